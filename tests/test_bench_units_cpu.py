"""The bench's roofline numerators against the per-unit figures they are
defined by (stated once here as numbers, not re-derived from bench.py's
code): algorithmic bytes and contraction FLOPs per token and head of the
delta-rule prefill at d = 64 and d = 128, and state bytes per decode step.
A changed workload shape or a dropped term in the bench's counting fails
here before it can skew a reported fraction."""
import os
import sys

import pytest

pytest.importorskip("torch")
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
import workloads as wl  # noqa: E402


def test_gpt2_prefill_units():
    w = wl.workload("gpt2_prefill")
    assert (w.ntok, w.H, w.dk, w.dv) == (16384, 12, 64, 64)
    nbytes, flops = bench.prefill_algo(w)
    # bf16 q, k, v, o (4 x 64 x 2 B) + one bf16 beta logit per token and head
    assert nbytes == 16384 * 12 * (4 * 64 * 2 + 2) == 101_056_512
    # 10 C d + 6 d^2 per token and head, C = 64, d = 64: 65 536
    assert flops == 16384 * 12 * 65_536


def test_gated_prefill_units():
    w = wl.workload("gated_prefill")
    assert (w.ntok, w.H, w.dk, w.dv) == (32768, 32, 128, 128)
    nbytes, flops = bench.prefill_algo(w)
    # + 128 bf16 gate logits per token and head
    assert nbytes == 32768 * 32 * (4 * 128 * 2 + 2 + 128 * 2)
    # 10 C d + 6 d^2 at d = 128: 180 224
    assert flops == 32768 * 32 * 180_224


def test_scalar_gate_counts_one_logit():
    w = wl.workload("gpt2_scalar_gate")
    assert w.gated and w.extra["scalar_gate"]
    nbytes, _ = bench.prefill_algo(w)
    assert nbytes == 16384 * 12 * (4 * 64 * 2 + 2 + 2)


def test_decode_state_bytes():
    w = wl.workload("decode")
    assert (w.n_seq, w.H, w.dk, w.dv) == (256, 32, 128, 128)
    # fp32 state read and written once: 8 bytes per element, 1 GiB per step
    assert bench.decode_state_bytes(w) == 256 * 32 * 128 * 128 * 8 == 1 << 30


def test_clock_summary_over_load_windows():
    """The clock median is taken over the samples inside the measured
    windows; throttle reasons are reported from those samples."""
    import bench
    cs = bench.ClockSampler(0, log_dir="/tmp")
    cs.proc = object()  # a sampler that ran
    row = lambda mhz, pc="Not Active": ["0", str(mhz), "2070", "500", "0x0", "Not Active",
                                        "Not Active", "Not Active", pc]
    cs.rows = [(0.0, row(800)), (1.0, row(2070)), (1.1, row(2060, "Active")), (3.0, row(900))]
    cs.windows = [(0.9, 1.2)]
    s = cs.summary()
    assert s["samples"] == 4 and s["samples_under_load"] == 2
    assert s["sm_mhz"] == 2065.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
