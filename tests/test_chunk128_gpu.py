"""Parity of the delta-rule prefill at chunk = 128 (bf16 I/O, dk = dv = 64):
the recurrence steps over 128-token chunks formed from pairs of 64-token
records, so every way a sequence can end relative to the pair boundary is
covered -- a last pair with one chunk of 1..64 tokens, a pair whose second
chunk is ragged, whole pairs, empty sequences -- against the oracle's
token-by-token recurrence, with and without gates and initial states."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _helpers import TOL, gpu_prefill_delta, oracle_prefill_delta, rel_err

pytestmark = pytest.mark.gpu

# lengths around the 64- and 128-token boundaries, an empty sequence
PAIRS = [1, 63, 64, 65, 127, 128, 129, 191, 192, 193, 0, 256, 300]


def check(la, inp, flags, oflags, scale=1.0):
    o, fS = gpu_prefill_delta(la, inp, flags=flags, scale=scale, chunk=128)
    ref_o, ref_S = oracle_prefill_delta(inp, flags=oflags, scale=scale)
    eo, es = rel_err(o.numpy(), ref_o), rel_err(fS.numpy(), ref_S)
    assert eo <= TOL[torch.bfloat16], f"output rel err {eo:.3e}"
    assert es <= TOL[torch.bfloat16], f"final state rel err {es:.3e}"


def test_chunk128_ragged_ungated(cuda_lib):
    inp = wl.prefill_inputs(PAIRS, 3, 64, 64, torch.bfloat16, False, seed=128, init_state=True)
    check(cuda_lib, inp, cuda_lib.LA_L2NORM_K, oracle.L2NORM_K)


def test_chunk128_ragged_per_channel_gate(cuda_lib):
    inp = wl.prefill_inputs(PAIRS, 2, 64, 64, torch.bfloat16, True, seed=129, init_state=True)
    check(cuda_lib, inp, cuda_lib.LA_L2NORM_K, oracle.L2NORM_K)


def test_chunk128_ragged_scalar_gate(cuda_lib):
    inp = wl.prefill_inputs(PAIRS, 2, 64, 64, torch.bfloat16, True, seed=130, init_state=True,
                            scalar_gate=True)
    check(cuda_lib, inp, cuda_lib.LA_L2NORM_K | cuda_lib.LA_GATE_SCALAR,
          oracle.L2NORM_K | oracle.SCALAR_GATE)


def test_chunk128_strong_gate(cuda_lib):
    """Decays close to 0 inside a chunk (gate logits around -1, so alpha
    down to ~0.3 per token): the pair's coupling multiplies e^{b_end} of the
    first chunk into the second chunk's operands."""
    inp = wl.prefill_inputs([200, 129, 64], 2, 64, 64, torch.bfloat16, True, seed=131,
                            init_state=True, gate_mean=-1.0)
    check(cuda_lib, inp, cuda_lib.LA_L2NORM_K, oracle.L2NORM_K)


@pytest.mark.parametrize("name", ["qnorm_silu", "additive"])
def test_chunk128_prologue_flags(cuda_lib, name):
    la = cuda_lib
    inp = wl.prefill_inputs([170, 64, 33], 2, 64, 64, torch.bfloat16, False, seed=132,
                            init_state=True)
    if name == "additive":
        check(la, inp, la.LA_L2NORM_K | la.LA_ADDITIVE, oracle.L2NORM_K | oracle.ADDITIVE, 0.5)
    else:
        check(la, inp, la.LA_L2NORM_K | la.LA_L2NORM_Q | la.LA_SILU_QK,
              oracle.L2NORM_K | oracle.L2NORM_Q | oracle.SILU_QK, 0.5)


def test_chunk128_many_sequences(cuda_lib):
    """More sequences than the intra-chunk kernel copies to shared memory
    (slot-major task order) and more (sequence, head) pairs than SMs."""
    rng = np.random.default_rng(133)
    lengths = [int(x) for x in rng.integers(0, 300, size=300)]
    inp = wl.prefill_inputs(lengths, 2, 64, 64, torch.bfloat16, False, seed=133)
    check(cuda_lib, inp, cuda_lib.LA_L2NORM_K, oracle.L2NORM_K)


def test_chunk128_gpt2_shape_full(cuda_lib):
    """The GPT-2-shaped workload (8 x 2048 tokens, 12 heads of 64) at chunk
    128, every head against the oracle, and against the chunk-64 path."""
    w = wl.workload("gpt2_prefill")
    inp = wl.inputs_for(w, seed=0)
    o128, s128 = gpu_prefill_delta(cuda_lib, inp, chunk=128)
    ref_o, ref_S = oracle_prefill_delta(inp)
    assert rel_err(o128.numpy(), ref_o) <= TOL[torch.bfloat16]
    assert rel_err(s128.numpy(), ref_S) <= TOL[torch.bfloat16]
    o64, s64 = gpu_prefill_delta(cuda_lib, inp, chunk=64)
    # two roundings of the same result: well inside the oracle tolerance
    assert rel_err(o128.numpy(), o64.numpy()) <= TOL[torch.bfloat16] / 2


def test_chunk128_repeated_calls_one_workspace(cuda_lib):
    """Back-to-back calls on one stream reuse the workspace; every result
    equals the first."""
    la = cuda_lib
    inp = wl.prefill_inputs([300, 129, 64], 4, 64, 64, torch.bfloat16, True, seed=134)
    dev = torch.device("cuda")
    t = {n: inp[n].to(dev) for n in ("q", "k", "v", "beta_logits", "gate_logits", "cu_seqlens")}
    ntok, H = t["q"].shape[0], t["q"].shape[1]
    need = la.la_prefill_delta_workspace_size(3, ntok, H, 64, 64, 128, la.LA_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(4):
        o = torch.empty((ntok, H, 64), dtype=torch.bfloat16, device=dev)
        la.la_prefill_delta(t["q"], t["k"], t["v"], t["beta_logits"], t["gate_logits"], o,
                            t["cu_seqlens"], chunk=128, workspace=ws)
        outs.append(o)
    assert la.la_check_device() == la.LA_OK
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
