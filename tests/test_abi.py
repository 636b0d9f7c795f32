"""Host-only checks of the C ABI: the library builds for sm_103a, loads, exports
every function that include/linattn.h declares, and rejects bad arguments on
the host before any launch (these calls never reach the GPU)."""
import ctypes
import os
import re

import pytest

import delta_rule_recurrent_chunkwise_gb300 as la

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    la.build()
    return la.library()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\w[\w\s\*]*?\b(la_\w+)\s*\(", text, flags=re.M))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("la_prefill_linear", "la_prefill_delta", "la_decode_step"):
        assert required in names
    assert set(la.EXPORTED) <= names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert la.la_status_string(la.LA_OK) == "LA_OK"
    for s in (1, 2, 3, 4, 5):
        assert la.la_status_string(s).startswith("LA_ERR_")
    assert la.la_status_string(99) == "LA_ERR_UNKNOWN"


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below is rejected first


def prefill_delta(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bl=FAKE, gl=None, o=FAKE, io=la.LA_BF16, cu=FAKE,
             cuh=None, N=2, ntok=40, H=4, dk=64, dv=64, chunk=64, scale=1.0,
             flags=la.LA_L2NORM_K, iS=None, fS=None, ws=FAKE, wsb=1 << 40, stream=None)
    a.update(kw)
    return lib.la_prefill_delta(a["q"], a["k"], a["v"], a["bl"], a["gl"], a["o"], a["io"],
                                a["cu"], a["cuh"], a["N"], a["ntok"], a["H"], a["dk"], a["dv"],
                                a["chunk"],
                                a["scale"], a["flags"], a["iS"], a["fS"], a["ws"], a["wsb"],
                                a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), la.LA_ERR_INVALID_ARG),
    (dict(bl=None), la.LA_ERR_INVALID_ARG),
    (dict(cu=None), la.LA_ERR_INVALID_ARG),
    (dict(N=0), la.LA_ERR_INVALID_ARG),
    (dict(H=-1), la.LA_ERR_INVALID_ARG),
    (dict(ntok=-5), la.LA_ERR_INVALID_ARG),
    (dict(io=7), la.LA_ERR_INVALID_ARG),
    (dict(flags=64), la.LA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), la.LA_ERR_INVALID_ARG),
    (dict(dk=96), la.LA_ERR_UNSUPPORTED),
    (dict(dv=32), la.LA_ERR_UNSUPPORTED),
    (dict(chunk=96), la.LA_ERR_UNSUPPORTED),
    (dict(chunk=256), la.LA_ERR_UNSUPPORTED),
    (dict(chunk=128, dk=128, dv=128), la.LA_ERR_UNSUPPORTED),   # chunk 128: d = 64 only
    (dict(chunk=128, io=la.LA_F32), la.LA_ERR_UNSUPPORTED),     # and the tensor-core path only
    (dict(chunk=0), la.LA_ERR_INVALID_ARG),
])
def test_prefill_delta_rejects_bad_arguments(lib, kw, code):
    assert prefill_delta(lib, **kw) == code


def test_non_monotone_host_cu_seqlens_rejected(lib):
    bad = (ctypes.c_int32 * 3)(0, 10, 5)
    assert prefill_delta(lib, cuh=bad) == la.LA_ERR_INVALID_ARG
    neg = (ctypes.c_int32 * 3)(-1, 10, 20)
    assert prefill_delta(lib, cuh=neg) == la.LA_ERR_INVALID_ARG
    past_end = (ctypes.c_int32 * 3)(0, 10, 41)   # beyond ntok = 40
    assert prefill_delta(lib, cuh=past_end) == la.LA_ERR_INVALID_ARG
    assert lib.la_prefill_linear(FAKE, FAKE, FAKE, FAKE, la.LA_F32, FAKE, bad, 2, 40, 1, 64, 64,
                                 None, None, None, None, None) == la.LA_ERR_INVALID_ARG


def test_decode_and_linear_reject_bad_arguments(lib):
    d = lib.la_decode_step
    assert d(FAKE, FAKE, FAKE, FAKE, None, FAKE, la.LA_BF16, 4, 2, 128, 128, 1.0, 1, None,
             None) == la.LA_ERR_INVALID_ARG          # no state
    assert d(FAKE, FAKE, FAKE, FAKE, None, FAKE, la.LA_BF16, 4, 2, 100, 128, 1.0, 1, FAKE,
             None) == la.LA_ERR_UNSUPPORTED
    assert d(FAKE, FAKE, FAKE, FAKE, None, FAKE, la.LA_BF16, 0, 2, 128, 128, 1.0, 1, FAKE,
             None) == la.LA_ERR_INVALID_ARG
    assert lib.la_prefill_linear(None, FAKE, FAKE, FAKE, la.LA_F32, FAKE, None, 1, 8, 1, 64, 64,
                                 None, None, None, None, None) == la.LA_ERR_INVALID_ARG
    assert lib.la_prefill_linear(FAKE, FAKE, FAKE, FAKE, la.LA_F32, FAKE, None, 1, 8, 1, 48, 64,
                                 None, None, None, None, None) == la.LA_ERR_UNSUPPORTED


def test_workspace_size_covers_the_chunk_records(lib):
    """The tensor-core path (bf16 I/O, dk == dv in {64, 128}) keeps one record
    per (64-token chunk slot, head), then one 4-byte flag per record and two
    task counters (256 bytes) for the launch that runs both halves together;
    every other configuration needs none."""
    ws = la.la_prefill_delta_workspace_size
    assert ws(4, 1024, 32, 128, 128, 64, la.LA_F32) == 0
    assert ws(4, 1024, 32, 64, 128, 64, la.LA_BF16) == 0
    rec = {64: 4 * 64 * 64 * 2 + 8192 + 4 * 64, 128: 4 * 64 * 128 * 2 + 8192 + 4 * 128}
    for D in (64, 128):
        rec_bytes = (rec[D] + 1023) // 1024 * 1024
        for N, ntok, H in ((1, 64, 1), (4, 1024, 32), (5, 65536, 16), (3, 100, 2)):
            slots = ntok // 64 + N + 1
            table = (slots * 8 + 1023) // 1024 * 1024
            flags = (slots * H * 4 + 255) // 256 * 256 + 256
            assert ws(N, ntok, H, D, D, 64, la.LA_BF16) == table + slots * H * rec_bytes + flags
    # chunk 128 (d = 64) keeps the 64-token records: the same bytes; no other
    # configuration takes it
    for N, ntok, H in ((1, 64, 1), (4, 1024, 32), (3, 100, 2)):
        assert ws(N, ntok, H, 64, 64, 128, la.LA_BF16) == ws(N, ntok, H, 64, 64, 64, la.LA_BF16)
    assert ws(4, 1024, 32, 128, 128, 128, la.LA_BF16) == 0
    assert ws(4, 1024, 32, 64, 64, 96, la.LA_BF16) == 0


def test_prefill_rejects_missing_workspace(lib):
    """A call that needs a workspace and gets none (or too little, or a
    misaligned one) is refused on the host before any launch."""
    need = la.la_prefill_delta_workspace_size(2, 256, 4, 64, 64, 64, la.LA_BF16)
    assert need > 0
    d = lib.la_prefill_delta
    args = (FAKE, FAKE, FAKE, FAKE, None, FAKE, la.LA_BF16, FAKE, None, 2, 256, 4, 64, 64, 64,
            1.0, 1, None, None)
    assert d(*args, None, 0, None) == la.LA_ERR_INVALID_ARG
    assert d(*args, FAKE, need - 1, None) == la.LA_ERR_INVALID_ARG
    assert d(*args, ctypes.c_void_p(0x1010), need, None) == la.LA_ERR_INVALID_ARG


def test_static_entry_point_refuses_requests_beyond_its_scratch(lib):
    """la_prefill_delta_static answers LA_ERR_TOO_LARGE, on the host and
    before any launch, when the sizes need more scratch than its static
    buffer; a request that fits is not refused for size."""
    d = lib.la_prefill_delta_static
    ws = la.la_prefill_delta_workspace_size
    big = (4, 8192 * 4, 32, 128, 128)
    assert ws(*big, 64, la.LA_BF16) > la.LA_STATIC_SCRATCH_BYTES
    assert d(FAKE, FAKE, FAKE, FAKE, None, FAKE, la.LA_BF16, FAKE, None, *big, 64, 1.0, 1,
             None, None, None) == la.LA_ERR_TOO_LARGE
    small = (2, 256, 4, 64, 64)
    assert ws(*small, 64, la.LA_BF16) <= la.LA_STATIC_SCRATCH_BYTES
    bad = (ctypes.c_int32 * 3)(0, 10, 5)   # rejected later, for its cu_seqlens_host
    assert d(FAKE, FAKE, FAKE, FAKE, None, FAKE, la.LA_BF16, FAKE, bad, *small, 64, 1.0, 1,
             None, None, None) == la.LA_ERR_INVALID_ARG


def test_scalar_gate_flag_needs_gate_logits(lib):
    """LA_GATE_SCALAR says how to read gate_logits; without them it is an
    argument error (prefill, allocation-free prefill and decode)."""
    args = (FAKE, FAKE, FAKE, FAKE, None, FAKE, la.LA_BF16, FAKE, None, 2, 40, 4, 64, 64, 64,
            1.0, la.LA_L2NORM_K | la.LA_GATE_SCALAR, None, None)
    assert lib.la_prefill_delta(*args, FAKE, 1 << 40, None) == la.LA_ERR_INVALID_ARG
    assert lib.la_prefill_delta_static(*args, None) == la.LA_ERR_INVALID_ARG
    assert lib.la_decode_step(FAKE, FAKE, FAKE, FAKE, None, FAKE, la.LA_BF16, 4, 2, 128, 128, 1.0,
                              la.LA_L2NORM_K | la.LA_GATE_SCALAR, FAKE, None) == la.LA_ERR_INVALID_ARG


def test_decode_slots_rejects_bad_arguments(lib):
    """The slot-map decode checks its own arguments (and la_decode_step's) on
    the host before touching the GPU."""
    d = lib.la_decode_step_slots
    base = (FAKE, FAKE, FAKE, FAKE, None, FAKE, la.LA_BF16, 4, 2, 128, 128, 1.0, 1)
    assert d(*base, FAKE, 8, None, None) == la.LA_ERR_INVALID_ARG       # no slot map
    assert d(*base, FAKE, 0, FAKE, None) == la.LA_ERR_INVALID_ARG       # empty pool
    assert d(*base, None, 8, FAKE, None) == la.LA_ERR_INVALID_ARG       # no pool
    assert d(FAKE, FAKE, FAKE, FAKE, None, FAKE, la.LA_BF16, 4, 2, 96, 128, 1.0, 1, FAKE, 8,
             FAKE, None) == la.LA_ERR_UNSUPPORTED
    assert d(FAKE, FAKE, FAKE, FAKE, None, FAKE, la.LA_BF16, 4, 2, 128, 128, 1.0,
             la.LA_GATE_SCALAR, FAKE, 8, FAKE, None) == la.LA_ERR_INVALID_ARG


def test_backward_checks_arguments_and_workspace(lib):
    """la_backward_delta: the forward call's checks, its own outputs, and a
    workspace of la_backward_delta_workspace_size bytes (chunk-start states
    plus per-token sums), all before any launch."""
    N, ntok, H, d = 2, 40, 4, 64
    need = la.la_backward_delta_workspace_size(N, ntok, H, d, d)
    slots = ntok // 64 + N + 1
    assert need >= slots * H * d * d * 4 + ntok * H * 3 * d * 4 + ntok * H * 4
    assert la.la_backward_delta_workspace_size(N, ntok, H, 96, d) == 0
    b = lib.la_backward_delta
    head = (FAKE, FAKE, FAKE, FAKE, None, FAKE, None, la.LA_BF16, FAKE, None, N, ntok, H, d, d,
            1.0, la.LA_L2NORM_K, None)
    outs = (FAKE, FAKE, FAKE, FAKE, None, None)
    assert b(*head, *outs, None, need, None) == la.LA_ERR_INVALID_ARG          # no workspace
    assert b(*head, *outs, FAKE, need - 1, None) == la.LA_ERR_INVALID_ARG      # too small
    assert b(*head, None, *outs[1:], FAKE, need, None) == la.LA_ERR_INVALID_ARG  # no dq
    gated = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, la.LA_BF16, FAKE, None, N, ntok, H, d, d,
             1.0, la.LA_L2NORM_K, None)
    assert b(*gated, *outs, FAKE, need, None) == la.LA_ERR_INVALID_ARG         # no d_gate_logits
    odd = head[:13] + (96,) + head[14:]
    assert b(*odd, *outs, FAKE, need, None) == la.LA_ERR_UNSUPPORTED


def test_training_pair_checks_arguments_and_saved_buffer(lib):
    """la_prefill_delta_train / la_backward_delta_saved: the forward call's
    checks, the chunkwise configurations only (bf16, dk = dv), and a saved
    buffer of la_backward_delta_workspace_size bytes, 256-byte aligned, all
    before any launch."""
    N, ntok, H, d = 2, 40, 4, 64
    need = la.la_backward_delta_workspace_size(N, ntok, H, d, d)
    MIS = ctypes.c_void_p(0x1000 + 128)   # not 256-byte aligned
    t = lib.la_prefill_delta_train
    fwd = (FAKE, FAKE, FAKE, FAKE, None, FAKE)
    tail = (1.0, la.LA_L2NORM_K, None, None)
    assert t(*fwd, la.LA_BF16, FAKE, None, N, ntok, H, d, d, *tail, None, need, None) == \
        la.LA_ERR_INVALID_ARG                                                       # no buffer
    assert t(*fwd, la.LA_BF16, FAKE, None, N, ntok, H, d, d, *tail, FAKE, need - 1, None) == \
        la.LA_ERR_INVALID_ARG                                                       # too small
    assert t(*fwd, la.LA_BF16, FAKE, None, N, ntok, H, d, d, *tail, MIS, need, None) == \
        la.LA_ERR_INVALID_ARG                                                       # misaligned
    assert t(*fwd, la.LA_F32, FAKE, None, N, ntok, H, d, d, *tail, FAKE, need, None) == \
        la.LA_ERR_UNSUPPORTED                                                       # fp32 I/O
    assert t(*fwd, la.LA_BF16, FAKE, None, N, ntok, H, d, 128, *tail, FAKE, need, None) == \
        la.LA_ERR_UNSUPPORTED                                                       # dk != dv
    assert t(*fwd[:5], None, la.LA_BF16, FAKE, None, N, ntok, H, d, d, *tail, FAKE, need,
             None) == la.LA_ERR_INVALID_ARG                                          # no o
    b = lib.la_backward_delta_saved
    head = (FAKE, FAKE, FAKE, FAKE, None, FAKE, None, la.LA_BF16, FAKE, None, N, ntok, H, d, d,
            1.0, la.LA_L2NORM_K, None)
    outs = (FAKE, FAKE, FAKE, FAKE, None, None)
    assert b(*head, *outs, None, need, None) == la.LA_ERR_INVALID_ARG
    assert b(*head, *outs, FAKE, need - 1, None) == la.LA_ERR_INVALID_ARG
    assert b(*head, *outs, MIS, need, None) == la.LA_ERR_INVALID_ARG
    assert b(*head, None, *outs[1:], FAKE, need, None) == la.LA_ERR_INVALID_ARG  # no dq
    f32 = head[:7] + (la.LA_F32,) + head[8:]
    assert b(*f32, *outs, FAKE, need, None) == la.LA_ERR_UNSUPPORTED


def test_launch_count_query(lib):
    """la_prefill_delta_launches: 1 for the CUDA-core path, 1 or 2 for the
    tensor-core path (2 wherever no device can hold the one-launch grid, as
    on a machine without a GPU), 0 for arguments la_prefill_delta rejects."""
    q = la.la_prefill_delta_launches
    assert q(2, 256, 4, 64, 64, io=la.LA_F32) == 1
    assert q(2, 256, 4, 128, 128, io=la.LA_BF16, has_gate=True) == 2
    assert q(2, 256, 4, 64, 64, io=la.LA_BF16) in (1, 2)
    import torch
    if not torch.cuda.is_available():
        assert q(2, 256, 4, 64, 64, io=la.LA_BF16) == 2
    assert q(2, 256, 4, 96, 96, io=la.LA_BF16) == 0          # unsupported head size
    assert q(0, 256, 4, 64, 64, io=la.LA_BF16) == 0           # no sequence
    assert q(2, 256, 4, 64, 64, io=la.LA_BF16, flags=la.LA_GATE_SCALAR) == 0  # scalar gate, no gate
    assert q(2, 256, 4, 64, 64, chunk=128, io=la.LA_BF16) == 2              # intra, then the 128-token recurrence
    assert q(2, 256, 4, 128, 128, chunk=128, io=la.LA_BF16) == 0
    assert q(2, 256, 4, 64, 64, chunk=128, io=la.LA_F32) == 0
