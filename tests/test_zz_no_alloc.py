"""The allocation-free prefill entry point, la_prefill_delta_static, which
takes its scratch from the library's static device buffer instead of a
caller workspace, gives exactly the results of la_prefill_delta.

Two different problems go through the static entry point back to back, then
the first again, so stale scratch contents from one call could only go
unnoticed if they never matter.  The file name keeps it last in collection;
it passes alone and after the other GPU tests."""
import pytest
import torch

import delta_rule_recurrent_chunkwise_gb300 as la
import workloads as wl

pytestmark = pytest.mark.gpu

# (lengths, heads, head size, gated): ragged sequences spanning several
# chunks; the tensor-core path (bf16, dk == dv) takes the static scratch.
PROBLEMS = [
    ((200, 64, 1, 130), 4, 64, False),
    ((300, 77, 129), 2, 128, True),
]


def _device_inputs(problem, seed):
    lengths, H, D, gated = problem
    inp = wl.prefill_inputs(list(lengths), H, D, D, torch.bfloat16, gated, seed=seed,
                            init_state=True)
    dev = torch.device("cuda")
    return {n: (None if t is None else t.to(dev)) for n, t in inp.items()}, inp["cu_seqlens"]


def _run(entry, t, cu_host):
    N, H, D = t["cu_seqlens"].numel() - 1, t["q"].shape[1], t["q"].shape[2]
    o = torch.full_like(t["v"], float("nan"))
    fS = torch.full((N, H, D, D), float("nan"), device=t["q"].device)
    entry(t["q"], t["k"], t["v"], t["beta_logits"], t["gate_logits"], o, t["cu_seqlens"],
          init_S=t["init_S"], final_S=fS, cu_seqlens_host=cu_host)
    assert la.la_check_device() == la.LA_OK
    return o, fS


def test_static_scratch_matches_workspace_entry_point():
    la.build()
    runs = [_device_inputs(p, seed=11 + i) for i, p in enumerate(PROBLEMS)]
    for t, _ in runs:
        N, H, D = t["cu_seqlens"].numel() - 1, t["q"].shape[1], t["q"].shape[2]
        need = la.la_prefill_delta_workspace_size(N, t["q"].shape[0], H, D, D)
        assert 0 < need <= la.LA_STATIC_SCRATCH_BYTES
    ref = [_run(la.la_prefill_delta, t, cu) for t, cu in runs]
    for i in (0, 1, 0):
        t, cu = runs[i]
        o, fS = _run(la.la_prefill_delta_static, t, cu)
        assert torch.isfinite(o.float()).all() and torch.isfinite(fS).all()
        assert torch.equal(o, ref[i][0]), f"problem {i}: outputs differ"
        assert torch.equal(fS, ref[i][1]), f"problem {i}: final states differ"


def test_static_scratch_at_chunk_128():
    """The same at chunk 128 (bf16, d = 64): the recurrence over 128-token
    chunks reads the 64-token records from the static scratch."""
    la.build()
    t, cu = _device_inputs(((200, 64, 1, 130), 4, 64, False), seed=21)

    def at128(entry):
        return lambda *a, **k: entry(*a, chunk=128, **k)
    ref = _run(at128(la.la_prefill_delta), t, cu)
    o, fS = _run(at128(la.la_prefill_delta_static), t, cu)
    assert torch.equal(o, ref[0]) and torch.equal(fS, ref[1])


def test_static_scratch_refuses_oversize_request():
    la.build()
    dev = torch.device("cuda")
    # 4 x 8192 tokens, 32 heads, d = 128: about 1.2 GB of chunk records
    H, D, ntok = 32, 128, 4 * 8192
    assert la.la_prefill_delta_workspace_size(4, ntok, H, D, D) > la.LA_STATIC_SCRATCH_BYTES
    q = torch.zeros((ntok, H, D), dtype=torch.bfloat16, device=dev)
    bl = torch.zeros((ntok, H), dtype=torch.bfloat16, device=dev)
    cu = torch.tensor([0, 8192, 16384, 24576, 32768], dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    with pytest.raises(la.LinAttnError) as e:
        la.la_prefill_delta_static(q, q, q, bl, None, o, cu)
    assert e.value.status == la.LA_ERR_TOO_LARGE
