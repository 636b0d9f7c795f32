"""GPU checks of the invariances the method fixes, on the tensor-core path
(bf16 I/O, dk = dv): a prefill split at a chunk boundary and resumed from its
final state equals the single prefill bit for bit; split mid-chunk it agrees
within the bf16 bar; 64 recurrent decode steps equal a 64-token prefill from
the same state; packing sequences into one varlen batch changes nothing; and
tokens outside every sequence are never written."""
import pytest
import torch

import workloads as wl
from _helpers import TOL, gpu_prefill_delta, oracle_prefill_delta, rel_err

pytestmark = pytest.mark.gpu

SEQ = ("q", "k", "v", "beta_logits", "gate_logits")


def _slice(inp, a, b, init_S):
    out = {n: (None if inp[n] is None else inp[n][a:b]) for n in SEQ}
    out.update(cu_seqlens=torch.tensor([0, b - a], dtype=torch.int32), init_S=init_S)
    return out


@pytest.mark.parametrize("D,gated", [(64, False), (128, True)])
def test_split_at_chunk_boundary_is_bitwise_identical(cuda_lib, D, gated):
    T, t1 = 300, 128
    inp = wl.prefill_inputs([T], 3, D, D, torch.bfloat16, gated, seed=21, init_state=True)
    full_o, full_S = gpu_prefill_delta(cuda_lib, inp)
    o1, S1 = gpu_prefill_delta(cuda_lib, _slice(inp, 0, t1, inp["init_S"]))
    o2, S2 = gpu_prefill_delta(cuda_lib, _slice(inp, t1, T, S1))
    assert torch.equal(torch.cat([o1, o2]), full_o)
    assert torch.equal(S2, full_S)


@pytest.mark.parametrize("D,gated", [(64, False), (128, True)])
def test_split_mid_chunk_agrees(cuda_lib, D, gated):
    T, t1 = 300, 131
    inp = wl.prefill_inputs([T], 3, D, D, torch.bfloat16, gated, seed=22, init_state=True)
    full_o, full_S = gpu_prefill_delta(cuda_lib, inp)
    o1, S1 = gpu_prefill_delta(cuda_lib, _slice(inp, 0, t1, inp["init_S"]))
    o2, S2 = gpu_prefill_delta(cuda_lib, _slice(inp, t1, T, S1))
    ref_o, ref_S = oracle_prefill_delta(inp)
    split_o = torch.cat([o1, o2]).numpy()
    assert rel_err(split_o, ref_o) <= TOL[torch.bfloat16]
    assert rel_err(S2.numpy(), ref_S) <= TOL[torch.bfloat16]
    assert rel_err(split_o, full_o.numpy()) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("D,gated", [(64, False), (128, True)])
def test_decode_steps_equal_prefill(cuda_lib, D, gated):
    """64 decode steps from a state give the outputs and state of a 64-token
    prefill from the same state (both paths against each other and the oracle)."""
    la = cuda_lib
    dev = torch.device("cuda")
    T, H = 64, 2
    inp = wl.prefill_inputs([T], H, D, D, torch.bfloat16, gated, seed=23, init_state=True)
    pre_o, pre_S = gpu_prefill_delta(la, inp)
    state = inp["init_S"][0:1].clone().to(dev)          # [1][H][D][D]
    dec_o = []
    for t in range(T):
        tok = {n: (None if inp[n] is None else inp[n][t:t + 1].to(dev)) for n in SEQ}
        o = torch.empty((1, H, D), dtype=torch.bfloat16, device=dev)
        la.la_decode_step(tok["q"], tok["k"], tok["v"], tok["beta_logits"], tok["gate_logits"], o,
                          state)
        dec_o.append(o)
    assert la.la_check_device() == la.LA_OK
    dec_o = torch.cat(dec_o).float().cpu().numpy()
    ref_o, ref_S = oracle_prefill_delta(inp)
    tol = TOL[torch.bfloat16]
    assert rel_err(dec_o, ref_o) <= tol
    assert rel_err(state.cpu().numpy(), ref_S) <= tol
    assert rel_err(dec_o, pre_o.numpy()) <= tol
    assert rel_err(state.cpu().numpy(), pre_S.numpy()) <= tol


@pytest.mark.parametrize("D,gated", [(64, False), (128, True)])
def test_varlen_packing_equals_separate_runs(cuda_lib, D, gated):
    lengths = [200, 77, 1, 0, 128, 65]
    inp = wl.prefill_inputs(lengths, 2, D, D, torch.bfloat16, gated, seed=24, init_state=True)
    packed_o, packed_S = gpu_prefill_delta(cuda_lib, inp)
    cu = inp["cu_seqlens"].tolist()
    for n, L in enumerate(lengths):
        if L == 0:  # an empty sequence hands its initial state through
            assert torch.equal(packed_S[n], inp["init_S"][n])
            continue
        alone = _slice(inp, cu[n], cu[n + 1], inp["init_S"][n:n + 1])
        o, S = gpu_prefill_delta(cuda_lib, alone)
        assert torch.equal(o, packed_o[cu[n]:cu[n + 1]]), f"sequence {n}"
        assert torch.equal(S[0], packed_S[n]), f"sequence {n} state"


def test_tokens_outside_sequences_are_not_written(cuda_lib):
    """ntok larger than cu_seqlens[N]: the trailing tokens belong to no
    sequence; their output rows keep what the caller put there."""
    la = cuda_lib
    dev = torch.device("cuda")
    lengths, extra, H, D = [130, 64], 90, 2, 64
    inp = wl.prefill_inputs(lengths + [extra], H, D, D, torch.bfloat16, False, seed=25)
    inp["cu_seqlens"] = inp["cu_seqlens"][:-1].clone()   # last "sequence" is not one
    t = {n: (None if inp[n] is None else inp[n].to(dev)) for n in SEQ}
    o = torch.full(t["v"].shape, float("nan"), dtype=torch.bfloat16, device=dev)
    la.la_prefill_delta(t["q"], t["k"], t["v"], t["beta_logits"], None, o,
                        inp["cu_seqlens"].to(dev), cu_seqlens_host=inp["cu_seqlens"])
    assert la.la_check_device() == la.LA_OK
    o = o.float().cpu()
    n_in = sum(lengths)
    assert torch.isnan(o[n_in:]).all()
    head = {n: (None if inp[n] is None else inp[n][:n_in]) for n in SEQ}
    head["cu_seqlens"] = inp["cu_seqlens"]
    ref_o, _ = oracle_prefill_delta(head, init=False)
    assert rel_err(o[:n_in].numpy(), ref_o) <= TOL[torch.bfloat16]
