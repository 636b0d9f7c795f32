"""GPU edge cases of the prefill paths against the oracle: batches whose
sequences are all empty, single-token sequences, many short sequences, a
write strength beta ~ 0, and decays strong enough that products of alpha
over a 16-token block leave the fp32 range (fast-forgetting key channels)."""
import pytest
import torch

import oracle
import workloads as wl
from _helpers import TOL, gpu_prefill_delta, oracle_prefill_delta, rel_err

pytestmark = pytest.mark.gpu

CASES = [(torch.float32, 64, 128), (torch.bfloat16, 64, 64), (torch.bfloat16, 128, 128)]


@pytest.mark.parametrize("dtype,dk,dv", CASES)
@pytest.mark.parametrize("gated", [False, True])
def test_all_sequences_empty_hand_states_through(cuda_lib, dtype, dk, dv, gated):
    """Every sequence empty (cu_seqlens all zero, some tokens outside every
    sequence): the final states are the initial states, no output is written."""
    la = cuda_lib
    dev = torch.device("cuda")
    inp = wl.prefill_inputs([5, 0, 0], 2, dk, dv, dtype, gated, seed=90, init_state=True)
    inp["cu_seqlens"] = torch.zeros(4, dtype=torch.int32)
    t = {n: (None if inp[n] is None else inp[n].to(dev))
         for n in ("q", "k", "v", "beta_logits", "gate_logits", "init_S")}
    o = torch.full(t["v"].shape, float("nan"), dtype=dtype, device=dev)
    fS = torch.full(t["init_S"].shape, float("nan"), device=dev)
    la.la_prefill_delta(t["q"], t["k"], t["v"], t["beta_logits"], t["gate_logits"], o,
                        inp["cu_seqlens"].to(dev), init_S=t["init_S"], final_S=fS,
                        cu_seqlens_host=inp["cu_seqlens"])
    assert la.la_check_device() == la.LA_OK
    assert torch.equal(fS.cpu(), inp["init_S"])
    assert torch.isnan(o.float().cpu()).all()


@pytest.mark.parametrize("dtype,dk,dv", CASES)
def test_single_token_sequences(cuda_lib, dtype, dk, dv):
    inp = wl.prefill_inputs([1] * 9, 3, dk, dv, dtype, True, seed=91, init_state=True)
    o, fS = gpu_prefill_delta(cuda_lib, inp)
    ref_o, ref_S = oracle_prefill_delta(inp)
    assert rel_err(o.numpy(), ref_o) <= TOL[dtype]
    assert rel_err(fS.numpy(), ref_S) <= TOL[dtype]


def test_many_short_sequences_tensor_core_path(cuda_lib):
    """600 sequences of 1..130 tokens, one head: many chunk slots and gaps."""
    g = torch.Generator().manual_seed(92)
    lengths = torch.randint(1, 131, (600,), generator=g).tolist()
    inp = wl.prefill_inputs(lengths, 1, 64, 64, torch.bfloat16, False, seed=93, init_state=True)
    o, fS = gpu_prefill_delta(cuda_lib, inp)
    ref_o, ref_S = oracle_prefill_delta(inp)
    assert rel_err(o.numpy(), ref_o) <= TOL[torch.bfloat16]
    assert rel_err(fS.numpy(), ref_S) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("dtype,dk,dv", CASES)
def test_beta_near_zero_only_decays(cuda_lib, dtype, dk, dv):
    inp = wl.prefill_inputs([150, 70], 2, dk, dv, dtype, True, seed=94, init_state=True)
    inp["beta_logits"] = torch.full_like(inp["beta_logits"], -30.0)
    o, fS = gpu_prefill_delta(cuda_lib, inp)
    ref_o, ref_S = oracle_prefill_delta(inp)
    assert rel_err(o.numpy(), ref_o) <= TOL[dtype]
    assert rel_err(fS.numpy(), ref_S) <= TOL[dtype]


@pytest.mark.parametrize("dtype,dk,dv", CASES)
@pytest.mark.parametrize("scalar", [False, True])
def test_strong_decay(cuda_lib, dtype, dk, dv, scalar):
    """Gate logits around +9 (alpha ~ 1e-4 per token: a 16-token product near
    1e-64) on a random half of the key channels (or of the tokens, with a
    scalar gate), ordinary ones elsewhere."""
    inp = wl.prefill_inputs([200, 77], 2, dk, dv, dtype, True, seed=95, init_state=True,
                            scalar_gate=scalar)
    g = torch.Generator().manual_seed(96)
    gl = inp["gate_logits"].float()
    strong = torch.rand(gl.shape, generator=g) < 0.5
    inp["gate_logits"] = torch.where(strong, gl + 7.0, gl).to(dtype)
    flags = cuda_lib.LA_L2NORM_K | (cuda_lib.LA_GATE_SCALAR if scalar else 0)
    oflags = oracle.L2NORM_K | (oracle.SCALAR_GATE if scalar else 0)
    o, fS = gpu_prefill_delta(cuda_lib, inp, flags=flags)
    ref_o, ref_S = oracle_prefill_delta(inp, flags=oflags)
    assert rel_err(o.numpy(), ref_o) <= TOL[dtype]
    assert rel_err(fS.numpy(), ref_S) <= TOL[dtype]
