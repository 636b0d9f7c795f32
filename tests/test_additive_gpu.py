"""GPU parity of the additive decayed rule (LA_ADDITIVE: u = v, the page's
Mamba-2 form S_t = alpha_t S_{t-1} + k_t v_t^T) against the oracle, on every
path: the CUDA-core prefill (fp32), the tensor-core prefill (bf16, dk = dv),
the decode step and the backward pass."""
import pytest
import torch

import oracle
import workloads as wl
from _helpers import TOL, f64, gpu_prefill_delta, oracle_prefill_delta, rel_err

pytestmark = pytest.mark.gpu

RAGGED = [200, 77, 1, 0, 128, 65]


def _flags(la, gate):
    return (la.LA_L2NORM_K | la.LA_ADDITIVE | (la.LA_GATE_SCALAR if gate == "scalar" else 0),
            oracle.L2NORM_K | oracle.ADDITIVE | (oracle.SCALAR_GATE if gate == "scalar" else 0))


@pytest.mark.parametrize("dtype,dk,dv", [(torch.float32, 64, 128), (torch.float32, 128, 64),
                                         (torch.bfloat16, 64, 64), (torch.bfloat16, 128, 128)])
@pytest.mark.parametrize("gate", ["none", "channel", "scalar"])
def test_additive_prefill_ragged(cuda_lib, dtype, dk, dv, gate):
    inp = wl.prefill_inputs(RAGGED, 2, dk, dv, dtype, gate != "none", seed=80 + dk + dv,
                            init_state=True, scalar_gate=gate == "scalar")
    inp["beta_logits"] = None          # ignored by the additive rule
    f, of = _flags(cuda_lib, gate)
    o, fS = gpu_prefill_delta(cuda_lib, inp, flags=f)
    ref_o, ref_S = oracle_prefill_delta(inp, flags=of)
    assert rel_err(o.numpy(), ref_o) <= TOL[dtype]
    assert rel_err(fS.numpy(), ref_S) <= TOL[dtype]


def test_additive_gpt2_shape_scalar_gate_full(cuda_lib):
    """The Mamba-2 form at the GPT-2 prefill shape (8 x 2048 tokens, 12 heads,
    d = 64, bf16, one decay per token and head), every output checked."""
    w = wl.workload("gpt2_scalar_gate")
    inp = wl.inputs_for(w, seed=3)
    f, of = _flags(cuda_lib, "scalar")
    o, fS = gpu_prefill_delta(cuda_lib, inp, flags=f)
    ref_o, ref_S = oracle_prefill_delta(inp, flags=of)
    assert rel_err(o.numpy(), ref_o) <= TOL[w.dtype]
    assert rel_err(fS.numpy(), ref_S) <= TOL[w.dtype]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("gate", ["channel", "scalar"])
def test_additive_decode(cuda_lib, dtype, gate):
    la = cuda_lib
    dev = torch.device("cuda")
    inp = wl.decode_inputs(5, 3, 128, 64, 3, dtype, seed=81, scalar_gate=gate == "scalar")
    f, of = _flags(la, gate)
    st = inp["state"].clone().to(dev)
    ref_st = f64(inp["state"])
    for t in range(3):
        tok = {n: inp[n][t] for n in ("q", "k", "v", "gate_logits")}
        o = torch.empty(tok["v"].shape, dtype=dtype, device=dev)
        la.la_decode_step(tok["q"].to(dev), tok["k"].to(dev), tok["v"].to(dev), None,
                          tok["gate_logits"].to(dev), o, st, flags=f)
        ref_o, ref_st = oracle.decode(f64(tok["q"]), f64(tok["k"]), f64(tok["v"]), None,
                                      f64(tok["gate_logits"]), ref_st, flags=of)
        assert rel_err(o.float().cpu().numpy(), ref_o) <= TOL[dtype]
    assert la.la_check_device() == la.LA_OK
    assert rel_err(st.cpu().numpy(), ref_st) <= TOL[dtype]


@pytest.mark.parametrize("gate", ["channel", "scalar"])
def test_additive_backward(cuda_lib, gate):
    la = cuda_lib
    dev = torch.device("cuda")
    inp = wl.prefill_inputs([150, 0, 70], 2, 64, 128, torch.float32, True, seed=82,
                            init_state=True, scalar_gate=gate == "scalar")
    f, of = _flags(la, gate)
    g = torch.Generator().manual_seed(83)
    d_o = torch.randn(inp["v"].shape, generator=g)
    d_fS = torch.randn(inp["init_S"].shape, generator=g) * 0.1
    t = {n: inp[n].to(dev) for n in ("q", "k", "v", "gate_logits", "init_S")}
    got = la.la_backward_delta(t["q"], t["k"], t["v"], None, t["gate_logits"], d_o.to(dev),
                               inp["cu_seqlens"].to(dev), d_final_S=d_fS.to(dev), flags=f,
                               init_S=t["init_S"], cu_seqlens_host=inp["cu_seqlens"])
    assert la.la_check_device() == la.LA_OK
    ref = oracle.delta_backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), None,
                                f64(inp["gate_logits"]), inp["cu_seqlens"].numpy(), f64(d_o),
                                f64(d_fS), flags=of, init_S=f64(inp["init_S"]))
    for n in ("dq", "dk", "dv", "d_gate_logits", "d_init_S"):
        assert rel_err(got[n].cpu().numpy(), ref[n]) <= 1e-4, n
    assert float(got["d_beta_logits"].abs().max()) == 0.0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("gate", ["none", "channel", "scalar"])
def test_additive_backward_chunkwise(cuda_lib, d, gate):
    """bf16, dk = dv: the chunkwise backward (beta = 1, W = 0, T = I), ragged
    lengths with an empty sequence, initial states and a final-state
    gradient, against the oracle."""
    la = cuda_lib
    dev = torch.device("cuda")
    inp = wl.prefill_inputs([150, 0, 70, 64], 2, d, d, torch.bfloat16, gate != "none", seed=84,
                            init_state=True, scalar_gate=gate == "scalar")
    f = la.LA_ADDITIVE | la.LA_L2NORM_K | (la.LA_GATE_SCALAR if gate == "scalar" else 0)
    of = oracle.ADDITIVE | oracle.L2NORM_K | (oracle.SCALAR_GATE if gate == "scalar" else 0)
    g = torch.Generator().manual_seed(85)
    d_o = torch.randn(inp["v"].shape, generator=g).to(torch.bfloat16)
    d_fS = torch.randn(inp["init_S"].shape, generator=g) * 0.1
    gl = None if inp["gate_logits"] is None else inp["gate_logits"].to(dev)
    t = {n: inp[n].to(dev) for n in ("q", "k", "v", "init_S")}
    got = la.la_backward_delta(t["q"], t["k"], t["v"], None, gl, d_o.to(dev),
                               inp["cu_seqlens"].to(dev), d_final_S=d_fS.to(dev), flags=f,
                               init_S=t["init_S"], cu_seqlens_host=inp["cu_seqlens"])
    assert la.la_check_device() == la.LA_OK
    ref = oracle.delta_backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), None,
                                None if inp["gate_logits"] is None else f64(inp["gate_logits"]),
                                inp["cu_seqlens"].numpy(), f64(d_o), f64(d_fS), flags=of,
                                init_S=f64(inp["init_S"]))
    names = ("dq", "dk", "dv", "d_init_S") + (("d_gate_logits",) if gate != "none" else ())
    for n in names:
        assert rel_err(got[n].cpu().numpy(), ref[n]) <= TOL[torch.bfloat16], n
    assert float(got["d_beta_logits"].abs().max()) == 0.0
