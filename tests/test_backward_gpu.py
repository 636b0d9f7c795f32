"""GPU parity of la_backward_delta against the oracle's reverse-mode
gradients (oracle.delta_backward, pinned by finite differences) on the same
seeded inputs, element by element, for every gradient the call returns."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _helpers import TOL, f64, rel_err

pytestmark = pytest.mark.gpu

RAGGED = [200, 77, 1, 0, 128, 65]
NAMES = ("dq", "dk", "dv", "d_beta_logits", "d_gate_logits", "d_init_S")


def _grad_inputs(inp, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    ntok, H, dv = inp["v"].shape
    N, _, dk, _ = inp["init_S"].shape
    d_o = torch.randn((ntok, H, dv), generator=g).to(dtype)
    d_fS = torch.randn((N, H, dk, dv), generator=g) * 0.1
    return d_o, d_fS


def _run(la, inp, d_o, d_fS, flags, scale=1.0):
    dev = torch.device("cuda")
    t = {n: (None if inp[n] is None else inp[n].to(dev))
         for n in ("q", "k", "v", "beta_logits", "gate_logits", "init_S")}
    out = la.la_backward_delta(t["q"], t["k"], t["v"], t["beta_logits"], t["gate_logits"],
                               d_o.to(dev), inp["cu_seqlens"].to(dev), d_final_S=d_fS.to(dev),
                               scale=scale, flags=flags, init_S=t["init_S"],
                               cu_seqlens_host=inp["cu_seqlens"])
    assert la.la_check_device() == la.LA_OK
    return {n: (None if v is None else v.cpu().numpy()) for n, v in out.items()}


def _oracle(inp, d_o, d_fS, flags, scale=1.0, heads=None):
    sel = (lambda x: x) if heads is None else (lambda x: x[:, heads])
    g = oracle.delta_backward(f64(sel(inp["q"])), f64(sel(inp["k"])), f64(sel(inp["v"])),
                              f64(sel(inp["beta_logits"])),
                              None if inp["gate_logits"] is None else f64(sel(inp["gate_logits"])),
                              inp["cu_seqlens"].numpy(), f64(sel(d_o)), f64(sel(d_fS)),
                              scale=scale, flags=flags,
                              init_S=None if inp["init_S"] is None else f64(sel(inp["init_S"])))
    return {"dq": g["dq"], "dk": g["dk"], "dv": g["dv"], "d_beta_logits": g["d_beta_logits"],
            "d_gate_logits": g["d_gate_logits"], "d_init_S": g["d_init_S"]}


def _compare(got, ref, tol, rows=None):
    errs = {}
    for n in NAMES:
        if ref[n] is None:
            assert got[n] is None
            continue
        g = got[n] if rows is None or n == "d_init_S" else got[n][rows]
        r = ref[n] if rows is None or n == "d_init_S" else ref[n][rows]
        errs[n] = rel_err(g, r)
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, (bad, errs)
    return errs


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("gate", ["none", "channel", "scalar"])
def test_backward_ragged_matches_oracle(cuda_lib, dtype, dk, dv, gate):
    """Ragged lengths (an empty and a one-token sequence, partial chunks),
    initial states and a final-state gradient."""
    la = cuda_lib
    inp = wl.prefill_inputs(RAGGED, 2, dk, dv, dtype, gate != "none", seed=70 + dk + dv,
                            init_state=True, scalar_gate=gate == "scalar")
    d_o, d_fS = _grad_inputs(inp, dtype, seed=71)
    flags = la.LA_L2NORM_K | (la.LA_GATE_SCALAR if gate == "scalar" else 0)
    oflags = oracle.L2NORM_K | (oracle.SCALAR_GATE if gate == "scalar" else 0)
    got = _run(la, inp, d_o, d_fS, flags)
    ref = _oracle(inp, d_o, d_fS, oflags)
    _compare(got, ref, TOL[dtype])


def test_backward_flags_and_scale(cuda_lib):
    """silu and L2 norm on q and k, a scale, per-channel gate, fp32."""
    la = cuda_lib
    inp = wl.prefill_inputs([150, 64], 3, 64, 64, torch.float32, True, seed=72, init_state=True)
    d_o, d_fS = _grad_inputs(inp, torch.float32, seed=73)
    flags = la.LA_L2NORM_K | la.LA_L2NORM_Q | la.LA_SILU_QK
    oflags = oracle.L2NORM_K | oracle.L2NORM_Q | oracle.SILU_QK
    got = _run(la, inp, d_o, d_fS, flags, scale=0.6)
    ref = _oracle(inp, d_o, d_fS, oflags, scale=0.6)
    _compare(got, ref, 1e-4)


def test_backward_gpt2_shape_sampled_heads(cuda_lib):
    """The GPT-2-shaped prefill (8 x 2048 tokens, 12 heads, d = 64, bf16): the
    whole backward on the GPU, the oracle on two heads of every sequence."""
    la = cuda_lib
    w = wl.workload("gpt2_prefill")
    inp = wl.inputs_for(w, seed=0, init_state=True)
    d_o, d_fS = _grad_inputs(inp, w.dtype, seed=74)
    got = _run(la, inp, d_o, d_fS, la.LA_L2NORM_K)
    heads = [3, 10]
    ref = _oracle(inp, d_o, d_fS, oracle.L2NORM_K, heads=heads)
    sub = {n: (None if v is None else v[:, heads]) for n, v in got.items()}
    _compare(sub, ref, TOL[w.dtype])


def test_backward_gated_shape_sampled_heads(cuda_lib):
    """The gated prefill shape (4 x 8192 tokens, 32 heads, d = 128, a decay per
    key channel, bf16): the whole backward on the GPU (chunkwise, per-channel
    decay kernel), the oracle on two heads of every sequence."""
    la = cuda_lib
    w = wl.workload("gated_prefill")
    inp = wl.inputs_for(w, seed=0, init_state=True)
    d_o, d_fS = _grad_inputs(inp, w.dtype, seed=75)
    got = _run(la, inp, d_o, d_fS, la.LA_L2NORM_K)
    heads = [5, 30]
    ref = _oracle(inp, d_o, d_fS, oracle.L2NORM_K, heads=heads)
    sub = {n: (None if v is None else v[:, heads]) for n, v in got.items()}
    _compare(sub, ref, TOL[w.dtype])


@pytest.mark.parametrize("d", [64, 128])
def test_backward_strong_channel_decay(cuda_lib, d):
    """Gate logits around 8 (alpha ~ e^-8 per token and channel): the decay
    across a 16-token block underflows fp32, so only the exact in-block terms
    and products of factors <= 1 may carry it."""
    la = cuda_lib
    inp = wl.prefill_inputs([190, 64, 33], 2, d, d, torch.bfloat16, True, seed=76,
                            init_state=True, gate_mean=8.0)
    d_o, d_fS = _grad_inputs(inp, torch.bfloat16, seed=77)
    got = _run(la, inp, d_o, d_fS, la.LA_L2NORM_K)
    ref = _oracle(inp, d_o, d_fS, oracle.L2NORM_K)
    _compare(got, ref, TOL[torch.bfloat16])


def test_backward_channel_flags_and_scale_d128(cuda_lib):
    """silu and L2 norm on q and k, a scale, per-channel gate, bf16, d = 128."""
    la = cuda_lib
    inp = wl.prefill_inputs([150, 64, 1], 3, 128, 128, torch.bfloat16, True, seed=78,
                            init_state=True)
    d_o, d_fS = _grad_inputs(inp, torch.bfloat16, seed=79)
    flags = la.LA_L2NORM_K | la.LA_L2NORM_Q | la.LA_SILU_QK
    oflags = oracle.L2NORM_K | oracle.L2NORM_Q | oracle.SILU_QK
    got = _run(la, inp, d_o, d_fS, flags, scale=0.6)
    ref = _oracle(inp, d_o, d_fS, oflags, scale=0.6)
    _compare(got, ref, TOL[torch.bfloat16])


def test_backward_varlen_shape_sampled_heads(cuda_lib):
    """The varlen prefill shape (65 536 packed tokens of seeded lengths, 16
    heads, d = 128, a decay per key channel, bf16; ragged last chunks): the
    whole backward on the GPU, the oracle on one head of every sequence."""
    la = cuda_lib
    w = wl.workload("varlen_prefill")
    inp = wl.inputs_for(w, seed=0, init_state=True)
    d_o, d_fS = _grad_inputs(inp, w.dtype, seed=80)
    got = _run(la, inp, d_o, d_fS, la.LA_L2NORM_K)
    heads = [11]
    ref = _oracle(inp, d_o, d_fS, oracle.L2NORM_K, heads=heads)
    sub = {n: (None if v is None else v[:, heads]) for n, v in got.items()}
    _compare(sub, ref, TOL[w.dtype])


@pytest.mark.parametrize("d", [64, 128])
def test_backward_many_short_sequences(cuda_lib, d):
    """130 sequences of 1..100 tokens (most shorter than a chunk, some
    spanning two, some empty), scalar gate at d = 64 and per-channel at 128:
    every chunk slot and tail of the chunkwise backward."""
    la = cuda_lib
    g = torch.Generator().manual_seed(86)
    lens = torch.randint(0, 101, (130,), generator=g).tolist()
    scalar = d == 64
    inp = wl.prefill_inputs(lens, 2, d, d, torch.bfloat16, True, seed=87, init_state=True,
                            scalar_gate=scalar)
    d_o, d_fS = _grad_inputs(inp, torch.bfloat16, seed=88)
    flags = la.LA_L2NORM_K | (la.LA_GATE_SCALAR if scalar else 0)
    oflags = oracle.L2NORM_K | (oracle.SCALAR_GATE if scalar else 0)
    got = _run(la, inp, d_o, d_fS, flags)
    ref = _oracle(inp, d_o, d_fS, oflags)
    _compare(got, ref, TOL[torch.bfloat16])


def test_backward_unaligned_tensor_takes_token_serial(cuda_lib):
    """A tensor that is not 16-byte aligned (here d_final_S, one float into a
    larger buffer) sends a bf16 call that the chunkwise form would take to
    the token-serial kernels instead; the gradients still match the oracle."""
    la = cuda_lib
    dev = torch.device("cuda")
    inp = wl.prefill_inputs([130, 64], 2, 64, 64, torch.bfloat16, True, seed=75, init_state=True)
    d_o, d_fS = _grad_inputs(inp, torch.bfloat16, seed=76)
    buf = torch.zeros(d_fS.numel() + 1, device=dev)
    d_fS_odd = buf[1:].view(d_fS.shape)
    d_fS_odd.copy_(d_fS.to(dev))
    assert d_fS_odd.data_ptr() % 16 != 0
    t = {n: inp[n].to(dev) for n in ("q", "k", "v", "beta_logits", "gate_logits", "init_S")}
    out = la.la_backward_delta(t["q"], t["k"], t["v"], t["beta_logits"], t["gate_logits"],
                               d_o.to(dev), inp["cu_seqlens"].to(dev), d_final_S=d_fS_odd,
                               init_S=t["init_S"], cu_seqlens_host=inp["cu_seqlens"])
    assert la.la_check_device() == la.LA_OK
    got = {n: (None if v is None else v.cpu().numpy()) for n, v in out.items()}
    _compare(got, _oracle(inp, d_o, d_fS, oracle.L2NORM_K), TOL[torch.bfloat16])
