"""GPU checks of the training pair la_prefill_delta_train / la_backward_delta_saved:
the forward's outputs are la_prefill_delta's bit for bit (the same kernels,
which then also keep their records, T and chunk-start states), and the
gradients taken from those saved tensors match the oracle's reverse-mode
gradients (oracle.delta_backward, pinned by finite differences) within the
bf16 bar, on a second call from the same saved tensors too."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _helpers import TOL, f64, rel_err
from test_backward_gpu import RAGGED, _compare, _grad_inputs, _oracle

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "beta_logits", "gate_logits", "init_S")


def _forward_pair(la, inp, flags, scale):
    """(o, final_S) from la_prefill_delta, then from la_prefill_delta_train,
    and the saved buffer the latter filled."""
    dev = torch.device("cuda")
    t = {n: (None if inp[n] is None else inp[n].to(dev)) for n in NAMES}
    cu = inp["cu_seqlens"].to(dev)
    ntok, H, d = t["q"].shape
    N = cu.numel() - 1
    outs = []
    for train in (False, True):
        o = torch.full_like(t["v"], 7.0)
        fS = torch.full((N, H, d, d), 7.0, device=dev)
        if train:
            saved = torch.empty(la.la_backward_delta_workspace_size(N, ntok, H, d, d),
                                dtype=torch.uint8, device=dev)
            la.la_prefill_delta_train(t["q"], t["k"], t["v"], t["beta_logits"], t["gate_logits"], o,
                                      cu, saved, scale=scale, flags=flags, init_S=t["init_S"],
                                      final_S=fS, cu_seqlens_host=inp["cu_seqlens"])
        else:
            la.la_prefill_delta(t["q"], t["k"], t["v"], t["beta_logits"], t["gate_logits"], o, cu,
                                scale=scale, flags=flags, init_S=t["init_S"], final_S=fS,
                                cu_seqlens_host=inp["cu_seqlens"])
        assert la.la_check_device() == la.LA_OK
        outs.append((o, fS))
    return outs, saved, t, cu


def _saved_grads(la, inp, t, cu, saved, d_o, d_fS, flags, scale):
    dev = torch.device("cuda")
    g = la.la_backward_delta_saved(t["q"], t["k"], t["v"], t["beta_logits"], t["gate_logits"],
                                   d_o.to(dev), cu, saved, d_final_S=d_fS.to(dev), scale=scale,
                                   flags=flags, init_S=t["init_S"],
                                   cu_seqlens_host=inp["cu_seqlens"])
    assert la.la_check_device() == la.LA_OK
    return {n: (None if v is None else v.cpu().numpy()) for n, v in g.items()}


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("gate", ["none", "channel", "scalar"])
def test_train_pair_matches_prefill_and_oracle(cuda_lib, d, gate):
    """Ragged lengths (an empty and a one-token sequence, partial chunks),
    initial states and a final-state gradient."""
    la = cuda_lib
    inp = wl.prefill_inputs(RAGGED, 2, d, d, torch.bfloat16, gate != "none", seed=90 + d,
                            init_state=True, scalar_gate=gate == "scalar")
    flags = la.LA_L2NORM_K | (la.LA_GATE_SCALAR if gate == "scalar" else 0)
    oflags = oracle.L2NORM_K | (oracle.SCALAR_GATE if gate == "scalar" else 0)
    ((o_ref, fs_ref), (o, fs)), saved, t, cu = _forward_pair(la, inp, flags, 1.0)
    assert torch.equal(o, o_ref)
    assert torch.equal(fs, fs_ref)
    d_o, d_fS = _grad_inputs(inp, torch.bfloat16, seed=91)
    ref = _oracle(inp, d_o, d_fS, oflags)
    got = _saved_grads(la, inp, t, cu, saved, d_o, d_fS, flags, 1.0)
    _compare(got, ref, TOL[torch.bfloat16])
    # the saved tensors are not consumed: the same gradients again (up to the
    # order of the per-chunk kernel's shared-memory sums)
    again = _saved_grads(la, inp, t, cu, saved, d_o, d_fS, flags, 1.0)
    for n, v in got.items():
        if v is not None:
            assert rel_err(again[n], v) <= 1e-5, n


def test_train_pair_flags_and_scale(cuda_lib):
    """silu and L2 norm on q and k, a scale and a per-channel gate at d = 64."""
    la = cuda_lib
    inp = wl.prefill_inputs([150, 64, 9], 3, 64, 64, torch.bfloat16, True, seed=92,
                            init_state=True)
    flags = la.LA_L2NORM_K | la.LA_L2NORM_Q | la.LA_SILU_QK
    oflags = oracle.L2NORM_K | oracle.L2NORM_Q | oracle.SILU_QK
    ((o_ref, fs_ref), (o, fs)), saved, t, cu = _forward_pair(la, inp, flags, 0.6)
    assert torch.equal(o, o_ref)
    assert torch.equal(fs, fs_ref)
    d_o, d_fS = _grad_inputs(inp, torch.bfloat16, seed=93)
    got = _saved_grads(la, inp, t, cu, saved, d_o, d_fS, flags, 0.6)
    _compare(got, _oracle(inp, d_o, d_fS, oflags, scale=0.6), TOL[torch.bfloat16])


def test_train_pair_additive_rule(cuda_lib):
    """The additive (Mamba-2) rule through the pair: no beta (u = v), and a
    zero beta-logit gradient."""
    la = cuda_lib
    inp = wl.prefill_inputs(RAGGED, 2, 64, 64, torch.bfloat16, True, seed=94, init_state=True,
                            scalar_gate=True)
    inp["beta_logits"] = None          # ignored by the additive rule
    flags = la.LA_GATE_SCALAR | la.LA_ADDITIVE | la.LA_L2NORM_K
    oflags = oracle.SCALAR_GATE | oracle.ADDITIVE | oracle.L2NORM_K
    ((o_ref, fs_ref), (o, fs)), saved, t, cu = _forward_pair(la, inp, flags, 1.0)
    assert torch.equal(o, o_ref)
    assert torch.equal(fs, fs_ref)
    d_o, d_fS = _grad_inputs(inp, torch.bfloat16, seed=95)
    got = _saved_grads(la, inp, t, cu, saved, d_o, d_fS, flags, 1.0)
    ref = oracle.delta_backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), None,
                                f64(inp["gate_logits"]), inp["cu_seqlens"].numpy(), f64(d_o),
                                f64(d_fS), flags=oflags, init_S=f64(inp["init_S"]))
    for n in ("dq", "dk", "dv", "d_gate_logits", "d_init_S"):
        assert rel_err(got[n], ref[n]) <= TOL[torch.bfloat16], n
    assert np.all(got["d_beta_logits"] == 0.0)


def test_train_forward_refuses_fp32(cuda_lib):
    """fp32 I/O has no chunkwise backward: la_prefill_delta_train says so."""
    la = cuda_lib
    inp = wl.prefill_inputs([70], 1, 64, 64, torch.float32, False, seed=96)
    dev = torch.device("cuda")
    t = {n: (None if inp[n] is None else inp[n].to(dev)) for n in NAMES}
    saved = torch.empty(la.la_backward_delta_workspace_size(1, 70, 1, 64, 64), dtype=torch.uint8,
                        device=dev)
    with pytest.raises(la.LinAttnError) as e:
        la.la_prefill_delta_train(t["q"], t["k"], t["v"], t["beta_logits"], None,
                                  torch.empty_like(t["v"]), inp["cu_seqlens"].to(dev), saved)
    assert e.value.status == la.LA_ERR_UNSUPPORTED


def test_delta_rule_autograd(cuda_lib):
    """delta_rule as a torch.autograd.Function: a loss over o and final_S
    back-propagates to every input the same gradients la_backward_delta
    returns for that loss's output gradients (cast to each input's dtype)."""
    la = cuda_lib
    dev = torch.device("cuda")
    inp = wl.prefill_inputs([150, 64, 9], 2, 64, 64, torch.bfloat16, True, seed=97,
                            init_state=True)
    leaves = {n: inp[n].to(dev).requires_grad_(True) for n in NAMES}
    cu = inp["cu_seqlens"].to(dev)
    o, fS = la.delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["beta_logits"],
                          leaves["gate_logits"], cu, init_S=leaves["init_S"],
                          cu_seqlens_host=inp["cu_seqlens"])
    d_o, d_fS = _grad_inputs(inp, torch.bfloat16, seed=98)
    loss = (o.float() * d_o.to(dev).float()).sum() + (fS * d_fS.to(dev)).sum()
    loss.backward()
    assert la.la_check_device() == la.LA_OK
    t = {n: inp[n].to(dev) for n in NAMES}
    ref = la.la_backward_delta(t["q"], t["k"], t["v"], t["beta_logits"], t["gate_logits"],
                               d_o.to(dev), cu, d_final_S=d_fS.to(dev), init_S=t["init_S"],
                               cu_seqlens_host=inp["cu_seqlens"])
    pairs = (("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta_logits", "d_beta_logits"),
             ("gate_logits", "d_gate_logits"), ("init_S", "d_init_S"))
    for leaf, name in pairs:
        g = leaves[leaf].grad
        assert g is not None and g.dtype == leaves[leaf].dtype, leaf
        # bf16 inputs get the fp32 gradient rounded to bf16 (relative 2^-9)
        bar = 1e-5 if g.dtype == torch.float32 else 4e-3
        assert rel_err(g.float().cpu().numpy(), ref[name].cpu().numpy()) <= bar, leaf


def test_delta_rule_autograd_optional_inputs(cuda_lib):
    """delta_rule's optional pieces: the additive rule with no beta, a
    scalar gate at d = 128, no initial state, and a loss on o alone (so no
    final-state gradient reaches the backward)."""
    la = cuda_lib
    dev = torch.device("cuda")
    inp = wl.prefill_inputs([130, 7, 64], 2, 128, 128, torch.bfloat16, True, seed=99,
                            scalar_gate=True)
    names = ("q", "k", "v", "gate_logits")
    leaves = {n: inp[n].to(dev).requires_grad_(True) for n in names}
    cu = inp["cu_seqlens"].to(dev)
    flags = la.LA_ADDITIVE | la.LA_GATE_SCALAR | la.LA_L2NORM_K
    o, fS = la.delta_rule(leaves["q"], leaves["k"], leaves["v"], None, leaves["gate_logits"], cu,
                          flags=flags, cu_seqlens_host=inp["cu_seqlens"])
    g = torch.Generator().manual_seed(100)
    d_o = torch.randn(inp["v"].shape, generator=g).to(torch.bfloat16)
    (o.float() * d_o.to(dev).float()).sum().backward()
    assert la.la_check_device() == la.LA_OK
    t = {n: inp[n].to(dev) for n in names}
    ref = la.la_backward_delta(t["q"], t["k"], t["v"], None, t["gate_logits"], d_o.to(dev), cu,
                               flags=flags, cu_seqlens_host=inp["cu_seqlens"])
    for leaf, name in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("gate_logits", "d_gate_logits")):
        got = leaves[leaf].grad
        assert got is not None and got.dtype == torch.bfloat16, leaf
        assert rel_err(got.float().cpu().numpy(), ref[name].cpu().numpy()) <= 4e-3, leaf
