"""GPU parity of the decode step over a state pool addressed by a slot map
(la_decode_step_slots): each sequence's state is one slot of the pool, a
negative slot marks a padding sequence, an out-of-range slot is reported by
la_check_device.  The expected values are the oracle's decode on the states
gathered from the pool; gathering and scattering are plain indexing."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _helpers import TOL, f64, rel_err

pytestmark = pytest.mark.gpu


def _pool(n_slots, H, dk, dv, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((n_slots, H, dk, dv), generator=g) * 0.02


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128)])
@pytest.mark.parametrize("gate", ["none", "channel", "scalar"])
def test_decode_slots_match_oracle(cuda_lib, dtype, dk, dv, gate):
    la = cuda_lib
    dev = torch.device("cuda")
    steps, N, H, P = 3, 5, 3, 9
    idx = np.array([7, -1, 0, 4, 8], dtype=np.int32)   # one padding sequence
    inp = wl.decode_inputs(N, H, dk, dv, steps, dtype, seed=50 + dk + dv, gated=gate != "none",
                           scalar_gate=gate == "scalar")
    flags = la.LA_L2NORM_K | (la.LA_GATE_SCALAR if gate == "scalar" else 0)
    oflags = oracle.L2NORM_K | (oracle.SCALAR_GATE if gate == "scalar" else 0)
    pool0 = _pool(P, H, dk, dv, seed=dk + dv)
    pool = pool0.clone().to(dev)
    sidx = torch.from_numpy(idx).to(dev)
    live = idx >= 0
    ref_st = f64(pool0)[idx[live]]
    for t in range(steps):
        tok = {n: (None if inp[n] is None else inp[n][t]) for n in
               ("q", "k", "v", "beta_logits", "gate_logits")}
        o = torch.full(tok["v"].shape, float("nan"), dtype=dtype, device=dev)
        d = {n: (None if x is None else x.to(dev)) for n, x in tok.items()}
        la.la_decode_step_slots(d["q"], d["k"], d["v"], d["beta_logits"], d["gate_logits"], o,
                                pool, sidx, flags=flags)
        assert la.la_check_device() == la.LA_OK
        sel = {n: (None if x is None else f64(x)[live]) for n, x in tok.items()}
        ref_o, ref_st = oracle.decode(sel["q"], sel["k"], sel["v"], sel["beta_logits"],
                                      sel["gate_logits"], ref_st, flags=oflags)
        got = o.float().cpu()
        assert rel_err(got[live].numpy(), ref_o) <= TOL[dtype]
        assert torch.isnan(got[~live]).all(), "padding sequence's output was written"
    got_pool = pool.cpu()
    assert rel_err(got_pool[idx[live]].numpy(), ref_st) <= TOL[dtype]
    unused = sorted(set(range(P)) - set(idx[live].tolist()))
    assert torch.equal(got_pool[unused], pool0[unused]), "a slot outside the map changed"


def test_decode_slots_identity_map_equals_plain_decode(cuda_lib):
    """The identity slot map over a pool of N states is la_decode_step, bit
    for bit."""
    la = cuda_lib
    dev = torch.device("cuda")
    inp = wl.decode_inputs(6, 4, 128, 128, 1, torch.bfloat16, seed=61)
    tok = {n: inp[n][0].to(dev) for n in ("q", "k", "v", "beta_logits", "gate_logits")}
    a, b = inp["state"].clone().to(dev), inp["state"].clone().to(dev)
    oa = torch.empty_like(tok["v"])
    ob = torch.empty_like(tok["v"])
    la.la_decode_step(tok["q"], tok["k"], tok["v"], tok["beta_logits"], tok["gate_logits"], oa, a)
    la.la_decode_step_slots(tok["q"], tok["k"], tok["v"], tok["beta_logits"],
                            tok["gate_logits"], ob, b,
                            torch.arange(6, dtype=torch.int32, device=dev))
    assert la.la_check_device() == la.LA_OK
    assert torch.equal(oa, ob) and torch.equal(a, b)


def test_decode_slots_out_of_range_is_reported(cuda_lib):
    """A slot >= n_slots touches nothing for its sequence and is reported as
    LA_ERR_INVALID_ARG by la_check_device; the other sequences still step."""
    la = cuda_lib
    dev = torch.device("cuda")
    N, H, d, P = 3, 2, 64, 4
    inp = wl.decode_inputs(N, H, d, d, 1, torch.float32, seed=62)
    tok = {n: inp[n][0].to(dev) for n in ("q", "k", "v", "beta_logits", "gate_logits")}
    pool0 = _pool(P, H, d, d, seed=3)
    pool = pool0.clone().to(dev)
    o = torch.full(tok["v"].shape, float("nan"), device=dev)
    sidx = torch.tensor([2, P, 0], dtype=torch.int32, device=dev)
    la.la_decode_step_slots(tok["q"], tok["k"], tok["v"], tok["beta_logits"], tok["gate_logits"],
                            o, pool, sidx)
    assert la.la_check_device() == la.LA_ERR_INVALID_ARG
    assert la.la_check_device() == la.LA_OK          # the error word was cleared
    got = pool.cpu()
    assert torch.equal(got[[1, 3]], pool0[[1, 3]])
    assert torch.isnan(o[1].cpu()).all()
    ref_o, ref_st = oracle.decode(f64(inp["q"][0])[[0, 2]], f64(inp["k"][0])[[0, 2]],
                                  f64(inp["v"][0])[[0, 2]], f64(inp["beta_logits"][0])[[0, 2]],
                                  f64(inp["gate_logits"][0])[[0, 2]], f64(pool0)[[2, 0]])
    assert rel_err(o.cpu()[[0, 2]].numpy(), ref_o) <= 1e-4
    assert rel_err(got[[2, 0]].numpy(), ref_st) <= 1e-4
