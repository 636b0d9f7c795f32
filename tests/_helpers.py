"""Shared helpers for the GPU parity tests: run the CUDA path through the
C ABI binding and the oracle on the same seeded inputs, then compare with
max|GPU - oracle| / max|oracle| (the acceptance metric)."""
import numpy as np
import torch

import oracle

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), "non-finite values in GPU output"
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


def f64(t):
    return None if t is None else t.detach().to("cpu").double().numpy()


def gpu_prefill_delta(la, inp, flags=None, scale=1.0, final=True, init=True, chunk=64):
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    bl = None if inp["beta_logits"] is None else inp["beta_logits"].to(dev)
    gl = None if inp["gate_logits"] is None else inp["gate_logits"].to(dev)
    cu = inp["cu_seqlens"].to(dev)
    N, H, dk, dv = cu.numel() - 1, q.shape[1], q.shape[2], v.shape[2]
    o = torch.full((q.shape[0], H, dv), float("nan"), dtype=q.dtype, device=dev)
    iS = inp["init_S"].to(dev) if (init and inp.get("init_S") is not None) else None
    fS = torch.full((N, H, dk, dv), float("nan"), device=dev) if final else None
    la.la_prefill_delta(q, k, v, bl, gl, o, cu, chunk=chunk, scale=scale,
                        flags=la.LA_L2NORM_K if flags is None else flags, init_S=iS, final_S=fS,
                        cu_seqlens_host=inp["cu_seqlens"])
    assert la.la_check_device() == la.LA_OK
    return o.float().cpu(), (fS.cpu() if final else None)


def oracle_prefill_delta(inp, heads=None, flags=oracle.L2NORM_K, scale=1.0, init=True):
    sel = (lambda t: t) if heads is None else (lambda t: t[:, heads])
    q, k, v = (sel(inp[n]) for n in ("q", "k", "v"))
    bl = None if inp["beta_logits"] is None else sel(inp["beta_logits"])
    gl = None if inp["gate_logits"] is None else sel(inp["gate_logits"])
    iS = inp.get("init_S") if init else None
    if iS is not None and heads is not None:
        iS = iS[:, heads]
    return oracle.delta(f64(q), f64(k), f64(v), f64(bl), f64(gl), inp["cu_seqlens"].numpy(),
                        scale=scale, flags=flags, init_S=f64(iS))
