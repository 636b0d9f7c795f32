"""GB300 (sm_103a) causal linear / delta-rule attention: thin Python binding.

The product is the C-ABI library ``_lib/liblinattn.so`` declared in
``include/linattn.h``.  This module only marshals torch tensors (device
pointers, sizes, the current CUDA stream) into those calls; every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback: if
the library is not built, the first call raises.

Functions (same names as the C ABI):
  la_prefill_linear, la_prefill_delta, la_prefill_delta_workspace_size,
  la_prefill_delta_launches,
  la_prefill_delta_static, la_decode_step, la_decode_step_slots,
  la_backward_delta, la_prefill_delta_train, la_backward_delta_saved,
  la_check_device, la_selftest_wait_timeout, la_status_string;
and delta_rule, a torch.autograd.Function over the training pair.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB_PATH, build  # noqa: F401  (build needs no GPU)

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_TIMEOUT = 0, 1, 2, 3, 4
LA_ERR_TOO_LARGE = 5
LA_STATIC_SCRATCH_BYTES = 256 << 20
LA_F32, LA_BF16 = 0, 1
LA_L2NORM_K, LA_L2NORM_Q, LA_SILU_QK, LA_GATE_SCALAR, LA_ADDITIVE = 1, 2, 4, 8, 16

EXPORTED = ("la_prefill_linear", "la_prefill_delta", "la_prefill_delta_workspace_size",
            "la_prefill_delta_launches",
            "la_prefill_delta_static", "la_decode_step", "la_decode_step_slots",
            "la_backward_delta", "la_backward_delta_workspace_size",
            "la_prefill_delta_train", "la_backward_delta_saved", "la_check_device",
            "la_selftest_wait_timeout", "la_status_string")


class LinAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {la_status_string(status)}")


_lib = None


def library():
    """Load the in-tree CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library missing at {LIB_PATH}: build it with "
                               "delta_rule_recurrent_chunkwise_gb300.build()")
        lib = ctypes.CDLL(LIB_PATH)
        vp, ip, fp = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        u, sz = ctypes.c_uint, ctypes.c_size_t
        lib.la_prefill_linear.argtypes = [vp, vp, vp, vp, ip, vp, vp, ip, ip, ip, ip, ip,
                                          vp, vp, vp, vp, vp]
        lib.la_prefill_delta.argtypes = [vp, vp, vp, vp, vp, vp, ip, vp, vp, ip, ip, ip, ip, ip,
                                         ip, fp, u, vp, vp, vp, sz, vp]
        lib.la_prefill_delta_static.argtypes = [vp, vp, vp, vp, vp, vp, ip, vp, vp, ip, ip, ip,
                                                ip, ip, ip, fp, u, vp, vp, vp]
        lib.la_prefill_delta_workspace_size.argtypes = [ip, ip, ip, ip, ip, ip, ip]
        lib.la_prefill_delta_workspace_size.restype = sz
        lib.la_prefill_delta_launches.argtypes = [ip, ip, ip, ip, ip, ip, ip, u, ip]
        lib.la_prefill_delta_launches.restype = ip
        lib.la_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, ip, ip, ip, ip, ip, fp, u, vp, vp]
        lib.la_decode_step_slots.argtypes = [vp, vp, vp, vp, vp, vp, ip, ip, ip, ip, ip, fp, u,
                                             vp, ip, vp, vp]
        lib.la_backward_delta.argtypes = [vp, vp, vp, vp, vp, vp, vp, ip, vp, vp, ip, ip, ip, ip,
                                          ip, fp, u, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.la_prefill_delta_train.argtypes = [vp, vp, vp, vp, vp, vp, ip, vp, vp, ip, ip, ip,
                                               ip, ip, fp, u, vp, vp, vp, sz, vp]
        lib.la_backward_delta_saved.argtypes = lib.la_backward_delta.argtypes
        lib.la_backward_delta_workspace_size.argtypes = [ip, ip, ip, ip, ip]
        lib.la_backward_delta_workspace_size.restype = sz
        lib.la_check_device.argtypes = [vp]
        lib.la_selftest_wait_timeout.argtypes = [vp]
        lib.la_status_string.argtypes = [ip]
        lib.la_status_string.restype = ctypes.c_char_p
        for f in ("la_prefill_linear", "la_prefill_delta", "la_prefill_delta_static",
                  "la_decode_step", "la_decode_step_slots", "la_backward_delta",
                  "la_prefill_delta_train", "la_backward_delta_saved",
                  "la_check_device", "la_selftest_wait_timeout"):
            getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def la_status_string(status: int) -> str:
    return library().la_status_string(int(status)).decode()


# ---------------------------------------------------------------- marshalling

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _io(t):
    import torch
    if t.dtype == torch.float32:
        return LA_F32
    if t.dtype == torch.bfloat16:
        return LA_BF16
    raise TypeError(f"unsupported I/O dtype {t.dtype} (float32 or bfloat16)")


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(tensors, dtype=None, device=None):
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
        if device is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, expected {device}")


def _host_cu(cu_seqlens_host):
    if cu_seqlens_host is None:
        return None, None
    import torch
    h = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
    return h, ctypes.c_void_p(h.data_ptr())


def la_prefill_linear(q, k, v, o, cu_seqlens, init_S=None, init_z=None, final_S=None,
                      final_z=None, cu_seqlens_host=None, stream=None):
    """ELU+1 linear attention prefill.  q,k [ntok,H,dk]; v,o [ntok,H,dv]."""
    import torch
    _check(dict(q=q, k=k, v=v, o=o), dtype=q.dtype, device=q.device)
    _check(dict(cu_seqlens=cu_seqlens), dtype=torch.int32, device=q.device)
    _check(dict(init_S=init_S, init_z=init_z, final_S=final_S, final_z=final_z),
           dtype=torch.float32, device=q.device)
    ntok, H, dk = q.shape
    dv = v.shape[2]
    N = cu_seqlens.numel() - 1
    hold, hptr = _host_cu(cu_seqlens_host)
    rc = library().la_prefill_linear(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _io(q), _ptr(cu_seqlens),
                                     hptr, N, ntok, H, dk, dv, _ptr(init_S), _ptr(init_z),
                                     _ptr(final_S), _ptr(final_z), _stream(stream))
    if rc != LA_OK:
        raise LinAttnError(rc, "la_prefill_linear")
    return o


def la_prefill_delta_workspace_size(N, ntok, H, dk, dv, chunk=64, io=LA_BF16) -> int:
    return int(library().la_prefill_delta_workspace_size(N, ntok, H, dk, dv, chunk, io))


def la_prefill_delta_launches(N, ntok, H, dk, dv, chunk=64, io=LA_BF16, flags=LA_L2NORM_K,
                              has_gate=False) -> int:
    """Kernels one la_prefill_delta call with these sizes launches on the
    current device (0: the call would be rejected)."""
    return int(library().la_prefill_delta_launches(N, ntok, H, dk, dv, chunk, io, flags,
                                                   1 if has_gate else 0))


def la_prefill_delta(q, k, v, beta_logits, gate_logits, o, cu_seqlens, chunk=64, scale=1.0,
                     flags=LA_L2NORM_K, init_S=None, final_S=None, workspace=None,
                     cu_seqlens_host=None, stream=None):
    """(Gated) delta-rule prefill.  q,k [ntok,H,dk]; v,o [ntok,H,dv];
    beta_logits [ntok,H]; gate_logits [ntok,H,dk] or None.  chunk: tokens
    per chunk of the state recurrence, 64, or 128 for bf16 with dk = dv = 64.
    workspace: a device buffer of at least la_prefill_delta_workspace_size(...)
    bytes; allocated here (on q's device) when not given."""
    import torch
    _check(dict(q=q, k=k, v=v, o=o, beta_logits=beta_logits, gate_logits=gate_logits),
           dtype=q.dtype, device=q.device)
    _check(dict(cu_seqlens=cu_seqlens), dtype=torch.int32, device=q.device)
    _check(dict(init_S=init_S, final_S=final_S), dtype=torch.float32, device=q.device)
    ntok, H, dk = q.shape
    dv = v.shape[2]
    N = cu_seqlens.numel() - 1
    hold, hptr = _host_cu(cu_seqlens_host)
    if workspace is None:
        need = la_prefill_delta_workspace_size(N, ntok, H, dk, dv, chunk, _io(q))
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = library().la_prefill_delta(_ptr(q), _ptr(k), _ptr(v), _ptr(beta_logits),
                                    _ptr(gate_logits), _ptr(o), _io(q), _ptr(cu_seqlens), hptr,
                                    N, ntok, H, dk, dv, int(chunk), float(scale), int(flags),
                                    _ptr(init_S), _ptr(final_S), _ptr(workspace), ws_bytes,
                                    _stream(stream))
    if rc != LA_OK:
        raise LinAttnError(rc, "la_prefill_delta")
    return o


def la_prefill_delta_static(q, k, v, beta_logits, gate_logits, o, cu_seqlens, chunk=64,
                            scale=1.0, flags=LA_L2NORM_K, init_S=None, final_S=None,
                            cu_seqlens_host=None, stream=None):
    """la_prefill_delta on the library's static scratch: allocates nothing.
    Calls on one device must not overlap in time (they share the scratch)."""
    import torch
    _check(dict(q=q, k=k, v=v, o=o, beta_logits=beta_logits, gate_logits=gate_logits),
           dtype=q.dtype, device=q.device)
    _check(dict(cu_seqlens=cu_seqlens), dtype=torch.int32, device=q.device)
    _check(dict(init_S=init_S, final_S=final_S), dtype=torch.float32, device=q.device)
    ntok, H, dk = q.shape
    dv = v.shape[2]
    N = cu_seqlens.numel() - 1
    hold, hptr = _host_cu(cu_seqlens_host)
    rc = library().la_prefill_delta_static(_ptr(q), _ptr(k), _ptr(v), _ptr(beta_logits),
                                           _ptr(gate_logits), _ptr(o), _io(q), _ptr(cu_seqlens),
                                           hptr, N, ntok, H, dk, dv, int(chunk), float(scale),
                                           int(flags), _ptr(init_S), _ptr(final_S),
                                           _stream(stream))
    if rc != LA_OK:
        raise LinAttnError(rc, "la_prefill_delta_static")
    return o


def la_backward_delta_workspace_size(N, ntok, H, dk, dv) -> int:
    return int(library().la_backward_delta_workspace_size(N, ntok, H, dk, dv))


def la_backward_delta(q, k, v, beta_logits, gate_logits, d_o, cu_seqlens, d_final_S=None,
                      scale=1.0, flags=LA_L2NORM_K, init_S=None, want_d_init_S=True,
                      workspace=None, cu_seqlens_host=None, stream=None):
    """Gradients of la_prefill_delta given d_o [ntok,H,dv] (q's dtype) and
    optionally d_final_S [N,H,dk,dv] fp32.  Returns a dict of fp32 tensors
    dq, dk, dv, d_beta_logits, d_gate_logits (None without gate), d_init_S
    (None unless want_d_init_S).  Rows of tokens outside every sequence are
    zero here (the library leaves them untouched; they are allocated zeroed
    unless cu_seqlens_host shows the sequences cover every row)."""
    return _backward("la_backward_delta", q, k, v, beta_logits, gate_logits, d_o, cu_seqlens,
                     d_final_S, scale, flags, init_S, want_d_init_S, workspace, cu_seqlens_host,
                     stream)


def la_prefill_delta_train(q, k, v, beta_logits, gate_logits, o, cu_seqlens, saved, scale=1.0,
                           flags=LA_L2NORM_K, init_S=None, final_S=None, cu_seqlens_host=None,
                           stream=None):
    """la_prefill_delta (chunk 64) that also keeps what the gradients need in
    `saved`, a device buffer of la_backward_delta_workspace_size(...) bytes,
    for la_backward_delta_saved.  bf16 with dk = dv in {64, 128} only."""
    import torch
    _check(dict(q=q, k=k, v=v, o=o, beta_logits=beta_logits, gate_logits=gate_logits),
           dtype=q.dtype, device=q.device)
    _check(dict(cu_seqlens=cu_seqlens), dtype=torch.int32, device=q.device)
    _check(dict(init_S=init_S, final_S=final_S), dtype=torch.float32, device=q.device)
    _check(dict(saved=saved), device=q.device)
    ntok, H, dk = q.shape
    dv = v.shape[2]
    N = cu_seqlens.numel() - 1
    hold, hptr = _host_cu(cu_seqlens_host)
    rc = library().la_prefill_delta_train(
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta_logits), _ptr(gate_logits), _ptr(o), _io(q),
        _ptr(cu_seqlens), hptr, N, ntok, H, dk, dv, float(scale), int(flags), _ptr(init_S),
        _ptr(final_S), _ptr(saved), saved.numel() * saved.element_size(), _stream(stream))
    if rc != LA_OK:
        raise LinAttnError(rc, "la_prefill_delta_train")
    return o


def la_backward_delta_saved(q, k, v, beta_logits, gate_logits, d_o, cu_seqlens, saved,
                            d_final_S=None, scale=1.0, flags=LA_L2NORM_K, init_S=None,
                            want_d_init_S=True, cu_seqlens_host=None, stream=None):
    """la_backward_delta from the tensors la_prefill_delta_train kept in
    `saved` (pass that call's inputs); the forward is not recomputed."""
    if saved is None:
        raise ValueError("saved: the buffer la_prefill_delta_train filled")
    return _backward("la_backward_delta_saved", q, k, v, beta_logits, gate_logits, d_o,
                     cu_seqlens, d_final_S, scale, flags, init_S, want_d_init_S, saved,
                     cu_seqlens_host, stream)


_DeltaRuleFn = None


def delta_rule(q, k, v, beta_logits, gate_logits, cu_seqlens, scale=1.0, flags=LA_L2NORM_K,
               init_S=None, cu_seqlens_host=None):
    """Differentiable delta-rule prefill for torch training: returns
    (o, final_S); the forward is la_prefill_delta_train, the backward
    la_backward_delta_saved from the buffer the forward filled (one buffer per
    call, held until the backward).  bf16 q, k, v, beta_logits, gate_logits
    (or None) with dk = dv in {64, 128}; init_S fp32 or None.  Gradients
    reach every tensor input that requires one, cast to its dtype."""
    global _DeltaRuleFn
    if _DeltaRuleFn is None:
        import torch

        class _Fn(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, beta_logits, gate_logits, init_S, cu_seqlens, scale, flags,
                        cu_host):
                ntok, H, dk = q.shape
                N = cu_seqlens.numel() - 1
                saved = torch.empty(la_backward_delta_workspace_size(N, ntok, H, dk, v.shape[2]),
                                    dtype=torch.uint8, device=q.device)
                o = torch.empty_like(v)
                final_S = torch.empty((N, H, dk, v.shape[2]), dtype=torch.float32,
                                      device=q.device)
                la_prefill_delta_train(q, k, v, beta_logits, gate_logits, o, cu_seqlens, saved,
                                       scale=scale, flags=flags, init_S=init_S, final_S=final_S,
                                       cu_seqlens_host=cu_host)
                ctx.save_for_backward(q, k, v, beta_logits, gate_logits, init_S, cu_seqlens,
                                      saved)
                ctx.scale, ctx.flags, ctx.cu_host = scale, flags, cu_host
                return o, final_S

            @staticmethod
            def backward(ctx, d_o, d_final_S):
                q, k, v, beta_logits, gate_logits, init_S, cu_seqlens, saved = ctx.saved_tensors
                if d_o is None:
                    d_o = torch.zeros_like(v)
                g = la_backward_delta_saved(
                    q, k, v, beta_logits, gate_logits, d_o.to(q.dtype).contiguous(), cu_seqlens,
                    saved, d_final_S=None if d_final_S is None else d_final_S.float().contiguous(),
                    scale=ctx.scale, flags=ctx.flags, init_S=init_S,
                    want_d_init_S=init_S is not None, cu_seqlens_host=ctx.cu_host)
                cast = lambda x, like: None if x is None or like is None else x.to(like.dtype)
                return (cast(g["dq"], q), cast(g["dk"], k), cast(g["dv"], v),
                        cast(g["d_beta_logits"], beta_logits),
                        cast(g["d_gate_logits"], gate_logits), cast(g["d_init_S"], init_S),
                        None, None, None, None)

        _DeltaRuleFn = _Fn
    return _DeltaRuleFn.apply(q, k, v, beta_logits, gate_logits, init_S, cu_seqlens, float(scale),
                              int(flags), cu_seqlens_host)


def _backward(fn, q, k, v, beta_logits, gate_logits, d_o, cu_seqlens, d_final_S, scale, flags,
              init_S, want_d_init_S, workspace, cu_seqlens_host, stream):
    import torch
    _check(dict(q=q, k=k, v=v, d_o=d_o, beta_logits=beta_logits, gate_logits=gate_logits),
           dtype=q.dtype, device=q.device)
    _check(dict(cu_seqlens=cu_seqlens), dtype=torch.int32, device=q.device)
    _check(dict(init_S=init_S, d_final_S=d_final_S), dtype=torch.float32, device=q.device)
    ntok, H, dk = q.shape
    dv = v.shape[2]
    N = cu_seqlens.numel() - 1
    hold, hptr = _host_cu(cu_seqlens_host)
    f32 = dict(dtype=torch.float32, device=q.device)
    covered = hold is not None and int(hold[0]) == 0 and int(hold[-1]) == ntok
    alloc = torch.empty if covered else torch.zeros
    out = {"dq": alloc((ntok, H, dk), **f32), "dk": alloc((ntok, H, dk), **f32),
           "dv": alloc((ntok, H, dv), **f32),
           "d_beta_logits": alloc((ntok, H), **f32),
           "d_gate_logits": None if gate_logits is None else alloc(gate_logits.shape, **f32),
           "d_init_S": torch.empty((N, H, dk, dv), **f32) if want_d_init_S else None}
    if workspace is None:
        workspace = torch.empty(la_backward_delta_workspace_size(N, ntok, H, dk, dv),
                                dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = getattr(library(), fn)(
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta_logits), _ptr(gate_logits), _ptr(d_o),
        _ptr(d_final_S), _io(q), _ptr(cu_seqlens), hptr, N, ntok, H, dk, dv, float(scale),
        int(flags), _ptr(init_S), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
        _ptr(out["d_beta_logits"]), _ptr(out["d_gate_logits"]), _ptr(out["d_init_S"]),
        _ptr(workspace), ws_bytes, _stream(stream))
    if rc != LA_OK:
        raise LinAttnError(rc, fn)
    return out


def la_decode_step(q, k, v, beta_logits, gate_logits, o, state, scale=1.0, flags=LA_L2NORM_K,
                   stream=None):
    """One decode step, state updated in place.  q,k [N,H,dk]; v,o [N,H,dv];
    beta_logits [N,H]; gate_logits [N,H,dk] or None; state [N,H,dk,dv] fp32."""
    import torch
    _check(dict(q=q, k=k, v=v, o=o, beta_logits=beta_logits, gate_logits=gate_logits),
           dtype=q.dtype, device=q.device)
    _check(dict(state=state), dtype=torch.float32, device=q.device)
    N, H, dk = q.shape
    dv = v.shape[2]
    rc = library().la_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(beta_logits), _ptr(gate_logits),
                                  _ptr(o), _io(q), N, H, dk, dv, float(scale), int(flags),
                                  _ptr(state), _stream(stream))
    if rc != LA_OK:
        raise LinAttnError(rc, "la_decode_step")
    return o


def la_decode_step_slots(q, k, v, beta_logits, gate_logits, o, state_pool, state_indices,
                         scale=1.0, flags=LA_L2NORM_K, stream=None):
    """One decode step over a state pool: sequence n updates
    state_pool[state_indices[n]] in place (a negative index skips sequence
    n).  q,k [N,H,dk]; v,o [N,H,dv]; beta_logits [N,H]; gate_logits
    [N,H,dk] or None; state_pool [P,H,dk,dv] fp32; state_indices [N] int32."""
    import torch
    _check(dict(q=q, k=k, v=v, o=o, beta_logits=beta_logits, gate_logits=gate_logits),
           dtype=q.dtype, device=q.device)
    _check(dict(state_pool=state_pool), dtype=torch.float32, device=q.device)
    _check(dict(state_indices=state_indices), dtype=torch.int32, device=q.device)
    N, H, dk = q.shape
    dv = v.shape[2]
    if state_indices.shape != (N,) or state_pool.shape[1:] != (H, dk, dv):
        raise ValueError("state_indices must be [N] and state_pool [P, H, dk, dv]")
    rc = library().la_decode_step_slots(_ptr(q), _ptr(k), _ptr(v), _ptr(beta_logits),
                                        _ptr(gate_logits), _ptr(o), _io(q), N, H, dk, dv,
                                        float(scale), int(flags), _ptr(state_pool),
                                        int(state_pool.shape[0]), _ptr(state_indices),
                                        _stream(stream))
    if rc != LA_OK:
        raise LinAttnError(rc, "la_decode_step_slots")
    return o


def la_check_device(stream=None) -> int:
    """Synchronise the stream and return (and clear) any device-side error."""
    return int(library().la_check_device(_stream(stream)))


def la_selftest_wait_timeout(stream=None) -> None:
    """Launch the failure-path self-test (a bounded in-kernel wait that runs
    out); the next la_check_device reports LA_ERR_TIMEOUT."""
    rc = library().la_selftest_wait_timeout(_stream(stream))
    if rc != LA_OK:
        raise LinAttnError(rc, "la_selftest_wait_timeout")
