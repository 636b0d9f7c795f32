"""fp64 CPU oracle for causal linear attention (ELU+1) and the gated delta rule.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library never imports, links or calls it, and it shares
no code with the CUDA path.

The arithmetic lives in ``linattn_oracle.c`` (plain token-by-token loops in
double precision).  This module only builds that file with gcc, marshals numpy
arrays into it and returns numpy arrays.

Parity status of each function (what pins it, see ``tests/test_oracle_pins.py``):

* ``linear``  -- pinned: brute-force causal-masked (phi(Q) phi(K)^T) V with
  row-sum normalisation; split-sequence resume; varlen packing.
* ``delta``   -- pinned: orthonormal-key read-back (v_i returned exactly);
  replace-on-rewrite; orthogonal keys reduce to additive attention
  tril(QK^T)V; an independent fp64 transcription of the chunkwise WY/UT
  algorithm (alpha = 1) and of a gated chunk form built from the cumulative
  decay; closed forms for one token and for beta = 0; alpha = 0 restarts.
* ``decode``  -- pinned: equals ``delta`` one token at a time, and a single
  step equals its closed form.
* ``delta`` with ``ADDITIVE`` (u = v, the decayed additive state) -- pinned:
  brute-force decayed causal attention written from the products of the
  decays, with an initial state and per-channel or scalar gates; no gate
  gives tril(QK^T) V.
* ``delta_backward`` -- pinned: central finite differences of ``delta``'s
  outputs (element by element on tiny inputs, along random directions on
  larger ones, with and without gate, scalar gate, silu / q-norm flags and
  an initial state); beta = 0 leaves v without gradient; with alpha = 1 and
  orthonormal keys written once, d v_i of a read-back is exactly the output
  gradient.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "linattn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liblinattn_oracle.so")

# Prologue option bits understood by the C oracle.
L2NORM_K = 1
L2NORM_Q = 2
SILU_QK = 4
SCALAR_GATE = 8   # gate_logits [ntok][H]: one decay per token and head
ADDITIVE = 16     # u = v: decayed additive state, no delta term and no beta

def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (no GPU needed)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleLib:
    """The oracle functions bound to one compiled copy of linattn_oracle.c.

    The default instance uses the committed source; tests may bind a
    deliberately altered copy (compiled with ``build_variant``) to check that
    the pins catch it."""

    def __init__(self, lib_path):
        lib = ctypes.CDLL(lib_path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        c_int, c_uint, c_double = ctypes.c_int, ctypes.c_uint, ctypes.c_double
        lib.la_oracle_linear.argtypes = [dp, dp, dp, dp, ip, c_int, c_int, c_int, c_int,
                                         dp, dp, dp, dp, c_int]
        lib.la_oracle_delta.argtypes = [dp, dp, dp, dp, dp, dp, ip, c_int, c_int, c_int, c_int,
                                        c_double, c_uint, dp, dp, c_int]
        lib.la_oracle_decode.argtypes = [dp, dp, dp, dp, dp, dp, c_int, c_int, c_int, c_int,
                                         c_double, c_uint, dp, c_int]
        lib.la_oracle_delta_backward.argtypes = [dp, dp, dp, dp, dp, ip, c_int, c_int, c_int,
                                                 c_int, c_double, c_uint, dp, dp, dp, dp, dp,
                                                 dp, dp, dp, dp, c_int]
        for f in (lib.la_oracle_linear, lib.la_oracle_delta, lib.la_oracle_decode,
                  lib.la_oracle_delta_backward):
            f.restype = c_int
        self.lib = lib
        self.L2NORM_K, self.L2NORM_Q, self.SILU_QK = L2NORM_K, L2NORM_Q, SILU_QK
        self.SCALAR_GATE = SCALAR_GATE

    def linear(self, *a, **k):
        return _linear(self.lib, *a, **k)

    def delta(self, *a, **k):
        return _delta(self.lib, *a, **k)

    def delta_backward(self, *a, **k):
        return _delta_backward(self.lib, *a, **k)

    def decode(self, *a, **k):
        return _decode(self.lib, *a, **k)


def build_variant(source_text: str, out_dir: str) -> str:
    """Compile an altered copy of the oracle source into out_dir (tests only)."""
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, "variant.c")
    with open(src, "w") as f:
        f.write(source_text)
    lib = os.path.join(out_dir, "libvariant.so")
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o", lib,
                    src, "-lm"], check=True)
    return lib


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


_default = None


def _load():
    global _default
    if _default is None:
        _default = OracleLib(build())
    return _default.lib


def _f64(x):
    """Widen any array-like (numpy, or a CPU torch tensor) to C-contiguous fp64."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen through float64 on the CPU
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _cu(cu_seqlens):
    a = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def default_threads() -> int:
    return os.cpu_count() or 1


def linear(q, k, v, cu_seqlens, init_S=None, init_z=None, nthreads=None):
    """ELU+1 causal linear attention (see _linear)."""
    return _linear(_load(), q, k, v, cu_seqlens, init_S, init_z, nthreads)


def delta(q, k, v, beta_logits, gate_logits, cu_seqlens, scale=1.0, flags=L2NORM_K,
          init_S=None, nthreads=None):
    """(Gated) delta rule (see _delta)."""
    return _delta(_load(), q, k, v, beta_logits, gate_logits, cu_seqlens, scale, flags, init_S,
                  nthreads)


def delta_backward(q, k, v, beta_logits, gate_logits, cu_seqlens, d_o, d_final_S=None,
                   scale=1.0, flags=L2NORM_K, init_S=None, nthreads=None):
    """Gradients of the (gated) delta rule (see _delta_backward)."""
    return _delta_backward(_load(), q, k, v, beta_logits, gate_logits, cu_seqlens, d_o,
                           d_final_S, scale, flags, init_S, nthreads)


def decode(q, k, v, beta_logits, gate_logits, state, scale=1.0, flags=L2NORM_K, nthreads=None):
    """One decode step (see _decode)."""
    return _decode(_load(), q, k, v, beta_logits, gate_logits, state, scale, flags, nthreads)


def _linear(lib, q, k, v, cu_seqlens, init_S=None, init_z=None, nthreads=None):
    """ELU+1 causal linear attention.  Shapes: q,k [ntok,H,dk], v [ntok,H,dv].

    Returns (o [ntok,H,dv], final_S [N,H,dk,dv], final_z [N,H,dk]) in fp64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu, cup = _cu(cu_seqlens)
    ntok, H, dk = q.shape
    dv = v.shape[2]
    N = len(cu) - 1
    o = np.zeros((ntok, H, dv))
    fS = np.zeros((N, H, dk, dv))
    fz = np.zeros((N, H, dk))
    iS, iz = _f64(init_S), _f64(init_z)
    rc = lib.la_oracle_linear(_ptr(q), _ptr(k), _ptr(v), _ptr(o), cup, N, H, dk, dv,
                              _ptr(iS), _ptr(iz), _ptr(fS), _ptr(fz),
                              nthreads or default_threads())
    if rc != 0:
        raise ValueError("la_oracle_linear rejected its arguments")
    return o, fS, fz


def _delta(lib, q, k, v, beta_logits, gate_logits, cu_seqlens, scale=1.0, flags=L2NORM_K,
           init_S=None, nthreads=None):
    """(Gated) delta rule, token by token.  gate_logits None means alpha = 1.

    Shapes: q,k [ntok,H,dk]; v [ntok,H,dv]; beta_logits [ntok,H];
    gate_logits [ntok,H,dk] (or [ntok,H] with flags & SCALAR_GATE);
    init_S [N,H,dk,dv].  Returns (o, final_S) in fp64.
    """
    q, k, v, bl, gl = _f64(q), _f64(k), _f64(v), _f64(beta_logits), _f64(gate_logits)
    cu, cup = _cu(cu_seqlens)
    ntok, H, dk = q.shape
    dv = v.shape[2]
    N = len(cu) - 1
    o = np.zeros((ntok, H, dv))
    fS = np.zeros((N, H, dk, dv))
    iS = _f64(init_S)
    rc = lib.la_oracle_delta(_ptr(q), _ptr(k), _ptr(v), _ptr(bl), _ptr(gl), _ptr(o), cup,
                             N, H, dk, dv, float(scale), int(flags), _ptr(iS), _ptr(fS),
                             nthreads or default_threads())
    if rc != 0:
        raise ValueError("la_oracle_delta rejected its arguments")
    return o, fS


def _decode(lib, q, k, v, beta_logits, gate_logits, state, scale=1.0, flags=L2NORM_K,
            nthreads=None):
    """One decode step for N sequences.  q,k [N,H,dk]; v [N,H,dv]; state [N,H,dk,dv].

    Returns (o [N,H,dv], new_state) in fp64; the input state is not modified.
    """
    q, k, v, bl, gl = _f64(q), _f64(k), _f64(v), _f64(beta_logits), _f64(gate_logits)
    st = _f64(state).copy()
    N, H, dk = q.shape
    dv = v.shape[2]
    o = np.zeros((N, H, dv))
    rc = lib.la_oracle_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(bl), _ptr(gl), _ptr(o),
                                  N, H, dk, dv, float(scale), int(flags), _ptr(st),
                                  nthreads or default_threads())
    if rc != 0:
        raise ValueError("la_oracle_decode rejected its arguments")
    return o, st


def _delta_backward(lib, q, k, v, beta_logits, gate_logits, cu_seqlens, d_o, d_final_S=None,
                    scale=1.0, flags=L2NORM_K, init_S=None, nthreads=None):
    """Gradients of ``_delta``'s outputs with respect to all its inputs,
    given the output gradient d_o [ntok,H,dv] and optionally the final-state
    gradient d_final_S [N,H,dk,dv].  Returns a dict of fp64 arrays: dq, dk,
    dv, d_beta_logits, d_gate_logits (None without gate), d_init_S.
    Rows of tokens outside every sequence stay zero."""
    q, k, v, bl, gl = _f64(q), _f64(k), _f64(v), _f64(beta_logits), _f64(gate_logits)
    do, dfS, iS = _f64(d_o), _f64(d_final_S), _f64(init_S)
    cu, cup = _cu(cu_seqlens)
    ntok, H, dk = q.shape
    dv = v.shape[2]
    N = len(cu) - 1
    out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
           "d_beta_logits": np.zeros(q.shape[:2]),
           "d_gate_logits": None if gl is None else np.zeros_like(gl),
           "d_init_S": np.zeros((N, H, dk, dv))}
    rc = lib.la_oracle_delta_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(bl), _ptr(gl), cup, N, H, dk, dv, float(scale),
        int(flags), _ptr(iS), _ptr(do), _ptr(dfS), _ptr(out["dq"]), _ptr(out["dk"]),
        _ptr(out["dv"]), _ptr(out["d_beta_logits"]), _ptr(out["d_gate_logits"]),
        _ptr(out["d_init_S"]), nthreads or default_threads())
    if rc != 0:
        raise ValueError("la_oracle_delta_backward rejected its arguments")
    return out
