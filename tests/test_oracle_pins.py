"""Pins for the fp64 oracle against facts that do not come from the oracle.

Every test here checks the oracle (``oracle/linattn_oracle.c``) against
something fixed independently of its code: brute-force matrix forms, closed
forms, exact special cases named on the page "From GPT-2 to Kimi K3,
explained", an independent fp64 transcription of the chunkwise WY/UT
algorithm, and structural invariants (resume, packing, restart).  A dropped
term, a wrong sign, a transposed state or a decay on the wrong axis in the
oracle fails at least one of them (dk != dv everywhere for that reason).
"""
import json
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.special

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
BIG = 1e4  # logit that makes sigmoid exactly 1 (or 0) in fp64


def rng(seed):
    return np.random.default_rng(seed)


def unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def log_alpha_from_logits(g):
    # log alpha = -softplus(g) = -log(1 + e^g), via the library's logaddexp
    return -np.logaddexp(0.0, g)


# ----------------------------------------------------------- ELU+1 (pin a)

def phi(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def brute_linear(q, k, v):
    """Causal-masked (phi(Q) phi(K)^T) V with row-sum normalisation."""
    A = np.tril(phi(q) @ phi(k).T)
    return (A @ v) / A.sum(axis=1, keepdims=True)


def test_linear_equals_bruteforce_masked_attention():
    r = rng(1)
    lens = [37, 1, 64]
    H, dk, dv = 3, 8, 5
    ntok = sum(lens)
    q, k, v = r.normal(size=(ntok, H, dk)), r.normal(size=(ntok, H, dk)), r.normal(size=(ntok, H, dv))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, fS, fz = oracle.linear(q, k, v, cu)
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        for h in range(H):
            ref = brute_linear(q[s:e, h], k[s:e, h], v[s:e, h])
            np.testing.assert_allclose(o[s:e, h], ref, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(fS[n, h], phi(k[s:e, h]).T @ v[s:e, h], rtol=1e-12)
            np.testing.assert_allclose(fz[n, h], phi(k[s:e, h]).sum(0), rtol=1e-12)


def test_linear_resume_equals_single_pass():
    r = rng(2)
    T, H, dk, dv = 50, 2, 6, 4
    q, k, v = r.normal(size=(T, H, dk)), r.normal(size=(T, H, dk)), r.normal(size=(T, H, dv))
    o, fS, fz = oracle.linear(q, k, v, [0, T])
    t1 = 17
    o1, S1, z1 = oracle.linear(q[:t1], k[:t1], v[:t1], [0, t1])
    o2, S2, z2 = oracle.linear(q[t1:], k[t1:], v[t1:], [0, T - t1], init_S=S1, init_z=z1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=1e-12)
    np.testing.assert_allclose(S2, fS, rtol=1e-12)
    np.testing.assert_allclose(z2, fz, rtol=1e-12)


# ------------------------------------------------- read-back (pin b)

def test_readback_golden_from_page():
    """One write then a read with the same key returns ||k||^2 v (page's
    DeltaNet (Fast Weight Programmers) remark); a unit key returns v."""
    g = json.load(open(os.path.join(HERE, "golden", "readback_norm_scaling.json")))
    k = np.array(g["k"])[None, None, :]
    v = np.array(g["v"])[None, None, :]
    bl = np.full((1, 1), BIG)
    # raw key (no normalisation): read-back is scaled by ||k||^2
    o, _ = oracle.delta(k, k, v, bl, None, [0, 1], flags=0)
    np.testing.assert_allclose(o[0, 0], g["read_back"], rtol=1e-14)
    # unit key: exact value
    o, _ = oracle.delta(k, k, v, bl, None, [0, 1], flags=oracle.L2NORM_K | oracle.L2NORM_Q)
    np.testing.assert_allclose(o[0, 0], g["read_back_unit_key"], rtol=1e-14)


def test_orthonormal_keys_read_back_exactly():
    r = rng(3)
    dk, dv, H = 16, 7, 2
    T = dk
    Qm, _ = np.linalg.qr(r.normal(size=(dk, dk)))
    k = np.stack([Qm.T * (1 + h) for h in range(H)], axis=1)  # scaled: L2 flag makes them unit
    v = r.normal(size=(T, H, dv))
    q = r.normal(size=(T, H, dk))
    bl = np.full((T, H), BIG)
    _, S = oracle.delta(q, k, v, bl, None, [0, T], flags=oracle.L2NORM_K)
    for h in range(H):
        kk = unit_rows(k[:, h])
        np.testing.assert_allclose(kk @ S[0, h], v[:, h], atol=1e-12)


def test_rewrite_replaces_old_value():
    """The delta rule removes what the key held and writes the new value in
    its place (section DeltaNet (Fast Weight Programmers))."""
    r = rng(4)
    dk, dv = 8, 5
    k1 = unit_rows(r.normal(size=dk))
    k = np.stack([k1, k1])[:, None, :]
    v = r.normal(size=(2, 1, dv))
    q = k.copy()
    o, S = oracle.delta(q, k, v, np.full((2, 1), BIG), None, [0, 2], flags=oracle.L2NORM_K)
    np.testing.assert_allclose(o[0, 0], v[0, 0], atol=1e-13)
    np.testing.assert_allclose(o[1, 0], v[1, 0], atol=1e-13)
    np.testing.assert_allclose(k1 @ S[0, 0], v[1, 0], atol=1e-13)


def test_orthogonal_keys_reduce_to_additive_attention():
    """With mutually orthogonal unit keys nothing is read back before a write,
    so u_t = beta_t v_t and O = tril(Q K^T) (beta * V)."""
    r = rng(5)
    dk, dv, T, H = 24, 9, 20, 2
    q = r.normal(size=(T, H, dk))
    v = r.normal(size=(T, H, dv))
    bl = r.normal(size=(T, H))
    k = np.zeros((T, H, dk))
    for h in range(H):
        Qm, _ = np.linalg.qr(r.normal(size=(dk, dk)))
        k[:, h] = Qm.T[:T]
    o, _ = oracle.delta(q, k, v, bl, None, [0, T], flags=oracle.L2NORM_K, scale=0.75)
    beta = scipy.special.expit(bl)
    for h in range(H):
        ref = 0.75 * np.tril(q[:, h] @ k[:, h].T) @ (beta[:, h, None] * v[:, h])
        np.testing.assert_allclose(o[:, h], ref, atol=1e-12)


# ------------------------------------------------- constant state (pin c)

@pytest.mark.parametrize("T", [1, 9, 130])
def test_state_size_independent_of_length(T):
    r = rng(6)
    H, dk, dv = 2, 8, 4
    q, k, v = r.normal(size=(T, H, dk)), r.normal(size=(T, H, dk)), r.normal(size=(T, H, dv))
    _, S = oracle.delta(q, k, v, r.normal(size=(T, H)), r.normal(size=(T, H, dk)), [0, T])
    _, S2, z2 = oracle.linear(q, k, v, [0, T])
    assert S.shape == (1, H, dk, dv) and S2.shape == (1, H, dk, dv) and z2.shape == (1, H, dk)
    assert S.nbytes == 1 * H * dk * dv * 8


# ---------------------------------------- chunkwise transcription (pin d)

def chunk_delta_wy(q, k, v, beta, C, S0=None):
    """Independent fp64 chunkwise delta rule (WY/UT form) for one head.

    Per chunk: A = strictly_lower(diag(beta) K K^T); T = (I + A)^{-1};
    W = T (beta K); U = T (beta V); u = U - W S; o = Q S + tril(Q K^T) u;
    S += K^T u.  The tail chunk may be shorter than C."""
    L, dk = k.shape
    S = np.zeros((dk, v.shape[1])) if S0 is None else S0.copy()
    out = np.zeros((L, v.shape[1]))
    for s in range(0, L, C):
        e = min(L, s + C)
        K, Q, V, b = k[s:e], q[s:e], v[s:e], beta[s:e]
        n = e - s
        A = np.tril(b[:, None] * (K @ K.T), -1)
        T = scipy.linalg.solve_triangular(np.eye(n) + A, np.eye(n), lower=True, unit_diagonal=True)
        assert np.allclose(T @ (np.eye(n) + A), np.eye(n), atol=1e-10)
        W, U = T @ (b[:, None] * K), T @ (b[:, None] * V)
        u = U - W @ S
        out[s:e] = Q @ S + np.tril(Q @ K.T) @ u
        S = S + K.T @ u
    return out, S


def chunk_delta_gated(q, k, v, beta, log_alpha, C, S0=None):
    """Independent fp64 chunk form with one decay per key channel.

    b = inclusive cumulative sum of log alpha inside the chunk (the page's
    cumulative decay: a token written at x and read at x+t has been scaled by
    alpha_x ... alpha_{x+t}).  Pairwise factors exp(b_r - b_i) <= 1 only."""
    L, dk = k.shape
    S = np.zeros((dk, v.shape[1])) if S0 is None else S0.copy()
    out = np.zeros((L, v.shape[1]))
    for s in range(0, L, C):
        e = min(L, s + C)
        K, Q, V, bt, la = k[s:e], q[s:e], v[s:e], beta[s:e], log_alpha[s:e]
        n = e - s
        bcum = np.cumsum(la, axis=0)                         # [n, dk]
        D = np.exp(bcum[:, None, :] - bcum[None, :, :])      # [r, i, c], used for i <= r
        lower = np.tril(np.ones((n, n)), -1)
        A = bt[:, None] * np.einsum("rc,ic,ric->ri", K, K, np.where(lower[..., None] > 0, D, 0.0))
        Aqk = np.einsum("rc,ic,ric->ri", Q, K, np.where(np.tril(np.ones((n, n)))[..., None] > 0, D, 0.0))
        T = scipy.linalg.solve_triangular(np.eye(n) + A, np.eye(n), lower=True, unit_diagonal=True)
        G = np.exp(bcum)                                     # decay from chunk start
        W = T @ (bt[:, None] * K * G)
        U = T @ (bt[:, None] * V)
        u = U - W @ S
        out[s:e] = (Q * G) @ S + Aqk @ u
        Gend = np.exp(bcum[-1])
        S = Gend[:, None] * S + (K * np.exp(bcum[-1][None, :] - bcum)).T @ u
    return out, S


@pytest.mark.parametrize("C", [16, 64])
def test_oracle_matches_chunkwise_wy_transcription(C):
    r = rng(7)
    T, H, dk, dv = 150, 2, 16, 12   # ragged tail
    q, k, v = r.normal(size=(T, H, dk)), r.normal(size=(T, H, dk)), r.normal(size=(T, H, dv))
    bl = r.normal(size=(T, H))
    S0 = r.normal(size=(1, H, dk, dv)) * 0.1
    o, S = oracle.delta(q, k, v, bl, None, [0, T], flags=oracle.L2NORM_K, init_S=S0)
    beta = scipy.special.expit(bl)
    for h in range(H):
        ref_o, ref_S = chunk_delta_wy(q[:, h], unit_rows(k[:, h]), v[:, h], beta[:, h], C, S0[0, h])
        np.testing.assert_allclose(o[:, h], ref_o, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(S[0, h], ref_S, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("C", [8, 64])
def test_gated_oracle_matches_gated_chunk_form(C):
    r = rng(8)
    T, H, dk, dv = 100, 2, 12, 10
    q, k, v = r.normal(size=(T, H, dk)), r.normal(size=(T, H, dk)), r.normal(size=(T, H, dv))
    bl = r.normal(size=(T, H))
    gl = r.normal(size=(T, H, dk)) + 2.0
    S0 = r.normal(size=(1, H, dk, dv)) * 0.02
    o, S = oracle.delta(q, k, v, bl, gl, [0, T], flags=oracle.L2NORM_K, init_S=S0)
    beta, la = scipy.special.expit(bl), log_alpha_from_logits(gl)
    for h in range(H):
        ref_o, ref_S = chunk_delta_gated(q[:, h], unit_rows(k[:, h]), v[:, h], beta[:, h],
                                         la[:, h], C, S0[0, h])
        np.testing.assert_allclose(o[:, h], ref_o, rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(S[0, h], ref_S, rtol=1e-9, atol=1e-11)


# ------------------------------------------------ special cases (pin e)

def test_beta_zero_only_decays_state_on_key_axis():
    r = rng(9)
    T, H, dk, dv = 5, 2, 6, 3
    S0 = r.normal(size=(1, H, dk, dv))
    q = r.normal(size=(T, H, dk))
    gl = r.normal(size=(T, H, dk))
    o, S = oracle.delta(q, r.normal(size=(T, H, dk)), r.normal(size=(T, H, dv)),
                        np.full((T, H), -BIG), gl, [0, T], init_S=S0, flags=0)
    cum = np.cumsum(log_alpha_from_logits(gl), axis=0)     # [T, H, dk]
    for h in range(H):
        np.testing.assert_allclose(S[0, h], np.exp(cum[-1, h])[:, None] * S0[0, h], rtol=1e-12)
        for t in range(T):
            ref = (np.exp(cum[t, h])[:, None] * S0[0, h]).T @ q[t, h]
            np.testing.assert_allclose(o[t, h], ref, rtol=1e-11, atol=1e-13)


def test_known_gate_and_beta_values():
    """logit log(3) gives alpha = 1/4 exactly; logit 0 gives beta = 1/2."""
    dk, dv = 4, 3
    S0 = np.arange(dk * dv, dtype=float).reshape(1, 1, dk, dv)
    e = np.eye(dk)[None, :1, :]                     # unit key e_0, one head
    v = np.array([[[2.0, -4.0, 6.0]]])
    gl = np.full((1, 1, dk), np.log(3.0))
    o, S = oracle.delta(e, e, v, np.zeros((1, 1)), gl, [0, 1], init_S=S0, flags=0)
    Sd = 0.25 * S0[0, 0]
    u = 0.5 * (v[0, 0] - Sd[0])
    ref = Sd.copy()
    ref[0] += u
    np.testing.assert_allclose(S[0, 0], ref, rtol=1e-15)
    np.testing.assert_allclose(o[0, 0], ref[0], rtol=1e-15)


def test_gate_one_equals_pure_delta_and_gate_zero_restarts():
    r = rng(10)
    T, H, dk, dv = 40, 2, 8, 6
    q, k, v = r.normal(size=(T, H, dk)), r.normal(size=(T, H, dk)), r.normal(size=(T, H, dv))
    bl = r.normal(size=(T, H))
    S0 = r.normal(size=(1, H, dk, dv))
    o_plain, S_plain = oracle.delta(q, k, v, bl, None, [0, T], init_S=S0)
    o_one, S_one = oracle.delta(q, k, v, bl, np.full((T, H, dk), -BIG), [0, T], init_S=S0)
    np.testing.assert_array_equal(o_one, o_plain)
    np.testing.assert_array_equal(S_one, S_plain)
    # alpha = 0 at token t0 clears everything written before it
    t0 = 13
    gl = r.normal(size=(T, H, dk))
    gl[t0] = BIG
    o_all, S_all = oracle.delta(q, k, v, bl, gl, [0, T], init_S=S0)
    o_tail, S_tail = oracle.delta(q[t0:], k[t0:], v[t0:], bl[t0:], gl[t0:], [0, T - t0])
    np.testing.assert_allclose(o_all[t0:], o_tail, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S_all, S_tail, rtol=1e-12, atol=1e-14)


def test_scalar_gate_decays_orthonormal_memories_exactly():
    """One decay per token and head (section Gated DeltaNet): with
    orthonormal keys and beta = 1 nothing interferes, so after T steps the
    memory written at step j reads back as prod_{t>j} alpha_t times v_j."""
    r = rng(30)
    dk, dv, H = 12, 5, 2
    T = dk
    Qm, _ = np.linalg.qr(r.normal(size=(dk, dk)))
    k = np.stack([Qm.T for _ in range(H)], axis=1)
    v = r.normal(size=(T, H, dv))
    q = r.normal(size=(T, H, dk))
    bl = np.full((T, H), BIG)
    gl = r.normal(size=(T, H)) + 1.0
    _, S = oracle.delta(q, k, v, bl, gl, [0, T], flags=oracle.L2NORM_K | oracle.SCALAR_GATE)
    la = log_alpha_from_logits(gl)                       # [T][H]
    for h in range(H):
        tail = np.exp(np.cumsum(la[::-1, h])[::-1])      # prod_{t>=j} alpha_t
        decay_after = np.append(tail[1:], 1.0)           # prod_{t>j} alpha_t
        np.testing.assert_allclose(k[:, h] @ S[0, h], decay_after[:, None] * v[:, h],
                                   rtol=1e-12, atol=1e-14)


def test_scalar_gate_is_the_per_channel_gate_held_constant_across_channels():
    r = rng(31)
    lens = [23, 1, 40]
    H, dk, dv = 3, 6, 4
    ntok = sum(lens)
    q, k, v = r.normal(size=(ntok, H, dk)), r.normal(size=(ntok, H, dk)), r.normal(size=(ntok, H, dv))
    bl = r.normal(size=(ntok, H))
    gl = r.normal(size=(ntok, H)) + 2.0
    cu = np.concatenate([[0], np.cumsum(lens)])
    S0 = r.normal(size=(len(lens), H, dk, dv))
    o_s, S_s = oracle.delta(q, k, v, bl, gl, cu, flags=oracle.L2NORM_K | oracle.SCALAR_GATE,
                            init_S=S0)
    o_c, S_c = oracle.delta(q, k, v, bl, np.repeat(gl[:, :, None], dk, axis=2), cu,
                            flags=oracle.L2NORM_K, init_S=S0)
    np.testing.assert_array_equal(o_s, o_c)
    np.testing.assert_array_equal(S_s, S_c)
    # a zero decay at one token restarts the memory from there (per head)
    t0 = 9
    gl2 = gl[:40].copy()
    gl2[t0] = BIG
    o_all, S_all = oracle.delta(q[:40], k[:40], v[:40], bl[:40], gl2, [0, 40],
                                flags=oracle.L2NORM_K | oracle.SCALAR_GATE, init_S=S0[:1])
    o_tail, S_tail = oracle.delta(q[t0:40], k[t0:40], v[t0:40], bl[t0:40], gl2[t0:], [0, 40 - t0],
                                  flags=oracle.L2NORM_K | oracle.SCALAR_GATE)
    np.testing.assert_allclose(o_all[t0:], o_tail, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S_all, S_tail, rtol=1e-12, atol=1e-14)


def test_one_token_closed_form_and_scale():
    r = rng(11)
    H, dk, dv = 3, 8, 5
    q, k, v = r.normal(size=(1, H, dk)), r.normal(size=(1, H, dk)), r.normal(size=(1, H, dv))
    bl = r.normal(size=(1, H))
    o, S = oracle.delta(q, k, v, bl, None, [0, 1], scale=0.5, flags=oracle.L2NORM_K)
    beta = scipy.special.expit(bl)
    for h in range(H):
        kn = k[0, h] / np.linalg.norm(k[0, h])
        np.testing.assert_allclose(S[0, h], np.outer(kn, beta[0, h] * v[0, h]), rtol=1e-13)
        np.testing.assert_allclose(o[0, h], 0.5 * beta[0, h] * (kn @ q[0, h]) * v[0, h], rtol=1e-12)


def test_silu_and_query_norm_flags():
    r = rng(12)
    H, dk, dv = 2, 6, 4
    q, k, v = r.normal(size=(1, H, dk)), r.normal(size=(1, H, dk)), r.normal(size=(1, H, dv))
    bl = r.normal(size=(1, H))
    flags = oracle.L2NORM_K | oracle.L2NORM_Q | oracle.SILU_QK
    o, _ = oracle.delta(q, k, v, bl, None, [0, 1], flags=flags)
    silu = lambda x: x * scipy.special.expit(x)
    for h in range(H):
        qn, kn = unit_rows(silu(q[0, h])), unit_rows(silu(k[0, h]))
        ref = scipy.special.expit(bl[0, h]) * (kn @ qn) * v[0, h]
        np.testing.assert_allclose(o[0, h], ref, rtol=1e-12)


# ------------------------------------------- structural invariants (pin f)

def test_varlen_packing_equals_separate_runs_and_resume():
    r = rng(13)
    lens = [7, 30, 1, 19]
    H, dk, dv = 2, 8, 5
    ntok = sum(lens)
    q, k, v = r.normal(size=(ntok, H, dk)), r.normal(size=(ntok, H, dk)), r.normal(size=(ntok, H, dv))
    bl, gl = r.normal(size=(ntok, H)), r.normal(size=(ntok, H, dk)) + 2
    S0 = r.normal(size=(len(lens), H, dk, dv)) * 0.1
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, S = oracle.delta(q, k, v, bl, gl, cu, init_S=S0)
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        o_n, S_n = oracle.delta(q[s:e], k[s:e], v[s:e], bl[s:e], gl[s:e], [0, e - s],
                                init_S=S0[n:n + 1])
        np.testing.assert_array_equal(o[s:e], o_n)
        np.testing.assert_array_equal(S[n], S_n[0])
    # resume: split the longest sequence in two calls
    s, e = cu[1], cu[2]
    mid = s + 11
    o1, S1 = oracle.delta(q[s:mid], k[s:mid], v[s:mid], bl[s:mid], gl[s:mid], [0, mid - s],
                          init_S=S0[1:2])
    o2, S2 = oracle.delta(q[mid:e], k[mid:e], v[mid:e], bl[mid:e], gl[mid:e], [0, e - mid],
                          init_S=S1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o[s:e], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(S2[0], S[1], rtol=1e-13, atol=1e-15)


def test_decode_steps_equal_prefill():
    r = rng(14)
    N, H, dk, dv, steps = 3, 2, 8, 6, 5
    q = r.normal(size=(steps, N, H, dk))
    k = r.normal(size=(steps, N, H, dk))
    v = r.normal(size=(steps, N, H, dv))
    bl = r.normal(size=(steps, N, H))
    gl = r.normal(size=(steps, N, H, dk)) + 2
    S = r.normal(size=(N, H, dk, dv)) * 0.02
    outs = []
    st = S
    for t in range(steps):
        o, st = oracle.decode(q[t], k[t], v[t], bl[t], gl[t], st)
        outs.append(o)
    # the same tokens as a packed prefill, sequence-major
    tr = lambda x: np.ascontiguousarray(np.swapaxes(x, 0, 1).reshape((N * steps,) + x.shape[2:]))
    cu = np.arange(N + 1) * steps
    o_p, S_p = oracle.delta(tr(q), tr(k), tr(v), tr(bl), tr(gl), cu, init_S=S)
    np.testing.assert_allclose(tr(np.stack(outs)), o_p, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(st, S_p, rtol=1e-13, atol=1e-15)


def test_thread_count_does_not_change_results():
    r = rng(15)
    lens = [20, 33, 5]
    H, dk, dv = 4, 8, 8
    ntok = sum(lens)
    args = (r.normal(size=(ntok, H, dk)), r.normal(size=(ntok, H, dk)), r.normal(size=(ntok, H, dv)),
            r.normal(size=(ntok, H)), r.normal(size=(ntok, H, dk)), np.concatenate([[0], np.cumsum(lens)]))
    o1, S1 = oracle.delta(*args, nthreads=1)
    o8, S8 = oracle.delta(*args, nthreads=8)
    np.testing.assert_array_equal(o1, o8)
    np.testing.assert_array_equal(S1, S8)


# ------------------------------------- additive decayed state (Mamba-2 form)

def _decayed_attention(q, k, v, log_a, S0):
    """Brute force from the products of the decays, one (sequence, head):
    o_t = sum_{i<=t} sum_c q_t[c] k_i[c] prod_{i<s<=t} alpha_s[c] v_i
          + sum_c q_t[c] prod_{s<=t} alpha_s[c] S0[c, :]."""
    T, dk = q.shape
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        for i in range(t + 1):
            dec = np.exp(log_a[i + 1:t + 1].sum(0))   # prod over s in (i, t]
            o[t] += (q[t] * k[i] * dec).sum() * v[i]
        o[t] += (q[t] * np.exp(log_a[:t + 1].sum(0))) @ S0
    fS = np.exp(log_a.sum(0))[:, None] * S0
    for i in range(T):
        fS += np.outer(k[i] * np.exp(log_a[i + 1:].sum(0)), v[i])
    return o, fS


@pytest.mark.parametrize("gate", ["channel", "scalar"])
def test_additive_rule_equals_bruteforce_decayed_attention(gate):
    """ADDITIVE: the page's Mamba-2 update S_t = alpha_t S_{t-1} + k_t v_t^T
    (section Gated DeltaNet): every value is written at full strength and
    only decays afterwards."""
    r = rng(31)
    lengths, H, dk, dv = [9, 4], 2, 5, 3
    ntok = sum(lengths)
    q, k, v = r.standard_normal((ntok, H, dk)), r.standard_normal((ntok, H, dk)), \
        r.standard_normal((ntok, H, dv))
    g = r.standard_normal((ntok, H) if gate == "scalar" else (ntok, H, dk)) + 0.5
    S0 = r.standard_normal((2, H, dk, dv))
    flags = oracle.ADDITIVE | (oracle.SCALAR_GATE if gate == "scalar" else 0)
    o, fS = oracle.delta(q, k, v, None, g, [0, 9, 13], scale=0.5, flags=flags, init_S=S0)
    la = log_alpha_from_logits(g)
    if gate == "scalar":
        la = np.repeat(la[:, :, None], dk, axis=2)
    for n, (a, b) in enumerate([(0, 9), (9, 13)]):
        for h in range(H):
            ro, rS = _decayed_attention(q[a:b, h], k[a:b, h], v[a:b, h], la[a:b, h], S0[n, h])
            assert np.abs(o[a:b, h] - 0.5 * ro).max() < 1e-12
            assert np.abs(fS[n, h] - rS).max() < 1e-12


def test_additive_rule_without_gate_is_unnormalised_linear_attention():
    """No decay: o = tril(Q K^T) V, the additive form the delta rule replaces."""
    r = rng(32)
    T, dk, dv = 11, 4, 6
    q, k, v = r.standard_normal((T, 1, dk)), r.standard_normal((T, 1, dk)), \
        r.standard_normal((T, 1, dv))
    o, fS = oracle.delta(q, k, v, r.standard_normal((T, 1)), None, [0, T], flags=oracle.ADDITIVE)
    want = np.tril(q[:, 0] @ k[:, 0].T) @ v[:, 0]
    assert np.abs(o[:, 0] - want).max() < 1e-12
    assert np.abs(fS[0, 0] - k[:, 0].T @ v[:, 0]).max() < 1e-12
