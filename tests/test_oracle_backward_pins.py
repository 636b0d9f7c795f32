"""Pins of the oracle's backward pass (oracle.delta_backward) against facts
that do not come from its own code: central finite differences of the
forward oracle (itself pinned in test_oracle_pins.py), and closed forms.

The scalar loss is  L = sum(d_o * o) + sum(d_final_S * final_S)  for fixed
random d_o, d_final_S, so its gradient with respect to every input is what
delta_backward returns for those output gradients.  fp64 central differences
with step 1e-6 are accurate to ~1e-9 relative here."""
import numpy as np
import pytest

import oracle

H_FD = 1e-6


def _case(lengths, H, dk, dv, gate, seed, init=True):
    rs = np.random.default_rng(seed)
    ntok = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    N = len(lengths)
    inp = {
        "q": rs.standard_normal((ntok, H, dk)),
        "k": rs.standard_normal((ntok, H, dk)),
        "v": rs.standard_normal((ntok, H, dv)),
        "beta_logits": rs.standard_normal((ntok, H)),
        "gate_logits": (None if gate == "none" else
                        rs.standard_normal((ntok, H) if gate == "scalar" else (ntok, H, dk)) + 1.0),
        "init_S": rs.standard_normal((N, H, dk, dv)) * 0.5 if init else None,
    }
    grads = {"d_o": rs.standard_normal((ntok, H, dv)),
             "d_final_S": rs.standard_normal((N, H, dk, dv))}
    return inp, cu, grads


def _flags(gate, extra=0):
    return oracle.L2NORM_K | extra | (oracle.SCALAR_GATE if gate == "scalar" else 0)


def _loss(inp, cu, grads, flags, scale):
    o, fS = oracle.delta(inp["q"], inp["k"], inp["v"], inp["beta_logits"], inp["gate_logits"],
                         cu, scale=scale, flags=flags, init_S=inp["init_S"], nthreads=1)
    return float((grads["d_o"] * o).sum() + (grads["d_final_S"] * fS).sum())


def _grads(inp, cu, grads, flags, scale):
    g = oracle.delta_backward(inp["q"], inp["k"], inp["v"], inp["beta_logits"],
                              inp["gate_logits"], cu, grads["d_o"], grads["d_final_S"],
                              scale=scale, flags=flags, init_S=inp["init_S"], nthreads=1)
    return {"q": g["dq"], "k": g["dk"], "v": g["dv"], "beta_logits": g["d_beta_logits"],
            "gate_logits": g["d_gate_logits"], "init_S": g["d_init_S"]}


def _fd_element(inp, cu, grads, flags, scale, name, idx):
    x = inp[name]
    keep = x[idx]
    x[idx] = keep + H_FD
    lp = _loss(inp, cu, grads, flags, scale)
    x[idx] = keep - H_FD
    lm = _loss(inp, cu, grads, flags, scale)
    x[idx] = keep
    return (lp - lm) / (2 * H_FD)


FD_CASES = [("channel", 0, 1.0), ("none", 0, 0.7), ("scalar", 0, 1.0),
            ("channel", oracle.SILU_QK | oracle.L2NORM_Q, 1.3),
            ("scalar", oracle.ADDITIVE, 1.0), ("channel", oracle.ADDITIVE, 0.8)]


@pytest.mark.parametrize("gate,extra,scale", FD_CASES)
def test_backward_equals_finite_differences_elementwise(gate, extra, scale):
    """Every element of every input of a tiny ragged batch (an empty sequence
    included): the gradient equals the central difference of the loss."""
    inp, cu, grads = _case([3, 0, 4], 2, 3, 2, gate, seed=7)
    flags = _flags(gate, extra)
    g = _grads(inp, cu, grads, flags, scale)
    for name, x in inp.items():
        if x is None:
            continue
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            fd[idx] = _fd_element(inp, cu, grads, flags, scale, name, idx)
        err = np.abs(fd - g[name]).max() / max(np.abs(fd).max(), 1e-3)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("gate", ["none", "channel", "scalar"])
def test_backward_equals_directional_differences(gate):
    """Longer sequences (70 and 5 tokens), 16-wide heads: the derivative of
    the loss along a random direction in each input equals the gradient's
    inner product with that direction."""
    inp, cu, grads = _case([70, 5], 2, 16, 8, gate, seed=11)
    flags = _flags(gate)
    g = _grads(inp, cu, grads, flags, 1.0)
    rs = np.random.default_rng(3)
    for name, x in inp.items():
        if x is None:
            continue
        d = rs.standard_normal(x.shape)
        base = x.copy()
        inp[name] = base + H_FD * d
        lp = _loss(inp, cu, grads, flags, 1.0)
        inp[name] = base - H_FD * d
        lm = _loss(inp, cu, grads, flags, 1.0)
        inp[name] = base
        fd = (lp - lm) / (2 * H_FD)
        an = float((g[name] * d).sum())
        assert abs(fd - an) <= 1e-6 * max(abs(fd), 1.0), (name, fd, an)


def test_zero_beta_gives_no_value_gradient():
    """beta -> 0 (logit -60): nothing is written, so the values receive no
    gradient and the state only decays."""
    inp, cu, grads = _case([9], 1, 4, 3, "channel", seed=5)
    inp["beta_logits"][:] = -60.0
    g = _grads(inp, cu, grads, _flags("channel"), 1.0)
    assert np.abs(g["v"]).max() < 1e-20


def test_orthonormal_readback_gradient_is_the_output_gradient():
    """alpha = 1, beta = 1 (logit 40), keys e_0..e_3 written once with zero
    queries, then one token reading q = e_i while writing along e_4: its
    output is exactly v_i, so dv_i equals that token's output gradient and
    every other value gets none (no final-state gradient)."""
    d, n, i_read = 5, 4, 2
    ntok = n + 1
    q = np.zeros((ntok, 1, d))
    k = np.zeros((ntok, 1, d))
    for t in range(n):
        k[t, 0, t] = 1.0
    k[n, 0, n] = 1.0
    q[n, 0, i_read] = 1.0
    rs = np.random.default_rng(9)
    v = rs.standard_normal((ntok, 1, 3))
    bl = np.full((ntok, 1), 40.0)
    do = np.zeros((ntok, 1, 3))
    do[n, 0] = rs.standard_normal(3)
    g = oracle.delta_backward(q, k, v, bl, None, [0, ntok], do, None, nthreads=1)
    want = np.zeros_like(v)
    want[i_read, 0] = do[n, 0]
    assert np.abs(g["dv"] - want).max() < 1e-15


# ------------------------------------------- the pins catch planted mistakes

BACKWARD_MUTATIONS = [
    ("read-path term of dk dropped", "dkh[i] -= beta * acc;", "dkh[i] -= 0.0 * acc;"),
    ("delta term of dS with the wrong sign", "dS[i * dv + j] -= beta * kk[i] * du[j];",
     "dS[i * dv + j] += beta * kk[i] * du[j];"),
    ("decay not applied to dS", "dS[i * dv + j] *= al[i];", "dS[i * dv + j] *= 1.0;"),
    ("scale dropped from dq", "dqh[i] = c->scale * acc;", "dqh[i] = acc;"),
    ("dq from the state before the write", "acc += St[i * dv + j] * dot[j];",
     "acc += Sp[i * dv + j] * dot[j];"),
    ("sigmoid derivative incomplete", "dbeta * beta * (1.0 - beta);", "dbeta * beta;"),
    ("norm projection dropped", "(dy[i] - y[i] * ydy) / nrm", "dy[i] / nrm"),
    ("silu derivative incomplete", "dx[i] = ds[i] * sg * (1.0 + x[i] * (1.0 - sg));",
     "dx[i] = ds[i] * sg;"),
    ("scalar gate from one channel", "-acc * al[0] * sigmoid(g)", "-da[0] * al[0] * sigmoid(g)"),
    ("decay gradient against the decayed state", "acc += dS[i * dv + j] * Sp[i * dv + j];",
     "acc += dS[i * dv + j] * Sd[i * dv + j];"),
    ("beta gradient without the read", "dbeta += du[j] * (vt[j] - old);",
     "dbeta += du[j] * vt[j];"),
    ("final-state gradient ignored", "if (c->d_final_S) memcpy(dS", "if (0) memcpy(dS"),
    ("additive rule keeps the read-path terms", "        if (!additive) {\n            for (int i = 0; i < dk; ++i) {\n                double acc = 0.0;",
     "        if (1) {\n            for (int i = 0; i < dk; ++i) {\n                double acc = 0.0;"),
]


def _backward_pins():
    calls = []
    for gate, extra, scale in FD_CASES:
        calls.append(lambda a=(gate, extra, scale):
                     test_backward_equals_finite_differences_elementwise(*a))
    calls += [test_zero_beta_gives_no_value_gradient,
              test_orthonormal_readback_gradient_is_the_output_gradient]
    return calls


@pytest.mark.parametrize("mut", BACKWARD_MUTATIONS, ids=[m[0] for m in BACKWARD_MUTATIONS])
def test_backward_pins_catch_planted_mistake(mut, tmp_path, monkeypatch):
    name, old, new = mut
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site not unique: {old}"
    variant = oracle.OracleLib(oracle.build_variant(src.replace(old, new), str(tmp_path)))
    monkeypatch.setattr(oracle, "delta_backward", variant.delta_backward)
    failed = 0
    for call in _backward_pins():
        try:
            call()
        except AssertionError:
            failed += 1
    assert failed, f"no pin caught: {name}"
