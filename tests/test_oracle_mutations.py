"""The oracle's pins are strong enough to catch plausible mistakes.

Each case plants one mistake in a temporary copy of oracle/linattn_oracle.c
(on the CPU, never in the committed file), compiles it, rebinds the oracle
functions to it and runs every pin in tests/test_oracle_pins.py.  At least one
pin must fail for every planted mistake: a dropped term, a wrong sign, a
decay on the wrong axis or in the wrong order, a read before the write, a
wrong feature map, a missing normaliser, an ignored initial state, a skipped
token."""
import pytest

import oracle
import test_oracle_pins as pins

MUTATIONS = [
    ("decay dropped", "S[i * dv + j] *= alpha[i];", "S[i * dv + j] *= 1.0;", 1),
    ("decay on the value axis", "S[i * dv + j] *= alpha[i];", "S[i * dv + j] *= alpha[j % dk];", 1),
    ("decay after the write",
     "S[i * dv + j] *= alpha[i];", "S[i * dv + j] *= 1.0;", 1,
     "S[i * dv + j] += kk[i] * u[j];", "S[i * dv + j] = (S[i * dv + j] + kk[i] * u[j]) * alpha[i];"),
    ("delta sign", ": beta * (vt[j] - old);", ": beta * (vt[j] + old);", 1),
    ("beta dropped", ": beta * (vt[j] - old);", ": (vt[j] - old);", 1),
    ("read before the write", "acc += qq[i] * S[i * dv + j];",
     "acc += qq[i] * (S[i * dv + j] - kk[i] * u[j]);", 1),
    ("scale dropped", "ot[j] = c->scale * acc;", "ot[j] = acc;", 1),
    ("sigmoid sign", "if (x >= 0.0) return 1.0 / (1.0 + exp(-x));",
     "if (x >= 0.0) return 1.0 / (1.0 + exp(x));", 1),
    ("softplus sign", ": exp(-softplus(scalar_gate", ": exp(softplus(scalar_gate", 1),
    ("norm without sqrt", "double nrm = sqrt(s);", "double nrm = s;", 1),
    ("feature map without +1", "return x > 0.0 ? x + 1.0 : exp(x);",
     "return x > 0.0 ? x : exp(x);", 1),
    ("normaliser dropped", "ot[j] = num / den;", "ot[j] = num;", 1),
    ("normaliser not accumulated", "z[i] += fk[i];", "z[i] = fk[i];", 1),
    ("write with the query features", "S[i * dv + j] += fk[i] * vt[j];",
     "S[i * dv + j] += fq[i] * vt[j];", 1),
    ("initial states ignored", "if (c->init_S) memcpy(S, c->init_S + sbase",
     "if (0) memcpy(S, c->init_S + sbase", 2),
    ("first token of each sequence skipped", "for (int64_t t = c->cu[n]; t < c->cu[n + 1]; ++t)",
     "for (int64_t t = c->cu[n] + 1; t < c->cu[n + 1]; ++t)", 2),
    ("scalar gate of head 0 for every head", "scalar_gate ? c->gate_logits[t * H + h]",
     "scalar_gate ? c->gate_logits[t * H]", 1),
    ("scalar gate taken as no decay", "alpha[i] = !c->gate_logits ? 1.0",
     "alpha[i] = (!c->gate_logits || scalar_gate) ? 1.0", 1),
    ("additive rule keeps the delta", "u[j] = additive ? vt[j] : beta * (vt[j] - old);",
     "u[j] = beta * (vt[j] - old);", 1),
]


def pin_calls():
    calls = []
    for name in dir(pins):
        fn = getattr(pins, name)
        if not (name.startswith("test_") and callable(fn)):
            continue
        if name == "test_state_size_independent_of_length":
            calls += [(name, lambda f=fn, T=T: f(T)) for T in (1, 9, 130)]
        elif name == "test_oracle_matches_chunkwise_wy_transcription":
            calls += [(name, lambda f=fn, C=C: f(C)) for C in (16, 64)]
        elif name == "test_gated_oracle_matches_gated_chunk_form":
            calls += [(name, lambda f=fn, C=C: f(C)) for C in (8, 64)]
        elif name == "test_additive_rule_equals_bruteforce_decayed_attention":
            calls += [(name, lambda f=fn, g=g: f(g)) for g in ("channel", "scalar")]
        else:
            calls.append((name, fn))
    return calls


@pytest.mark.parametrize("mut", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(mut, tmp_path, monkeypatch):
    src = oracle.source_text()
    name, old, new, count = mut[:4]
    assert src.count(old) >= count, f"mutation site not found: {old}"
    src = src.replace(old, new, count)
    if len(mut) > 4:
        assert mut[4] in src
        src = src.replace(mut[4], mut[5], 1)
    variant = oracle.OracleLib(oracle.build_variant(src, str(tmp_path)))
    monkeypatch.setattr(oracle, "delta", variant.delta)
    monkeypatch.setattr(oracle, "linear", variant.linear)
    monkeypatch.setattr(oracle, "decode", variant.decode)
    failed = []
    for pin, call in pin_calls():
        try:
            call()
        except Exception:  # assertion or numerical failure of the pin
            failed.append(pin)
    assert failed, f"no pin caught: {name}"


def test_unmutated_source_passes_every_pin(tmp_path, monkeypatch):
    variant = oracle.OracleLib(oracle.build_variant(oracle.source_text(), str(tmp_path)))
    monkeypatch.setattr(oracle, "delta", variant.delta)
    monkeypatch.setattr(oracle, "linear", variant.linear)
    monkeypatch.setattr(oracle, "decode", variant.decode)
    for pin, call in pin_calls():
        call()
