"""Seeded synthetic inputs for the five linear/delta-rule attention workloads.

This module is shared by the tests, the bench and the oracle checks.  It holds
random draws, rounding to the I/O dtype and shape bookkeeping only: none of the
method's arithmetic (no feature map, normalisation, sigmoid, softplus or
recurrence) happens here.  The kernels and the oracle each apply the prologue
to the raw tensors produced below.

Recipe (fixed draw order from one ``torch.Generator('cpu')`` per call):
q, k, v ~ N(0, 1); beta logits ~ N(0, 1); gate logits ~ N(0, 1) + 2 (gated
workloads, giving alpha = exp(-softplus(.)) per token, head and key channel);
initial/decode state ~ N(0, 0.02^2) in fp32.  Every tensor is drawn in fp32 and
then rounded (round-to-nearest-even) to the I/O dtype, so both sides see the
same rounded values.

Packed layouts: token tensors [ntok][H][d] with sequences back to back as
``cu_seqlens`` says; beta logits [ntok][H]; gate logits [ntok][H][dk];
states [N][H][dk][dv] fp32.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "prefill_linear", "prefill_delta", "decode"
    H: int
    dk: int
    dv: int
    dtype: torch.dtype
    gated: bool = False
    lengths: tuple = ()  # prefill: per-sequence token counts
    n_seq: int = 0       # decode: number of sequences
    steps: int = 0       # decode: consecutive steps
    varlen: tuple = ()   # (total, lo, hi) for seeded length draws
    extra: dict = field(default_factory=dict)

    @property
    def ntok(self) -> int:
        return sum(self.lengths)


def varlen_lengths(total: int, lo: int, hi: int, seed: int) -> list[int]:
    """Draw integer lengths uniform in [lo, hi] until they reach ``total``;
    the last one is cut so that the lengths sum to exactly ``total``."""
    g = torch.Generator().manual_seed(seed + 7919)
    out: list[int] = []
    s = 0
    while s < total:
        L = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        L = min(L, total - s)
        out.append(L)
        s += L
    return out


def workload(name: str, seed: int = 0) -> Workload:
    """The named workloads, shaped like the models the page walks through."""
    if name == "tiny_linear":      # ELU+1 linear attention, fp32, one sequence
        return Workload(name, "prefill_linear", 1, 64, 64, torch.float32, lengths=(256,))
    if name == "tiny_delta":       # delta rule, k L2-normalised, alpha = 1, fp32
        return Workload(name, "prefill_delta", 1, 64, 64, torch.float32, lengths=(256,))
    if name == "gpt2_prefill":     # GPT-2-small-shaped: 12 heads of 64, 8 x 2048 tokens
        return Workload(name, "prefill_delta", 12, 64, 64, torch.bfloat16, lengths=(2048,) * 8)
    if name == "gpt2_scalar_gate":  # the GPT-2 shape with one decay per token and head
        return Workload(name, "prefill_delta", 12, 64, 64, torch.bfloat16, gated=True,
                        lengths=(2048,) * 8, extra={"scalar_gate": True})
    if name == "gpt2_chunk128":    # the GPT-2 shape with the recurrence over 128-token chunks
        return Workload(name, "prefill_delta", 12, 64, 64, torch.bfloat16, lengths=(2048,) * 8,
                        extra={"chunk": 128})
    if name == "gated_prefill":    # per-channel decay, 32 heads of 128, 4 x 8192 tokens
        return Workload(name, "prefill_delta", 32, 128, 128, torch.bfloat16, gated=True,
                        lengths=(8192,) * 4)
    if name == "decode":           # 256 sequences x 32 heads, 128x128 fp32 state, 64 steps
        return Workload(name, "decode", 32, 128, 128, torch.bfloat16, gated=True,
                        n_seq=256, steps=64)
    if name == "varlen_prefill":   # 65536 packed tokens, lengths uniform in [1024, 16384]
        lens = varlen_lengths(65536, 1024, 16384, seed)
        return Workload(name, "prefill_delta", 16, 128, 128, torch.bfloat16, gated=True,
                        lengths=tuple(lens), varlen=(65536, 1024, 16384))
    raise KeyError(name)


ALL_WORKLOADS = ("tiny_linear", "tiny_delta", "gpt2_prefill", "gated_prefill", "decode",
                 "varlen_prefill", "gpt2_scalar_gate", "gpt2_chunk128")


def cu_seqlens(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def _randn(g, shape, dtype, mean=0.0, std=1.0):
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(dtype)


def prefill_inputs(lengths, H, dk, dv, dtype, gated, seed=0, init_state=False,
                   gate_mean=2.0, scalar_gate=False):
    """Raw prefill inputs on the CPU: q, k, v, beta/gate logits, optional state.
    scalar_gate: one gate logit per token and head ([ntok][H]) instead of one
    per key channel."""
    g = torch.Generator().manual_seed(seed)
    ntok = int(sum(lengths))
    out = {
        "q": _randn(g, (ntok, H, dk), dtype),
        "k": _randn(g, (ntok, H, dk), dtype),
        "v": _randn(g, (ntok, H, dv), dtype),
        "beta_logits": _randn(g, (ntok, H), dtype),
        "gate_logits": (_randn(g, (ntok, H) if scalar_gate else (ntok, H, dk), dtype,
                               mean=gate_mean) if gated else None),
        "cu_seqlens": cu_seqlens(lengths),
    }
    out["init_S"] = (_randn(g, (len(lengths), H, dk, dv), torch.float32, std=0.02)
                     if init_state else None)
    return out


def decode_inputs(n_seq, H, dk, dv, steps, dtype, seed=0, gated=True, gate_mean=2.0,
                  scalar_gate=False):
    """Raw decode inputs: ``steps`` tokens per sequence and the pre-filled state
    (scalar_gate: gate logits [steps][n_seq][H])."""
    g = torch.Generator().manual_seed(seed)
    return {
        "q": _randn(g, (steps, n_seq, H, dk), dtype),
        "k": _randn(g, (steps, n_seq, H, dk), dtype),
        "v": _randn(g, (steps, n_seq, H, dv), dtype),
        "beta_logits": _randn(g, (steps, n_seq, H), dtype),
        "gate_logits": (_randn(g, (steps, n_seq, H) if scalar_gate else (steps, n_seq, H, dk),
                               dtype, mean=gate_mean) if gated else None),
        "state": _randn(g, (n_seq, H, dk, dv), torch.float32, std=0.02),
    }


def inputs_for(w: Workload, seed=0, init_state=False):
    if w.kind == "decode":
        return decode_inputs(w.n_seq, w.H, w.dk, w.dv, w.steps, w.dtype, seed, gated=w.gated)
    return prefill_inputs(w.lengths, w.H, w.dk, w.dv, w.dtype, w.gated, seed,
                          init_state=init_state, scalar_gate=w.extra.get("scalar_gate", False))


def shard_sequences(inp: dict, rank: int, world: int) -> tuple[dict, list[int]]:
    """Rank `rank`'s share of one packed prefill batch across `world` ranks:
    sequences rank, rank + world, ... with their tokens, states and a fresh
    cu_seqlens (the delta rule and ELU+1 treat every sequence on its own, so
    no rank needs another's data).  Also returns the global indices of the
    sequences taken, for putting the outputs back with gather_sequences."""
    cu = [int(x) for x in inp["cu_seqlens"]]
    n_seq = len(cu) - 1
    mine = list(range(rank, n_seq, world))
    rows = [torch.arange(cu[n], cu[n + 1]) for n in mine]
    idx = torch.cat(rows) if rows else torch.zeros(0, dtype=torch.long)
    out = {}
    for name, t in inp.items():
        if name == "cu_seqlens":
            out[name] = cu_seqlens([cu[n + 1] - cu[n] for n in mine])
        elif t is None:
            out[name] = None
        elif name in ("init_S", "state"):
            out[name] = t[mine]
        else:
            out[name] = t[idx]
    return out, mine


def gather_sequences(shards: list[tuple[torch.Tensor, list[int]]], cu_full) -> torch.Tensor:
    """Per-token outputs of every rank's shard (tensor [tokens of its
    sequences, ...], global sequence indices) back in the packed order of
    the full batch."""
    cu = [int(x) for x in cu_full]
    first = shards[0][0]
    full = torch.empty((cu[-1],) + tuple(first.shape[1:]), dtype=first.dtype)
    for part, seqs in shards:
        at = 0
        for n in seqs:
            L = cu[n + 1] - cu[n]
            full[cu[n]:cu[n + 1]] = part[at:at + L]
            at += L
    return full
