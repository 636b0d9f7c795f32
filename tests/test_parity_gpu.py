"""GPU parity: every C-ABI entry point against the fp64 oracle on the same
seeded inputs.  Metric: max|GPU - oracle| / max|oracle|, over outputs and,
separately, over final states; bar 1e-4 for fp32 I/O and 2e-2 for bf16 I/O
(fp32 state in both).  Small cases compare every element and cover ragged
tails (lengths 1, 63, 64, 65, 130), empty sequences and every head size;
full-size workloads compare every (sequence, head) the oracle can afford and
sampled heads where it cannot."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from _helpers import TOL, f64, gpu_prefill_delta, oracle_prefill_delta, rel_err

pytestmark = pytest.mark.gpu

RAGGED = [1, 63, 64, 65, 130, 0, 7]


# ------------------------------------------------------------- delta prefill

def check_delta(la, inp, dtype, heads=None, flags=oracle.L2NORM_K, scale=1.0):
    o, fS = gpu_prefill_delta(la, inp, flags=flags, scale=scale)
    ref_o, ref_S = oracle_prefill_delta(inp, heads=heads, flags=flags, scale=scale)
    if heads is not None:
        o, fS = o[:, heads], fS[:, heads]
    eo, es = rel_err(o.numpy(), ref_o), rel_err(fS.numpy(), ref_S)
    assert eo <= TOL[dtype], f"output rel err {eo:.3e}"
    assert es <= TOL[dtype], f"final state rel err {es:.3e}"
    return eo, es


def test_tiny_delta_fp32(cuda_lib):
    w = wl.workload("tiny_delta")
    check_delta(cuda_lib, wl.inputs_for(w, seed=0), torch.float32)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("gated", [False, True])
def test_delta_ragged_fp32(cuda_lib, dk, dv, gated):
    inp = wl.prefill_inputs(RAGGED, 2, dk, dv, torch.float32, gated, seed=dk + dv + gated,
                            init_state=True)
    check_delta(cuda_lib, inp, torch.float32)


@pytest.mark.parametrize("flags", [0, oracle.L2NORM_K | oracle.L2NORM_Q,
                                   oracle.L2NORM_K | oracle.L2NORM_Q | oracle.SILU_QK])
def test_delta_prologue_flags_fp32(cuda_lib, flags):
    inp = wl.prefill_inputs([70, 33], 2, 64, 64, torch.float32, True, seed=3)
    if flags == 0:  # unnormalised keys: keep the recurrence contractive
        inp["k"] = inp["k"] * 0.1
    check_delta(cuda_lib, inp, torch.float32, flags=flags, scale=0.5)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128)])
def test_delta_ragged_bf16(cuda_lib, dk, dv):
    inp = wl.prefill_inputs([200, 77, 1, 0, 128], 3, dk, dv, torch.bfloat16, True, seed=11,
                            init_state=True)
    check_delta(cuda_lib, inp, torch.bfloat16)


@pytest.mark.parametrize("flags", [oracle.L2NORM_K, oracle.L2NORM_K | oracle.ADDITIVE])
def test_delta_ragged_bf16_d64_ungated(cuda_lib, flags):
    """d = 64 without a per-channel gate: the one-launch path that runs the
    intra-chunk tasks and the recurrence together (ragged lengths, an empty
    sequence, initial states, with and without the delta term)."""
    inp = wl.prefill_inputs(RAGGED, 3, 64, 64, torch.bfloat16, False, seed=12, init_state=True)
    check_delta(cuda_lib, inp, torch.bfloat16, flags=flags)


def test_delta_bf16_d64_many_chains(cuda_lib):
    """160 (sequence, head) chains, more than half the resident grid: the
    same configuration takes the two-launch path."""
    lens = [70, 1, 129, 64] * 10
    inp = wl.prefill_inputs(lens, 4, 64, 64, torch.bfloat16, False, seed=13, init_state=True)
    check_delta(cuda_lib, inp, torch.bfloat16, heads=[0, 3])


def test_delta_resume_matches_single_pass(cuda_lib):
    la = cuda_lib
    T, t1 = 300, 131
    inp = wl.prefill_inputs([T], 2, 128, 128, torch.float32, True, seed=5, init_state=True)
    full_o, full_S = gpu_prefill_delta(la, inp)
    part1 = {n: (None if inp[n] is None else inp[n][:t1]) for n in
             ("q", "k", "v", "beta_logits", "gate_logits")}
    part1.update(cu_seqlens=torch.tensor([0, t1], dtype=torch.int32), init_S=inp["init_S"])
    o1, S1 = gpu_prefill_delta(la, part1)
    part2 = {n: (None if inp[n] is None else inp[n][t1:]) for n in
             ("q", "k", "v", "beta_logits", "gate_logits")}
    part2.update(cu_seqlens=torch.tensor([0, T - t1], dtype=torch.int32), init_S=S1)
    o2, S2 = gpu_prefill_delta(la, part2)
    assert rel_err(torch.cat([o1, o2]).numpy(), full_o.numpy()) <= 1e-5
    assert rel_err(S2.numpy(), full_S.numpy()) <= 1e-5


def test_gpt2_prefill_full(cuda_lib):
    """Full-size GPT-2-shaped workload (8 x 2048 tokens, 12 heads of 64), every head."""
    w = wl.workload("gpt2_prefill")
    check_delta(cuda_lib, wl.inputs_for(w, seed=0), torch.bfloat16)


def test_gated_prefill_full_sampled_heads(cuda_lib):
    """Full-size gated workload (4 x 8192 tokens, 32 heads of 128); the oracle
    runs on 3 of the 32 heads for all four sequences."""
    w = wl.workload("gated_prefill")
    check_delta(cuda_lib, wl.inputs_for(w, seed=0), torch.bfloat16, heads=[0, 17, 31])


def test_varlen_prefill_full_sampled_heads(cuda_lib):
    """65536 packed tokens with seeded lengths in [1024, 16384]; final states compared."""
    w = wl.workload("varlen_prefill", seed=0)
    assert sum(w.lengths) == 65536 and len(w.lengths) > 1
    check_delta(cuda_lib, wl.inputs_for(w, seed=0), torch.bfloat16, heads=[0, 9, 15])


# ------------------------------------------------------------ ELU+1 linear

def check_linear(la, inp, dtype, init=False, host_cu=True):
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    cu = inp["cu_seqlens"]
    N, H, dk, dv = cu.numel() - 1, q.shape[1], q.shape[2], v.shape[2]
    g = torch.Generator().manual_seed(99)
    iS = torch.rand((N, H, dk, dv), generator=g) if init else None
    iz = torch.rand((N, H, dk), generator=g) + 1.0 if init else None
    o = torch.full((q.shape[0], H, dv), float("nan"), dtype=q.dtype, device=dev)
    fS = torch.full((N, H, dk, dv), float("nan"), device=dev)
    fz = torch.full((N, H, dk), float("nan"), device=dev)
    la.la_prefill_linear(q, k, v, o, cu.to(dev), init_S=None if iS is None else iS.to(dev),
                         init_z=None if iz is None else iz.to(dev), final_S=fS, final_z=fz,
                         cu_seqlens_host=cu if host_cu else None)
    assert la.la_check_device() == la.LA_OK
    ro, rS, rz = oracle.linear(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), cu.numpy(),
                               init_S=f64(iS), init_z=f64(iz))
    tol = TOL[dtype]
    assert rel_err(o.float().cpu().numpy(), ro) <= tol
    assert rel_err(fS.cpu().numpy(), rS) <= tol
    assert rel_err(fz.cpu().numpy(), rz) <= tol


def test_tiny_linear_fp32(cuda_lib):
    w = wl.workload("tiny_linear")
    check_linear(cuda_lib, wl.inputs_for(w, seed=0), torch.float32)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_linear_ragged_fp32(cuda_lib, dk, dv):
    inp = wl.prefill_inputs(RAGGED, 2, dk, dv, torch.float32, False, seed=21)
    check_linear(cuda_lib, inp, torch.float32, init=True)


def test_linear_bf16(cuda_lib):
    inp = wl.prefill_inputs([300, 64, 5], 4, 64, 64, torch.bfloat16, False, seed=22)
    check_linear(cuda_lib, inp, torch.bfloat16)


# Sequences of at most 8 chunks (512 tokens) take the chunk-parallel kernel,
# longer ones the chunk-by-chunk scan: both, and the boundary between them.
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128)])
def test_linear_long_sequences_fp32(cuda_lib, dk, dv):
    inp = wl.prefill_inputs([700, 513, 64, 0], 2, dk, dv, torch.float32, False, seed=23)
    check_linear(cuda_lib, inp, torch.float32, init=True)


def test_linear_long_sequences_bf16(cuda_lib):
    inp = wl.prefill_inputs([600, 200], 3, 64, 128, torch.bfloat16, False, seed=24)
    check_linear(cuda_lib, inp, torch.bfloat16, init=True)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64)])
def test_linear_eight_chunk_boundary(cuda_lib, dk, dv):
    inp = wl.prefill_inputs([512, 511, 1, 0, 448], 2, dk, dv, torch.float32, False, seed=25)
    check_linear(cuda_lib, inp, torch.float32, init=True)


def test_linear_tensor_core_ragged(cuda_lib):
    """bf16, dk = dv = 64, sequences past 8 chunks: the tensor-core kernel
    (ragged tails, a 1-token and an empty sequence, initial states)."""
    inp = wl.prefill_inputs([700, 129, 64, 1, 0, 513], 3, 64, 64, torch.bfloat16, False, seed=27)
    check_linear(cuda_lib, inp, torch.bfloat16, init=True)
    check_linear(cuda_lib, inp, torch.bfloat16, init=False, host_cu=False)


def test_linear_tensor_core_gpt2_shape(cuda_lib):
    """The GPT-2 shape (8 x 2048 tokens, 12 heads of 64) in bf16, every head."""
    inp = wl.prefill_inputs((2048,) * 8, 12, 64, 64, torch.bfloat16, False, seed=28)
    check_linear(cuda_lib, inp, torch.bfloat16)


@pytest.mark.parametrize("lengths", [[200, 0, 57], [400, 300]])
def test_linear_without_host_cu_seqlens(cuda_lib, lengths):
    """No host copy of cu_seqlens: a packed total of at most 512 tokens
    still takes the chunk-parallel kernel, a larger one the scan."""
    inp = wl.prefill_inputs(lengths, 2, 64, 64, torch.float32, False, seed=26)
    check_linear(cuda_lib, inp, torch.float32, init=True, host_cu=False)


# ------------------------------------------------------------------ decode

def run_decode(la, inp, steps, scale=1.0, flags=1, gated=True):
    dev = torch.device("cuda")
    st = inp["state"].clone().to(dev)
    outs = []
    for t in range(steps):
        q, k, v, bl = (inp[n][t].to(dev) for n in ("q", "k", "v", "beta_logits"))
        gl = inp["gate_logits"][t].to(dev) if gated else None
        o = torch.full(v.shape, float("nan"), dtype=v.dtype, device=dev)
        la.la_decode_step(q, k, v, bl, gl, o, st, scale=scale, flags=flags)
        outs.append(o.float().cpu())
    assert la.la_check_device() == la.LA_OK
    return torch.stack(outs), st.cpu()


def oracle_decode(inp, steps, pairs=None, scale=1.0, flags=1, gated=True):
    sel = (lambda t: t) if pairs is None else (lambda t: t[:, pairs[0], pairs[1]][:, :, None])
    st = inp["state"] if pairs is None else inp["state"][pairs[0], pairs[1]][:, None]
    st = f64(st)
    outs = []
    for t in range(steps):
        g = f64(sel(inp["gate_logits"])[t]) if gated else None
        o, st = oracle.decode(f64(sel(inp["q"])[t]), f64(sel(inp["k"])[t]), f64(sel(inp["v"])[t]),
                              f64(sel(inp["beta_logits"])[t]), g, st, scale=scale, flags=flags)
        outs.append(o)
    return np.stack(outs), st


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("gated", [False, True])
def test_decode_small(cuda_lib, dtype, dk, dv, gated):
    inp = wl.decode_inputs(5, 3, dk, dv, 4, dtype, seed=dk * 3 + dv + gated, gated=gated)
    o, st = run_decode(cuda_lib, inp, 4, scale=0.75, gated=gated)
    ro, rst = oracle_decode(inp, 4, scale=0.75, gated=gated)
    assert rel_err(o.numpy(), ro) <= TOL[dtype]
    assert rel_err(st.numpy(), rst) <= TOL[dtype]


def test_decode_flags(cuda_lib):
    flags = oracle.L2NORM_K | oracle.L2NORM_Q | oracle.SILU_QK
    inp = wl.decode_inputs(3, 2, 128, 128, 3, torch.float32, seed=4)
    o, st = run_decode(cuda_lib, inp, 3, flags=flags)
    ro, rst = oracle_decode(inp, 3, flags=flags)
    assert rel_err(o.numpy(), ro) <= 1e-4
    assert rel_err(st.numpy(), rst) <= 1e-4


def test_decode_full_sampled(cuda_lib):
    """Full decode workload: 256 sequences x 32 heads, 128x128 fp32 states, 64
    consecutive steps; the oracle follows 12 sampled (sequence, head) pairs."""
    w = wl.workload("decode")
    inp = wl.inputs_for(w, seed=0)
    o, st = run_decode(cuda_lib, inp, w.steps)
    rs = np.random.default_rng(0)
    pairs = (rs.integers(0, w.n_seq, 12), rs.integers(0, w.H, 12))
    ro, rst = oracle_decode(inp, w.steps, pairs=pairs)
    got_o = o[:, pairs[0], pairs[1]][:, :, None].numpy()
    got_st = st[pairs[0], pairs[1]][:, None].numpy()
    assert rel_err(got_o, ro) <= TOL[torch.bfloat16]
    assert rel_err(got_st, rst) <= TOL[torch.bfloat16]


# ------------------------------------------------- scalar gate (one decay per token and head)

@pytest.mark.parametrize("dtype,dk,dv", [(torch.float32, 64, 64), (torch.float32, 64, 128),
                                         (torch.float32, 128, 128), (torch.bfloat16, 64, 64),
                                         (torch.bfloat16, 128, 128)])
def test_delta_scalar_gate_ragged(cuda_lib, dtype, dk, dv):
    """LA_GATE_SCALAR: fp32 I/O on the CUDA-core kernel, bf16 (dk == dv) on the
    tensor-core kernels; ragged lengths, empty sequence, initial states."""
    inp = wl.prefill_inputs(RAGGED, 2, dk, dv, dtype, True, seed=40 + dk + dv, init_state=True,
                            scalar_gate=True)
    o, fS = gpu_prefill_delta(cuda_lib, inp, flags=cuda_lib.LA_L2NORM_K | cuda_lib.LA_GATE_SCALAR)
    ref_o, ref_S = oracle_prefill_delta(inp, flags=oracle.L2NORM_K | oracle.SCALAR_GATE)
    assert rel_err(o.numpy(), ref_o) <= TOL[dtype]
    assert rel_err(fS.numpy(), ref_S) <= TOL[dtype]


def test_gpt2_shape_scalar_gate_full(cuda_lib):
    """The GPT-2-shaped workload (8 x 2048 tokens, 12 heads of 64) with a
    scalar gate per token and head, every head against the oracle."""
    w = wl.workload("gpt2_prefill")
    inp = wl.prefill_inputs(w.lengths, w.H, w.dk, w.dv, w.dtype, True, seed=1, scalar_gate=True)
    o, fS = gpu_prefill_delta(cuda_lib, inp, flags=cuda_lib.LA_L2NORM_K | cuda_lib.LA_GATE_SCALAR)
    ref_o, ref_S = oracle_prefill_delta(inp, flags=oracle.L2NORM_K | oracle.SCALAR_GATE)
    assert rel_err(o.numpy(), ref_o) <= TOL[torch.bfloat16]
    assert rel_err(fS.numpy(), ref_S) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_scalar_gate(cuda_lib, dtype):
    inp = wl.decode_inputs(5, 3, 128, 128, 4, dtype, seed=41, scalar_gate=True)
    o, st = run_decode(cuda_lib, inp, 4, flags=cuda_lib.LA_L2NORM_K | cuda_lib.LA_GATE_SCALAR)
    ro, rst = oracle_decode(inp, 4, flags=oracle.L2NORM_K | oracle.SCALAR_GATE)
    assert rel_err(o.numpy(), ro) <= TOL[dtype]
    assert rel_err(st.numpy(), rst) <= TOL[dtype]
