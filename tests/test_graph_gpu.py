"""The library's calls inside CUDA graphs: each entry point is captured once
(after one uncaptured call, which resolves the library's per-device lookups
outside the capture), the graph is replayed on new values written into the
captured input tensors, and its outputs must equal, bit for bit, those of the
same calls made without a graph on the new values.  (The library neither
allocates nor synchronises inside its calls, and its launches take the
caller's stream, so a capture records exactly the kernels a call launches.)"""
import pytest
import torch

import workloads as wl
from test_backward_gpu import RAGGED

pytestmark = pytest.mark.gpu

PREFILL = ("q", "k", "v", "beta_logits", "gate_logits", "init_S")


def _refill(dst, src):
    for n, t in dst.items():
        if t is not None:
            t.copy_(src[n])


def _capture(fn):
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()                                   # outside the capture first
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("d,gate", [(64, False), (128, True)])
def test_prefill_graph_replay(cuda_lib, d, gate):
    la = cuda_lib
    dev = torch.device("cuda")
    a = wl.prefill_inputs(RAGGED, 2, d, d, torch.bfloat16, gate, seed=110, init_state=True)
    b = wl.prefill_inputs(RAGGED, 2, d, d, torch.bfloat16, gate, seed=111, init_state=True)
    t = {n: (None if a[n] is None else a[n].to(dev)) for n in PREFILL}
    cu = a["cu_seqlens"].to(dev)
    N, H = cu.numel() - 1, t["q"].shape[1]
    o = torch.empty_like(t["v"])
    fS = torch.empty((N, H, d, d), device=dev)
    ws = torch.empty(la.la_prefill_delta_workspace_size(N, t["q"].shape[0], H, d, d, 64, la.LA_BF16),
                     dtype=torch.uint8, device=dev)

    def call():
        la.la_prefill_delta(t["q"], t["k"], t["v"], t["beta_logits"], t["gate_logits"], o, cu,
                            init_S=t["init_S"], final_S=fS, workspace=ws,
                            cu_seqlens_host=a["cu_seqlens"])

    g = _capture(call)
    _refill(t, {n: (None if b[n] is None else b[n].to(dev)) for n in PREFILL})
    g.replay()
    torch.cuda.synchronize()
    assert la.la_check_device() == la.LA_OK
    o_graph, fs_graph = o.clone(), fS.clone()
    o.fill_(7.0)
    call()
    assert la.la_check_device() == la.LA_OK
    assert torch.equal(o_graph, o)
    assert torch.equal(fs_graph, fS)


def test_decode_64_steps_in_one_graph(cuda_lib):
    """64 consecutive decode steps captured as one graph (the decode
    workload's form), replayed from a new state on new tokens."""
    la = cuda_lib
    dev = torch.device("cuda")
    steps, N, H, d = 64, 8, 4, 128
    a = wl.decode_inputs(N, H, d, d, steps, torch.bfloat16, seed=112)
    b = wl.decode_inputs(N, H, d, d, steps, torch.bfloat16, seed=113)
    names = ("q", "k", "v", "beta_logits", "gate_logits")
    t = {n: a[n].to(dev) for n in names}
    state = a["state"].to(dev)
    o = torch.empty((steps, N, H, d), dtype=torch.bfloat16, device=dev)

    def run():
        for s in range(steps):
            la.la_decode_step(t["q"][s], t["k"][s], t["v"][s], t["beta_logits"][s],
                              t["gate_logits"][s], o[s], state)

    g = _capture(run)
    _refill(t, {n: b[n].to(dev) for n in names})
    state.copy_(b["state"])
    g.replay()
    torch.cuda.synchronize()
    assert la.la_check_device() == la.LA_OK
    o_graph, state_graph = o.clone(), state.clone()
    state.copy_(b["state"])
    o.fill_(7.0)
    run()
    assert la.la_check_device() == la.LA_OK
    assert torch.equal(o_graph, o)
    assert torch.equal(state_graph, state)


def test_training_pair_graph_replay(cuda_lib):
    """la_prefill_delta_train then la_backward_delta_saved in one graph
    (gated, d = 128).  The per-chunk gradient kernel adds some partial sums
    with shared-memory atomics, so the gradients are compared to the last
    bits' spread rather than bit for bit; o and the final states exactly."""
    la = cuda_lib
    dev = torch.device("cuda")
    d = 128
    a = wl.prefill_inputs(RAGGED, 2, d, d, torch.bfloat16, True, seed=114, init_state=True)
    b = wl.prefill_inputs(RAGGED, 2, d, d, torch.bfloat16, True, seed=115, init_state=True)
    t = {n: a[n].to(dev) for n in PREFILL}
    cu = a["cu_seqlens"].to(dev)
    ntok, H = t["q"].shape[:2]
    N = cu.numel() - 1
    gen = torch.Generator().manual_seed(116)
    d_o = torch.randn((ntok, H, d), generator=gen).to(torch.bfloat16).to(dev)
    saved = torch.empty(la.la_backward_delta_workspace_size(N, ntok, H, d, d), dtype=torch.uint8,
                        device=dev)
    o = torch.empty_like(t["v"])
    fS = torch.empty((N, H, d, d), device=dev)
    grads = {n: torch.empty(t[x].shape, device=dev) for n, x in
             (("dq", "q"), ("dk", "k"), ("dv", "v"), ("db", "beta_logits"), ("dg", "gate_logits"),
              ("di", "init_S"))}
    lib = la.library()
    import ctypes
    p = lambda x: ctypes.c_void_p(x.data_ptr())

    def step():
        la.la_prefill_delta_train(t["q"], t["k"], t["v"], t["beta_logits"], t["gate_logits"], o,
                                  cu, saved, init_S=t["init_S"], final_S=fS,
                                  cu_seqlens_host=a["cu_seqlens"])
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = lib.la_backward_delta_saved(p(t["q"]), p(t["k"]), p(t["v"]), p(t["beta_logits"]),
                                         p(t["gate_logits"]), p(d_o), None, la.LA_BF16, p(cu),
                                         None, N, ntok, H, d, d, 1.0, la.LA_L2NORM_K,
                                         p(t["init_S"]), p(grads["dq"]), p(grads["dk"]),
                                         p(grads["dv"]), p(grads["db"]), p(grads["dg"]),
                                         p(grads["di"]), p(saved), saved.numel(), s)
        assert rc == la.LA_OK

    g = _capture(step)
    _refill(t, {n: b[n].to(dev) for n in PREFILL})
    g.replay()
    torch.cuda.synchronize()
    assert la.la_check_device() == la.LA_OK
    first = {n: x.clone() for n, x in grads.items()}
    o_graph, fs_graph = o.clone(), fS.clone()
    for x in grads.values():
        x.fill_(7.0)
    step()
    assert la.la_check_device() == la.LA_OK
    assert torch.equal(o_graph, o)
    assert torch.equal(fs_graph, fS)
    for n, x in grads.items():
        den = float(x.abs().max())
        assert float((first[n] - x).abs().max()) <= 1e-5 * max(den, 1e-30), n
