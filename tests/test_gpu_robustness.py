"""Robustness of the CUDA path: nothing is written past a buffer the caller
passed (canary words after every output and state buffer), a learner that
drops out of a step leaves an average of the others equal to the oracle's,
AdaComp's state is the caller's residue (save, restore, resume bit for
bit), and a whole step replays from a CUDA graph.  No test here faults or
hangs a GPU: a failure is made on the host.
"""
import numpy as np
import pytest

import oracle
from conftest import rel_err
from gradient_compression_sgd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CANARY = 0x5A5AA5A5  # int32 bit pattern written after every buffer
PAD = 64             # canary words (or pairs) after each buffer


def guarded(shape, dtype, fill=0):
    """A tensor of `shape` at the start of a larger allocation whose tail
    holds PAD canary elements; returns (view, whole)."""
    import torch
    n = int(np.prod(shape))
    whole = torch.full((n + PAD,), fill, dtype=dtype, device="cuda")
    whole[n:].view(torch.int32 if dtype in (torch.int32, torch.float32) else dtype).fill_(CANARY)
    return whole[:n].view(shape), whole


def guarded_pairs(K, cap):
    import torch
    whole = torch.zeros(((K * cap + PAD) * 2,), dtype=torch.int32, device="cuda")
    whole[K * cap * 2:] = CANARY
    return whole[:K * cap * 2].view(K, cap, 2), whole


def canary_intact(whole, n_elems):
    import torch
    tail = whole[n_elems:]
    bits = tail.view(torch.int32) if tail.dtype in (torch.int32, torch.float32) else tail
    return bool(torch.all(bits == CANARY).item())


def guarded_workspace(nbytes):
    """Scratch bytes followed by 4096 bytes of 0xA5."""
    import torch
    whole = torch.full((nbytes + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    return whole[:nbytes], whole


def workspace_intact(whole, nbytes):
    import torch
    return bool(torch.all(whole[nbytes:] == 0xA5).item())


@pytest.mark.parametrize("nesterov", [False, True])
def test_dgc_writes_nothing_past_its_buffers(cuda_lib, nesterov):
    """Ragged layout with empty, tiny, raw and pool segments, K = 3, clipping
    on: out, counts, totals, u, v and the workspace keep their canaries, and
    the result still equals the oracle's."""
    import torch
    gc = cuda_lib
    sizes = [0, 7, 1, 33, 70001, 0, 4097, 50001, 3]
    off = wl.layout_offsets(sizes)
    K, N, S = 3, int(off[-1]), len(sizes)
    density, m = 0.01, 0.9
    cap = sum(gc.dgc_k(density, s) for s in sizes)
    rng = np.random.default_rng(21)
    G = rng.standard_normal((K, N)).astype(np.float32) * 1e-2
    out, out_w = guarded_pairs(K, cap)
    counts, counts_w = guarded((K, S), torch.int64)
    totals, totals_w = guarded((K,), torch.int64)
    u, u_w = guarded((K, N), torch.float32)
    v, v_w = guarded((K, N), torch.float32)
    ws_n = gc.dgc_workspace_size(off, K, density)
    ws, ws_w = guarded_workspace(ws_n)
    u_o = np.zeros((K, N), np.float32)
    v_o = np.zeros((K, N), np.float32)
    for t in range(2):
        gc.dgc_compress(off, torch.from_numpy(G * (t + 1)).cuda(), u, v, out, counts, ws, density, m, 0.5, 2,
                        totals=totals, nesterov=nesterov)
        torch.cuda.synchronize()
        idx_o, val_o, counts_o, _ = oracle.dgc_step(off, G * (t + 1), u_o, v_o, density, m, 0.5, 2, cap=cap,
                                                    nesterov=nesterov)
        np.testing.assert_array_equal(counts.cpu().numpy(), counts_o)
        np.testing.assert_array_equal(gc.pair_indices(out).cpu().numpy(), idx_o.astype(np.int64))
        assert rel_err(u.cpu().numpy(), u_o) <= 1e-6 and rel_err(v.cpu().numpy(), v_o) <= 1e-6
    assert canary_intact(out_w, K * cap * 2)
    assert canary_intact(counts_w, K * S) and canary_intact(totals_w, K)
    assert canary_intact(u_w, K * N) and canary_intact(v_w, K * N)
    assert workspace_intact(ws_w, ws_n)


def test_adacomp_writes_nothing_past_its_buffers(cuda_lib):
    """Warp-chunk, tile and big-bin lengths on a ragged layout, K = 3: out,
    counts, scales, totals, the residue and the workspace keep their
    canaries, and the result equals the oracle's."""
    import torch
    gc = cuda_lib
    sizes = [7, 50001, 0, 13, 4097, 99999]
    lt = [2, 50, 7, 5, 700, 7000]
    off = wl.layout_offsets(sizes)
    K, N, S = 3, int(off[-1]), len(sizes)
    cap = N
    rng = np.random.default_rng(22)
    out, out_w = guarded_pairs(K, cap)
    counts, counts_w = guarded((K, S), torch.int64)
    scales, scales_w = guarded((K, S), torch.float32)
    totals, totals_w = guarded((K,), torch.int64)
    R, R_w = guarded((K, N), torch.float32)
    ws_n = gc.adacomp_workspace_size(off, lt, K, cap)
    ws, ws_w = guarded_workspace(ws_n)
    R_o = np.zeros((K, N), np.float32)
    for t in range(2):
        dW = rng.laplace(0, 1e-2, size=(K, N)).astype(np.float32)
        gc.adacomp_compress(off, lt, torch.from_numpy(dW).cuda(), R, out, counts, scales, totals, ws)
        torch.cuda.synchronize()
        idx_o, val_o, counts_o, scales_o, totals_o = oracle.adacomp_step(off, lt, dW, R_o, cap=cap)
        np.testing.assert_array_equal(counts.cpu().numpy(), counts_o)
        np.testing.assert_array_equal(totals.cpu().numpy(), totals_o)
        idx_g = gc.pair_indices(out).cpu().numpy()
        for k in range(K):
            n = int(totals_o[k])
            np.testing.assert_array_equal(idx_g[k, :n], idx_o[k, :n].astype(np.int64))
        assert rel_err(scales.cpu().numpy(), scales_o) <= 1e-6
    assert canary_intact(out_w, K * cap * 2)
    assert canary_intact(counts_w, K * S) and canary_intact(scales_w, K * S) and canary_intact(totals_w, K)
    assert canary_intact(R_w, K * N)
    assert workspace_intact(ws_w, ws_n)


def test_average_without_a_dropped_learner(cuda_lib):
    """A learner that fails this step (its message never arrives) is left out
    on the host: the average of the K - 1 others equals the oracle's."""
    import torch
    gc = cuda_lib
    w = wl.workload(2, small=True)
    K, N = w.learners, w.n
    d = gc.DGC(w.offsets, K, w.density, w.momentum)
    u = torch.zeros((K, N), device="cuda")
    v = torch.zeros((K, N), device="cuda")
    out, totals = d(wl.gradients(w, 0).cuda(), u, v)
    keep = [k for k in range(K) if k != 1]  # learner 1 dropped out
    lists = out[keep].contiguous()
    tot = totals[keep].contiguous()
    avg = torch.empty(N, device="cuda")
    gc.sparse_average(lists, tot, N, avg)
    torch.cuda.synchronize()
    want = oracle.sparse_average(gc.pair_indices(lists).cpu().numpy().astype(np.uint32),
                                 gc.pair_values(lists).cpu().numpy(), tot.cpu().numpy(), N)
    np.testing.assert_array_equal(avg.cpu().numpy(), want)


def test_adacomp_checkpoint_resume_is_bit_identical(cuda_lib):
    """AdaComp's state is the caller's residue: 3 steps straight equal 1 step,
    a save/restore of R through host memory, then 2 more steps."""
    import torch
    gc = cuda_lib
    w = wl.workload(3, small=True)
    K, N = w.learners, w.n
    dWs = [wl.gradients(w, t).cuda() for t in range(3)]
    a = gc.AdaComp(w.offsets, w.lt, K, N // 4)
    R = torch.zeros((K, N), device="cuda")
    outs = []
    for t in range(3):
        o, tot = a(dWs[t], R)
        outs.append((o.clone(), tot.clone()))
    a2 = gc.AdaComp(w.offsets, w.lt, K, N // 4)
    R2 = torch.zeros((K, N), device="cuda")
    a2(dWs[0], R2)
    R3 = R2.cpu().clone().cuda()
    for t in (1, 2):
        o, tot = a2(dWs[t], R3)
        assert torch.equal(tot, outs[t][1])
        for k in range(K):
            n = int(tot[k])
            assert torch.equal(o[k, :n], outs[t][0][k, :n])
    assert torch.equal(R3, R)


@pytest.mark.parametrize("method", ["dgc", "adacomp"])
def test_step_replays_from_a_cuda_graph(cuda_lib, method):
    """A whole step (compress + average) captured once into a CUDA graph and
    replayed: the library allocates nothing and never synchronises, so the
    replays give the same bits as eager calls from the same state."""
    import torch
    gc = cuda_lib
    w = wl.workload(2 if method == "dgc" else 3, small=True)
    K, N = w.learners, w.n
    grads = [wl.gradients(w, t).cuda() for t in range(3)]
    g_in = grads[0].clone()

    def make():
        if method == "dgc":
            obj = gc.DGC(w.offsets, K, w.density, w.momentum)
            state = [torch.zeros((K, N), device="cuda"), torch.zeros((K, N), device="cuda")]
        else:
            obj = gc.AdaComp(w.offsets, w.lt, K, N // 4)
            state = [torch.zeros((K, N), device="cuda")]
        return obj, state, torch.empty(N, device="cuda")

    def step(obj, state, g, avg):
        out, tot = obj(g, *state)
        gc.sparse_average(out, tot, N, avg)

    # eager reference
    obj_e, st_e, avg_e = make()
    ref = []
    for t in range(3):
        step(obj_e, st_e, grads[t], avg_e)
        ref.append((avg_e.clone(), [x.clone() for x in st_e]))
    torch.cuda.synchronize()
    # captured: warm up the library (first-call attributes) on a side stream, then capture
    obj_g, st_g, avg_g = make()
    scratch = [torch.zeros_like(x) for x in st_g]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(obj_g, scratch, g_in, avg_g)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(obj_g, st_g, g_in, avg_g)
    for x in st_g:
        x.zero_()
    for t in range(3):
        g_in.copy_(grads[t])
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(avg_g, ref[t][0])
        for a, b in zip(st_g, ref[t][1]):
            assert torch.equal(a, b)


def test_trace_events_captured_into_a_graph_time_its_replay(cuda_lib):
    """Tracing on while a step is captured: the traced kernel's two events
    become event nodes of the graph, and a read after a replay returns one
    launch of that kernel with a positive duration (the replay's)."""
    import torch
    gc = cuda_lib
    w = wl.workload(2, small=True)
    K, N = w.learners, w.n
    d = gc.DGC(w.offsets, K, w.density, w.momentum)
    u = torch.zeros((K, N), device="cuda")
    v = torch.zeros((K, N), device="cuda")
    g_in = wl.gradients(w, 0).cuda()
    s = torch.cuda.Stream()
    gc.trace_only("dgc_update")
    gc.trace_enable(True)
    try:
        with torch.cuda.stream(s):  # eager traced call: first-call attributes, events in the pool
            d(g_in, u, v)
        torch.cuda.synchronize()
        gc.trace_read()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            d(g_in, u, v)
        gc.trace_enable(False)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        tr = gc.trace_read()
    finally:
        gc.trace_enable(False)
        gc.trace_only(None)
    assert set(tr) == {"dgc_update"}
    n, ms = tr["dgc_update"]
    assert n == 1 and 0.0 < ms < 1000.0
