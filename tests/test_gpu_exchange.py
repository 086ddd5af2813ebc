"""The per-rank kernels of the multi-GPU paths, on one GPU.

DCD-PSGD across ranks: dcd_step_rows steps a rank's own nodes beside copies
of its two ring neighbours and packs the C(z) of its first and last node;
dcd_copy_add adds a neighbour's C to a copy.  Here W ranks are emulated in
one process: every rank's rows live on the one GPU, each iteration steps all
of them, then hands each rank's lists to its neighbours' copies directly
(the transfer itself, torch.distributed send/recv, is covered on CPU by
tests/test_exchange.py).  After every iteration every row, own or copy, must
equal the oracle's single-process ring bit for bit.
"""
import numpy as np
import pytest

import oracle
from gradient_compression_sgd_gb300 import exchange

pytestmark = pytest.mark.gpu

RING_W = (0.25, 0.45, 0.3)


def ring_inputs(n, d, iters, seed):
    rng = np.random.default_rng(seed)
    x0 = (rng.standard_normal(d) * 1e-2).astype(np.float32)
    x0[::977] = -0.0  # a starting model with -0 entries: the copies' first update takes the zero pass
    grads = [(rng.standard_normal((n, d)) * 1e-3).astype(np.float32) for _ in range(iters)]
    return x0, grads


@pytest.mark.parametrize("n,world,p,d", [(8, 2, 0.01, 10001), (5, 3, 0.2, 4096), (2, 2, 0.5, 777), (8, 8, 0.05, 3),
                                         (7, 2, 1.0, 20000), (13, 4, 0.01, 65537)])
def test_dcd_rows_emulated_ranks(cuda_lib, n, world, p, d):
    import torch
    gc = cuda_lib
    iters, seed, gamma = 4, 1234, 0.1
    x0, grads = ring_inputs(n, d, iters, 40 + n)
    parts = [exchange.RingPartition(n, world, r) for r in range(world)]
    dev = torch.device("cuda")
    rings = [exchange.GpuRing(part, d, RING_W, gamma, p, seed, dev) for part in parts]
    local = [torch.from_numpy(np.tile(x0, (part.rows, 1))).to(dev) for part in parts]
    x = np.ascontiguousarray(np.tile(x0, (n, 1)))
    for t in range(iters):
        sent = []
        for r, part in enumerate(parts):
            g_own = torch.from_numpy(np.ascontiguousarray(grads[t][part.a:part.b])).to(dev)
            first, last = rings[r].step(local[r], g_own, t)
            sent.append((first.clone(), last.clone()))
        for r, part in enumerate(parts):
            rings[r].copy_add(local[r][0], sent[part.left_rank][1])
            rings[r].copy_add(local[r][-1], sent[part.right_rank][0])
        oracle.dcd_step(x, grads[t], RING_W, gamma, p, seed, t)
        torch.cuda.synchronize()
        for r, part in enumerate(parts):
            got = local[r].cpu().numpy()
            for row, node in enumerate(part.row_nodes()):
                np.testing.assert_array_equal(got[row].view(np.uint32), x[node].view(np.uint32),
                                              err_msg=f"iteration {t}, rank {r}, row {row} (node {node})")


def test_dcd_rows_lists_are_the_kept_entries(cuda_lib):
    """The packed lists hold every kept entry exactly once; scattered into
    zeros they are the oracle's C of the first and last own node."""
    import torch
    gc = cuda_lib
    rng = np.random.default_rng(3)
    rows, d, first_node, p = 5, 20003, 4, 0.05
    xr = (rng.standard_normal((rows, d)) * 1e-2).astype(np.float32)
    g = (rng.standard_normal((rows - 2, d)) * 1e-3).astype(np.float32)
    xg = torch.from_numpy(xr).cuda()
    cf = torch.zeros((d, 2), dtype=torch.int32, device="cuda")
    cl = torch.zeros((d, 2), dtype=torch.int32, device="cuda")
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    gc.dcd_step_rows(xg, torch.from_numpy(g).cuda(), RING_W, 0.1, p, 99, 7, first_node, cf, cl, counts)
    c_first, c_last = oracle.dcd_step_rows(xr, g, RING_W, 0.1, p, 99, 7, first_node)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(xg.cpu().numpy(), xr)
    thr = oracle.keep_threshold(p)
    for lst, cnt, want, node in ((cf, counts[0], c_first, first_node), (cl, counts[1], c_last, first_node + rows - 3)):
        m = int(cnt)
        a = lst[:m].cpu().numpy()
        idx = a[:, 0].view(np.uint32).astype(np.int64)
        assert len(np.unique(idx)) == m
        kept = np.zeros(d, bool)  # the keep draw, word e % 4 of Philox at counter (e / 4, node, t, 0)
        for q in range((d + 3) // 4):
            words = oracle.philox4x32_10([q, node, 7, 0], [99, 0])
            for j in range(min(4, d - 4 * q)):
                kept[4 * q + j] = words[j] < thr
        np.testing.assert_array_equal(np.sort(idx), np.nonzero(kept)[0])
        dense = np.zeros(d, np.float32)
        dense[idx] = a[:, 1].view(np.float32)
        np.testing.assert_array_equal(dense.view(np.uint32), want.view(np.uint32))


def test_dcd_rows_counts_past_capacity(cuda_lib):
    """A list smaller than the kept count: the count is still exact, nothing is
    written past the capacity (a guard record after it stays untouched)."""
    import torch
    gc = cuda_lib
    rng = np.random.default_rng(4)
    rows, d, cap = 3, 4096, 100
    xr = torch.from_numpy((rng.standard_normal((rows, d)) * 1e-2).astype(np.float32)).cuda()
    g = torch.from_numpy((rng.standard_normal((1, d)) * 1e-3).astype(np.float32)).cuda()
    buf = torch.full((2, cap + 1, 2), 7, dtype=torch.int32, device="cuda")
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    gc.dcd_step_rows(xr, g, RING_W, 0.1, 0.5, 5, 0, 0, buf[0, :cap], buf[1, :cap], counts)
    torch.cuda.synchronize()
    assert int(counts[0]) == int(counts[1]) > cap  # one own node: both lists are its C
    assert (buf[:, cap] == 7).all()
