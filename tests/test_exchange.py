"""The exchange step across ranks, on CPU with gloo process groups.

K learners are split over 2 or 3 ranks; each rank steps its own learners
with the CPU oracle (DGC or AdaComp), then `exchange.exchange_average`
all-gathers the counts and the padded lists and averages them in global
learner order, with the oracle's sparse average as the averager.  Every rank
must end with the dense average a single process holding all K learners
computes, bit for bit, step after step ("Deep Gradient Compression",
Appendix A; "AdaComp", Proposed method).  Nothing here touches a GPU.
"""
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from gradient_compression_sgd_gb300 import exchange  # noqa: E402
from gradient_compression_sgd_gb300 import workloads as wl  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def oracle_average(lists, counts, n, out):
    """The oracle's sparse average over [K, cap, 2] int32 pair records."""
    import oracle
    a = lists.numpy()
    idx = a[..., 0].view(np.uint32)
    val = a[..., 1].view(np.float32)
    out.copy_(torch.from_numpy(oracle.sparse_average(idx, val, counts.numpy(), n)))


def to_pairs(idx, val, counts_per_learner):
    """Oracle (idx, val) arrays as a [K, cap, 2] int32 pair tensor."""
    K, cap = idx.shape
    rec = np.zeros((K, cap, 2), np.int32)
    rec[..., 0] = idx.view(np.int32)
    rec[..., 1] = val.view(np.int32)
    return torch.from_numpy(rec), torch.as_tensor(np.asarray(counts_per_learner, np.int64))


def case_inputs(method, K, steps):
    """Seeded gradients of a small mixed layout for every learner and step."""
    sizes = [300, 5000, 17, 4096, 20000]
    off = wl.layout_offsets(sizes)
    rng = np.random.default_rng(7 + K)
    grads = [(rng.standard_normal((K, off[-1])) * rng.choice([1e-3, 1e-1], size=(K, 1))).astype(np.float32)
             for _ in range(steps)]
    lt = [50, 4, 1, 500, 64] if method == "adacomp" else None
    return off, grads, lt


def run_learners(method, off, G, state, lt, cap):
    """One oracle step of the given learners: (pairs [K_r, cap, 2], totals [K_r])."""
    import oracle
    if method == "dgc":
        u, v = state
        idx, val, counts, _ = oracle.dgc_step(off, G, u, v, 0.01, 0.9, cap=cap)
        return to_pairs(idx, val, counts.sum(axis=1))
    (R,) = state
    idx, val, counts, _, totals = oracle.adacomp_step(off, lt, G, R, cap=cap)
    return to_pairs(idx, val, totals)


def _worker(rank, world, port, out_dir, method, K, steps):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        off, grads, lt = case_inputs(method, K, steps)
        N = int(off[-1])
        lo, hi = exchange.learner_range(K, world, rank)
        state = [np.zeros((hi - lo, N), np.float32) for _ in range(2 if method == "dgc" else 1)]
        cap = N
        res = []
        for t in range(steps):
            pairs, totals = run_learners(method, off, np.ascontiguousarray(grads[t][lo:hi]), state, lt, cap)
            out = torch.empty(N, dtype=torch.float32)
            lists_all, totals_all = exchange.exchange_average(pairs, totals, K, N, out, average=oracle_average)
            res.append({"avg": out.numpy().view(np.uint32).tolist(), "totals": totals_all.tolist(),
                        "cap_pad": int(lists_all.shape[1])})
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(res, f)
    finally:
        dist.destroy_process_group()


def single_process(method, K, steps):
    off, grads, lt = case_inputs(method, K, steps)
    N = int(off[-1])
    state = [np.zeros((K, N), np.float32) for _ in range(2 if method == "dgc" else 1)]
    want = []
    for t in range(steps):
        pairs, totals = run_learners(method, off, grads[t], state, lt, N)
        out = torch.empty(N, dtype=torch.float32)
        oracle_average(pairs, totals, N, out)
        want.append((out.numpy().view(np.uint32).tolist(), totals.tolist()))
    return want


@pytest.mark.parametrize("method,K,world", [("dgc", 4, 2), ("dgc", 5, 2), ("adacomp", 5, 3), ("adacomp", 2, 2)])
def test_exchange_average_equals_one_process(tmp_path, method, K, world):
    steps = 3
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path), method, K, steps), nprocs=world, join=True)
    want = single_process(method, K, steps)
    for r in range(world):
        got = json.load(open(tmp_path / f"rank{r}.json"))
        for t in range(steps):
            assert got[t]["totals"] == want[t][1], f"rank {r} step {t}: gathered counts"
            assert got[t]["avg"] == want[t][0], f"rank {r} step {t}: dense average differs"
            assert got[t]["cap_pad"] == max(1, max(want[t][1]))


def test_learner_range_partitions():
    for K in (1, 2, 5, 8, 13):
        for world in range(1, K + 1):
            spans = [exchange.learner_range(K, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == K
            assert all(spans[r][1] == spans[r + 1][0] for r in range(world - 1))
            sizes = [hi - lo for lo, hi in spans]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
    with pytest.raises(ValueError):
        exchange.learner_range(3, 2, 2)


# ------------------------------------------------------------ DCD-PSGD ring

RING_W = (0.25, 0.45, 0.3)  # asymmetric: a mirrored neighbour would show


def ring_inputs(n, d, iters):
    rng = np.random.default_rng(100 + n)
    x0 = (rng.standard_normal(d) * 1e-2).astype(np.float32)
    grads = [(rng.standard_normal((n, d)) * 1e-3).astype(np.float32) for _ in range(iters)]
    return x0, grads


def pack_nonzero(c):
    """Entries of a dense C whose bits are not +0, as [m, 2] int32 pair records."""
    bits = c.view(np.uint32)
    idx = np.nonzero(bits)[0].astype(np.uint32)
    rec = np.zeros((idx.size, 2), np.int32)
    rec[:, 0] = idx.view(np.int32)
    rec[:, 1] = bits[idx].view(np.int32)
    return torch.from_numpy(rec)


def add_pairs(row, pairs):
    """row + C, C the pairs' values at their indices and +0 elsewhere (what the
    owner added, entry by entry)."""
    c = np.zeros_like(row)
    a = pairs.numpy()
    c[a[:, 0].view(np.uint32)] = a[:, 1].view(np.float32)
    row[:] = row + c


def _ring_worker(rank, world, port, out_dir, n, d, iters, p, seed):
    import oracle
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        part = exchange.RingPartition(n, world, rank)
        x0, grads = ring_inputs(n, d, iters)
        local = np.ascontiguousarray(np.tile(x0, (part.rows, 1)))
        def step(xrows, g_own, t):
            c_first, c_last = oracle.dcd_step_rows(xrows, g_own, RING_W, 0.1, p, seed, t, part.a)
            return pack_nonzero(c_first), pack_nonzero(c_last)

        for t in range(iters):
            g_own = np.ascontiguousarray(grads[t][part.a:part.b])
            exchange.ring_iteration(part, local, g_own, t, step, add_pairs)
        np.save(os.path.join(out_dir, f"rows{rank}.npy"), local)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("n,world,p", [(8, 2, 0.01), (5, 3, 0.2), (2, 2, 0.5), (3, 3, 1.0)])
def test_ring_exchange_equals_one_process(tmp_path, n, world, p):
    """DCD-PSGD across ranks: each rank steps its own nodes beside copies of
    its two neighbours, sends the first and last own node's C(z) to the
    neighbouring ranks and adds theirs to its copies.  After every rank's
    iterations the own rows, and the copies, equal the single-process ring
    bit for bit (n = 2 on 2 ranks: both copies are the other node)."""
    import oracle
    d, iters, seed = 3000, 4, 77
    mp.spawn(_ring_worker, args=(world, _free_port(), str(tmp_path), n, d, iters, p, seed), nprocs=world,
             join=True)
    x0, grads = ring_inputs(n, d, iters)
    x = np.ascontiguousarray(np.tile(x0, (n, 1)))
    for t in range(iters):
        oracle.dcd_step(x, grads[t], RING_W, 0.1, p, seed, t)
    for r in range(world):
        part = exchange.RingPartition(n, world, r)
        local = np.load(tmp_path / f"rows{r}.npy")
        for row, node in enumerate(part.row_nodes()):
            np.testing.assert_array_equal(local[row].view(np.uint32), x[node].view(np.uint32),
                                          err_msg=f"rank {r} row {row} (node {node})")


def test_ring_rows_over_the_whole_ring_is_the_ring_step():
    """The rows step with the whole ring laid out as [n-1, 0 .. n-1, 0] is
    the ring step, and its first and last C are the ones nodes 0 and n-1
    added."""
    import oracle
    rng = np.random.default_rng(5)
    n, d = 6, 2000
    x = (rng.standard_normal((n, d)) * 1e-2).astype(np.float32)
    g = (rng.standard_normal((n, d)) * 1e-3).astype(np.float32)
    rows = np.ascontiguousarray(np.concatenate([x[-1:], x, x[:1]]))
    c_first, c_last = oracle.dcd_step_rows(rows, g, RING_W, 0.1, 0.05, 9, 3, 0)
    ring = x.copy()
    oracle.dcd_step(ring, g, RING_W, 0.1, 0.05, 9, 3)
    np.testing.assert_array_equal(rows[1:-1], ring)
    np.testing.assert_array_equal(x[0] + c_first, ring[0])
    np.testing.assert_array_equal(x[-1] + c_last, ring[-1])
