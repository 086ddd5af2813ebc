"""AdaComp, sparse-average and DCD parity: CUDA library against the CPU oracle.

Indices, counts and masks are compared bit for bit; fp32 values within 1e-6
relative (1e-5 for the K-way averages, where the contract allows a different
summation order; the kernel keeps learner order, so they are expected exact).
"""
import numpy as np
import pytest

import oracle
from conftest import rel_err
from gradient_compression_sgd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

VAL_RTOL = 1e-6
AVG_RTOL = 1e-5


# ------------------------------------------------------------------ AdaComp

def shifted(a, offset):
    """A CUDA copy of `a` starting `offset` floats past an allocation's start."""
    import torch
    flat = torch.zeros(a.size + offset, dtype=torch.float32, device="cuda")
    view = flat[offset:].view(a.shape)
    view.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return view


def run_adacomp(gc, offsets, lt, dWs, cap=None, R0=None, offset=0):
    import torch
    offsets = np.asarray(offsets, np.int64)
    K, N = dWs[0].shape
    cap = cap if cap is not None else max(1, N)
    R_o = np.zeros((K, N), np.float32) if R0 is None else R0.copy()
    R_g = shifted(R_o, offset)
    a = gc.AdaComp(offsets, lt, K, cap)
    results = []
    for t, dW in enumerate(dWs):
        G = R_o + dW  # fp32, the value the residue is measured against
        try:
            idx_o, val_o, counts_o, scales_o, totals_o = oracle.adacomp_step(offsets, lt, dW, R_o, cap=cap)
            over = False
        except oracle.OracleError:
            over = True
        out, totals = a(shifted(dW, offset), R_g)
        torch.cuda.synchronize()
        tot_g = totals.cpu().numpy()
        if over:
            results.append(("overflow", tot_g))
            assert np.any(tot_g > cap)
            assert rel_err(R_g.cpu().numpy(), R_o) <= VAL_RTOL
            continue
        np.testing.assert_array_equal(a.counts.cpu().numpy(), counts_o, err_msg=f"counts t={t}")
        np.testing.assert_array_equal(tot_g, totals_o)
        assert rel_err(a.scales.cpu().numpy(), scales_o) <= VAL_RTOL, f"scales t={t}"
        idx_g = gc.pair_indices(out).cpu().numpy()
        val_g = gc.pair_values(out).cpu().numpy()
        for k in range(K):
            n = int(totals_o[k])
            np.testing.assert_array_equal(idx_g[k, :n], idx_o[k, :n].astype(np.int64), err_msg=f"idx k={k} t={t}")
            assert rel_err(val_g[k, :n], val_o[k, :n]) <= VAL_RTOL
        # residue: relative to |G| (cancellation near G ~ scale makes |R| a poor yardstick)
        Rg = R_g.cpu().numpy()
        denom = np.maximum(np.abs(G), np.abs(R_o))
        err = np.abs(Rg.astype(np.float64) - R_o) / np.maximum(denom, np.finfo(np.float32).tiny)
        assert float(err.max(initial=0.0)) <= VAL_RTOL, f"residue t={t}"
        results.append(("ok", tot_g))
    return a, results


def test_config1_adacomp_lt50(cuda_lib):
    """The config-1 tensor (1,048,576 values N(0, 1e-3)) with L_T = 50
    (20,972 bins, the last one of 26 values), 3 steps with the residue carried."""
    w = wl.workload(1)
    dWs = [wl.gradients(w, t).numpy() for t in range(w.steps)]
    run_adacomp(cuda_lib, w.offsets, [w.also_adacomp_lt], dWs)


def test_config3_small(cuda_lib):
    """LSTM (hidden 150, vocab 1000; L_T = 500) + VGG-16 convs at 1/8 width
    (L_T = 50), Laplace gradients, K = 8, 5 steps."""
    w = wl.workload(3, small=True)
    dWs = [wl.gradients(w, t).numpy() for t in range(w.steps)]
    run_adacomp(cuda_lib, w.offsets, w.lt, dWs)


@pytest.mark.parametrize("L", [1, 3, 4, 50, 64, 500, 4096, 5000, 123457])
def test_bin_lengths(cuda_lib, L):
    """Bin lengths below 4, odd, a whole tile, longer than a tile (bins that
    straddle tiles), and one bin for the whole segment."""
    rng = np.random.default_rng(L)
    sizes = [123457, 0, 4099, 77]
    off = wl.layout_offsets(sizes)
    K = 2
    dWs = [rng.laplace(0, 1e-3, size=(K, off[-1])).astype(np.float32) for _ in range(3)]
    run_adacomp(cuda_lib, off, [L] * len(sizes), dWs)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_buffers_not_16_byte_aligned(cuda_lib, offset):
    """dW and R starting 4, 8 or 12 bytes past a 16-byte boundary."""
    rng = np.random.default_rng(offset + 40)
    sizes, lt = [50001, 8000, 4096], [50, 500, 64]
    off = wl.layout_offsets(sizes)
    dWs = [rng.laplace(0, 1e-3, size=(2, off[-1])).astype(np.float32) for _ in range(2)]
    run_adacomp(cuda_lib, off, lt, dWs, offset=offset)


def test_nan_entries_are_never_sent(cuda_lib):
    """A NaN in G never wins a bin maximum and is never sent (every comparison
    with NaN is false); its residue stays NaN; the rest is unaffected."""
    import torch
    gc = cuda_lib
    rng = np.random.default_rng(17)
    sizes, lt = [5000, 30000, 9000], [50, 500, 7000]
    off = wl.layout_offsets(sizes)
    K, N = 2, off[-1]
    dW = rng.laplace(0, 1e-3, size=(K, N)).astype(np.float32)
    dW[0, [3, 77, 5123, 30001, 36000]] = np.nan
    dW[1, [0, 4999, 35000]] = np.nan
    R_o = np.zeros((K, N), np.float32)
    idx_o, val_o, counts_o, scales_o, totals_o = oracle.adacomp_step(off, lt, dW, R_o, cap=N)
    R_g = torch.zeros((K, N), device="cuda")
    a = gc.AdaComp(off, lt, K, N)
    out, totals = a(torch.from_numpy(dW).cuda(), R_g)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(a.counts.cpu().numpy(), counts_o)
    np.testing.assert_array_equal(totals.cpu().numpy(), totals_o)
    assert rel_err(a.scales.cpu().numpy(), scales_o) <= VAL_RTOL
    idx_g, val_g = gc.pair_indices(out).cpu().numpy(), gc.pair_values(out).cpu().numpy()
    for k in range(K):
        n = int(totals_o[k])
        np.testing.assert_array_equal(idx_g[k, :n], idx_o[k, :n].astype(np.int64))
        assert not np.isnan(val_g[k, :n]).any() and rel_err(val_g[k, :n], val_o[k, :n]) <= VAL_RTOL
    Rg = R_g.cpu().numpy()
    np.testing.assert_array_equal(np.isnan(Rg), np.isnan(R_o))
    fin = ~np.isnan(R_o)
    assert rel_err(Rg[fin], R_o[fin]) <= VAL_RTOL


def test_mixed_bins_and_ragged_offsets(cuda_lib):
    rng = np.random.default_rng(5)
    sizes = [7, 50001, 13, 4096, 4097, 99999]
    lt = [2, 50, 5, 500, 4096, 7000]
    off = wl.layout_offsets(sizes)
    dWs = [rng.laplace(0, 1e-2, size=(3, off[-1])).astype(np.float32) for _ in range(3)]
    dWs[1][:, 100:400] = 0.0  # all-zero bins select nothing
    run_adacomp(cuda_lib, off, lt, dWs)


def test_capacity_overflow_sends_nothing_and_keeps_the_residue(cuda_lib):
    rng = np.random.default_rng(6)
    off = wl.layout_offsets([20000])
    dWs = [rng.laplace(0, 1.0, size=(2, 20000)).astype(np.float32) for _ in range(2)]
    dWs[0][1] *= 0  # learner 1 sends nothing at step 0: fits
    _, res = run_adacomp(cuda_lib, off, [1], dWs, cap=5000)
    assert res[0][0] == "overflow"


def test_capacity_overflow_leaves_the_list_and_reports_would_be_counts(cuda_lib):
    """A learner over cap: its list is not written (sentinel words stay), its
    counts add up to its would-be total, and its residue is G = R + dW; the
    learner that fits sends as usual."""
    import torch
    gc = cuda_lib
    rng = np.random.default_rng(61)
    off = wl.layout_offsets([20000])
    dW = rng.laplace(0, 1.0, size=(2, 20000)).astype(np.float32)
    R0 = rng.laplace(0, 0.1, size=(2, 20000)).astype(np.float32)
    dW[1, 100:] = 0.0  # learner 1: G = 0 past its first 100 values, so it sends at most 100
    R0[1] = 0.0
    a = gc.AdaComp(off, [1], 2, 5000)
    a.out.fill_(0x7A7A7A7A)
    R = torch.from_numpy(R0.copy()).cuda()
    out, totals = a(torch.from_numpy(dW).cuda(), R)
    torch.cuda.synchronize()
    tot = totals.cpu().numpy()
    assert tot[0] > 5000 >= tot[1]
    assert int(a.counts[0].sum().item()) == tot[0]
    assert bool(torch.all(out[0] == 0x7A7A7A7A).item())
    np.testing.assert_array_equal(R[0].cpu().numpy(), R0[0] + dW[0])
    Ro = R0.copy()
    idx_o, val_o, counts_o, scales_o, totals_o = oracle.adacomp_step(off, [1], dW[1:], Ro[1:], cap=5000)
    n1 = int(totals_o[0])
    assert tot[1] == n1
    np.testing.assert_array_equal(gc.pair_indices(out)[1, :n1].cpu().numpy(), idx_o[0, :n1].astype(np.int64))


# ------------------------------------------------------------ sparse average

def padded(idx, val, cap):
    """The same lists in a wider buffer (the sparse average picks its kernel
    from K * cap against n: a quarter entry per output or more is dense)."""
    K, c = idx.shape
    if cap <= c:
        return idx, val
    i2 = np.zeros((K, cap), np.uint32)
    v2 = np.zeros((K, cap), np.float32)
    i2[:, :c], v2[:, :c] = idx, val
    return i2, v2


def run_average(gc, idx, val, counts, n, out_offset=0):
    import torch
    K, cap = idx.shape
    pairs = torch.zeros((K, cap, 2), dtype=torch.int32)
    pairs[..., 0] = torch.from_numpy(idx.astype(np.int64)).to(torch.int32)
    pairs[..., 1] = torch.from_numpy(val.view(np.int32))
    pairs = pairs.cuda()
    # NaN everywhere, so an output the kernel fails to write shows
    buf = torch.full((max(n, 1) + out_offset + 5,), float("nan"), device="cuda")
    out = buf[out_offset:out_offset + max(n, 1)]
    gc.sparse_average(pairs, torch.from_numpy(counts.astype(np.int64)).cuda(), n, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()[:n]
    rest = buf.cpu().numpy()
    assert np.isnan(rest[:out_offset]).all() and np.isnan(rest[out_offset + n:]).all()  # nothing outside out
    want = oracle.sparse_average(idx, val, counts, n)
    assert rel_err(got, want) <= AVG_RTOL
    np.testing.assert_array_equal(np.nonzero(got)[0], np.nonzero(want)[0])
    return got, want


@pytest.mark.parametrize("kernel", ["tiles", "warp_spans"])
@pytest.mark.parametrize("K", [1, 2, 4, 8, 33])
@pytest.mark.parametrize("n", [1, 4095, 4096, 100003])
def test_sparse_average_random_lists(cuda_lib, K, n, kernel):
    rng = np.random.default_rng(K * 7 + n)
    cap = max(1, min(n, 3000, n // (4 * K) - 1 if kernel == "tiles" else n))
    if kernel == "tiles" and K * cap >= n // 4:
        pytest.skip("no list capacity this small is sparse")
    idx = np.zeros((K, cap), np.uint32)
    val = np.zeros((K, cap), np.float32)
    counts = np.zeros(K, np.int64)
    for k in range(K):
        c = int(rng.integers(0, cap + 1))
        idx[k, :c] = np.sort(rng.choice(n, size=c, replace=False))
        val[k, :c] = rng.standard_normal(c).astype(np.float32)
        counts[k] = c
    if kernel == "warp_spans":
        idx, val = padded(idx, val, max(cap, -(-n // (4 * K))))
    got, want = run_average(cuda_lib, idx, val, counts, n)
    np.testing.assert_array_equal(got, want)  # learner order kept: exact


@pytest.mark.parametrize("offset", [1, 2, 3])
@pytest.mark.parametrize("K", [3, 4])
def test_sparse_average_unaligned_output(cuda_lib, offset, K):
    """The output vector need not start on a 16-byte boundary."""
    rng = np.random.default_rng(offset * 10 + K)
    n, cap = 50001, 400
    idx = np.zeros((K, cap), np.uint32)
    val = np.zeros((K, cap), np.float32)
    counts = np.zeros(K, np.int64)
    for k in range(K):
        c = int(rng.integers(1, cap + 1))
        pick = np.concatenate([[0, n - 1], rng.choice(np.arange(1, n - 1), size=c - 2, replace=False)])[:c]
        idx[k, :c] = np.sort(pick)
        val[k, :c] = rng.standard_normal(c).astype(np.float32)
        counts[k] = c
    got, want = run_average(cuda_lib, idx, val, counts, n, out_offset=offset)
    np.testing.assert_array_equal(got, want)
    idx, val = padded(idx, val, -(-n // (4 * K)))  # the same lists through the warp-span kernel
    got, want = run_average(cuda_lib, idx, val, counts, n, out_offset=offset)
    np.testing.assert_array_equal(got, want)


def test_sparse_average_of_dgc_messages(cuda_lib):
    """The K = 4 messages of the small ResNet-50 layout after DGC step 1."""
    import torch
    gc = cuda_lib
    w = wl.workload(2, small=True)
    G = wl.gradients(w, 0)
    d = gc.DGC(w.offsets, w.learners, w.density, w.momentum)
    u = torch.zeros((w.learners, w.n), device="cuda")
    v = torch.zeros((w.learners, w.n), device="cuda")
    out, totals = d(G.cuda(), u, v)
    torch.cuda.synchronize()
    idx = gc.pair_indices(out).cpu().numpy().astype(np.uint32)
    val = gc.pair_values(out).cpu().numpy()
    run_average(gc, idx, val, totals.cpu().numpy(), w.n)


def test_sparse_average_dense_lists(cuda_lib):
    """Every index in every list (density 1): each output is a K-term sum."""
    rng = np.random.default_rng(1)
    K, n = 5, 9000
    idx = np.tile(np.arange(n, dtype=np.uint32), (K, 1))
    val = rng.standard_normal((K, n)).astype(np.float32)
    got, want = run_average(cuda_lib, idx, val, np.full(K, n, np.int64), n)
    np.testing.assert_array_equal(got, want)


def test_sparse_average_512_lists(cuda_lib):
    """The largest K the call takes: 64 batches of eight lists per span."""
    rng = np.random.default_rng(512)
    K, n, cap = 512, 20011, 60
    idx = np.zeros((K, cap), np.uint32)
    val = np.zeros((K, cap), np.float32)
    counts = rng.integers(0, cap + 1, size=K).astype(np.int64)
    for k in range(K):
        idx[k, :counts[k]] = np.sort(rng.choice(n, size=int(counts[k]), replace=False))
        val[k, :counts[k]] = rng.standard_normal(int(counts[k])).astype(np.float32)
    got, want = run_average(cuda_lib, idx, val, counts, n)
    np.testing.assert_array_equal(got, want)


def test_sparse_average_malformed_lists_stay_in_range(cuda_lib):
    """Unsorted lists, repeated and out-of-range indices: the result is not
    defined, but the call ends, writes every output and nothing else."""
    import torch
    gc = cuda_lib
    rng = np.random.default_rng(3)
    K, n, cap = 3, 5000, 700
    pairs = torch.zeros((K, cap, 2), dtype=torch.int32)
    idx = rng.integers(0, n, size=(K, cap)).astype(np.int64)
    idx[0, ::7] = n + 5           # past the end
    idx[1, :50] = 4999            # one index repeated
    idx[2] = np.sort(idx[2])[::-1]  # descending
    pairs[..., 0] = torch.from_numpy(idx).to(torch.int32)
    pairs[..., 1] = torch.from_numpy(rng.standard_normal((K, cap)).astype(np.float32)).view(torch.int32)
    buf = torch.full((n + 8,), float("nan"), device="cuda")
    out = buf[4:4 + n]
    gc.sparse_average(pairs.cuda(), torch.full((K,), cap, dtype=torch.int64, device="cuda"), n, out)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.isnan(b[:4]).all() and np.isnan(b[4 + n:]).all()
    assert not np.isnan(b[4:4 + n]).any()


# --------------------------------------------- averaged sparse weight update

def run_update(gc, idx, val, counts, n, lr, seed=0, w_offset=0):
    """Weights after the fused average-update, CUDA vs oracle, bit for bit
    (untouched weights included: -0.0 and a NaN payload among them)."""
    import torch
    K, cap = idx.shape
    rng = np.random.default_rng(seed)
    w0 = rng.standard_normal(max(n, 1)).astype(np.float32)
    if n > 2:
        w0[n // 2] = -0.0
        w0[n - 1] = np.frombuffer(np.uint32(0x7FC00321).tobytes(), np.float32)[0]
    pairs = torch.zeros((K, cap, 2), dtype=torch.int32)
    pairs[..., 0] = torch.from_numpy(idx.astype(np.int64)).to(torch.int32)
    pairs[..., 1] = torch.from_numpy(val.view(np.int32))
    w_g = shifted(w0, w_offset)
    gc.sparse_average_update(pairs.cuda(), torch.from_numpy(counts.astype(np.int64)).cuda(), n, lr, w_g)
    torch.cuda.synchronize()
    want = oracle.sparse_average_update(idx, val, counts, n, lr, w0.copy())
    got = w_g.cpu().numpy()[:n]
    # bit for bit, except that a NaN weight that gets updated is NaN on both
    # sides with whatever payload the hardware's subtraction returns
    both_nan = np.isnan(got) & np.isnan(want[:n])
    carried = np.zeros(n, bool)
    for k in range(K):
        carried[idx[k, :counts[k]]] = True
    np.testing.assert_array_equal(got.view(np.uint32)[~both_nan | ~carried], want[:n].view(np.uint32)[~both_nan | ~carried])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want[:n]))


@pytest.mark.parametrize("K", [1, 2, 4, 8, 33])
@pytest.mark.parametrize("n", [1, 4095, 4096, 100003])
def test_update_random_lists(cuda_lib, K, n):
    rng = np.random.default_rng(K * 11 + n)
    cap = max(1, min(n, 3000))
    idx = np.zeros((K, cap), np.uint32)
    val = np.zeros((K, cap), np.float32)
    counts = np.zeros(K, np.int64)
    for k in range(K):
        c = int(rng.integers(0, cap + 1))
        idx[k, :c] = np.sort(rng.choice(n, size=c, replace=False))
        val[k, :c] = rng.standard_normal(c).astype(np.float32)
        counts[k] = c
    run_update(cuda_lib, idx, val, counts, n, 0.05, seed=K + n)


@pytest.mark.parametrize("offset", [1, 3])
def test_update_unaligned_weights_and_dense_lists(cuda_lib, offset):
    """Every index in every list (the dense, windowed path) and weights off a 16-byte boundary."""
    rng = np.random.default_rng(offset)
    K, n = 5, 9000
    idx = np.tile(np.arange(n, dtype=np.uint32), (K, 1))
    val = rng.standard_normal((K, n)).astype(np.float32)
    run_update(cuda_lib, idx, val, np.full(K, n, np.int64), n, -0.01, seed=offset, w_offset=offset)


def test_update_of_dgc_messages(cuda_lib):
    """The K = 4 messages of the small ResNet-50 layout after DGC step 1."""
    import torch
    gc = cuda_lib
    w = wl.workload(2, small=True)
    G = wl.gradients(w, 0)
    d = gc.DGC(w.offsets, w.learners, w.density, w.momentum)
    u = torch.zeros((w.learners, w.n), device="cuda")
    v = torch.zeros((w.learners, w.n), device="cuda")
    out, totals = d(G.cuda(), u, v)
    torch.cuda.synchronize()
    idx = gc.pair_indices(out).cpu().numpy().astype(np.uint32)
    val = gc.pair_values(out).cpu().numpy()
    run_update(gc, idx, val, totals.cpu().numpy(), w.n, 0.1, seed=3, w_offset=2)


# ---------------------------------------------------------------------- DCD

def run_dcd(gc, n, d, T, p, w=(1 / 3, 1 / 3, 1 / 3), gamma=0.1, seed=0x5EED):
    import torch
    rng = np.random.default_rng(n * 1000 + d)
    x0 = (rng.standard_normal(d) * 1e-2).astype(np.float32)
    x_o = np.tile(x0, (n, 1)).copy()
    x_g = torch.from_numpy(x_o.copy()).cuda()
    for t in range(T):
        g = (rng.standard_normal((n, d)) * 1e-3).astype(np.float32)
        oracle.dcd_step(x_o, g, w, gamma, p, seed, t)
        gc.dcd_step(x_g, torch.from_numpy(g).cuda(), w, gamma, p, seed, t)
    torch.cuda.synchronize()
    got = x_g.cpu().numpy()
    np.testing.assert_array_equal(got == x0[None, :], x_o == x0[None, :])  # identical keep masks
    assert rel_err(got, x_o) <= VAL_RTOL


def test_config5_small(cuda_lib):
    """Ring of 8 nodes, d = 262,144, W = 1/3, gamma = 0.1, keep 1% scaled x100, 10 iterations."""
    w = wl.workload(5, small=True)
    run_dcd(cuda_lib, w.learners, w.n, w.steps, w.keep_p, w.ring_w, w.gamma, wl.dcd_seed(w))


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 9, 13])
@pytest.mark.parametrize("d", [1, 7, 4096, 10001])
def test_dcd_nodes_and_sizes(cuda_lib, n, d):
    run_dcd(cuda_lib, n, d, 3, 0.3)


def test_dcd_keep_all_and_weights(cuda_lib):
    run_dcd(cuda_lib, 4, 5000, 2, 1.0, w=(0.25, 0.5, 0.25))
    run_dcd(cuda_lib, 1, 5000, 2, 1.0, w=(0.0, 1.0, 0.0))


@pytest.mark.parametrize("n", [5, 13])
def test_dcd_asymmetric_ring_weights(cuda_lib, n):
    """w_ring = (left, self, right) with unequal weights, p = 1 and p = 0.3:
    the fixed-size (n = 5) and rolling (n = 13) kernels take node i - 1 as
    the left neighbour, as the oracle does (3 steps, so the models differ)."""
    run_dcd(cuda_lib, n, 5003, 3, 1.0, w=(0.6, 0.3, 0.1))
    run_dcd(cuda_lib, n, 5003, 3, 0.3, w=(0.1, 0.25, 0.65))


@pytest.mark.parametrize("n", [3, 9])
def test_ecd_asymmetric_ring_weights(cuda_lib, n):
    run_ecd(cuda_lib, n, 4099, 3, 0.5, w=(0.6, 0.3, 0.1))


def test_philox_matches_curand_device_api(cuda_lib, tmp_path):
    """The oracle's Philox4x32-10 word block at counter (q, node, t, q >> 32)
    under key (seed) equals cuRAND's curand4 after curand_init(seed,
    subsequence = t, offset = 4 (q + node 2^32)) -- a library routine."""
    import ctypes
    import subprocess

    import torch
    from gradient_compression_sgd_gb300 import build as gbuild
    src = __import__("os").path.join(__import__("os").path.dirname(__file__), "curand_philox.cu")
    so = str(tmp_path / "curand_philox.so")
    subprocess.check_call([gbuild.nvcc(), *gbuild.ARCH, "-O2", "-shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
                           src, "-o", so])
    L = ctypes.CDLL(so)
    rng = np.random.default_rng(3)
    seed = 0x5EED000000000005
    qs = np.concatenate([[0, 1, 2, 3, 6_399_999], rng.integers(0, 1 << 31, size=59)]).astype(np.uint64)
    nodes = rng.integers(0, 8, size=len(qs)).astype(np.uint64)
    ts = rng.integers(0, 10, size=len(qs)).astype(np.uint64)
    sub = torch.from_numpy(ts.astype(np.int64)).cuda()
    off = torch.from_numpy((4 * (qs + (nodes << np.uint64(32)))).astype(np.int64)).cuda()
    out = torch.zeros((len(qs), 4), dtype=torch.int32, device="cuda")
    assert L.curand_philox_blocks(ctypes.c_ulonglong(seed), ctypes.c_void_p(sub.data_ptr()),
                                  ctypes.c_void_p(off.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                  ctypes.c_int(len(qs))) == 0
    got = out.cpu().numpy().view(np.uint32)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for i in range(len(qs)):
        want = oracle.philox4x32_10([int(qs[i]) & 0xFFFFFFFF, int(nodes[i]), int(ts[i]), int(qs[i]) >> 32], key)
        np.testing.assert_array_equal(got[i], want)


# ----------------------------------------------------------------- ECD-PSGD

def run_ecd(gc, n, d, T, p, w=(1 / 3, 1 / 3, 1 / 3), gamma=0.1, seed=0xEC0, offset=0):
    """T iterations (t = 1..T) on both sides, the caller swapping x and
    x_prev after each; models and estimates compared after every step."""
    rng = np.random.default_rng(n * 1000 + d + offset)
    x0 = (rng.standard_normal(d) * 1e-2).astype(np.float32)
    xo, xpo, xto = (np.tile(x0, (n, 1)).copy() for _ in range(3))
    xg, xpg, xtg = (shifted(np.tile(x0, (n, 1)), offset) for _ in range(3))
    for t in range(1, T + 1):
        g = (rng.standard_normal((n, d)) * 1e-3).astype(np.float32)
        oracle.ecd_step(xo, xpo, xto, g, w, gamma, p, seed, t)
        gc.ecd_step(xg, xpg, xtg, shifted(g, offset), w, gamma, p, seed, t)
        xo, xpo = xpo, xo
        xg, xpg = xpg, xg
        import torch
        torch.cuda.synchronize()
        np.testing.assert_array_equal(xg.cpu().numpy().view(np.uint32), xo.view(np.uint32), err_msg=f"model t={t}")
        np.testing.assert_array_equal(xtg.cpu().numpy().view(np.uint32), xto.view(np.uint32), err_msg=f"est t={t}")


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 9, 13])
@pytest.mark.parametrize("d", [1, 7, 4096, 10001])
def test_ecd_nodes_and_sizes(cuda_lib, n, d):
    run_ecd(cuda_lib, n, d, 4, 0.3)


@pytest.mark.parametrize("offset", [1, 3])
def test_ecd_ring8_sparsified_unaligned(cuda_lib, offset):
    """The config-5 ring (8 nodes, keep 1 % scaled x100) at d = 262,144, 6 iterations, buffers off 16 bytes."""
    run_ecd(cuda_lib, 8, 262144, 6, 0.01, offset=offset)
