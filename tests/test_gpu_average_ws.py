"""sparse_average_ws: the K-way average through the cursor table and the
region kernel, against the oracle's average bit for bit ("AdaComp ...",
Proposed method; "Deep Gradient Compression", Appendix A).

Cases: random lists sparse and dense, list ranges that fill and overflow a
region's stage, regions with no entries, ragged last regions, K up to 512,
outputs and lists that start off the 16- and 8-byte boundaries, a workspace
reused across calls of other shapes (its stale table must not matter), the
argument errors, malformed lists, and the K = 8 AdaComp messages of the
LSTM + VGG-16 layout at full size.
"""
import numpy as np
import pytest

import oracle
from gradient_compression_sgd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def pairs_of(idx, val, list_offset_words=0):
    """[K, cap, 2] int32 records on the GPU; list_offset_words = 1 places them
    4 bytes past an 8-byte boundary."""
    import torch
    K, cap = idx.shape
    flat = torch.zeros(2 * K * cap + list_offset_words, dtype=torch.int32)
    view = flat[list_offset_words:].view(K, cap, 2)
    view[..., 0] = torch.from_numpy(idx.astype(np.int64)).to(torch.int32)
    view[..., 1] = torch.from_numpy(np.ascontiguousarray(val, np.float32).view(np.int32))
    g = flat.cuda()
    return g[list_offset_words:].view(K, cap, 2)


def run_ws(gc, idx, val, counts, n, out_offset=0, list_offset_words=0, ws=None):
    import torch
    K, cap = idx.shape
    pairs = pairs_of(idx, val, list_offset_words)
    assert (pairs.data_ptr() % 8 == 0) == (list_offset_words == 0)
    if ws is None:
        ws = torch.empty(gc.sparse_average_workspace_size(K, n), dtype=torch.uint8, device="cuda")
    buf = torch.full((max(n, 1) + out_offset + 5,), float("nan"), device="cuda")
    out = buf[out_offset:out_offset + max(n, 1)]
    gc.sparse_average_ws(pairs, torch.from_numpy(np.asarray(counts, np.int64)).cuda(), n, out, ws)
    torch.cuda.synchronize()
    rest = buf.cpu().numpy()
    assert np.isnan(rest[:out_offset]).all() and np.isnan(rest[out_offset + n:]).all()  # nothing outside out
    got = out.cpu().numpy()[:n]
    if n > 0:
        assert gc.sparse_average_status(ws, K, n) == 0  # every bulk copy completed
    want = oracle.sparse_average(idx, val, counts, n)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
    return got


def random_lists(rng, K, n, cap, fill=None):
    idx = np.zeros((K, cap), np.uint32)
    val = np.zeros((K, cap), np.float32)
    counts = np.zeros(K, np.int64)
    for k in range(K):
        c = int(rng.integers(0, min(cap, n) + 1)) if fill is None else min(cap, n, int(fill * n))
        idx[k, :c] = np.sort(rng.choice(n, size=c, replace=False))
        val[k, :c] = rng.standard_normal(c).astype(np.float32)
        counts[k] = c
    return idx, val, counts


@pytest.mark.parametrize("K", [1, 2, 4, 8, 33])
@pytest.mark.parametrize("n", [1, 4095, 8192, 8193, 100003])
@pytest.mark.parametrize("cap_frac", [0.01, 0.3])
def test_ws_random_lists(cuda_lib, K, n, cap_frac):
    rng = np.random.default_rng(K * 1009 + n + int(cap_frac * 100))
    cap = max(1, int(cap_frac * n))
    idx, val, counts = random_lists(rng, K, n, cap)
    run_ws(cuda_lib, idx, val, counts, n)


@pytest.mark.parametrize("K,n,fill", [(8, 3 * 8192 + 77, 1.0), (5, 9000, 1.0), (3, 200000, 0.6), (16, 40000, 0.5)])
def test_ws_stage_overflow(cuda_lib, K, n, fill):
    """Lists dense enough that a region's ranges exceed a 6048-entry stage
    buffer (8 full lists: 32,768 entries per 4096-output region), so the
    regions are added straight from global memory."""
    rng = np.random.default_rng(K + n)
    idx, val, counts = random_lists(rng, K, n, n, fill=fill)
    run_ws(cuda_lib, idx, val, counts, n)


@pytest.mark.parametrize("K,cap_extra", [(4, 0), (3, 1), (7, 3)])
def test_ws_mixed_dense_and_sparse_regions(cuda_lib, K, cap_extra):
    """Every list full over [50000, 90000) and 2 % dense elsewhere: staged
    regions and regions added from global memory alternate in one call, in
    both stage buffers; odd capacities put list starts off the 16-byte
    boundary (first and last pairs copied alone)."""
    rng = np.random.default_rng(K * 31 + cap_extra)
    n = 200003
    dense = np.arange(50000, 90000)
    cap = len(dense) + n // 40 + cap_extra
    idx = np.zeros((K, cap), np.uint32)
    val = np.zeros((K, cap), np.float32)
    counts = np.zeros(K, np.int64)
    for k in range(K):
        rest = np.setdiff1d(np.arange(n), dense)
        pick = np.sort(np.concatenate([dense, rng.choice(rest, size=int(0.02 * len(rest)), replace=False)]))
        c = min(cap, len(pick))
        idx[k, :c], counts[k] = pick[:c], c
        val[k, :c] = rng.standard_normal(c).astype(np.float32)
    assert K * cap >= n // 4
    run_ws(cuda_lib, idx, val, counts, n)


@pytest.mark.parametrize("K,n,density", [(8, 4096 * 40 + 3, 0.05), (2, 4096 * 25, 0.15), (5, 77777, 0.12)])
def test_ws_staged_regions(cuda_lib, K, n, density):
    """AdaComp-like densities: every region fits a stage buffer and goes
    through the bulk copies; odd K and odd capacities misalign list starts."""
    rng = np.random.default_rng(K * 7 + n)
    cap = int(density * n) + K  # K * cap >= n / 4 at these densities
    idx, val, counts = random_lists(rng, K, n, cap, fill=density)
    assert K * cap >= n // 4
    run_ws(cuda_lib, idx, val, counts, n)


def shared_lists(rng, K, n, cap, density, shared):
    """K lists of density * n sorted indices (the same indices in every list
    when `shared`), normal values with -0.0 among them."""
    c = int(density * n)
    idx = np.zeros((K, cap), np.uint32)
    val = np.zeros((K, cap), np.float32)
    common = np.sort(rng.choice(n, size=c, replace=False))
    for k in range(K):
        idx[k, :c] = common if shared else np.sort(rng.choice(n, size=c, replace=False))
        v = rng.standard_normal(c).astype(np.float32)
        v[rng.choice(c, size=max(1, c // 50), replace=False)] = -0.0
        val[k, :c] = v
    return idx, val, np.full(K, c, np.int64)


@pytest.mark.parametrize("K,density,shared", [(8, 0.05, False), (8, 0.09, False), (8, 0.04, True), (3, 0.1, True),
                                              (1, 0.1, False), (7, 0.06, False), (2, 0.08, True)])
def test_ws_shared_indices(cuda_lib, K, density, shared):
    """Up to 8 lists whose ranges in a region fit the consumers' read-ahead
    (at most 512 staged entries per list), some carrying the same outputs:
    the learner-order sum bit for bit.  `shared`: every list carries the
    same indices, so each carried output is a sum of K values; -0.0 values
    check that the first add is 0 + value."""
    rng = np.random.default_rng(K * 31 + int(density * 1000) + shared)
    n = 12 * 4096 + 1234
    idx, val, counts = shared_lists(rng, K, n, n // 2, density, shared)  # K * cap >= n / 4: the region kernel
    run_ws(cuda_lib, idx, val, counts, n)


@pytest.mark.parametrize("K,shared", [(8, True), (8, False), (5, True)])
def test_update_ws_shared_indices(cuda_lib, K, shared):
    """The update mode on the same kind of lists."""
    rng = np.random.default_rng(K + 7 * shared)
    n = 9 * 4096 + 77
    idx, val, counts = shared_lists(rng, K, n, n // 2, 0.05, shared)
    run_update_ws(cuda_lib, idx, val, counts, n, 0.03, seed=K)


def test_ws_empty_regions_and_ragged_tail(cuda_lib):
    """Entries only near the ends of a long output (capacities large enough
    for the region kernel): most regions have none, a checkpoint owns a long
    run of regions, the last region is ragged."""
    rng = np.random.default_rng(9)
    K, n, cap = 4, 100 * 4096 + 1234, 26000
    idx = np.zeros((K, cap), np.uint32)
    val = rng.standard_normal((K, cap)).astype(np.float32)
    counts = np.array([200, 200, 0, 7], np.int64)
    for k in range(K):
        c = int(counts[k])
        pick = np.concatenate([rng.choice(5000, size=c // 2, replace=False),
                               n - 1 - rng.choice(5000, size=c - c // 2, replace=False)])
        idx[k, :c] = np.sort(pick)
    run_ws(cuda_lib, idx, val, counts, n)


@pytest.mark.parametrize("out_offset,list_offset_words", [(1, 0), (2, 1), (3, 1), (0, 1)])
def test_ws_unaligned(cuda_lib, out_offset, list_offset_words):
    """Outputs off the 16-byte boundary; lists 4 bytes off the 8-byte one
    (copied a word at a time)."""
    rng = np.random.default_rng(out_offset * 3 + list_offset_words)
    K, n = 4, 70001
    idx, val, counts = random_lists(rng, K, n, 20000)
    run_ws(cuda_lib, idx, val, counts, n, out_offset=out_offset, list_offset_words=list_offset_words)


def test_ws_512_lists(cuda_lib):
    rng = np.random.default_rng(512)
    K, n, cap = 512, 20011, 60
    idx, val, counts = random_lists(rng, K, n, cap)
    run_ws(cuda_lib, idx, val, counts, n)


def test_ws_reused_workspace(cuda_lib):
    """One workspace across calls of different K and n, largest first: the
    table a call finds is the previous call's, and must not matter."""
    import torch
    gc = cuda_lib
    ws = torch.empty(gc.sparse_average_workspace_size(33, 300000), dtype=torch.uint8, device="cuda")
    ws.fill_(0xA5)
    rng = np.random.default_rng(21)
    for K, n, cap in [(33, 300000, 5000), (4, 100000, 30000), (8, 8193, 8193), (2, 300000, 100), (4, 300000, 30001)]:
        idx, val, counts = random_lists(rng, K, n, cap)
        run_ws(gc, idx, val, counts, n, ws=ws)


def test_ws_equals_sparse_average_on_dgc_messages(cuda_lib):
    """The K = 4 messages of the small ResNet-50 layout after one DGC step:
    both entry points give the same bits."""
    import torch
    gc = cuda_lib
    w = wl.workload(2, small=True)
    d = gc.DGC(w.offsets, w.learners, w.density, w.momentum)
    u = torch.zeros((w.learners, w.n), device="cuda")
    v = torch.zeros((w.learners, w.n), device="cuda")
    out, totals = d(wl.gradients(w, 0).cuda(), u, v)
    a = torch.empty(w.n, device="cuda")
    b = torch.empty(w.n, device="cuda")
    gc.sparse_average(out, totals, w.n, a)
    ws = torch.empty(gc.sparse_average_workspace_size(w.learners, w.n), dtype=torch.uint8, device="cuda")
    gc.sparse_average_ws(out, totals, w.n, b, ws)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_ws_argument_errors(cuda_lib):
    import torch
    gc = cuda_lib
    K, n, cap = 3, 10000, 100
    pairs = torch.zeros((K, cap, 2), dtype=torch.int32, device="cuda")
    counts = torch.zeros(K, dtype=torch.int64, device="cuda")
    out = torch.empty(n, device="cuda")
    need = gc.sparse_average_workspace_size(K, n)
    assert need % 256 == 0 and need >= 4 * K * (-(-n // 8192) + 1)
    with pytest.raises(gc.GcsgdError) as e:
        gc.sparse_average_ws(pairs, counts, n, out, torch.empty(need - 1, dtype=torch.uint8, device="cuda"))
    assert e.value.code == -3  # GCSGD_ERR_WORKSPACE
    big = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(gc.GcsgdError) as e:
        gc.sparse_average_ws(pairs, counts, n, out, big[8:])
    assert e.value.code == -1  # GCSGD_ERR_INVALID_ARG
    with pytest.raises(gc.GcsgdError):
        gc.sparse_average_workspace_size(0, n)
    with pytest.raises(gc.GcsgdError):
        gc.sparse_average_workspace_size(513, n)
    gc.sparse_average_ws(pairs, counts, 0, out, big)  # n = 0: nothing to do
    out.fill_(float("nan"))
    gc.sparse_average_ws(pairs, counts, n, out, big)  # empty lists: all +0
    torch.cuda.synchronize()
    assert (out.view(torch.int32) == 0).all()


def test_ws_malformed_lists_stay_in_range(cuda_lib):
    """Unsorted lists, repeated and out-of-range indices: the result is not
    defined, but the call ends, writes every output and nothing else."""
    import torch
    gc = cuda_lib
    rng = np.random.default_rng(3)
    K, n, cap = 3, 50000, 7000
    pairs = torch.zeros((K, cap, 2), dtype=torch.int32)
    idx = rng.integers(0, n, size=(K, cap)).astype(np.int64)
    idx[0, ::7] = n + 5           # past the end
    idx[1, :50] = 4999            # one index repeated
    idx[2] = np.sort(idx[2])[::-1]  # descending
    pairs[..., 0] = torch.from_numpy(idx).to(torch.int32)
    pairs[..., 1] = torch.from_numpy(rng.standard_normal((K, cap)).astype(np.float32)).view(torch.int32)
    buf = torch.full((n + 8,), float("nan"), device="cuda")
    out = buf[4:4 + n]
    ws = torch.empty(gc.sparse_average_workspace_size(K, n), dtype=torch.uint8, device="cuda")
    gc.sparse_average_ws(pairs.cuda(), torch.full((K,), cap, dtype=torch.int64, device="cuda"), n, out, ws)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.isnan(b[:4]).all() and np.isnan(b[4 + n:]).all()
    assert not np.isnan(b[4:4 + n]).any()


def test_ws_adacomp_full_size(cuda_lib):
    """The K = 8 AdaComp messages of the LSTM + VGG-16 layout (80,748,688
    outputs) after one step, in the benchmark's launch configuration: the
    whole average against the oracle's, bit for bit."""
    import torch
    gc = cuda_lib
    w = wl.workload(3)
    K, N = w.learners, w.n
    a = gc.AdaComp(w.offsets, w.lt, K, N // 8)
    R = torch.zeros((K, N), device="cuda")
    out, totals = a(wl.gradients(w, 0, device="cuda"), R)
    del R
    avg = torch.empty(N, device="cuda")
    ws = torch.empty(gc.sparse_average_workspace_size(K, N), dtype=torch.uint8, device="cuda")
    gc.sparse_average_ws(out, totals, N, avg, ws)
    torch.cuda.synchronize()
    tot = totals.cpu().numpy()
    m = int(tot.max())
    want = oracle.sparse_average(gc.pair_indices(out[:, :m]).cpu().numpy().astype(np.uint32),
                                 gc.pair_values(out[:, :m]).cpu().numpy(), tot, N)
    np.testing.assert_array_equal(avg.cpu().numpy().view(np.uint32), want.view(np.uint32))


# ---------------------------------------- averaged weight update, workspace

def run_update_ws(gc, idx, val, counts, n, lr, seed=0, w_offset=0, list_offset_words=0, ws=None):
    """Weights after sparse_average_update_ws against the oracle's update, bit
    for bit (untouched weights included: -0.0 and a NaN payload among them;
    a carried NaN weight is NaN on both sides)."""
    import torch
    K, cap = idx.shape
    rng = np.random.default_rng(seed)
    w0 = rng.standard_normal(max(n, 1)).astype(np.float32)
    if n > 2:
        w0[n // 2] = -0.0
        w0[n - 1] = np.frombuffer(np.uint32(0x7FC00321).tobytes(), np.float32)[0]
    flat = torch.zeros(max(n, 1) + w_offset + 3, dtype=torch.float32)
    flat[:] = float("nan")
    flat[w_offset:w_offset + max(n, 1)] = torch.from_numpy(w0)
    buf = flat.cuda()
    w_g = buf[w_offset:w_offset + max(n, 1)]
    if ws is None:
        ws = torch.empty(gc.sparse_average_workspace_size(K, n), dtype=torch.uint8, device="cuda")
    gc.sparse_average_update_ws(pairs_of(idx, val, list_offset_words),
                                torch.from_numpy(np.asarray(counts, np.int64)).cuda(), n, lr, w_g, ws)
    torch.cuda.synchronize()
    if n > 0:
        assert gc.sparse_average_status(ws, K, n) == 0
    rest = buf.cpu().numpy()
    assert np.isnan(rest[:w_offset]).all() and np.isnan(rest[w_offset + max(n, 1):]).all()
    want = oracle.sparse_average_update(idx, val, np.asarray(counts, np.int64), n, lr, w0.copy())
    got = w_g.cpu().numpy()[:n]
    both_nan = np.isnan(got) & np.isnan(want[:n])
    carried = np.zeros(n, bool)
    for k in range(K):
        carried[idx[k, :counts[k]]] = True
    keep = ~(both_nan & carried)
    np.testing.assert_array_equal(got.view(np.uint32)[keep], want[:n].view(np.uint32)[keep])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want[:n]))


@pytest.mark.parametrize("K", [1, 2, 4, 8, 33])
@pytest.mark.parametrize("n", [1, 4095, 8193, 100003])
@pytest.mark.parametrize("cap_frac", [0.01, 0.3])
def test_update_ws_random_lists(cuda_lib, K, n, cap_frac):
    rng = np.random.default_rng(K * 17 + n + int(cap_frac * 100))
    cap = max(1, int(cap_frac * n))
    idx, val, counts = random_lists(rng, K, n, cap)
    run_update_ws(cuda_lib, idx, val, counts, n, 0.05, seed=K + n)


@pytest.mark.parametrize("K,n,fill", [(8, 3 * 4096 + 77, 1.0), (3, 200000, 0.6), (5, 77777, 0.12)])
def test_update_ws_staged_and_overflowing_regions(cuda_lib, K, n, fill):
    """Regions that fit the stage (AdaComp-like density) and regions added
    from global memory (full lists), with a negative learning rate."""
    rng = np.random.default_rng(K + n)
    idx, val, counts = random_lists(rng, K, n, n, fill=fill)
    run_update_ws(cuda_lib, idx, val, counts, n, -0.01, seed=K)


@pytest.mark.parametrize("w_offset,list_offset_words", [(1, 0), (3, 0), (2, 1)])
def test_update_ws_unaligned(cuda_lib, w_offset, list_offset_words):
    """Weights off the 16-byte boundary (scalar writes of the carried values
    only); lists 4 bytes off the 8-byte boundary (sparse_average_update)."""
    rng = np.random.default_rng(w_offset * 5 + list_offset_words)
    K, n = 4, 70001
    idx, val, counts = random_lists(rng, K, n, 20000)
    run_update_ws(cuda_lib, idx, val, counts, n, 0.1, seed=w_offset, w_offset=w_offset,
                  list_offset_words=list_offset_words)


def test_update_ws_512_lists_and_reuse(cuda_lib):
    import torch
    gc = cuda_lib
    ws = torch.empty(gc.sparse_average_workspace_size(512, 300000), dtype=torch.uint8, device="cuda")
    ws.fill_(0x5A)
    rng = np.random.default_rng(7)
    for K, n, cap in [(512, 20011, 60), (4, 300000, 30000), (8, 8193, 8193)]:
        idx, val, counts = random_lists(rng, K, n, cap)
        run_update_ws(gc, idx, val, counts, n, 0.02, seed=K, ws=ws)


def test_update_ws_adacomp_full_size(cuda_lib):
    """The K = 8 AdaComp messages of the LSTM + VGG-16 layout: the weights
    after sparse_average_update_ws equal sparse_average_update's bit for bit,
    and on a sample of 20,000 indices the oracle's update of those indices."""
    import torch
    gc = cuda_lib
    w = wl.workload(3)
    K, N = w.learners, w.n
    a = gc.AdaComp(w.offsets, w.lt, K, N // 8)
    R = torch.zeros((K, N), device="cuda")
    out, totals = a(wl.gradients(w, 0, device="cuda"), R)
    del R
    g = torch.Generator(device="cpu").manual_seed(5)
    w0 = torch.randn(N, generator=g).cuda()
    w1, w2 = w0.clone(), w0.clone()
    gc.sparse_average_update(out, totals, N, 0.03, w1)
    ws = torch.empty(gc.sparse_average_workspace_size(K, N), dtype=torch.uint8, device="cuda")
    gc.sparse_average_update_ws(out, totals, N, 0.03, w2, ws)
    torch.cuda.synchronize()
    assert gc.sparse_average_status(ws, K, N) == 0
    assert torch.equal(w1.view(torch.int32), w2.view(torch.int32))
    tot = totals.cpu().numpy()
    m = int(tot.max())
    idx = gc.pair_indices(out[:, :m]).cpu().numpy().astype(np.uint32)
    val = gc.pair_values(out[:, :m]).cpu().numpy()
    want = oracle.sparse_average_update(idx, val, tot, N, 0.03, w0.cpu().numpy().copy())
    sample = np.random.default_rng(1).choice(N, size=20000, replace=False)
    np.testing.assert_array_equal(w2.cpu().numpy()[sample].view(np.uint32), want[sample].view(np.uint32))
