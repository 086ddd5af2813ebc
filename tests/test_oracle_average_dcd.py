"""Pins of the oracle's sparse average and DCD-PSGD step (CPU only)."""
import numpy as np
import pytest

import oracle
from conftest import ulp32


# ----------------------------------------------------------- sparse average

def _lists(rng, K, n, cap, fill):
    idx = np.zeros((K, cap), np.uint32)
    val = np.zeros((K, cap), np.float32)
    counts = np.zeros(K, np.int64)
    for k in range(K):
        c = int(rng.integers(0, fill + 1))
        sel = np.sort(rng.choice(n, size=c, replace=False))
        idx[k, :c] = sel
        val[k, :c] = rng.standard_normal(c).astype(np.float32)
        counts[k] = c
    return idx, val, counts


def test_single_list_is_decompression():
    rng = np.random.default_rng(0)
    idx, val, counts = _lists(rng, 1, 500, 64, 64)
    out = oracle.sparse_average(idx, val, counts, 500)
    want = np.zeros(500, np.float32)
    want[idx[0, :counts[0]]] = val[0, :counts[0]]
    np.testing.assert_array_equal(out, want)


@pytest.mark.parametrize("K", [2, 3, 4, 8])
def test_matches_numpy_ordered_scatter_add(K):
    """numpy's unbuffered ufunc.at adds duplicates in the order given, so the
    lists concatenated in learner order reproduce the K-ordered fp32 sum."""
    rng = np.random.default_rng(K)
    n, cap = 3000, 400
    idx, val, counts = _lists(rng, K, n, cap, cap)
    acc = np.zeros(n, np.float32)
    for k in range(K):
        np.add.at(acc, idx[k, :counts[k]].astype(np.int64), val[k, :counts[k]])
    want = acc / np.float32(K)
    out = oracle.sparse_average(idx, val, counts, n)
    np.testing.assert_array_equal(out, want)
    # mass and support
    assert abs(out.astype(np.float64).sum() * K - sum(val[k, :counts[k]].astype(np.float64).sum() for k in range(K))) < 1e-4
    support = set()
    for k in range(K):
        support |= set(idx[k, :counts[k]].tolist())
    assert set(np.nonzero(out)[0].tolist()) <= support


def test_index_out_of_range_is_rejected():
    idx = np.array([[5]], np.uint32)
    val = np.array([[1.0]], np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.sparse_average(idx, val, np.array([1]), 5)


# ------------------------------------------- averaged sparse weight update

@pytest.mark.parametrize("K", [1, 2, 4, 7])
def test_update_matches_numpy(K):
    """w[j] -= lr * avg[j] on the support, with avg from numpy's ordered
    ufunc.at and one float32 rounding per operation; every other weight keeps
    its bits (including -0.0 and a NaN payload)."""
    rng = np.random.default_rng(100 + K)
    n, cap = 4000, 300
    idx, val, counts = _lists(rng, K, n, cap, cap)
    w0 = rng.standard_normal(n).astype(np.float32)
    support = np.zeros(n, bool)
    for k in range(K):
        support[idx[k, :counts[k]]] = True
    off = np.nonzero(~support)[0]
    w0[off[0]] = -0.0
    w0[off[1]] = np.frombuffer(np.uint32(0x7FC00123).tobytes(), np.float32)[0]
    acc = np.zeros(n, np.float32)
    for k in range(K):
        np.add.at(acc, idx[k, :counts[k]].astype(np.int64), val[k, :counts[k]])
    avg = acc / np.float32(K)
    lr = np.float32(0.0375)
    want = w0.copy()
    want[support] = want[support] - lr * avg[support]
    got = oracle.sparse_average_update(idx, val, counts, n, lr, w0.copy())
    np.testing.assert_array_equal(got.view(np.uint32)[~support], w0.view(np.uint32)[~support])
    np.testing.assert_array_equal(got[support], want[support])


def test_update_single_list_dyadic_is_exact():
    """K = 1, lr = 1/2 and dyadic values: every step is exact, w - v/2."""
    idx = np.array([[1, 4, 7]], np.uint32)
    val = np.array([[2.0, -0.5, 3.0]], np.float32)
    w = np.array([1, 1, 1, 1, 1, 1, 1, 1], np.float32)
    oracle.sparse_average_update(idx, val, np.array([3]), 8, 0.5, w)
    np.testing.assert_array_equal(w, np.array([1, 0, 1, 1, 1.25, 1, 1, -0.5], np.float32))


# -------------------------------------------------------------------- Philox

def test_philox_known_answers(golden):
    ex = golden("philox4x32_10_kat.txt")
    with open(__import__("os").path.join(__import__("conftest").GOLDEN, "philox4x32_10_kat.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        w = [int(x, 16) for x in r]
        assert list(oracle.philox4x32_10(w[0:4], w[4:6])) == w[6:10]
    assert ex is not None


def test_keep_threshold():
    assert oracle.keep_threshold(0.01) == 42_949_673
    assert oracle.keep_threshold(1.0) == 1 << 32
    assert oracle.keep_threshold(0.5) == 1 << 31


# ---------------------------------------------------------------------- DCD

RING = (1.0 / 3.0, 1.0 / 3.0, 1.0 / 3.0)


def _ring_matrix(n, w):
    W = np.zeros((n, n))
    for i in range(n):
        W[i, (i - 1) % n] += w[0]
        W[i, i] += w[1]
        W[i, (i + 1) % n] += w[2]
    return W


def test_keep_all_is_dpsgd():
    """p = 1 (C is the identity): the model becomes x_half = W x - gamma g, which
    numpy computes in fp64 with the ring's mixing matrix."""
    rng = np.random.default_rng(4)
    n, d, gamma = 6, 1001, 0.1
    w = np.float32(RING).astype(np.float64)
    x = rng.standard_normal((n, d)).astype(np.float32)
    g = rng.standard_normal((n, d)).astype(np.float32)
    x_half = _ring_matrix(n, w) @ x.astype(np.float64) - np.float64(np.float32(gamma)) * g
    got = oracle.dcd_step(x.copy(), g, RING, gamma, 1.0, 123, 0)
    scale = np.maximum(np.abs(x_half), np.abs(x)).max()
    assert np.abs(got - x_half).max() <= 8 * np.spacing(np.float32(scale))


def test_left_weight_takes_the_previous_node():
    """w_ring is (left, self, right) with node i's left neighbour i - 1 (mod n):
    with W = (1, 0, 0), p = 1 and g = 0 every node's model becomes its left
    neighbour's, exactly (small integers: every sum and difference is exact);
    with W = (0, 0, 1) its right neighbour's."""
    n, d = 5, 37
    x = np.arange(n * d, dtype=np.float32).reshape(n, d) % 97
    g = np.zeros((n, d), np.float32)
    left = oracle.dcd_step(x.copy(), g, (1.0, 0.0, 0.0), 0.1, 1.0, 9, 0)
    np.testing.assert_array_equal(left, np.roll(x, 1, axis=0))
    right = oracle.dcd_step(x.copy(), g, (0.0, 0.0, 1.0), 0.1, 1.0, 9, 0)
    np.testing.assert_array_equal(right, np.roll(x, -1, axis=0))


def test_single_node_is_sgd():
    rng = np.random.default_rng(5)
    d = 777
    x = rng.standard_normal((1, d)).astype(np.float32)
    g = rng.standard_normal((1, d)).astype(np.float32)
    got = oracle.dcd_step(x.copy(), g, (0.0, 1.0, 0.0), 0.05, 1.0, 9, 3)
    want = x[0].astype(np.float64) - np.float64(np.float32(0.05)) * g[0]
    # a few fp32 roundings, each at most half an ulp of the largest operand
    assert np.all(np.abs(got[0] - want) <= 2 * ulp32(np.maximum(np.abs(want), np.abs(x[0]))))


def test_random_sparsification_mask_and_scale():
    """From x = 0 on one node with W = (0, 1, 0), z = -gamma g and the new model
    is exactly C(z): kept entries are z/p, the others 0.  The kept set is the
    set of words of Philox(counter (e/4, node, t, 0), key seed) below
    round(p 2^32); its size is within 5 sigma of the binomial mean, and alpha^2 =
    ||z - C(z)||^2 / ||z||^2 is near its expectation (1 - p) / p."""
    rng = np.random.default_rng(6)
    d, p, t, seed = 200_000, 0.01, 7, 0xDEADBEEF12345678
    g = rng.standard_normal((1, d)).astype(np.float32)
    x = np.zeros((1, d), np.float32)
    cz = oracle.dcd_step(x, g, (0.0, 1.0, 0.0), 0.1, p, seed, t)[0]
    z = -(np.float32(0.1) * g[0])
    kept = cz != 0
    thr = oracle.keep_threshold(p)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for e in rng.choice(d, size=300, replace=False):
        word = oracle.philox4x32_10([e // 4, 0, t, 0], key)[e % 4]
        assert bool(word < thr) == bool(kept[e])
    np.testing.assert_array_equal(cz[kept], z[kept] * np.float32(1.0 / p))
    mean, sd = d * p, np.sqrt(d * p * (1 - p))
    assert abs(kept.sum() - mean) < 5 * sd
    alpha2 = np.sum((z.astype(np.float64) - cz) ** 2) / np.sum(z.astype(np.float64) ** 2)
    assert abs(alpha2 - (1 - p) / p) < 0.15 * (1 - p) / p


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_replica_identity(n):
    """Every node keeps its own copies of its neighbours' models and applies the
    C(z_j) it receives; starting equal, those copies stay bit-identical to the
    single shared array xhat (DCD-PSGD step 3)."""
    rng = np.random.default_rng(n)
    d, T, gamma, p, seed = 53, 6, 0.1, 0.3, 77
    x0 = rng.standard_normal(d).astype(np.float32)
    xhat = np.tile(x0, (n, 1)).copy()
    rep = np.tile(x0, (n, n, 1)).copy()
    for t in range(T):
        g = rng.standard_normal((n, d)).astype(np.float32)
        oracle.dcd_step(xhat, g, RING, gamma, p, seed, t)
        oracle.dcd_step_replicas(rep, g, RING, gamma, p, seed, t)
        for i in range(n):
            for j in {i, (i - 1) % n, (i + 1) % n}:
                np.testing.assert_array_equal(rep[i, j], xhat[j])


def test_nodes_read_the_previous_iterate():
    """The step is a function of the old models only: permuting the order in
    which a reference computes nodes cannot matter, so node i's result equals a
    one-node evaluation on the old neighbours."""
    rng = np.random.default_rng(8)
    n, d = 4, 64
    x = rng.standard_normal((n, d)).astype(np.float32)
    g = rng.standard_normal((n, d)).astype(np.float32)
    full = oracle.dcd_step(x.copy(), g, RING, 0.1, 1.0, 1, 0)
    for i in range(n):
        l, r = (i - 1) % n, (i + 1) % n
        acc = np.float32(RING[0]) * x[l]
        acc = acc + np.float32(RING[1]) * x[i]
        acc = acc + np.float32(RING[2]) * x[r]
        xh = acc - np.float32(0.1) * g[i]
        want = x[i] + (xh - x[i])
        np.testing.assert_array_equal(full[i], want)


def test_window_matches_full_step():
    """A column window computed on its own equals the same columns of the full step."""
    rng = np.random.default_rng(12)
    n, d = 5, 2000
    x = rng.standard_normal((n, d)).astype(np.float32)
    g = rng.standard_normal((n, d)).astype(np.float32)
    full = oracle.dcd_step(x.copy(), g, RING, 0.1, 0.2, 99, 4)
    for e0, e1 in [(0, 7), (13, 500), (1999, 2000), (1024, 2000)]:
        win = oracle.dcd_step_window(np.ascontiguousarray(x[:, e0:e1]), g[:, e0:e1], RING, 0.1, 0.2, 99, 4, e0)
        np.testing.assert_array_equal(win, full[:, e0:e1])


# ------------------------------------------------------------------ ECD-PSGD

def _ecd_state(rng, n, d):
    x_prev = (rng.standard_normal((n, d)) * 1e-2).astype(np.float32)
    x = (x_prev + rng.standard_normal((n, d)) * 1e-3).astype(np.float32)
    g = (rng.standard_normal((n, d)) * 1e-3).astype(np.float32)
    return x, x_prev, g


def test_ecd_t2_identity_compression_is_d_psgd():
    """At t = 2 the extrapolation weights are (0, 1) and the estimate weights
    (0, 1), so with C the identity the estimate is x_t itself and the step is
    D-PSGD: W x_t - gamma g, added left, self, right in fp32."""
    rng = np.random.default_rng(0)
    n, d = 5, 777
    x, x_prev, g = _ecd_state(rng, n, d)
    xt = rng.standard_normal((n, d)).astype(np.float32)  # the old estimate is weighted by 0
    w = np.array([0.25, 0.5, 0.25], np.float32)
    new, est = oracle.ecd_step(x, x_prev.copy(), xt, g, w, np.float32(0.1), 1.0, 5, 2)
    np.testing.assert_array_equal(est, x)
    want = (w[0] * np.roll(x, 1, axis=0) + w[1] * x) + w[2] * np.roll(x, -1, axis=0)
    want = want - np.float32(0.1) * g
    np.testing.assert_array_equal(new, want.astype(np.float32))


@pytest.mark.parametrize("t", [1, 3, 7, 40])
def test_ecd_estimate_tracks_the_model_without_compression(t):
    """With C the identity and a consistent estimate (xt = x_{t-1}),
    equations (3) and (4) give xt_t = x_t up to fp32 rounding."""
    rng = np.random.default_rng(t)
    n, d = 3, 4000
    x, x_prev, g = _ecd_state(rng, n, d)
    xt = x_prev.copy()
    _, est = oracle.ecd_step(x, x_prev.copy(), xt, g, np.array([1 / 3] * 3, np.float32), np.float32(0.1), 1.0, 9, t)
    # the terms are O(t |x|), so the rounding error scales with t
    assert np.max(np.abs(est - x)) <= 4 * t * np.finfo(np.float32).eps * np.max(np.abs(x))


def test_ecd_self_weight_one_is_sgd():
    rng = np.random.default_rng(3)
    x, x_prev, g = _ecd_state(rng, 4, 1000)
    new, _ = oracle.ecd_step(x, x_prev.copy(), x_prev.copy(), g, np.array([0, 1, 0], np.float32),
                             np.float32(0.05), 0.01, 11, 6)
    np.testing.assert_array_equal(new, x - np.float32(0.05) * g)


def test_ecd_t2_keep_mask_from_philox():
    """At t = 2, xt = C(x_t): x_t / p where Philox keeps it, 0 elsewhere; the
    counter is (e / 4, node, t, e / 2^34), the word e mod 4, key = the seed."""
    rng = np.random.default_rng(4)
    n, d, p, seed = 2, 2048, 0.25, 0x1234_5678_9ABC_DEF0
    x, x_prev, g = _ecd_state(rng, n, d)
    _, est = oracle.ecd_step(x, x_prev.copy(), np.zeros((n, d), np.float32), g, np.array([1 / 3] * 3, np.float32),
                             np.float32(0.1), p, seed, 2)
    thr = oracle.keep_threshold(p)
    key = (seed & 0xFFFFFFFF, seed >> 32)
    for i in range(n):
        for e in range(0, d, 4):
            words = oracle.philox4x32_10((e // 4, i, 2, 0), key)
            for q in range(4):
                want = np.float32(x[i, e + q] * np.float32(1 / p)) if words[q] < thr else np.float32(0)
                assert est[i, e + q] == want
