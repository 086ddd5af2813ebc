"""Pins of the oracle's AdaComp step (CPU only): a hand-worked example, the
special cases L_T = 1 and L_T = n, the scale against numpy's per-bin maxima,
bin locality, and residue conservation over steps."""
import numpy as np
import pytest

import oracle
from conftest import f32, ulp32


def test_worked_example(golden):
    ex = golden("adacomp_worked_example.txt")
    sizes = [int(x) for x in ex["sizes"]]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    R = f32(ex["R"])[None].copy()
    idx, val, counts, scales, totals = oracle.adacomp_step(off, [int(x) for x in ex["lt"]], f32(ex["dW"])[None], R)
    tot = int(totals[0])
    assert list(idx[0, :tot]) == [int(x) for x in ex["sent_idx"]]
    np.testing.assert_array_equal(val[0, :tot], f32(ex["sent_val"]))
    assert list(counts[0]) == [int(x) for x in ex["counts"]]
    np.testing.assert_array_equal(scales[0], f32(ex["scales"]))
    np.testing.assert_array_equal(R[0], f32(ex["R_new"]))


def _rand(rng, shape, scale=1.0):
    return (rng.laplace(0.0, scale, size=shape)).astype(np.float32)


@pytest.mark.parametrize("seed", range(5))
def test_single_element_bins(seed):
    """L_T = 1: each entry is its own bin, so it is sent iff |G + dW| >= |G| and G != 0."""
    rng = np.random.default_rng(seed)
    n = 257
    dW = _rand(rng, (1, n))
    R = _rand(rng, (1, n))
    R[0, ::7] = -dW[0, ::7]  # some G == 0 exactly
    G = R[0] + dW[0]
    H = G + dW[0]
    want = np.nonzero((np.abs(H) >= np.abs(G)) & (np.abs(G) > 0))[0]
    idx, val, counts, scales, totals = oracle.adacomp_step([0, n], [1], dW, R)
    assert list(idx[0, :totals[0]]) == list(want)
    # scale is the mean |G| over all entries
    assert scales[0, 0] == np.float32(np.abs(G.astype(np.float64)).mean())


@pytest.mark.parametrize("seed", range(5))
def test_one_bin_layer(seed):
    """L_T = n: one bin, the scale is max |G| and the test is |G + dW| >= max |G|."""
    rng = np.random.default_rng(100 + seed)
    n = 300
    dW = _rand(rng, (1, n))
    R = _rand(rng, (1, n), 3.0)
    G = R[0] + dW[0]
    gmax = np.abs(G).max()
    want = np.nonzero((np.abs(G + dW[0]) >= gmax) & (G != 0))[0]
    idx, val, counts, scales, totals = oracle.adacomp_step([0, n], [n], dW, R)
    assert scales[0, 0] == gmax
    assert list(idx[0, :totals[0]]) == list(want)
    np.testing.assert_array_equal(val[0, :totals[0]], np.sign(G[want]) * gmax)


@pytest.mark.parametrize("L", [2, 3, 50, 64, 500])
def test_scale_is_mean_of_bin_maxima_and_selection_is_per_bin(L):
    rng = np.random.default_rng(L)
    sizes = [1000, 37, 0, 2048]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    N = off[-1]
    K = 2
    dW = _rand(rng, (K, N), 1e-3)
    R = _rand(rng, (K, N), 1e-3)
    R0 = R.copy()
    idx, val, counts, scales, totals = oracle.adacomp_step(off, [L] * len(sizes), dW, R)
    for k in range(K):
        got = set(int(i) for i in idx[k, :totals[k]])
        pos = 0
        for s, n in enumerate(sizes):
            if n == 0:
                assert counts[k, s] == 0
                continue
            G = R0[k, off[s]:off[s + 1]] + dW[k, off[s]:off[s + 1]]
            nb = -(-n // L)
            pad = np.full(nb * L, -1.0, np.float32)
            pad[:n] = np.abs(G)
            bmax = pad.reshape(nb, L).max(axis=1)
            assert scales[k, s] == np.float32(bmax.astype(np.float64).mean())
            H = G + dW[k, off[s]:off[s + 1]]
            m = np.repeat(bmax, L)[:n]
            sel = (np.abs(H) >= m) & (m > 0) & (G != 0)
            want = set((off[s] + np.nonzero(sel)[0]).tolist())
            assert want == {i for i in got if off[s] <= i < off[s + 1]}
            assert counts[k, s] == sel.sum()
            # residue: exact where not sent; where sent it is G - q correctly
            # rounded (the difference of two fp32 values is exact in fp64)
            Rn = R[k, off[s]:off[s + 1]]
            np.testing.assert_array_equal(Rn[~sel], G[~sel])
            q = np.sign(G[sel]) * scales[k, s]
            exact = G[sel].astype(np.float64) - q.astype(np.float64)
            assert np.all(np.abs(Rn[sel] - exact) <= 0.5 * ulp32(Rn[sel]))
            np.testing.assert_array_equal(val[k, pos:pos + sel.sum()], q)
            pos += sel.sum()


def test_bin_locality():
    """Changing the gradient inside one bin changes nothing outside it except
    the layer's scale (selection needs no global sort)."""
    rng = np.random.default_rng(1)
    n, L = 1000, 50
    dW = _rand(rng, (1, n))
    R = _rand(rng, (1, n))
    a = oracle.adacomp_step([0, n], [L], dW, R.copy())
    dW2 = dW.copy()
    dW2[0, 300:350] = _rand(rng, (50,), 5.0)
    b = oracle.adacomp_step([0, n], [L], dW2, R.copy())
    sa = set(a[0][0, :a[4][0]].tolist())
    sb = set(b[0][0, :b[4][0]].tolist())
    outside = lambda S: {i for i in S if not 300 <= i < 350}
    assert outside(sa) == outside(sb)


def test_residue_carries_unsent_mass():
    """Over many steps, everything sent plus the final residue equals the sum of
    all new gradients, up to fp32 rounding of the per-step adds."""
    rng = np.random.default_rng(2)
    n, T = 2000, 20
    R = np.zeros((1, n), np.float32)
    sent = np.zeros(n, np.float64)
    total = np.zeros(n, np.float64)
    for _ in range(T):
        dW = _rand(rng, (1, n), 1e-2)
        idx, val, counts, scales, totals = oracle.adacomp_step([0, n], [50], dW, R)
        np.add.at(sent, idx[0, :totals[0]].astype(np.int64), val[0, :totals[0]].astype(np.float64))
        total += dW[0]
    err = np.abs(sent + R[0] - total)
    assert err.max() < 1e-6 * T


def test_capacity_overflow_reports_total():
    n = 100
    dW = np.ones((1, n), np.float32)
    R = np.zeros((1, n), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.adacomp_step([0, n], [10], dW, R, cap=5)
