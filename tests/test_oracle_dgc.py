"""Pins of the oracle's Deep Gradient Compression step (CPU only).

Each test checks the oracle against something other than itself: a worked
example, brute force over all subsets, closed forms of the momentum-corrected
accumulation in exact rational arithmetic, and numpy's norm routine.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle
from conftest import f32


def _step(off, G, u, v, density, m, clip=0.0, nodes=1):
    return oracle.dgc_step(off, G[None, :] if G.ndim == 1 else G, u, v, density, m, clip, nodes)


def test_worked_example(golden):
    ex = golden("dgc_worked_example.txt")
    sizes = [int(x) for x in ex["sizes"]]
    off = np.array([0, sizes[0], sizes[0] + sizes[1]], dtype=np.int64)
    N = off[-1]
    u = np.zeros((1, N), np.float32)
    v = np.zeros((1, N), np.float32)
    for t in (1, 2):
        idx, val, counts, cs = oracle.dgc_step(off, f32(ex[f"grad{t}"])[None], u, v,
                                               float(ex["density"][0]), float(ex["momentum"][0]))
        tot = counts.sum()
        assert list(idx[0, :tot]) == [int(x) for x in ex[f"sent{t}_idx"]]
        np.testing.assert_array_equal(val[0, :tot], f32(ex[f"sent{t}_val"]))
        np.testing.assert_array_equal(u[0], f32(ex[f"u{t}"]))
        np.testing.assert_array_equal(v[0], f32(ex[f"v{t}"]))
        assert cs[0] == 1.0


def _brute_force_topk(vals, k):
    """The unique k-subset S with |v_i| > |v_j|, or equal and i < j, for i in S, j not in S."""
    n = len(vals)
    found = []
    for S in itertools.combinations(range(n), k):
        Sset = set(S)
        ok = all(abs(vals[i]) > abs(vals[j]) or (abs(vals[i]) == abs(vals[j]) and i < j)
                 for i in Sset for j in range(n) if j not in Sset)
        if ok:
            found.append(S)
    assert len(found) == 1, found
    return list(found[0])


@pytest.mark.parametrize("seed", range(40))
def test_topk_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 10))
    pool = np.array([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, -3.0, 3.0], np.float32)
    G = rng.choice(pool, size=n).astype(np.float32)
    density = float(rng.choice([0.1, 0.25, 0.5, 0.75, 1.0]))
    k = oracle.dgc_k(density, n)
    u = np.zeros((1, n), np.float32)
    v = np.zeros((1, n), np.float32)
    idx, val, counts, _ = _step(np.array([0, n], np.int64), G, u, v, density, 0.9)
    assert counts[0, 0] == k
    want = _brute_force_topk([float(x) for x in G], k)
    assert list(idx[0, :k]) == want
    # from a zero state the accumulated velocity equals the gradient
    np.testing.assert_array_equal(val[0, :k], G[want])
    # momentum factor masking: zero exactly where sent, untouched elsewhere
    rest = [i for i in range(n) if i not in want]
    assert np.all(u[0, want] == 0) and np.all(v[0, want] == 0)
    np.testing.assert_array_equal(u[0, rest], G[rest])
    np.testing.assert_array_equal(v[0, rest], G[rest])


def test_k_rule():
    # k = ceil(density * n) in fp64, at least 1, at most n
    assert oracle.dgc_k(0.001, 1_048_576) == 1049
    assert oracle.dgc_k(0.001, 1000) == 1
    assert oracle.dgc_k(0.001, 64) == 1
    assert oracle.dgc_k(0.001, 2_359_296) == 2360
    assert oracle.dgc_k(1.0, 7) == 7
    assert oracle.dgc_k(0.5, 0) == 0


def test_momentum_correction_closed_form():
    """With m = 1/2 and small integer gradients every fp32 operation is exact, so
    an entry that is never sent must follow the closed form of the corrected
    accumulation: u_T = sum_j m^(T-j) G_j and v_T = sum_j G_j (1 - m^(T-j+1)) / (1 - m).
    Entry 0 carries a huge gradient and is sent every step (k = 1), so it must
    restart from zero each step: sent_t = G_t at entry 0."""
    rng = np.random.default_rng(7)
    n, T, m = 16, 6, Fraction(1, 2)
    Gs = rng.integers(-8, 9, size=(T, n)).astype(np.float32)
    Gs[:, 0] = 1e6 * np.array([1, -1, 1, -1, 1, -1])[:T]
    u = np.zeros((1, n), np.float32)
    v = np.zeros((1, n), np.float32)
    off = np.array([0, n], np.int64)
    for t in range(T):
        idx, val, counts, _ = _step(off, Gs[t], u, v, 1.0 / n, 0.5)
        assert counts[0, 0] == 1 and idx[0, 0] == 0 and val[0, 0] == Gs[t, 0]
    for i in range(1, n):
        uT = sum(m ** (T - 1 - j) * Fraction(float(Gs[j, i])) for j in range(T))
        vT = sum(Fraction(float(Gs[j, i])) * (1 - m ** (T - j)) / (1 - m) for j in range(T))
        assert Fraction(float(u[0, i])) == uT
        assert Fraction(float(v[0, i])) == vT


def test_density_one_sends_the_gradient():
    """Sending everything resets u and v each step, so what is sent is G itself."""
    rng = np.random.default_rng(3)
    K, n = 2, 33
    off = np.array([0, 5, 5, 33], np.int64)  # includes an empty tensor
    u = np.zeros((K, n), np.float32)
    v = np.zeros((K, n), np.float32)
    for t in range(3):
        G = rng.standard_normal((K, n)).astype(np.float32)
        idx, val, counts, _ = oracle.dgc_step(off, G, u, v, 1.0, 0.9)
        assert list(counts[0]) == [5, 0, 28]
        for k in range(K):
            assert list(idx[k]) == list(range(n))
            np.testing.assert_array_equal(val[k], G[k])
        assert not u.any() and not v.any()


def test_zero_momentum_is_plain_residual_accumulation():
    """m = 0: v accumulates G and sent + residual conserves the total exactly
    (integer-valued gradients keep fp32 exact)."""
    rng = np.random.default_rng(11)
    n, T = 50, 8
    off = np.array([0, n], np.int64)
    u = np.zeros((1, n), np.float32)
    v = np.zeros((1, n), np.float32)
    total_sent = np.zeros(n, np.float64)
    total_grad = np.zeros(n, np.float64)
    for _ in range(T):
        G = rng.integers(-4, 5, size=n).astype(np.float32)
        idx, val, counts, _ = _step(off, G, u, v, 0.1, 0.0)
        total_sent[idx[0, :counts.sum()]] += val[0, :counts.sum()]
        total_grad += G
        np.testing.assert_array_equal(u[0][v[0] != 0], G[v[0] != 0])
    np.testing.assert_array_equal(total_sent + v[0], total_grad)


def test_clipping_norm_spans_every_tensor_of_a_learner():
    """The clipping norm is the learner's whole gradient, across tensors (DGC,
    Appendix C: the local gradient's L2 norm), and each learner has its own:
    the scale is thr / ||G_k|| over all of learner k's values (numpy's fp64
    norm), not over one tensor, and at density 1 what is sent has norm thr."""
    rng = np.random.default_rng(7)
    sizes = [1000, 3000, 96]
    off = np.array([0, 1000, 4000, 4096], np.int64)
    K, N = 2, 4096
    G = np.concatenate([rng.standard_normal((K, n)) * s for n, s in zip(sizes, (0.2, 0.01, 0.5))], axis=1)
    G = G.astype(np.float32)
    thr = 1.0
    u = np.zeros((K, N), np.float32)
    v = np.zeros((K, N), np.float32)
    _, val, _, cs = _step(off, G, u, v, 1.0, 0.0, clip=thr, nodes=1)
    for k in range(K):
        whole = np.linalg.norm(G[k].astype(np.float64))
        first = np.linalg.norm(G[k, :1000].astype(np.float64))
        assert whole > thr and abs(whole - first) > 0.1 * whole
        assert cs[k] == np.float32(thr / whole)
        sent = val[k].astype(np.float64)
        assert abs(np.linalg.norm(sent) - thr) <= 1e-6 * thr
    assert cs[0] != cs[1]


@pytest.mark.parametrize("nodes", [1, 4])
def test_local_gradient_clipping(nodes):
    """The scale is thr_k / ||G|| with thr_k = thr / sqrt(N) (Appendix C), from
    numpy's fp64 norm; it depends on G only (clipping happens before the
    gradient joins the accumulation), and the clipped gradient's norm is
    within fp32 rounding of thr_k."""
    rng = np.random.default_rng(nodes)
    n = 4096
    G = (rng.standard_normal(n) * 0.05).astype(np.float32)  # ||G|| ~ 3.2
    thr = 1.0
    thr_k = thr / np.sqrt(nodes)
    norm = np.linalg.norm(G.astype(np.float64))
    assert norm > thr_k
    off = np.array([0, n], np.int64)
    u = np.zeros((1, n), np.float32)
    v = np.zeros((1, n), np.float32)
    _, val, _, cs = _step(off, G, u, v, 1.0, 0.0, clip=thr, nodes=nodes)
    assert cs[0] == np.float32(thr_k / norm)
    Gc = G * cs[0]
    np.testing.assert_array_equal(val[0], Gc)  # density 1, zero state: what is sent is c*G
    assert np.linalg.norm(Gc.astype(np.float64)) <= thr_k * (1 + 1e-6)
    # with a non-zero state the scale is unchanged: it is a property of G alone
    u2 = rng.standard_normal((1, n)).astype(np.float32)
    v2 = rng.standard_normal((1, n)).astype(np.float32)
    _, val, _, cs2 = _step(off, G, u2, v2, 1.0, 0.9, clip=thr, nodes=nodes)
    assert cs2[0] == cs[0]
    # below the threshold nothing is scaled
    small = G * np.float32(0.01)
    _, val, _, cs3 = _step(off, small, np.zeros((1, n), np.float32), np.zeros((1, n), np.float32), 1.0, 0.0,
                           clip=thr, nodes=nodes)
    assert cs3[0] == 1.0
    np.testing.assert_array_equal(val[0], small)


def test_multi_learner_independence():
    """Learners share nothing: running K together equals running each alone."""
    rng = np.random.default_rng(5)
    off = np.array([0, 100, 130, 400], np.int64)
    K, n = 3, 400
    G = rng.standard_normal((K, n)).astype(np.float32)
    u = rng.standard_normal((K, n)).astype(np.float32)
    v = rng.standard_normal((K, n)).astype(np.float32)
    u0, v0 = u.copy(), v.copy()
    idx, val, counts, _ = oracle.dgc_step(off, G, u, v, 0.05, 0.9, 1.0, 2)
    for k in range(K):
        uk, vk = u0[k:k + 1].copy(), v0[k:k + 1].copy()
        i1, v1, c1, _ = oracle.dgc_step(off, G[k:k + 1], uk, vk, 0.05, 0.9, 1.0, 2)
        np.testing.assert_array_equal(i1[0], idx[k])
        np.testing.assert_array_equal(v1[0], val[k])
        np.testing.assert_array_equal(uk[0], u[k])
        np.testing.assert_array_equal(vk[0], v[k])


def test_sent_plus_residual_is_accumulation():
    """v_acc = v_new + sent, bit for bit, where v_acc is observed by running
    the same step with nothing extra sent (density small) on a copy."""
    rng = np.random.default_rng(9)
    off = np.array([0, 300, 1000], np.int64)
    n = 1000
    G = rng.standard_normal((1, n)).astype(np.float32)
    u = rng.standard_normal((1, n)).astype(np.float32)
    v = rng.standard_normal((1, n)).astype(np.float32)
    # v_acc from density 1 (everything sent, so the sent values are v_acc)
    _, vacc, _, _ = oracle.dgc_step(off, G, u.copy(), v.copy(), 1.0, 0.9)
    idx, val, counts, _ = oracle.dgc_step(off, G, u, v, 0.02, 0.9)
    tot = counts.sum()
    recon = v[0].copy()
    recon[idx[0, :tot]] += val[0, :tot]  # v is exactly 0 there
    np.testing.assert_array_equal(recon, vacc[0])


# ------------------------------------------------------- sampled threshold

def test_sampled_hand_example():
    """n = 20480, density 0.001 (k = 21), a 1 % sample: m = 192 values in 3
    blocks of 64 at stride 6826 ([0, 64), [6826, 6890), [13652, 13716));
    a = round(21 * 192 / 20480) = 0 -> 1, so tau is the largest sampled |v|
    (5.0, planted at 6830).  |v| >= 5.0 holds at 100 (6.0), 200 (7.0), 6830
    and 20000 (5.0, a tie with tau): 4 < 21 entries, all of them sent."""
    n = 20480
    G = np.full((1, n), 1e-3, np.float32)
    G[0, 6830] = 5.0
    G[0, 100] = 6.0
    G[0, 200] = -7.0
    G[0, 20000] = 5.0
    G[0, 300] = 4.9
    u = np.zeros((1, n), np.float32)
    v = np.zeros((1, n), np.float32)
    idx, val, counts, _ = oracle.dgc_step_sampled([0, n], G, u, v, 0.001, 0.01, 0.9)
    assert counts.tolist() == [[4]]
    assert idx[0, :4].tolist() == [100, 200, 6830, 20000]
    assert val[0, :4].tolist() == [6.0, -7.0, 5.0, 5.0]
    assert not v[0, [100, 200, 6830, 20000]].any() and not u[0, [100, 200, 6830, 20000]].any()
    assert v[0, 300] == np.float32(4.9) and u[0, 300] == np.float32(4.9)


def sampled_example(ex, name):
    n = int(ex[f"{name}_n"][0])
    G = np.full((1, n), float(ex[f"{name}_base"][0]), np.float32)
    if f"{name}_ramp" in ex:
        r = int(ex[f"{name}_ramp"][0])
        G[0, :r] = np.arange(1, r + 1, dtype=np.float32)
    G[0, [int(x) for x in ex[f"{name}_at"]]] = f32(ex[f"{name}_val"])
    return n, G


@pytest.mark.parametrize("name", ["A", "B", "C", "D"])
def test_sampled_small_tensor_examples(golden, name):
    """Hand-worked examples (tests/golden/dgc_sampled_small_examples.txt): a
    tensor of 6400 values sampled by one block, a density of 0.5 sampled, a
    sample of 20480 values, and a tensor whose 1 % sample is under one block
    selected exactly."""
    ex = golden("dgc_sampled_small_examples.txt")
    n, G = sampled_example(ex, name)
    u = np.zeros((1, n), np.float32)
    v = np.zeros((1, n), np.float32)
    idx, val, counts, _ = oracle.dgc_step_sampled([0, n], G, u, v, float(ex[f"{name}_density"][0]),
                                                  float(ex[f"{name}_frac"][0]), 0.9)
    want_idx = [int(x) for x in ex[f"{name}_sent_idx"]]
    c = len(want_idx)
    assert counts.tolist() == [[c]]
    assert idx[0, :c].tolist() == want_idx
    np.testing.assert_array_equal(val[0, :c], f32(ex[f"{name}_sent_val"]))
    assert not v[0, want_idx].any() and not u[0, want_idx].any()
    keep = np.ones(n, bool)
    keep[want_idx] = False
    np.testing.assert_array_equal(v[0, keep], G[0, keep])


def sample_blocks(n, frac):
    """Whole 64-value blocks in floor(frac * n) values (0: the tensor is exact)."""
    m = int(frac * n)
    return (m - m % 64) // 64


@pytest.mark.parametrize("frac", [0.001, 0.003, 0.01, 0.2])
def test_sampled_is_a_top_set_and_exact_when_full(frac):
    """Whatever the sample, the sent set is the top of |v| (everything sent is
    at least as large as everything kept); when it reaches k it is exactly
    the exact step's top-k; a tensor whose sample holds no whole 64-value
    block is exact."""
    rng = np.random.default_rng(int(frac * 1e4))
    sizes = [16384, 50000, 200000, 33333, 6400, 700]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    K, N = 2, int(off[-1])
    for step in range(3):
        G = (rng.standard_normal((K, N)) * rng.choice([1e-4, 1e-2], size=(K, 1))).astype(np.float32)
        u0 = rng.standard_normal((K, N)).astype(np.float32) * 1e-3
        v0 = rng.standard_normal((K, N)).astype(np.float32) * 1e-3
        us, vs = u0.copy(), v0.copy()
        ue, ve = u0.copy(), v0.copy()
        idx_s, val_s, cnt_s, _ = oracle.dgc_step_sampled(off, G, us, vs, 0.002, frac, 0.9)
        idx_e, val_e, cnt_e, _ = oracle.dgc_step(off, G, ue, ve, 0.002, 0.9)
        vacc = ve.copy()  # the accumulated v before masking: reconstruct from the exact run
        for k in range(K):
            vacc[k, idx_e[k, :cnt_e[k].sum()]] = val_e[k, :cnt_e[k].sum()]
        for k in range(K):
            ps, pe = 0, 0
            for s in range(len(sizes)):
                cs, ce = int(cnt_s[k, s]), int(cnt_e[k, s])
                assert cs <= ce
                sent = idx_s[k, ps:ps + cs].astype(np.int64)
                if sample_blocks(sizes[s], frac) == 0 or cs == ce:
                    np.testing.assert_array_equal(sent, idx_e[k, pe:pe + ce])
                mag = np.abs(vacc[k, off[s]:off[s + 1]])
                mask = np.zeros(sizes[s], bool)
                mask[sent - off[s]] = True
                if cs and (~mask).any():
                    assert mag[mask].min() >= mag[~mask].max()
                np.testing.assert_array_equal(val_s[k, ps:ps + cs], vacc[k, sent])
                ps, pe = ps + cs, pe + ce
        G_sent = vs.copy()
        assert not any(G_sent[k, idx_s[k, :cnt_s[k].sum()]].any() for k in range(K))


@pytest.mark.parametrize("density,frac", [(0.01, 0.01), (0.1, 0.001), (0.05, 0.01), (0.3, 0.003)])
def test_sampled_count_near_k(density, frac):
    """On i.i.d. normal values the sample's a-th largest sits near the
    population's k-th largest, so the sent count is close to k, never above
    it, and what was sent plus what stays in v is the accumulated v, bit for
    bit.  a = round(k m / n) is at least 20 in every case here, so the
    relative spread of the count is about 1 / sqrt(a) < 0.25."""
    rng = np.random.default_rng(int(density * 1000 + frac * 1e5))
    n = 1 << 20
    G = rng.standard_normal((1, n)).astype(np.float32)
    u = np.zeros((1, n), np.float32)
    v = np.zeros((1, n), np.float32)
    idx, val, counts, _ = oracle.dgc_step_sampled([0, n], G, u, v, density, frac, 0.0)
    k = oracle.dgc_k(density, n)
    m = sample_blocks(n, frac) * 64
    assert round(k * m / n) >= 20
    c = int(counts[0, 0])
    assert 0.5 * k <= c <= k
    recon = v[0].copy()
    recon[idx[0, :c].astype(np.int64)] += val[0, :c]
    np.testing.assert_array_equal(recon, G[0])


def test_sampled_hand_example_rank_above_one():
    """n = 20480, k = 21, a 50 % sample: m = 10240 values in 160 blocks of 64
    at stride 128 (positions 128 b .. 128 b + 63); a = round(21 * 10240 /
    20480) = 11.  Twelve sampled values 100..111 (at 128 b, b = 0..11) put tau
    at the 11th largest, 101; unsampled 150 (at 64) is above it, unsampled
    100.5 (at 65) below: 11 + 1 = 12 < 21 entries sent."""
    n = 20480
    G = np.full((1, n), 1e-3, np.float32)
    for b in range(12):
        G[0, 128 * b] = 100.0 + b
    G[0, 64] = 150.0
    G[0, 65] = 100.5
    u = np.zeros((1, n), np.float32)
    v = np.zeros((1, n), np.float32)
    idx, val, counts, _ = oracle.dgc_step_sampled([0, n], G, u, v, 0.001, 0.5, 0.9)
    want = sorted([128 * b for b in range(1, 12)] + [64])
    assert counts.tolist() == [[12]]
    assert idx[0, :12].tolist() == want
    assert v[0, 65] == np.float32(100.5) and v[0, 0] == np.float32(100.0)


# ------------------------------------------------ Nesterov momentum (reading)

def test_nesterov_worked_example(golden):
    """The hand-worked two-step example of the Nesterov reading (v takes m*u + G)."""
    ex = golden("dgc_nesterov_worked_example.txt")
    sizes = [int(x) for x in ex["sizes"]]
    off = np.array([0, sizes[0], sizes[0] + sizes[1]], dtype=np.int64)
    N = off[-1]
    u = np.zeros((1, N), np.float32)
    v = np.zeros((1, N), np.float32)
    for t in (1, 2):
        idx, val, counts, _ = oracle.dgc_step(off, f32(ex[f"grad{t}"])[None], u, v, float(ex["density"][0]),
                                              float(ex["momentum"][0]), nesterov=True)
        tot = counts.sum()
        assert list(idx[0, :tot]) == [int(x) for x in ex[f"sent{t}_idx"]]
        np.testing.assert_array_equal(val[0, :tot], f32(ex[f"sent{t}_val"]))
        np.testing.assert_array_equal(u[0], f32(ex[f"u{t}"]))
        np.testing.assert_array_equal(v[0], f32(ex[f"v{t}"]))


def test_nesterov_closed_form():
    """Exact rationals: an entry never sent follows u_T = sum_j m^(T-1-j) G_j and
    v_T = sum_j G_j (1 + m (1 - m^(T-j)) / (1 - m)); the entry sent every step
    restarts from zero, so it sends (1 + m) G_t."""
    rng = np.random.default_rng(11)
    n, T, m = 16, 6, Fraction(1, 2)
    Gs = rng.integers(-8, 9, size=(T, n)).astype(np.float32)
    Gs[:, 0] = 1e6 * np.array([1, -1, 1, -1, 1, -1])[:T]
    u = np.zeros((1, n), np.float32)
    v = np.zeros((1, n), np.float32)
    off = np.array([0, n], np.int64)
    for t in range(T):
        idx, val, counts, _ = oracle.dgc_step(off, Gs[t][None], u, v, 1.0 / n, 0.5, nesterov=True)
        assert counts[0, 0] == 1 and idx[0, 0] == 0 and val[0, 0] == np.float32(1.5) * Gs[t, 0]
    for i in range(1, n):
        uT = sum(m ** (T - 1 - j) * Fraction(float(Gs[j, i])) for j in range(T))
        vT = sum(Fraction(float(Gs[j, i])) * (1 + m * (1 - m ** (T - j)) / (1 - m)) for j in range(T))
        assert Fraction(float(u[0, i])) == uT
        assert Fraction(float(v[0, i])) == vT


def test_nesterov_with_zero_momentum_is_the_vanilla_step():
    """m = 0: u = G and v += G either way, so the two steps agree bit for bit."""
    rng = np.random.default_rng(12)
    off = np.array([0, 300, 1000, 1001], np.int64)
    G = rng.standard_normal((2, 1001)).astype(np.float32)
    runs = []
    for nest in (False, True):
        u = np.zeros((2, 1001), np.float32)
        v = np.full((2, 1001), 0.25, np.float32)
        out = oracle.dgc_step(off, G, u, v, 0.05, 0.0, nesterov=nest)
        runs.append((out, u, v))
    for a, b in zip(runs[0][0], runs[1][0]):
        np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(runs[0][1], runs[1][1])
    np.testing.assert_array_equal(runs[0][2], runs[1][2])
