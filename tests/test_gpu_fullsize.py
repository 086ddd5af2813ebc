"""Full-size workloads, in the launch configuration the benchmark times.

At these sizes the oracle runs on one learner (learners share nothing, so
learner 0 of a K-learner call must equal the oracle run on learner 0 alone),
on sampled windows (DCD), and properties that hold at any size are checked
for every learner: exact counts, ascending in-segment indices, every sent
magnitude at least every unsent one in its segment (ties to the lower
index), and the masked state.
"""
import numpy as np
import pytest

import oracle
from conftest import rel_err
from gradient_compression_sgd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def check_topk_properties(gc, off, idx, val, counts, v_before_mask, v_after, u_after, density):
    """Properties of one learner's DGC message (numpy arrays)."""
    pos = 0
    for s in range(len(off) - 1):
        n = int(off[s + 1] - off[s])
        k = gc.dgc_k(density, n)
        assert counts[s] == k
        seg_idx = idx[pos:pos + k]
        pos += k
        if k == 0:
            continue
        assert np.all(np.diff(seg_idx) > 0) and seg_idx[0] >= off[s] and seg_idx[-1] < off[s + 1]
        vb = np.abs(v_before_mask[off[s]:off[s + 1]])
        sent = np.zeros(n, bool)
        sent[seg_idx - off[s]] = True
        if k < n:
            lo, hi = vb[sent].min(), vb[~sent].max()
            assert lo >= hi
            if lo == hi:  # ties: every sent tie precedes every unsent tie
                assert np.nonzero(sent & (vb == lo))[0].max() < np.nonzero(~sent & (vb == lo))[0].min()
        assert not np.any(v_after[off[s]:off[s + 1]][sent]) and not np.any(u_after[off[s]:off[s + 1]][sent])
    assert pos == int(np.sum(counts))


@pytest.mark.parametrize("config", [2, 4])
def test_dgc_full_size(cuda_lib, config):
    """ResNet-50 (25,557,032 values, 161 tensors, K = 4) and the GRU layout
    (98,378,240 values, K = 8) at density 0.001, momentum 0.9: two steps;
    learner 0 against the oracle, every learner against the properties; then
    the sparse average of the K messages against the oracle."""
    import torch
    gc = cuda_lib
    w = wl.workload(config)
    off, K, N = w.offsets, w.learners, w.n
    d = gc.DGC(off, K, w.density, w.momentum)
    u = torch.zeros((K, N), device="cuda")
    v = torch.zeros((K, N), device="cuda")
    u0 = np.zeros((1, N), np.float32)
    v0 = np.zeros((1, N), np.float32)
    for t in range(2):
        G = wl.gradients(w, t, device="cuda")
        u_prev, v_prev = u.clone(), v.clone()
        out, totals = d(G, u, v)
        torch.cuda.synchronize()
        st = d.stats()
        assert st["hint_failed"] == 0 and st["raw_global"] == 0, st  # the fast paths served every segment
        # learner 0 against the oracle
        idx_o, val_o, counts_o, _ = oracle.dgc_step(off, G[0:1].cpu().numpy(), u0, v0, w.density, w.momentum,
                                                    cap=d.cap)
        idx_g = gc.pair_indices(out).cpu().numpy()
        val_g = gc.pair_values(out).cpu().numpy()
        n0 = int(counts_o[0].sum())
        np.testing.assert_array_equal(idx_g[0, :n0], idx_o[0, :n0].astype(np.int64))
        assert rel_err(val_g[0, :n0], val_o[0, :n0]) <= 1e-6
        assert rel_err(u[0].cpu().numpy(), u0[0]) <= 1e-6
        assert rel_err(v[0].cpu().numpy(), v0[0]) <= 1e-6
        # every learner: properties; the pre-mask velocity is v_after plus the sent values
        counts = d.counts.cpu().numpy()
        for k in range(K):
            va = v[k].cpu().numpy()
            ua = u[k].cpu().numpy()
            n = int(counts[k].sum())
            vb = va.copy()
            vb[idx_g[k, :n]] = val_g[k, :n]
            check_topk_properties(gc, off, idx_g[k, :n], val_g[k, :n], counts[k], vb, va, ua, w.density)
            # unsent entries followed the corrected accumulation (checked on a sample)
            rng = np.random.default_rng(k)
            sample = rng.choice(N, size=4096, replace=False)
            sample = sample[va[sample] != 0]
            up = u_prev[k].cpu().numpy()[sample]
            vp = v_prev[k].cpu().numpy()[sample]
            g = G[k].cpu().numpy()[sample]
            un = np.float32(w.momentum) * up + g
            np.testing.assert_array_equal(ua[sample], un)
            np.testing.assert_array_equal(va[sample], vp + un)
    # sparse average of the K messages
    avg = torch.empty(N, device="cuda")
    gc.sparse_average(out, totals, N, avg)
    torch.cuda.synchronize()
    want = oracle.sparse_average(gc.pair_indices(out).cpu().numpy().astype(np.uint32),
                                 gc.pair_values(out).cpu().numpy(), totals.cpu().numpy(), N)
    np.testing.assert_array_equal(avg.cpu().numpy(), want)


def check_adacomp_bins(gc, a, off, lt, dW, R_prev, R, out, totals, seed, bins_per_learner=64):
    """Every learner, sampled bins: the sent indices of a bin are exactly those
    with |G + dW| >= the bin's max |G| and G != 0 (G = R_prev + dW in fp32),
    each sent as sign(G) * the segment's scale, and the residue is G minus
    what was sent.  Holds at any size; uses only the GPU's inputs."""
    K = dW.shape[0]
    counts = a.counts.cpu().numpy()
    scales = a.scales.cpu().numpy()
    tot = totals.cpu().numpy()
    rng = np.random.default_rng(seed)
    segs = [s for s in range(len(off) - 1) if off[s + 1] > off[s]]
    for k in range(K):
        n_k = int(tot[k])
        idx = gc.pair_indices(out)[k, :n_k].cpu().numpy()
        val = gc.pair_values(out)[k, :n_k].cpu().numpy()
        assert n_k == int(counts[k].sum()) and np.all(np.diff(idx) > 0)
        for _ in range(bins_per_learner):
            s = int(rng.choice(segs))
            L, n = int(lt[s]), int(off[s + 1] - off[s])
            b = int(rng.integers(0, (n + L - 1) // L))
            lo, hi = int(off[s]) + b * L, int(off[s]) + min((b + 1) * L, n)
            G = (R_prev[k, lo:hi] + dW[k, lo:hi]).cpu().numpy()
            d = dW[k, lo:hi].cpu().numpy()
            gmax = np.float32(np.nanmax(np.abs(np.where(np.isnan(G), 0, G)))) if hi > lo else np.float32(0)
            with np.errstate(invalid="ignore"):
                sel = (np.abs(G + d) >= gmax) & (gmax > 0) & (G != 0)
            a0, a1 = np.searchsorted(idx, [lo, hi])
            np.testing.assert_array_equal(idx[a0:a1], lo + np.nonzero(sel)[0], err_msg=f"k={k} s={s} bin={b}")
            q = np.where(G > 0, scales[k, s], -scales[k, s]).astype(np.float32)
            np.testing.assert_array_equal(val[a0:a1], q[sel])
            r_want = np.where(sel, G - q, G).astype(np.float32)
            np.testing.assert_array_equal(R[k, lo:hi].cpu().numpy(), r_want)


def test_adacomp_full_size(cuda_lib):
    """LSTM (66,034,000 values, L_T = 500) + VGG-16 convs (14,714,688, L_T = 50),
    K = 8, two steps; learner 0 against the oracle; selection rule checked for
    every learner on sampled bins."""
    import torch
    gc = cuda_lib
    w = wl.workload(3)
    off, K, N = w.offsets, w.learners, w.n
    cap = N // 8
    a = gc.AdaComp(off, w.lt, K, cap)
    R = torch.zeros((K, N), device="cuda")
    R0 = np.zeros((1, N), np.float32)
    for t in range(2):
        dW = wl.gradients(w, t, device="cuda")
        R_prev = R.clone()
        out, totals = a(dW, R)
        torch.cuda.synchronize()
        check_adacomp_bins(gc, a, off, w.lt, dW, R_prev, R, out, totals, seed=t)
        idx_o, val_o, counts_o, scales_o, totals_o = oracle.adacomp_step(off, w.lt, dW[0:1].cpu().numpy(), R0,
                                                                         cap=cap)
        np.testing.assert_array_equal(a.counts[0].cpu().numpy(), counts_o[0])
        assert rel_err(a.scales[0].cpu().numpy(), scales_o[0]) <= 1e-6
        n0 = int(totals_o[0])
        np.testing.assert_array_equal(gc.pair_indices(out)[0, :n0].cpu().numpy(), idx_o[0, :n0].astype(np.int64))
        assert rel_err(gc.pair_values(out)[0, :n0].cpu().numpy(), val_o[0, :n0]) <= 1e-6
        assert np.all(totals.cpu().numpy() <= cap)
    avg = torch.empty(N, device="cuda")
    gc.sparse_average(out, totals, N, avg)
    torch.cuda.synchronize()
    want = oracle.sparse_average(gc.pair_indices(out).cpu().numpy().astype(np.uint32),
                                 gc.pair_values(out).cpu().numpy(), totals.cpu().numpy(), N)
    assert rel_err(avg.cpu().numpy(), want) <= 1e-5


def test_dcd_full_size(cuda_lib):
    """Ring of 8 nodes, 25.6M values each, 3 iterations; four 4096-column
    windows (including the last) against the oracle's windowed step."""
    import torch
    gc = cuda_lib
    w = wl.workload(5)
    n, D = w.learners, w.n
    x = wl.dcd_initial_model(w, device="cuda")
    seed = wl.dcd_seed(w)
    windows = [(0, 4096), (12_345_678, 12_349_774), (D - 4096, D), (777, 4873)]
    x_win = [x[:, a:b].cpu().numpy().copy() for a, b in windows]
    for t in range(3):
        g = torch.stack([wl.gradient(w, i, t, device="cuda") for i in range(n)])
        gc.dcd_step(x, g, w.ring_w, w.gamma, w.keep_p, seed, t)
        for j, (a, b) in enumerate(windows):
            oracle.dcd_step_window(x_win[j], np.ascontiguousarray(g[:, a:b].cpu().numpy()), w.ring_w, w.gamma,
                                   w.keep_p, seed, t, a)
    torch.cuda.synchronize()
    for j, (a, b) in enumerate(windows):
        np.testing.assert_array_equal(x[:, a:b].cpu().numpy(), x_win[j])
