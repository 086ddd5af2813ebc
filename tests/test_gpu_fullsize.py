"""Full-size workloads, in the launch configuration the benchmark times.

Every learner is compared with the oracle element by element: learners
share nothing, so learner k of a K-learner call must equal the oracle run
on learner k alone, and the K oracle runs go to a thread pool (the oracle's
C calls release the GIL).  DCD columns are independent, so the ring is
checked over every column in windows.  Properties that hold at any size
are checked beside the oracle: exact counts, ascending in-segment indices,
every sent magnitude at least every unsent one in its segment (ties to the
lower index), and the masked state (DGC); the selection rule on sampled
bins (AdaComp).
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
from conftest import rel_err
from gradient_compression_sgd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def oracle_map(fn, items):
    """fn over items in threads (the oracle's C calls run in parallel)."""
    with ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        return list(ex.map(fn, items))


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
    every learner's message, u and v against the oracle, learners 0 and K-1
    also against the properties; then the sparse average of the K messages
    against the oracle."""
    import torch
    gc = cuda_lib
    w = wl.workload(config)
    off, K, N = w.offsets, w.learners, w.n
    d = gc.DGC(off, K, w.density, w.momentum)
    u = torch.zeros((K, N), device="cuda")
    v = torch.zeros((K, N), device="cuda")
    u_o = np.zeros((K, N), np.float32)  # the oracle's state, learner by learner
    v_o = np.zeros((K, N), np.float32)
    for t in range(2):
        G = wl.gradients(w, t, device="cuda")
        u_prev, v_prev = u.clone(), v.clone()
        out, totals = d(G, u, v)
        torch.cuda.synchronize()
        st = d.stats()
        assert st["hint_failed"] == 0 and st["raw_global"] == 0, st  # the fast paths served every segment
        Gh = G.cpu().numpy()
        idx_g = gc.pair_indices(out).cpu().numpy()
        val_g = gc.pair_values(out).cpu().numpy()
        counts = d.counts.cpu().numpy()
        ug, vg = u.cpu().numpy(), v.cpu().numpy()

        def learner(k):
            idx_o, val_o, counts_o, _ = oracle.dgc_step(off, Gh[k:k + 1], u_o[k:k + 1], v_o[k:k + 1], w.density,
                                                        w.momentum, cap=d.cap)
            return idx_o[0], val_o[0], counts_o[0]

        for k, (idx_o, val_o, counts_o) in enumerate(oracle_map(learner, range(K))):
            n_k = int(counts_o.sum())
            np.testing.assert_array_equal(counts[k], counts_o, err_msg=f"t={t} k={k}")
            np.testing.assert_array_equal(idx_g[k, :n_k], idx_o[:n_k].astype(np.int64), err_msg=f"t={t} k={k}")
            assert rel_err(val_g[k, :n_k], val_o[:n_k]) <= 1e-6, (t, k)
            assert rel_err(ug[k], u_o[k]) <= 1e-6, (t, k)
            assert rel_err(vg[k], v_o[k]) <= 1e-6, (t, k)
        # learners 0 and K-1: properties; the pre-mask velocity is v_after plus the sent values
        for k in sorted({0, K - 1}):
            va = vg[k]
            ua = ug[k]
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
            g = Gh[k][sample]
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
    K = 8, two steps; every learner's message, scales and residue against the
    oracle (the residue relative to max(|G|, |R|), G = R_prev + dW in fp32);
    the selection rule checked for every learner on sampled bins."""
    import torch
    gc = cuda_lib
    w = wl.workload(3)
    off, K, N = w.offsets, w.learners, w.n
    cap = N // 8
    a = gc.AdaComp(off, w.lt, K, cap)
    R = torch.zeros((K, N), device="cuda")
    R_o = np.zeros((K, N), np.float32)  # the oracle's residue, learner by learner
    for t in range(2):
        dW = wl.gradients(w, t, device="cuda")
        R_prev = R.clone()
        out, totals = a(dW, R)
        torch.cuda.synchronize()
        check_adacomp_bins(gc, a, off, w.lt, dW, R_prev, R, out, totals, seed=t)
        assert np.all(totals.cpu().numpy() <= cap)
        dWh = dW.cpu().numpy()
        Rp = R_prev.cpu().numpy()
        Rg = R.cpu().numpy()
        counts_g, scales_g = a.counts.cpu().numpy(), a.scales.cpu().numpy()
        idx_g = gc.pair_indices(out).cpu().numpy()
        val_g = gc.pair_values(out).cpu().numpy()

        def learner(k):
            idx_o, val_o, counts_o, scales_o, totals_o = oracle.adacomp_step(off, w.lt, dWh[k:k + 1],
                                                                             R_o[k:k + 1], cap=cap)
            return idx_o[0], val_o[0], counts_o[0], scales_o[0], int(totals_o[0])

        for k, (idx_o, val_o, counts_o, scales_o, n_k) in enumerate(oracle_map(learner, range(K))):
            np.testing.assert_array_equal(counts_g[k], counts_o, err_msg=f"t={t} k={k}")
            assert rel_err(scales_g[k], scales_o) <= 1e-6, (t, k)
            np.testing.assert_array_equal(idx_g[k, :n_k], idx_o[:n_k].astype(np.int64), err_msg=f"t={t} k={k}")
            assert rel_err(val_g[k, :n_k], val_o[:n_k]) <= 1e-6, (t, k)
            G = Rp[k] + dWh[k]
            denom = np.maximum(np.maximum(np.abs(G), np.abs(R_o[k])), np.finfo(np.float32).tiny)
            assert float((np.abs(Rg[k].astype(np.float64) - R_o[k]) / denom).max(initial=0.0)) <= 1e-6, (t, k)
    avg = torch.empty(N, device="cuda")
    gc.sparse_average(out, totals, N, avg)
    torch.cuda.synchronize()
    want = oracle.sparse_average(gc.pair_indices(out).cpu().numpy().astype(np.uint32),
                                 gc.pair_values(out).cpu().numpy(), totals.cpu().numpy(), N)
    assert rel_err(avg.cpu().numpy(), want) <= 1e-5


def test_dcd_full_size(cuda_lib):
    """Ring of 8 nodes, 25.6M values each, 3 iterations; every column against
    the oracle's step, run on 64 column windows (columns are independent;
    the keep draws take the absolute column, so the windows' boundaries do
    not matter), bit for bit after every iteration."""
    import torch
    gc = cuda_lib
    w = wl.workload(5)
    n, D = w.learners, w.n
    x = wl.dcd_initial_model(w, device="cuda")
    seed = wl.dcd_seed(w)
    cuts = [D * j // 64 for j in range(65)]
    windows = list(zip(cuts[:-1], cuts[1:]))
    xh = x.cpu().numpy()
    x_win = [np.ascontiguousarray(xh[:, a:b]) for a, b in windows]
    del xh
    for t in range(3):
        g = torch.stack([wl.gradient(w, i, t, device="cuda") for i in range(n)])
        gc.dcd_step(x, g, w.ring_w, w.gamma, w.keep_p, seed, t)
        gh = g.cpu().numpy()
        oracle_map(lambda j: oracle.dcd_step_window(x_win[j], np.ascontiguousarray(gh[:, windows[j][0]:windows[j][1]]),
                                                    w.ring_w, w.gamma, w.keep_p, seed, t, windows[j][0]),
                   range(len(windows)))
        torch.cuda.synchronize()
        xg = x.cpu().numpy()
        for j, (a, b) in enumerate(windows):
            np.testing.assert_array_equal(xg[:, a:b], x_win[j], err_msg=f"t={t} columns [{a}, {b})")
