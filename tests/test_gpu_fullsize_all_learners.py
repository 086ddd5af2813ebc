"""Full-size workloads, every learner against the oracle.

Learners share nothing, so the oracle runs each learner of the K-learner
call on its own (every gradient drawn by the CPU generator from the same
seed on both sides), all of them at once in spawned processes on the host's
cores (the pool starts before any GPU work in this test and never touches
the GPU).  Per learner and step: the message (indices and per-tensor counts
bit for bit, values bit for bit) and the state, u and v for DGC or the
residue for AdaComp, compared through two exact checksums of the fp32 bit
patterns (the sum of the 32-bit words and their position-weighted sum, both
in 64-bit integers), so no state has to cross between processes.
"""
import multiprocessing as mp
import os

import numpy as np
import pytest

from gradient_compression_sgd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

STEPS = 2


def checksums_np(a: np.ndarray) -> tuple[int, int]:
    w = a.reshape(-1).view(np.int32).astype(np.int64)
    pos = (np.arange(w.size, dtype=np.int64) % 1021) + 1
    return int(w.sum()), int((w * pos).sum())


def checksums_gpu(t) -> tuple[int, int]:
    import torch
    w = t.reshape(-1).view(torch.int32).to(torch.int64)
    pos = (torch.arange(w.numel(), dtype=torch.int64, device=w.device) % 1021) + 1
    return int(w.sum().item()), int((w * pos).sum().item())


def oracle_learner(args):
    """One learner's STEPS oracle steps, in a spawned process: per step the
    message and the state's checksums."""
    import oracle
    config, k, cap = args
    w = wl.workload(config)
    N = w.n
    out = []
    if w.method == "dgc":
        u = np.zeros((1, N), np.float32)
        v = np.zeros((1, N), np.float32)
        for t in range(STEPS):
            G = wl.gradient(w, k, t).numpy()[None]
            idx, val, counts, _ = oracle.dgc_step(w.offsets, G, u, v, w.density, w.momentum, cap=cap)
            n = int(counts.sum())
            out.append({"idx": idx[0, :n].copy(), "val": val[0, :n].copy(), "counts": counts[0].copy(),
                        "u": checksums_np(u), "v": checksums_np(v)})
    else:
        R = np.zeros((1, N), np.float32)
        for t in range(STEPS):
            dW = wl.gradient(w, k, t).numpy()[None]
            idx, val, counts, scales, totals = oracle.adacomp_step(w.offsets, w.lt, dW, R, cap=cap)
            n = int(totals[0])
            out.append({"idx": idx[0, :n].copy(), "val": val[0, :n].copy(), "counts": counts[0].copy(),
                        "scales": scales[0].copy(), "R": checksums_np(R)})
    return out


def run_oracles(config, K, cap):
    ctx = mp.get_context("spawn")
    with ctx.Pool(processes=min(K, max(1, os.cpu_count() or 1))) as pool:
        return pool.map(oracle_learner, [(config, k, cap) for k in range(K)])


@pytest.mark.parametrize("config", [2, 4])
def test_dgc_every_learner_full_size(cuda_lib, config):
    """ResNet-50 layout (K = 4, 25,557,032 values) and the GRU layout (K = 8,
    98,378,240 values), density 0.001, momentum 0.9, two steps."""
    import torch
    gc = cuda_lib
    w = wl.workload(config)
    off, K, N = w.offsets, w.learners, w.n
    cap = sum(gc.dgc_k(w.density, int(off[s + 1] - off[s])) for s in range(len(off) - 1))
    want = run_oracles(config, K, cap)  # before the first GPU call of this test
    d = gc.DGC(off, K, w.density, w.momentum)
    u = torch.zeros((K, N), device="cuda")
    v = torch.zeros((K, N), device="cuda")
    for t in range(STEPS):
        out, totals = d(wl.gradients(w, t).cuda(), u, v)  # the CPU generator's bytes, as the workers draw them
        torch.cuda.synchronize()
        idx = gc.pair_indices(out).cpu().numpy()
        val = gc.pair_values(out).cpu().numpy()
        counts = d.counts.cpu().numpy()
        for k in range(K):
            o = want[k][t]
            n = len(o["idx"])
            np.testing.assert_array_equal(counts[k], o["counts"], err_msg=f"counts, learner {k}, step {t}")
            np.testing.assert_array_equal(idx[k, :n], o["idx"].astype(np.int64), err_msg=f"learner {k}, step {t}")
            np.testing.assert_array_equal(val[k, :n].view(np.uint32), o["val"].view(np.uint32))
            assert checksums_gpu(u[k]) == o["u"], f"u, learner {k}, step {t}"
            assert checksums_gpu(v[k]) == o["v"], f"v, learner {k}, step {t}"


def test_adacomp_every_learner_full_size(cuda_lib):
    """LSTM (66,034,000 values, L_T = 500) + VGG-16 convs (14,714,688, L_T =
    50), K = 8, two steps with the residue carried."""
    import torch
    gc = cuda_lib
    w = wl.workload(3)
    K, N = w.learners, w.n
    a = gc.AdaComp(w.offsets, w.lt, K, N // 8)
    want = run_oracles(3, K, a.cap)
    R = torch.zeros((K, N), device="cuda")
    for t in range(STEPS):
        out, totals = a(wl.gradients(w, t).cuda(), R)
        torch.cuda.synchronize()
        idx = gc.pair_indices(out).cpu().numpy()
        val = gc.pair_values(out).cpu().numpy()
        counts = a.counts.cpu().numpy()
        scales = a.scales.cpu().numpy()
        for k in range(K):
            o = want[k][t]
            n = len(o["idx"])
            assert int(totals[k]) == n
            np.testing.assert_array_equal(counts[k], o["counts"], err_msg=f"counts, learner {k}, step {t}")
            np.testing.assert_array_equal(idx[k, :n], o["idx"].astype(np.int64), err_msg=f"learner {k}, step {t}")
            np.testing.assert_array_equal(scales[k].view(np.uint32), o["scales"].view(np.uint32))
            np.testing.assert_array_equal(val[k, :n].view(np.uint32), o["val"].view(np.uint32))
            assert checksums_gpu(R[k]) == o["R"], f"residue, learner {k}, step {t}"
