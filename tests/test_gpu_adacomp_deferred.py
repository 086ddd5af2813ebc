"""AdaComp with the residue fix-up deferred to the next call
(adacomp_compress_deferred, adacomp_settle) against adacomp_compress and the
oracle ("AdaComp ...", Proposed method).

The deferred calls make the same fp32 operations in the same order, only at
another time, so every message word, count, scale and total must equal the
eager call's bit for bit at every step, and the residue after a settle must
equal the eager residue bit for bit.  The eager path is pinned to the oracle
by tests/test_gpu_adacomp_average_dcd.py; here the settled residue and the
messages are also checked against the oracle directly on small cases.
"""
import numpy as np
import pytest

import oracle
from conftest import rel_err
from gradient_compression_sgd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def words(t):
    import torch
    return t.contiguous().view(torch.int32).cpu().numpy()


def shifted(a, offset):
    import torch
    flat = torch.zeros(a.size + offset, dtype=torch.float32, device="cuda")
    view = flat[offset:].view(a.shape)
    view.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return view


def compare_step(gc, eager, deferred, t):
    tot_e, tot_d = words(eager.totals), words(deferred.totals)
    np.testing.assert_array_equal(tot_d, tot_e, err_msg=f"totals t={t}")
    np.testing.assert_array_equal(words(deferred.counts), words(eager.counts), err_msg=f"counts t={t}")
    np.testing.assert_array_equal(words(deferred.scales), words(eager.scales), err_msg=f"scales t={t}")
    te = eager.totals.cpu().numpy()
    oe, od = words(eager.out), words(deferred.out)
    for k in range(eager.K):
        n = int(te[k])
        if n <= eager.cap:
            np.testing.assert_array_equal(od[k, :n], oe[k, :n], err_msg=f"message k={k} t={t}")


def run_pair(gc, off, lt, dWs, cap=None, settle_at=(), offset=0, R0=None):
    """Eager and deferred AdaComp on the same inputs; returns the final eager
    residue (CPU) after checking every step and the settled residues."""
    import torch
    K, N = dWs[0].shape
    cap = cap if cap is not None else max(1, N)
    R_init = np.zeros((K, N), np.float32) if R0 is None else R0
    Re, Rd = shifted(R_init, offset), shifted(R_init, offset)
    eager = gc.AdaComp(off, lt, K, cap)
    deferred = gc.AdaComp(off, lt, K, cap, deferred=True)
    for t, dW in enumerate(dWs):
        d = shifted(dW, offset)
        eager(d, Re)
        deferred(d, Rd)
        torch.cuda.synchronize()
        compare_step(gc, eager, deferred, t)
        if t in settle_at or t == len(dWs) - 1:
            deferred.settle(Rd)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(words(Rd), words(Re), err_msg=f"settled residue t={t}")
    return eager, Re.cpu().numpy()


def test_mixed_bins_deferred_equals_eager(cuda_lib):
    """Warp-chunk segments (L_T 50, 500, 512, 5) beside tile (L_T 2, 4096)
    and big-bin (7000) segments, ragged sizes, 5 steps, a settle in the
    middle (the next call then starts from a settled residue)."""
    rng = np.random.default_rng(5)
    sizes = [7, 50001, 13, 4096, 4097, 99999, 30000, 1025]
    lt = [2, 50, 5, 500, 4096, 7000, 512, 4]
    off = wl.layout_offsets(sizes)
    dWs = [rng.laplace(0, 1e-2, size=(3, off[-1])).astype(np.float32) for _ in range(5)]
    dWs[1][:, 100:400] = 0.0  # all-zero bins select nothing
    run_pair(cuda_lib, off, lt, dWs, settle_at=(2,))


def test_config3_small_deferred_against_oracle(cuda_lib):
    """LSTM + VGG-16 at small size (L_T 500 and 50), K = 8, 5 steps: equal
    to the eager calls, and the messages and the settled residue of every
    step within the eager path's tolerance of the oracle."""
    import torch
    gc = cuda_lib
    w = wl.workload(3, small=True)
    dWs = [wl.gradients(w, t).numpy() for t in range(w.steps)]
    K, N = dWs[0].shape
    off = np.asarray(w.offsets, np.int64)
    eager = gc.AdaComp(off, w.lt, K, N)
    deferred = gc.AdaComp(off, w.lt, K, N, deferred=True)
    Re = torch.zeros((K, N), device="cuda")
    Rd = torch.zeros((K, N), device="cuda")
    R_o = np.zeros((K, N), np.float32)
    for t, dW in enumerate(dWs):
        G = R_o + dW  # fp32: what the residue is measured against
        idx_o, val_o, counts_o, scales_o, totals_o = oracle.adacomp_step(off, w.lt, dW, R_o, cap=N)
        d = torch.from_numpy(dW).cuda()
        eager(d, Re)
        out, totals = deferred(d, Rd)
        torch.cuda.synchronize()
        compare_step(gc, eager, deferred, t)
        np.testing.assert_array_equal(totals.cpu().numpy(), totals_o)
        np.testing.assert_array_equal(deferred.counts.cpu().numpy(), counts_o)
        idx_g = gc.pair_indices(out).cpu().numpy()
        val_g = gc.pair_values(out).cpu().numpy()
        for k in range(K):
            n = int(totals_o[k])
            np.testing.assert_array_equal(idx_g[k, :n], idx_o[k, :n].astype(np.int64))
            assert rel_err(val_g[k, :n], val_o[k, :n]) <= 1e-6
    deferred.settle(Rd)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(words(Rd), words(Re))
    Rg = Rd.cpu().numpy()  # against the oracle as the eager tests measure it: relative to max(|G|, |R|)
    denom = np.maximum(np.maximum(np.abs(G), np.abs(R_o)), np.finfo(np.float32).tiny)
    assert float((np.abs(Rg.astype(np.float64) - R_o) / denom).max(initial=0.0)) <= 1e-6


def test_deferred_over_capacity(cuda_lib):
    """A learner over cap sends nothing and keeps G, so the next call must
    apply no fix-up for it; the other learner's fix-up still applies.  With
    L_T = 4 every bin sends at least one value: learner 0 fits at step 0
    (its gradient is zero past index 100) and is over the cap of 2000 from
    step 1 on; learner 1 always fits."""
    import torch
    gc = cuda_lib
    rng = np.random.default_rng(61)
    off = wl.layout_offsets([20000, 3000])
    lt = [4, 500]
    dWs = [rng.laplace(0, 1.0, size=(2, 23000)).astype(np.float32) for _ in range(4)]
    dWs[0][0, 100:] = 0.0
    for dW in dWs:
        dW[1, 100:] = 0.0
    dWs[3][0] = 0.0
    eager, _ = run_pair(gc, off, lt, dWs, cap=2000)
    # the last step: learner 0 over the cap, learner 1 not
    tot = eager.totals.cpu().numpy()
    assert tot[0] > 2000 >= tot[1]


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_deferred_unaligned_buffers(cuda_lib, offset):
    """dW and R starting 4, 8 or 12 bytes past a 16-byte boundary (the bin
    pass takes its 4-byte copy path)."""
    rng = np.random.default_rng(offset + 90)
    sizes, lt = [50001, 8000, 4096], [50, 500, 64]
    off = wl.layout_offsets(sizes)
    dWs = [rng.laplace(0, 1e-3, size=(2, off[-1])).astype(np.float32) for _ in range(3)]
    run_pair(cuda_lib, off, lt, dWs, offset=offset)


def test_deferred_nan_entries(cuda_lib):
    """NaN in dW is never sent; its residue stays NaN with the same bits as
    the eager call's."""
    rng = np.random.default_rng(17)
    sizes, lt = [5000, 30000, 9000], [50, 500, 7000]
    off = wl.layout_offsets(sizes)
    dWs = [rng.laplace(0, 1e-3, size=(2, off[-1])).astype(np.float32) for _ in range(3)]
    dWs[0][0, [3, 77, 5123, 30001, 36000]] = np.nan
    dWs[1][1, [0, 4999, 35000]] = np.nan
    run_pair(cuda_lib, off, lt, dWs)


def test_deferred_residue_tensors_switch(cuda_lib):
    """One deferred object used on two residue tensors in turn: each call on
    the other tensor settles the previous one first, so both stay equal to
    their eager twins."""
    import torch
    gc = cuda_lib
    rng = np.random.default_rng(33)
    off = wl.layout_offsets([40000, 7000])
    lt = [50, 500]
    K, N = 2, int(off[-1])
    eager = gc.AdaComp(off, lt, K, N)
    deferred = gc.AdaComp(off, lt, K, N, deferred=True)
    Re = [torch.zeros((K, N), device="cuda") for _ in range(2)]
    Rd = [torch.zeros((K, N), device="cuda") for _ in range(2)]
    for t in range(6):
        j = (t // 2) % 2  # R0, R0, R1, R1, R0, R0
        d = torch.from_numpy(rng.laplace(0, 1e-3, size=(K, N)).astype(np.float32)).cuda()
        eager(d, Re[j])
        deferred(d, Rd[j])
        torch.cuda.synchronize()
        compare_step(gc, eager, deferred, t)
    deferred.settle()
    torch.cuda.synchronize()
    for j in range(2):
        np.testing.assert_array_equal(words(Rd[j]), words(Re[j]), err_msg=f"residue {j}")


def test_deferred_argument_errors(cuda_lib):
    """A bin length below 1, a short workspace and a pending flag other than
    0 or 1 are refused before anything is enqueued."""
    import ctypes
    import torch
    gc = cuda_lib
    off = wl.layout_offsets([1000])
    a = gc.AdaComp(off, [50], 2, 1000, deferred=True)
    R = torch.zeros((2, 1000), device="cuda")
    dW = torch.zeros((2, 1000), device="cuda")
    with pytest.raises(gc.GcsgdError):
        gc.adacomp_settle(off, [0], R, a.out, a.counts, a.totals, a.workspace)
    with pytest.raises(gc.GcsgdError) as e:
        gc.adacomp_settle(off, [50], R, a.out, a.counts, a.totals, a.workspace[:100])
    assert e.value.code == -3  # GCSGD_ERR_WORKSPACE
    o = np.ascontiguousarray(np.asarray(off, np.int64))
    lt = np.array([50], np.int32)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = gc.lib().adacomp_compress_deferred(o.ctypes.data_as(ctypes.c_void_p), 1, lt.ctypes.data_as(ctypes.c_void_p),
                                            2, p(dW), p(R), p(a.out), 1000, p(a.counts), p(a.scales), p(a.totals), 2,
                                            p(a.workspace), a.workspace.numel(), None)
    assert rc == -1  # GCSGD_ERR_INVALID_ARG


def test_deferred_full_size_lstm_vgg(cuda_lib):
    """LSTM + VGG-16 layout (80,748,688 values), K = 8, three steps in the
    benchmark's launch configuration: every message word and, after a settle,
    every residue word equal to the eager calls'."""
    import torch
    gc = cuda_lib
    w = wl.workload(3)
    K, N = w.learners, w.n
    eager = gc.AdaComp(w.offsets, w.lt, K, N // 8)
    deferred = gc.AdaComp(w.offsets, w.lt, K, N // 8, deferred=True)
    Re = torch.zeros((K, N), device="cuda")
    Rd = torch.zeros((K, N), device="cuda")
    for t in range(3):
        d = wl.gradients(w, t, device="cuda")
        eager(d, Re)
        deferred(d, Rd)
        torch.cuda.synchronize()
        assert torch.equal(eager.totals, deferred.totals)
        assert torch.equal(eager.counts, deferred.counts)
        assert torch.equal(eager.scales.view(torch.int32), deferred.scales.view(torch.int32))
        m = int(eager.totals.max().item())
        assert m <= eager.cap
        assert torch.equal(eager.out[:, :m], deferred.out[:, :m])
        del d
    deferred.settle(Rd)
    torch.cuda.synchronize()
    assert torch.equal(Re.view(torch.int32), Rd.view(torch.int32))
