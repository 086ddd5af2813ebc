"""Wire formats: the CUDA encoders against the oracle's byte streams, and
decode(encode(message)) == message."""
import numpy as np
import pytest

import oracle
from gradient_compression_sgd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _pairs(idx, val):
    import torch
    K, cap = idx.shape
    p = torch.zeros((K, cap, 2), dtype=torch.int32)
    p[..., 0] = torch.from_numpy(idx.astype(np.int64)).to(torch.int32)
    p[..., 1] = torch.from_numpy(val.astype(np.float32).view(np.int32))
    return p.cuda()


def _encode_dgc(gc, pairs, totals, stream_cap):
    import torch
    K = pairs.shape[0]
    streams = torch.zeros((K, stream_cap), dtype=torch.uint8, device="cuda")
    nbytes = torch.zeros(K, dtype=torch.int64, device="cuda")
    gc.dgc_encode(pairs, totals, streams, nbytes)
    torch.cuda.synchronize()
    return streams, nbytes


def _check_dgc_round_trip(gc, idx, val, totals_np):
    import torch
    K, cap = idx.shape
    pairs = _pairs(idx, val)
    totals = torch.from_numpy(totals_np.astype(np.int64)).cuda()
    need = max(len(oracle.dgc_encode(idx[k, :int(totals_np[k])], val[k, :int(totals_np[k])])) for k in range(K))
    streams, nbytes = _encode_dgc(gc, pairs, totals, need + 16 - need % 16)
    nb = nbytes.cpu().numpy()
    st = streams.cpu().numpy()
    for k in range(K):
        n = int(totals_np[k])
        want = oracle.dgc_encode(idx[k, :n], val[k, :n])
        assert nb[k] == len(want)
        assert st[k, :nb[k]].tobytes() == want
    lists = torch.zeros((K, cap, 2), dtype=torch.int32, device="cuda")
    tot2 = torch.zeros(K, dtype=torch.int64, device="cuda")
    gc.dgc_decode(streams, nbytes, lists, tot2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tot2.cpu().numpy(), totals_np)
    li = lists.cpu().numpy()
    for k in range(K):
        n = int(totals_np[k])
        np.testing.assert_array_equal(li[k, :n, 0].view(np.uint32), idx[k, :n])
        np.testing.assert_array_equal(li[k, :n, 1].view(np.float32), val[k, :n])


def test_dgc_stream_of_a_dgc_step(cuda_lib):
    import torch
    gc = cuda_lib
    w = wl.workload(2, small=True)
    d = gc.DGC(w.offsets, w.learners, w.density, w.momentum)
    u = torch.zeros((w.learners, w.n), device="cuda")
    v = torch.zeros((w.learners, w.n), device="cuda")
    out, totals = d(wl.gradients(w, 0).cuda(), u, v)
    torch.cuda.synchronize()
    idx = gc.pair_indices(out).cpu().numpy().astype(np.uint32)
    val = gc.pair_values(out).cpu().numpy()
    _check_dgc_round_trip(gc, idx, val, totals.cpu().numpy())


def test_dgc_stream_long_gaps_and_edges(cuda_lib):
    """Gaps of 65535, 65536, 131072 and more (escapes), index 0, the last
    index below 2^32, an empty list."""
    idx = np.zeros((3, 8), np.uint32)
    val = np.zeros((3, 8), np.float32)
    rows = [[0, 65536, 65537 + 65536, 400000, 400001, 4294967295],
            [65535, 65536 + 65535 + 1, 9_000_000],
            []]
    for k, r in enumerate(rows):
        idx[k, :len(r)] = r
        val[k, :len(r)] = np.arange(1, len(r) + 1, dtype=np.float32) * (-1.5) ** np.arange(len(r))
    _check_dgc_round_trip(cuda_lib, idx, val, np.array([len(r) for r in rows]))


def test_dgc_stream_refuses_short_buffers_and_unsorted_lists(cuda_lib):
    import torch
    idx = np.array([[1, 2, 3, 0], [5, 4, 0, 0]], np.uint32)
    val = np.ones((2, 4), np.float32)
    pairs = _pairs(idx, val)
    streams, nbytes = _encode_dgc(cuda_lib, pairs, torch.tensor([3, 2], device="cuda"), 16)
    assert nbytes.cpu().tolist() == [-1, -1]  # 18 bytes do not fit 16; 5, 4 do not ascend


def test_adacomp_stream_of_an_adacomp_step(cuda_lib):
    import torch
    gc = cuda_lib
    w = wl.workload(3, small=True)
    K = w.learners
    a = gc.AdaComp(w.offsets, w.lt, K, w.n)
    R = torch.zeros((K, w.n), device="cuda")
    out, totals = a(wl.gradients(w, 0).cuda(), R)
    torch.cuda.synchronize()
    S = len(w.sizes)
    cap_b = 8 * S + 4 * int(totals.max().item())
    cap_b += (-cap_b) % 16
    streams = torch.zeros((K, cap_b), dtype=torch.uint8, device="cuda")
    nbytes = torch.zeros(K, dtype=torch.int64, device="cuda")
    gc.adacomp_encode(w.offsets, out, a.counts, a.scales, streams, nbytes)
    torch.cuda.synchronize()
    idx = gc.pair_indices(out).cpu().numpy().astype(np.uint32)
    val = gc.pair_values(out).cpu().numpy()
    counts, scales, tot = a.counts.cpu().numpy(), a.scales.cpu().numpy(), totals.cpu().numpy()
    nb, st = nbytes.cpu().numpy(), streams.cpu().numpy()
    for k in range(K):
        n = int(tot[k])
        want = oracle.adacomp_encode(w.offsets, idx[k, :n], val[k, :n], counts[k], scales[k])
        assert nb[k] == len(want) and st[k, :nb[k]].tobytes() == want
    lists = torch.zeros_like(out)
    tot2 = torch.zeros(K, dtype=torch.int64, device="cuda")
    gc.adacomp_decode(w.offsets, streams, nbytes, lists, tot2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tot2.cpu().numpy(), tot)
    li = lists.cpu().numpy()
    for k in range(K):
        n = int(tot[k])
        np.testing.assert_array_equal(li[k, :n, 0].view(np.uint32), idx[k, :n])
        np.testing.assert_array_equal(li[k, :n, 1].view(np.float32), val[k, :n])


def test_adacomp_stream_refuses_counts_beyond_the_list(cuda_lib):
    """After a capacity overflow the list is empty while the counts are not:
    the encoder must not read past the list."""
    import torch
    off = [0, 100, 300]
    lists = torch.zeros((2, 4, 2), dtype=torch.int32, device="cuda")
    counts = torch.tensor([[3, 2], [1, 0]], dtype=torch.int64, device="cuda")  # 5 > cap 4 for learner 0
    scales = torch.ones((2, 2), device="cuda")
    streams = torch.zeros((2, 64), dtype=torch.uint8, device="cuda")
    nbytes = torch.zeros(2, dtype=torch.int64, device="cuda")
    cuda_lib.adacomp_encode(off, lists, counts, scales, streams, nbytes)
    torch.cuda.synchronize()
    assert nbytes.cpu().tolist() == [-1, 8 * 2 + 4 * 1]
