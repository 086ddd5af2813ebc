"""The largest tensor count a call accepts (gc.MAX_SEGMENTS tensors, which
takes the many-segment instantiations of the plan and hint kernels): DGC
(vanilla, Nesterov, sampled threshold), AdaComp with mixed bin lengths, the
sparse average of their messages and the AdaComp wire format, all against
the oracle on a ragged layout with empty, tiny and candidate-pool tensors."""
import numpy as np
import pytest

import oracle
from gradient_compression_sgd_gb300 import workloads as wl
from test_gpu_adacomp_average_dcd import run_adacomp
from test_gpu_dgc import run_dgc, run_dgc_sampled

pytestmark = pytest.mark.gpu


def max_layout(seed):
    """gc.MAX_SEGMENTS tensor sizes: most in [0, 600), 40 empty, 6 large
    enough for DGC's candidate pool."""
    import gradient_compression_sgd_gb300 as gc
    rng = np.random.default_rng(seed)
    S = gc.MAX_SEGMENTS
    sizes = rng.integers(0, 600, size=S)
    sizes[rng.choice(S, 40, replace=False)] = 0
    sizes[rng.choice(S, 6, replace=False)] = rng.integers(20_000, 70_000, size=6)
    return [int(x) for x in sizes]


@pytest.mark.parametrize("nesterov", [False, True])
def test_dgc_at_the_maximum_tensor_count(cuda_lib, nesterov):
    sizes = max_layout(31)
    off = wl.layout_offsets(sizes)
    assert len(sizes) == cuda_lib.MAX_SEGMENTS
    rng = np.random.default_rng(32)
    K, N = 3, int(off[-1])
    grads = [(rng.standard_normal((K, N)) * 1e-3).astype(np.float32) for _ in range(2)]
    d = run_dgc(cuda_lib, off, grads, 0.01, 0.9, nesterov=nesterov)
    st = d.stats()
    assert st["pool"] > 0 and st["empty"] > 0 and st["raw"] > 0


def test_dgc_sampled_at_the_maximum_tensor_count(cuda_lib):
    sizes = max_layout(33)
    off = wl.layout_offsets(sizes)
    rng = np.random.default_rng(34)
    K, N = 2, int(off[-1])
    grads = [(rng.standard_normal((K, N)) * 1e-3).astype(np.float32) for _ in range(2)]
    run_dgc_sampled(cuda_lib, off, grads, 0.01, 0.05, 0.9)


def test_adacomp_average_and_wire_at_the_maximum_tensor_count(cuda_lib):
    import torch
    gc = cuda_lib
    sizes = max_layout(35)
    off = wl.layout_offsets(sizes)
    rng = np.random.default_rng(36)
    lt = [int(x) for x in rng.choice([2, 7, 50, 500, 4096, 7000], size=len(sizes))]
    K, N = 3, int(off[-1])
    dWs = [rng.laplace(0, 1e-2, size=(K, N)).astype(np.float32) for _ in range(2)]
    a, results = run_adacomp(gc, off, lt, dWs)
    assert all(r[0] == "ok" for r in results)
    out, counts, scales, totals = a.out, a.counts, a.scales, a.totals
    # the average of the last step's messages
    avg = torch.empty(N, device="cuda")
    gc.sparse_average(out, totals, N, avg)
    torch.cuda.synchronize()
    idx = gc.pair_indices(out).cpu().numpy().astype(np.uint32)
    val = gc.pair_values(out).cpu().numpy()
    tot = totals.cpu().numpy()
    np.testing.assert_array_equal(avg.cpu().numpy(), oracle.sparse_average(idx, val, tot, N))
    # the wire format: per-layer count and scale for every one of the tensors, then the entries
    cap_b = 8 * len(sizes) + 4 * int(tot.max())
    cap_b += (-cap_b) % 16
    streams = torch.zeros((K, cap_b), dtype=torch.uint8, device="cuda")
    nbytes = torch.zeros(K, dtype=torch.int64, device="cuda")
    gc.adacomp_encode(off, out, counts, scales, streams, nbytes)
    torch.cuda.synchronize()
    nb, stm = nbytes.cpu().numpy(), streams.cpu().numpy()
    cnt, sc = counts.cpu().numpy(), scales.cpu().numpy()
    for k in range(K):
        n = int(tot[k])
        want = oracle.adacomp_encode(off, idx[k, :n], val[k, :n], cnt[k], sc[k])
        assert nb[k] == len(want) and stm[k, :nb[k]].tobytes() == want
    lists = torch.zeros_like(out)
    tot2 = torch.zeros(K, dtype=torch.int64, device="cuda")
    gc.adacomp_decode(off, streams, nbytes, lists, tot2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tot2.cpu().numpy(), tot)
    li = lists.cpu().numpy()
    for k in range(K):
        n = int(tot[k])
        np.testing.assert_array_equal(li[k, :n, 0].view(np.uint32), idx[k, :n])
        np.testing.assert_array_equal(li[k, :n, 1].view(np.float32), val[k, :n])


def test_adacomp_learner_limit_at_the_maximum_tensor_count(cuda_lib):
    """At 2048 tensors 24 learners fit ada_emit's tables and match the
    oracle; 25 are refused before anything runs, leaving the residue as it
    was."""
    import torch
    gc = cuda_lib
    S = gc.MAX_SEGMENTS
    sizes = [3] * S
    off = wl.layout_offsets(sizes)
    lt = [2] * S
    rng = np.random.default_rng(37)
    dWs = [rng.laplace(0, 1e-2, size=(24, 3 * S)).astype(np.float32)]
    run_adacomp(gc, off, lt, dWs)
    R = torch.from_numpy(rng.standard_normal((25, 3 * S)).astype(np.float32)).cuda()
    R0 = R.clone()
    a = gc.AdaComp(off, lt, 25, 3 * S)
    with pytest.raises(gc.GcsgdError, match="emit tables"):
        a(torch.from_numpy(rng.laplace(0, 1e-2, size=(25, 3 * S)).astype(np.float32)).cuda(), R)
    torch.cuda.synchronize()
    assert torch.equal(R, R0)
