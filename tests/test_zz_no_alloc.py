"""dgc_compress_noalloc: the DGC step for callers that cannot allocate device
memory (a plugin whose host framework's allocator owns the memory budget, or
a loop that must not call into the driver's allocator mid-step).  Checked
against the CPU oracle on two calls in a row (indices and counts bit for bit,
values, u and v within the contract's 1e-6), bit for bit against
dgc_compress with a caller workspace, and for what it claims: after the
first call on the device, a call changes the device's free memory by nothing.
Layouts that need more than its fixed scratch are refused.

This file is named so that pytest collects it last: if it fails, a run that
stops at the first failure has already run every other test.  It passes on
its own in a fresh process as well.
"""
import numpy as np
import pytest

import oracle
from conftest import rel_err
from gradient_compression_sgd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

VAL_RTOL = 1e-6


def _state(K, N):
    import torch
    return torch.zeros((K, N), device="cuda"), torch.zeros((K, N), device="cuda")


@pytest.mark.parametrize("config,small", [(1, False), (2, True)])
def test_noalloc_matches_the_oracle_two_calls(cuda_lib, config, small):
    """The one-tensor clipping workload at full size and the 1/8-width
    ResNet-50 layout (K = 4): both calls against the oracle's DGC step."""
    import torch
    gc = cuda_lib
    w = wl.workload(config, small=small)
    off, K, N = w.offsets, w.learners, w.n
    cap = gc.DGC(off, K, w.density, w.momentum, w.clip_thr, w.clip_nodes).cap
    u_g, v_g = _state(K, N)
    u_o = np.zeros((K, N), np.float32)
    v_o = np.zeros((K, N), np.float32)
    out = gc.pairs_buffer(K, cap)
    counts = torch.zeros((K, len(w.sizes)), dtype=torch.int64, device="cuda")
    totals = torch.zeros(K, dtype=torch.int64, device="cuda")
    for t in range(2):  # two calls in a row: the shared scratch keeps the first call's contents
        G = wl.gradients(w, t)
        idx_o, val_o, counts_o, _ = oracle.dgc_step(off, G.numpy(), u_o, v_o, w.density, w.momentum, w.clip_thr,
                                                    w.clip_nodes, cap=cap)
        gc.dgc_compress_noalloc(off, G.cuda(), u_g, v_g, out, counts, w.density, w.momentum, w.clip_thr,
                                w.clip_nodes, totals=totals)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(counts.cpu().numpy(), counts_o, err_msg=f"counts, call {t}")
        assert totals.cpu().numpy().tolist() == counts_o.sum(axis=1).tolist()
        idx_g = gc.pair_indices(out).cpu().numpy()
        val_g = gc.pair_values(out).cpu().numpy()
        for k in range(K):
            n = int(counts_o[k].sum())
            np.testing.assert_array_equal(idx_g[k, :n], idx_o[k, :n].astype(np.int64), err_msg=f"idx k={k} t={t}")
            assert rel_err(val_g[k, :n], val_o[k, :n]) <= VAL_RTOL
        assert rel_err(u_g.cpu().numpy(), u_o) <= VAL_RTOL, f"u, call {t}"
        assert rel_err(v_g.cpu().numpy(), v_o) <= VAL_RTOL, f"v, call {t}"


def test_noalloc_matches_workspace_entry_point_and_allocates_nothing(cuda_lib):
    """The full ResNet-50 layout, K = 4: bit for bit the same as dgc_compress
    on two calls, and the second call leaves the device's free memory as it
    was (the first call may place the library's scratch array)."""
    import torch
    gc = cuda_lib
    w = wl.workload(2)
    off, K, N = w.offsets, w.learners, w.n
    ref = gc.DGC(off, K, w.density, w.momentum, w.clip_thr, w.clip_nodes)
    u1, v1 = _state(K, N)
    u2, v2 = _state(K, N)
    out2 = gc.pairs_buffer(K, ref.cap)
    counts2 = torch.zeros((K, len(w.sizes)), dtype=torch.int64, device="cuda")
    totals2 = torch.zeros(K, dtype=torch.int64, device="cuda")
    grads = [wl.gradients(w, t, device="cuda") for t in range(2)]
    for t in range(2):
        out1, totals1 = ref(grads[t], u1, v1)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        gc.dgc_compress_noalloc(off, grads[t], u2, v2, out2, counts2, w.density, w.momentum, w.clip_thr,
                                w.clip_nodes, totals=totals2)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        if t == 1:
            assert free_after == free_before, f"the call changed free device memory by {free_before - free_after} B"
        assert torch.equal(totals1, totals2) and torch.equal(ref.counts, counts2)
        assert torch.equal(gc.pair_indices(out1), gc.pair_indices(out2))
        assert torch.equal(gc.pair_values(out1), gc.pair_values(out2))
        assert torch.equal(u1, u2) and torch.equal(v1, v2)


def test_noalloc_rejects_layouts_beyond_its_scratch(cuda_lib):
    import torch
    gc = cuda_lib
    w = wl.workload(4)  # 8 learners x 98M values: about 74 MiB of scratch
    need = gc.dgc_workspace_size(w.offsets, w.learners, w.density)
    assert need > gc.NOALLOC_SCRATCH_BYTES
    x = torch.zeros((w.learners, 4), device="cuda")  # never read: the call is refused first
    out = gc.pairs_buffer(w.learners, 8)
    counts = torch.zeros((w.learners, len(w.sizes)), dtype=torch.int64, device="cuda")
    with pytest.raises(gc.GcsgdError) as e:
        gc.dgc_compress_noalloc(w.offsets, x, x, x, out, counts, w.density, w.momentum)
    assert e.value.code == -3 and "scratch" in str(e.value)
