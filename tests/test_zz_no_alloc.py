"""dgc_compress_noalloc: the DGC step for callers that cannot allocate device
memory (a plugin whose host framework's allocator owns the memory budget, or
a loop that must not call into the driver's allocator mid-step).  It must give
the same results as dgc_compress with a caller workspace, call after call,
and refuse layouts that need more than its fixed scratch.

This file is named so that pytest collects it last: if it fails, a run that
stops at the first failure has already run every other test.  It passes on
its own in a fresh process as well.
"""
import numpy as np
import pytest

from conftest import rel_err
from gradient_compression_sgd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _state(K, N):
    import torch
    return torch.zeros((K, N), device="cuda"), torch.zeros((K, N), device="cuda")


@pytest.mark.parametrize("config", [1, 2])
def test_noalloc_matches_workspace_entry_point_two_calls(cuda_lib, config):
    import torch
    gc = cuda_lib
    w = wl.workload(config)
    off, K, N = w.offsets, w.learners, w.n
    ref = gc.DGC(off, K, w.density, w.momentum, w.clip_thr, w.clip_nodes)
    u1, v1 = _state(K, N)
    u2, v2 = _state(K, N)
    out2 = gc.pairs_buffer(K, ref.cap)
    counts2 = torch.zeros((K, len(w.sizes)), dtype=torch.int64, device="cuda")
    totals2 = torch.zeros(K, dtype=torch.int64, device="cuda")
    for t in range(2):  # two calls in a row: the shared scratch keeps the first call's contents
        G = wl.gradients(w, t, device="cuda")
        out1, totals1 = ref(G, u1, v1)
        gc.dgc_compress_noalloc(off, G, u2, v2, out2, counts2, w.density, w.momentum, w.clip_thr, w.clip_nodes,
                                totals=totals2)
        torch.cuda.synchronize()
        assert torch.equal(totals1, totals2) and torch.equal(ref.counts, counts2)
        assert torch.equal(gc.pair_indices(out1), gc.pair_indices(out2))
        assert rel_err(gc.pair_values(out2).cpu().numpy(), gc.pair_values(out1).cpu().numpy()) <= 1e-6
        assert rel_err(u2.cpu().numpy(), u1.cpu().numpy()) <= 1e-6
        assert rel_err(v2.cpu().numpy(), v1.cpu().numpy()) <= 1e-6


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
