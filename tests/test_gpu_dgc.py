"""DGC parity: the CUDA library against the CPU oracle, element by element.

Indices, counts and the masked state are compared bit for bit; values within
the 1e-6 relative tolerance of the contract (the kernels use the same
per-operation fp32 rounding, so they are expected to be exact).
"""
import zlib

import numpy as np
import pytest

import oracle
from conftest import rel_err
from gradient_compression_sgd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

VAL_RTOL = 1e-6


def shifted(a, offset):
    """A CUDA copy of `a` that starts `offset` floats past an allocation's start
    (offset 1..3: not 16-byte aligned)."""
    import torch
    flat = torch.zeros(a.size + offset, dtype=torch.float32, device="cuda")
    view = flat[offset:].view(a.shape)
    view.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return view


def run_dgc(gc, offsets, grads, density, momentum, clip_thr=0.0, clip_nodes=1, u0=None, v0=None, offset=0,
            nesterov=False):
    """Step both sides through the gradient list and compare after every step."""
    import torch
    offsets = np.asarray(offsets, np.int64)
    K, N = grads[0].shape
    u_o = np.zeros((K, N), np.float32) if u0 is None else u0.copy()
    v_o = np.zeros((K, N), np.float32) if v0 is None else v0.copy()
    u_g = shifted(u_o, offset)
    v_g = shifted(v_o, offset)
    d = gc.DGC(offsets, K, density, momentum, clip_thr, clip_nodes, nesterov=nesterov)
    for t, G in enumerate(grads):
        idx_o, val_o, counts_o, _ = oracle.dgc_step(offsets, G, u_o, v_o, density, momentum, clip_thr, clip_nodes,
                                                    cap=d.cap, nesterov=nesterov)
        out, totals = d(shifted(G, offset), u_g, v_g)
        torch.cuda.synchronize()
        counts_g = d.counts.cpu().numpy()
        np.testing.assert_array_equal(counts_g, counts_o, err_msg=f"counts, step {t}")
        assert list(totals.cpu().numpy()) == [int(counts_o[k].sum()) for k in range(K)]
        idx_g = gc.pair_indices(out).cpu().numpy()
        val_g = gc.pair_values(out).cpu().numpy()
        for k in range(K):
            n = int(counts_o[k].sum())
            np.testing.assert_array_equal(idx_g[k, :n], idx_o[k, :n].astype(np.int64), err_msg=f"idx k={k} t={t}")
            assert rel_err(val_g[k, :n], val_o[k, :n]) <= VAL_RTOL, f"values k={k} t={t}"
        assert rel_err(u_g.cpu().numpy(), u_o) <= VAL_RTOL, f"u, step {t}"
        assert rel_err(v_g.cpu().numpy(), v_o) <= VAL_RTOL, f"v, step {t}"
        # masking: zero exactly at the sent indices
        vg = v_g.cpu().numpy()
        for k in range(K):
            n = int(counts_o[k].sum())
            assert not np.any(vg[k, idx_o[k, :n]])
    return d


def test_config1_dgc_single_tensor_with_clipping(cuda_lib):
    """1,048,576 values N(0, 1e-3), density 0.001 (k = 1049), clip thr 1.0
    (the norm is ~1.02, so clipping fires), momentum 0.9, 3 steps."""
    w = wl.workload(1)
    grads = [wl.gradients(w, t).numpy() for t in range(w.steps)]
    d = run_dgc(cuda_lib, w.offsets, grads, w.density, w.momentum, w.clip_thr, w.clip_nodes)
    assert d.cap == 1049


@pytest.mark.parametrize("config", [2, 4])
def test_small_configs(cuda_lib, config):
    """The ResNet-50 layout at 1/8 width (161 tensors, K = 4, 5 steps) and the
    GRU layout shrunk to 256x768 (K = 8, 10 steps)."""
    w = wl.workload(config, small=True)
    grads = [wl.gradients(w, t).numpy() for t in range(w.steps)]
    d = run_dgc(cuda_lib, w.offsets, grads, w.density, w.momentum)
    st = d.stats()
    assert st["units"] == w.learners * len(w.sizes) and st["hint_failed"] == 0


EDGE_LAYOUTS = {
    "single_1": [1],
    "tiny": [3, 1, 2],
    "empty_segments": [0, 5, 0, 0, 17, 0],
    "tile_plus_one": [4097],
    "misaligned": [7, 33, 65537, 12, 50001, 3],
    "pool_segment": [40000],
    "two_pool_segments_ragged": [100003, 70001],
}


@pytest.mark.parametrize("name", list(EDGE_LAYOUTS))
@pytest.mark.parametrize("density", [0.001, 0.05, 1.0])
def test_edge_layouts(cuda_lib, name, density):
    sizes = EDGE_LAYOUTS[name]
    off = wl.layout_offsets(sizes)
    rng = np.random.default_rng(zlib.crc32(f"{name}/{density}".encode()))
    K = 3
    grads = [(rng.standard_normal((K, off[-1])) * rng.uniform(1e-4, 1e-1)).astype(np.float32) for _ in range(3)]
    run_dgc(cuda_lib, off, grads, density, 0.9)


@pytest.mark.parametrize("levels", [1, 3, 7])
def test_ties_and_zeros(cuda_lib, levels):
    """Few distinct magnitudes (and all-zero gradients for levels = 1): the
    threshold value is shared by many entries and the lower indices must win."""
    rng = np.random.default_rng(levels)
    off = wl.layout_offsets([50000, 1000, 70000])
    K = 2
    grads = []
    for t in range(3):
        q = rng.integers(-(levels // 2), levels // 2 + 1, size=(K, off[-1])).astype(np.float32) * 0.25
        grads.append(q)
    run_dgc(cuda_lib, off, grads, 0.01, 0.0)
    run_dgc(cuda_lib, off, grads, 0.003, 0.5)


@pytest.mark.parametrize("n,density", [(40000, 0.003), (2359296, 0.001)])
def test_hint_above_the_kth_value_falls_back(cuda_lib, n, density):
    """Values planted where the threshold sample reads push the candidate
    threshold above the k-th value: exactly a sampled values are 3.0 (so the
    hint is 3.0 and only a < k entries qualify), the other sampled values 1.0
    (ties), some unsampled ones 0.5, the rest tiny.  The select must fall
    back to the whole segment and still be exact, also for a tensor of
    ResNet-50's largest size (2,359,296 values, the emission sweeping it from
    global memory).  (The sample layout mirrors the kernel's plan: R = max(2.5
    k, 512), m = min(48 n / R, 16384) rounded down to 64, blocks of 64 at
    stride n / (m / 64), a = round(R m / n).)"""
    k = oracle.dgc_k(density, n)
    R = max(5 * k // 2, 512)
    m = min(48 * n // R, 16384) & ~63
    nblk, stride = m // 64, n // (m // 64)
    a = (R * m + n // 2) // n
    assert a < k
    G = np.full((1, n), 1e-6, np.float32)
    pos = np.concatenate([np.arange(b * stride, b * stride + 64) for b in range(nblk)])
    G[0, pos] = 1.0
    G[0, pos[np.linspace(0, len(pos) - 1, a).astype(int)]] = 3.0
    G[0, 30001:30050] = 0.5
    d = run_dgc(cuda_lib, [0, n], [G], density, 0.9)
    assert d.stats()["hint_failed"] == 1


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_buffers_not_16_byte_aligned(cuda_lib, offset):
    """g, u and v starting 4, 8 or 12 bytes past a 16-byte boundary."""
    rng = np.random.default_rng(offset)
    off = wl.layout_offsets([5000, 70001, 4096, 20000])
    grads = [rng.standard_normal((2, off[-1])).astype(np.float32) for _ in range(2)]
    run_dgc(cuda_lib, off, grads, 0.01, 0.9, offset=offset)


def test_nonzero_initial_state_and_momentum_zero(cuda_lib):
    rng = np.random.default_rng(11)
    off = wl.layout_offsets([1000, 200000, 36864])
    K, N = 2, off[-1]
    u0 = rng.standard_normal((K, N)).astype(np.float32) * 0.1
    v0 = rng.standard_normal((K, N)).astype(np.float32)
    grads = [rng.standard_normal((K, N)).astype(np.float32) for _ in range(2)]
    run_dgc(cuda_lib, off, grads, 0.002, 0.9, u0=u0, v0=v0)
    run_dgc(cuda_lib, off, grads, 0.002, 0.0, u0=u0, v0=v0)


@pytest.mark.parametrize("nodes", [1, 4])
def test_clipping_multi_learner(cuda_lib, nodes):
    rng = np.random.default_rng(nodes)
    off = wl.layout_offsets([300000, 5000])
    K, N = 3, off[-1]
    scale = np.array([1e-4, 1e-3, 1e-2], np.float32)[:, None]  # some learners clip, some do not
    grads = [(rng.standard_normal((K, N)) * scale).astype(np.float32) for _ in range(3)]
    run_dgc(cuda_lib, off, grads, 0.001, 0.9, clip_thr=1.0, clip_nodes=nodes)


def test_checkpoint_resume_is_bit_identical(cuda_lib):
    """The state is the caller's u and v: 3 steps straight equal 1 step, a
    save/restore of (u, v) through host memory, then 2 more steps."""
    import torch
    gc = cuda_lib
    w = wl.workload(2, small=True)
    off = w.offsets
    K, N = w.learners, w.n
    grads = [wl.gradients(w, t).cuda() for t in range(3)]
    d = gc.DGC(off, K, w.density, w.momentum)
    u = torch.zeros((K, N), device="cuda")
    v = torch.zeros((K, N), device="cuda")
    outs = []
    for t in range(3):
        o, _ = d(grads[t], u, v)
        outs.append(o.clone())
    u2 = torch.zeros((K, N), device="cuda")
    v2 = torch.zeros((K, N), device="cuda")
    d2 = gc.DGC(off, K, w.density, w.momentum)
    o0, _ = d2(grads[0], u2, v2)
    saved = (u2.cpu().clone(), v2.cpu().clone())
    u3, v3 = saved[0].cuda(), saved[1].cuda()
    for t in (1, 2):
        o, _ = d2(grads[t], u3, v3)
        assert torch.equal(o, outs[t])
    assert torch.equal(u3, u) and torch.equal(v3, v)


def test_async_on_side_stream(cuda_lib):
    """Calls enqueue on the given stream and never synchronise."""
    import torch
    gc = cuda_lib
    off = wl.layout_offsets([100000, 3000])
    K, N = 2, off[-1]
    g = torch.randn((K, N), device="cuda") * 1e-3
    u = torch.zeros((K, N), device="cuda")
    v = torch.zeros((K, N), device="cuda")
    d = gc.DGC(off, K, 0.01, 0.9)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out, totals = d(g, u, v, stream=s)
    s.synchronize()
    assert int(totals[0]) == sum(gc.dgc_k(0.01, int(off[i + 1] - off[i])) for i in range(2))


# ------------------------------------------- pools larger than one CTA's stage

def test_big_pool_ties_across_cluster_ranks(cuda_lib):
    """Pools of up to ~52K candidates are selected by a thread-block cluster,
    each CTA holding an eighth of the tiles.  Values from a small discrete set
    put thousands of exact ties at the k-th value, spread over every rank;
    the ties must go to the lowest indices across ranks."""
    rng = np.random.default_rng(21)
    n, density = 1 << 21, 0.01  # k = 20972, expected candidates 52430: more than one stage
    off = wl.layout_offsets([n, 5000])
    grads = [(rng.integers(0, 200, size=(2, off[-1])) * 1e-3).astype(np.float32) for _ in range(2)]
    run_dgc(cuda_lib, off, grads, density, 0.0)


def test_big_pool_heavy_duplicates(cuda_lib):
    """Most candidates share one value and one candidate is huge, so the key
    range is wide and a single radix bucket holds far more keys than the
    candidate buffer: every digit runs across the cluster until the last one
    names the threshold, and the ties at 0.5 go to the lowest indices."""
    rng = np.random.default_rng(22)
    n, density = 3 << 20, 0.004  # k = 12583
    G = np.full((1, n), 1e-4, np.float32)
    G[0, rng.choice(n, 40000, replace=False)] = 0.5
    G[0, rng.choice(n, 3000, replace=False)] = np.float32(0.5) * np.float32(1.0000001)
    G[0, 12345] = 1e6
    run_dgc(cuda_lib, [0, n], [G, G], density, 0.9)


def test_big_pool_skewed_to_one_rank_falls_back(cuda_lib):
    """Every candidate in the first eighth of the tiles: one rank's share is
    above its stage, so the cluster's first CTA selects the pool alone."""
    rng = np.random.default_rng(23)
    n, density = 1 << 21, 0.01
    G = (rng.standard_normal((1, n)) * 1e-6).astype(np.float32)
    G[0, : n // 8] = (rng.standard_normal(n // 8) * 1.0).astype(np.float32)
    d = run_dgc(cuda_lib, [0, n], [G], density, 0.9)
    assert d.stats()["hint_failed"] == 0


@pytest.mark.parametrize("frac", [0.01, 0.3])
def test_big_pool_sampled_threshold(cuda_lib, frac):
    """The sampled threshold on pools larger than one stage (the cluster also
    sends every candidate when there are fewer than k)."""
    rng = np.random.default_rng(int(frac * 100))
    off = wl.layout_offsets([1 << 21, 3 << 19])
    grads = [(rng.standard_normal((2, off[-1])) * 1e-3).astype(np.float32) for _ in range(2)]
    run_dgc_sampled(cuda_lib, off, grads, 0.01, frac, 0.9)


# ------------------------------------------------------- sampled threshold

def run_dgc_sampled(gc, offsets, grads, density, frac, momentum, offset=0):
    """The sampled-threshold step, CUDA against the oracle after every step:
    per-tensor counts, the packed lists, u and v."""
    offsets = np.asarray(offsets, np.int64)
    K, N = grads[0].shape
    u_o = np.zeros((K, N), np.float32)
    v_o = np.zeros((K, N), np.float32)
    u_g = shifted(u_o, offset)
    v_g = shifted(v_o, offset)
    d = gc.DGC(offsets, K, density, momentum, sample_frac=frac)
    short = 0
    for t, G in enumerate(grads):
        idx_o, val_o, counts_o, _ = oracle.dgc_step_sampled(offsets, G, u_o, v_o, density, frac, momentum, cap=d.cap)
        out, totals = d(shifted(G, offset), u_g, v_g)
        import torch
        torch.cuda.synchronize()
        np.testing.assert_array_equal(d.counts.cpu().numpy(), counts_o, err_msg=f"counts, step {t}")
        tot = totals.cpu().numpy()
        assert tot.tolist() == counts_o.sum(axis=1).tolist()
        idx_g = gc.pair_indices(out).cpu().numpy()
        val_g = gc.pair_values(out).cpu().numpy()
        for k in range(K):
            n = int(tot[k])
            np.testing.assert_array_equal(idx_g[k, :n], idx_o[k, :n].astype(np.int64), err_msg=f"idx k={k} t={t}")
            assert rel_err(val_g[k, :n], val_o[k, :n]) <= VAL_RTOL
        assert rel_err(u_g.cpu().numpy(), u_o) <= VAL_RTOL and rel_err(v_g.cpu().numpy(), v_o) <= VAL_RTOL
        short += int((counts_o < np.array([[oracle.dgc_k(density, int(offsets[s + 1] - offsets[s]))
                                             for s in range(len(offsets) - 1)]])).sum())
    return short


@pytest.mark.parametrize("frac", [0.001, 0.003, 0.01, 0.2])
def test_sampled_threshold(cuda_lib, frac):
    """Tensors of every kind: small ones sampled from the select kernel's
    stage (6400 .. 16384 values), pool tensors, samples above 16384 keys
    (700000 and 2.4M values at 0.2 and 0.01), ones under one block."""
    rng = np.random.default_rng(int(frac * 1000) + 7)
    off = wl.layout_offsets([16384, 50000, 200000, 33333, 0, 700000, 6400, 9000, 700, 2359296])
    grads = [(rng.standard_normal((2, off[-1])) * 1e-3).astype(np.float32) for _ in range(3)]
    run_dgc_sampled(cuda_lib, off, grads, 0.002, frac, 0.9)


@pytest.mark.parametrize("density", [0.05, 0.3, 0.9])
def test_sampled_threshold_high_density(cuda_lib, density):
    """Densities with 5 k > n: every tensor with a whole sample block is
    sampled, small (staged) and large (pool) alike."""
    rng = np.random.default_rng(int(density * 100) + 3)
    off = wl.layout_offsets([640, 6400, 16384, 40000, 300000])
    grads = [(rng.standard_normal((2, off[-1])) * 1e-2).astype(np.float32) for _ in range(3)]
    run_dgc_sampled(cuda_lib, off, grads, density, 0.1, 0.9)


def test_sampled_small_tensor_examples_on_the_gpu(cuda_lib):
    """The hand-worked examples of tests/golden/dgc_sampled_small_examples.txt."""
    from conftest import load_golden
    from test_oracle_dgc import sampled_example

    ex = load_golden("dgc_sampled_small_examples.txt")
    for name in "ABCD":
        n, G = sampled_example(ex, name)
        run_dgc_sampled(cuda_lib, [0, n], [G], float(ex[f"{name}_density"][0]), float(ex[f"{name}_frac"][0]), 0.9)


def test_sampled_threshold_resnet50_small_layout(cuda_lib):
    """The 1/8-width ResNet-50 layout, K = 4, 1 % samples, 5 steps; some
    tensors send fewer than k (the approximation the sample makes)."""
    w = wl.workload(2, small=True)
    grads = [wl.gradients(w, t).numpy() for t in range(5)]
    short = run_dgc_sampled(cuda_lib, w.offsets, grads, w.density, 0.01, w.momentum, offset=1)
    assert short > 0


def test_sampled_hand_examples_on_the_gpu(cuda_lib):
    n = 20480
    G = np.full((1, n), 1e-3, np.float32)
    G[0, 6830], G[0, 100], G[0, 200], G[0, 20000], G[0, 300] = 5.0, 6.0, -7.0, 5.0, 4.9
    run_dgc_sampled(cuda_lib, [0, n], [G], 0.001, 0.01, 0.9)
    G = np.full((1, n), 1e-3, np.float32)
    for b in range(12):
        G[0, 128 * b] = 100.0 + b
    G[0, 64], G[0, 65] = 150.0, 100.5
    run_dgc_sampled(cuda_lib, [0, n], [G], 0.001, 0.5, 0.9)


# ------------------------------------------------ Nesterov momentum (reading)

@pytest.mark.parametrize("config", [2, 4])
def test_nesterov_small_configs(cuda_lib, config):
    """dgc_compress_nesterov on the small ResNet-50 and GRU layouts, every step
    against the oracle's Nesterov step."""
    w = wl.workload(config, small=True)
    grads = [wl.gradients(w, t).numpy() for t in range(w.steps)]
    d = run_dgc(cuda_lib, w.offsets, grads, w.density, w.momentum, nesterov=True)
    assert d.stats()["hint_failed"] == 0


@pytest.mark.parametrize("name", ["tiny", "empty_segments", "misaligned", "two_pool_segments_ragged"])
def test_nesterov_edge_layouts_with_clipping(cuda_lib, name):
    sizes = EDGE_LAYOUTS[name]
    off = wl.layout_offsets(sizes)
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    grads = [rng.standard_normal((3, off[-1])).astype(np.float32) * 1e-2 for _ in range(3)]
    run_dgc(cuda_lib, off, grads, 0.01, 0.9, clip_thr=0.5, clip_nodes=2, nesterov=True)


def test_nesterov_with_zero_momentum_matches_dgc_compress(cuda_lib):
    """m = 0: the Nesterov entry point and dgc_compress give identical bits."""
    import torch
    gc = cuda_lib
    off = wl.layout_offsets([50001, 300, 70001])
    rng = np.random.default_rng(3)
    G = torch.from_numpy(rng.standard_normal((2, off[-1])).astype(np.float32)).cuda()
    res = []
    for nest in (False, True):
        u = torch.zeros((2, off[-1]), device="cuda")
        v = torch.full((2, off[-1]), 0.25, device="cuda")
        d = gc.DGC(off, 2, 0.01, 0.0, nesterov=nest)
        out, totals = d(G, u, v)
        torch.cuda.synchronize()
        res.append((out.cpu().clone(), totals.cpu().clone(), u.cpu(), v.cpu()))
    for a, b in zip(res[0], res[1]):
        assert torch.equal(a, b)
