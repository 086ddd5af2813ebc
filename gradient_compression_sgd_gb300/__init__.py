"""GB300 gradient compression for data-parallel SGD: a thin Python binding.

Every step of the path runs in ``libgcsgd.so`` (hand-written sm_103a CUDA
behind the C ABI declared in ``include/gcsgd.h``).  This module only
marshals torch tensors (device memory) and streams into those calls; there is
no CPU or PyTorch fallback, and calling an entry point without the built
library raises.

Entry points mirror the C names: :func:`dgc_compress`,
:func:`adacomp_compress`, :func:`sparse_average`, :func:`dcd_step`, plus the
workspace-size queries and the tracing helpers.  :class:`DGC` and
:class:`AdaComp` keep the workspace, message buffers and counters of one
layout so that a training loop makes one call per step.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgcsgd.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "gcsgd.h")

GCSGD_OK = 0
ERRORS = {-1: "invalid argument", -2: "capacity", -3: "workspace", -4: "cuda"}
MAX_SEGMENTS = 2048

_lock = threading.Lock()
_lib = None


class GcsgdError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed ({ERRORS.get(code, code)}): {msg}")
        self.code = code


class DgcStats(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int64) for name in
                ("units", "empty", "raw", "pool", "pool_global", "raw_global", "hint_failed")]


class TraceEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


def declared_functions() -> list[str]:
    """Names of the functions include/gcsgd.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\*?([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return [n for n in names if n not in ("defined",)]


def lib():
    """Load libgcsgd.so (it must have been built: gradient_compression_sgd_gb300.build.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m gradient_compression_sgd_gb300.build` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, f32, f64, u32, u64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                                ctypes.c_double, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_size_t)
        L.gcsgd_last_error.restype = ctypes.c_char_p
        L.gcsgd_version.restype = i32
        L.gcsgd_launch_count.restype = i64
        L.gcsgd_launch_count_reset.restype = None
        L.gcsgd_trace_enable.argtypes = [i32]
        L.gcsgd_trace_read.argtypes = [vp, i32, vp]
        L.gcsgd_trace_only.argtypes = [ctypes.c_char_p]
        L.gcsgd_dgc_k.restype = i64
        L.gcsgd_dgc_k.argtypes = [f64, i64]
        L.gcsgd_dgc_workspace_size.argtypes = [vp, i32, i32, f64, vp]
        L.dgc_compress.argtypes = [vp, i32, i32, vp, vp, vp, f64, f32, f32, i32, vp, i64, vp, vp, vp, sz, vp]
        L.dgc_compress_nesterov.argtypes = L.dgc_compress.argtypes
        L.dgc_compress_noalloc.argtypes = [vp, i32, i32, vp, vp, vp, f64, f32, f32, i32, vp, i64, vp, vp, vp]
        L.gcsgd_dgc_sampled_workspace_size.argtypes = [vp, i32, i32, f64, f64, vp]
        L.dgc_compress_sampled.argtypes = [vp, i32, i32, vp, vp, vp, f64, f64, f32, f32, i32, vp, i64, vp, vp, vp,
                                           sz, vp]
        L.gcsgd_dgc_stats.argtypes = [vp, i32, i32, f64, vp, vp, vp]
        L.gcsgd_adacomp_workspace_size.argtypes = [vp, i32, vp, i32, i64, vp]
        L.adacomp_compress.argtypes = [vp, i32, vp, i32, vp, vp, vp, i64, vp, vp, vp, vp, sz, vp]
        L.adacomp_compress_deferred.argtypes = [vp, i32, vp, i32, vp, vp, vp, i64, vp, vp, vp, i32, vp, sz, vp]
        L.adacomp_settle.argtypes = [vp, i32, vp, i32, vp, vp, i64, vp, vp, vp, sz, vp]
        L.sparse_average.argtypes = [vp, i64, vp, i32, i64, vp, vp]
        L.sparse_average_update.argtypes = [vp, i64, vp, i32, i64, f32, vp, vp]
        L.gcsgd_sparse_average_workspace_size.argtypes = [i32, i64, vp]
        L.sparse_average_ws.argtypes = [vp, i64, vp, i32, i64, vp, vp, sz, vp]
        L.gcsgd_sparse_average_status.argtypes = [vp, i32, i64, vp, vp]
        L.sparse_average_update_ws.argtypes = [vp, i64, vp, i32, i64, f32, vp, vp, sz, vp]
        L.dcd_step.argtypes = [i32, i64, vp, vp, vp, f32, f64, u64, u32, vp]
        L.ecd_step.argtypes = [i32, i64, vp, vp, vp, vp, vp, f32, f64, u64, u32, vp]
        L.dcd_step_rows.argtypes = [i32, i64, i64, vp, vp, vp, f32, f64, u64, u32, vp, vp, i64, vp, vp]
        L.dcd_copy_add.argtypes = [vp, i64, vp, vp, i64, i32, vp]
        L.dgc_encode.argtypes = [vp, i64, vp, i32, vp, i64, vp, vp]
        L.dgc_decode.argtypes = [vp, i64, vp, i32, vp, i64, vp, vp]
        L.adacomp_encode.argtypes = [vp, i32, vp, i64, vp, vp, i32, vp, i64, vp, vp]
        L.adacomp_decode.argtypes = [vp, i32, vp, i64, vp, i32, vp, i64, vp, vp]
        _lib = L
        return L


def _check(fn: str, rc: int):
    if rc != GCSGD_OK:
        raise GcsgdError(fn, rc, lib().gcsgd_last_error().decode(errors="replace"))


def last_error() -> str:
    return lib().gcsgd_last_error().decode(errors="replace")


def version() -> int:
    return int(lib().gcsgd_version())


# ----------------------------------------------------------------- helpers

def _offsets(offsets) -> np.ndarray:
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    if off.ndim != 1 or len(off) < 2:
        raise ValueError("offsets must be a 1-D array of n_seg + 1 entries")
    return off


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dev(t, name, dtype=None):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def ecd_step(x, x_prev, xtilde, grad, w_ring, gamma: float, keep_p: float, seed: int, t: int, stream=None):
    """One ECD-PSGD ring iteration t >= 1 (see ecd_step in include/gcsgd.h): x_prev receives x_{t+1},
    xtilde is updated in place."""
    import torch
    n, d = x.shape
    w = np.ascontiguousarray(np.asarray(w_ring, dtype=np.float32))
    if w.shape != (3,):
        raise ValueError("w_ring must hold 3 weights (left, self, right)")
    _check("ecd_step", lib().ecd_step(int(n), int(d), _ptr(w), _dev(x, "x", torch.float32),
                                      _dev(x_prev, "x_prev", torch.float32), _dev(xtilde, "xtilde", torch.float32),
                                      _dev(grad, "grad", torch.float32), float(gamma), float(keep_p),
                                      int(seed) & 0xFFFFFFFFFFFFFFFF, int(t) & 0xFFFFFFFF, _stream(stream)))


def dgc_encode(lists, totals, streams, nbytes, stream=None):
    """DGC messages [K, cap] -> byte streams [K, stream_cap] (uint8); nbytes [K] (see dgc_encode in include/gcsgd.h)."""
    import torch
    K, cap = lists.shape[0], lists.shape[1]
    _check("dgc_encode", lib().dgc_encode(_dev(lists, "lists", torch.int32), int(cap), _dev(totals, "totals", torch.int64),
                                          int(K), _dev(streams, "streams", torch.uint8), int(streams.shape[1]),
                                          _dev(nbytes, "nbytes", torch.int64), _stream(stream)))


def dgc_decode(streams, nbytes, lists, totals, stream=None):
    import torch
    K = streams.shape[0]
    _check("dgc_decode", lib().dgc_decode(_dev(streams, "streams", torch.uint8), int(streams.shape[1]),
                                          _dev(nbytes, "nbytes", torch.int64), int(K), _dev(lists, "lists", torch.int32),
                                          int(lists.shape[1]), _dev(totals, "totals", torch.int64), _stream(stream)))


def adacomp_encode(offsets, lists, counts, scales, streams, nbytes, stream=None):
    import torch
    off = _offsets(offsets)
    K, cap = lists.shape[0], lists.shape[1]
    _check("adacomp_encode", lib().adacomp_encode(
        _ptr(off), len(off) - 1, _dev(lists, "lists", torch.int32), int(cap), _dev(counts, "counts", torch.int64),
        _dev(scales, "scales", torch.float32), int(K), _dev(streams, "streams", torch.uint8), int(streams.shape[1]),
        _dev(nbytes, "nbytes", torch.int64), _stream(stream)))


def adacomp_decode(offsets, streams, nbytes, lists, totals, stream=None):
    import torch
    off = _offsets(offsets)
    K = streams.shape[0]
    _check("adacomp_decode", lib().adacomp_decode(
        _ptr(off), len(off) - 1, _dev(streams, "streams", torch.uint8), int(streams.shape[1]),
        _dev(nbytes, "nbytes", torch.int64), int(K), _dev(lists, "lists", torch.int32), int(lists.shape[1]),
        _dev(totals, "totals", torch.int64), _stream(stream)))


def pairs_buffer(K: int, cap: int, device="cuda"):
    """[K, cap, 2] int32 tensor holding gcsgd_pair records (index, value bits)."""
    import torch
    return torch.zeros((K, max(cap, 1), 2), dtype=torch.int32, device=device)


def pair_indices(pairs):
    """uint32 indices of a pairs buffer, as int64."""
    import torch
    return pairs[..., 0].to(torch.int64) & 0xFFFFFFFF


def pair_values(pairs):
    """fp32 values of a pairs buffer (a view)."""
    import torch
    return pairs[..., 1].view(torch.float32)


# ------------------------------------------------------------------- DGC

def dgc_k(density: float, n: int) -> int:
    return int(lib().gcsgd_dgc_k(float(density), int(n)))


def dgc_workspace_size(offsets, K: int, density: float) -> int:
    off = _offsets(offsets)
    out = ctypes.c_size_t(0)
    _check("gcsgd_dgc_workspace_size",
           lib().gcsgd_dgc_workspace_size(_ptr(off), len(off) - 1, int(K), float(density), ctypes.byref(out)))
    return int(out.value)


def dgc_compress(offsets, grad, u, v, out, counts, workspace, density, momentum, clip_thr=0.0, clip_nodes=1,
                 totals=None, stream=None, nesterov=False):
    """One DGC step of K learners (see dgc_compress and, with nesterov,
    dgc_compress_nesterov in include/gcsgd.h)."""
    import torch
    off = _offsets(offsets)
    K = grad.shape[0]
    cap = out.shape[1]
    fn = "dgc_compress_nesterov" if nesterov else "dgc_compress"
    _check(fn, getattr(lib(), fn)(
        _ptr(off), len(off) - 1, int(K), _dev(grad, "grad", torch.float32), _dev(u, "u", torch.float32),
        _dev(v, "v", torch.float32), float(density), float(momentum), float(clip_thr), int(clip_nodes),
        _dev(out, "out", torch.int32), int(cap), _dev(counts, "counts", torch.int64),
        _dev(totals, "totals", torch.int64), _dev(workspace, "workspace", torch.uint8), int(workspace.numel()),
        _stream(stream)))


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def dgc_sampled_workspace_size(offsets, K: int, density: float, sample_frac: float) -> int:
    off = _offsets(offsets)
    out = ctypes.c_size_t(0)
    _check("gcsgd_dgc_sampled_workspace_size",
           lib().gcsgd_dgc_sampled_workspace_size(_ptr(off), len(off) - 1, int(K), float(density), float(sample_frac),
                                                  ctypes.byref(out)))
    return int(out.value)


def dgc_compress_sampled(offsets, grad, u, v, out, counts, workspace, density, sample_frac, momentum, clip_thr=0.0,
                         clip_nodes=1, totals=None, stream=None):
    """The DGC step with the sampled threshold (see dgc_compress_sampled in include/gcsgd.h)."""
    import torch
    off = _offsets(offsets)
    K = grad.shape[0]
    cap = out.shape[1]
    _check("dgc_compress_sampled", lib().dgc_compress_sampled(
        _ptr(off), len(off) - 1, int(K), _dev(grad, "grad", torch.float32), _dev(u, "u", torch.float32),
        _dev(v, "v", torch.float32), float(density), float(sample_frac), float(momentum), float(clip_thr),
        int(clip_nodes), _dev(out, "out", torch.int32), int(cap), _dev(counts, "counts", torch.int64),
        _dev(totals, "totals", torch.int64), _dev(workspace, "workspace", torch.uint8), int(workspace.numel()),
        _stream(stream)))


def dgc_compress_noalloc(offsets, grad, u, v, out, counts, density, momentum, clip_thr=0.0, clip_nodes=1,
                         totals=None, stream=None):
    """dgc_compress with the library's fixed scratch instead of a workspace, for
    callers that may not allocate device memory (see dgc_compress_noalloc in
    include/gcsgd.h: at most NOALLOC_SCRATCH_BYTES of scratch; overlapping
    calls race on the shared scratch)."""
    import torch
    off = _offsets(offsets)
    K = grad.shape[0]
    cap = out.shape[1]
    _check("dgc_compress_noalloc", lib().dgc_compress_noalloc(
        _ptr(off), len(off) - 1, int(K), _dev(grad, "grad", torch.float32), _dev(u, "u", torch.float32),
        _dev(v, "v", torch.float32), float(density), float(momentum), float(clip_thr), int(clip_nodes),
        _dev(out, "out", torch.int32), int(cap), _dev(counts, "counts", torch.int64),
        _dev(totals, "totals", torch.int64), _stream(stream)))


class DGC:
    """Buffers of DGC on one layout: workspace, [K, cap] messages and counters."""

    def __init__(self, offsets, K: int, density: float, momentum: float, clip_thr: float = 0.0,
                 clip_nodes: int = 1, device="cuda", sample_frac: float = 0.0, nesterov: bool = False):
        import torch
        self.offsets = _offsets(offsets)
        self.S = len(self.offsets) - 1
        self.K, self.density, self.momentum = int(K), float(density), float(momentum)
        self.clip_thr, self.clip_nodes = float(clip_thr), int(clip_nodes)
        self.sample_frac = float(sample_frac)  # > 0: the sampled threshold (dgc_compress_sampled)
        self.nesterov = bool(nesterov)  # Nesterov momentum (dgc_compress_nesterov)
        if self.nesterov and self.sample_frac > 0:
            raise ValueError("Nesterov momentum is available with the exact top-k only")
        self.cap = sum(dgc_k(density, int(self.offsets[s + 1] - self.offsets[s])) for s in range(self.S))
        ws = (dgc_sampled_workspace_size(self.offsets, K, density, self.sample_frac) if self.sample_frac > 0
              else dgc_workspace_size(self.offsets, K, density))
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=device)
        self.out = pairs_buffer(K, self.cap, device)
        self.counts = torch.zeros((K, self.S), dtype=torch.int64, device=device)
        self.totals = torch.zeros(K, dtype=torch.int64, device=device)

    def stats(self, stream=None) -> dict:
        """How the last call selected each (learner, segment) (gcsgd_dgc_stats; synchronises)."""
        st = DgcStats()
        _check("gcsgd_dgc_stats", lib().gcsgd_dgc_stats(
            _ptr(self.offsets), self.S, self.K, self.density, ctypes.c_void_p(self.workspace.data_ptr()),
            _stream(stream), ctypes.byref(st)))
        return {name: int(getattr(st, name)) for name, _ in DgcStats._fields_}

    def __call__(self, grad, u, v, stream=None):
        if self.sample_frac > 0:
            dgc_compress_sampled(self.offsets, grad, u, v, self.out, self.counts, self.workspace, self.density,
                                 self.sample_frac, self.momentum, self.clip_thr, self.clip_nodes, totals=self.totals,
                                 stream=stream)
        else:
            dgc_compress(self.offsets, grad, u, v, self.out, self.counts, self.workspace, self.density,
                         self.momentum, self.clip_thr, self.clip_nodes, totals=self.totals, stream=stream,
                         nesterov=self.nesterov)
        return self.out, self.totals


# ---------------------------------------------------------------- AdaComp

def adacomp_workspace_size(offsets, lt, K: int, cap: int) -> int:
    off = _offsets(offsets)
    lt = np.ascontiguousarray(np.asarray(lt, dtype=np.int32))
    out = ctypes.c_size_t(0)
    _check("gcsgd_adacomp_workspace_size", lib().gcsgd_adacomp_workspace_size(
        _ptr(off), len(off) - 1, _ptr(lt), int(K), int(cap), ctypes.byref(out)))
    return int(out.value)


def adacomp_compress(offsets, lt, dW, residue, out, counts, scales, totals, workspace, stream=None):
    """One AdaComp step of K learners (see adacomp_compress in include/gcsgd.h)."""
    import torch
    off = _offsets(offsets)
    lt = np.ascontiguousarray(np.asarray(lt, dtype=np.int32))
    K = dW.shape[0]
    cap = out.shape[1]
    _check("adacomp_compress", lib().adacomp_compress(
        _ptr(off), len(off) - 1, _ptr(lt), int(K), _dev(dW, "dW", torch.float32),
        _dev(residue, "residue", torch.float32), _dev(out, "out", torch.int32), int(cap),
        _dev(counts, "counts", torch.int64), _dev(scales, "scales", torch.float32),
        _dev(totals, "totals", torch.int64), _dev(workspace, "workspace", torch.uint8), int(workspace.numel()),
        _stream(stream)))


def adacomp_compress_deferred(offsets, lt, dW, residue, out, counts, scales, totals, workspace, pending: bool,
                              stream=None):
    """One AdaComp step with the residue fix-up deferred to the next call (see
    adacomp_compress_deferred in include/gcsgd.h)."""
    import torch
    off = _offsets(offsets)
    lt = np.ascontiguousarray(np.asarray(lt, dtype=np.int32))
    K = dW.shape[0]
    cap = out.shape[1]
    _check("adacomp_compress_deferred", lib().adacomp_compress_deferred(
        _ptr(off), len(off) - 1, _ptr(lt), int(K), _dev(dW, "dW", torch.float32),
        _dev(residue, "residue", torch.float32), _dev(out, "out", torch.int32), int(cap),
        _dev(counts, "counts", torch.int64), _dev(scales, "scales", torch.float32),
        _dev(totals, "totals", torch.int64), 1 if pending else 0, _dev(workspace, "workspace", torch.uint8),
        int(workspace.numel()), _stream(stream)))


def adacomp_settle(offsets, lt, residue, out, counts, totals, workspace, stream=None):
    """Applies a deferred call's pending residue fix-up (see adacomp_settle in include/gcsgd.h)."""
    import torch
    off = _offsets(offsets)
    lt = np.ascontiguousarray(np.asarray(lt, dtype=np.int32))
    K = out.shape[0]
    _check("adacomp_settle", lib().adacomp_settle(
        _ptr(off), len(off) - 1, _ptr(lt), int(K), _dev(residue, "residue", torch.float32),
        _dev(out, "out", torch.int32), int(out.shape[1]), _dev(counts, "counts", torch.int64),
        _dev(totals, "totals", torch.int64), _dev(workspace, "workspace", torch.uint8), int(workspace.numel()),
        _stream(stream)))


class AdaComp:
    """Buffers of AdaComp on one layout; ``cap`` bounds the entries per learner.

    With ``deferred=True`` each call leaves the residue fix-up of its sent
    entries to the next call on the same residue tensor (adacomp_compress_deferred);
    ``settle(residue)`` applies a pending one, and a call on another residue
    tensor settles the previous tensor first."""

    def __init__(self, offsets, lt, K: int, cap: int, device="cuda", deferred: bool = False):
        import torch
        self.offsets = _offsets(offsets)
        self.lt = np.ascontiguousarray(np.asarray(lt, dtype=np.int32))
        self.S = len(self.offsets) - 1
        self.K, self.cap = int(K), int(cap)
        self.workspace = torch.empty(adacomp_workspace_size(self.offsets, self.lt, K, cap), dtype=torch.uint8,
                                     device=device)
        self.out = pairs_buffer(K, cap, device)
        self.counts = torch.zeros((K, self.S), dtype=torch.int64, device=device)
        self.scales = torch.zeros((K, self.S), dtype=torch.float32, device=device)
        self.totals = torch.zeros(K, dtype=torch.int64, device=device)
        self.deferred = bool(deferred)
        self._pending = None  # the residue tensor whose fix-up is pending

    def __call__(self, dW, residue, stream=None):
        if not self.deferred:
            adacomp_compress(self.offsets, self.lt, dW, residue, self.out, self.counts, self.scales, self.totals,
                             self.workspace, stream=stream)
            return self.out, self.totals
        if self._pending is not None and self._pending.data_ptr() != residue.data_ptr():
            self.settle(self._pending, stream=stream)
        pending = self._pending is not None
        adacomp_compress_deferred(self.offsets, self.lt, dW, residue, self.out, self.counts, self.scales,
                                  self.totals, self.workspace, pending, stream=stream)
        self._pending = residue
        return self.out, self.totals

    def settle(self, residue=None, stream=None):
        """Applies the pending fix-up to `residue` (default: the pending tensor), if any."""
        r = self._pending if residue is None else residue
        if self._pending is None or r is None or r.data_ptr() != self._pending.data_ptr():
            return
        adacomp_settle(self.offsets, self.lt, r, self.out, self.counts, self.totals, self.workspace, stream=stream)
        self._pending = None


# ---------------------------------------------------------- sparse average

def sparse_average(lists, counts, n: int, out, stream=None):
    """Dense K-way average of sparse messages (see sparse_average in include/gcsgd.h)."""
    import torch
    K, cap = lists.shape[0], lists.shape[1]
    if counts.numel() != K:
        raise ValueError("counts must have K entries")
    _check("sparse_average", lib().sparse_average(
        _dev(lists, "lists", torch.int32), int(cap), _dev(counts, "counts", torch.int64), int(K), int(n),
        _dev(out, "out", torch.float32), _stream(stream)))


def sparse_average_workspace_size(K: int, n: int) -> int:
    """Bytes of workspace sparse_average_ws needs (see gcsgd_sparse_average_workspace_size in include/gcsgd.h)."""
    b = ctypes.c_size_t(0)
    _check("gcsgd_sparse_average_workspace_size",
           lib().gcsgd_sparse_average_workspace_size(int(K), int(n), ctypes.byref(b)))
    return int(b.value)


def sparse_average_ws(lists, counts, n: int, out, workspace, stream=None):
    """sparse_average through the cursor-table kernels; workspace: a uint8 device
    tensor of at least sparse_average_workspace_size(K, n) bytes (see
    sparse_average_ws in include/gcsgd.h)."""
    import torch
    K, cap = lists.shape[0], lists.shape[1]
    if counts.numel() != K:
        raise ValueError("counts must have K entries")
    _check("sparse_average_ws", lib().sparse_average_ws(
        _dev(lists, "lists", torch.int32), int(cap), _dev(counts, "counts", torch.int64), int(K), int(n),
        _dev(out, "out", torch.float32), _dev(workspace, "workspace", torch.uint8), int(workspace.numel()),
        _stream(stream)))


def sparse_average_update_ws(lists, counts, n: int, lr: float, w, workspace, stream=None):
    """w[j] -= lr * (K-way average)[j] at every carried index, through the
    cursor-table kernels (see sparse_average_update_ws in include/gcsgd.h)."""
    import torch
    K, cap = lists.shape[0], lists.shape[1]
    if counts.numel() != K:
        raise ValueError("counts must have K entries")
    _check("sparse_average_update_ws", lib().sparse_average_update_ws(
        _dev(lists, "lists", torch.int32), int(cap), _dev(counts, "counts", torch.int64), int(K), int(n),
        float(lr), _dev(w, "w", torch.float32), _dev(workspace, "workspace", torch.uint8), int(workspace.numel()),
        _stream(stream)))


def sparse_average_status(workspace, K: int, n: int, stream=None) -> int:
    """Status word of the last sparse_average_ws call with this workspace, K and n
    (0: every bulk copy completed); waits for the stream."""
    st = ctypes.c_int32(-1)
    _check("gcsgd_sparse_average_status", lib().gcsgd_sparse_average_status(
        ctypes.c_void_p(workspace.data_ptr()), int(K), int(n), _stream(stream), ctypes.byref(st)))
    return int(st.value)


def sparse_average_update(lists, counts, n: int, lr: float, w, stream=None):
    """w[j] -= lr * (K-way average)[j] at every carried index (see sparse_average_update in include/gcsgd.h)."""
    import torch
    K, cap = lists.shape[0], lists.shape[1]
    if counts.numel() != K:
        raise ValueError("counts must have K entries")
    _check("sparse_average_update", lib().sparse_average_update(
        _dev(lists, "lists", torch.int32), int(cap), _dev(counts, "counts", torch.int64), int(K), int(n),
        float(lr), _dev(w, "w", torch.float32), _stream(stream)))


# -------------------------------------------------------------------- DCD

def dcd_step(xhat, grad, w_ring, gamma: float, keep_p: float, seed: int, t: int, stream=None):
    """One DCD-PSGD ring iteration, xhat [n, d] updated in place (see dcd_step in include/gcsgd.h)."""
    import torch
    n, d = xhat.shape
    w = np.ascontiguousarray(np.asarray(w_ring, dtype=np.float32))
    if w.shape != (3,):
        raise ValueError("w_ring must hold 3 weights (left, self, right)")
    _check("dcd_step", lib().dcd_step(int(n), int(d), _ptr(w), _dev(xhat, "xhat", torch.float32),
                                      _dev(grad, "grad", torch.float32), float(gamma), float(keep_p),
                                      int(seed) & 0xFFFFFFFFFFFFFFFF, int(t) & 0xFFFFFFFF, _stream(stream)))


def dcd_step_rows(xrows, grad, w_ring, gamma: float, keep_p: float, seed: int, t: int, first_node: int,
                  c_first, c_last, counts, stream=None):
    """DCD-PSGD on the own rows 1..R-2 of xrows [R, d] beside the neighbours'
    copies in rows 0 and R-1 (see dcd_step_rows in include/gcsgd.h).  c_first,
    c_last: [cap, 2] int32 pair buffers; counts: [2] int64, set on the device."""
    import torch
    R, d = xrows.shape
    if grad.shape != (R - 2, d):
        raise ValueError(f"grad must be [{R - 2}, {d}]")
    if c_first.shape != c_last.shape or c_first.dim() != 2 or c_first.shape[1] != 2 or counts.numel() != 2:
        raise ValueError("c_first, c_last: [cap, 2] int32 pair buffers; counts: 2 int64")
    w = np.ascontiguousarray(np.asarray(w_ring, dtype=np.float32))
    if w.shape != (3,):
        raise ValueError("w_ring must hold 3 weights (left, self, right)")
    _check("dcd_step_rows", lib().dcd_step_rows(
        int(R), int(d), int(first_node), _ptr(w), _dev(xrows, "xrows", torch.float32), _dev(grad, "grad", torch.float32),
        float(gamma), float(keep_p), int(seed) & 0xFFFFFFFFFFFFFFFF, int(t) & 0xFFFFFFFF,
        _dev(c_first, "c_first", torch.int32), _dev(c_last, "c_last", torch.int32), int(c_first.shape[0]),
        _dev(counts, "counts", torch.int64), _stream(stream)))


def dcd_copy_add(x_row, pairs, count, zero_pass: bool = False, stream=None):
    """x_row [d] += the C(z) a neighbour sent as pairs [cap, 2] int32, count a
    device int64 (see dcd_copy_add in include/gcsgd.h)."""
    import torch
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs: [cap, 2] int32")
    _check("dcd_copy_add", lib().dcd_copy_add(
        _dev(x_row, "x_row", torch.float32), int(x_row.numel()), _dev(pairs, "pairs", torch.int32) if pairs.numel() else None,
        _dev(count, "count", torch.int64), int(pairs.shape[0]), 1 if zero_pass else 0, _stream(stream)))


# ------------------------------------------------------- counting, tracing

def launch_count() -> int:
    return int(lib().gcsgd_launch_count())


def launch_count_reset():
    lib().gcsgd_launch_count_reset()


def trace_enable(on: bool = True):
    lib().gcsgd_trace_enable(1 if on else 0)


def trace_only(name=None):
    """Trace only the launches of kernel `name` (None: every kernel)."""
    _check("gcsgd_trace_only", lib().gcsgd_trace_only(name.encode() if name else None))


def trace_read() -> dict:
    """{kernel name: (launches, total ms)} recorded since the last read (waits for the events)."""
    n = ctypes.c_int32(0)
    buf = (TraceEntry * 64)()
    _check("gcsgd_trace_read", lib().gcsgd_trace_read(ctypes.cast(buf, ctypes.c_void_p), 64, ctypes.byref(n)))
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(min(n.value, 64))}
