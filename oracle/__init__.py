"""CPU oracle of the gradient-compression step -- TEST INFRASTRUCTURE ONLY.

A ctypes binding of ``gcsgd_oracle.c``: a plain, single-threaded C statement
of Deep Gradient Compression, AdaComp, the sparse decompress-and-average and
the DCD-PSGD replica update.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package; the product path never
does, and the two share no code.  Inputs come from
``gradient_compression_sgd_gb300.workloads`` (random draws only).

Parity pins: every function is checked in ``tests/test_oracle_*.py`` against
brute force, closed forms, library routines and published known answers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gcsgd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgcsgd_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction) into ``libgcsgd_oracle.so``."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            i64p = ctypes.POINTER(ctypes.c_int64)
            vp = ctypes.c_void_p
            L.oracle_dgc_k.restype = ctypes.c_int64
            L.oracle_dgc_k.argtypes = [ctypes.c_double, ctypes.c_int64]
            L.oracle_dgc_step.restype = ctypes.c_int
            L.oracle_dgc_step.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, ctypes.c_double,
                                          ctypes.c_float, ctypes.c_float, ctypes.c_int, vp, vp,
                                          ctypes.c_int64, vp, vp]
            L.oracle_dgc_step_nesterov.restype = ctypes.c_int
            L.oracle_dgc_step_nesterov.argtypes = L.oracle_dgc_step.argtypes
            L.oracle_dgc_step_sampled.restype = ctypes.c_int
            L.oracle_dgc_step_sampled.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, ctypes.c_double,
                                                  ctypes.c_double, ctypes.c_float, ctypes.c_float, ctypes.c_int, vp,
                                                  vp, ctypes.c_int64, vp, vp]
            L.oracle_adacomp_step.restype = ctypes.c_int
            L.oracle_adacomp_step.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, vp,
                                              ctypes.c_int64, vp, vp, vp]
            L.oracle_sparse_average.restype = ctypes.c_int
            L.oracle_sparse_average.argtypes = [ctypes.c_int, vp, vp, ctypes.c_int64, vp, ctypes.c_int64, vp]
            L.oracle_sparse_average_update.restype = ctypes.c_int
            L.oracle_sparse_average_update.argtypes = [ctypes.c_int, vp, vp, ctypes.c_int64, vp, ctypes.c_int64,
                                                       ctypes.c_float, vp]
            L.oracle_philox4x32_10.restype = None
            L.oracle_philox4x32_10.argtypes = [vp, vp, vp]
            L.oracle_keep_threshold.restype = ctypes.c_uint64
            L.oracle_keep_threshold.argtypes = [ctypes.c_double]
            L.oracle_ecd_step.restype = ctypes.c_int
            L.oracle_ecd_step.argtypes = [ctypes.c_int, ctypes.c_int64, vp, vp, vp, vp, vp, ctypes.c_float,
                                          ctypes.c_double, ctypes.c_uint64, ctypes.c_uint32]
            L.oracle_dgc_encode.restype = ctypes.c_int64
            L.oracle_dgc_encode.argtypes = [vp, vp, ctypes.c_int64, vp, ctypes.c_int64]
            L.oracle_dgc_decode.restype = ctypes.c_int
            L.oracle_dgc_decode.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, vp]
            L.oracle_adacomp_encode.restype = ctypes.c_int64
            L.oracle_adacomp_encode.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, vp, ctypes.c_int64]
            L.oracle_adacomp_decode.restype = ctypes.c_int
            L.oracle_adacomp_decode.argtypes = [vp, ctypes.c_int64, vp, ctypes.c_int, vp]
            L.oracle_dcd_step_window.restype = ctypes.c_int
            L.oracle_dcd_step_window.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, vp, vp, vp,
                                                 ctypes.c_float, ctypes.c_double, ctypes.c_uint64, ctypes.c_uint32]
            L.oracle_dcd_step_rows.restype = ctypes.c_int
            L.oracle_dcd_step_rows.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, vp, vp, vp,
                                               ctypes.c_float, ctypes.c_double, ctypes.c_uint64, ctypes.c_uint32,
                                               vp, vp]
            for f in (L.oracle_dcd_step, L.oracle_dcd_step_replicas):
                f.restype = ctypes.c_int
                f.argtypes = [ctypes.c_int, ctypes.c_int64, vp, vp, vp, ctypes.c_float, ctypes.c_double,
                              ctypes.c_uint64, ctypes.c_uint32]
            _ = i64p
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} returned {rc}")


def dgc_k(density: float, n: int) -> int:
    return int(lib().oracle_dgc_k(float(density), int(n)))


def dgc_step(offsets, grad, u, v, density, momentum, clip_thr=0.0, clip_nodes=1, cap=None, nesterov=False):
    """One DGC step of K learners. ``u``/``v`` ([K, N] float32) are updated in place.
    ``nesterov``: the accumulated state takes the look-ahead step m*u + g.

    Returns (idx [K, cap] uint32, val [K, cap] float32, counts [K, S] int64,
    clip_scale [K] float32).
    """
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    S = len(off) - 1
    grad = _f32(grad)
    K = grad.shape[0]
    assert u.dtype == np.float32 and v.dtype == np.float32 and u.flags["C_CONTIGUOUS"] and v.flags["C_CONTIGUOUS"]
    if cap is None:
        cap = max(1, sum(dgc_k(density, int(off[s + 1] - off[s])) for s in range(S)))
    idx = np.zeros((K, cap), dtype=np.uint32)
    val = np.zeros((K, cap), dtype=np.float32)
    counts = np.zeros((K, S), dtype=np.int64)
    cs = np.zeros(K, dtype=np.float32)
    fn = lib().oracle_dgc_step_nesterov if nesterov else lib().oracle_dgc_step
    rc = fn(K, S, _p(off), _p(grad), _p(u), _p(v), float(density), float(momentum),
            float(clip_thr), int(clip_nodes), _p(idx), _p(val), int(cap), _p(counts), _p(cs))
    _check(rc, "oracle_dgc_step")
    return idx, val, counts, cs


def dgc_step_sampled(offsets, grad, u, v, density, sample_frac, momentum, clip_thr=0.0, clip_nodes=1, cap=None):
    """The DGC step with the sampled threshold (every tensor whose sample of
    floor(sample_frac * n) values holds a whole 64-value block; the others exact).

    Same returns as ``dgc_step``; learner k's list has ``counts[k].sum()`` entries."""
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    S = len(off) - 1
    grad = _f32(grad)
    K = grad.shape[0]
    assert u.dtype == np.float32 and v.dtype == np.float32 and u.flags["C_CONTIGUOUS"] and v.flags["C_CONTIGUOUS"]
    if cap is None:
        cap = max(1, sum(dgc_k(density, int(off[s + 1] - off[s])) for s in range(S)))
    idx = np.zeros((K, cap), dtype=np.uint32)
    val = np.zeros((K, cap), dtype=np.float32)
    counts = np.zeros((K, S), dtype=np.int64)
    cs = np.zeros(K, dtype=np.float32)
    rc = lib().oracle_dgc_step_sampled(K, S, _p(off), _p(grad), _p(u), _p(v), float(density), float(sample_frac),
                                       float(momentum), float(clip_thr), int(clip_nodes), _p(idx), _p(val), int(cap),
                                       _p(counts), _p(cs))
    _check(rc, "oracle_dgc_step_sampled")
    return idx, val, counts, cs


def adacomp_step(offsets, lt, dW, R, cap=None):
    """One AdaComp step of K learners. ``R`` ([K, N] float32) is updated in place.

    Returns (idx [K, cap], val [K, cap], counts [K, S], scales [K, S], totals [K]).
    """
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    S = len(off) - 1
    lt = np.ascontiguousarray(lt, dtype=np.int32)
    dW = _f32(dW)
    K = dW.shape[0]
    assert R.dtype == np.float32 and R.flags["C_CONTIGUOUS"]
    if cap is None:
        cap = max(1, int(off[-1]))
    idx = np.zeros((K, cap), dtype=np.uint32)
    val = np.zeros((K, cap), dtype=np.float32)
    counts = np.zeros((K, S), dtype=np.int64)
    scales = np.zeros((K, S), dtype=np.float32)
    totals = np.zeros(K, dtype=np.int64)
    rc = lib().oracle_adacomp_step(K, S, _p(off), _p(lt), _p(dW), _p(R), _p(idx), _p(val), int(cap),
                                   _p(counts), _p(scales), _p(totals))
    _check(rc, "oracle_adacomp_step")
    return idx, val, counts, scales, totals


def sparse_average(idx, val, counts, n):
    """Dense [n] float32 average of K sparse lists (idx/val [K, cap], counts [K])."""
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    val = _f32(val)
    counts = np.ascontiguousarray(counts, dtype=np.int64)
    K, cap = idx.shape
    out = np.zeros(int(n), dtype=np.float32)
    rc = lib().oracle_sparse_average(K, _p(idx), _p(val), int(cap), _p(counts), int(n), _p(out))
    _check(rc, "oracle_sparse_average")
    return out


def sparse_average_update(idx, val, counts, n, lr, w):
    """w[j] -= lr * avg[j] at every index some list carries; ``w`` ([n] float32) is updated in place."""
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    val = _f32(val)
    counts = np.ascontiguousarray(counts, dtype=np.int64)
    assert w.dtype == np.float32 and w.flags["C_CONTIGUOUS"] and w.size >= n
    K, cap = idx.shape
    rc = lib().oracle_sparse_average_update(K, _p(idx), _p(val), int(cap), _p(counts), int(n), float(lr), _p(w))
    _check(rc, "oracle_sparse_average_update")
    return w


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    o = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_p(c), _p(k), _p(o))
    return o


def keep_threshold(p: float) -> int:
    return int(lib().oracle_keep_threshold(float(p)))


def dcd_step(xhat, g, w, gamma, p, seed, t):
    """One DCD-PSGD iteration; ``xhat`` ([n, d] float32) is updated in place."""
    assert xhat.dtype == np.float32 and xhat.flags["C_CONTIGUOUS"]
    g = _f32(g)
    w3 = _f32(w)
    n, d = xhat.shape
    rc = lib().oracle_dcd_step(n, d, _p(w3), _p(xhat), _p(g), float(gamma), float(p), int(seed), int(t))
    _check(rc, "oracle_dcd_step")
    return xhat


def dcd_step_window(xhat, g, w, gamma, p, seed, t, e_base):
    """DCD-PSGD iteration on the column window [e_base, e_base + d) of a longer model."""
    assert xhat.dtype == np.float32 and xhat.flags["C_CONTIGUOUS"]
    g = _f32(g)
    w3 = _f32(w)
    n, d = xhat.shape
    rc = lib().oracle_dcd_step_window(n, d, int(e_base), _p(w3), _p(xhat), _p(g), float(gamma), float(p), int(seed),
                                      int(t))
    _check(rc, "oracle_dcd_step_window")
    return xhat


def dcd_step_rows(xrows, g, w, gamma, p, seed, t, first_node):
    """One DCD iteration of the own rows 1..R-2 of ``xrows`` ([R, d] float32,
    updated in place; rows 0 and R-1 are the neighbours' copies, read only),
    own nodes first_node.. ; g: [R-2, d].  Returns (C of row 1, C of row R-2)."""
    assert xrows.dtype == np.float32 and xrows.flags["C_CONTIGUOUS"]
    R, d = xrows.shape
    g = _f32(g)
    assert g.shape == (R - 2, d)
    wr = np.ascontiguousarray(w, dtype=np.float32)
    c_first = np.zeros(d, np.float32)
    c_last = np.zeros(d, np.float32)
    rc = lib().oracle_dcd_step_rows(int(R), int(d), int(first_node), _p(wr), _p(xrows), _p(g), float(gamma),
                                    float(p), int(seed), int(t), _p(c_first), _p(c_last))
    _check(rc, "oracle_dcd_step_rows")
    return c_first, c_last


def dcd_step_replicas(rep, g, w, gamma, p, seed, t):
    """DCD-PSGD iteration with explicit replicas ``rep`` [n, n, d] (node i's copy of node j)."""
    assert rep.dtype == np.float32 and rep.flags["C_CONTIGUOUS"]
    g = _f32(g)
    w3 = _f32(w)
    n, _, d = rep.shape
    rc = lib().oracle_dcd_step_replicas(n, d, _p(w3), _p(rep), _p(g), float(gamma), float(p), int(seed), int(t))
    _check(rc, "oracle_dcd_step_replicas")
    return rep


def ecd_step(x, x_prev, xt, g, w, gamma, p, seed, t):
    """One ECD-PSGD iteration t >= 1: ``xt`` updated in place, ``x_prev`` receives x_{t+1}."""
    for a in (x, x_prev, xt):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    g = _f32(g)
    w3 = _f32(w)
    n, d = x.shape
    rc = lib().oracle_ecd_step(n, d, _p(w3), _p(x), _p(x_prev), _p(xt), _p(g), float(gamma), float(p), int(seed),
                               int(t))
    _check(rc, "oracle_ecd_step")
    return x_prev, xt


def dgc_encode(idx, val) -> bytes:
    """DGC's byte stream of one learner's ascending (idx, val) list."""
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    val = _f32(val)
    cap = 6 * (len(idx) + int(idx.max(initial=0)) // 65536 + 2)
    buf = np.zeros(max(cap, 6), np.uint8)
    nb = lib().oracle_dgc_encode(_p(idx), _p(val), len(idx), _p(buf), len(buf))
    if nb < 0:
        raise OracleError("oracle_dgc_encode: indices do not ascend or the buffer is short")
    return buf[:nb].tobytes()


def dgc_decode(stream: bytes, n: int) -> np.ndarray:
    buf = np.frombuffer(stream, np.uint8).copy() if stream else np.zeros(1, np.uint8)
    out = np.zeros(max(int(n), 1), np.float32)
    _check(lib().oracle_dgc_decode(_p(buf), len(stream), int(n), _p(out)), "oracle_dgc_decode")
    return out[:n]


def adacomp_encode(offsets, idx, val, counts, scales) -> bytes:
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    S = len(off) - 1
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    val = _f32(val)
    counts = np.ascontiguousarray(counts, dtype=np.int64)
    scales = _f32(scales)
    buf = np.zeros(8 * S + 4 * int(counts.sum()) + 1, np.uint8)
    nb = lib().oracle_adacomp_encode(_p(off), S, _p(idx), _p(val), _p(counts), _p(scales), _p(buf), len(buf))
    if nb < 0:
        raise OracleError("oracle_adacomp_encode: buffer too short")
    return buf[:nb].tobytes()


def adacomp_decode(stream: bytes, offsets) -> np.ndarray:
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    buf = np.frombuffer(stream, np.uint8).copy() if stream else np.zeros(1, np.uint8)
    out = np.zeros(max(int(off[-1]), 1), np.float32)
    _check(lib().oracle_adacomp_decode(_p(buf), len(stream), _p(off), len(off) - 1, _p(out)), "oracle_adacomp_decode")
    return out[:int(off[-1])]
