"""The C-ABI library builds, loads and exports every function include/gcsgd.h
declares; host-side functions and argument checks work without a GPU."""
import ctypes
import subprocess

import numpy as np
import pytest

import gradient_compression_sgd_gb300 as gc
from gradient_compression_sgd_gb300 import build


@pytest.fixture(scope="module")
def L():
    build.build()
    return gc.lib()


def test_exports_every_declared_function(L):
    names = gc.declared_functions()
    assert {"dgc_compress", "adacomp_compress", "sparse_average", "dcd_step", "gcsgd_last_error"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", gc.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)


def test_host_helpers(L):
    assert gc.version() >= 100
    assert gc.dgc_k(0.001, 1_048_576) == 1049
    assert gc.dgc_k(0.001, 1000) == 1
    assert gc.dgc_k(0.5, 0) == 0
    off = np.array([0, 1000, 1000, 50_000], np.int64)
    a = gc.dgc_workspace_size(off, 4, 0.001)
    b = gc.dgc_workspace_size(off, 8, 0.001)
    assert 0 < a < b and a % 256 == 0
    c = gc.adacomp_workspace_size(off, [50, 50, 500], 2, 10_000)
    assert c >= 2 * 10_000 * 8


def _call(L, fn, *args):
    rc = getattr(L, fn)(*args)
    return rc, gc.last_error()


@pytest.mark.parametrize("case", ["density0", "density_gt1", "bad_offsets", "k0", "too_many_segments", "null_grad"])
def test_dgc_rejects_bad_arguments(L, case):
    off = np.array([0, 100, 300], np.int64)
    S, K, density, nodes = 2, 2, 0.01, 1
    grad = ctypes.c_void_p(0x1000)
    if case == "density0":
        density = 0.0
    elif case == "density_gt1":
        density = 1.5
    elif case == "bad_offsets":
        off = np.array([0, 300, 100], np.int64)
    elif case == "k0":
        K = 0
    elif case == "too_many_segments":
        S = gc.MAX_SEGMENTS + 1
        off = np.arange(S + 1, dtype=np.int64)
    elif case == "null_grad":
        grad = None
    p = off.ctypes.data_as(ctypes.c_void_p)
    rc, msg = _call(L, "dgc_compress", p, S, K, grad, ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000), density,
                    0.9, 0.0, nodes, ctypes.c_void_p(0x1000), 100, ctypes.c_void_p(0x1000), None,
                    ctypes.c_void_p(0x1000 * 256), 1 << 30, None)
    assert rc == -1 and msg


def test_dgc_capacity_and_workspace_checked_before_launch(L):
    off = np.array([0, 1000, 5000], np.int64)
    p = off.ctypes.data_as(ctypes.c_void_p)
    need = gc.dgc_workspace_size(off, 1, 0.01)
    x = ctypes.c_void_p(0x1000)
    rc, msg = _call(L, "dgc_compress", p, 2, 1, x, x, x, 0.01, 0.9, 0.0, 1, x, 100, x, None,
                    ctypes.c_void_p(0x10000), need - 256, None)
    assert rc == -3 and "workspace" in msg
    rc, msg = _call(L, "dgc_compress", p, 2, 1, x, x, x, 0.01, 0.9, 0.0, 1, x, 49, x, None,
                    ctypes.c_void_p(0x10000), need, None)
    assert rc == -2 and "cap" in msg
    rc, msg = _call(L, "dgc_compress", p, 2, 1, x, x, x, 0.01, 0.9, 0.0, 1, x, 50, x, None,
                    ctypes.c_void_p(0x10001), need, None)
    assert rc == -1 and "aligned" in msg


def test_other_entry_points_reject_bad_arguments(L):
    x = ctypes.c_void_p(0x1000)
    off = np.array([0, 10], np.int64)
    lt = np.array([0], np.int32)
    rc, msg = _call(L, "adacomp_compress", off.ctypes.data_as(ctypes.c_void_p), 1, lt.ctypes.data_as(ctypes.c_void_p),
                    1, x, x, x, 10, x, x, x, x, 1 << 20, None)
    assert rc == -1 and "lt" in msg
    rc, msg = _call(L, "sparse_average", x, 10, x, 0, 100, x, None)
    assert rc == -1
    rc, msg = _call(L, "sparse_average_update", x, 10, x, 4, 100, ctypes.c_float(float("nan")), x, None)
    assert rc == -1 and "lr" in msg
    rc, msg = _call(L, "sparse_average_update", x, 10, x, 513, 100, ctypes.c_float(0.1), x, None)
    assert rc == -1 and "K" in msg
    w = np.array([1, 1, 1], np.float32)
    rc, msg = _call(L, "dcd_step", 8, 100, w.ctypes.data_as(ctypes.c_void_p), x, x, ctypes.c_float(0.1), 0.0,
                    ctypes.c_uint64(1), ctypes.c_uint32(0), None)
    assert rc == -1 and "keep_p" in msg
    rc, msg = _call(L, "dcd_step", 0, 100, w.ctypes.data_as(ctypes.c_void_p), x, x, ctypes.c_float(0.1), 0.5,
                    ctypes.c_uint64(1), ctypes.c_uint32(0), None)
    assert rc == -1


def test_binding_refuses_cpu_tensors(L):
    torch = pytest.importorskip("torch")
    off = np.array([0, 8], np.int64)
    g = torch.zeros((1, 8))
    with pytest.raises(TypeError):
        gc.dgc_compress(off, g, g, g, torch.zeros((1, 1, 2), dtype=torch.int32), torch.zeros((1, 1), dtype=torch.int64),
                        torch.zeros(1024, dtype=torch.uint8), 0.5, 0.9)


def test_trace_filter_takes_and_clears_a_name(L):
    """Selective tracing is host state: a name is accepted, an over-long one is
    refused, and None goes back to tracing every kernel."""
    gc.trace_only("dgc_update")
    with pytest.raises(gc.GcsgdError):
        gc.trace_only("x" * 48)
    gc.trace_only(None)
    assert L.gcsgd_trace_only(None) == 0


def test_adacomp_emit_table_limit_checked_before_launch(L):
    """K * (4 n_seg + 8) bytes of emit tables above 200 KiB: refused before
    anything is enqueued (no GPU is touched here)."""
    S = gc.MAX_SEGMENTS
    off = np.arange(S + 1, dtype=np.int64)
    lt = np.full(S, 50, np.int32)
    x = ctypes.c_void_p(0x1000)
    ws = ctypes.c_void_p(0x1000 * 256)
    K = 25  # 25 * (4 * 2048 + 8) = 205,000 > 204,800
    rc, msg = _call(L, "adacomp_compress", off.ctypes.data_as(ctypes.c_void_p), S, lt.ctypes.data_as(ctypes.c_void_p),
                    K, x, x, x, S, x, x, x, ws, 1 << 40, None)
    assert rc == -1 and "emit tables" in msg
