"""Pins of the oracle's wire encodings (CPU only)."""
import numpy as np
import pytest

import oracle
from conftest import load_golden


def test_dgc_hand_example():
    g = load_golden("wire_examples.txt")
    idx = np.array([int(x) for x in g["dgc_idx"]], np.uint32)
    val = np.array([float(x) for x in g["dgc_val"]], np.float32)
    stream = oracle.dgc_encode(idx, val)
    assert stream.hex() == g["dgc_bytes"][0]
    dense = oracle.dgc_decode(stream, 70001)
    want = np.zeros(70001, np.float32)
    want[idx] = val
    np.testing.assert_array_equal(dense, want)


@pytest.mark.parametrize("seed", range(4))
def test_dgc_round_trip_and_size(seed):
    """Decoding gives the dense vector back; the size is 6 bytes per entry
    plus 6 per full 65536-position escape inside a gap."""
    rng = np.random.default_rng(seed)
    n = 3_000_000
    c = int(rng.integers(1, 400))
    idx = np.sort(rng.choice(n, size=c, replace=False)).astype(np.uint32)
    val = rng.standard_normal(c).astype(np.float32)
    stream = oracle.dgc_encode(idx, val)
    gaps = np.diff(np.concatenate([[-1], idx.astype(np.int64)])) - 1
    assert len(stream) == 6 * (c + int((gaps // 65536).sum()))
    want = np.zeros(n, np.float32)
    want[idx] = val
    np.testing.assert_array_equal(oracle.dgc_decode(stream, n), want)


def test_dgc_rejects_unsorted():
    with pytest.raises(oracle.OracleError):
        oracle.dgc_encode(np.array([5, 3], np.uint32), np.array([1, 1], np.float32))


def test_adacomp_hand_example():
    g = load_golden("wire_examples.txt")
    off = [int(x) for x in g["ada_off"]]
    stream = oracle.adacomp_encode(off, np.array([int(x) for x in g["ada_idx"]], np.uint32),
                                   np.array([float(x) for x in g["ada_val"]], np.float32),
                                   np.array([int(x) for x in g["ada_counts"]], np.int64),
                                   np.array([float(x) for x in g["ada_scales"]], np.float32))
    assert stream.hex() == g["ada_bytes"][0]
    dense = oracle.adacomp_decode(stream, off)
    want = np.zeros(30, np.float32)
    want[[3, 7, 29]] = [0.5, -0.5, -0.25]
    np.testing.assert_array_equal(dense, want)


def test_adacomp_round_trip_of_a_step():
    """The message of one AdaComp step decodes to sign * scale at exactly
    the sent entries; 8 bytes per layer plus 4 per entry."""
    rng = np.random.default_rng(9)
    sizes, lt = [5000, 12000, 77], [50, 500, 10]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    dW = rng.laplace(0, 1e-3, size=(1, off[-1])).astype(np.float32)
    idx, val, counts, scales, totals = oracle.adacomp_step(off, lt, dW, np.zeros_like(dW))
    n = int(totals[0])
    stream = oracle.adacomp_encode(off, idx[0, :n], val[0, :n], counts[0], scales[0])
    assert len(stream) == 8 * len(sizes) + 4 * n
    want = np.zeros(off[-1], np.float32)
    want[idx[0, :n]] = val[0, :n]
    np.testing.assert_array_equal(oracle.adacomp_decode(stream, off), want)
