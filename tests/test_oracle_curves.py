"""Pins of the oracle's space-filling-curve codes (CPU only).

The pages name z_order_encode/decode and hilbert_encode/decode ("Contribution
Tasks — JeffreyXiang/FlexGEMM", §二 module table, kernels.cuda.serialize) but
print no values; these tests tie the oracle to properties that define the two
curves rather than to its own formulas: each is a bijection of the 2^b cube onto
[0, 8^b) (checked by exhaustion), decode inverts encode (batch index included),
the z-order code nests (a cell's code without its lowest 3 bits is its parent
cell's code, and the 8 children of a cell hold 8 consecutive codes), and the
Hilbert curve is a path: consecutive codes are face neighbours.  A planted
mistake (Hilbert without its Gray coding, or z-order with two axes swapped) fails
one of them.
"""
import numpy as np
import pytest

import oracle


def _cube(bits, b=0):
    R = 1 << bits
    g = np.stack(np.meshgrid(np.arange(R), np.arange(R), np.arange(R), indexing="ij"), -1).reshape(-1, 3)
    return np.concatenate([np.full((g.shape[0], 1), b, np.int32), g.astype(np.int32)], axis=1)


@pytest.mark.parametrize("curve", [oracle.ZORDER, oracle.HILBERT])
@pytest.mark.parametrize("bits", [0, 1, 2, 3, 4])
def test_curve_is_a_bijection_of_the_cube(curve, bits):
    c = _cube(bits)
    codes = oracle.curve_encode(c, bits, curve)
    assert np.array_equal(np.sort(codes), np.arange(8 ** bits, dtype=np.uint64))
    assert np.array_equal(oracle.curve_decode(codes, bits, curve), c)


@pytest.mark.parametrize("curve", [oracle.ZORDER, oracle.HILBERT])
def test_decode_inverts_encode_with_batch(curve):
    rng = np.random.default_rng(4)
    bits = 10
    c = np.concatenate([rng.integers(0, 7, (5000, 1)), rng.integers(0, 1 << bits, (5000, 3))], 1).astype(np.int32)
    codes = oracle.curve_encode(c, bits, curve)
    assert np.array_equal(codes >> np.uint64(3 * bits), c[:, 0].astype(np.uint64))
    assert np.array_equal(oracle.curve_decode(codes, bits, curve), c)


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5])
def test_hilbert_steps_are_unit(bits):
    cells = oracle.curve_decode(np.arange(8 ** bits, dtype=np.uint64), bits, oracle.HILBERT)
    step = np.abs(np.diff(cells[:, 1:].astype(np.int64), axis=0)).sum(axis=1)
    assert np.all(step == 1)
    assert np.array_equal(cells[0], [0, 0, 0, 0])


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_zorder_nests(bits):
    c = _cube(bits)
    codes = oracle.curve_encode(c, bits, oracle.ZORDER)
    parent = c.copy()
    parent[:, 1:] >>= 1
    assert np.array_equal(codes >> np.uint64(3), oracle.curve_encode(parent, bits - 1, oracle.ZORDER))
    # the x bit sits above y, y above z within each level
    one = np.array([[0, 1, 0, 0], [0, 0, 1, 0], [0, 0, 0, 1]], np.int32)
    assert list(oracle.curve_encode(one, bits, oracle.ZORDER)) == [4, 2, 1]


def test_planted_curve_mistakes_are_caught():
    # Hilbert without the Gray coding step of the transposed index is not a path
    bits = 3
    cells = oracle.curve_decode(np.arange(8 ** bits, dtype=np.uint64), bits, oracle.HILBERT)
    # undo a Gray code on the codes: code -> code ^ (code >> 1) reorders the path
    wrong = cells[np.argsort(np.arange(8 ** bits) ^ (np.arange(8 ** bits) >> 1))]
    step = np.abs(np.diff(wrong[:, 1:].astype(np.int64), axis=0)).sum(axis=1)
    assert not np.all(step == 1)
    # z-order with x and z swapped breaks the documented bit positions
    c = np.array([[0, 1, 0, 0]], np.int32)
    assert oracle.curve_encode(c[:, [0, 3, 2, 1]], bits, oracle.ZORDER)[0] != 4


def test_curve_rejects_out_of_range():
    with pytest.raises(oracle.OracleError):
        oracle.curve_encode(np.array([[0, 8, 0, 0]], np.int32), 3, oracle.HILBERT)
    with pytest.raises(oracle.OracleError):
        oracle.curve_encode(np.array([[0, 0, 0, 0]], np.int32), 21, oracle.ZORDER)
