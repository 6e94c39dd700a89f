"""Pins of the oracle's regular (strided / transposed) sparse convolution (CPU only).

The reading ("Contribution Tasks — JeffreyXiang/FlexGEMM", §二: sparse_conv3d and
sparse_neighbor_map, output sites that differ from the input sites) is the
convolution torch's dense conv3d computes on the densified grid, kept at the
output sites whose window holds an input; its transposed form is torch's
conv_transpose3d read at the original sites.  Each test ties the oracle to those
library routines (and their autograd), not to the oracle's own loops.
"""
import numpy as np
import pytest
import torch

import oracle
from voxel_gemm_gb300 import synth

NONE = oracle.NONE
CASES = [(2, 2), (3, 2), (3, 1), (2, 1)]  # (kernel, stride)


def _pad27(W, K):
    """[K^3, Cin, Cout] weights as the oracle's 27-tap layout (absent taps zero)."""
    out = np.zeros((27,) + W.shape[1:])
    out[: K ** 3] = W
    return out


def _torch_w(W, K):
    # W[k][ci][co], k = (tx*K + ty)*K + tz  <->  conv3d weight [co][ci][tx][ty][tz]
    cin, cout = W.shape[1], W.shape[2]
    return torch.from_numpy(np.ascontiguousarray(W.transpose(2, 1, 0))).reshape(cout, cin, K, K, K)


def _torch_wt(W, K):
    # conv_transpose3d weight [ci][co][tx][ty][tz]
    cin, cout = W.shape[1], W.shape[2]
    return torch.from_numpy(np.ascontiguousarray(W.transpose(1, 2, 0))).reshape(cin, cout, K, K, K)


def _densify(coords, shape, vals):
    B, X, Y, Z = shape
    d = torch.zeros(B, vals.shape[1], X, Y, Z, dtype=torch.float64)
    c = torch.from_numpy(coords.astype(np.int64))
    d[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]] = torch.from_numpy(vals)
    return d


def _at(dense, coords):
    c = torch.from_numpy(coords.astype(np.int64))
    return dense[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]]


def _case(K, s, seed=0, grid=(2, 8, 10, 6), n=260, cin=3, cout=4):
    coords = synth.random_coords(seed + 10 * K + s, n, *grid)
    rng = np.random.default_rng(seed + 7)
    T = K ** 3
    f = rng.standard_normal((coords.shape[0], cin))
    W = rng.standard_normal((T, cin, cout))
    b = rng.standard_normal(cout)
    return coords, grid, f, W, b


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("K,s", CASES)
def test_output_set_and_order(K, s):
    coords, grid, *_ = _case(K, s)
    co, down, up = oracle.sparse_map(coords, *grid, K, s)
    p = 1 if K == 3 else 0
    occ = _densify(coords, grid, np.ones((coords.shape[0], 1)))
    cnt = torch.nn.functional.conv3d(occ, torch.ones(1, 1, K, K, K, dtype=torch.float64), stride=s, padding=p)
    want = torch.nonzero(cnt[:, 0] > 0.5).numpy().astype(np.int32)  # (b, x, y, z), row-major = linear key order
    assert np.array_equal(co, want)
    # down and up describe the same (output, tap, input) triples
    pairs_d = {(o, k, int(j)) for o, k in zip(*np.nonzero(down != NONE)) for j in [down[o, k]]}
    pairs_u = {(int(up[j, k]), k, j) for j, k in zip(*np.nonzero(up != NONE))}
    assert pairs_d == pairs_u and len(pairs_d) > 0
    assert np.all(down[:, K ** 3:] == NONE) and np.all(up[:, K ** 3:] == NONE)


@pytest.mark.parametrize("K,s", CASES)
def test_strided_conv_equals_dense_conv3d_and_autograd(K, s):
    coords, grid, f, W, b = _case(K, s)
    co, down, up = oracle.sparse_map(coords, *grid, K, s)
    rng = np.random.default_rng(3)
    dY = rng.standard_normal((co.shape[0], W.shape[2]))
    W27 = _pad27(W, K)
    out = oracle.fwd(down, f, W27, b)
    dX = oracle.dgrad_scatter_to(down, dY, W27, coords.shape[0])
    dW, db = oracle.wgrad(down, f, dY)
    p = 1 if K == 3 else 0
    x = _densify(coords, grid, f).requires_grad_(True)
    w = _torch_w(W, K).clone().requires_grad_(True)
    bias = torch.from_numpy(b).clone().requires_grad_(True)
    y = torch.nn.functional.conv3d(x, w, bias, stride=s, padding=p)
    ys = _at(y, co)
    assert _rel(out, ys.detach().numpy()) < 1e-12
    (ys * torch.from_numpy(dY)).sum().backward()
    assert _rel(dX, _at(x.grad, coords).numpy()) < 1e-12
    cout, cin = w.shape[0], w.shape[1]
    assert _rel(dW[: K ** 3], w.grad.reshape(cout, cin, K ** 3).permute(2, 1, 0).numpy()) < 1e-12
    assert np.all(dW[K ** 3:] == 0)
    assert _rel(db, bias.grad.numpy()) < 1e-12


@pytest.mark.parametrize("K,s", CASES)
def test_transposed_conv_equals_dense_conv_transpose3d_and_autograd(K, s):
    coords, grid, _, W, b = _case(K, s, seed=5)
    co, down, up = oracle.sparse_map(coords, *grid, K, s)
    rng = np.random.default_rng(4)
    g = rng.standard_normal((co.shape[0], W.shape[1]))      # features on the coarse sites
    dY = rng.standard_normal((coords.shape[0], W.shape[2]))  # gradient on the fine sites
    W27 = _pad27(W, K)
    out = oracle.fwd(up, g, W27, b)
    dG = oracle.dgrad_scatter_to(up, dY, W27, co.shape[0])
    dW, db = oracle.wgrad(up, g, dY)
    p = 1 if K == 3 else 0
    B, X, Y, Z = grid
    Xo, Yo, Zo = ((v + 2 * p - K) // s + 1 for v in (X, Y, Z))
    # output_padding restores the fine extent exactly
    op = tuple(v - ((vo - 1) * s - 2 * p + K) for v, vo in zip((X, Y, Z), (Xo, Yo, Zo)))
    x = _densify(co, (B, Xo, Yo, Zo), g).requires_grad_(True)
    w = _torch_wt(W, K).clone().requires_grad_(True)
    bias = torch.from_numpy(b).clone().requires_grad_(True)
    y = torch.nn.functional.conv_transpose3d(x, w, bias, stride=s, padding=p, output_padding=op)
    assert tuple(y.shape[2:]) == (X, Y, Z)
    ys = _at(y, coords)
    assert _rel(out, ys.detach().numpy()) < 1e-12
    (ys * torch.from_numpy(dY)).sum().backward()
    assert _rel(dG, _at(x.grad, co).numpy()) < 1e-12
    cin, cout = w.shape[0], w.shape[1]
    assert _rel(dW[: K ** 3], w.grad.reshape(cin, cout, K ** 3).permute(2, 0, 1).numpy()) < 1e-12
    assert _rel(db, bias.grad.numpy()) < 1e-12


@pytest.mark.parametrize("K,s", CASES)
def test_adjoint_identity(K, s):
    coords, grid, f, W, b = _case(K, s, seed=9)
    co, down, up = oracle.sparse_map(coords, *grid, K, s)
    dY = np.random.default_rng(2).standard_normal((co.shape[0], W.shape[2]))
    W27 = _pad27(W, K)
    lhs = float(np.sum(dY * oracle.fwd(down, f, W27, None)))
    rhs = float(np.sum(oracle.dgrad_scatter_to(down, dY, W27, coords.shape[0]) * f))
    assert abs(lhs - rhs) <= 1e-12 * (abs(lhs) + 1.0)


def test_planted_sparse_mistakes_are_caught():
    coords, grid, f, W, b = _case(3, 2, seed=13)
    co, down, up = oracle.sparse_map(coords, *grid, 3, 2)
    x = _densify(coords, grid, f)
    ref = _at(torch.nn.functional.conv3d(x, _torch_w(W, 3), torch.from_numpy(b), stride=2, padding=1), co).numpy()
    # taps in reverse order (the offset sign flipped)
    assert _rel(oracle.fwd(down[:, list(range(26, -1, -1))], f, _pad27(W, 3), b), ref) > 1e-2
    # the up map used as if it were the down map's transpose with flipped taps
    assert not np.array_equal(up[:, :27], up[:, 26::-1])


def test_sparse_map_rejects_bad_arguments():
    c = np.zeros((1, 4), np.int32)
    for K, s in [(4, 2), (3, 3), (1, 1)]:
        with pytest.raises(oracle.OracleError):
            oracle.sparse_map(c, 1, 4, 4, 4, K, s)
    with pytest.raises(oracle.OracleError):
        oracle.sparse_map(np.array([[0, 4, 0, 0]], np.int32), 1, 4, 4, 4, 3, 2)
