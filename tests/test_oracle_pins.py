"""Pins of the CPU oracle to things other than itself (CPU only).

Each test ties one oracle function to a fact fixed by the mathematics or by a
library routine: brute-force neighbour search, the dense torch conv3d on the
densified grid (and its autograd), the 1x1x1 special case (a plain matmul), an
all-ones closed form, permutation equivariance, the adjoint identity and
central finite differences.  The ``planted`` tests feed the oracle a
plausible mistake (a flipped tap order, a transposed weight, a wrong offset
sign) and check that the pins reject it.
"""
import numpy as np
import pytest
import torch

import oracle
from voxel_gemm_gb300 import synth

NONE = oracle.NONE


def _offsets():
    return np.array([(k // 9 - 1, (k // 3) % 3 - 1, k % 3 - 1) for k in range(27)], dtype=np.int64)


def _small_case(seed=0, n=200, B=2, R=8, cin=3, cout=5):
    coords = synth.random_coords(seed, n, B, R, R, R)
    rng = np.random.default_rng(seed + 100)
    f = rng.standard_normal((coords.shape[0], cin))
    W = rng.standard_normal((27, cin, cout))
    b = rng.standard_normal(cout)
    dY = rng.standard_normal((coords.shape[0], cout))
    return coords, (B, R, R, R), f, W, b, dY


def _sphere_case(cin=4, cout=6, seed=3):
    wl = synth.WORKLOADS["sphere16_c32_f32"]
    coords = synth.make_coords(wl)
    rng = np.random.default_rng(seed)
    f = rng.standard_normal((coords.shape[0], cin))
    W = rng.standard_normal((27, cin, cout))
    b = rng.standard_normal(cout)
    dY = rng.standard_normal((coords.shape[0], cout))
    return coords, wl.grid, f, W, b, dY


def _aniso_case(seed=7, n=300, cin=3, cout=4):
    # a grid with three different extents and three batch elements, so a mix-up of
    # the axes in the linearisation or in the tap offsets cannot go unnoticed
    grid = (3, 5, 9, 13)
    coords = synth.random_coords(seed, n, *grid)
    rng = np.random.default_rng(seed + 100)
    f = rng.standard_normal((coords.shape[0], cin))
    W = rng.standard_normal((27, cin, cout))
    b = rng.standard_normal(cout)
    dY = rng.standard_normal((coords.shape[0], cout))
    return coords, grid, f, W, b, dY


CASES = {"random8": _small_case, "sphere16": _sphere_case, "aniso_3x5x9x13": _aniso_case}


def _brute_nbr(coords, grid):
    B, X, Y, Z = grid
    c = coords.astype(np.int64)
    n = c.shape[0]
    nbr = np.full((n, 27), NONE, dtype=np.uint32)
    for k, (dx, dy, dz) in enumerate(_offsets()):
        t = c + np.array([0, dx, dy, dz])
        eq = np.all(t[:, None, :] == c[None, :, :], axis=2)  # [n, n]
        hit = eq.any(axis=1)
        nbr[hit, k] = eq[hit].argmax(axis=1).astype(np.uint32)
    return nbr


def _dense_torch_w(W):
    # W[k][ci][co] with k = 9(dx+1)+3(dy+1)+(dz+1)  <->  torch w[co][ci][dx+1][dy+1][dz+1]
    cin, cout = W.shape[1], W.shape[2]
    return torch.from_numpy(np.ascontiguousarray(W.transpose(2, 1, 0))).reshape(cout, cin, 3, 3, 3)


def _densify(coords, grid, vals):
    B, X, Y, Z = grid
    d = torch.zeros(B, vals.shape[1], X, Y, Z, dtype=torch.float64)
    c = torch.from_numpy(coords.astype(np.int64))
    d[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]] = torch.from_numpy(vals)
    return d


def _read_sites(dense, coords):
    c = torch.from_numpy(coords.astype(np.int64))
    return dense[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]].numpy()


def _dense_fwd_bwd(coords, grid, f, W, b, dY):
    """Dense conv3d(padding=1) on the densified grid, read at the active sites, and its autograd."""
    x = _densify(coords, grid, f).requires_grad_(True)
    w = _dense_torch_w(W).clone().requires_grad_(True)
    bias = torch.from_numpy(b).clone().requires_grad_(True)
    out = torch.nn.functional.conv3d(x, w, bias, padding=1)
    c = torch.from_numpy(coords.astype(np.int64))
    out_sites = out[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]]
    loss = (out_sites * torch.from_numpy(dY)).sum()
    loss.backward()
    dX = _read_sites(x.grad, coords)
    cout, cin = w.shape[0], w.shape[1]
    dW = w.grad.reshape(cout, cin, 27).permute(2, 1, 0).numpy()
    return out_sites.detach().numpy(), dX, dW, bias.grad.numpy()


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ---------------------------------------------------------------- generator
def test_generator_sphere_matches_bruteforce():
    wl = synth.WORKLOADS["sphere16_c32_f32"]
    coords = synth.make_coords(wl)
    g = np.stack(np.meshgrid(*[np.arange(16)] * 3, indexing="ij"), -1).reshape(-1, 3)
    d = synth.surface_distance("sphere", (8.0, 8.0, 8.0), (5.0,), g[:, 0], g[:, 1], g[:, 2])
    ref = {tuple(v) for v in g[np.abs(d) <= 0.5]}
    got = {tuple(v) for v in coords[:, 1:].tolist()}
    assert got == ref and coords.shape[0] == len(ref)
    assert np.all(coords[:, 0] == 0)


@pytest.mark.parametrize("kind,centre,radii", [
    ("torus", (15.3, 16.7, 14.2), (9.0, 2.6)),
    ("torus", (2.0, 30.0, 16.0), (8.0, 0.4)),     # thin tube, clipped by the grid
    ("sphere", (31.0, 1.5, 20.0), (12.25,)),       # clipped by the grid
])
def test_generator_shell_matches_bruteforce(kind, centre, radii):
    got = synth.shell_voxels(kind, centre, radii, 32)
    g = np.stack(np.meshgrid(*[np.arange(32)] * 3, indexing="ij"), -1).reshape(-1, 3)
    d = synth.surface_distance(kind, centre, radii, g[:, 0], g[:, 1], g[:, 2])
    ref = {tuple(v) for v in g[np.abs(d) <= 0.5]}
    assert {tuple(v) for v in got.tolist()} == ref


def test_generator_is_seeded_and_deduplicated():
    wl = synth.WORKLOADS["b4_r64_spheres_c64_f16"]
    a, b = synth.make_coords(wl), synth.make_coords(wl)
    assert np.array_equal(a, b)
    keys = ((a[:, 0].astype(np.int64) * 64 + a[:, 1]) * 64 + a[:, 2]) * 64 + a[:, 3]
    assert np.unique(keys).size == keys.size
    assert a.min() >= 0 and a[:, 1:].max() < 64 and a[:, 0].max() < 4


# ---------------------------------------------------------------- neighbour map
@pytest.mark.parametrize("case", list(CASES))
def test_nbrmap_matches_bruteforce(case):
    coords, grid, *_ = CASES[case]()
    nbr, mask = oracle.nbrmap(coords, *grid)
    ref = _brute_nbr(coords, grid)
    assert np.array_equal(nbr, ref)
    bits = (nbr != NONE).astype(np.uint64) << np.arange(27, dtype=np.uint64)
    assert np.array_equal(mask.astype(np.uint64), bits.sum(axis=1))


@pytest.mark.parametrize("case", list(CASES))
def test_nbrmap_invariants(case):
    coords, grid, *_ = CASES[case]()
    nbr, mask = oracle.nbrmap(coords, *grid)
    n = coords.shape[0]
    assert np.array_equal(nbr[:, 13], np.arange(n, dtype=np.uint32))
    # symmetry: nbr[i][k] = j  <=>  nbr[j][26-k] = i
    i, k = np.nonzero(nbr != NONE)
    j = nbr[i, k].astype(np.int64)
    assert np.array_equal(nbr[j, 26 - k].astype(np.int64), i)
    pop = np.array([bin(int(m)).count("1") for m in mask])
    assert np.array_equal(pop, (nbr != NONE).sum(axis=1))
    P = int(pop.sum())
    assert (P - n) % 2 == 0
    # batches never interact
    valid = nbr != NONE
    rows = np.nonzero(valid)
    assert np.array_equal(coords[rows[0], 0], coords[nbr[rows].astype(np.int64), 0])


def test_nbrmap_thin_shell_density():
    # a 1-voxel-thick sphere shell is locally a plane: about 9-11 of the 27 taps are active
    coords = synth.make_coords(synth.WORKLOADS["b4_r64_spheres_c64_f16"])
    _, mask = oracle.nbrmap(coords, 4, 64, 64, 64)
    pn = sum(bin(int(m)).count("1") for m in mask) / coords.shape[0]
    assert 8.0 < pn < 13.0


def test_nbrmap_errors_and_empty():
    c = np.array([[0, 1, 2, 3], [0, 1, 2, 4]], dtype=np.int32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.nbrmap(np.array([[0, 1, 2, 3], [0, 1, 2, 3]], np.int32), 1, 8, 8, 8)
    assert e.value.code == oracle.DUPLICATE
    for bad in ([1, 0, 0, 0], [0, 8, 0, 0], [0, 0, -1, 0], [0, 0, 0, 8]):
        with pytest.raises(oracle.OracleError) as e:
            oracle.nbrmap(np.array([bad], np.int32), 1, 8, 8, 8)
        assert e.value.code == oracle.OUT_OF_RANGE
    nbr, mask = oracle.nbrmap(np.zeros((0, 4), np.int32), 1, 8, 8, 8)
    assert nbr.shape == (0, 27) and mask.shape == (0,)
    nbr, mask = oracle.nbrmap(c, 1, 8, 8, 8)
    assert nbr[0, 14] == 1 and nbr[1, 12] == 0 and bin(int(mask[0])).count("1") == 2


def test_nbrmap_grid_boundary_is_absent():
    # corner voxels: neighbours outside the grid do not wrap around
    c = np.array([[0, 0, 0, 0], [0, 3, 3, 3], [0, 3, 0, 0], [0, 0, 3, 3]], dtype=np.int32)
    nbr, mask = oracle.nbrmap(c, 1, 4, 4, 4)
    assert np.all(mask == (1 << 13))


# ---------------------------------------------------------------- forward
@pytest.mark.parametrize("case", list(CASES))
def test_fwd_equals_dense_conv3d(case):
    coords, grid, f, W, b, dY = CASES[case]()
    nbr, _ = oracle.nbrmap(coords, *grid)
    out = oracle.fwd(nbr, f, W, b)
    ref = _dense_fwd_bwd(coords, grid, f, W, b, dY)[0]
    assert _rel(out, ref) < 1e-12


def test_fwd_1x1x1_is_matmul():
    coords, grid, f, W, b, _ = _small_case(cin=7, cout=4)
    W1 = np.zeros_like(W)
    W1[13] = W[13]
    nbr, _ = oracle.nbrmap(coords, *grid)
    out = oracle.fwd(nbr, f, W1, b)
    assert _rel(out, f @ W[13] + b) < 1e-14


def test_fwd_all_ones_closed_form():
    coords, grid, f, W, b, _ = _sphere_case(cin=5, cout=3)
    nbr, mask = oracle.nbrmap(coords, *grid)
    out = oracle.fwd(nbr, np.ones_like(f), np.ones_like(W), b)
    pop = np.array([bin(int(m)).count("1") for m in mask], dtype=np.float64)
    assert np.array_equal(out, pop[:, None] * 5 + b[None, :])


def test_fwd_bias_none_is_zero_bias():
    coords, grid, f, W, b, _ = _small_case()
    nbr, _ = oracle.nbrmap(coords, *grid)
    assert np.array_equal(oracle.fwd(nbr, f, W, None), oracle.fwd(nbr, f, W, np.zeros_like(b)))


def test_permutation_equivariance():
    coords, grid, f, W, b, dY = _small_case(seed=5)
    nbr, _ = oracle.nbrmap(coords, *grid)
    perm = np.random.default_rng(9).permutation(coords.shape[0])
    nbr_p, _ = oracle.nbrmap(coords[perm], *grid)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    relabel = np.where(nbr[perm] == NONE, NONE, inv[np.minimum(nbr[perm], perm.size - 1)])
    assert np.array_equal(nbr_p, relabel.astype(np.uint32))
    out = oracle.fwd(nbr, f, W, b)
    out_p = oracle.fwd(nbr_p, f[perm], W, b)
    assert _rel(out_p, out[perm]) < 1e-13
    dX = oracle.dgrad_scatter(nbr, dY, W)
    dX_p = oracle.dgrad_scatter(nbr_p, dY[perm], W)
    assert _rel(dX_p, dX[perm]) < 1e-13
    dW, db = oracle.wgrad(nbr, f, dY)
    dW_p, db_p = oracle.wgrad(nbr_p, f[perm], dY[perm])
    assert _rel(dW_p, dW) < 1e-13 and _rel(db_p, db) < 1e-13


# ---------------------------------------------------------------- backward
@pytest.mark.parametrize("case", list(CASES))
def test_bwd_equals_dense_autograd(case):
    coords, grid, f, W, b, dY = CASES[case]()
    nbr, _ = oracle.nbrmap(coords, *grid)
    _, dX_ref, dW_ref, db_ref = _dense_fwd_bwd(coords, grid, f, W, b, dY)
    assert _rel(oracle.dgrad_scatter(nbr, dY, W), dX_ref) < 1e-12
    assert _rel(oracle.dgrad_rows(nbr, dY, W), dX_ref) < 1e-12
    dW, db = oracle.wgrad(nbr, f, dY)
    assert _rel(dW, dW_ref) < 1e-12
    # grad_bias from the dense convolution's own autograd (torch's bias gradient of
    # conv3d reduces over the whole grid; only active sites carry a non-zero dY)
    assert _rel(db, db_ref) < 1e-12


@pytest.mark.parametrize("case", list(CASES))
def test_adjoint_identity(case):
    coords, grid, f, W, b, dY = CASES[case]()
    nbr, _ = oracle.nbrmap(coords, *grid)
    lhs = float(np.sum(dY * oracle.fwd(nbr, f, W, None)))
    rhs = float(np.sum(oracle.dgrad_scatter(nbr, dY, W) * f))
    assert abs(lhs - rhs) <= 1e-12 * (abs(lhs) + 1.0)


def test_dgrad_rows_subset_equals_scatter():
    coords, grid, f, W, b, dY = _sphere_case(cin=6, cout=5)
    nbr, _ = oracle.nbrmap(coords, *grid)
    full = oracle.dgrad_scatter(nbr, dY, W)
    rows = np.random.default_rng(1).choice(coords.shape[0], 40, replace=False)
    sub = oracle.dgrad_rows(nbr[rows], dY, W)
    assert _rel(sub, full[rows]) < 1e-13


def test_wgrad_finite_differences():
    coords, grid, f, W, b, dY = _small_case(seed=11, cin=4, cout=3)
    nbr, _ = oracle.nbrmap(coords, *grid)
    dW, _ = oracle.wgrad(nbr, f, dY)
    rng = np.random.default_rng(12)
    for _ in range(3):
        E = rng.standard_normal(W.shape)
        h = 1e-3
        lp = np.sum(dY * oracle.fwd(nbr, f, W + h * E, b))
        lm = np.sum(dY * oracle.fwd(nbr, f, W - h * E, b))
        fd = (lp - lm) / (2 * h)
        assert abs(fd - np.sum(dW * E)) <= 1e-8 * (abs(fd) + 1.0)


# ---------------------------------------------------------------- planted mistakes
def test_planted_flipped_taps_is_caught():
    coords, grid, f, W, b, dY = _small_case(seed=21)
    nbr, _ = oracle.nbrmap(coords, *grid)
    ref = _dense_fwd_bwd(coords, grid, f, W, b, dY)[0]
    wrong = oracle.fwd(nbr, f, W[::-1].copy(), b)       # taps in reverse order (o_k -> -o_k)
    assert _rel(wrong, ref) > 1e-2


def test_planted_transposed_weight_is_caught():
    coords, grid, f, W, b, dY = _small_case(seed=22, cin=4, cout=4)
    nbr, _ = oracle.nbrmap(coords, *grid)
    ref, dX_ref, _, _ = _dense_fwd_bwd(coords, grid, f, W, b, dY)
    assert _rel(oracle.fwd(nbr, f, W.transpose(0, 2, 1).copy(), b), ref) > 1e-2
    assert _rel(oracle.dgrad_rows(nbr, dY, W.transpose(0, 2, 1).copy()), dX_ref) > 1e-2


def test_planted_wrong_offset_sign_is_caught():
    coords, grid, *_ = _small_case(seed=23)
    nbr, _ = oracle.nbrmap(coords, *grid)
    ref = _brute_nbr(coords, grid)
    assert not np.array_equal(nbr[:, ::-1], ref)      # a map built with -o_k fails brute force


def test_planted_dropped_bias_is_caught():
    coords, grid, f, W, b, dY = _small_case(seed=24)
    nbr, _ = oracle.nbrmap(coords, *grid)
    ref = _dense_fwd_bwd(coords, grid, f, W, b, dY)[0]
    assert _rel(oracle.fwd(nbr, f, W, None), ref) > 1e-3


def test_planted_masked_bias_gradient_is_caught():
    # a grad_bias that sums dY only over rows with some neighbour besides the centre
    # (a plausible slip when db is folded into the per-tap weight-gradient loop)
    coords, grid, f, W, b, dY = _small_case(seed=25, n=60)
    nbr, mask = oracle.nbrmap(coords, *grid)
    db_ref = _dense_fwd_bwd(coords, grid, f, W, b, dY)[3]
    lonely = mask == (1 << 13)
    assert lonely.any()
    wrong = dY[~lonely].sum(axis=0)
    assert _rel(wrong, db_ref) > 1e-3
    _, db = oracle.wgrad(nbr, f, dY)
    assert _rel(db, db_ref) < 1e-12

