"""GPU neighbour map vs the oracle: bit-exact nbr and mask on every workload, plus
the sorted row order, tile masks, key-width equivalence and the error records."""
import numpy as np
import pytest
import torch

import oracle
from helpers import coords_of, oracle_map, u32
from voxel_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu

MAP_WORKLOADS = ["sphere16_c32_f32", "b4_r64_spheres_c64_f16", "b2_r256_shapes_c128_bf16",
                 "b1_r512_shapes_c256_bf16", "b1_r1024_shapes_c64_f16"]


def gpu_map(coords_np, grid, flags=0):
    c = torch.from_numpy(coords_np).cuda()
    m = ops.NbrMap.alloc(coords_np.shape[0], grid, flags)
    m.build(c)
    st = m.status()
    return m, st


def order_keys(coords, mask, grid):
    """The documented sort key: batch element (1024^3 Morton block), the tap mask, then the top G fine Morton bits."""
    B, X, Y, Z = grid
    L = int(np.ceil(np.log2(max(X, Y, Z)))) if max(X, Y, Z) > 1 else 0
    c = coords.astype(np.uint64)
    m = c[:, 0] << np.uint64(3 * L)
    for b in range(L):
        for col, pos in ((1, 2), (2, 1), (3, 0)):
            m |= ((c[:, col] >> np.uint64(b)) & np.uint64(1)) << np.uint64(3 * b + pos)
    lb = int(np.ceil(np.log2(B))) if B > 1 else 0
    F = min(3 * L, 30)
    G = min(F, 6)
    coarse = lb + 3 * L - F
    if coarse + 27 + G > 32 and coarse + 27 <= 32:
        G = 32 - 27 - coarse
    F, G = np.uint64(F), np.uint64(G)
    fine = (m & ((np.uint64(1) << F) - np.uint64(1))) >> (F - G)
    return ((m >> F) << (np.uint64(27) + G)) | (mask.astype(np.uint64) << G) | fine


@pytest.mark.parametrize("name", MAP_WORKLOADS)
def test_nbrmap_bit_exact(name):
    wl = synth.WORKLOADS[name]
    coords = coords_of(name)
    nbr_ref, mask_ref = oracle_map(name)
    m, st = gpu_map(coords, wl.grid, wl.key_flag)
    assert st == ops.VG_OK
    assert np.array_equal(u32(m.nbr), nbr_ref)
    assert np.array_equal(u32(m.mask), mask_ref)
    # sorted order: a permutation, stable-sorted by the Morton key
    order = u32(m.sorted_idx()).astype(np.int64)
    n = coords.shape[0]
    assert np.array_equal(np.sort(order), np.arange(n))
    keys = order_keys(coords, mask_ref, wl.grid)[order]
    assert np.all(keys[1:] >= keys[:-1])
    ties = keys[1:] == keys[:-1]
    assert np.all(order[1:][ties] > order[:-1][ties])
    # tile masks: OR of the valid-tap masks of each block of 128 sorted rows
    T = (n + 127) // 128
    pad = np.zeros(T * 128, dtype=np.uint32)
    pad[:n] = mask_ref[order]
    want = np.bitwise_or.reduce(pad.reshape(T, 128), axis=1)
    assert np.array_equal(u32(m.tile_mask()), want)
    # neighbour lists in processing order, padded with VG_NONE to whole tiles
    sn = u32(m.sorted_nbr())
    assert sn.shape == (T * 128, 27)
    assert np.array_equal(sn[:n], nbr_ref[order]) and np.all(sn[n:] == 0xFFFFFFFF)


def test_key_width_does_not_change_the_map():
    name = "b2_r256_shapes_c128_bf16"
    wl = synth.WORKLOADS[name]
    coords = coords_of(name)
    m32, s32 = gpu_map(coords, wl.grid, ops.VG_KEY32 | ops.VG_MAP_HASH)
    m64, s64 = gpu_map(coords, wl.grid, ops.VG_KEY64 | ops.VG_MAP_HASH)
    assert s32 == s64 == ops.VG_OK
    assert torch.equal(m32.nbr, m64.nbr) and torch.equal(m32.mask, m64.mask)
    assert torch.equal(m32.sorted_idx(), m64.sorted_idx())


def test_large_grid_forces_64bit_keys_and_matches():
    # B*X*Y*Z = 2^33 cannot use 32-bit keys; coordinates near the far corner
    coords = synth.random_coords(3, 3000, 8, 1024, 1024, 1024)
    coords[:, 1:] = np.minimum(coords[:, 1:] // 64 + 1000, 1023)  # cluster them
    keys = ((coords[:, 0].astype(np.int64) * 1024 + coords[:, 1]) * 1024 + coords[:, 2]) * 1024 + coords[:, 3]
    _, first = np.unique(keys, return_index=True)
    coords = coords[np.sort(first)]
    nbr_ref, mask_ref = oracle.nbrmap(coords, 8, 1024, 1024, 1024)
    m, st = gpu_map(coords, (8, 1024, 1024, 1024))
    assert st == ops.VG_OK
    assert np.array_equal(u32(m.nbr), nbr_ref) and np.array_equal(u32(m.mask), mask_ref)


@pytest.mark.parametrize("name", MAP_WORKLOADS)
def test_column_index_equals_hash_table(name):
    """The (b, x, y) column index and the hash table must give the same map, row
    order and tiles (the bit-exact test above covers whichever is the default)."""
    wl = synth.WORKLOADS[name]
    coords = coords_of(name)
    n = coords.shape[0]
    assert ops.vg_nbrmap_describe(n, *wl.grid, wl.key_flag | ops.VG_MAP_COLUMNS)["index"] == "columns"
    assert ops.vg_nbrmap_describe(n, *wl.grid, wl.key_flag | ops.VG_MAP_HASH)["index"] == "hash"
    mc, sc = gpu_map(coords, wl.grid, wl.key_flag | ops.VG_MAP_COLUMNS)
    mh, sh = gpu_map(coords, wl.grid, wl.key_flag | ops.VG_MAP_HASH)
    assert sc == sh == ops.VG_OK
    assert torch.equal(mc.nbr, mh.nbr) and torch.equal(mc.mask, mh.mask)
    assert torch.equal(mc.sorted_idx(), mh.sorted_idx()) and torch.equal(mc.tile_mask(), mh.tile_mask())
    assert torch.equal(mc.sorted_nbr(), mh.sorted_nbr())


@pytest.mark.parametrize("flags", [ops.VG_MAP_COLUMNS, ops.VG_MAP_HASH])
@pytest.mark.parametrize("n", [1, 127, 128, 129, 4097, 5000])
def test_ragged_sizes(n, flags):
    coords = synth.random_coords(n, n, 2, 12, 12, 12)
    nbr_ref, mask_ref = oracle.nbrmap(coords, 2, 12, 12, 12)
    m, st = gpu_map(coords, (2, 12, 12, 12), flags)
    assert st == ops.VG_OK
    assert np.array_equal(u32(m.nbr), nbr_ref) and np.array_equal(u32(m.mask), mask_ref)


@pytest.mark.parametrize("flags", [ops.VG_MAP_COLUMNS, ops.VG_MAP_HASH])
def test_solid_block_and_long_columns(flags):
    """Dense input: a solid 14^3 block (every tap of its inner voxels valid) and
    full z-columns of 600 voxels, long enough for the column index's binary search."""
    g = np.stack(np.meshgrid(np.arange(1, 15), np.arange(2, 16), np.arange(3, 17), indexing="ij"), -1).reshape(-1, 3)
    solid = np.concatenate([np.zeros((g.shape[0], 1), np.int64), g], 1)
    zs = np.arange(600)
    cols = [np.stack([np.full(600, b), np.full(600, x), np.full(600, y), zs], 1)
            for b, x, y in [(0, 20, 20), (0, 20, 21), (0, 21, 21), (1, 0, 0), (1, 0, 1), (1, 23, 23)]]
    coords = np.concatenate([solid] + cols).astype(np.int32)
    coords = coords[np.random.default_rng(5).permutation(coords.shape[0])]
    grid = (2, 24, 24, 600)
    assert ops.vg_nbrmap_describe(coords.shape[0], *grid, flags)["index"] == (
        "hash" if flags == ops.VG_MAP_HASH else "columns")
    nbr_ref, mask_ref = oracle.nbrmap(coords, *grid)
    m, st = gpu_map(coords, grid, flags)
    assert st == ops.VG_OK
    assert np.array_equal(u32(m.nbr), nbr_ref) and np.array_equal(u32(m.mask), mask_ref)


def test_empty_map():
    m = ops.NbrMap.alloc(0, (1, 8, 8, 8))
    m.build(torch.zeros(0, 4, dtype=torch.int32, device="cuda"))
    assert m.status() == ops.VG_OK


@pytest.mark.parametrize("flags", [ops.VG_MAP_COLUMNS, ops.VG_MAP_HASH])
def test_duplicate_and_out_of_range_are_reported(flags):
    c = np.array([[0, 1, 1, 1], [0, 2, 2, 2], [0, 1, 1, 1]], dtype=np.int32)
    _, st = gpu_map(c, (1, 8, 8, 8), flags)
    assert st == ops.VG_ERR_DUPLICATE_COORD
    # a duplicate among many voxels, in a long column
    c = np.array([[0, 3, 4, z] for z in range(40)] + [[0, 3, 4, 17]], dtype=np.int32)
    _, st = gpu_map(c, (1, 8, 8, 64), flags)
    assert st == ops.VG_ERR_DUPLICATE_COORD
    for bad in ([1, 0, 0, 0], [0, 8, 0, 0], [0, 0, -1, 0], [0, 0, 0, 9], [-1, 0, 0, 0]):
        c = np.array([[0, 1, 1, 1], bad], dtype=np.int32)
        _, st = gpu_map(c, (1, 8, 8, 8), flags)
        assert st == ops.VG_ERR_COORD_OUT_OF_RANGE


def test_hash_overflow_is_reported():
    coords = synth.random_coords(7, 4000, 1, 32, 32, 32)
    _, st = gpu_map(coords, (1, 32, 32, 32), ops.VG_TEST_SMALL_HASH)
    assert st == ops.VG_ERR_HASH_FULL


def test_bad_map_blocks_the_convolution():
    # a map with a duplicate must make the convolution write nothing
    c = np.array([[0, 1, 1, 1], [0, 2, 2, 2], [0, 1, 1, 1]], dtype=np.int32)
    m, st = gpu_map(c, (1, 8, 8, 8))
    assert st == ops.VG_ERR_DUPLICATE_COORD
    f = torch.randn(3, 16, device="cuda")
    W = torch.randn(27, 16, 16, device="cuda")
    out = torch.full((3, 16), 7.0, device="cuda")
    ws = ops.conv_workspace(3, 16, 16, torch.float32)
    ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, None, out, ws)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


# ---------------------------------------------------------------- serialisation (z-order / Hilbert)
@pytest.mark.parametrize("mode", [ops.VG_CURVE_ZORDER, ops.VG_CURVE_HILBERT])
@pytest.mark.parametrize("bits", [0, 1, 5, 10, 20])
def test_encode_decode_seq_bit_exact(mode, bits):
    rng = np.random.default_rng(bits * 3 + mode)
    n = 20000
    b = rng.integers(0, 5, (n, 1))
    xyz = rng.integers(0, 1 << bits, (n, 3))
    c = np.concatenate([b, xyz], 1).astype(np.int32)
    codes = torch.empty(n, dtype=torch.int64, device="cuda")
    ops.vg_encode_seq(torch.from_numpy(c).cuda(), bits, mode, codes)
    ref = oracle.curve_encode(c, bits, mode)
    assert np.array_equal(codes.cpu().numpy().view(np.uint64), ref)
    back = torch.empty(n, 4, dtype=torch.int32, device="cuda")
    ops.vg_decode_seq(codes, bits, mode, back)
    assert np.array_equal(back.cpu().numpy(), c)


def test_encode_seq_marks_out_of_range_rows():
    c = np.array([[0, 8, 0, 0], [0, 1, 2, 3], [-1, 0, 0, 0]], np.int32)
    codes = torch.empty(3, dtype=torch.int64, device="cuda")
    ops.vg_encode_seq(torch.from_numpy(c).cuda(), 3, ops.VG_CURVE_HILBERT, codes)
    got = codes.cpu().numpy().view(np.uint64)
    assert got[0] == np.uint64(0xFFFFFFFFFFFFFFFF) and got[2] == np.uint64(0xFFFFFFFFFFFFFFFF)
    assert got[1] == oracle.curve_encode(c[1:2], 3, oracle.HILBERT)[0]


def hilbert_order_keys(coords, mask, grid):
    """The documented sort key with the Hilbert code (from the oracle) in place of Morton."""
    B, X, Y, Z = grid
    L = int(np.ceil(np.log2(max(X, Y, Z)))) if max(X, Y, Z) > 1 else 0
    m = oracle.curve_encode(coords, L, oracle.HILBERT)
    lb = int(np.ceil(np.log2(B))) if B > 1 else 0
    F = min(3 * L, 30)
    G = min(F, 6)
    coarse = lb + 3 * L - F
    if coarse + 27 + G > 32 and coarse + 27 <= 32:
        G = 32 - 27 - coarse
    F, G = np.uint64(F), np.uint64(G)
    fine = (m & ((np.uint64(1) << F) - np.uint64(1))) >> (F - G)
    return ((m >> F) << (np.uint64(27) + G)) | (mask.astype(np.uint64) << G) | fine


@pytest.mark.parametrize("name", ["b4_r64_spheres_c64_f16", "b2_r256_shapes_c128_bf16", "b1_r512_shapes_c256_bf16"])
def test_hilbert_row_order(name):
    # VG_ORDER_HILBERT leaves the map unchanged and sorts the rows by the Hilbert key
    wl = synth.WORKLOADS[name]
    coords = coords_of(name)
    nbr_ref, mask_ref = oracle_map(name)
    m, st = gpu_map(coords, wl.grid, wl.key_flag | ops.VG_ORDER_HILBERT)
    assert st == ops.VG_OK
    assert np.array_equal(u32(m.nbr), nbr_ref) and np.array_equal(u32(m.mask), mask_ref)
    order = u32(m.sorted_idx()).astype(np.int64)
    n = coords.shape[0]
    assert np.array_equal(np.sort(order), np.arange(n))
    keys = hilbert_order_keys(coords, mask_ref, wl.grid)[order]
    assert np.all(keys[1:] >= keys[:-1])
    ties = keys[1:] == keys[:-1]
    assert np.all(order[1:][ties] > order[:-1][ties])
    T = (n + 127) // 128
    pad = np.zeros(T * 128, dtype=np.uint32)
    pad[:n] = mask_ref[order]
    assert np.array_equal(u32(m.tile_mask()), np.bitwise_or.reduce(pad.reshape(T, 128), axis=1))
    sn = u32(m.sorted_nbr())
    assert np.array_equal(sn[:n], nbr_ref[order]) and np.all(sn[n:] == 0xFFFFFFFF)
