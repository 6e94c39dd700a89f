"""The C-ABI library builds, loads and exports every symbol include/vg.h declares (CPU only).

Only host-side calls are made here (sizes, strings, argument validation that
returns before any device work); nothing computes without a GPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ops():
    from voxel_gemm_gb300 import build, ops
    build.build()
    return ops


def declared_symbols():
    syms = set()
    for name in os.listdir(os.path.join(ROOT, "include")):
        if name.endswith(".h"):
            text = open(os.path.join(ROOT, "include", name)).read()
            syms |= set(re.findall(r"^VG_API\s+[\w\s\*]+?\b(vg_\w+)\s*\(", text, flags=re.M))
    return syms


def test_every_declared_symbol_is_exported(ops):
    syms = declared_symbols()
    assert len(syms) >= 11
    L = ctypes.CDLL(ops.LIB_PATH)
    for s in sorted(syms):
        assert hasattr(L, s), s


def test_host_only_queries(ops):
    assert ops.vg_version() >= 100
    assert ops.vg_strerror(ops.VG_ERR_DUPLICATE_COORD) == "duplicate coordinate"
    assert ops.vg_strerror(12345) == "unknown status"
    n32 = ops.vg_nbrmap_workspace_bytes(1000, 1, 64, 64, 64, ops.VG_MAP_HASH)
    n64 = ops.vg_nbrmap_workspace_bytes(1000, 1, 64, 64, 64, ops.VG_KEY64 | ops.VG_MAP_HASH)
    assert n64 > n32 > 0
    assert ops.vg_nbrmap_workspace_bytes(-1, 1, 8, 8, 8, 0) == 0
    assert ops.vg_nbrmap_workspace_bytes(10, 0, 8, 8, 8, 0) == 0
    assert ops.vg_nbrmap_workspace_bytes(10, 1, 8, 8, 8, ops.VG_KEY32 | ops.VG_KEY64) == 0
    # 32-bit keys cannot address a 2^32-cell grid
    assert ops.vg_nbrmap_workspace_bytes(10, 4, 1024, 1024, 1024, ops.VG_KEY32) == 0
    assert ops.vg_conv_workspace_bytes(1000, 64, 64, ops.VG_F16) > 0
    assert ops.vg_conv_workspace_bytes(1000, 60, 64, ops.VG_F16) == 0      # Cin % 8 != 0
    assert ops.vg_conv_workspace_bytes(1000, 64, 64, 7) == 0               # bad dtype
    assert ops.vg_conv_workspace_bytes(0, 64, 64, ops.VG_BF16) > 0
    # sort-key width of the documented row order: bits of m above F + the 27-bit tap
    # mask + G kept fine bits (G = 6, or fewer so that the key fits 32 bits); 8-bit digits
    for (B, R, bits) in [(4, 64, 2 + 27 + 3), (2, 256, 1 + 27 + 4),
                         (1, 512, 0 + 27 + 5), (1, 1024, 0 + 27 + 5), (1, 2, 0 + 27 + 3)]:
        d = ops.vg_nbrmap_describe(1000, B, R, R, R)
        assert d["sort_bits"] == bits and d["sort_passes"] == (bits + 7) // 8, (B, R, d)
    # kernels per build: (hash) insert, probe, keys or (column index) count, scan,
    # scatter, rank, probe, keys; the radix passes, tile rows, and above 2^17
    # voxels one more pass ordering the tiles region by region
    H = ops.VG_MAP_HASH
    assert ops.vg_nbrmap_describe(1 << 17, 1, 512, 512, 512, H)["launches"] == 4 + 4
    assert ops.vg_nbrmap_describe((1 << 17) + 1, 1, 512, 512, 512, H)["launches"] == 4 + 4 + 1
    C = ops.VG_MAP_COLUMNS
    assert ops.vg_nbrmap_describe(1 << 17, 1, 512, 512, 512, C)["launches"] == 7 + 4
    assert ops.vg_nbrmap_describe((1 << 17) + 1, 1, 512, 512, 512, C)["launches"] == 7 + 4 + 1
    # the 64-bit hash path leaves the plan otherwise unchanged
    d32 = ops.vg_nbrmap_describe(5000, 1, 512, 512, 512, ops.VG_KEY32 | H)
    d64 = ops.vg_nbrmap_describe(5000, 1, 512, 512, 512, ops.VG_KEY64 | H)
    assert (d32["key64"], d64["key64"]) == (0, 1) and d32["sort_passes"] == d64["sort_passes"]
    assert d32["index"] == d64["index"] == "hash"


def test_column_index_choice(ops):
    """Column index by default when the hash table would exceed 64 MiB and the
    (b, x, y) columns number at most 8 N + 2^20 (and at most 2^28); VG_MAP_HASH
    and VG_MAP_COLUMNS force one or the other."""
    d = ops.vg_nbrmap_describe
    assert d(4_915_386, 1, 1024, 1024, 1024)["index"] == "columns"   # 268 MB table
    assert d(602_492, 1, 512, 512, 512)["index"] == "hash"           # 16 MB table
    assert d(25_179, 4, 64, 64, 64)["index"] == "hash"
    assert d(4_915_386, 1, 4096, 1024, 1024)["index"] == "columns"    # 2^22 columns <= 8 N + 2^20
    assert d(4_915_386, 16, 4096, 1024, 1024)["index"] == "hash"      # 2^26 columns > 8 N + 2^20
    assert d(4_915_386, 1, 1024, 1024, 1024, ops.VG_MAP_HASH)["index"] == "hash"
    assert d(25_179, 4, 64, 64, 64, ops.VG_MAP_COLUMNS)["index"] == "columns"
    assert d(3000, 8, 1024, 1024, 1024, ops.VG_MAP_COLUMNS)["index"] == "columns"  # 2^23 columns allowed when forced
    assert d(4000, 1, 32, 32, 32, ops.VG_TEST_SMALL_HASH)["index"] == "hash"
    with pytest.raises(RuntimeError):
        d(1000, 1, 8, 8, 8, ops.VG_MAP_HASH | ops.VG_MAP_COLUMNS)
    with pytest.raises(RuntimeError):
        d(1000, 1, 1 << 15, 1 << 14, 8, ops.VG_MAP_COLUMNS)           # above 2^28 columns
    assert d(1 << 30, 1, 1 << 15, 1 << 14, 8)["index"] == "hash"
    # the column layout keeps its arrays 256-byte aligned for any size (else the
    # query would return 0)
    for n in (1, 2, 3, 255, 4097, 100_003, 4_915_386):
        for grid in ((1, 8, 8, 8), (3, 65, 33, 17), (1, 1024, 1024, 1024), (2, 700, 301, 5)):
            assert d(n, *grid, ops.VG_MAP_COLUMNS)["index"] == "columns"
            assert ops.vg_nbrmap_workspace_bytes(n, *grid, ops.VG_MAP_COLUMNS) > 0, (n, grid)
    # both layouts are valid workspaces of their own size
    assert ops.vg_nbrmap_workspace_bytes(4_915_386, 1, 1024, 1024, 1024) > 0
    assert ops.vg_nbrmap_workspace_bytes(4_915_386, 1, 1024, 1024, 1024, ops.VG_MAP_HASH) > 0


@pytest.mark.parametrize("sms", [152, 148, 76])
def test_split_k_plan(ops, sms):
    """Split-K chunks of the tensor-core weight gradient: about four work units per SM,
    at most 256 tiles per chunk, at least 4 tiles per chunk when there are enough,
    and fp32 partial sums of at most 768 MiB."""
    for N, C in [(25179, 64), (319057, 128), (602492, 256), (602492, 512), (602492, 1024),
                 (4915386, 64), (1000, 64), (128, 256)]:
        d = ops.vg_conv_describe(N, C, C, ops.VG_BF16, sm_count=sms)
        assert d["tensor_core"] == 1
        S, T = d["splits"], (N + 127) // 128
        tpc = (T + S - 1) // S  # tiles per chunk
        assert 1 <= S <= T and (S - 1) * tpc < T, (N, C, S)  # every chunk non-empty
        assert S * 27 * C * C * 4 <= (3 << 28) or S == 1, (N, C, S)
        if T >= 4:
            assert tpc >= 4 or S == 1, (N, C, S)
        if (T + 255) // 256 * 27 * C * C * 4 <= (3 << 28):  # 256-tile chunks fit the cap
            assert tpc <= 256, (N, C, S)


def test_argument_errors_return_before_any_launch(ops):
    L = ops.lib()
    P = ctypes.c_void_p
    # null workspace / coords: rejected on the host
    st = L.vg_nbrmap_build(None, 10, 1, 8, 8, 8, 0, None, 0, None, None, None)
    assert st == ops.VG_ERR_INVALID_ARG
    # misaligned workspace pointer
    st = L.vg_nbrmap_build(P(16), 10, 1, 8, 8, 8, 0, P(0x1001), 1 << 20, P(64), P(64), None)
    assert st == ops.VG_ERR_INVALID_ARG
    # workspace too small
    need = ops.vg_nbrmap_workspace_bytes(10, 1, 8, 8, 8, 0)
    st = L.vg_nbrmap_build(P(256), 10, 1, 8, 8, 8, 0, P(0x10000), need - 1, P(256), P(256), None)
    assert st == ops.VG_ERR_WORKSPACE_TOO_SMALL
    # conv: unsupported channels, unknown flags
    st = L.vg_subm_conv3d_fwd(P(256), P(256), P(256), 10, ops.VG_F16, P(256), P(256), None, P(256),
                              12, 64, 0, P(256), 1 << 20, None)
    assert st == ops.VG_ERR_UNSUPPORTED
    st = L.vg_subm_conv3d_fwd(P(256), P(256), P(256), 10, ops.VG_F16, P(256), P(256), None, P(256),
                              64, 64, 0x80, P(256), 1 << 20, None)
    assert st == ops.VG_ERR_UNSUPPORTED
    st = L.vg_subm_conv3d_bwd(P(256), P(256), P(256), 10, ops.VG_F16, P(256), P(256), P(256),
                              P(256), None, None, 64, 64, 0, P(256), 16, None)
    assert st == ops.VG_ERR_WORKSPACE_TOO_SMALL
    assert L.vg_conv_status(None, None) == ops.VG_ERR_INVALID_ARG
    assert L.vg_nbrmap_status(None, None) == ops.VG_ERR_INVALID_ARG


def test_plans_follow_the_sm_count(ops):
    """The split-K chunk count and the sort grid follow the device's SM count (passed
    explicitly here; 0 means the current device's)."""
    # 319k voxels, C = 128: 14 (M group, N block) units per chunk, about 4 units per SM
    s152 = ops.vg_conv_describe(319057, 128, 128, ops.VG_BF16, sm_count=152)["splits"]
    s76 = ops.vg_conv_describe(319057, 128, 128, ops.VG_BF16, sm_count=76)["splits"]
    assert s152 * 14 >= 4 * 152 and s76 * 14 >= 4 * 76 and s76 < s152, (s76, s152)
    with pytest.raises(ops.VGError):
        ops.vg_conv_describe(1000, 64, 64, ops.VG_BF16, sm_count=-1)
    with pytest.raises(ops.VGError):
        ops.vg_nbrmap_describe(1000, 1, 8, 8, 8, sm_count=-1)
    # without a device, 0 plans for the default count
    import torch
    if not torch.cuda.is_available():
        assert (ops.vg_conv_describe(319057, 128, 128, ops.VG_BF16)["splits"] == s152)

