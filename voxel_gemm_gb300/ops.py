"""Thin ctypes binding of include/vg.h: argument marshalling only.

Each ``vg_*`` function has the C name and takes torch CUDA tensors (device
memory comes from torch; the library allocates nothing).  Status codes other
than VG_OK raise ``VGError``.  All computation happens inside
``libvoxelgemm.so``; if that library is missing the first call raises, there
is no fallback.

The small ``NbrMap`` / ``ConvWorkspace`` helpers only allocate the caller-owned
buffers with torch and keep the pointers together.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

VG_OK, VG_ERR_INVALID_ARG, VG_ERR_COORD_OUT_OF_RANGE, VG_ERR_DUPLICATE_COORD = 0, 1, 2, 3
VG_ERR_HASH_FULL, VG_ERR_UNSUPPORTED, VG_ERR_WORKSPACE_TOO_SMALL, VG_ERR_CUDA = 4, 5, 6, 7
VG_ERR_DEVICE_TIMEOUT = 8
VG_F32, VG_F16, VG_BF16 = 0, 1, 2
VG_KEY32, VG_KEY64, VG_ORDER_HILBERT, VG_MAP_HASH, VG_MAP_COLUMNS = 0x1, 0x2, 0x4, 0x8, 0x40
VG_TEST_SMALL_HASH = 0x100
VG_CURVE_ZORDER, VG_CURVE_HILBERT = 0, 1
VG_ALLOW_TF32, VG_NO_SMALL_N_SPLIT = 0x10, 0x20
VG_NONE = 0xFFFFFFFF
VG_TILE_ROWS = 128

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libvoxelgemm.so")
_lock = threading.Lock()
_lib = None

_DT = {torch.float32: VG_F32, torch.float16: VG_F16, torch.bfloat16: VG_BF16}


class SparseMapStruct(ctypes.Structure):
    """Mirror of vg_sparse_map (include/vg.h)."""
    _fields_ = [("n_in", ctypes.c_int64), ("n_out", ctypes.c_int64), ("kernel", ctypes.c_int),
                ("stride", ctypes.c_int), ("taps", ctypes.c_int), ("out_grid", ctypes.c_int * 4),
                ("side_in", ctypes.c_void_p), ("side_out", ctypes.c_void_p), ("down", ctypes.c_void_p),
                ("down_mask", ctypes.c_void_p), ("up", ctypes.c_void_p), ("up_mask", ctypes.c_void_p),
                ("coords_out", ctypes.c_void_p)]


class VGError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {vg_strerror(status)} (status {status})")
        self.status = status


def lib():
    """The loaded libvoxelgemm.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m voxel_gemm_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, U, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint, ctypes.c_size_t
        sig = {
            "vg_strerror": ([I], ctypes.c_char_p),
            "vg_version": ([], I),
            "vg_nbrmap_workspace_bytes": ([I64, I, I, I, I, U], SZ),
            "vg_nbrmap_build": ([P, I64, I, I, I, I, U, P, SZ, P, P, P], I),
            "vg_nbrmap_status": ([P, P], I),
            "vg_nbrmap_sorted_idx": ([P], P),
            "vg_nbrmap_tile_mask": ([P, I64], P),
            "vg_nbrmap_sorted_nbr": ([P, I64], P),
            "vg_conv_workspace_bytes": ([I64, I, I, I, U], SZ),
            "vg_subm_conv3d_fwd": ([P, P, P, I64, I, P, P, P, P, I, I, U, P, SZ, P], I),
            "vg_subm_conv3d_bwd": ([P, P, P, I64, I, P, P, P, P, P, P, I, I, U, P, SZ, P], I),
            "vg_conv_status": ([P, P], I),
            "vg_nbrmap_describe": ([I64, I, I, I, I, U, I, ctypes.POINTER(ctypes.c_int)], I),
            "vg_conv_describe": ([I64, I, I, I, U, I, ctypes.POINTER(ctypes.c_int)], I),
            "vg_subm_conv3d_fwd_noalloc": ([P, P, P, I64, I, P, P, P, P, I, I, U, P], I),
            "vg_subm_conv3d_fwd_noalloc_status": ([P], I),
            "vg_sum_ordered": ([P, I, I64, I, P, P], I),
            "vg_encode_seq": ([P, I64, I, I, P, P], I),
            "vg_sparse_map_workspace_bytes": ([I64, I, I, I, I, I, I, U], SZ),
            "vg_sparse_map_build": ([P, I64, I, I, I, I, I, I, U, P, SZ, ctypes.POINTER(SparseMapStruct), P], I),
            "vg_sparse_conv_workspace_bytes": ([ctypes.POINTER(SparseMapStruct), I, I, I, I, U], SZ),
            "vg_sparse_conv3d_fwd": ([ctypes.POINTER(SparseMapStruct), I, I, P, P, P, P, I, I, U, P, SZ, P], I),
            "vg_sparse_conv3d_bwd": ([ctypes.POINTER(SparseMapStruct), I, I, P, P, P, P, P, P, I, I, U, P, SZ, P],
                                     I),
            "vg_decode_seq": ([P, I64, I, I, P, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
        return L


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st: int, where: str):
    if st != VG_OK:
        raise VGError(st, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _DT[t.dtype]


def vg_strerror(status: int) -> str:
    return lib().vg_strerror(int(status)).decode()


def vg_version() -> int:
    return lib().vg_version()


def vg_nbrmap_workspace_bytes(N: int, B: int, X: int, Y: int, Z: int, flags: int = 0) -> int:
    return int(lib().vg_nbrmap_workspace_bytes(N, B, X, Y, Z, flags))


def vg_nbrmap_build(coords, B, X, Y, Z, flags, ws, nbr, mask, stream=None) -> None:
    N = coords.shape[0]
    _check(lib().vg_nbrmap_build(_p(coords), N, B, X, Y, Z, flags, _p(ws), ws.numel() * ws.element_size(),
                                 _p(nbr), _p(mask), _s(stream)), "vg_nbrmap_build")


def vg_nbrmap_status(ws, stream=None) -> int:
    return lib().vg_nbrmap_status(_p(ws), _s(stream))


def vg_nbrmap_sorted_idx(ws, N: int) -> torch.Tensor:
    """View of the workspace's sorted_idx [N] (int32 storage of uint32 values)."""
    off = lib().vg_nbrmap_sorted_idx(_p(ws)) - ws.data_ptr()
    return ws.view(torch.uint8)[off: off + 4 * N].view(torch.int32)


def vg_nbrmap_tile_mask(ws, N: int) -> torch.Tensor:
    """View of the workspace's per-tile masks [ceil(N/128)] (int32 storage of uint32 values)."""
    off = lib().vg_nbrmap_tile_mask(_p(ws), N) - ws.data_ptr()
    T = (N + VG_TILE_ROWS - 1) // VG_TILE_ROWS
    return ws.view(torch.uint8)[off: off + 4 * T].view(torch.int32)


def vg_nbrmap_sorted_nbr(ws, N: int) -> torch.Tensor:
    """View of the workspace's neighbour lists in processing order [ceil(N/128)*128, 27]."""
    off = lib().vg_nbrmap_sorted_nbr(_p(ws), N) - ws.data_ptr()
    R = (N + VG_TILE_ROWS - 1) // VG_TILE_ROWS * VG_TILE_ROWS
    return ws.view(torch.uint8)[off: off + 4 * 27 * R].view(torch.int32).view(R, 27)


def vg_conv_workspace_bytes(N: int, Cin: int, Cout: int, dtype, flags: int = 0) -> int:
    code = dtype if isinstance(dtype, int) else _DT[dtype]
    return int(lib().vg_conv_workspace_bytes(N, Cin, Cout, code, flags))


def vg_subm_conv3d_fwd(nbr_ws, nbr, mask, feats, weight, bias, out, conv_ws, flags=0, stream=None) -> None:
    N, Cin = feats.shape
    Cout = weight.shape[2]
    _check(lib().vg_subm_conv3d_fwd(_p(nbr_ws), _p(nbr), _p(mask), N, _dtype_code(feats), _p(feats),
                                    _p(weight), _p(bias), _p(out), Cin, Cout, flags, _p(conv_ws),
                                    conv_ws.numel() * conv_ws.element_size(), _s(stream)),
           "vg_subm_conv3d_fwd")


def vg_subm_conv3d_fwd_noalloc(nbr_ws, nbr, mask, feats, weight, bias, out, flags=0, stream=None) -> None:
    """Forward without a workspace argument (scratch is a fixed array inside the library)."""
    N, Cin = feats.shape
    Cout = weight.shape[2]
    _check(lib().vg_subm_conv3d_fwd_noalloc(_p(nbr_ws), _p(nbr), _p(mask), N, _dtype_code(feats), _p(feats),
                                            _p(weight), _p(bias), _p(out), Cin, Cout, flags, _s(stream)),
           "vg_subm_conv3d_fwd_noalloc")


def vg_subm_conv3d_fwd_noalloc_status(stream=None) -> int:
    """Device-side status of the last no-allocation forward on the current device (syncs `stream`)."""
    return lib().vg_subm_conv3d_fwd_noalloc_status(_s(stream))


def vg_subm_conv3d_bwd(nbr_ws, nbr, mask, grad_out, feats, weight, grad_feats, grad_weight, grad_bias,
                       conv_ws, flags=0, stream=None) -> None:
    N, Cout = grad_out.shape
    Cin = weight.shape[1]
    _check(lib().vg_subm_conv3d_bwd(_p(nbr_ws), _p(nbr), _p(mask), N, _dtype_code(grad_out), _p(grad_out),
                                    _p(feats), _p(weight), _p(grad_feats), _p(grad_weight), _p(grad_bias),
                                    Cin, Cout, flags, _p(conv_ws), conv_ws.numel() * conv_ws.element_size(),
                                    _s(stream)),
           "vg_subm_conv3d_bwd")


def vg_nbrmap_describe(N, B, X, Y, Z, flags=0, sm_count=0) -> dict:
    info = (ctypes.c_int * 4)()
    _check(lib().vg_nbrmap_describe(N, B, X, Y, Z, flags, sm_count, info), "vg_nbrmap_describe")
    return {"key64": 1 if info[0] == 1 else 0, "index": "columns" if info[0] == 2 else "hash",
            "sort_bits": info[1], "sort_passes": info[2], "launches": info[3]}


def vg_conv_describe(N, Cin, Cout, dtype, flags=0, sm_count=0) -> dict:
    code = dtype if isinstance(dtype, int) else _DT[dtype]
    info = (ctypes.c_int * 4)()
    _check(lib().vg_conv_describe(N, Cin, Cout, code, flags, sm_count, info), "vg_conv_describe")
    return {"tensor_core": info[0], "splits": info[1], "launches_fwd": info[2], "launches_bwd": info[3]}


def vg_sum_ordered(parts, out, stream=None) -> None:
    """out = parts[0] + parts[1] + ... (fp32 adds in index order, one rounding); parts [n, *out.shape]."""
    if parts.dtype != out.dtype or parts.shape[1:] != out.shape or not parts.is_contiguous() \
            or not out.is_contiguous():
        raise ValueError("vg_sum_ordered: parts must be [n, *out.shape], contiguous, of out's dtype")
    _check(lib().vg_sum_ordered(_p(parts), parts.shape[0], out.numel(), _dtype_code(out), _p(out), _s(stream)),
           "vg_sum_ordered")


def vg_encode_seq(coords, bits: int, mode: int, codes, stream=None) -> None:
    """codes[i] (int64 storage of uint64) = (b << 3*bits) | curve(x, y, z) of coords[i]."""
    _check(lib().vg_encode_seq(_p(coords), coords.shape[0], bits, mode, _p(codes), _s(stream)), "vg_encode_seq")


def vg_decode_seq(codes, bits: int, mode: int, coords, stream=None) -> None:
    """coords[i] = (b, x, y, z) of codes[i] (the inverse of vg_encode_seq)."""
    _check(lib().vg_decode_seq(_p(codes), codes.shape[0], bits, mode, _p(coords), _s(stream)), "vg_decode_seq")


def vg_conv_status(conv_ws, stream=None) -> int:
    return lib().vg_conv_status(_p(conv_ws), _s(stream))


# ---------------------------------------------------------------- buffer helpers
@dataclass
class NbrMap:
    """Caller-owned buffers of one neighbour map (allocated with torch)."""
    N: int
    grid: tuple
    flags: int
    ws: torch.Tensor     # uint8 workspace (the neighbour cache)
    nbr: torch.Tensor    # int32 [N,27] storage of uint32 entries
    mask: torch.Tensor   # int32 [N] storage of uint32 bitmasks

    @staticmethod
    def alloc(N, grid, flags=0, device="cuda") -> "NbrMap":
        B, X, Y, Z = grid
        nb = vg_nbrmap_workspace_bytes(N, B, X, Y, Z, flags)
        if nb == 0:
            raise VGError(VG_ERR_INVALID_ARG, "vg_nbrmap_workspace_bytes")
        ws = torch.empty(nb, dtype=torch.uint8, device=device)
        nbr = torch.empty(N, 27, dtype=torch.int32, device=device)
        mask = torch.empty(N, dtype=torch.int32, device=device)
        return NbrMap(N, tuple(grid), flags, ws, nbr, mask)

    def build(self, coords, stream=None) -> "NbrMap":
        vg_nbrmap_build(coords, *self.grid, self.flags, self.ws, self.nbr, self.mask, stream)
        return self

    def status(self, stream=None) -> int:
        return vg_nbrmap_status(self.ws, stream)

    def sorted_idx(self) -> torch.Tensor:
        return vg_nbrmap_sorted_idx(self.ws, self.N)

    def tile_mask(self) -> torch.Tensor:
        return vg_nbrmap_tile_mask(self.ws, self.N)

    def sorted_nbr(self) -> torch.Tensor:
        return vg_nbrmap_sorted_nbr(self.ws, self.N)


def conv_workspace(N, Cin, Cout, dtype, device="cuda", flags=0) -> torch.Tensor:
    nb = vg_conv_workspace_bytes(N, Cin, Cout, dtype, flags)
    if nb == 0:
        raise VGError(VG_ERR_UNSUPPORTED, "vg_conv_workspace_bytes")
    return torch.zeros(nb, dtype=torch.uint8, device=device)  # zero error record before any call


# ---------------------------------------------------------------- regular (strided / transposed) conv
class SparseMap:
    """A regular-convolution map (input sites -> strided output sites) in a torch-owned workspace."""

    def __init__(self, coords, grid, kernel: int, stride: int, flags: int = 0, stream=None):
        B, X, Y, Z = grid
        N = coords.shape[0]
        nb = int(lib().vg_sparse_map_workspace_bytes(N, B, X, Y, Z, kernel, stride, flags))
        if nb == 0:
            raise VGError(VG_ERR_INVALID_ARG, "vg_sparse_map_workspace_bytes")
        self.ws = torch.empty(nb, dtype=torch.uint8, device=coords.device)
        self.coords = coords
        self.m = SparseMapStruct()
        _check(lib().vg_sparse_map_build(_p(coords), N, B, X, Y, Z, kernel, stride, flags, _p(self.ws), nb,
                                         ctypes.byref(self.m), _s(stream)), "vg_sparse_map_build")

    @property
    def n_in(self) -> int:
        return self.m.n_in

    @property
    def n_out(self) -> int:
        return self.m.n_out

    @property
    def taps(self) -> int:
        return self.m.taps

    def _view(self, ptr, nbytes, dtype, shape):
        off = ptr - self.ws.data_ptr()
        return self.ws.view(torch.uint8)[off: off + nbytes].view(dtype).view(*shape)

    def coords_out(self) -> torch.Tensor:
        return self._view(self.m.coords_out, 16 * self.n_out, torch.int32, (self.n_out, 4))

    def down(self) -> torch.Tensor:
        return self._view(self.m.down, 4 * 27 * self.n_out, torch.int32, (self.n_out, 27))

    def up(self) -> torch.Tensor:
        return self._view(self.m.up, 4 * 27 * self.n_in, torch.int32, (self.n_in, 27))

    def workspace(self, transposed, Cin, Cout, dtype, flags=0) -> torch.Tensor:
        code = dtype if isinstance(dtype, int) else _DT[dtype]
        nb = int(lib().vg_sparse_conv_workspace_bytes(ctypes.byref(self.m), int(transposed), Cin, Cout, code, flags))
        if nb == 0:
            raise VGError(VG_ERR_UNSUPPORTED, "vg_sparse_conv_workspace_bytes")
        return torch.zeros(nb, dtype=torch.uint8, device=self.ws.device)

    def fwd(self, transposed, feats, weight, bias, out, conv_ws, flags=0, stream=None) -> None:
        Cin, Cout = weight.shape[1], weight.shape[2]
        _check(lib().vg_sparse_conv3d_fwd(ctypes.byref(self.m), int(transposed), _dtype_code(weight), _p(feats),
                                          _p(weight), _p(bias), _p(out), Cin, Cout, flags, _p(conv_ws),
                                          conv_ws.numel(), _s(stream)), "vg_sparse_conv3d_fwd")

    def bwd(self, transposed, grad_out, feats, weight, grad_feats, grad_weight, grad_bias, conv_ws, flags=0,
            stream=None) -> None:
        Cin, Cout = weight.shape[1], weight.shape[2]
        _check(lib().vg_sparse_conv3d_bwd(ctypes.byref(self.m), int(transposed), _dtype_code(weight), _p(grad_out),
                                          _p(feats), _p(weight), _p(grad_feats), _p(grad_weight), _p(grad_bias),
                                          Cin, Cout, flags, _p(conv_ws), conv_ws.numel(), _s(stream)),
               "vg_sparse_conv3d_bwd")

