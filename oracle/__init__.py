"""CPU oracle for submanifold sparse 3D convolution — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never loads it and it
never loads the GPU library: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, fp64, a sorted-array
dictionary for the neighbour lookup, loops over voxels x taps x channels).
This module compiles it with gcc and wraps it with ctypes (argument
marshalling only).  Every function's header comment in ``oracle.c`` states
the definition it follows and the page section that defines the operator:
"Contribution Tasks — JeffreyXiang/FlexGEMM" §一/§二 for the operator and the
neighbour-map/neighbour-cache structure, and "From CUDA to Triton: Triton JIT
and autotuning" §六 6.2 for the kernel arguments (V = 27 taps, uint32
neighbour table, contraction over V * Ci).

Parity status of each function (what pins it, in ``tests/test_oracle_pins.py``):
  nbrmap        brute-force O(N^2) search, tap symmetry, centre tap, popcounts
  fwd           dense torch conv3d on the densified grid, 1x1x1 = matmul,
                all-ones closed form, permutation equivariance
  dgrad_scatter dense conv3d autograd, adjoint identity
  dgrad_rows    equal to dgrad_scatter (it is a regrouping of the same sum)
  wgrad         dense conv3d autograd (dW and db), central finite differences
  sparse_map    (regular strided / transposed convolution) dense torch conv3d and
                conv_transpose3d on the densified grid (outputs, output set,
                autograd), adjoint identity
  dgrad_scatter_to  dense conv3d autograd (the strided convolution's input gradient)
  curve_encode / curve_decode (z-order, Hilbert)
                bijection onto [0, 8^bits) by exhaustion on small cubes, decode is
                the inverse of encode, z-order's parent/child nesting, Hilbert's
                unit steps between consecutive codes
No function is left unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

NONE = 0xFFFFFFFF
OK, BAD_ARG, OUT_OF_RANGE, DUPLICATE, NO_MEMORY = range(5)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, OpenMP). Returns the path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.oracle_nbrmap.argtypes = [P, I64, I, I, I, I, P, P]
        lib.oracle_nbrmap.restype = I
        lib.oracle_fwd.argtypes = [P, I64, P, I64, P, P, I, I, P]
        lib.oracle_fwd.restype = None
        lib.oracle_dgrad_scatter.argtypes = [P, I64, P, P, I, I, P]
        lib.oracle_dgrad_scatter.restype = None
        lib.oracle_dgrad_rows.argtypes = [P, I64, P, I64, P, I, I, P]
        lib.oracle_dgrad_rows.restype = None
        lib.oracle_wgrad.argtypes = [P, I64, P, I64, P, I, I, P, P]
        lib.oracle_wgrad.restype = None
        lib.oracle_dgrad_scatter_to.argtypes = [P, I64, P, P, I, I, I64, P]
        lib.oracle_dgrad_scatter_to.restype = None
        lib.oracle_sparse_map.argtypes = [P, I64, I, I, I, I, I, I, P, P, P, P]
        lib.oracle_sparse_map.restype = I
        lib.oracle_curve_encode.argtypes = [P, I64, I, I, P]
        lib.oracle_curve_encode.restype = I
        lib.oracle_curve_decode.argtypes = [P, I64, I, I, P]
        lib.oracle_curve_decode.restype = I
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = I
        lib.oracle_set_num_threads.argtypes = [I]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


class OracleError(RuntimeError):
    def __init__(self, code: int):
        names = {BAD_ARG: "bad argument", OUT_OF_RANGE: "coordinate out of range",
                 DUPLICATE: "duplicate coordinate", NO_MEMORY: "out of memory"}
        super().__init__(names.get(code, f"oracle error {code}"))
        self.code = code


def nbrmap(coords, B: int, X: int, Y: int, Z: int):
    """Neighbour map of int32 (b,x,y,z) rows: returns (nbr uint32 [N,27], mask uint32 [N])."""
    c = np.ascontiguousarray(np.asarray(coords, dtype=np.int32).reshape(-1, 4))
    n = c.shape[0]
    nbr = np.empty((n, 27), dtype=np.uint32)
    mask = np.empty((n,), dtype=np.uint32)
    rc = _load().oracle_nbrmap(_ptr(c), n, B, X, Y, Z, _ptr(nbr), _ptr(mask))
    if rc != OK:
        raise OracleError(rc)
    return nbr, mask


def fwd(nbr, f, W, bias=None):
    """out [R,Cout] (fp64) for the R rows whose neighbour lists are nbr [R,27] (indices into f)."""
    nbr = np.ascontiguousarray(nbr, dtype=np.uint32)
    f = _f64(f)
    W = _f64(W)
    _, cin, cout = W.shape
    assert W.shape[0] == 27 and f.shape[1] == cin
    b = None if bias is None else _f64(bias)
    out = np.empty((nbr.shape[0], cout), dtype=np.float64)
    _load().oracle_fwd(_ptr(nbr), nbr.shape[0], _ptr(f), f.shape[0], _ptr(W),
                       None if b is None else _ptr(b), cin, cout, _ptr(out))
    return out


def dgrad_scatter(nbr, dY, W):
    """dX [N,Cin] (fp64) by scattering every valid pair; nbr is the full [N,27] map."""
    nbr = np.ascontiguousarray(nbr, dtype=np.uint32)
    dY = _f64(dY)
    W = _f64(W)
    _, cin, cout = W.shape
    dX = np.empty((nbr.shape[0], cin), dtype=np.float64)
    _load().oracle_dgrad_scatter(_ptr(nbr), nbr.shape[0], _ptr(dY), _ptr(W), cin, cout, _ptr(dX))
    return dX


def dgrad_rows(nbr, dY, W):
    """dX rows [R,Cin] (fp64) for the R rows whose neighbour lists are nbr [R,27] (indices into dY)."""
    nbr = np.ascontiguousarray(nbr, dtype=np.uint32)
    dY = _f64(dY)
    W = _f64(W)
    _, cin, cout = W.shape
    dX = np.empty((nbr.shape[0], cin), dtype=np.float64)
    _load().oracle_dgrad_rows(_ptr(nbr), nbr.shape[0], _ptr(dY), dY.shape[0], _ptr(W),
                              cin, cout, _ptr(dX))
    return dX


def wgrad(nbr, f, dY, with_bias: bool = True):
    """(dW [27,Cin,Cout], db [Cout] or None), fp64; nbr is the full [N,27] map."""
    nbr = np.ascontiguousarray(nbr, dtype=np.uint32)
    f = _f64(f)
    dY = _f64(dY)
    cin, cout = f.shape[1], dY.shape[1]
    dW = np.empty((27, cin, cout), dtype=np.float64)
    db = np.empty((cout,), dtype=np.float64) if with_bias else None
    _load().oracle_wgrad(_ptr(nbr), nbr.shape[0], _ptr(f), f.shape[0], _ptr(dY), cin, cout,
                         _ptr(dW), None if db is None else _ptr(db))
    return dW, db


ZORDER, HILBERT = 0, 1


def curve_encode(coords, bits: int, curve: int):
    """uint64 codes (b << 3*bits) | curve(x, y, z) of int32 (b,x,y,z) rows; curve ZORDER or HILBERT."""
    c = np.ascontiguousarray(np.asarray(coords, dtype=np.int32).reshape(-1, 4))
    out = np.empty(c.shape[0], dtype=np.uint64)
    rc = _load().oracle_curve_encode(_ptr(c), c.shape[0], bits, curve, _ptr(out))
    if rc != OK:
        raise OracleError(rc)
    return out


def curve_decode(codes, bits: int, curve: int):
    """int32 (b,x,y,z) rows of uint64 curve codes (the inverse of curve_encode)."""
    k = np.ascontiguousarray(np.asarray(codes, dtype=np.uint64).reshape(-1))
    out = np.empty((k.shape[0], 4), dtype=np.int32)
    rc = _load().oracle_curve_decode(_ptr(k), k.shape[0], bits, curve, _ptr(out))
    if rc != OK:
        raise OracleError(rc)
    return out


def dgrad_scatter_to(nbr, dY, W, n_x: int):
    """dX [n_x, Cin] (fp64): every valid pair (i, k) of nbr [R,27] adds W_k dY[i] to dX[nbr[i][k]]."""
    nbr = np.ascontiguousarray(nbr, dtype=np.uint32)
    dY = _f64(dY)
    W = _f64(W)
    _, cin, cout = W.shape
    dX = np.empty((n_x, cin), dtype=np.float64)
    _load().oracle_dgrad_scatter_to(_ptr(nbr), nbr.shape[0], _ptr(dY), _ptr(W), cin, cout, n_x, _ptr(dX))
    return dX


def sparse_map(coords, B: int, X: int, Y: int, Z: int, kernel: int, stride: int):
    """Regular sparse convolution map: (coords_out int32 [No,4] in ascending linear key,
    down uint32 [No,27] -> input rows, up uint32 [N,27] -> output rows).  Kernel 2 or 3
    (padding 0 or 1), stride 1 or 2; taps k >= kernel^3 are absent."""
    c = np.ascontiguousarray(np.asarray(coords, dtype=np.int32).reshape(-1, 4))
    n = c.shape[0]
    T = kernel ** 3
    cap = max(1, n * T)
    out = np.empty((cap, 4), dtype=np.int32)
    down = np.empty((cap, 27), dtype=np.uint32)
    up = np.empty((max(1, n), 27), dtype=np.uint32)
    no = ctypes.c_int64(0)
    rc = _load().oracle_sparse_map(_ptr(c), n, B, X, Y, Z, kernel, stride, ctypes.byref(no), _ptr(out),
                                   _ptr(down), _ptr(up))
    if rc != OK:
        raise OracleError(rc)
    k = no.value
    return out[:k].copy(), down[:k].copy(), up[:n].copy()

