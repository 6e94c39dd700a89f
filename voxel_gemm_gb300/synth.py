"""Seeded synthetic voxel workloads (inputs only; none of the convolution's arithmetic).

Both the GPU library's tests/benchmark and the CPU oracle's tests draw their
inputs from here, so this module must stay free of anything the method
computes: it only voxelises analytic surfaces and draws random numbers.

Workloads stand in for the pages' training benchmark ("Contribution Tasks —
JeffreyXiang/FlexGEMM" §一: voxel data with C = 64..1024 channels and grid
resolutions 8..1024 on an A100; the real data is not available here).  The
pages name the project's test-data generator ``sphere_coords`` (same page,
§三, pitfalls list, item 6), a voxelised sphere; spheres and tori are
voxelised the same way here:

* a voxel (integer cell, centre at +0.5) is on a surface when the signed
  distance d from its centre to the surface satisfies |d| <= 0.5;
* sphere: d = |p - c| - r;  torus with its axis along z:
  d = sqrt((sqrt(px^2 + py^2) - R)^2 + pz^2) - r;
* shapes are clipped to the grid, the union over shapes is deduplicated, and
  rows are emitted in a seeded random permutation.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Tuple

import numpy as np

NO_KEY_FORCE, KEY32, KEY64 = 0, 1, 2


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int                 # batch elements
    res: int               # grid is res^3 per batch element
    shapes_per_sample: int
    kinds: Tuple[str, ...]  # ("sphere",) or ("sphere", "torus")
    cin: int
    cout: int
    dtype: str             # "f32" | "f16" | "bf16"
    seed: int
    w_var_num: float       # weight variance = w_var_num / (27 * cin)
    fixed_sphere: Tuple[float, float, float, float] | None = None  # (cx, cy, cz, r)
    key_flag: int = NO_KEY_FORCE

    @property
    def grid(self) -> Tuple[int, int, int, int]:
        return (self.B, self.res, self.res, self.res)


def _mk(name, B, res, n, kinds, c, dtype, seed, w_var_num=2.0, fixed=None, key_flag=NO_KEY_FORCE):
    return Workload(name, B, res, n, kinds, c, c, dtype, seed, w_var_num, fixed, key_flag)


# The five seeded workloads (seed = position in this list).
WORKLOADS: Dict[str, Workload] = {w.name: w for w in [
    # one sphere, centre (8,8,8), radius 5, in a 16^3 grid; fp32; W ~ N(0, 1/(27 Cin))
    _mk("sphere16_c32_f32", 1, 16, 1, ("sphere",), 32, "f32", 0, w_var_num=1.0,
        fixed=(8.0, 8.0, 8.0, 5.0)),
    # batch 4, 64^3, 3 random spheres per sample, r ~ U[0.1, 0.35] * 64; fp16; He init
    _mk("b4_r64_spheres_c64_f16", 4, 64, 3, ("sphere",), 64, "f16", 1),
    # batch 2, 256^3, 6 random spheres/tori per sample; bf16
    _mk("b2_r256_shapes_c128_bf16", 2, 256, 6, ("sphere", "torus"), 128, "bf16", 2),
    # batch 1, 512^3, 6 random spheres/tori; channel sweep; bf16
    _mk("b1_r512_shapes_c256_bf16", 1, 512, 6, ("sphere", "torus"), 256, "bf16", 3),
    _mk("b1_r512_shapes_c512_bf16", 1, 512, 6, ("sphere", "torus"), 512, "bf16", 3),
    _mk("b1_r512_shapes_c1024_bf16", 1, 512, 6, ("sphere", "torus"), 1024, "bf16", 3),
    # batch 1, 1024^3, 8 random spheres/tori, 64-bit hash keys; fp16
    _mk("b1_r1024_shapes_c64_f16", 1, 1024, 8, ("sphere", "torus"), 64, "f16", 4,
        key_flag=KEY64),
    # a smaller case of the 512^3 C = 1024 kernels (256^3 grid, same generator), for
    # counter captures that must stay a few GB on the device; its DRAM bytes per valid
    # pair scale to the large case
    _mk("b1_r256_shapes_c1024_bf16", 1, 256, 6, ("sphere", "torus"), 1024, "bf16", 3),
    # small inference case (forward only, few voxels): batch 1, 64^3, 2 random spheres,
    # C = 256 bf16 -- fewer (tile, channel block) units than SMs
    _mk("b1_r64_spheres_c256_bf16_infer", 1, 64, 2, ("sphere",), 256, "bf16", 5),
]}


def _shape_params(wl: Workload, rng: np.random.Generator) -> List[Tuple[int, str, Tuple[float, ...], Tuple[float, ...]]]:
    """(batch, kind, centre, radii) for every shape of the workload, in draw order."""
    out = []
    if wl.fixed_sphere is not None:
        cx, cy, cz, r = wl.fixed_sphere
        for b in range(wl.B):
            out.append((b, "sphere", (cx, cy, cz), (r,)))
        return out
    R = float(wl.res)
    for b in range(wl.B):
        for _ in range(wl.shapes_per_sample):
            kind = "sphere"
            if len(wl.kinds) > 1:
                kind = "torus" if rng.random() < 0.5 else "sphere"
            centre = tuple(float(v) for v in rng.uniform(0.0, R, size=3))
            if kind == "sphere":
                radii = (float(rng.uniform(0.10, 0.35)) * R,)
            else:
                radii = (float(rng.uniform(0.15, 0.35)) * R, float(rng.uniform(0.03, 0.08)) * R)
            out.append((b, kind, centre, radii))
    return out


def _expand(lo: np.ndarray, hi: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """For integer intervals [lo, hi] (inclusive) return (interval id, value) of every member."""
    n = np.maximum(hi - lo + 1, 0)
    total = int(n.sum())
    ids = np.repeat(np.arange(lo.size), n)
    starts = np.repeat(np.cumsum(n) - n, n)
    vals = np.repeat(lo, n) + (np.arange(total) - starts)
    return ids, vals


def surface_distance(kind: str, centre, radii, x, y, z) -> np.ndarray:
    """Signed distance from voxel centres (x+.5, y+.5, z+.5) to the surface."""
    px = np.asarray(x, dtype=np.float64) + 0.5 - centre[0]
    py = np.asarray(y, dtype=np.float64) + 0.5 - centre[1]
    pz = np.asarray(z, dtype=np.float64) + 0.5 - centre[2]
    if kind == "sphere":
        return np.sqrt(px * px + py * py + pz * pz) - radii[0]
    R, r = radii
    return np.sqrt((np.sqrt(px * px + py * py) - R) ** 2 + pz * pz) - r


def shell_voxels(kind: str, centre, radii, res: int) -> np.ndarray:
    """int64 [n,3] (x,y,z) of the voxels with |d| <= 0.5 inside [0,res)^3."""
    cx, cy, cz = centre
    if kind == "sphere":
        r = radii[0]
        reach = r + 1.0
    else:
        R, r = radii
        reach = R + r + 1.0
    x0, x1 = max(0, math.floor(cx - reach) - 1), min(res, math.ceil(cx + reach) + 1)
    y0, y1 = max(0, math.floor(cy - reach) - 1), min(res, math.ceil(cy + reach) + 1)
    if x0 >= x1 or y0 >= y1:
        return np.zeros((0, 3), dtype=np.int64)
    xs, ys = np.meshgrid(np.arange(x0, x1), np.arange(y0, y1), indexing="ij")
    xs, ys = xs.ravel(), ys.ravel()
    px = xs + 0.5 - cx
    py = ys + 0.5 - cy
    q = px * px + py * py
    e = q if kind == "sphere" else (np.sqrt(q) - radii[0]) ** 2
    lo_r, hi_r = max(0.0, r - 0.5), r + 0.5
    top = hi_r * hi_r - e
    keep = top >= 0.0
    xs, ys, e, top = xs[keep], ys[keep], e[keep], top[keep]
    sb = np.sqrt(top)
    sa = np.sqrt(np.maximum(lo_r * lo_r - e, 0.0))
    # |pz| in [sa, sb], pz = z + 0.5 - cz; candidate z ranges widened by one cell,
    # then every candidate is tested exactly below.
    up_lo = np.ceil(cz - 0.5 + sa).astype(np.int64) - 1
    up_hi = np.floor(cz - 0.5 + sb).astype(np.int64) + 1
    dn_lo = np.ceil(cz - 0.5 - sb).astype(np.int64) - 1
    dn_hi = np.floor(cz - 0.5 - sa).astype(np.int64) + 1
    lo = np.maximum(np.concatenate([up_lo, dn_lo]), 0)
    hi = np.minimum(np.concatenate([up_hi, dn_hi]), res - 1)
    ids, zs = _expand(lo, hi)
    cx_ = np.concatenate([xs, xs])[ids]
    cy_ = np.concatenate([ys, ys])[ids]
    d = surface_distance(kind, centre, radii, cx_, cy_, zs)
    ok = np.abs(d) <= 0.5
    return np.stack([cx_[ok], cy_[ok], zs[ok]], axis=1).astype(np.int64)


def _sorted_unique(a: np.ndarray) -> np.ndarray:
    """Sorted distinct values of a 1-D array (np.unique's result, by sort + compare)."""
    a = np.sort(a)
    if a.size == 0:
        return a
    keep = np.empty(a.size, dtype=bool)
    keep[0] = True
    np.not_equal(a[1:], a[:-1], out=keep[1:])
    return a[keep]


def make_coords(wl: Workload) -> np.ndarray:
    """int32 [N,4] (b,x,y,z), deduplicated, rows in a seeded random permutation."""
    rng = np.random.default_rng(wl.seed)
    res = wl.res
    keys = []
    for b, kind, centre, radii in _shape_params(wl, rng):
        v = shell_voxels(kind, centre, radii, res)
        keys.append(((b * res + v[:, 0]) * res + v[:, 1]) * res + v[:, 2])
    allk = _sorted_unique(np.concatenate(keys)) if keys else np.zeros(0, np.int64)
    perm = rng.permutation(allk.size)
    allk = allk[perm]
    out = np.empty((allk.size, 4), dtype=np.int32)
    out[:, 3] = allk % res
    t = allk // res
    out[:, 2] = t % res
    t //= res
    out[:, 1] = t % res
    out[:, 0] = t // res
    return out


TORCH_DTYPES = {"f32": "float32", "f16": "float16", "bf16": "bfloat16"}


def torch_dtype(name: str):
    import torch
    return getattr(torch, TORCH_DTYPES[name])


def make_tensors(wl: Workload, n: int, device="cpu", dtype: str | None = None):
    """Seeded (feats [N,Cin], weight [27,Cin,Cout], bias [Cout], grad_out [N,Cout]).

    feats and grad_out ~ N(0,1); weight ~ N(0, w_var_num / (27 Cin)) (He init
    for w_var_num = 2); bias ~ N(0, 0.1^2).  Drawn in fp32 with torch's
    generator on ``device`` and rounded to the workload's dtype.
    """
    import torch
    dt = torch_dtype(dtype or wl.dtype)
    g = torch.Generator(device=device)
    g.manual_seed(1_000_003 * (wl.seed + 1) + wl.cin * 7 + wl.cout)
    f = torch.randn(n, wl.cin, generator=g, device=device, dtype=torch.float32).to(dt)
    wstd = math.sqrt(wl.w_var_num / (27.0 * wl.cin))
    W = (torch.randn(27, wl.cin, wl.cout, generator=g, device=device, dtype=torch.float32)
         * wstd).to(dt)
    bias = (torch.randn(wl.cout, generator=g, device=device, dtype=torch.float32) * 0.1).to(dt)
    dy = torch.randn(n, wl.cout, generator=g, device=device, dtype=torch.float32).to(dt)
    return f, W, bias, dy


def random_coords(seed: int, n: int, B: int, X: int, Y: int, Z: int) -> np.ndarray:
    """n distinct uniformly random (b,x,y,z) int32 rows (for small edge-case tests)."""
    rng = np.random.default_rng(seed)
    vol = B * X * Y * Z
    n = min(n, vol)
    keys = rng.choice(vol, size=n, replace=False)
    z = keys % Z
    t = keys // Z
    y = t % Y
    t //= Y
    x = t % X
    b = t // X
    return np.stack([b, x, y, z], axis=1).astype(np.int32)
