"""Shared test helpers: cached workloads, oracle sub-problems, error metrics."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from voxel_gemm_gb300 import synth

NONE = oracle.NONE
TOL = {"f32": 1e-5, "f16": 1e-2, "bf16": 1e-2}


def rel_fro(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


@functools.lru_cache(maxsize=None)
def coords_of(name: str) -> np.ndarray:
    return synth.make_coords(synth.WORKLOADS[name])


@functools.lru_cache(maxsize=None)
def oracle_map(name: str):
    wl = synth.WORKLOADS[name]
    return oracle.nbrmap(coords_of(name), *wl.grid)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def u32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint32)


def compact(nbr_rows: np.ndarray):
    """Remap the neighbour lists of a row subset onto the distinct rows they use."""
    valid = nbr_rows != NONE
    used = np.unique(nbr_rows[valid]).astype(np.int64)
    remap = np.full(nbr_rows.shape, NONE, dtype=np.uint32)
    remap[valid] = np.searchsorted(used, nbr_rows[valid].astype(np.int64)).astype(np.uint32)
    return remap, used


def oracle_fwd_rows(nbr, rows, cols, f, W, bias):
    """Oracle forward restricted to output rows x output columns (exact restriction)."""
    sub, used = compact(nbr[rows])
    fb = f64(f[torch.from_numpy(used)]) if used.size else np.zeros((0, f.shape[1]))
    Wc = f64(W[:, :, torch.from_numpy(cols)])
    bc = None if bias is None else f64(bias[torch.from_numpy(cols)])
    return oracle.fwd(sub, fb, Wc, bc)


def oracle_dgrad_rows(nbr, rows, cols, dY, W):
    """Oracle input gradient for rows x input-channel columns (gathered form)."""
    sub, used = compact(nbr[rows])
    gb = f64(dY[torch.from_numpy(used)]) if used.size else np.zeros((0, dY.shape[1]))
    Wc = f64(W[:, torch.from_numpy(cols), :])
    return oracle.dgrad_rows(sub, gb, Wc)


def oracle_wgrad_cols(nbr, f, dY, ci_cols, co_cols):
    """Oracle dW[:, ci_cols, co_cols] and db[co_cols] (each entry a full sum over all rows)."""
    fc = f64(f[:, torch.from_numpy(ci_cols)])
    gc = f64(dY[:, torch.from_numpy(co_cols)])
    return oracle.wgrad(nbr, fc, gc)
