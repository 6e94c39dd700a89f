"""Regular (strided and transposed) sparse convolution on the GPU vs the oracle.

The map (output sites in linear-key order, down and up tables) must equal the
oracle's bit for bit; the forward, input gradient, weight and bias gradient of
both directions must be within the dtype's relative Frobenius bound, on all four
(kernel, stride) cases and on ragged sizes, through the tensor-core, TF32 and
FFMA paths.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, f64, rel_fro, u32
from voxel_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu
TF32_TOL = 5e-3


def _pad27(W):
    out = np.zeros((27,) + tuple(W.shape[1:]))
    out[: W.shape[0]] = f64(W)
    return out


def _problem(K, s, n, grid, cin, cout, dtype, seed):
    coords = synth.random_coords(seed, n, *grid)
    rng = torch.Generator().manual_seed(seed)
    dt = synth.torch_dtype(dtype)
    T = K ** 3
    f_in = torch.randn(coords.shape[0], cin, generator=rng).to(dt)
    W = (torch.randn(T, cin, cout, generator=rng) * (2.0 / (T * cin)) ** 0.5).to(dt)
    b = (torch.randn(cout, generator=rng) * 0.1).to(dt)
    return coords, f_in, W, b


@pytest.mark.parametrize("K,s", [(2, 2), (3, 2), (3, 1), (2, 1)])
def test_sparse_map_bit_exact(K, s):
    grid = (2, 18, 11, 14)
    coords = synth.random_coords(K * 10 + s, 1500, *grid)
    co_ref, down_ref, up_ref = oracle.sparse_map(coords, *grid, K, s)
    m = ops.SparseMap(torch.from_numpy(coords).cuda(), grid, K, s)
    assert m.n_out == co_ref.shape[0] and m.taps == K ** 3
    assert np.array_equal(m.coords_out().cpu().numpy(), co_ref)
    assert np.array_equal(u32(m.down()), down_ref)
    assert np.array_equal(u32(m.up()), up_ref)


CASES = [(K, s, dt, c) for (K, s) in [(2, 2), (3, 2), (3, 1), (2, 1)] for dt, c in
         [("bf16", (64, 128)), ("f16", (128, 64)), ("f32", (24, 40))]]


@pytest.mark.parametrize("K,s,dtype,chan", CASES)
def test_strided_and_transposed_conv_match_oracle(K, s, dtype, chan):
    cin, cout = chan
    grid = (2, 16, 14, 12)
    coords, f_in, W, b = _problem(K, s, 1700, grid, cin, cout, dtype, K * 100 + s * 10 + cin)
    co, down, up = oracle.sparse_map(coords, *grid, K, s)
    m = ops.SparseMap(torch.from_numpy(coords).cuda(), grid, K, s)
    assert m.n_out == co.shape[0]
    tol = TOL[dtype]
    W27 = _pad27(W)
    dt = f_in.dtype
    Wd, bd = W.cuda(), b.cuda()
    # ---- strided: input sites -> output sites
    fi = f_in.cuda()
    dY = torch.randn(m.n_out, cout, generator=torch.Generator().manual_seed(1)).to(dt)
    ws = m.workspace(0, cin, cout, dt)
    out = torch.empty(m.n_out, cout, dtype=dt, device="cuda")
    m.fwd(0, fi, Wd, bd, out, ws)
    dX = torch.empty(m.n_in, cin, dtype=dt, device="cuda")
    dW = torch.empty_like(Wd)
    db = torch.empty_like(bd)
    m.bwd(0, dY.cuda(), fi, Wd, dX, dW, db, ws)
    torch.cuda.synchronize()
    assert ops.vg_conv_status(ws) == ops.VG_OK
    out_ref = oracle.fwd(down, f64(f_in), W27, f64(b))
    dX_ref = oracle.dgrad_scatter_to(down, f64(dY), W27, m.n_in)
    dW_ref, db_ref = oracle.wgrad(down, f64(f_in), f64(dY))
    errs = {"out": rel_fro(f64(out), out_ref), "dX": rel_fro(f64(dX), dX_ref),
            "dW": rel_fro(f64(dW), dW_ref[: K ** 3]), "db": rel_fro(f64(db), db_ref)}
    assert all(e <= tol for e in errs.values()), errs
    # ---- transposed: output sites -> input sites (the same map, the other way)
    g = torch.randn(m.n_out, cin, generator=torch.Generator().manual_seed(2)).to(dt)
    dYt = torch.randn(m.n_in, cout, generator=torch.Generator().manual_seed(3)).to(dt)
    wst = m.workspace(1, cin, cout, dt)
    outt = torch.empty(m.n_in, cout, dtype=dt, device="cuda")
    m.fwd(1, g.cuda(), Wd, bd, outt, wst)
    dG = torch.empty(m.n_out, cin, dtype=dt, device="cuda")
    m.bwd(1, dYt.cuda(), g.cuda(), Wd, dG, dW, db, wst)
    torch.cuda.synchronize()
    assert ops.vg_conv_status(wst) == ops.VG_OK
    out_ref = oracle.fwd(up, f64(g), W27, f64(b))
    dG_ref = oracle.dgrad_scatter_to(up, f64(dYt), W27, m.n_out)
    dW_ref, db_ref = oracle.wgrad(up, f64(g), f64(dYt))
    errs = {"out": rel_fro(f64(outt), out_ref), "dG": rel_fro(f64(dG), dG_ref),
            "dW": rel_fro(f64(dW), dW_ref[: K ** 3]), "db": rel_fro(f64(db), db_ref)}
    assert all(e <= tol for e in errs.values()), errs


@pytest.mark.parametrize("K,s", [(2, 2), (3, 2)])
def test_sparse_conv_tf32(K, s):
    grid = (1, 20, 20, 20)
    coords, f_in, W, b = _problem(K, s, 2500, grid, 64, 32, "f32", 77 + K)
    co, down, up = oracle.sparse_map(coords, *grid, K, s)
    m = ops.SparseMap(torch.from_numpy(coords).cuda(), grid, K, s)
    fl = ops.VG_ALLOW_TF32
    ws = m.workspace(0, 64, 32, torch.float32, fl)
    out = torch.empty(m.n_out, 32, device="cuda")
    m.fwd(0, f_in.cuda(), W.cuda(), b.cuda(), out, ws, flags=fl)
    dY = torch.randn(m.n_out, 32)
    dX = torch.empty(m.n_in, 64, device="cuda")
    dW = torch.empty_like(W).cuda()
    db = torch.empty(32, device="cuda")
    m.bwd(0, dY.cuda(), f_in.cuda(), W.cuda(), dX, dW, db, ws, flags=fl)
    torch.cuda.synchronize()
    assert ops.vg_conv_status(ws) == ops.VG_OK
    W27 = _pad27(W)
    assert rel_fro(f64(out), oracle.fwd(down, f64(f_in), W27, f64(b))) <= TF32_TOL
    assert rel_fro(f64(dX), oracle.dgrad_scatter_to(down, f64(dY), W27, m.n_in)) <= TF32_TOL
    dW_ref, db_ref = oracle.wgrad(down, f64(f_in), f64(dY))
    assert rel_fro(f64(dW), dW_ref[: K ** 3]) <= TF32_TOL and rel_fro(f64(db), db_ref) <= TF32_TOL


def test_sparse_map_rejects_bad_sites_and_arguments():
    grid = (1, 8, 8, 8)
    c = torch.tensor([[0, 1, 1, 1], [0, 1, 1, 1]], dtype=torch.int32, device="cuda")
    with pytest.raises(ops.VGError) as e:
        ops.SparseMap(c, grid, 3, 2)
    assert e.value.status == ops.VG_ERR_DUPLICATE_COORD
    c = torch.tensor([[0, 8, 1, 1]], dtype=torch.int32, device="cuda")
    with pytest.raises(ops.VGError) as e:
        ops.SparseMap(c, grid, 2, 2)
    assert e.value.status == ops.VG_ERR_COORD_OUT_OF_RANGE
    assert ops.lib().vg_sparse_map_workspace_bytes(10, 1, 8, 8, 8, 4, 2, 0) == 0
    assert ops.lib().vg_sparse_map_workspace_bytes(10, 1, 8, 8, 8, 3, 3, 0) == 0


def test_sparse_map_empty_input():
    m = ops.SparseMap(torch.zeros(0, 4, dtype=torch.int32, device="cuda"), (1, 8, 8, 8), 3, 2)
    assert m.n_out == 0
    W = torch.randn(27, 64, 64, device="cuda").bfloat16()
    ws = m.workspace(0, 64, 64, torch.bfloat16)
    dW = torch.full_like(W, 3.0)
    db = torch.full((64,), 3.0, dtype=torch.bfloat16, device="cuda")
    m.bwd(0, torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda"), torch.zeros(0, 64, dtype=torch.bfloat16,
          device="cuda"), W, None, dW, db, ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dW) == 0 and torch.count_nonzero(db) == 0


def test_sparse_map_large_grid_and_hilbert_order():
    # a grid of more than 2^31 cells (64-bit hash and candidate keys) with the Hilbert
    # row order: the map stays bit-exact and a bf16 strided pass stays within bound
    grid = (3, 1100, 1000, 900)
    coords = synth.random_coords(91, 3000, *grid)
    # cluster half of the voxels so that windows hold several inputs
    coords[:1500, 1:] = (coords[:1500, 1:] % 16) + 500
    coords = np.unique(coords, axis=0)
    coords = coords[np.random.default_rng(1).permutation(len(coords))].astype(np.int32)
    co, down, up = oracle.sparse_map(coords, *grid, 3, 2)
    m = ops.SparseMap(torch.from_numpy(coords).cuda(), grid, 3, 2, flags=ops.VG_ORDER_HILBERT)
    assert m.n_out == co.shape[0]
    assert np.array_equal(m.coords_out().cpu().numpy(), co)
    assert np.array_equal(u32(m.down()), down) and np.array_equal(u32(m.up()), up)
    g = torch.Generator().manual_seed(4)
    f = torch.randn(coords.shape[0], 64, generator=g).bfloat16()
    W = (torch.randn(27, 64, 64, generator=g) * 0.03).bfloat16()
    ws = m.workspace(0, 64, 64, torch.bfloat16)
    out = torch.empty(m.n_out, 64, dtype=torch.bfloat16, device="cuda")
    m.fwd(0, f.cuda(), W.cuda(), None, out, ws)
    torch.cuda.synchronize()
    ref = oracle.fwd(down, f64(f), _pad27(W), None)
    assert rel_fro(f64(out), ref) <= TOL["bf16"]


def test_sparse_conv_16bit_cuda_core_channels_and_graph_capture():
    # 16-bit channels that are not multiples of 64 take the CUDA-core kernels; the
    # strided forward and backward replay from a CUDA graph with the same bits
    grid = (1, 20, 20, 20)
    coords, f_in, W, b = _problem(3, 2, 1500, grid, 40, 24, "f16", 5)
    co, down, up = oracle.sparse_map(coords, *grid, 3, 2)
    m = ops.SparseMap(torch.from_numpy(coords).cuda(), grid, 3, 2)
    dt = torch.float16
    fi, Wd, bd = f_in.cuda(), W.cuda(), b.cuda()
    dY = torch.randn(m.n_out, 24, generator=torch.Generator().manual_seed(6)).half().cuda()
    ws = m.workspace(0, 40, 24, dt)
    out = torch.empty(m.n_out, 24, dtype=dt, device="cuda")
    dX = torch.empty(m.n_in, 40, dtype=dt, device="cuda")
    dW = torch.empty_like(Wd)
    db = torch.empty_like(bd)
    s = torch.cuda.Stream()

    def step():
        m.fwd(0, fi, Wd, bd, out, ws, stream=s)
        m.bwd(0, dY, fi, Wd, dX, dW, db, ws, stream=s)

    with torch.cuda.stream(s):
        step()
    s.synchronize()
    eager = [t.clone() for t in (out, dX, dW, db)]
    W27 = _pad27(W)
    assert rel_fro(f64(out), oracle.fwd(down, f64(f_in), W27, f64(b))) <= TOL["f16"]
    assert rel_fro(f64(dX), oracle.dgrad_scatter_to(down, f64(dY), W27, m.n_in)) <= TOL["f16"]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for t in (out, dX, dW, db):
        t.zero_()
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    for a_, b_ in zip(eager, (out, dX, dW, db)):
        assert torch.equal(a_, b_)


@pytest.mark.parametrize("cin,cout", [(64, 256), (256, 64)])
def test_regular_conv_tile_pairs_match_oracle(cin, cout):
    """Enough output (or input) sites that the 256-column gather passes run on the
    tile-pair kernel (at least two 128-row tiles per SM): the forward at Cout = 256 and
    the input gradient at Cin = 256, strided and transposed, every element against the
    oracle (bf16)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grid = (1, 96, 96, 96)
    coords, f_in, W, b = _problem(2, 2, 80000, grid, cin, cout, "bf16", 77 + cin)
    co, down, up = oracle.sparse_map(coords, *grid, 2, 2)
    m = ops.SparseMap(torch.from_numpy(coords).cuda(), grid, 2, 2)
    assert m.n_out == co.shape[0] and min(m.n_in, m.n_out) >= 2 * sms * 128
    dt, tol = f_in.dtype, TOL["bf16"]
    W27, Wd, bd = _pad27(W), W.cuda(), b.cuda()
    for transposed, nbr, n_src, n_dst in ((0, down, m.n_in, m.n_out), (1, up, m.n_out, m.n_in)):
        x = torch.randn(n_src, cin, generator=torch.Generator().manual_seed(5 + transposed)).to(dt)
        dY = torch.randn(n_dst, cout, generator=torch.Generator().manual_seed(7 + transposed)).to(dt)
        ws = m.workspace(transposed, cin, cout, dt)
        out = torch.empty(n_dst, cout, dtype=dt, device="cuda")
        dX = torch.empty(n_src, cin, dtype=dt, device="cuda")
        dW, db = torch.empty_like(Wd), torch.empty_like(bd)
        m.fwd(transposed, x.cuda(), Wd, bd, out, ws)
        m.bwd(transposed, dY.cuda(), x.cuda(), Wd, dX, dW, db, ws)
        torch.cuda.synchronize()
        assert ops.vg_conv_status(ws) == ops.VG_OK
        out_ref = oracle.fwd(nbr, f64(x), W27, f64(b))
        dX_ref = oracle.dgrad_scatter_to(nbr, f64(dY), W27, n_src)
        dW_ref, db_ref = oracle.wgrad(nbr, f64(x), f64(dY))
        errs = {"out": rel_fro(f64(out), out_ref), "dX": rel_fro(f64(dX), dX_ref),
                "dW": rel_fro(f64(dW), dW_ref[:8]), "db": rel_fro(f64(db), db_ref)}
        assert all(e <= tol for e in errs.values()), (transposed, errs)
