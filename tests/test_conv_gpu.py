"""GPU forward / input gradient / weight and bias gradient vs the oracle.

Small workloads are compared element by element in full; the large ones on
seeded samples the oracle computes one by one (4096 output rows x up to 64
columns for fwd and dgrad, 27 x 16 x 16 full-sum dW entries, all of db), in the
same launch configuration the benchmark times.  Bound: relative Frobenius
error <= 1e-5 (fp32, FFMA) and <= 1e-2 (fp16/bf16 with fp32 accumulation).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import (TOL, coords_of, f64, oracle_dgrad_rows, oracle_fwd_rows, oracle_map,
                     oracle_wgrad_cols, rel_fro, u32)
from voxel_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def run_gpu(coords_np, grid, f, W, b, dY, key_flag=0, flags=0):
    dev = "cuda"
    c = torch.from_numpy(coords_np).to(dev)
    N = coords_np.shape[0]
    m = ops.NbrMap.alloc(N, grid, key_flag).build(c)
    fd, Wd, dYd = f.to(dev), W.to(dev), dY.to(dev)
    bd = None if b is None else b.to(dev)
    Cin, Cout = W.shape[1], W.shape[2]
    ws = ops.conv_workspace(N, Cin, Cout, f.dtype, flags=flags)
    res = {}
    out = torch.empty(N, Cout, dtype=f.dtype, device=dev)
    ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, fd, Wd, bd, out, ws, flags=flags)
    dX = torch.empty(N, Cin, dtype=f.dtype, device=dev)
    dW = torch.empty(27, Cin, Cout, dtype=f.dtype, device=dev)
    db = torch.empty(Cout, dtype=f.dtype, device=dev)
    ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dYd, fd, Wd, dX, dW, db, ws, flags=flags)
    assert m.status() == ops.VG_OK
    assert ops.vg_conv_status(ws) == ops.VG_OK
    res.update(out=out.cpu(), dX=dX.cpu(), dW=dW.cpu(), db=db.cpu(), nbr=u32(m.nbr))
    return res


def full_check(coords, grid, f, W, b, dY, tol, key_flag=0, flags=0):
    nbr_ref, _ = oracle.nbrmap(coords, *grid)
    r = run_gpu(coords, grid, f, W, b, dY, key_flag, flags)
    assert np.array_equal(r["nbr"], nbr_ref)
    out_ref = oracle.fwd(nbr_ref, f64(f), f64(W), None if b is None else f64(b))
    dX_ref = oracle.dgrad_scatter(nbr_ref, f64(dY), f64(W))
    dW_ref, db_ref = oracle.wgrad(nbr_ref, f64(f), f64(dY))
    errs = {"out": rel_fro(f64(r["out"]), out_ref), "dX": rel_fro(f64(r["dX"]), dX_ref),
            "dW": rel_fro(f64(r["dW"]), dW_ref), "db": rel_fro(f64(r["db"]), db_ref)}
    for k, e in errs.items():
        assert e <= tol, (k, e, errs)
    return errs


@pytest.mark.parametrize("name", ["sphere16_c32_f32", "b4_r64_spheres_c64_f16"])
def test_workload_full(name):
    wl = synth.WORKLOADS[name]
    coords = coords_of(name)
    f, W, b, dY = synth.make_tensors(wl, coords.shape[0])
    full_check(coords, wl.grid, f, W, b, dY, TOL[wl.dtype], wl.key_flag)


SAMPLED = ["b2_r256_shapes_c128_bf16", "b1_r512_shapes_c256_bf16", "b1_r512_shapes_c512_bf16",
           "b1_r512_shapes_c1024_bf16", "b1_r1024_shapes_c64_f16"]


@pytest.mark.parametrize("name", SAMPLED)
def test_workload_sampled(name):
    wl = synth.WORKLOADS[name]
    coords = coords_of(name)
    N = coords.shape[0]
    nbr_ref, _ = oracle_map(name)
    f, W, b, dY = synth.make_tensors(wl, N)
    r = run_gpu(coords, wl.grid, f, W, b, dY, wl.key_flag)
    assert np.array_equal(r["nbr"], nbr_ref)
    rng = np.random.default_rng(1234 + wl.seed)
    rows = np.sort(rng.choice(N, size=min(N, 4096), replace=False))
    ncol = min(wl.cout, 64)
    cols_out = np.sort(rng.choice(wl.cout, size=ncol, replace=False))
    cols_in = np.sort(rng.choice(wl.cin, size=min(wl.cin, 64), replace=False))
    out_ref = oracle_fwd_rows(nbr_ref, rows, cols_out, f, W, b)
    e_out = rel_fro(f64(r["out"][rows][:, cols_out]), out_ref)
    dX_ref = oracle_dgrad_rows(nbr_ref, rows, cols_in, dY, W)
    e_dx = rel_fro(f64(r["dX"][rows][:, cols_in]), dX_ref)
    # 27 taps x 16 x 16 = 6912 seeded full-sum dW entries (each a sum over every valid
    # pair of its tap), and every db entry
    ci = np.sort(rng.choice(wl.cin, size=16, replace=False))
    co = np.sort(rng.choice(wl.cout, size=16, replace=False))
    dW_ref, _ = oracle_wgrad_cols(nbr_ref, f, dY, ci, co)
    e_dw = rel_fro(f64(r["dW"][:, ci][:, :, co]), dW_ref)
    _, db_ref = oracle_wgrad_cols(nbr_ref, f[:, :1], dY, np.arange(1), np.arange(wl.cout))
    e_db = rel_fro(f64(r["db"]), db_ref)
    tol = TOL[wl.dtype]
    assert max(e_out, e_dx, e_dw, e_db) <= tol, (e_out, e_dx, e_dw, e_db)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("cin,cout", [(64, 64), (64, 128), (128, 64), (192, 64), (40, 24), (8, 8)])
def test_ragged_and_shapes(dtype, cin, cout):
    # N not a multiple of the tile, Cin != Cout, both tensor-core-shaped and CUDA-core-shaped channels
    coords = synth.random_coords(cin * 7 + cout, 1111, 2, 14, 14, 14)
    wl = synth.Workload("t", 2, 14, 0, ("sphere",), cin, cout, dtype, 9, 2.0)
    f, W, b, dY = synth.make_tensors(wl, coords.shape[0])
    full_check(coords, (2, 14, 14, 14), f, W, b, dY, TOL[dtype])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("cin,cout,n", [(256, 256, 1111), (64, 256, 1280), (256, 512, 1400), (512, 64, 600)])
def test_wide_blocks_one_unit_per_tile(dtype, cin, cout, n):
    """256-column output blocks with one unit per (tile, block) (no tap groups),
    odd and even tile counts, with and without bias: every element against the oracle."""
    coords = synth.random_coords(cin + cout + n, n, 1, 18, 18, 18)
    N = coords.shape[0]
    wl = synth.Workload("t", 1, 18, 0, ("sphere",), cin, cout, dtype, 21, 2.0)
    f, W, b, dY = synth.make_tensors(wl, N)
    full_check(coords, (1, 18, 18, 18), f, W, b, dY, TOL[dtype], flags=ops.VG_NO_SMALL_N_SPLIT)
    full_check(coords, (1, 18, 18, 18), f, W, None, dY, TOL[dtype], flags=ops.VG_NO_SMALL_N_SPLIT)


@pytest.mark.parametrize("dtype,cout", [("bf16", 256), ("f16", 512), ("f32", 256)])
def test_tile_pairs_rows_and_ragged_tail(dtype, cout):
    """256-column output blocks with at least as many tile pairs as SMs run on the
    kernel that feeds each weight tile to two consecutive tiles (each skipping its own
    absent taps).  Surface voxels (tiles with different tap masks) and an odd tile
    count whose last tile is partial: every column of 4096 sampled rows and of every
    row of the last three tiles in processing order, for out and dX, and sampled
    full-sum dW entries, against the oracle (fp32 runs as TF32)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = (2 * sms + 1) * 128 - 77
    wl = synth.Workload("t", 4, 112, 4, ("sphere", "torus"), 256, cout, dtype, 41, 2.0)
    coords_all = synth.make_coords(wl)
    assert coords_all.shape[0] >= n
    coords = coords_all[np.random.default_rng(41).permutation(coords_all.shape[0])[:n]]
    flags = ops.VG_ALLOW_TF32 if dtype == "f32" else 0
    f, W, b, dY = synth.make_tensors(wl, n)
    c = torch.from_numpy(coords).cuda()
    m = ops.NbrMap.alloc(n, wl.grid).build(c)
    fd, Wd, bd, dYd = (t.cuda() for t in (f, W, b, dY))
    ws = ops.conv_workspace(n, 256, cout, f.dtype, flags=flags)
    out = torch.empty(n, cout, dtype=f.dtype, device="cuda")
    dX = torch.empty(n, 256, dtype=f.dtype, device="cuda")
    dW = torch.empty_like(Wd)
    db = torch.empty_like(bd)
    ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, fd, Wd, bd, out, ws, flags=flags)
    ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dYd, fd, Wd, dX, dW, db, ws, flags=flags)
    assert m.status() == ops.VG_OK and ops.vg_conv_status(ws) == ops.VG_OK
    nbr_ref, _ = oracle.nbrmap(coords, *wl.grid)
    assert np.array_equal(u32(m.nbr), nbr_ref)
    order = m.sorted_idx().cpu().numpy().astype(np.int64)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([rng.choice(n, size=4096, replace=False), order[(n // 128 - 2) * 128:]]))
    tol = 5e-3 if dtype == "f32" else TOL[dtype]
    e_out = rel_fro(f64(out.cpu()[rows]), oracle_fwd_rows(nbr_ref, rows, np.arange(cout), f, W, b))
    e_dx = rel_fro(f64(dX.cpu()[rows]), oracle_dgrad_rows(nbr_ref, rows, np.arange(256), dY, W))
    ci = np.sort(rng.choice(256, size=16, replace=False))
    co = np.sort(rng.choice(cout, size=16, replace=False))
    dW_ref, _ = oracle_wgrad_cols(nbr_ref, f, dY, ci, co)
    e_dw = rel_fro(f64(dW.cpu()[:, ci][:, :, co]), dW_ref)
    assert max(e_out, e_dx, e_dw) <= tol, (e_out, e_dx, e_dw)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n", [3000, 60000])
def test_workspace_contents_do_not_matter(n, dtype):
    """The GEMM kernels hand out work units through counters in the conv workspace
    (reset before a launch with more units than CTAs; with fewer, every claim ends
    the sequence whatever the counter holds).  A workspace full of 0xFF bytes and a
    zeroed one must give the same bits, in both regimes (bf16, and fp32 as TF32)."""
    coords = synth.random_coords(n, n, 1, 64, 64, 64)
    N = coords.shape[0]
    wl = synth.Workload("t", 1, 64, 0, ("sphere",), 256, 256, dtype, 31, 2.0)
    f, W, b, dY = (t.cuda() for t in synth.make_tensors(wl, N))
    flags = ops.VG_NO_SMALL_N_SPLIT | (ops.VG_ALLOW_TF32 if dtype == "f32" else 0)
    m = ops.NbrMap.alloc(N, (1, 64, 64, 64)).build(torch.from_numpy(coords).cuda())
    res = []
    for fill in (0x00, 0xFF):
        ws = ops.conv_workspace(N, 256, 256, f.dtype, flags=flags)
        ws.view(torch.uint8).fill_(fill)
        out = torch.empty(N, 256, dtype=f.dtype, device="cuda")
        dX = torch.empty_like(out)
        dW = torch.empty_like(W)
        db = torch.empty_like(b)
        ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, out, ws, flags=flags)
        ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, dX, dW, db, ws, flags=flags)
        assert ops.vg_conv_status(ws) == ops.VG_OK
        res.append((out, dX, dW, db))
    for a, b_ in zip(*res):
        assert torch.equal(a, b_)


def test_bias_none_and_closed_form():
    # all-ones features and weights: out[i] = popcount(mask_i) * Cin exactly (small integers)
    coords = coords_of("b4_r64_spheres_c64_f16")
    N = coords.shape[0]
    _, mask_ref = oracle_map("b4_r64_spheres_c64_f16")
    f = torch.ones(N, 64, dtype=torch.float16)
    W = torch.ones(27, 64, 64, dtype=torch.float16)
    r = run_gpu(coords, (4, 64, 64, 64), f, W, None, torch.zeros(N, 64, dtype=torch.float16))
    pop = np.array([bin(int(x)).count("1") for x in mask_ref], dtype=np.float64)
    assert np.array_equal(f64(r["out"]), np.repeat(pop[:, None] * 64, 64, axis=1))
    assert torch.count_nonzero(r["dW"]) == 0 and torch.count_nonzero(r["db"]) == 0


def test_wgrad_is_deterministic():
    name = "b2_r256_shapes_c128_bf16"
    wl = synth.WORKLOADS[name]
    coords = coords_of(name)
    f, W, b, dY = synth.make_tensors(wl, coords.shape[0])
    outs = [run_gpu(coords, wl.grid, f, W, b, dY) for _ in range(3)]
    for o in outs[1:]:
        for k in ("out", "dX", "dW", "db"):
            assert torch.equal(o[k].view(torch.int16), outs[0][k].view(torch.int16)), k


def test_empty_input():
    m = ops.NbrMap.alloc(0, (1, 8, 8, 8)).build(torch.zeros(0, 4, dtype=torch.int32, device="cuda"))
    ws = ops.conv_workspace(0, 64, 64, torch.bfloat16)
    f = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.randn(27, 64, 64, device="cuda").bfloat16()
    out = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, None, out, ws)
    dW = torch.full((27, 64, 64), 3.0, dtype=torch.bfloat16, device="cuda")
    db = torch.full((64,), 3.0, dtype=torch.bfloat16, device="cuda")
    ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, f, f, W, f, dW, db, ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dW) == 0 and torch.count_nonzero(db) == 0


def test_cuda_graph_capture_matches_eager():
    # the whole step (map build, fwd, bwd) is stream-ordered and capturable
    wl = synth.WORKLOADS["b4_r64_spheres_c64_f16"]
    coords = torch.from_numpy(coords_of(wl.name)).cuda()
    N = coords.shape[0]
    f, W, b, dY = (t.cuda() for t in synth.make_tensors(wl, N))
    s = torch.cuda.Stream()
    outs = {}
    for mode in ("eager", "graph"):
        m = ops.NbrMap.alloc(N, wl.grid)
        ws = ops.conv_workspace(N, 64, 64, f.dtype)
        out = torch.empty(N, 64, dtype=f.dtype, device="cuda")
        dX = torch.empty_like(out)
        dW = torch.empty_like(W)
        db = torch.empty_like(b)

        def step():
            m.build(coords, s)
            ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, out, ws, stream=s)
            ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, dX, dW, db, ws, stream=s)

        if mode == "eager":
            with torch.cuda.stream(s):
                step()
        else:
            with torch.cuda.stream(s):
                step()  # first call outside capture (kernel attributes are set here)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                step()
            for t_ in (out, dX, dW, db):
                t_.zero_()
            g.replay()
        s.synchronize()
        assert m.status(s) == ops.VG_OK
        outs[mode] = [t_.clone() for t_ in (out, dX, dW, db)]
    for a_, b_ in zip(outs["eager"], outs["graph"]):
        assert torch.equal(a_, b_)


@pytest.mark.parametrize("name", ["b4_r64_spheres_c64_f16", "b2_r256_shapes_c128_bf16"])
def test_three_streams_match_one_stream(name):
    # the benchmark's step: after the map build, forward, input gradient and weight
    # gradient run on three streams, each with its own conv workspace, sharing the map;
    # replayed from a CUDA graph it must give the same bits as the calls on one stream
    wl = synth.WORKLOADS[name]
    coords = torch.from_numpy(coords_of(name)).cuda()
    N = coords.shape[0]
    f, W, b, dY = (t.cuda() for t in synth.make_tensors(wl, N))
    m = ops.NbrMap.alloc(N, wl.grid, wl.key_flag)
    ws = [ops.conv_workspace(N, wl.cin, wl.cout, f.dtype) for _ in range(3)]
    s0, s1, s2 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def outputs():
        return (torch.empty(N, wl.cout, dtype=f.dtype, device="cuda"),
                torch.empty(N, wl.cin, dtype=f.dtype, device="cuda"),
                torch.empty_like(W), torch.empty_like(b))

    ref = outputs()
    with torch.cuda.stream(s0):
        m.build(coords, s0)
        ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, ref[0], ws[0], stream=s0)
        ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, ref[1], ref[2], ref[3], ws[0], stream=s0)
    s0.synchronize()
    got = outputs()

    def step():
        m.build(coords, s0)
        s1.wait_stream(s0)
        s2.wait_stream(s0)
        ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, got[0], ws[0], stream=s0)
        ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, got[1], None, None, ws[1], stream=s1)
        ops.vg_subm_conv3d_bwd(m.ws, m.nbr, m.mask, dY, f, W, None, got[2], got[3], ws[2], stream=s2)
        s0.wait_stream(s1)
        s0.wait_stream(s2)

    with torch.cuda.stream(s0):
        step()  # eager, also sets kernel attributes before the capture
    s0.synchronize()
    for t_, r_ in zip(got, ref):
        assert torch.equal(t_, r_)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s0):
        step()
    for t_ in got:
        t_.zero_()
    with torch.cuda.stream(s0):
        g.replay()
    s0.synchronize()
    assert m.status(s0) == ops.VG_OK
    assert all(ops.vg_conv_status(w, s0) == ops.VG_OK for w in ws)
    for t_, r_ in zip(got, ref):
        assert torch.equal(t_, r_)


@pytest.mark.parametrize("dtype,cin,cout", [("f16", 64, 128), ("f32", 24, 16)])
def test_anisotropic_grid(dtype, cin, cout):
    # three different grid extents and three batch elements: the linearisation,
    # the tap offsets and the row order must keep the axes apart
    grid = (3, 5, 9, 13)
    coords = synth.random_coords(77, 700, *grid)
    wl = synth.Workload("t", 3, 13, 0, ("sphere",), cin, cout, dtype, 11, 2.0)
    f, W, b, dY = synth.make_tensors(wl, coords.shape[0])
    full_check(coords, grid, f, W, b, dY, TOL[dtype])


# ---------------------------------------------------------------- TF32 (VG_ALLOW_TF32)
TF32_TOL = 5e-3


def test_tf32_sphere_workload():
    # the fp32 16^3 sphere (Cin = Cout = 32): forward and input gradient on the tensor
    # cores as TF32, within the TF32 bound of the oracle
    wl = synth.WORKLOADS["sphere16_c32_f32"]
    coords = coords_of(wl.name)
    f, W, b, dY = synth.make_tensors(wl, coords.shape[0])
    assert ops.vg_conv_describe(coords.shape[0], 32, 32, torch.float32, ops.VG_ALLOW_TF32)["tensor_core"] == 2
    errs = full_check(coords, wl.grid, f, W, b, dY, TF32_TOL, flags=ops.VG_ALLOW_TF32)
    assert errs["out"] > 1e-5  # the TF32 path really ran (the FFMA path is ~3e-7 on this case)


@pytest.mark.parametrize("cin,cout", [(32, 32), (64, 64), (64, 128), (128, 64), (192, 64), (32, 96), (256, 256),
                                      (160, 512)])
def test_tf32_ragged_and_shapes(cin, cout):
    coords = synth.random_coords(cin * 5 + cout, 1111, 2, 14, 14, 14)
    wl = synth.Workload("t", 2, 14, 0, ("sphere",), cin, cout, "f32", 13, 2.0)
    f, W, b, dY = synth.make_tensors(wl, coords.shape[0])
    full_check(coords, (2, 14, 14, 14), f, W, b, dY, TF32_TOL, flags=ops.VG_ALLOW_TF32)


def test_tf32_anisotropic_grid():
    grid = (3, 5, 9, 13)
    coords = synth.random_coords(78, 700, *grid)
    wl = synth.Workload("t", 3, 13, 0, ("sphere",), 32, 64, "f32", 12, 2.0)
    f, W, b, dY = synth.make_tensors(wl, coords.shape[0])
    full_check(coords, grid, f, W, b, dY, TF32_TOL, flags=ops.VG_ALLOW_TF32)


def test_tf32_flag_falls_back_to_ffma_for_other_channels():
    # channels that are not multiples of 32 keep the exact FFMA path under the flag
    coords = synth.random_coords(3, 500, 1, 12, 12, 12)
    wl = synth.Workload("t", 1, 12, 0, ("sphere",), 24, 40, "f32", 14, 2.0)
    f, W, b, dY = synth.make_tensors(wl, coords.shape[0])
    assert ops.vg_conv_describe(coords.shape[0], 24, 40, torch.float32, ops.VG_ALLOW_TF32)["tensor_core"] == 0
    full_check(coords, (1, 12, 12, 12), f, W, b, dY, TOL["f32"], flags=ops.VG_ALLOW_TF32)


# ---------------------------------------------------------------- small-N forward (tap groups)
@pytest.mark.parametrize("dtype,c,n", [("bf16", 256, 2000), ("f16", 64, 900), ("f32", 128, 1500)])
def test_small_n_split_matches_oracle_and_unsplit(dtype, c, n):
    # few voxels: fewer (tile, channel block) units than SMs, so the forward and the
    # input gradient cut each unit's taps into groups summed by a second kernel
    coords = synth.random_coords(c + n, n, 1, 20, 20, 20)
    N = coords.shape[0]
    flags = ops.VG_ALLOW_TF32 if dtype == "f32" else 0
    d_split = ops.vg_conv_describe(N, c, c, synth.torch_dtype(dtype), flags)
    d_plain = ops.vg_conv_describe(N, c, c, synth.torch_dtype(dtype), flags | ops.VG_NO_SMALL_N_SPLIT)
    assert d_split["launches_fwd"] == 3 and d_plain["launches_fwd"] == 2
    wl = synth.Workload("t", 1, 20, 0, ("sphere",), c, c, dtype, 15, 2.0)
    f, W, b, dY = synth.make_tensors(wl, N)
    tol = TF32_TOL if dtype == "f32" else TOL[dtype]
    errs = full_check(coords, (1, 20, 20, 20), f, W, b, dY, tol, flags=flags)
    r_plain = run_gpu(coords, (1, 20, 20, 20), f, W, b, dY, flags=flags | ops.VG_NO_SMALL_N_SPLIT)
    r_split = run_gpu(coords, (1, 20, 20, 20), f, W, b, dY, flags=flags)
    for k in ("out", "dX"):
        assert rel_fro(f64(r_split[k]), f64(r_plain[k])) <= tol, (k, errs)
    # the split pass is deterministic: the same bits twice
    r_again = run_gpu(coords, (1, 20, 20, 20), f, W, b, dY, flags=flags)
    for k in ("out", "dX"):
        assert torch.equal(r_again[k], r_split[k]), k



def test_hilbert_row_order_gives_the_same_convolution():
    # the row order only changes the schedule: results stay within the dtype bound of
    # the oracle (sampled rows and dW entries at full size)
    name = "b2_r256_shapes_c128_bf16"
    wl = synth.WORKLOADS[name]
    coords = coords_of(name)
    N = coords.shape[0]
    nbr_ref, _ = oracle_map(name)
    f, W, b, dY = synth.make_tensors(wl, N)
    r = run_gpu(coords, wl.grid, f, W, b, dY, wl.key_flag | ops.VG_ORDER_HILBERT)
    rng = np.random.default_rng(99)
    rows = np.sort(rng.choice(N, size=2048, replace=False))
    cols = np.sort(rng.choice(wl.cout, size=32, replace=False))
    e_out = rel_fro(f64(r["out"][rows][:, cols]), oracle_fwd_rows(nbr_ref, rows, cols, f, W, b))
    e_dx = rel_fro(f64(r["dX"][rows][:, cols]), oracle_dgrad_rows(nbr_ref, rows, cols, dY, W))
    ci = np.sort(rng.choice(wl.cin, size=8, replace=False))
    co = np.sort(rng.choice(wl.cout, size=8, replace=False))
    dW_ref, _ = oracle_wgrad_cols(nbr_ref, f, dY, ci, co)
    e_dw = rel_fro(f64(r["dW"][:, ci][:, :, co]), dW_ref)
    assert max(e_out, e_dx, e_dw) <= TOL[wl.dtype], (e_out, e_dx, e_dw)


def test_tf32_weight_gradient_sampled_at_full_size():
    # the 512^3 voxels with fp32 features under VG_ALLOW_TF32 (Cin = Cout = 256): the
    # tensor-core TF32 weight gradient on 6912 full-sum dW entries and all of db
    name = "b1_r512_shapes_c256_bf16"
    base = synth.WORKLOADS[name]
    wl = synth.Workload("tf32_512", base.B, base.res, base.shapes_per_sample, base.kinds, 256, 256, "f32",
                        base.seed, 2.0)
    coords = coords_of(name)
    N = coords.shape[0]
    nbr_ref, _ = oracle_map(name)
    f, W, b, dY = synth.make_tensors(wl, N)
    r = run_gpu(coords, wl.grid, f, W, b, dY, flags=ops.VG_ALLOW_TF32)
    rng = np.random.default_rng(5)
    ci = np.sort(rng.choice(256, size=16, replace=False))
    co = np.sort(rng.choice(256, size=16, replace=False))
    dW_ref, _ = oracle_wgrad_cols(nbr_ref, f, dY, ci, co)
    _, db_ref = oracle_wgrad_cols(nbr_ref, f[:, :1], dY, np.arange(1), np.arange(256))
    e_dw = rel_fro(f64(r["dW"][:, ci][:, :, co]), dW_ref)
    e_db = rel_fro(f64(r["db"]), db_ref)
    rows = np.sort(rng.choice(N, size=2048, replace=False))
    e_out = rel_fro(f64(r["out"][rows][:, co]), oracle_fwd_rows(nbr_ref, rows, co, f, W, b))
    assert max(e_dw, e_db, e_out) <= TF32_TOL, (e_dw, e_db, e_out)
    assert e_dw > 1e-6  # TF32 products, not the exact FFMA path

