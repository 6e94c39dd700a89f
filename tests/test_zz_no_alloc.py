"""vg_subm_conv3d_fwd_noalloc against vg_subm_conv3d_fwd and the oracle (GPU).

The no-allocation forward serves callers that cannot allocate device memory
(plug-ins under a runtime that owns all device memory, paths that cannot pay
for cudaMalloc's synchronisation): its scratch
is a fixed array inside the library instead of a caller workspace.  It runs the
same kernels as the workspace forward, so its output must be bit-identical to
it; a second call must not see stale state from the first, because every call
shares that array; and its device-side status word must read back VG_OK.
This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, f64, rel_fro, u32
from voxel_gemm_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def _case(seed, cin, cout, dtype, n=3000):
    coords = synth.random_coords(seed, n, 2, 20, 20, 20)
    wl = synth.Workload("noalloc", 2, 20, 0, ("sphere",), cin, cout, dtype, seed, 2.0)
    f, W, b, _ = synth.make_tensors(wl, coords.shape[0])
    m = ops.NbrMap.alloc(coords.shape[0], (2, 20, 20, 20)).build(torch.from_numpy(coords).cuda())
    return coords, m, f.cuda(), W.cuda(), b.cuda()


def _noalloc_raw(m, f, W, b, out):
    """Call the C ABI symbol directly (ctypes), no workspace argument."""
    L = ops.lib()
    N, cin = f.shape
    cout = W.shape[2]
    code = {torch.float32: ops.VG_F32, torch.float16: ops.VG_F16, torch.bfloat16: ops.VG_BF16}[f.dtype]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return L.vg_subm_conv3d_fwd_noalloc(p(m.ws), p(m.nbr), p(m.mask), N, code, p(f), p(W), p(b), p(out),
                                        cin, cout, 0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _noalloc_status():
    L = ops.lib()
    return L.vg_subm_conv3d_fwd_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("cin,cout,dtype", [(64, 64, "f16"), (128, 64, "bf16"), (32, 32, "f32")])
def test_noalloc_matches_fwd_on_two_calls(cin, cout, dtype):
    for seed in (1, 2):  # two calls in a row, different inputs
        coords, m, f, W, b = _case(seed * 31 + cin, cin, cout, dtype)
        ref = torch.empty(f.shape[0], cout, dtype=f.dtype, device="cuda")
        # the workspace forward in the same schedule (one unit per tile and channel
        # block; the no-allocation forward has no room for split partial sums)
        fl = ops.VG_NO_SMALL_N_SPLIT
        ws = ops.conv_workspace(f.shape[0], cin, cout, f.dtype, flags=fl)
        ops.vg_subm_conv3d_fwd(m.ws, m.nbr, m.mask, f, W, b, ref, ws, flags=fl)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc_raw(m, f, W, b, out) == ops.VG_OK
        assert _noalloc_status() == ops.VG_OK
        assert m.status() == ops.VG_OK and ops.vg_conv_status(ws) == ops.VG_OK
        # the same kernels on the same inputs: identical bits
        assert torch.equal(out.view(torch.uint8), ref.view(torch.uint8))
        # and against the oracle directly, within the dtype's bound
        nbr_ref, _ = oracle.nbrmap(coords, 2, 20, 20, 20)
        assert np.array_equal(u32(m.nbr), nbr_ref)
        err = rel_fro(f64(out), oracle.fwd(nbr_ref, f64(f), f64(W), f64(b)))
        assert err <= TOL[dtype], err


def test_noalloc_rejects_sizes_beyond_its_scratch():
    _, m, f, W, b = _case(5, 64, 64, "bf16", n=200)
    W_big = torch.zeros(27, 512, 512, dtype=torch.bfloat16, device="cuda")  # 14 MiB of packed weights
    f_big = torch.zeros(f.shape[0], 512, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(f.shape[0], 512, dtype=torch.bfloat16, device="cuda")
    assert _noalloc_raw(m, f_big, W_big, None, out) == ops.VG_ERR_WORKSPACE_TOO_SMALL
