"""vg_sum_ordered (the data-parallel gradient exchange's arithmetic) against a
plain PyTorch CPU fp32 sum in the same order: identical bits."""
import pytest
import torch

from voxel_gemm_gb300 import ops

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("nparts,count", [(1, 1000), (2, 27 * 64 * 64), (5, 1000003)])
def test_sum_is_rank_ordered_fp32_with_one_rounding(dtype, nparts, count):
    g = torch.Generator().manual_seed(nparts * 7 + count)
    parts = torch.randn(nparts, count, generator=g).to(dtype)
    ref = parts[0].float()
    for p in range(1, nparts):
        ref = ref + parts[p].float()
    ref = ref.to(dtype)
    out = torch.empty(count, dtype=dtype, device="cuda")
    ops.vg_sum_ordered(parts.cuda(), out)
    torch.cuda.synchronize()
    view = torch.int32 if dtype == torch.float32 else torch.int16
    assert torch.equal(out.cpu().view(view), ref.view(view))


def test_sum_rejects_bad_arguments():
    L = ops.lib()
    assert L.vg_sum_ordered(None, 0, 10, ops.VG_F32, None, None) == ops.VG_ERR_INVALID_ARG
    assert L.vg_sum_ordered(None, 2, 10, 9, None, None) == ops.VG_ERR_INVALID_ARG
