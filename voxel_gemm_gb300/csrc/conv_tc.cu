// Tensor-core (tcgen05 / TMEM) masked implicit GEMM — placeholder until the kernel lands.
#include "common.cuh"
#include "internal.h"

namespace vg {
int tc_supported(int, int, int) { return 0; }
int tc_wgrad_splits(int64_t, int, int) { return 1; }
size_t tc_packed_weight_bytes(int, int, int) { return 0; }
int tc_pack_weights(const void*, int, int, int, int, void*, const uint32_t*, cudaStream_t) { return VG_ERR_UNSUPPORTED; }
int tc_gather_pass(const GatherPass&, const void*, cudaStream_t) { return VG_ERR_UNSUPPORTED; }
int tc_wgrad(const WgradPass&, cudaStream_t) { return VG_ERR_UNSUPPORTED; }
int tc_fwd_launches() { return 2; }
int tc_bwd_launches() { return 6; }
}  // namespace vg
