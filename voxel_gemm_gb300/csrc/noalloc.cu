// Forward pass for callers that cannot allocate device memory.
//
// vg_subm_conv3d_fwd needs a caller-provided conv workspace (for the repacked
// weight tiles of the tensor-core path and a device error word).  Some callers
// cannot obtain one: plug-ins hosted by a runtime that owns all device memory and
// forbids allocation after start-up, and hot paths that cannot afford the
// device-wide synchronisation cudaMalloc/cudaFree imply.
// This entry point keeps its scratch in a fixed, file-scope __device__ array
// instead, so the caller passes only inputs and outputs.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace vg {
namespace {

// Largest packed-weight image the fixed scratch holds: 27 * Cin * Cout 16-bit
// values <= 8 MiB (for example Cin = Cout = 384).  Plus 256 bytes for the error word.
constexpr size_t kNoAllocWeightBytes = size_t(8) << 20;
constexpr size_t kNoAllocScratchBytes = 256 + kNoAllocWeightBytes;

// Every GPU that loads the library holds this array until the process exits.
// In host code the name is only a host-side stand-in: the device address is
// obtained with cudaGetSymbolAddress below and passed to the kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];  // null until a lookup on that device succeeded

// Device address of the scratch array on the current device.  Only a successful
// lookup is kept; a failed one (for example under a sticky error) returns
// VG_ERR_CUDA and is retried by the next call.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return VG_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return VG_OK;
}

}  // namespace
}  // namespace vg

using namespace vg;

extern "C" int vg_subm_conv3d_fwd_noalloc(const void* nbr_ws, const uint32_t* nbr, const uint32_t* mask,
                                          int64_t N, int dtype, const void* feats, const void* weight,
                                          const void* bias, void* out, int Cin, int Cout, unsigned flags,
                                          void* stream) {
    if (N < 0 || N >= (int64_t(1) << 31) || Cin <= 0 || Cout <= 0) return VG_ERR_INVALID_ARG;
    if (dtype != VG_F32 && dtype != VG_F16 && dtype != VG_BF16) return VG_ERR_INVALID_ARG;
    if (flags != 0 || Cin % 8 || Cout % 8) return VG_ERR_UNSUPPORTED;
    const bool tc = tc_supported(dtype, Cin, Cout) != 0;
    if (tc && tc_packed_weight_bytes(dtype, Cin, Cout) > kNoAllocWeightBytes) return VG_ERR_WORKSPACE_TOO_SMALL;
    auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
    if (!nbr_ws || mis(nbr_ws, 256)) return VG_ERR_INVALID_ARG;
    if (!weight || mis(weight, 16) || (bias && mis(bias, 16))) return VG_ERR_INVALID_ARG;
    if (N > 0 && (!nbr || !mask || !feats || !out || mis(nbr, 4) || mis(mask, 4) || mis(feats, 16) ||
                  mis(out, 16)))
        return VG_ERR_INVALID_ARG;
    void* scratch = nullptr;
    int st = scratch_address(&scratch);
    if (st != VG_OK) return st;
    if (N == 0) return VG_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    char* base = static_cast<char*>(scratch);
    uint32_t* err = reinterpret_cast<uint32_t*>(base);
    cudaMemsetAsync(err, 0, 4, s);  // the array keeps the previous call's contents
    GatherPass g;
    g.sorted_idx = vg_nbrmap_sorted_idx(nbr_ws);
    g.tile_mask = vg_nbrmap_tile_mask(nbr_ws, N);
    g.nbr = nbr;
    g.sorted_nbr = vg_nbrmap_sorted_nbr(nbr_ws, N);
    g.nbr_status = static_cast<const uint32_t*>(nbr_ws);
    g.n = N;
    g.A = feats;
    g.Kdim = Cin;
    g.W = weight;
    g.Cin = Cin;
    g.Cout = Cout;
    g.dgrad = 0;
    g.bias = bias;
    g.out = out;
    g.Ndim = Cout;
    g.dtype = dtype;
    g.err = err;
    if (tc) {
        st = tc_pack_weights(weight, dtype, Cin, Cout, 0, kTaps, base + 256, g.nbr_status, s);
        if (st == VG_OK) st = tc_gather_pass(g, base + 256, s);
    } else {
        st = simt_gather_pass(g, s);
    }
    if (st != VG_OK) return st;
    return cudaGetLastError() == cudaSuccess ? VG_OK : VG_ERR_CUDA;
}

extern "C" int vg_subm_conv3d_fwd_noalloc_status(void* stream) {
    void* scratch = nullptr;
    if (scratch_address(&scratch) != VG_OK) return VG_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t h = 0;
    if (cudaMemcpyAsync(&h, scratch, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return VG_ERR_CUDA;
    if (cudaMemsetAsync(scratch, 0, sizeof(h), s) != cudaSuccess) return VG_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return VG_ERR_CUDA;
    return (h & kErrTimeout) ? VG_ERR_DEVICE_TIMEOUT : VG_OK;
}
