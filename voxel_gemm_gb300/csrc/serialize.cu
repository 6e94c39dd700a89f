// Serialisation of voxel coordinates into space-filling-curve codes and back
// ("Contribution Tasks — JeffreyXiang/FlexGEMM", §二 module table,
// kernels.cuda.serialize: z_order_encode/decode and hilbert_encode/decode;
// ops.serialize encode_seq/decode_seq(coords, shape, mode)).
//
// code = (b << 3 * bits) | curve(x, y, z), one thread per voxel.
#include "common.cuh"
#include "curves.cuh"
#include "internal.h"

namespace vg {
namespace {

// A row with a coordinate outside [0, 2^bits), or a batch index that does not fit
// above the 3*bits curve bits, gets the code ~0 (no valid code has all bits set).
__global__ void __launch_bounds__(256)
k_encode(const int4* __restrict__ coords, int64_t n, int bits, int curve, uint64_t* __restrict__ codes) {
    const uint32_t lim = 1u << bits;
    const uint64_t b_lim = uint64_t(1) << (63 - 3 * bits);  // keeps the top bit of every valid code clear
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
        const int4 c = coords[i];
        if (c.x < 0 || (uint64_t)c.x >= b_lim || (uint32_t)c.y >= lim || (uint32_t)c.z >= lim ||
            (uint32_t)c.w >= lim) {
            codes[i] = ~0ull;
            continue;
        }
        const uint64_t h = curve == kCurveHilbert ? hilbert3((uint32_t)c.y, (uint32_t)c.z, (uint32_t)c.w, bits)
                                                  : zorder3((uint32_t)c.y, (uint32_t)c.z, (uint32_t)c.w);
        codes[i] = ((uint64_t)(uint32_t)c.x << (3 * bits)) | h;
    }
}

__global__ void __launch_bounds__(256)
k_decode(const uint64_t* __restrict__ codes, int64_t n, int bits, int curve, int4* __restrict__ coords) {
    const uint64_t low_mask = bits > 0 ? (uint64_t(1) << (3 * bits)) - 1 : 0;
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
        const uint64_t c = codes[i];
        uint32_t x, y, z;
        if (curve == kCurveHilbert) {
            hilbert3_inverse(c & low_mask, bits, x, y, z);
        } else {
            x = gather3((c & low_mask) >> 2);
            y = gather3((c & low_mask) >> 1);
            z = gather3(c & low_mask);
        }
        coords[i] = make_int4((int)(c >> (3 * bits)), (int)x, (int)y, (int)z);
    }
}

}  // namespace

int curve_encode(const int32_t* coords, int64_t n, int bits, int curve, uint64_t* codes, cudaStream_t s) {
    if (n == 0) return VG_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, 16 * (int64_t)plan_sms(0));
    k_encode<<<blocks, 256, 0, s>>>(reinterpret_cast<const int4*>(coords), n, bits, curve, codes);
    return VG_OK;
}

int curve_decode(const uint64_t* codes, int64_t n, int bits, int curve, int32_t* coords, cudaStream_t s) {
    if (n == 0) return VG_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, 16 * (int64_t)plan_sms(0));
    k_decode<<<blocks, 256, 0, s>>>(codes, n, bits, curve, reinterpret_cast<int4*>(coords));
    return VG_OK;
}

}  // namespace vg
