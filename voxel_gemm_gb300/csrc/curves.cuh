// Space-filling-curve codes of voxel coordinates on the GPU: z-order (Morton)
// and Hilbert, as the pages' serialize module names them ("Contribution Tasks —
// JeffreyXiang/FlexGEMM", §二 module table, kernels.cuda.serialize:
// z_order_encode/decode, hilbert_encode/decode).
//
// A code packs the curve position of (x, y, z) in [0, 2^L)^3 into 3L bits;
// level j (bit j of each coordinate) occupies bits 3j+2 (x), 3j+1 (y), 3j (z).
// The Hilbert curve is J. Skilling's ("Programming the Hilbert curve", AIP
// Conf. Proc. 707, 2004): its "transposed" index is formed by undoing, level by
// level from the top, each sub-cube's rotation/reflection and then Gray-coding;
// the transposed words are then interleaved like a z-order code.
#pragma once
#include <cstdint>

namespace vg {

constexpr int kCurveZOrder = 0;
constexpr int kCurveHilbert = 1;

// Bit j of v moved to bit 3j (j < 21).
__host__ __device__ __forceinline__ uint64_t spread3(uint32_t v) {
    uint64_t x = v & 0x1FFFFFu;
    x = (x | (x << 32)) & 0x001F00000000FFFFull;
    x = (x | (x << 16)) & 0x001F0000FF0000FFull;
    x = (x | (x << 8)) & 0x100F00F00F00F00Full;
    x = (x | (x << 4)) & 0x10C30C30C30C30C3ull;
    x = (x | (x << 2)) & 0x1249249249249249ull;
    return x;
}
// Bits 3j of v gathered to bit j (the inverse of spread3).
__host__ __device__ __forceinline__ uint32_t gather3(uint64_t v) {
    uint64_t x = v & 0x1249249249249249ull;
    x = (x | (x >> 2)) & 0x10C30C30C30C30C3ull;
    x = (x | (x >> 4)) & 0x100F00F00F00F00Full;
    x = (x | (x >> 8)) & 0x001F0000FF0000FFull;
    x = (x | (x >> 16)) & 0x001F00000000FFFFull;
    x = (x | (x >> 32)) & 0x1FFFFFull;
    return (uint32_t)x;
}

__host__ __device__ __forceinline__ uint64_t zorder3(uint32_t x, uint32_t y, uint32_t z) {
    return (spread3(x) << 2) | (spread3(y) << 1) | spread3(z);
}

__host__ __device__ __forceinline__ uint64_t hilbert3(uint32_t x, uint32_t y, uint32_t z, int bits) {
    if (bits <= 0) return 0;
    // level by level from the top: a set bit of an axis reflects the lower bits of
    // x; a clear bit swaps the lower bits of x and that axis
    for (int lvl = bits - 1; lvl >= 1; --lvl) {
        const uint32_t q = 1u << lvl, lo = q - 1u;
        if (x & q) x ^= lo;
        if (y & q) {
            x ^= lo;
        } else {
            const uint32_t s = (x ^ y) & lo;
            x ^= s;
            y ^= s;
        }
        if (z & q) {
            x ^= lo;
        } else {
            const uint32_t s = (x ^ z) & lo;
            x ^= s;
            z ^= s;
        }
    }
    y ^= x;  // Gray code across the three words
    z ^= y;
    uint32_t flip = 0;
    for (int lvl = bits - 1; lvl >= 1; --lvl)
        if (z & (1u << lvl)) flip ^= (1u << lvl) - 1u;
    return zorder3(x ^ flip, y ^ flip, z ^ flip);
}

__host__ __device__ __forceinline__ void hilbert3_inverse(uint64_t c, int bits, uint32_t& x, uint32_t& y,
                                                          uint32_t& z) {
    x = gather3(c >> 2);
    y = gather3(c >> 1);
    z = gather3(c);
    if (bits <= 0) return;
    const uint32_t g = z >> 1;  // undo the Gray code
    z ^= y;
    y ^= x;
    x ^= g;
    for (int lvl = 1; lvl < bits; ++lvl) {  // redo the sub-cube transforms, bottom level first
        const uint32_t q = 1u << lvl, lo = q - 1u;
        if (z & q) {
            x ^= lo;
        } else {
            const uint32_t s = (x ^ z) & lo;
            x ^= s;
            z ^= s;
        }
        if (y & q) {
            x ^= lo;
        } else {
            const uint32_t s = (x ^ y) & lo;
            x ^= s;
            y ^= s;
        }
        if (x & q) x ^= lo;
    }
}

}  // namespace vg
