// Shared device/host helpers of the GPU library (not used by the CPU oracle).
#pragma once
#include <cstdint>
#include <cstddef>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "vg.h"

namespace vg {

constexpr uint32_t kNone = VG_NONE;
constexpr int kTaps = 27;
constexpr int kTileRows = VG_TILE_ROWS;

// Device-side error record bits (nbr-map header word 0 and the conv workspace word).
constexpr uint32_t kErrRange = 1u;
constexpr uint32_t kErrDup = 2u;
constexpr uint32_t kErrFull = 4u;
constexpr uint32_t kErrTimeout = 8u;
// A conv pass's error record is the first word of a 256-byte block; further
// words of that block hold the unit counters of the dynamically scheduled
// kernels (zeroed before each launch).
constexpr int kWgradUnitCounter = 16;
constexpr int kGatherUnitCounter = 32;

// Bound on mbarrier polls before a kernel gives up (~seconds at GB300 clocks).
constexpr uint32_t kSpinLimit = 1u << 26;

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// -------- element conversion --------
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// -------- neighbour-map workspace layout (byte offsets; computed identically on host) --------
struct NbrLayout {
    int64_t n = 0;
    int key64 = 0;          // hash keys are 64-bit
    int sort64 = 0;         // Morton sort keys are 64-bit
    int sort_bits = 0;      // significant bits of the Morton key
    int fine_keep = 0;      // G: fine Morton bits kept below the tap mask
    int cap_log2 = 0;       // hash capacity = 2^cap_log2
    int64_t num_tiles = 0;  // ceil(n / 128)
    int64_t sort_blocks = 0;
    int sort_items = 16;    // keys per thread in the radix sort
    size_t off_hdr = 0, off_sorted = 0, off_tmask = 0, off_table = 0;
    size_t off_skeys_a = 0, off_skeys_b = 0, off_svals_b = 0, off_hist = 0, off_nbr_sorted = 0, total = 0;
    size_t off_status = 0, off_tickets = 0;
    size_t off_torder = 0, off_tkey_a = 0, off_tkey_b = 0, off_torder_b = 0;  // tile region sort
    int sms = 0;             // SM count the sort grid is sized for
    int curve = 0;           // curve of the row order: 0 z-order (Morton), 1 Hilbert
    int tile_passes = 1;     // radix passes of the tile region sort
    int64_t tile_blocks = 1; // blocks of one tile-sort pass
    // column index (instead of the hash table): B*X*Y columns, their counts and
    // starts, the scan's published chunk sums, and the voxels as {z, row}
    int cols = 0;
    int64_t ncols = 0, cchunks = 0;
    size_t off_ccnt = 0, off_cpart = 0, off_cticket = 0, off_cstart = 0, off_carr = 0, off_cent_a = 0,
           off_cent_b = 0, off_ccol_a = 0, off_ccol_b = 0, off_cpos = 0, off_crec = 0;
};

// Workspace layout of a regular (strided / transposed) convolution map: a header
// (status word, number of output sites), one submanifold-layout block per side
// (input sites, output sites: row order, tile masks, lists in processing order,
// tile order, hash table, sort scratch), the down/up neighbour tables and masks,
// the output coordinates, and the output-site candidate sort.
struct SparseLayout {
    int64_t n_in = 0, n_out = -1, cap_out = 0;
    int K = 3, stride = 2, pad = 1, T = 27;
    int B = 1, X = 1, Y = 1, Z = 1;
    int64_t Xo = 1, Yo = 1, Zo = 1;
    unsigned flags = 0;
    NbrLayout li, lo_cap, lo;  // input side; output side sized for cap_out; output side for n_out
    size_t side_o_bytes = 0;
    int cand64 = 0, cand_passes = 1, cand_items = 16;
    int64_t cand_n = 0, cand_blocks = 1, scan_blocks = 1;
    uint64_t sentinel = 0;     // key meaning "no output cell": the output grid's volume
    size_t off_hdr = 0, off_side_i = 0, off_side_o = 0, off_nbr_down = 0, off_mask_down = 0, off_nbr_up = 0,
           off_mask_up = 0, off_coords_out = 0, off_cand_a = 0, off_cand_b = 0, off_cand_va = 0, off_cand_vb = 0,
           off_cand_hist = 0, off_cand_status = 0, off_cand_tickets = 0, off_scan = 0, total = 0;
};

// dY in processing order as the weight gradient's B-operand image (Cout a
// multiple of 128): 8 KB tiles of 64 sorted rows x 64 channels, ordered [row
// group r / 64][channel block c / 64], each tile in the 128-byte-swizzled
// MN-major layout the MMA reads (row rr at (rr / 8) * 1024 + (rr % 8) * 128
// bytes, its 16-byte chunk cc stored at chunk cc ^ (rr % 8)); the B tile of one
// stage (64 rows, BN channels) is then one contiguous bulk copy.  Offset, in
// 16-bit elements, of chunk c8 (channels 8 * c8 .. 8 * c8 + 7) of sorted row r.
__host__ __device__ __forceinline__ int64_t dy_image_offset(int64_t r, int c8, int Cout) {
    const int rr = (int)(r & 63), cc = c8 & 7;
    return ((r >> 6) * (Cout >> 6) + (c8 >> 3)) * 4096 + (rr >> 3) * 512 + (rr & 7) * 64 + ((cc ^ (rr & 7)) << 3);
}

// fp32 dY in processing order as the TF32 weight gradient's B-operand image
// (K-major: the contraction runs over rows): per group of 32 sorted rows, each
// channel's 32 values form a 128-byte row, channels in order, in the 128-byte
// swizzle (channel c at (c / 8) * 1024 + (c % 8) * 128 bytes of its group, its
// 16-byte chunk of rows 4kc..4kc+3 stored at chunk kc ^ (c % 8)); the B tile of
// a stage (32 rows, BN channels) is then one contiguous bulk copy.  Offset, in
// floats, of sorted row r, channel c.
__host__ __device__ __forceinline__ int64_t tf32_dy_image_offset(int64_t r, int c, int Cout) {
    const int kc = (int)((r & 31) >> 2);
    return (r >> 5) * (int64_t)Cout * 32 + (c >> 3) * 256 + (c & 7) * 32 + ((kc ^ (c & 7)) << 2) + (int)(r & 3);
}

constexpr int kSortThreads = 256;
constexpr int kMaxSortPasses = 8;                     // 64-bit keys, 8-bit digits
constexpr int kRadixBits = 8;
constexpr int kRadix = 1 << kRadixBits;
constexpr int kFineOrderBits = 30;                    // Morton bits below the tap mask (1024^3 blocks)
constexpr int kKeptFineBits = 6;                      // of those, at most this many kept in the key (4x4x4 split)

}  // namespace vg
