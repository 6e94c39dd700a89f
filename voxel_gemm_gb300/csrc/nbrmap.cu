// Neighbour map on the GPU: validate + linearise + hash insert, 27-tap probe with
// valid-tap mask, Morton (z-order) keys + stable LSD radix sort, per-tile masks.
//
// Follows "Contribution Tasks — JeffreyXiang/FlexGEMM", §二 module table:
// kernels.cuda.hash (hashmap_insert_3d_idx_as_val: the table maps a voxel's
// linearised coordinate to its row index), kernels.cuda.spconv
// (subm_neighbor_map: probe all 27 offsets of every voxel; migemm_neighmap_pp:
// row order + valid-tap summaries for the masked implicit GEMM), and
// kernels.cuda.serialize (z_order_encode) plus ops.utils.init_hashmap (32- or
// 64-bit keys chosen by grid volume).
#include "common.cuh"
#include "internal.h"

namespace vg {

// ------------------------------------------------------------------ hashing
// Fibonacci (multiplicative) hashing onto a power-of-two table, linear probing.
__device__ __forceinline__ uint32_t hash_slot(uint32_t key, int cap_log2) {
    return (key * 0x9E3779B1u) >> (32 - cap_log2);
}
__device__ __forceinline__ uint32_t hash_slot(uint64_t key, int cap_log2) {
    return (uint32_t)((key * 0x9E3779B97F4A7C15ull) >> (64 - cap_log2));
}
__device__ __forceinline__ uint32_t cas(uint32_t* p, uint32_t cmp, uint32_t v) {
    return atomicCAS(reinterpret_cast<unsigned int*>(p), cmp, v);
}
__device__ __forceinline__ uint64_t cas(uint64_t* p, uint64_t cmp, uint64_t v) {
    return (uint64_t)atomicCAS(reinterpret_cast<unsigned long long*>(p),
                               (unsigned long long)cmp, (unsigned long long)v);
}

template <typename K>
__global__ void k_insert(const int4* __restrict__ coords, int64_t n, int B, int X, int Y, int Z,
                         K* __restrict__ hkeys, uint32_t* __restrict__ hvals, int cap_log2,
                         uint32_t* __restrict__ status) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int4 c = coords[i];
    if (c.x < 0 || c.x >= B || c.y < 0 || c.y >= X || c.z < 0 || c.z >= Y || c.w < 0 || c.w >= Z) {
        atomicOr(status, kErrRange);
        return;
    }
    const K key = (K)((((int64_t)c.x * X + c.y) * Y + c.z) * Z + c.w);
    const uint32_t cmask = (1u << cap_log2) - 1u;
    const K empty = ~K(0);
    uint32_t slot = hash_slot(key, cap_log2);
    for (uint32_t p = 0; p <= cmask; ++p) {
        const K prev = cas(&hkeys[slot], empty, key);
        if (prev == empty) {
            hvals[slot] = (uint32_t)i;
            return;
        }
        if (prev == key) {
            atomicOr(status, kErrDup);
            return;
        }
        slot = (slot + 1u) & cmask;
    }
    atomicOr(status, kErrFull);
}

// One thread per (voxel, tap); a block covers 32 voxels x 27 taps so the
// nbr rows it writes are one contiguous, coalesced range.
constexpr int kProbeVoxels = 32;
constexpr int kProbeThreads = kProbeVoxels * kTaps;  // 864

template <typename K>
__global__ void __launch_bounds__(kProbeThreads)
k_probe(const int4* __restrict__ coords, int64_t n, int X, int Y, int Z,
        const K* __restrict__ hkeys, const uint32_t* __restrict__ hvals, int cap_log2,
        uint32_t* __restrict__ nbr, uint32_t* __restrict__ mask) {
    __shared__ uint32_t smask[kProbeVoxels];
    const int t = threadIdx.x;
    const int local = t / kTaps;
    const int k = t - local * kTaps;
    const int64_t i = (int64_t)blockIdx.x * kProbeVoxels + local;
    if (t < kProbeVoxels) smask[t] = 0;
    __syncthreads();
    if (i < n) {
        const int4 c = coords[i];
        const int x = c.y + (k / 9 - 1), y = c.z + ((k / 3) % 3 - 1), z = c.w + (k % 3 - 1);
        uint32_t j = kNone;
        if (x >= 0 && x < X && y >= 0 && y < Y && z >= 0 && z < Z) {
            const K key = (K)((((int64_t)c.x * X + x) * Y + y) * Z + z);
            const uint32_t cmask = (1u << cap_log2) - 1u;
            const K empty = ~K(0);
            uint32_t slot = hash_slot(key, cap_log2);
            for (uint32_t p = 0; p <= cmask; ++p) {
                const K kk = hkeys[slot];
                if (kk == key) { j = hvals[slot]; break; }
                if (kk == empty) break;
                slot = (slot + 1u) & cmask;
            }
        }
        nbr[i * kTaps + k] = j;
        if (j != kNone) atomicOr(&smask[local], 1u << k);
    }
    __syncthreads();
    if (t < kProbeVoxels) {
        const int64_t ii = (int64_t)blockIdx.x * kProbeVoxels + t;
        if (ii < n) mask[ii] = smask[t];
    }
}

// ------------------------------------------------------------------ row order
// Sort key of voxel i (the page's sorted_idx groups rows for the masked GEMM):
//   m      = (b << 3L) | interleave(x, y, z)            Morton (z-order) code
//   key    = ((m >> F) << (27 + F)) | (mask_i << F) | (m & (2^F - 1)),  F = min(3L, 21)
// i.e. coarse Morton block of 128^3 voxels, then the valid-tap mask, then the
// fine Morton order.  Rows of one tile then share most of their taps (few
// zero-filled rows in the MMA) while a block's rows stay spatially close
// (gathered neighbours are reused from L2).
template <typename SK>
__global__ void k_order_key(const int4* __restrict__ coords, const uint32_t* __restrict__ mask, int64_t n,
                            int L, SK* __restrict__ keys) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int4 c = coords[i];
    uint64_t m = (uint64_t)(uint32_t)c.x << (3 * L);
    for (int b = 0; b < L; ++b) {
        m |= (uint64_t)(((uint32_t)c.y >> b) & 1u) << (3 * b + 2);
        m |= (uint64_t)(((uint32_t)c.z >> b) & 1u) << (3 * b + 1);
        m |= (uint64_t)(((uint32_t)c.w >> b) & 1u) << (3 * b);
    }
    const int F = min(3 * L, kFineOrderBits);
    const uint64_t fine = m & ((uint64_t(1) << F) - 1);
    keys[i] = (SK)(((m >> F) << (kTaps + F)) | ((uint64_t)mask[i] << F) | fine);
}

// Stable LSD radix sort, 8-bit digits.  Pass = histogram -> scan -> scatter.
template <typename SK>
__global__ void __launch_bounds__(kSortThreads)
k_radix_hist(const SK* __restrict__ keys, int64_t n, int shift, uint32_t* __restrict__ hist,
             int64_t nblocks) {
    __shared__ uint32_t h[kRadix];
    const int t = threadIdx.x;
    h[t] = 0;
    __syncthreads();
    const int64_t base = (int64_t)blockIdx.x * kSortTile;
#pragma unroll 4
    for (int it = 0; it < kSortItems; ++it) {
        const int64_t idx = base + (int64_t)it * kSortThreads + t;
        if (idx < n) atomicAdd(&h[(uint32_t)(keys[idx] >> shift) & (kRadix - 1)], 1u);
    }
    __syncthreads();
    hist[(int64_t)t * nblocks + blockIdx.x] = h[t];
}

// Exclusive scan of `total` counters, one block of 1024 threads, each owning a
// contiguous segment (digit-major, block-minor order gives stable offsets).
__global__ void __launch_bounds__(1024) k_scan_exclusive(uint32_t* __restrict__ v, int64_t total) {
    __shared__ uint32_t wsum[32];
    const int t = threadIdx.x;
    const int64_t per = (total + 1023) / 1024;
    const int64_t b = t * per, e = min(total, b + per);
    uint32_t s = 0;
    for (int64_t i = b; i < e; ++i) s += v[i];
    // inclusive scan of s across the block
    uint32_t x = s;
    const int lane = t & 31, w = t >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[w] = x;
    __syncthreads();
    if (w == 0) {
        uint32_t y = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t z = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += z;
        }
        wsum[lane] = y;
    }
    __syncthreads();
    uint32_t run = x - s + (w > 0 ? wsum[w - 1] : 0u);
    for (int64_t i = b; i < e; ++i) {
        const uint32_t c = v[i];
        v[i] = run;
        run += c;
    }
}

template <typename SK>
__global__ void __launch_bounds__(kSortThreads)
k_radix_scatter(const SK* __restrict__ kin, const uint32_t* __restrict__ vin, SK* __restrict__ kout,
                uint32_t* __restrict__ vout, int64_t n, int shift,
                const uint32_t* __restrict__ hist, int64_t nblocks) {
    constexpr int kWarps = kSortThreads / 32;
    __shared__ uint32_t offs[kRadix];
    __shared__ uint32_t wcount[kWarps][kRadix];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    offs[t] = hist[(int64_t)t * nblocks + blockIdx.x];
    const int64_t base = (int64_t)blockIdx.x * kSortTile;
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int it = 0; it < kSortItems; ++it) {
        const int64_t idx = base + (int64_t)it * kSortThreads + t;
        const bool valid = idx < n;
        SK key = 0;
        uint32_t val = 0, d = kRadix;  // invalid lanes use a digit no bucket has
        if (valid) {
            key = kin[idx];
            val = vin ? vin[idx] : (uint32_t)idx;
            d = (uint32_t)(key >> shift) & (kRadix - 1);
        }
#pragma unroll
        for (int w = 0; w < kWarps; ++w) wcount[w][t] = 0;
        __syncthreads();
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        const uint32_t rank = __popc(peers & lt_mask);
        if (valid && lane == __ffs(peers) - 1) wcount[warp][d] = __popc(peers);
        __syncthreads();
        {
            uint32_t run = offs[t];
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const uint32_t c = wcount[w][t];
                wcount[w][t] = run;
                run += c;
            }
            offs[t] = run;
        }
        __syncthreads();
        if (valid) {
            const uint32_t pos = wcount[warp][d] + rank;
            kout[pos] = key;
            vout[pos] = val;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kTileRows)
k_tile_mask(const uint32_t* __restrict__ sorted_idx, const uint32_t* __restrict__ mask, int64_t n,
            uint32_t* __restrict__ tmask) {
    __shared__ uint32_t w[kTileRows / 32];
    const int64_t r = (int64_t)blockIdx.x * kTileRows + threadIdx.x;
    uint32_t m = r < n ? mask[sorted_idx[r]] : 0u;
    m = __reduce_or_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0) w[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t o = 0;
        for (int i = 0; i < kTileRows / 32; ++i) o |= w[i];
        tmask[blockIdx.x] = o;
    }
}

// nbr_sorted[r][k] = nbr[sorted_idx[r]][k] for r < n, VG_NONE for the padding rows
// up to a whole number of 128-row tiles.  One thread per entry (coalesced writes).
__global__ void k_sort_rows(const uint32_t* __restrict__ sorted_idx, const uint32_t* __restrict__ nbr,
                            int64_t n, int64_t total, uint32_t* __restrict__ nbr_sorted) {
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= total) return;
    const int64_t r = e / kTaps;
    const int k = (int)(e - r * kTaps);
    nbr_sorted[e] = r < n ? nbr[(int64_t)sorted_idx[r] * kTaps + k] : kNone;
}

// ------------------------------------------------------------------ host side
static int ceil_log2(int64_t v) {
    int b = 0;
    while ((int64_t(1) << b) < v) ++b;
    return b;
}

int nbr_layout(int64_t N, int B, int X, int Y, int Z, unsigned flags, NbrLayout* L) {
    if (N < 0 || N >= (int64_t(1) << 31) || B <= 0 || X <= 0 || Y <= 0 || Z <= 0) return VG_ERR_INVALID_ARG;
    if ((flags & VG_KEY32) && (flags & VG_KEY64)) return VG_ERR_INVALID_ARG;
    if (flags & ~(VG_KEY32 | VG_KEY64 | VG_TEST_SMALL_HASH)) return VG_ERR_INVALID_ARG;
    const double vol = (double)B * X * Y * Z;
    if (vol >= 18446744073709551615.0) return VG_ERR_UNSUPPORTED;
    NbrLayout l;
    l.n = N;
    if (flags & VG_KEY64) l.key64 = 1;
    else if (flags & VG_KEY32) {
        if (vol > 4294967294.0) return VG_ERR_INVALID_ARG;  // all-ones is the empty-slot marker
        l.key64 = 0;
    } else l.key64 = vol >= 1073741824.0 ? 1 : 0;
    const int lb = ceil_log2(B);
    const int lg = ceil_log2(std::max(X, std::max(Y, Z)));
    l.sort_bits = lb + 3 * lg + kTaps;  // Morton code + the 27-bit valid-tap mask
    if (l.sort_bits > 64) return VG_ERR_UNSUPPORTED;
    l.sort64 = l.sort_bits > 32 ? 1 : 0;
    if (flags & VG_TEST_SMALL_HASH) {
        int c = 4;
        while ((int64_t(1) << (c + 1)) <= N / 2) ++c;
        l.cap_log2 = c;
    } else {
        l.cap_log2 = std::max(6, ceil_log2(2 * std::max<int64_t>(N, 1)));
    }
    if (l.cap_log2 > 31) return VG_ERR_UNSUPPORTED;
    const size_t cap = size_t(1) << l.cap_log2;
    l.num_tiles = (N + kTileRows - 1) / kTileRows;
    l.sort_blocks = (N + kSortTile - 1) / kSortTile;
    const size_t ks = l.key64 ? 8 : 4, ss = l.sort64 ? 8 : 4;
    size_t o = 0;
    l.off_hdr = o;      o += 256;
    l.off_sorted = o;   o += align_up(4 * (size_t)N, 256);
    l.off_tmask = o;    o += align_up(4 * (size_t)l.num_tiles, 256);
    l.off_nbr_sorted = o; o += align_up(4 * (size_t)kTaps * kTileRows * l.num_tiles, 256);
    l.off_hkeys = o;    o += align_up(ks * cap, 256);
    l.off_hvals = o;    o += align_up(4 * cap, 256);
    l.off_skeys_a = o;  o += align_up(ss * (size_t)N, 256);
    l.off_skeys_b = o;  o += align_up(ss * (size_t)N, 256);
    l.off_svals_b = o;  o += align_up(4 * (size_t)N, 256);
    l.off_hist = o;     o += align_up(4 * (size_t)kRadix * l.sort_blocks, 256);
    l.total = o;
    *L = l;
    return VG_OK;
}

template <typename K>
static void launch_hash(const int4* coords, const NbrLayout& l, int B, int X, int Y, int Z,
                        char* ws, uint32_t* nbr, uint32_t* mask, cudaStream_t s) {
    const int64_t n = l.n;
    K* hk = reinterpret_cast<K*>(ws + l.off_hkeys);
    uint32_t* hv = reinterpret_cast<uint32_t*>(ws + l.off_hvals);
    uint32_t* status = reinterpret_cast<uint32_t*>(ws + l.off_hdr);
    const size_t cap = size_t(1) << l.cap_log2;
    cudaMemsetAsync(hk, 0xFF, cap * sizeof(K), s);
    k_insert<K><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(coords, n, B, X, Y, Z, hk, hv,
                                                          l.cap_log2, status);
    k_probe<K><<<(unsigned)((n + kProbeVoxels - 1) / kProbeVoxels), kProbeThreads, 0, s>>>(
        coords, n, X, Y, Z, hk, hv, l.cap_log2, nbr, mask);
}

template <typename SK>
static void launch_sort(const int4* coords, const uint32_t* mask, const NbrLayout& l, int X, int Y, int Z,
                        char* ws, cudaStream_t s) {
    const int64_t n = l.n;
    const int L = ceil_log2(std::max(X, std::max(Y, Z)));
    SK* ka = reinterpret_cast<SK*>(ws + l.off_skeys_a);
    SK* kb = reinterpret_cast<SK*>(ws + l.off_skeys_b);
    uint32_t* v0 = reinterpret_cast<uint32_t*>(ws + l.off_sorted);
    uint32_t* v1 = reinterpret_cast<uint32_t*>(ws + l.off_svals_b);
    uint32_t* hist = reinterpret_cast<uint32_t*>(ws + l.off_hist);
    k_order_key<SK><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(coords, mask, n, L, ka);
    const int passes = std::max(1, (l.sort_bits + kRadixBits - 1) / kRadixBits);
    const unsigned g = (unsigned)l.sort_blocks;
    const uint32_t* vin = nullptr;
    for (int p = 0; p < passes; ++p) {
        const SK* kin = (p % 2 == 0) ? ka : kb;
        SK* kout = (p % 2 == 0) ? kb : ka;
        uint32_t* vout = ((passes - 1 - p) % 2 == 0) ? v0 : v1;
        const int shift = p * kRadixBits;
        k_radix_hist<SK><<<g, kSortThreads, 0, s>>>(kin, n, shift, hist, l.sort_blocks);
        k_scan_exclusive<<<1, 1024, 0, s>>>(hist, (int64_t)kRadix * l.sort_blocks);
        k_radix_scatter<SK><<<g, kSortThreads, 0, s>>>(kin, vin, kout, vout, n, shift, hist,
                                                      l.sort_blocks);
        vin = vout;
    }
}

int nbr_build(const int32_t* coords, int64_t N, int B, int X, int Y, int Z, unsigned flags,
              void* ws_, size_t ws_bytes, uint32_t* nbr, uint32_t* mask, cudaStream_t s) {
    NbrLayout l;
    int st = nbr_layout(N, B, X, Y, Z, flags, &l);
    if (st != VG_OK) return st;
    if (!ws_ || (reinterpret_cast<uintptr_t>(ws_) & 255)) return VG_ERR_INVALID_ARG;
    if (ws_bytes < l.total) return VG_ERR_WORKSPACE_TOO_SMALL;
    if (N > 0 && (!coords || !nbr || !mask)) return VG_ERR_INVALID_ARG;
    if (N > 0 && ((reinterpret_cast<uintptr_t>(coords) & 15) || (reinterpret_cast<uintptr_t>(nbr) & 3) ||
                  (reinterpret_cast<uintptr_t>(mask) & 3)))
        return VG_ERR_INVALID_ARG;
    char* ws = static_cast<char*>(ws_);
    cudaGetLastError();  // clear any stale error so the check below is ours
    cudaMemsetAsync(ws + l.off_hdr, 0, 256, s);
    if (N > 0) {
        const int4* c4 = reinterpret_cast<const int4*>(coords);
        if (l.key64) launch_hash<uint64_t>(c4, l, B, X, Y, Z, ws, nbr, mask, s);
        else launch_hash<uint32_t>(c4, l, B, X, Y, Z, ws, nbr, mask, s);
        if (l.sort64) launch_sort<uint64_t>(c4, mask, l, X, Y, Z, ws, s);
        else launch_sort<uint32_t>(c4, mask, l, X, Y, Z, ws, s);
        k_tile_mask<<<(unsigned)l.num_tiles, kTileRows, 0, s>>>(
            reinterpret_cast<const uint32_t*>(ws + l.off_sorted), mask, N,
            reinterpret_cast<uint32_t*>(ws + l.off_tmask));
        const int64_t total = (int64_t)kTaps * kTileRows * l.num_tiles;
        k_sort_rows<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
            reinterpret_cast<const uint32_t*>(ws + l.off_sorted), nbr, N, total,
            reinterpret_cast<uint32_t*>(ws + l.off_nbr_sorted));
    }
    return cudaGetLastError() == cudaSuccess ? VG_OK : VG_ERR_CUDA;
}

int nbr_status(const void* ws, cudaStream_t s) {
    if (!ws) return VG_ERR_INVALID_ARG;
    uint32_t h = 0;
    if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return VG_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return VG_ERR_CUDA;
    if (h & kErrRange) return VG_ERR_COORD_OUT_OF_RANGE;
    if (h & kErrDup) return VG_ERR_DUPLICATE_COORD;
    if (h & kErrFull) return VG_ERR_HASH_FULL;
    return VG_OK;
}

}  // namespace vg
