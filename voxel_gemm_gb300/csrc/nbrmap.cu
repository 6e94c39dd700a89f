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
#include "curves.cuh"
#include "internal.h"

namespace vg {

// ------------------------------------------------------------------ hashing
// Open addressing with linear probing over a power-of-two table of slots, each
// slot holding {key, row} together (one 8- or 16-byte access per probe).  The
// start slot keeps runs of 8 consecutive linear keys (8 voxels along z) in 8
// adjacent slots: group = key >> 3 is Fibonacci-hashed to a group of slots and
// key & 7 picks the slot inside it, so the 27 probes of one voxel touch about a
// dozen slot groups instead of 27 unrelated slots.
template <typename K> struct Slot;
template <> struct Slot<uint32_t> { using T = uint2; };       // {key, row}
template <> struct Slot<uint64_t> { using T = ulonglong2; };  // {key, row}

__device__ __forceinline__ uint32_t group_hash(uint32_t g, int bits) {
    return bits > 0 ? (g * 0x9E3779B1u) >> (32 - bits) : 0u;
}
__device__ __forceinline__ uint32_t group_hash(uint64_t g, int bits) {
    return bits > 0 ? (uint32_t)((g * 0x9E3779B97F4A7C15ull) >> (64 - bits)) : 0u;
}
template <typename K>
__device__ __forceinline__ uint32_t start_slot(K key, int cap_log2) {
    const int gb = cap_log2 - 3;
    return ((group_hash((K)(key >> 3), gb) << 3) | (uint32_t)(key & 7)) & ((1u << cap_log2) - 1u);
}
__device__ __forceinline__ uint32_t cas_key(uint2* s, uint32_t cmp, uint32_t v) {
    return atomicCAS(reinterpret_cast<unsigned int*>(&s->x), cmp, v);
}
__device__ __forceinline__ uint64_t cas_key(ulonglong2* s, uint64_t cmp, uint64_t v) {
    return (uint64_t)atomicCAS(reinterpret_cast<unsigned long long*>(&s->x), (unsigned long long)cmp,
                               (unsigned long long)v);
}

template <typename K>
__global__ void k_insert(const int4* __restrict__ coords, int64_t n, int B, int X, int Y, int Z,
                         typename Slot<K>::T* __restrict__ table, int cap_log2, uint32_t* __restrict__ status) {
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
    uint32_t slot = start_slot(key, cap_log2);
    for (uint32_t p = 0; p <= cmask; ++p) {
        const K prev = cas_key(&table[slot], empty, key);
        if (prev == empty) {
            table[slot].y = i;
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

// Row-order key of one voxel (see k_key_hist): coarse Morton block, tap mask, then
// the top G fine Morton bits (a 4x4x4 split of the block).  Below that the stable sort keeps
// the input order; dropping the low Morton bits saves radix passes, and rows with
// equal masks in one sub-block are gathered alike whatever their order.
// Curve code (b << 3L) | curve(x, y, z) of a voxel: the Morton (z-order) code,
// or the Hilbert code when the build asks for the Hilbert row order (L <= 20
// whenever the layout is valid).
__device__ __forceinline__ uint64_t curve_code(int4 c, int L, int curve) {
    const uint64_t h = curve == kCurveHilbert ? hilbert3((uint32_t)c.y, (uint32_t)c.z, (uint32_t)c.w, L)
                                              : zorder3((uint32_t)c.y, (uint32_t)c.z, (uint32_t)c.w);
    return ((uint64_t)(uint32_t)c.x << (3 * L)) | h;
}

__device__ __forceinline__ uint64_t order_key(int4 c, uint32_t mask, int L, int G, int curve) {
    const uint64_t m = curve_code(c, L, curve);
    const int F = min(3 * L, kFineOrderBits);
    const uint64_t fine = (m & ((uint64_t(1) << F) - 1)) >> (F - G);
    return ((m >> F) << (kTaps + G)) | ((uint64_t)mask << G) | fine;
}

// Probe of the 13 taps k < 13 (offsets with dx < 0, or dx = 0 and dy < 0, or
// dx = dy = 0 and dz < 0) plus the centre.  Since o_{26-k} = -o_k, finding j at
// tap k of voxel i also fixes nbr[j][26-k] = i, which this thread writes too;
// every entry is written by exactly one thread, the rest keep the VG_NONE fill.
// One block = 32 voxels x 14 threads.
constexpr int kProbeVoxels = 32;
constexpr int kHalfTaps = 14;  // taps 0..12 and the centre 13
constexpr int kProbeThreads = kProbeVoxels * kHalfTaps;  // 448

template <typename K>
__global__ void __launch_bounds__(kProbeThreads)
k_probe_half(const int4* __restrict__ coords, int64_t n, int X, int Y, int Z,
             const typename Slot<K>::T* __restrict__ table, int cap_log2, uint32_t* __restrict__ nbr) {
    const int t = threadIdx.x;
    const int local = t / kHalfTaps;
    const int k = t - local * kHalfTaps;
    const int64_t i = (int64_t)blockIdx.x * kProbeVoxels + local;
    if (i >= n) return;
    if (k == 13) {
        nbr[i * kTaps + 13] = (uint32_t)i;
        return;
    }
    const int4 c = coords[i];
    const int x = c.y + (k / 9 - 1), y = c.z + ((k / 3) % 3 - 1), z = c.w + (k % 3 - 1);
    if (x < 0 || x >= X || y < 0 || y >= Y || z < 0 || z >= Z) return;
    const K key = (K)((((int64_t)c.x * X + x) * Y + y) * Z + z);
    const uint32_t cmask = (1u << cap_log2) - 1u;
    const K empty = ~K(0);
    uint32_t slot = start_slot(key, cap_log2);
    for (uint32_t p = 0; p <= cmask; ++p) {
        const typename Slot<K>::T e = table[slot];
        if ((K)e.x == key) {
            const uint32_t j = (uint32_t)e.y;
            nbr[i * kTaps + k] = j;
            nbr[(int64_t)j * kTaps + (26 - k)] = (uint32_t)i;
            return;
        }
        if ((K)e.x == empty) return;
        slot = (slot + 1u) & cmask;
    }
}

// Valid-tap mask from a voxel's neighbour row.
__device__ __forceinline__ uint32_t row_mask(const uint32_t* __restrict__ row) {
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < kTaps; ++k) m |= (row[k] != kNone ? 1u : 0u) << k;
    return m;
}

// Row-order sort key of every voxel, its valid-tap mask, and the digit
// histograms of every radix pass (all passes in one read of the keys):
//   m   = (b << 3L) | interleave(x, y, z)            Morton (z-order) code
//   key = ((m >> F) << (27 + G)) | (mask << G) | ((m mod 2^F) >> (F - G))
// with F = min(3L, 30): the batch element (a 1024^3 block of a larger grid),
// then the valid-tap mask, then the top G fine Morton bits (the page's
// sorted_idx groups rows for the masked GEMM).  Rows of one tile then share
// nearly all of their taps (few zero-filled rows in the MMA: 88 % of the rows
// useful on a 512^3 surface, 95 % on 1024^3) while rows of one mask stay in
// Morton order (neighbours of consecutive tiles reused from L2).
template <typename SK>
__global__ void __launch_bounds__(kSortThreads)
k_key_globalhist(const int4* __restrict__ coords, const uint32_t* __restrict__ nbr, int64_t n, int L, int G,
                 int curve, int passes, uint32_t* __restrict__ mask, SK* __restrict__ keys,
                 uint32_t* __restrict__ ghist) {
    __shared__ uint32_t h[kMaxSortPasses][kRadix];
    const int t = threadIdx.x;
    for (int p = 0; p < passes; ++p) h[p][t] = 0;
    __syncthreads();
    for (int64_t i = (int64_t)blockIdx.x * kSortThreads + t; i < n; i += (int64_t)gridDim.x * kSortThreads) {
        const uint32_t m = row_mask(nbr + i * kTaps);
        mask[i] = m;
        const SK key = (SK)order_key(coords[i], m, L, G, curve);
        keys[i] = key;
        for (int p = 0; p < passes; ++p) atomicAdd(&h[p][(uint32_t)(key >> (p * kRadixBits)) & (kRadix - 1)], 1u);
    }
    __syncthreads();
    for (int p = 0; p < passes; ++p)
        if (h[p][t]) atomicAdd(&ghist[p * kRadix + t], h[p][t]);
}

// One stable counting pass of the LSD radix sort in a single kernel ("one
// sweep"): each block takes the next virtual tile (ticket order, so every block
// it waits on has already started), counts its digits, publishes the counts,
// looks back over earlier tiles' published counts for its global offsets, and
// scatters.  status[tile][digit] = flag (bits 62-63: 1 aggregate, 2 inclusive
// prefix) | count.  The look-back wait is bounded; giving up marks the map bad.
constexpr uint64_t kFlagAgg = 1ull << 62, kFlagInc = 2ull << 62, kCountMask = (1ull << 62) - 1;

__device__ __forceinline__ void st_release(uint64_t* p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_acquire(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

template <typename SK>
__global__ void __launch_bounds__(kSortThreads)
k_onesweep(const SK* __restrict__ kin, const uint32_t* __restrict__ vin, SK* __restrict__ kout,
           uint32_t* __restrict__ vout, int64_t n, int shift, const uint32_t* __restrict__ ghist_pass,
           uint64_t* __restrict__ status, uint32_t* __restrict__ ticket, int items, uint32_t* __restrict__ err) {
    constexpr int kWarps = kSortThreads / 32;
    extern __shared__ uint8_t dsm[];
    SK* s_keys = reinterpret_cast<SK*>(dsm);                                     // [items * 256]
    uint32_t* s_vals = reinterpret_cast<uint32_t*>(s_keys + items * kSortThreads);  // [items * 256]
    __shared__ uint32_t offs[kRadix];
    __shared__ uint32_t wcount[kWarps][kRadix];
    __shared__ uint32_t s_vid;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    if (t == 0) s_vid = atomicAdd(ticket, 1u);
    // bin bases: exclusive scan of this pass's global digit counts
    {
        const uint32_t c = ghist_pass[t];
        uint32_t inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) wcount[0][warp] = inc;
        __syncthreads();
        uint32_t base = inc - c;
        for (int w = 0; w < warp; ++w) base += wcount[0][w];
        offs[t] = base;
        __syncthreads();
    }
    const int64_t vid = s_vid;
    const int64_t tile0 = vid * kSortThreads * items;
    // load the tile and count its digits
    uint32_t cnt = 0;
    for (int w = 0; w < kWarps; ++w) wcount[w][t] = 0;
    __syncthreads();
    for (int it = 0; it < items; ++it) {
        const int64_t idx = tile0 + (int64_t)it * kSortThreads + t;
        SK key = 0;
        uint32_t val = 0;
        if (idx < n) {
            key = kin[idx];
            val = vin ? vin[idx] : (uint32_t)idx;
            atomicAdd(&wcount[0][(uint32_t)(key >> shift) & (kRadix - 1)], 1u);
        }
        s_keys[it * kSortThreads + t] = key;
        s_vals[it * kSortThreads + t] = val;
    }
    __syncthreads();
    cnt = wcount[0][t];  // this tile's count of digit t
    uint64_t* my = status + vid * kRadix;
    st_release(&my[t], (vid == 0 ? kFlagInc : kFlagAgg) | cnt);
    // look back for the count of digit t in all earlier tiles
    uint64_t prefix = 0;
    bool timed_out = false;
    if (vid > 0) {
        // walk back 8 tiles per round (independent loads), consuming them in order
        constexpr int kW = 8;
        int64_t q = vid - 1;
        const uint64_t t0 = now_ns();
        bool done = false;
        while (!done && q >= 0) {
            uint64_t st[kW];
#pragma unroll
            for (int u = 0; u < kW; ++u) st[u] = q - u >= 0 ? ld_acquire(&status[(q - u) * kRadix + t]) : 0ull;
            int used = 0;
#pragma unroll
            for (int u = 0; u < kW; ++u) {
                if (done || used < u || q - u < 0) continue;  // stop at the first unpublished tile
                const uint64_t flag = st[u] & ~kCountMask;
                if (flag == kFlagInc) {
                    prefix += st[u] & kCountMask;
                    done = true;
                } else if (flag == kFlagAgg) {
                    prefix += st[u] & kCountMask;
                    used = u + 1;
                }
            }
            q -= used;
            if (!done && used < kW && q >= 0 && now_ns() - t0 > 1000000000ull) {  // 1 s: a tile never published
                timed_out = true;
                break;
            }
        }
        st_release(&my[t], kFlagInc | (prefix + cnt));
    }
    if (timed_out) atomicOr(err, kErrTimeout);
    offs[t] += (uint32_t)prefix;
    __syncthreads();
    // stable scatter, one sub-step of 256 consecutive keys at a time
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int it = 0; it < items; ++it) {
        const int64_t idx = tile0 + (int64_t)it * kSortThreads + t;
        const bool valid = idx < n;
        const SK key = s_keys[it * kSortThreads + t];
        const uint32_t val = s_vals[it * kSortThreads + t];
        const uint32_t d = valid ? (uint32_t)(key >> shift) & (kRadix - 1) : (uint32_t)kRadix;
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
        if (valid && !timed_out) {
            const uint32_t pos = wcount[warp][d] + rank;
            kout[pos] = key;
            vout[pos] = val;
        }
        __syncthreads();
    }
}

// Per 128-row tile of the processing order: the OR of the rows' tap masks, and
// the tile's neighbour lists copied into processing order,
// sorted_nbr[r][k] = nbr[sorted_idx[r]][k] (VG_NONE for padding rows past n).
// Also the tile's region key (Morton bits above F - G of its first row: the
// spatial region its rows were sorted within) and that key's digit counts for
// the tile sort that orders the weight gradient's tiles region by region.
__global__ void __launch_bounds__(kTileRows)
k_tile_rows(const uint32_t* __restrict__ sorted_idx, const uint32_t* __restrict__ nbr,
            const uint32_t* __restrict__ mask, int64_t n, uint32_t* __restrict__ tmask,
            uint32_t* __restrict__ sorted_nbr, const int4* __restrict__ coords, int L, int G, int curve,
            int tile_passes, uint32_t* __restrict__ tkey, uint32_t* __restrict__ thist,
            uint32_t* __restrict__ torder) {
    __shared__ uint32_t rows[kTileRows];
    __shared__ uint32_t w[kTileRows / 32];
    const int64_t r = (int64_t)blockIdx.x * kTileRows + threadIdx.x;
    const uint32_t v = r < n ? sorted_idx[r] : kNone;
    rows[threadIdx.x] = v;
    uint32_t m = v != kNone ? mask[v] : 0u;
    m = __reduce_or_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0) w[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t o = 0;
        for (int i = 0; i < kTileRows / 32; ++i) o |= w[i];
        tmask[blockIdx.x] = o;
        if (tile_passes == 0) {  // no tile sort: the visiting order is the sorted order
            torder[blockIdx.x] = blockIdx.x;
        } else {
            const int F = min(3 * L, kFineOrderBits);
            const uint32_t key = (uint32_t)(curve_code(coords[rows[0]], L, curve) >> (F - G));  // rows[0] < n always
            tkey[blockIdx.x] = key;
            for (int p = 0; p < tile_passes; ++p)
                atomicAdd(&thist[p * kRadix + ((key >> (p * kRadixBits)) & (kRadix - 1))], 1u);
        }
    }
    uint32_t* dst = sorted_nbr + (int64_t)blockIdx.x * kTileRows * kTaps;
    for (int e = threadIdx.x; e < kTileRows * kTaps; e += kTileRows) {
        const int rr = e / kTaps, k = e - rr * kTaps;
        const uint32_t vv = rows[rr];
        dst[e] = vv != kNone ? nbr[(int64_t)vv * kTaps + k] : kNone;
    }
}

// ------------------------------------------------------------------ host side
static int ceil_log2(int64_t v) {
    int b = 0;
    while ((int64_t(1) << b) < v) ++b;
    return b;
}

int nbr_layout(int64_t N, int B, int X, int Y, int Z, unsigned flags, int sms, NbrLayout* L) {
    if (N < 0 || N >= (int64_t(1) << 31) || B <= 0 || X <= 0 || Y <= 0 || Z <= 0) return VG_ERR_INVALID_ARG;
    if ((flags & VG_KEY32) && (flags & VG_KEY64)) return VG_ERR_INVALID_ARG;
    if (flags & ~(VG_KEY32 | VG_KEY64 | VG_ORDER_HILBERT | VG_TEST_SMALL_HASH)) return VG_ERR_INVALID_ARG;
    const double vol = (double)B * X * Y * Z;
    if (vol >= 18446744073709551615.0) return VG_ERR_UNSUPPORTED;
    NbrLayout l;
    l.n = N;
    l.sms = plan_sms(sms);
    l.curve = (flags & VG_ORDER_HILBERT) ? kCurveHilbert : kCurveZOrder;
    if (flags & VG_KEY64) l.key64 = 1;
    else if (flags & VG_KEY32) {
        if (vol > 4294967294.0) return VG_ERR_INVALID_ARG;  // all-ones is the empty-slot marker
        l.key64 = 0;
    } else l.key64 = vol >= 1073741824.0 ? 1 : 0;
    const int lb = ceil_log2(B);
    const int lg = ceil_log2(std::max(X, std::max(Y, Z)));
    // Morton code without its low F - G fine bits, plus the 27-bit valid-tap mask
    const int fine = std::min(3 * lg, kFineOrderBits);
    // G = min(F, 6) fine bits, fewer when that lets the whole key fit 32 bits
    const int coarse = lb + 3 * lg - fine;
    l.fine_keep = std::min(fine, kKeptFineBits);
    if (coarse + kTaps + l.fine_keep > 32 && coarse + kTaps <= 32) l.fine_keep = 32 - kTaps - coarse;
    l.sort_bits = coarse + kTaps + l.fine_keep;
    if (l.sort_bits > 64) return VG_ERR_UNSUPPORTED;
    l.sort64 = l.sort_bits > 32 ? 1 : 0;
    if (flags & VG_TEST_SMALL_HASH) {
        int c = 4;
        while ((int64_t(1) << (c + 1)) <= N / 2) ++c;
        l.cap_log2 = c;
    } else {
        // load <= 1/4 up to 2^21 voxels, where the map build is latency-bound and the
        // longest probe chain sets the insert and probe times (measured: 25k voxels
        // 0.102 -> 0.091 ms); load <= 1/2 above, where the larger table's memset and
        // random reads cost more than the shorter chains save
        const int64_t slots = (N <= (int64_t(1) << 21) ? 4 : 2) * std::max<int64_t>(N, 1);
        l.cap_log2 = std::max(6, ceil_log2(slots));
    }
    if (l.cap_log2 > 31) return VG_ERR_UNSUPPORTED;
    const size_t cap = size_t(1) << l.cap_log2;
    l.num_tiles = (N + kTileRows - 1) / kTileRows;
    // keys per thread in the radix sort: enough blocks to fill the GPU (about
    // 2 per SM), at most 16 keys per thread
    const int64_t per_block_target = std::max<int64_t>(1, N / (2 * (int64_t)l.sms));
    l.sort_items = (int)std::min<int64_t>(16, std::max<int64_t>(1, (per_block_target + kSortThreads - 1) / kSortThreads));
    int64_t tile = (int64_t)kSortThreads * l.sort_items;
    l.sort_blocks = std::max<int64_t>(1, (N + tile - 1) / tile);
    (void)tile;
    const size_t slot = l.key64 ? 16 : 8, ss = l.sort64 ? 8 : 4;
    size_t o = 0;
    l.off_hdr = o;      o += 256;
    l.off_sorted = o;   o += align_up(4 * (size_t)N, 256);
    l.off_tmask = o;    o += align_up(4 * (size_t)l.num_tiles, 256);
    l.off_nbr_sorted = o; o += align_up(4 * (size_t)kTaps * kTileRows * l.num_tiles, 256);
    l.off_torder = o;   o += align_up(4 * (size_t)l.num_tiles, 256);  // offset depends on N only
    l.off_tkey_a = o;   o += align_up(4 * (size_t)l.num_tiles, 256);
    l.off_tkey_b = o;   o += align_up(4 * (size_t)l.num_tiles, 256);
    l.off_torder_b = o; o += align_up(4 * (size_t)l.num_tiles, 256);
    l.off_table = o;    o += align_up(slot * cap, 256);
    l.off_skeys_a = o;  o += align_up(ss * (size_t)N, 256);
    l.off_skeys_b = o;  o += align_up(ss * (size_t)N, 256);
    l.off_svals_b = o;  o += align_up(4 * (size_t)N, 256);
    // one-sweep radix sort: global digit counts of every pass, then per pass the
    // tiles' published counts and a ticket counter (all zeroed by one memset)
    // (the tile region sort's passes follow the row sort's in the same arrays)
    // (up to 2^17 voxels the features of a layer stay in L2 whatever the order:
    // no tile sort, the visiting order is the sorted order)
    const int region_bits = std::min(32, coarse + l.fine_keep);
    l.tile_passes = N <= (int64_t(1) << 17) ? 0 : std::max(1, (region_bits + kRadixBits - 1) / kRadixBits);
    l.tile_blocks = std::max<int64_t>(1, (l.num_tiles + (int64_t)kSortThreads * l.sort_items - 1) /
                                             ((int64_t)kSortThreads * l.sort_items));
    const int passes = std::max(1, (l.sort_bits + kRadixBits - 1) / kRadixBits);
    const int all = passes + l.tile_passes;
    const int64_t sblocks = std::max(l.sort_blocks, l.tile_blocks);
    l.off_hist = o;     o += align_up(4 * (size_t)kRadix * all, 256);
    l.off_status = o;   o += align_up(8 * (size_t)kRadix * sblocks * all, 256);
    l.off_tickets = o;  o += align_up(4 * (size_t)all, 256);
    l.total = o;
    *L = l;
    return VG_OK;
}

int nbr_sort_passes(const NbrLayout& l) { return std::max(1, (l.sort_bits + kRadixBits - 1) / kRadixBits); }

// The row-order half of a build, for any neighbour table nbr [n][27] of the n
// rows whose coordinates are `coords` in a grid with extents < 2^L: tap masks,
// sort keys and their digit counts, the radix passes (sorted_idx), tile masks,
// the map in processing order, and the tiles' visiting order.
template <typename SK>
static void launch_layout(const int4* coords, const NbrLayout& l, int L, char* ws, const uint32_t* nbr,
                          uint32_t* mask, cudaStream_t s) {
    const int64_t n = l.n;
    uint32_t* status = reinterpret_cast<uint32_t*>(ws + l.off_hdr);
    SK* ka = reinterpret_cast<SK*>(ws + l.off_skeys_a);
    SK* kb = reinterpret_cast<SK*>(ws + l.off_skeys_b);
    uint32_t* v0 = reinterpret_cast<uint32_t*>(ws + l.off_sorted);
    uint32_t* v1 = reinterpret_cast<uint32_t*>(ws + l.off_svals_b);
    uint32_t* hist = reinterpret_cast<uint32_t*>(ws + l.off_hist);
    const int passes = nbr_sort_passes(l);
    const unsigned g = (unsigned)l.sort_blocks;
    const int all = passes + l.tile_passes;
    const int64_t sblocks = std::max(l.sort_blocks, l.tile_blocks);
    cudaMemsetAsync(hist, 0, l.off_tickets + 4 * (size_t)all - l.off_hist, s);  // counts, status, tickets
    const int gh_blocks = (int)std::min<int64_t>(l.sort_blocks, 4 * (int64_t)l.sms);
    k_key_globalhist<SK><<<gh_blocks, kSortThreads, 0, s>>>(coords, nbr, n, L, l.fine_keep, l.curve, passes, mask,
                                                            ka, hist);
    const uint32_t* vin = nullptr;
    const size_t smem = (size_t)kSortThreads * l.sort_items * (sizeof(SK) + 4);
    cudaFuncSetAttribute(k_onesweep<SK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    for (int p = 0; p < passes; ++p) {
        const SK* kin = (p % 2 == 0) ? ka : kb;
        SK* kout = (p % 2 == 0) ? kb : ka;
        uint32_t* vout = ((passes - 1 - p) % 2 == 0) ? v0 : v1;
        k_onesweep<SK><<<g, kSortThreads, smem, s>>>(
            kin, vin, kout, vout, n, p * kRadixBits, hist + p * kRadix,
            reinterpret_cast<uint64_t*>(ws + l.off_status) + (size_t)p * kRadix * sblocks,
            reinterpret_cast<uint32_t*>(ws + l.off_tickets) + p, l.sort_items, status);
        vin = vout;
    }
    uint32_t* tka = reinterpret_cast<uint32_t*>(ws + l.off_tkey_a);
    uint32_t* tkb = reinterpret_cast<uint32_t*>(ws + l.off_tkey_b);
    uint32_t* to0 = reinterpret_cast<uint32_t*>(ws + l.off_torder);
    uint32_t* to1 = reinterpret_cast<uint32_t*>(ws + l.off_torder_b);
    k_tile_rows<<<(unsigned)l.num_tiles, kTileRows, 0, s>>>(
        v0, nbr, mask, n, reinterpret_cast<uint32_t*>(ws + l.off_tmask),
        reinterpret_cast<uint32_t*>(ws + l.off_nbr_sorted), coords, L, l.fine_keep, l.curve, l.tile_passes, tka,
        hist + passes * kRadix, to0);
    // stable sort of the tiles by region key: the weight gradient's visiting order
    const size_t tsmem = (size_t)kSortThreads * l.sort_items * (sizeof(uint32_t) + 4);
    cudaFuncSetAttribute(k_onesweep<uint32_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tsmem);
    const uint32_t* tvin = nullptr;
    for (int p = 0; p < l.tile_passes; ++p) {
        const int q = passes + p;
        const uint32_t* kin = (p % 2 == 0) ? tka : tkb;
        uint32_t* kout = (p % 2 == 0) ? tkb : tka;
        uint32_t* vout = ((l.tile_passes - 1 - p) % 2 == 0) ? to0 : to1;
        k_onesweep<uint32_t><<<(unsigned)l.tile_blocks, kSortThreads, tsmem, s>>>(
            kin, tvin, kout, vout, l.num_tiles, p * kRadixBits, hist + q * kRadix,
            reinterpret_cast<uint64_t*>(ws + l.off_status) + (size_t)q * kRadix * sblocks,
            reinterpret_cast<uint32_t*>(ws + l.off_tickets) + q, l.sort_items, status);
        tvin = vout;
    }
}

template <typename K, typename SK>
static void launch_build(const int4* coords, const NbrLayout& l, int B, int X, int Y, int Z, char* ws,
                         uint32_t* nbr, uint32_t* mask, cudaStream_t s) {
    const int64_t n = l.n;
    using T = typename Slot<K>::T;
    T* table = reinterpret_cast<T*>(ws + l.off_table);
    uint32_t* status = reinterpret_cast<uint32_t*>(ws + l.off_hdr);
    const size_t cap = size_t(1) << l.cap_log2;
    cudaMemsetAsync(table, 0xFF, cap * sizeof(T), s);  // empty keys (row fields are don't-care)
    cudaMemsetAsync(nbr, 0xFF, (size_t)n * kTaps * sizeof(uint32_t), s);  // VG_NONE everywhere
    k_insert<K><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(coords, n, B, X, Y, Z, table, l.cap_log2, status);
    k_probe_half<K><<<(unsigned)((n + kProbeVoxels - 1) / kProbeVoxels), kProbeThreads, 0, s>>>(
        coords, n, X, Y, Z, table, l.cap_log2, nbr);
    launch_layout<SK>(coords, l, ceil_log2(std::max(X, std::max(Y, Z))), ws, nbr, mask, s);
}

int nbr_build(const int32_t* coords, int64_t N, int B, int X, int Y, int Z, unsigned flags,
              void* ws_, size_t ws_bytes, uint32_t* nbr, uint32_t* mask, cudaStream_t s) {
    NbrLayout l;
    int st = nbr_layout(N, B, X, Y, Z, flags, 0, &l);
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
        if (l.key64) {
            if (l.sort64) launch_build<uint64_t, uint64_t>(c4, l, B, X, Y, Z, ws, nbr, mask, s);
            else launch_build<uint64_t, uint32_t>(c4, l, B, X, Y, Z, ws, nbr, mask, s);
        } else {
            if (l.sort64) launch_build<uint32_t, uint64_t>(c4, l, B, X, Y, Z, ws, nbr, mask, s);
            else launch_build<uint32_t, uint32_t>(c4, l, B, X, Y, Z, ws, nbr, mask, s);
        }
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
    if (h & kErrTimeout) return VG_ERR_DEVICE_TIMEOUT;
    return VG_OK;
}

// ================================================================== regular (strided / transposed) map
// "Contribution Tasks — JeffreyXiang/FlexGEMM", §二: sparse_conv3d and
// kernels.cuda.spconv sparse_neighbor_map -- a convolution whose output sites
// differ from its input sites.  The map holds the output sites (every cell of
// the strided output grid whose K^3 window holds an input, numbered by linear
// key), down[o][k] (input row at s*o + d_k) and up[j][k] (output row o with
// s*o + d_k = coord_j), and for each side the row order and tiles the GEMM
// kernels read, laid out as a submanifold neighbour-map workspace so that the
// same kernels run on it.
namespace {

constexpr int kScanItems = 16;                          // candidates per thread in the unique pass
constexpr int kScanChunk = kSortThreads * kScanItems;   // candidates per block

__device__ __forceinline__ void tap_delta(int k, int K, int pad, int& dx, int& dy, int& dz) {
    dx = k / (K * K) - pad;
    dy = (k / K) % K - pad;
    dz = k % K - pad;
}

// Output cell of input coordinate v (one axis) through offset d, or -1.
__device__ __forceinline__ int64_t out_cell(int64_t v, int d, int stride, int64_t lim) {
    const int64_t u = v - d;
    if (u < 0 || u % stride != 0) return -1;
    const int64_t o = u / stride;
    return o < lim ? o : -1;
}

// cand[i*T + k] = linear key of the output cell input i reaches through tap k, or
// `sentinel` (the output grid's volume: larger than every key) when there is none.
template <typename CK>
__global__ void __launch_bounds__(256)
k_candidates(const int4* __restrict__ coords, int64_t n, int B, int X, int Y, int Z, int K, int stride, int pad,
             int T, int64_t Xo, int64_t Yo, int64_t Zo, CK sentinel, CK* __restrict__ cand) {
    const int64_t total = n * T;
    for (int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x; e < total; e += (int64_t)gridDim.x * 256) {
        const int64_t i = e / T;
        const int k = (int)(e - i * T);
        const int4 c = coords[i];
        CK key = sentinel;
        if (c.x >= 0 && c.x < B && c.y >= 0 && c.y < X && c.z >= 0 && c.z < Y && c.w >= 0 && c.w < Z) {
            int dx, dy, dz;
            tap_delta(k, K, pad, dx, dy, dz);
            const int64_t ox = out_cell(c.y, dx, stride, Xo), oy = out_cell(c.z, dy, stride, Yo),
                          oz = out_cell(c.w, dz, stride, Zo);
            if (ox >= 0 && oy >= 0 && oz >= 0) key = (CK)((((int64_t)c.x * Xo + ox) * Yo + oy) * Zo + oz);
        }
        cand[e] = key;
    }
}

// Digit counts of every radix pass over n keys.
template <typename CK>
__global__ void __launch_bounds__(kSortThreads)
k_key_hist(const CK* __restrict__ keys, int64_t n, int passes, uint32_t* __restrict__ ghist) {
    __shared__ uint32_t h[kMaxSortPasses][kRadix];
    const int t = threadIdx.x;
    for (int p = 0; p < passes; ++p) h[p][t] = 0;
    __syncthreads();
    for (int64_t i = (int64_t)blockIdx.x * kSortThreads + t; i < n; i += (int64_t)gridDim.x * kSortThreads) {
        const CK key = keys[i];
        for (int p = 0; p < passes; ++p) atomicAdd(&h[p][(uint32_t)(key >> (p * kRadixBits)) & (kRadix - 1)], 1u);
    }
    __syncthreads();
    for (int p = 0; p < passes; ++p)
        if (h[p][t]) atomicAdd(&ghist[p * kRadix + t], h[p][t]);
}

// The first occurrence of each key of the sorted candidates, sentinel excluded.
template <typename CK>
__device__ __forceinline__ bool first_of_run(const CK* keys, int64_t i, CK sentinel) {
    const CK k = keys[i];
    return k != sentinel && (i == 0 || keys[i - 1] != k);
}

// Block b counts the distinct keys starting in its chunk of kScanChunk candidates.
template <typename CK>
__global__ void __launch_bounds__(kSortThreads)
k_unique_count(const CK* __restrict__ keys, int64_t n, CK sentinel, uint32_t* __restrict__ counts) {
    __shared__ uint32_t red[kSortThreads / 32];
    const int64_t base = (int64_t)blockIdx.x * kScanChunk + (int64_t)threadIdx.x * kScanItems;
    uint32_t c = 0;
    for (int q = 0; q < kScanItems; ++q)
        if (base + q < n && first_of_run(keys, base + q, sentinel)) ++c;
    c = __reduce_add_sync(0xffffffffu, c);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int w = 0; w < kSortThreads / 32; ++w) t += red[w];
        counts[blockIdx.x] = t;
    }
}

// Exclusive scan of the block counts in place (one block); the total is the
// number of output sites, stored as int64 at n_out.
__global__ void __launch_bounds__(1024) k_unique_scan(uint32_t* __restrict__ counts, int64_t nb, int64_t* n_out) {
    __shared__ uint32_t warp_tot[32];
    __shared__ uint64_t carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t b0 = 0; b0 < nb; b0 += 1024) {
        const int64_t i = b0 + threadIdx.x;
        const uint32_t v = i < nb ? counts[i] : 0u;
        uint32_t inc = v;
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) warp_tot[warp] = inc;
        __syncthreads();
        uint32_t before = 0;
        for (int w = 0; w < warp; ++w) before += warp_tot[w];
        if (i < nb) counts[i] = (uint32_t)(carry + before + inc - v);
        __syncthreads();
        if (threadIdx.x == 1023) carry += before + inc;
        __syncthreads();
    }
    if (threadIdx.x == 0) *n_out = (int64_t)carry;
}

// uniq[offset of block + rank] = each first-of-run key, in order.
template <typename CK>
__global__ void __launch_bounds__(kSortThreads)
k_unique_write(const CK* __restrict__ keys, int64_t n, CK sentinel, const uint32_t* __restrict__ offsets,
               CK* __restrict__ uniq) {
    __shared__ uint32_t warp_tot[kSortThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t base = (int64_t)blockIdx.x * kScanChunk + (int64_t)threadIdx.x * kScanItems;
    uint32_t c = 0;
    for (int q = 0; q < kScanItems; ++q)
        if (base + q < n && first_of_run(keys, base + q, sentinel)) ++c;
    uint32_t inc = c;
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    uint32_t pos = offsets[blockIdx.x] + inc - c;
    for (int w = 0; w < warp; ++w) pos += warp_tot[w];
    for (int q = 0; q < kScanItems; ++q)
        if (base + q < n && first_of_run(keys, base + q, sentinel)) uniq[pos++] = keys[base + q];
}

template <typename CK>
__global__ void __launch_bounds__(256)
k_decode_out(const CK* __restrict__ uniq, const int64_t* __restrict__ n_out, int64_t Xo, int64_t Yo, int64_t Zo,
             int4* __restrict__ coords_out) {
    const int64_t n = *n_out;
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
        uint64_t key = (uint64_t)uniq[i];
        const int z = (int)(key % Zo);
        key /= Zo;
        const int y = (int)(key % Yo);
        key /= Yo;
        const int x = (int)(key % Xo);
        coords_out[i] = make_int4((int)(key / Xo), x, y, z);
    }
}

// Row of `key` in an open-addressing table, or VG_NONE.
template <typename K>
__device__ __forceinline__ uint32_t hash_find(const typename Slot<K>::T* __restrict__ table, int cap_log2, K key) {
    const uint32_t cmask = (1u << cap_log2) - 1u;
    const K empty = ~K(0);
    uint32_t slot = start_slot(key, cap_log2);
    for (uint32_t p = 0; p <= cmask; ++p) {
        const typename Slot<K>::T e = table[slot];
        if ((K)e.x == key) return (uint32_t)e.y;
        if ((K)e.x == empty) return kNone;
        slot = (slot + 1u) & cmask;
    }
    return kNone;
}

// down[o][k] = input row at s*o + d_k (k < T); one thread per (o, k).
template <typename K>
__global__ void __launch_bounds__(256)
k_probe_down(const int4* __restrict__ coords_out, int64_t n_out, int X, int Y, int Z, int K_, int stride, int pad,
             int T, const typename Slot<K>::T* __restrict__ table_in, int cap_log2, uint32_t* __restrict__ down) {
    const int64_t total = n_out * T;
    for (int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x; e < total; e += (int64_t)gridDim.x * 256) {
        const int64_t o = e / T;
        const int k = (int)(e - o * T);
        const int4 c = coords_out[o];
        int dx, dy, dz;
        tap_delta(k, K_, pad, dx, dy, dz);
        const int64_t x = (int64_t)stride * c.y + dx, y = (int64_t)stride * c.z + dy, z = (int64_t)stride * c.w + dz;
        if (x < 0 || x >= X || y < 0 || y >= Y || z < 0 || z >= Z) continue;
        down[o * kTaps + k] = hash_find<K>(table_in, cap_log2, (K)((((int64_t)c.x * X + x) * Y + y) * Z + z));
    }
}

// up[j][k] = output row o with s*o + d_k = coord_j (k < T); one thread per (j, k).
template <typename K>
__global__ void __launch_bounds__(256)
k_probe_up(const int4* __restrict__ coords, int64_t n, int64_t Xo, int64_t Yo, int64_t Zo, int K_, int stride,
           int pad, int T, const typename Slot<K>::T* __restrict__ table_out, int cap_log2,
           uint32_t* __restrict__ up) {
    const int64_t total = n * T;
    for (int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x; e < total; e += (int64_t)gridDim.x * 256) {
        const int64_t j = e / T;
        const int k = (int)(e - j * T);
        const int4 c = coords[j];
        int dx, dy, dz;
        tap_delta(k, K_, pad, dx, dy, dz);
        const int64_t ox = out_cell(c.y, dx, stride, Xo), oy = out_cell(c.z, dy, stride, Yo),
                      oz = out_cell(c.w, dz, stride, Zo);
        if (ox < 0 || oy < 0 || oz < 0) continue;
        up[j * kTaps + k] = hash_find<K>(table_out, cap_log2, (K)((((int64_t)c.x * Xo + ox) * Yo + oy) * Zo + oz));
    }
}

// Every side's status word becomes the OR of all three (the whole map is good or bad).
__global__ void k_merge_status(uint32_t* a, uint32_t* b, uint32_t* c) {
    const uint32_t v = *a | *b | *c;
    *a = v;
    *b = v;
    *c = v;
}

}  // namespace

int sparse_layout(int64_t N, int B, int X, int Y, int Z, int K, int stride, unsigned flags, int sms,
                  int64_t n_out, SparseLayout* S) {
    if (N < 0 || N >= (int64_t(1) << 31) || B <= 0 || X <= 0 || Y <= 0 || Z <= 0) return VG_ERR_INVALID_ARG;
    if ((K != 2 && K != 3) || (stride != 1 && stride != 2)) return VG_ERR_INVALID_ARG;
    if (flags & ~VG_ORDER_HILBERT) return VG_ERR_INVALID_ARG;
    SparseLayout l;
    l.n_in = N;
    l.K = K;
    l.stride = stride;
    l.pad = K == 3 ? 1 : 0;
    l.T = K * K * K;
    l.B = B; l.X = X; l.Y = Y; l.Z = Z;
    if (X + 2 * l.pad < K || Y + 2 * l.pad < K || Z + 2 * l.pad < K) return VG_ERR_INVALID_ARG;
    l.Xo = (X + 2 * l.pad - K) / stride + 1;
    l.Yo = (Y + 2 * l.pad - K) / stride + 1;
    l.Zo = (Z + 2 * l.pad - K) / stride + 1;
    l.flags = flags;
    const double vol_out = (double)B * l.Xo * l.Yo * l.Zo;
    if (vol_out >= 9.0e18) return VG_ERR_UNSUPPORTED;
    l.sentinel = (uint64_t)B * l.Xo * l.Yo * l.Zo;
    l.cap_out = std::min<int64_t>(N * l.T, (int64_t)std::min(vol_out, 2147483647.0));
    l.cap_out = std::min<int64_t>(l.cap_out, (int64_t(1) << 31) - 1);
    const int sms_ = plan_sms(sms);
    int st = nbr_layout(N, B, X, Y, Z, flags, sms_, &l.li);
    if (st != VG_OK) return st;
    st = nbr_layout(l.cap_out, B, l.Xo, l.Yo, l.Zo, flags, sms_, &l.lo_cap);
    if (st != VG_OK) return st;
    if (n_out >= 0) {  // the output side as laid out for the actual number of output sites
        if (n_out > l.cap_out) return VG_ERR_INVALID_ARG;
        st = nbr_layout(n_out, B, l.Xo, l.Yo, l.Zo, flags, sms_, &l.lo);
        if (st != VG_OK) return st;
    }
    l.n_out = n_out;
    l.cand64 = l.sentinel >= 0xFFFFFFFFull ? 1 : 0;
    int bits = 0;
    while (bits < 64 && (l.sentinel >> bits) != 0) ++bits;
    l.cand_passes = std::max(1, (bits + kRadixBits - 1) / kRadixBits);
    l.cand_n = N * l.T;
    const int64_t per_block_target = std::max<int64_t>(1, l.cand_n / (2 * (int64_t)sms_));
    l.cand_items = (int)std::min<int64_t>(16, std::max<int64_t>(1, (per_block_target + kSortThreads - 1) / kSortThreads));
    l.cand_blocks = std::max<int64_t>(1, (l.cand_n + (int64_t)kSortThreads * l.cand_items - 1) /
                                             ((int64_t)kSortThreads * l.cand_items));
    l.scan_blocks = std::max<int64_t>(1, (l.cand_n + kScanChunk - 1) / kScanChunk);
    const size_t ck = l.cand64 ? 8 : 4;
    size_t o = 0;
    l.off_hdr = o;          o += 256;
    l.off_side_i = o;       o += align_up(l.li.total, 256);
    // the output side is laid out for the actual count later; its sort-scratch block
    // count is not monotone in the row count, so leave room for the largest
    l.side_o_bytes = align_up(l.lo_cap.total + 8 * (size_t)kRadix * (2 * (size_t)sms_ + 2) * (kMaxSortPasses + 4), 256);
    l.off_side_o = o;       o += l.side_o_bytes;
    l.off_nbr_down = o;     o += align_up(4 * (size_t)kTaps * l.cap_out, 256);
    l.off_mask_down = o;    o += align_up(4 * (size_t)l.cap_out, 256);
    l.off_nbr_up = o;       o += align_up(4 * (size_t)kTaps * N, 256);
    l.off_mask_up = o;      o += align_up(4 * (size_t)N, 256);
    l.off_coords_out = o;   o += align_up(16 * (size_t)l.cap_out, 256);
    l.off_cand_a = o;       o += align_up(ck * l.cand_n, 256);
    l.off_cand_b = o;       o += align_up(ck * l.cand_n, 256);
    l.off_cand_va = o;      o += align_up(4 * (size_t)l.cand_n, 256);
    l.off_cand_vb = o;      o += align_up(4 * (size_t)l.cand_n, 256);
    l.off_cand_hist = o;    o += align_up(4 * (size_t)kRadix * l.cand_passes, 256);
    l.off_cand_status = o;  o += align_up(8 * (size_t)kRadix * l.cand_blocks * l.cand_passes, 256);
    l.off_cand_tickets = o; o += align_up(4 * (size_t)l.cand_passes, 256);
    l.off_scan = o;         o += align_up(4 * (size_t)l.scan_blocks, 256);
    l.total = o;
    *S = l;
    return VG_OK;
}

template <typename K>
static void insert_sites(const int4* coords, int64_t n, int B, int X, int Y, int Z, const NbrLayout& l, char* side,
                         cudaStream_t s) {
    using T = typename Slot<K>::T;
    T* table = reinterpret_cast<T*>(side + l.off_table);
    cudaMemsetAsync(table, 0xFF, (size_t(1) << l.cap_log2) * sizeof(T), s);
    if (n > 0)
        k_insert<K><<<(unsigned)((n + 255) / 256), 256, 0, s>>>(coords, n, B, X, Y, Z, table, l.cap_log2,
                                                                reinterpret_cast<uint32_t*>(side + l.off_hdr));
}

template <typename CK>
static void sparse_front(const int4* coords, const SparseLayout& l, char* ws, cudaStream_t s) {
    uint32_t* status = reinterpret_cast<uint32_t*>(ws + l.off_hdr);
    CK* ca = reinterpret_cast<CK*>(ws + l.off_cand_a);
    CK* cb = reinterpret_cast<CK*>(ws + l.off_cand_b);
    uint32_t* va = reinterpret_cast<uint32_t*>(ws + l.off_cand_va);
    uint32_t* vb = reinterpret_cast<uint32_t*>(ws + l.off_cand_vb);
    uint32_t* hist = reinterpret_cast<uint32_t*>(ws + l.off_cand_hist);
    const int sms = l.li.sms;
    const unsigned gblocks = (unsigned)std::min<int64_t>((l.cand_n + 255) / 256, 16 * (int64_t)sms);
    k_candidates<CK><<<gblocks, 256, 0, s>>>(coords, l.n_in, l.B, l.X, l.Y, l.Z, l.K, l.stride, l.pad, l.T, l.Xo,
                                             l.Yo, l.Zo, (CK)l.sentinel, ca);
    cudaMemsetAsync(hist, 0, l.off_scan - l.off_cand_hist, s);  // counts, look-back status, tickets
    k_key_hist<CK><<<(unsigned)std::min<int64_t>(l.cand_blocks, 4 * (int64_t)sms), kSortThreads, 0, s>>>(
        ca, l.cand_n, l.cand_passes, hist);
    const size_t smem = (size_t)kSortThreads * l.cand_items * (sizeof(CK) + 4);
    cudaFuncSetAttribute(k_onesweep<CK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const uint32_t* vin = nullptr;
    for (int p = 0; p < l.cand_passes; ++p) {
        const CK* kin = (p % 2 == 0) ? ca : cb;
        CK* kout = (p % 2 == 0) ? cb : ca;
        uint32_t* vout = (p % 2 == 0) ? va : vb;
        k_onesweep<CK><<<(unsigned)l.cand_blocks, kSortThreads, smem, s>>>(
            kin, vin, kout, vout, l.cand_n, p * kRadixBits, hist + p * kRadix,
            reinterpret_cast<uint64_t*>(ws + l.off_cand_status) + (size_t)p * kRadix * l.cand_blocks,
            reinterpret_cast<uint32_t*>(ws + l.off_cand_tickets) + p, l.cand_items, status);
        vin = vout;
    }
    const CK* sorted = (l.cand_passes % 2 == 1) ? cb : ca;
    CK* uniq = (l.cand_passes % 2 == 1) ? ca : cb;
    uint32_t* counts = reinterpret_cast<uint32_t*>(ws + l.off_scan);
    int64_t* n_out = reinterpret_cast<int64_t*>(ws + l.off_hdr + 8);
    k_unique_count<CK><<<(unsigned)l.scan_blocks, kSortThreads, 0, s>>>(sorted, l.cand_n, (CK)l.sentinel, counts);
    k_unique_scan<<<1, 1024, 0, s>>>(counts, l.scan_blocks, n_out);
    k_unique_write<CK><<<(unsigned)l.scan_blocks, kSortThreads, 0, s>>>(sorted, l.cand_n, (CK)l.sentinel, counts,
                                                                       uniq);
    k_decode_out<CK><<<(unsigned)std::min<int64_t>((l.cap_out + 255) / 256, 16 * (int64_t)sms), 256, 0, s>>>(
        uniq, n_out, l.Xo, l.Yo, l.Zo, reinterpret_cast<int4*>(ws + l.off_coords_out));
}

template <typename KI, typename KO>
static void sparse_probes(const int4* coords, const SparseLayout& l, char* ws, cudaStream_t s) {
    char* side_i = ws + l.off_side_i;
    char* side_o = ws + l.off_side_o;
    const int4* cout_ = reinterpret_cast<const int4*>(ws + l.off_coords_out);
    uint32_t* down = reinterpret_cast<uint32_t*>(ws + l.off_nbr_down);
    uint32_t* up = reinterpret_cast<uint32_t*>(ws + l.off_nbr_up);
    const int sms = l.li.sms;
    insert_sites<KO>(cout_, l.n_out, l.B, (int)l.Xo, (int)l.Yo, (int)l.Zo, l.lo, side_o, s);
    cudaMemsetAsync(down, 0xFF, 4 * (size_t)kTaps * l.n_out, s);
    cudaMemsetAsync(up, 0xFF, 4 * (size_t)kTaps * l.n_in, s);
    if (l.n_out > 0)
        k_probe_down<KI><<<(unsigned)std::min<int64_t>((l.n_out * l.T + 255) / 256, 16 * (int64_t)sms), 256, 0, s>>>(
            cout_, l.n_out, l.X, l.Y, l.Z, l.K, l.stride, l.pad, l.T,
            reinterpret_cast<const typename Slot<KI>::T*>(side_i + l.li.off_table), l.li.cap_log2, down);
    k_probe_up<KO><<<(unsigned)std::min<int64_t>((l.n_in * l.T + 255) / 256, 16 * (int64_t)sms), 256, 0, s>>>(
        coords, l.n_in, l.Xo, l.Yo, l.Zo, l.K, l.stride, l.pad, l.T,
        reinterpret_cast<const typename Slot<KO>::T*>(side_o + l.lo.off_table), l.lo.cap_log2, up);
}

template <typename SK>
static void layout_side(const int4* coords, const NbrLayout& l, int X, int Y, int Z, char* side, const uint32_t* nbr,
                        uint32_t* mask, cudaStream_t s) {
    if (l.n > 0) launch_layout<SK>(coords, l, ceil_log2(std::max(X, std::max(Y, Z))), side, nbr, mask, s);
}

int sparse_build(const int32_t* coords, int64_t N, int B, int X, int Y, int Z, int K, int stride, unsigned flags,
                 void* ws_, size_t ws_bytes, int64_t* n_out_host, cudaStream_t s) {
    SparseLayout l;
    int st = sparse_layout(N, B, X, Y, Z, K, stride, flags, 0, -1, &l);
    if (st != VG_OK) return st;
    if (!ws_ || (reinterpret_cast<uintptr_t>(ws_) & 255) || !n_out_host) return VG_ERR_INVALID_ARG;
    if (ws_bytes < l.total) return VG_ERR_WORKSPACE_TOO_SMALL;
    if (N > 0 && (!coords || (reinterpret_cast<uintptr_t>(coords) & 15))) return VG_ERR_INVALID_ARG;
    char* ws = static_cast<char*>(ws_);
    char* side_i = ws + l.off_side_i;
    char* side_o = ws + l.off_side_o;
    cudaGetLastError();
    cudaMemsetAsync(ws + l.off_hdr, 0, 256, s);
    cudaMemsetAsync(side_i + l.li.off_hdr, 0, 256, s);
    cudaMemsetAsync(side_o + l.lo_cap.off_hdr, 0, 256, s);
    *n_out_host = 0;
    if (N == 0) return cudaStreamSynchronize(s) == cudaSuccess && cudaGetLastError() == cudaSuccess ? VG_OK : VG_ERR_CUDA;
    const int4* c4 = reinterpret_cast<const int4*>(coords);
    // phase 1: input sites into their hash table (range and duplicate checks), output sites
    if (l.li.key64) insert_sites<uint64_t>(c4, N, B, X, Y, Z, l.li, side_i, s);
    else insert_sites<uint32_t>(c4, N, B, X, Y, Z, l.li, side_i, s);
    if (l.cand64) sparse_front<uint64_t>(c4, l, ws, s);
    else sparse_front<uint32_t>(c4, l, ws, s);
    int64_t n_out = 0;
    uint32_t st_in = 0, st_hdr = 0;
    if (cudaMemcpyAsync(&n_out, ws + l.off_hdr + 8, 8, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(&st_in, side_i + l.li.off_hdr, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(&st_hdr, ws + l.off_hdr, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return VG_ERR_CUDA;
    const uint32_t early = st_in | st_hdr;
    if (early) {  // record the error in every side so that convolutions on this map write nothing
        k_merge_status<<<1, 1, 0, s>>>(reinterpret_cast<uint32_t*>(ws + l.off_hdr),
                                      reinterpret_cast<uint32_t*>(side_i + l.li.off_hdr),
                                      reinterpret_cast<uint32_t*>(side_o + l.lo_cap.off_hdr));
        cudaStreamSynchronize(s);
        if (early & kErrRange) return VG_ERR_COORD_OUT_OF_RANGE;
        if (early & kErrDup) return VG_ERR_DUPLICATE_COORD;
        if (early & kErrFull) return VG_ERR_HASH_FULL;
        return VG_ERR_DEVICE_TIMEOUT;
    }
    // phase 2: with the number of output sites known, the output hash, both maps and both row orders
    st = sparse_layout(N, B, X, Y, Z, K, stride, flags, 0, n_out, &l);
    if (st != VG_OK) return st;
    if (l.lo.total > l.side_o_bytes) return VG_ERR_UNSUPPORTED;
    if (l.li.key64) {
        if (l.lo.key64) sparse_probes<uint64_t, uint64_t>(c4, l, ws, s);
        else sparse_probes<uint64_t, uint32_t>(c4, l, ws, s);
    } else {
        if (l.lo.key64) sparse_probes<uint32_t, uint64_t>(c4, l, ws, s);
        else sparse_probes<uint32_t, uint32_t>(c4, l, ws, s);
    }
    const int4* cout_ = reinterpret_cast<const int4*>(ws + l.off_coords_out);
    uint32_t* down = reinterpret_cast<uint32_t*>(ws + l.off_nbr_down);
    uint32_t* up = reinterpret_cast<uint32_t*>(ws + l.off_nbr_up);
    uint32_t* mdown = reinterpret_cast<uint32_t*>(ws + l.off_mask_down);
    uint32_t* mup = reinterpret_cast<uint32_t*>(ws + l.off_mask_up);
    if (l.lo.sort64) layout_side<uint64_t>(cout_, l.lo, (int)l.Xo, (int)l.Yo, (int)l.Zo, side_o, down, mdown, s);
    else layout_side<uint32_t>(cout_, l.lo, (int)l.Xo, (int)l.Yo, (int)l.Zo, side_o, down, mdown, s);
    if (l.li.sort64) layout_side<uint64_t>(c4, l.li, X, Y, Z, side_i, up, mup, s);
    else layout_side<uint32_t>(c4, l.li, X, Y, Z, side_i, up, mup, s);
    k_merge_status<<<1, 1, 0, s>>>(reinterpret_cast<uint32_t*>(ws + l.off_hdr),
                                  reinterpret_cast<uint32_t*>(side_i + l.li.off_hdr),
                                  reinterpret_cast<uint32_t*>(side_o + l.lo.off_hdr));
    uint32_t h = 0;
    if (cudaMemcpyAsync(&h, ws + l.off_hdr, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess || cudaGetLastError() != cudaSuccess)
        return VG_ERR_CUDA;
    *n_out_host = n_out;
    if (h & kErrFull) return VG_ERR_HASH_FULL;
    if (h & kErrTimeout) return VG_ERR_DEVICE_TIMEOUT;
    if (h) return VG_ERR_INVALID_ARG;
    return VG_OK;
}

}  // namespace vg
