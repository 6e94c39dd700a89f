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

// Published partial results of the single-pass scans below: flag bits 62-63
// (1 this block's own count, 2 inclusive prefix) over a 62-bit count.
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

// ------------------------------------------------------------------ column index
// Where the grid has few (b, x, y) columns for its voxels, the map is built
// without a hash table.  Column c = (b*X + x)*Y + y of a voxel:
//   cnt[c]    voxels in column c (k_col_count, which also validates coordinates)
//   start[c]  exclusive prefix sum of cnt, start[C] = number of valid voxels (k_col_scan)
//   ent[start[c] .. start[c+1])  the column's voxels as {z, row}, ascending z,
//             with col[] holding c beside each entry and pos[row] the entry's
//             index (k_col_scatter in arrival order, then k_col_rank)
// The probe (k_col_probe) walks the entries in that column order and searches
// each voxel's 9 neighbouring columns for z - 1, z, z + 1: the threads of a warp
// hold voxels of one or a few adjacent columns, so their lookups share cache
// lines.  It writes each neighbour row with its mask as a 128-byte record in
// column order (whole cache lines); k_col_emit then moves the records to the
// caller's order (nbr, mask, sort keys) with one line read per row.  Scattering
// 4-byte neighbour entries straight
// into the caller's order was measured 1.7 ms slower at 4.9 M voxels: the GPU's
// L2 handles each partial-sector write as its own request.
__device__ __forceinline__ bool in_grid(int4 c, int B, int X, int Y, int Z) {
    return c.x >= 0 && c.x < B && c.y >= 0 && c.y < X && c.z >= 0 && c.z < Y && c.w >= 0 && c.w < Z;
}

__global__ void __launch_bounds__(256)
k_col_count(const int4* __restrict__ coords, int64_t n, int B, int X, int Y, int Z, uint32_t* __restrict__ cnt,
            uint32_t* __restrict__ arrival, uint32_t* __restrict__ status) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int4 c = coords[i];
    if (!in_grid(c, B, X, Y, Z)) {
        atomicOr(status, kErrRange);
        return;
    }
    arrival[i] = atomicAdd(&cnt[((int64_t)c.x * X + c.y) * Y + c.z], 1u);
}

// start[j] = cnt[0] + ... + cnt[j-1] for j < m, in one pass: each block takes the
// next chunk of 4096 counts (ticket order), publishes its sum, and one thread
// looks back over the earlier chunks' published sums (flag bits 62-63 as in the
// radix sort: 1 chunk sum, 2 inclusive prefix).  The wait is bounded; giving up
// marks the map bad (and the readers clamp every position to [0, n]).
constexpr int kColScanItems = 16;
constexpr int kColScanChunk = kSortThreads * kColScanItems;
// shared-memory slot of chunk element p: one pad word per 32 (conflict-free both
// when a warp reads 32 consecutive elements and when each thread reads its own 16)
__device__ __forceinline__ int col_pad(int p) { return p + (p >> 5); }

__global__ void __launch_bounds__(kSortThreads)
k_col_scan(const uint32_t* __restrict__ cnt, int64_t m, uint32_t* __restrict__ start, uint64_t* __restrict__ part,
           uint32_t* __restrict__ ticket, uint32_t* __restrict__ err) {
    __shared__ uint32_t sv[kColScanChunk + kColScanChunk / 32];
    __shared__ uint32_t wsum[kSortThreads / 32];
    __shared__ uint32_t s_vid;
    __shared__ uint32_t s_prefix;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    if (t == 0) s_vid = atomicAdd(ticket, 1u);
    __syncthreads();
    const int64_t vid = s_vid;
    const int64_t base = vid * kColScanChunk;
    for (int j = 0; j < kColScanItems; ++j) {
        const int64_t idx = base + (int64_t)j * kSortThreads + t;
        sv[col_pad(j * kSortThreads + t)] = idx < m ? cnt[idx] : 0u;
    }
    __syncthreads();
    uint32_t v[kColScanItems], sum = 0;
#pragma unroll
    for (int j = 0; j < kColScanItems; ++j) {
        v[j] = sv[col_pad(t * kColScanItems + j)];
        sum += v[j];
    }
    uint32_t inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    uint32_t before = inc - sum, total = 0;
    for (int w = 0; w < kSortThreads / 32; ++w) {
        if (w < warp) before += wsum[w];
        total += wsum[w];
    }
    if (t == 0) {
        uint64_t prefix = 0;
        if (vid == 0) {
            st_release(&part[0], kFlagInc | total);
        } else {
            st_release(&part[vid], kFlagAgg | total);
            int64_t q = vid - 1;
            const uint64_t t0 = now_ns();
            while (q >= 0) {
                const uint64_t st = ld_acquire(&part[q]);
                const uint64_t flag = st & ~kCountMask;
                if (flag == kFlagInc) {
                    prefix += st & kCountMask;
                    break;
                }
                if (flag == kFlagAgg) {
                    prefix += st & kCountMask;
                    --q;
                    continue;
                }
                if (now_ns() - t0 > 1000000000ull) {  // 1 s: a chunk never published
                    atomicOr(err, kErrTimeout);
                    break;
                }
            }
            st_release(&part[vid], kFlagInc | (prefix + total));
        }
        s_prefix = (uint32_t)prefix;
    }
    __syncthreads();
    uint32_t run = s_prefix + before;
#pragma unroll
    for (int j = 0; j < kColScanItems; ++j) {
        sv[col_pad(t * kColScanItems + j)] = run;
        run += v[j];
    }
    __syncthreads();
    for (int j = 0; j < kColScanItems; ++j) {
        const int64_t idx = base + (int64_t)j * kSortThreads + t;
        if (idx < m) start[idx] = sv[col_pad(j * kSortThreads + t)];
    }
}

// Column range [s, e) of column col, clamped to [0, n] (a scan that gave up
// leaves the starts undefined; the map is then flagged bad, but no access may leave the arrays).
__device__ __forceinline__ void col_range(const uint32_t* __restrict__ start, int64_t col, int64_t n, uint32_t& s,
                                          uint32_t& e) {
    s = min((uint32_t)n, start[col]);
    e = max(s, min((uint32_t)n, start[col + 1]));
}

__global__ void __launch_bounds__(256)
k_col_scatter(const int4* __restrict__ coords, int64_t n, int B, int X, int Y, int Z,
              const uint32_t* __restrict__ start, const uint32_t* __restrict__ arrival, uint2* __restrict__ ent,
              uint32_t* __restrict__ ecol) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int4 c = coords[i];
    if (!in_grid(c, B, X, Y, Z)) return;
    const int64_t col = ((int64_t)c.x * X + c.y) * Y + c.z;
    const uint64_t pos = (uint64_t)start[col] + arrival[i];
    if (pos < (uint64_t)n) {
        ent[pos] = make_uint2((uint32_t)c.w, (uint32_t)i);
        ecol[pos] = (uint32_t)col;
    }
}

// Entries in column order: j < start[C] (clamped to n).  A column id read from
// an entry is checked against C before it indexes anything.
__device__ __forceinline__ int64_t col_entries(const uint32_t* __restrict__ start, int64_t ncols, int64_t n) {
    return min((int64_t)start[ncols], n);
}

// Final slot of entry j in its column: the number of the column's entries with a
// smaller z, or the same z and a smaller row (slots stay distinct even with
// duplicates, which are reported).  One thread per entry, in column order.
__global__ void __launch_bounds__(256)
k_col_rank(const uint32_t* __restrict__ start, int64_t ncols, int64_t n, const uint2* __restrict__ ent_in,
           const uint32_t* __restrict__ col_in, uint2* __restrict__ ent_out, uint32_t* __restrict__ col_out,
           uint32_t* __restrict__ pos, uint32_t* __restrict__ status) {
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= col_entries(start, ncols, n)) return;
    const uint2 q = ent_in[j];
    const uint32_t col = col_in[j];
    if (col >= (uint64_t)ncols) return;
    uint32_t s, e;
    col_range(start, col, n, s, e);
    uint32_t r = 0;
    bool dup = false;
    for (uint32_t p = s; p < e; ++p) {
        const uint2 o = ent_in[p];
        r += (o.x < q.x || (o.x == q.x && o.y < q.y)) ? 1u : 0u;
        dup |= o.x == q.x && o.y != q.y;
    }
    if (dup) atomicOr(status, kErrDup);
    if (s + r < e) {
        ent_out[s + r] = q;
        col_out[s + r] = col;
        if (q.y < (uint64_t)n) pos[q.y] = s + r;
    }
}

// The 27-tap probe over the column index, one thread per entry in column order:
// for the voxel (b, x, y, z) of entry j, each of the columns (x + dx, y + dy)
// inside the grid is searched for z - 1, z, z + 1 (a scan of a short column, a
// binary search for z - 1 in a long one, then at most three entries).  The block
// stages its 256 records (27 neighbour rows + the valid-tap mask) in shared
// memory (stride 29: conflict-free) and writes them to rec[j][0..27] as one run.
constexpr int kShortColumn = 8;
// 27 neighbour rows + mask + 4 padding words: one 128-byte line per record
// (measured: 112-byte records cost 0.19 ms more at 4.9 M voxels, most of them
// straddling two lines)
constexpr int kRecWords = 32;
constexpr int kRecStride = 29;

__global__ void __launch_bounds__(256)
k_col_probe(const uint32_t* __restrict__ start, int64_t ncols, int64_t n, int X, int Y,
            const uint2* __restrict__ ent, const uint32_t* __restrict__ ecol, uint32_t* __restrict__ rec) {
    __shared__ uint32_t srec[256 * kRecStride];
    const int t = threadIdx.x;
    const int64_t total = col_entries(start, ncols, n);
    const int64_t j0 = (int64_t)blockIdx.x * 256;
    if (j0 >= total) return;  // whole block
    const int64_t j = j0 + t;
    uint32_t* my = srec + t * kRecStride;
    if (j < total) {
        const uint2 q = ent[j];
        const uint32_t col = ecol[j];
        uint32_t m = 0;
        const bool ok = col < (uint64_t)ncols;
        const uint32_t bx = ok ? col / (uint32_t)Y : 0u;
        const int y = (int)(col - bx * (uint32_t)Y);
        const int x = (int)(bx % (uint32_t)X);
        const int z = (int)q.x;
#pragma unroll
        for (int dx = -1; dx <= 1; ++dx) {
#pragma unroll
            for (int dy = -1; dy <= 1; ++dy) {
                const int k0 = (dx + 1) * 9 + (dy + 1) * 3;  // tap of dz = -1
                uint32_t v0 = kNone, v1 = kNone, v2 = kNone;
                if (ok && x + dx >= 0 && x + dx < X && y + dy >= 0 && y + dy < Y) {
                    uint32_t s, e;
                    col_range(start, (int64_t)col + (int64_t)dx * Y + dy, n, s, e);
                    if (e - s > kShortColumn) {  // first entry with z' >= z - 1
                        uint32_t lo = s, hi = e;
                        while (lo < hi) {
                            const uint32_t mid = (lo + hi) >> 1;
                            if ((int)ent[mid].x < z - 1) lo = mid + 1;
                            else hi = mid;
                        }
                        s = lo;
                    }
                    for (uint32_t p = s; p < e; ++p) {
                        const uint2 o = ent[p];
                        const int d = (int)o.x - z;
                        if (d > 1) break;
                        if (d == -1) v0 = o.y;
                        else if (d == 0) v1 = o.y;
                        else if (d == 1) v2 = o.y;
                    }
                }
                my[k0] = v0;
                my[k0 + 1] = v1;
                my[k0 + 2] = v2;
                m |= (v0 != kNone ? 1u : 0u) << k0 | (v1 != kNone ? 2u : 0u) << k0 | (v2 != kNone ? 4u : 0u) << k0;
            }
        }
        my[kTaps] = m;
    }
    __syncthreads();
    const int64_t words = (total - j0 < 256 ? total - j0 : (int64_t)256) * kRecWords;
    uint32_t* out = rec + j0 * kRecWords;
    for (int64_t w = t; w < words; w += 256) {
        const int r = (int)(w / kRecWords), k = (int)(w - (int64_t)r * kRecWords);
        out[w] = k <= kTaps ? srec[r * kRecStride + k] : 0u;  // words past the mask: padding
    }
}

// Record of voxel i for the caller-order passes: rec + pos[i] * 28, or null when
// the voxel has none (outside the grid, or a build that gave up).
__device__ __forceinline__ const uint32_t* col_record(const uint32_t* __restrict__ rec,
                                                      const uint32_t* __restrict__ pos, int64_t total, uint32_t i,
                                                      bool valid) {
    if (!valid) return nullptr;
    const uint32_t p = pos[i];
    return p < (uint64_t)total ? rec + (int64_t)p * kRecWords : nullptr;
}

// Copies the first 28 words (rows + mask) of the records of 32 rows into
// srow[32][29] with 16-byte loads, a warp at a time: each load instruction moves
// four records (7 lanes each).
__device__ __forceinline__ void warp_load_records(const uint32_t* src, uint32_t* srow, int lane) {
    const int sub = lane / 7, c = lane - sub * 7;  // record of the group, 16-byte chunk
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int r = it * 4 + (sub < 4 ? sub : 0);
        const unsigned long long a = __shfl_sync(0xffffffffu, (unsigned long long)src, r);
        if (sub < 4) {
            const uint32_t* rp = reinterpret_cast<const uint32_t*>(a);
            uint4 v = make_uint4(kNone, kNone, kNone, c == 6 ? 0u : kNone);  // no record: empty row, mask 0
            if (rp) v = *reinterpret_cast<const uint4*>(rp + 4 * c);
            uint32_t* d = srow + r * kRecStride + 4 * c;
            d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
        }
    }
}

// Caller-order pass: nbr[i], mask[i] from voxel i's record, and the row-order
// sort keys with the digit counts of every radix pass (every voxel counted once,
// so the passes' offsets always match their keys).  A voxel without a record
// gets an empty row and mask (the map is flagged bad then).
template <typename SK>
__global__ void __launch_bounds__(kSortThreads)
k_col_emit(const int4* __restrict__ coords, int64_t n, int B, int X, int Y, int Z, const uint32_t* __restrict__ start,
           int64_t ncols, const uint32_t* __restrict__ rec, const uint32_t* __restrict__ pos, int L, int G,
           int curve, int passes, uint32_t* __restrict__ nbr, uint32_t* __restrict__ mask, SK* __restrict__ keys,
           uint32_t* __restrict__ ghist) {
    __shared__ uint32_t srow[kSortThreads * kRecStride];
    __shared__ uint32_t h[kMaxSortPasses][kRadix];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    for (int p = 0; p < passes; ++p) h[p][t] = 0;
    __syncthreads();
    const int64_t total = col_entries(start, ncols, n);
    uint32_t* ws_rows = srow + warp * 32 * kRecStride;
    for (int64_t base = (int64_t)blockIdx.x * kSortThreads; base < n; base += (int64_t)gridDim.x * kSortThreads) {
        const int64_t i = base + t;
        const int64_t wbase = base + warp * 32;
        int4 c = make_int4(0, 0, 0, 0);
        const uint32_t* src = nullptr;
        if (i < n) {
            c = coords[i];
            src = col_record(rec, pos, total, (uint32_t)i, in_grid(c, B, X, Y, Z));
        }
        warp_load_records(src, ws_rows, lane);
        __syncwarp();
        if (i < n) {
            const uint32_t m = ws_rows[lane * kRecStride + kTaps];
            mask[i] = m;
            const SK key = (SK)order_key(c, m, L, G, curve);
            keys[i] = key;
            for (int p = 0; p < passes; ++p)
                atomicAdd(&h[p][(uint32_t)(key >> (p * kRadixBits)) & (kRadix - 1)], 1u);
        }
        if (wbase < n) {  // the warp's rows, contiguous in nbr
            const int rows = n - wbase < 32 ? (int)(n - wbase) : 32;
            uint32_t* out = nbr + wbase * kTaps;
            for (int w = lane; w < rows * kTaps; w += 32) {
                const int r = w / kTaps;
                out[w] = ws_rows[r * kRecStride + (w - r * kTaps)];
            }
        }
        __syncwarp();
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
    if (flags & ~(VG_KEY32 | VG_KEY64 | VG_ORDER_HILBERT | VG_MAP_HASH | VG_MAP_COLUMNS | VG_TEST_SMALL_HASH))
        return VG_ERR_INVALID_ARG;
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
    // Column index instead of the hash table when the table would not stay in L2
    // (above 64 MiB; measured at 4.9 M voxels, 268 MB table: 2.69 -> 1.51 ms; at
    // 602k voxels, 16 MB table: 0.307 ms hashed, 0.326 ms by column) and the
    // (b, x, y) columns are few for the voxels (their counts and starts cost 8
    // bytes per column); VG_MAP_COLUMNS / VG_MAP_HASH force one or the other.
    const double ncols = (double)B * X * Y;
    const bool cols_ok = ncols <= (double)(1 << 28);
    if ((flags & VG_MAP_COLUMNS) && (flags & (VG_MAP_HASH | VG_TEST_SMALL_HASH))) return VG_ERR_INVALID_ARG;
    if ((flags & VG_MAP_COLUMNS) && !cols_ok) return VG_ERR_UNSUPPORTED;
    const bool table_big = (double)(l.key64 ? 16 : 8) * (double)cap > 64.0 * 1048576.0;
    l.cols = (flags & VG_MAP_COLUMNS) ||
             (!(flags & (VG_MAP_HASH | VG_TEST_SMALL_HASH)) && cols_ok && table_big &&
              ncols <= 8.0 * (double)N + (double)(1 << 20));
    l.num_tiles = (N + kTileRows - 1) / kTileRows;
    // keys per thread in the radix sort: enough blocks to fill the GPU (about
    // 2 per SM), 4 to 16 keys per thread (below 4, the blocks' look-back chain
    // costs more than their parallelism gives: map build at 25k voxels 0.112 ms
    // with 1 key per thread, 0.107 ms with 4, 0.139 ms with 16)
    const int64_t per_block_target = std::max<int64_t>(1, N / (2 * (int64_t)l.sms));
    l.sort_items = (int)std::min<int64_t>(16, std::max<int64_t>(4, (per_block_target + kSortThreads - 1) / kSortThreads));
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
    if (l.cols) {
        // zeroed together: counts, the scan's chunk sums and its ticket
        l.ncols = (int64_t)ncols;
        l.cchunks = (l.ncols + 1 + kColScanChunk - 1) / kColScanChunk;
        l.off_ccnt = o;    o += align_up(4 * (size_t)(l.ncols + 1), 16);
        l.off_cpart = o;   o += 8 * (size_t)l.cchunks;
        l.off_cticket = o; o += 4;
        o = align_up(o, 256);  // every array below starts on a 256-byte boundary (16-byte record loads)
        l.off_cstart = o;  o += align_up(4 * (size_t)(l.ncols + 1), 256);
        l.off_carr = o;    o += align_up(4 * (size_t)N, 256);
        l.off_cent_a = o;  o += align_up(8 * (size_t)N, 256);
        l.off_cent_b = o;  o += align_up(8 * (size_t)N, 256);
        l.off_ccol_a = o;  o += align_up(4 * (size_t)N, 256);
        l.off_ccol_b = o;  o += align_up(4 * (size_t)N, 256);
        l.off_cpos = o;    o += align_up(4 * (size_t)N, 256);
        l.off_crec = o;    o += align_up(4 * (size_t)kRecWords * N, 256);
        for (const size_t off : {l.off_cstart, l.off_carr, l.off_cent_a, l.off_cent_b, l.off_ccol_a, l.off_ccol_b,
                                 l.off_cpos, l.off_crec})
            if (off & 255) return VG_ERR_UNSUPPORTED;  // layout invariant (never taken)
    } else {
        l.off_table = o;    o += align_up(slot * cap, 256);
    }
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
// With keys_ready, the masks, sort keys and digit counts were written by the
// probe already (after this half's memset, done by the caller).
static void layout_memset(const NbrLayout& l, char* ws, cudaStream_t s) {
    const int all = nbr_sort_passes(l) + l.tile_passes;
    cudaMemsetAsync(ws + l.off_hist, 0, l.off_tickets + 4 * (size_t)all - l.off_hist, s);  // counts, status, tickets
}

template <typename SK>
static void launch_layout(const int4* coords, const NbrLayout& l, int L, char* ws, const uint32_t* nbr,
                          uint32_t* mask, cudaStream_t s, bool keys_ready = false) {
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
    if (!keys_ready) {
        layout_memset(l, ws, s);
        // (a grid-stride loop: one key per thread up to four blocks per SM)
        const int gh_blocks =
            (int)std::max<int64_t>(1, std::min<int64_t>((n + kSortThreads - 1) / kSortThreads, 4 * (int64_t)l.sms));
        k_key_globalhist<SK><<<gh_blocks, kSortThreads, 0, s>>>(coords, nbr, n, L, l.fine_keep, l.curve, passes,
                                                                mask, ka, hist);
    }
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
    // (the column build gathers from nbr too: reading its 128-byte records here
    // through pos[] was measured slower, one more dependent load per row)
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

// Map build over the column index: count, scan, scatter, rank, probe (records in
// column order), emit (caller order: nbr, mask, sort keys and digit counts), then
// the row order.
template <typename SK>
static void launch_build_cols(const int4* coords, const NbrLayout& l, int B, int X, int Y, int Z, char* ws,
                              uint32_t* nbr, uint32_t* mask, cudaStream_t s) {
    const int64_t n = l.n;
    uint32_t* status = reinterpret_cast<uint32_t*>(ws + l.off_hdr);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + l.off_ccnt);
    uint32_t* start = reinterpret_cast<uint32_t*>(ws + l.off_cstart);
    uint32_t* arrival = reinterpret_cast<uint32_t*>(ws + l.off_carr);
    uint2* ent_a = reinterpret_cast<uint2*>(ws + l.off_cent_a);
    uint2* ent_b = reinterpret_cast<uint2*>(ws + l.off_cent_b);
    const unsigned vb = (unsigned)((n + 255) / 256);
    const int L = ceil_log2(std::max(X, std::max(Y, Z)));
    cudaMemsetAsync(cnt, 0, l.off_cticket + 4 - l.off_ccnt, s);  // counts, chunk sums, ticket
    layout_memset(l, ws, s);
    k_col_count<<<vb, 256, 0, s>>>(coords, n, B, X, Y, Z, cnt, arrival, status);
    k_col_scan<<<(unsigned)l.cchunks, kSortThreads, 0, s>>>(cnt, l.ncols + 1, start,
                                                            reinterpret_cast<uint64_t*>(ws + l.off_cpart),
                                                            reinterpret_cast<uint32_t*>(ws + l.off_cticket), status);
    uint32_t* col_a = reinterpret_cast<uint32_t*>(ws + l.off_ccol_a);
    uint32_t* col_b = reinterpret_cast<uint32_t*>(ws + l.off_ccol_b);
    k_col_scatter<<<vb, 256, 0, s>>>(coords, n, B, X, Y, Z, start, arrival, ent_a, col_a);
    uint32_t* pos = reinterpret_cast<uint32_t*>(ws + l.off_cpos);
    uint32_t* rec = reinterpret_cast<uint32_t*>(ws + l.off_crec);  // 16-byte records: 256-aligned offset
    k_col_rank<<<vb, 256, 0, s>>>(start, l.ncols, n, ent_a, col_a, ent_b, col_b, pos, status);
    k_col_probe<<<vb, 256, 0, s>>>(start, l.ncols, n, X, Y, ent_b, col_b, rec);
    const int passes = nbr_sort_passes(l);
    const unsigned kb = (unsigned)std::min<int64_t>(l.sort_blocks, 4 * (int64_t)l.sms);
    k_col_emit<SK><<<kb, kSortThreads, 0, s>>>(coords, n, B, X, Y, Z, start, l.ncols, rec, pos, L, l.fine_keep,
                                               l.curve, passes, nbr, mask, reinterpret_cast<SK*>(ws + l.off_skeys_a),
                                               reinterpret_cast<uint32_t*>(ws + l.off_hist));
    launch_layout<SK>(coords, l, L, ws, nbr, mask, s, true);
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
        if (l.cols) {
            if (l.sort64) launch_build_cols<uint64_t>(c4, l, B, X, Y, Z, ws, nbr, mask, s);
            else launch_build_cols<uint32_t>(c4, l, B, X, Y, Z, ws, nbr, mask, s);
        } else if (l.key64) {
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
    // each side keeps its hash table: the down / up lookups use it
    const unsigned side_flags = flags | VG_MAP_HASH;
    int st = nbr_layout(N, B, X, Y, Z, side_flags, sms_, &l.li);
    if (st != VG_OK) return st;
    st = nbr_layout(l.cap_out, B, l.Xo, l.Yo, l.Zo, side_flags, sms_, &l.lo_cap);
    if (st != VG_OK) return st;
    if (n_out >= 0) {  // the output side as laid out for the actual number of output sites
        if (n_out > l.cap_out) return VG_ERR_INVALID_ARG;
        st = nbr_layout(n_out, B, l.Xo, l.Yo, l.Zo, side_flags, sms_, &l.lo);
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
