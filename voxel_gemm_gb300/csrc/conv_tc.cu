// Tensor-core (tcgen05 / TMEM) masked implicit GEMM: the forward pass and the
// input-gradient pass over the sorted row tiles, for fp16/bf16 features
// (kind::f16) and for fp32 features read as TF32 (kind::tf32, when the caller
// allows TF32).
//
// Method: "From CUDA to Triton: Triton JIT and autotuning", §六 6.2 — the
// masked implicit GEMM kernel takes (input, weight, bias, neighbor,
// sorted_idx, output), gathers input rows per tap and contracts over V * Ci,
// skipping taps no row of the tile uses.  The backward reuses the same
// neighbour cache ("Contribution Tasks — JeffreyXiang/FlexGEMM", §二 call flow).
//
// GB300 design (one CTA per SM, two for tiles up to 128 columns; persistent over
// (128-row tile, N block) units):
//   warps 0-3  gather: per tap and 128-byte K block (64 16-bit or 32 fp32
//              channels), 128 rows x 128 B of the
//              feature matrix via 16-byte cp.async with zero fill for missing
//              neighbours, written in the 128-byte-swizzled K-major layout; each
//              thread's copies arrive on the stage barrier by themselves
//              (cp.async.mbarrier.arrive.noinc), so up to S stages are in flight;
//              each thread reads its eight source rows once per tap and reuses
//              them for every K block; thread 0 also bulk-copies, one unit ahead,
//              the tile's 13.5 KB neighbour block.  (L2 prefetching of later taps'
//              rows was measured to slow the gathers.)
//   warp 4     TMEM allocation and the single MMA-issuing thread:
//              tcgen05.mma M=128, N=BN, K=16 (K=8 for TF32), fp32 accumulators
//              in TMEM, several accumulator buffers so the epilogue overlaps
//              the next tiles.
//   warps 5-8  epilogue: tcgen05.ld, + bias, round to the output type, scatter
//              rows back to the caller's order through sorted_idx.
//   warp 9     weight-tile loader: one bulk copy (TMA engine) of the prepacked
//              weight tile per stage, kept off the gather warps' issue path.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace vg {

namespace {

using namespace ptx;

constexpr int kThreads = 320;          // 10 warps
constexpr int kBM = 128;               // rows per tile (MMA M)
constexpr int kKBytes = 128;           // bytes of one K block of a row (64 16-bit or 32 fp32 values)
constexpr int kABytes = kBM * kKBytes;  // 16 KB
constexpr int kMaxBiasCols = 2048;     // 16-bit bias staged in shared memory up to this many columns
constexpr int kMaxTapGroups = 6;      // most tap groups per (tile, N block) at small N

// Work units are handed out dynamically: gather thread 0 claims units from a
// global counter, one unit ahead (so that the next unit's neighbour lists can be
// copied in while the current one is gathered), and publishes each in an
// 8-slot ring that the MMA, epilogue and weight-loader roles read in order
// (-1 ends the sequence).  A CTA that
// draws units with few taps takes more of them; with the fixed round-robin the
// busiest CTA had 37 % more tap stages than the mean at 319k voxels, C = 128
// (12 % at 602k voxels, C = 256).
constexpr int kUnitRing = 8;
constexpr int kUnitReaders = 1 + 4 + 1;  // the MMA thread, the epilogue warps, the weight loader

// Element types of the kernel: A, B, bias and output share one.
constexpr int kF16 = VG_F16, kBF16 = VG_BF16, kTF32 = VG_F32;
template <int DT> struct Elt { static constexpr int size = DT == kTF32 ? 4 : 2; };

int choose_bn(int ndim) {
    if (ndim % 256 == 0) return 256;
    if (ndim % 128 == 0) return 128;
    if (ndim % 64 == 0) return 64;
    return 32;  // TF32 only (channels multiples of 32)
}

// Tiles up to 128 columns are issue-bound at the single MMA thread (four short
// MMAs per stage): two CTAs share each SM there, with 3 stages each at BN <= 64
// and 2 stages + 2 accumulator buffers at BN = 128, so that two MMA threads feed
// each tensor core (measured: forward 0.0389 -> 0.0305 ms at 25k voxels and
// 1.734 -> 1.600 ms at 4.9M, C = 64; 0.258 -> 0.195 ms at 319k voxels, C = 128;
// 4 stages with one CTA per SM: no gain).
template <int BN>
constexpr int ctas_per_sm() { return BN <= 128 ? 2 : 1; }

template <int BN>
struct Cfg {
    static constexpr int S = BN == 256 ? 4 : (BN == 128 ? 2 : 3);  // pipeline stages
    static constexpr int kBBytes = BN * kKBytes;
    static constexpr int NBUF = BN <= 64 ? 4 : 2;                   // TMEM accumulator buffers
    static constexpr int kTmemCols = NBUF * BN;                      // 128, 256 or 512 columns
    static constexpr size_t kSmemA = (size_t)S * kABytes;
    static constexpr size_t kSmemB = (size_t)S * kBBytes;
    static constexpr size_t kNbrTileBytes = (size_t)kBM * kTaps * 4;  // one tile of neighbour lists
    // full, empty, tfull, tempty, done, nbr x2, unit ring full and empty
    static constexpr int kNumBars = 2 * S + 2 * NBUF + 3 + 2 * kUnitRing;
    static constexpr size_t kSmem = 1024 + kSmemA + kSmemB + 2 * kNbrTileBytes + 8 * kNumBars + 8 * (kUnitRing + 2) + 16 +
                                    2 * kMaxBiasCols;
};

struct TcArgs {
    const uint32_t* sorted_idx;
    const uint32_t* tile_mask;
    const uint32_t* sorted_nbr;  // [tiles*128][27]
    const uint32_t* nbr_status;
    int64_t n;
    int64_t num_tiles;
    const uint8_t* A;     // [n][Kdim] elements
    int Kdim;
    const uint8_t* Bimg;  // packed weight tiles
    const void* bias;     // [Ndim] or null
    uint8_t* out;         // [n][Ndim]
    int Ndim;
    int ksplit;           // tap groups per (tile, N block); > 1: fp32 partials, reduced by a second kernel
    float* partial;       // [ksplit][num_tiles*128][Ndim] when ksplit > 1
    uint32_t* err;
    uint32_t* unit_ctr;   // next unit to claim (zero before the launch)
};

// Taps of group ks (of ks_count) of a tile's tap mask: its set bits, in order,
// cut into ks_count runs of near-equal length (run g holds the j-th set bit when
// floor(j * ks_count / popcount) = g).  ks_count = 1: the whole mask.
__device__ __forceinline__ uint32_t tap_group(uint32_t tm, int ks, int ks_count) {
    if (ks_count == 1) return tm;
    const int c = __popc(tm);
    uint32_t out = 0;
    int j = 0;
    for (uint32_t m = tm; m != 0u; m &= m - 1u, ++j)
        if (j * ks_count / c == ks) out |= m & (0u - m);
    return out;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}
template <bool BF16>
__device__ __forceinline__ float bits_to_f32(uint16_t b) {
    if constexpr (BF16) return __uint_as_float((uint32_t)b << 16);
    else return __half2float(__ushort_as_half(b));
}

// Add the bias to 32 fp32 accumulators of one row (columns col..col+31) and round
// them to the output type: 16 words of two 16-bit values, or 32 fp32 words.
template <int DT>
__device__ __forceinline__ void pack_row32(uint32_t* dst, const uint32_t (&acc)[32], const void* s_bias,
                                           const void* g_bias, int col) {
    const bool has_bias = g_bias != nullptr;
    if constexpr (DT == kTF32) {
        const float* gb = static_cast<const float*>(g_bias);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            dst[i] = __float_as_uint(__uint_as_float(acc[i]) + (has_bias ? __ldg(gb + col + i) : 0.f));
    } else {
        const uint16_t* sb = static_cast<const uint16_t*>(s_bias);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float lo = __uint_as_float(acc[2 * i]), hi = __uint_as_float(acc[2 * i + 1]);
            if (has_bias) {
                lo += bits_to_f32<DT == kBF16>(sb[col + 2 * i]);
                hi += bits_to_f32<DT == kBF16>(sb[col + 2 * i + 1]);
            }
            dst[i] = pack2<DT == kBF16>(lo, hi);
        }
    }
}

// Store one 128-byte line of output per row for a warp's 32 rows (lane i holds
// row i's line, output columns col.. of row v; kNone: no row).
template <int ES>
__device__ __forceinline__ void store_lines(uint8_t* out, int Ndim, uint32_t v, uint32_t (&z)[32], int col, int lane,
                                            bool v8ok) {
    store_lines_quad(v != kNone ? out + ((int64_t)v * Ndim + col) * ES : nullptr, z, lane, v8ok);
}

// Reads of unit-ring slot qi % R (phase parity (qi / R) & 1): by one thread, or
// warp-wide; the reader then releases the slot.  -1 when the sequence has ended
// or the wait gave up.
__device__ __forceinline__ int64_t read_unit_one(const volatile int64_t* s_unit, uint32_t ufull0, uint32_t uempty0,
                                                 uint32_t qi, const volatile uint32_t* abort) {
    const uint32_t slot = qi % kUnitRing;
    const int64_t u = mbar_wait(ufull0 + 8 * slot, (qi / kUnitRing) & 1u, abort) ? s_unit[slot] : -1;
    mbar_arrive(uempty0 + 8 * slot);
    return u;
}
__device__ __forceinline__ int64_t read_unit_warp(const volatile int64_t* s_unit, uint32_t ufull0, uint32_t uempty0,
                                                  uint32_t qi, int lane, const volatile uint32_t* abort) {
    const uint32_t slot = qi % kUnitRing;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(ufull0 + 8 * slot, (qi / kUnitRing) & 1u, abort));
    const int64_t u = ok ? s_unit[slot] : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(uempty0 + 8 * slot);
    return u;
}

template <int BN, int DT>
__global__ void __launch_bounds__(kThreads, ctas_per_sm<BN>()) k_gather_gemm_tc(TcArgs a) {
    using C = Cfg<BN>;
    constexpr int S = C::S;
    constexpr int ES = Elt<DT>::size;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::kSmemA;
    uint32_t* s_nbr = reinterpret_cast<uint32_t*>(sB + C::kSmemB);  // [2][128*27]
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_nbr + 2 * kBM * kTaps);
    volatile int64_t* s_unit = reinterpret_cast<volatile int64_t*>(bars + C::kNumBars);  // unit ring
    volatile int64_t* s_gu = s_unit + kUnitRing;  // [2]: the gather threads' current and next unit
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::kNumBars + kUnitRing + 2);
    volatile uint32_t* s_abort = s_tmem + 1;
    uint8_t* s_bias = reinterpret_cast<uint8_t*>(s_tmem + 4);  // [Ndim] elements when bias is given

    if (*a.nbr_status) return;  // bad neighbour map: write nothing (uniform over the block)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    constexpr int NBUF = C::NBUF;
    const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + NBUF);
    const uint32_t done_bar = smem_u32(bars + 2 * S + 2 * NBUF);
    const uint32_t nbar0 = smem_u32(bars + 2 * S + 2 * NBUF + 1);
    const uint32_t ufull0 = smem_u32(bars + 2 * S + 2 * NBUF + 3), uempty0 = ufull0 + 8 * kUnitRing;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kUnitRing; ++i) {
            mbar_init(ufull0 + 8 * i, 1);             // gather thread 0's publication of the slot
            mbar_init(uempty0 + 8 * i, kUnitReaders);  // every reader of the slot
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(full0 + 8 * i, 128 + 1);  // 128 gather threads + the weight-tile expect_tx
            mbar_init(empty0 + 8 * i, 1);       // one tcgen05.commit
        }
        for (int i = 0; i < NBUF; ++i) {
            mbar_init(tfull0 + 8 * i, 1);
            mbar_init(tempty0 + 8 * i, 4);      // one arrive per epilogue warp
        }
        mbar_init(done_bar, 1);
        mbar_init(nbar0, 1);
        mbar_init(nbar0 + 8, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(smem_u32(s_tmem), C::kTmemCols);
        tmem_relinquish();
    }
    if (DT != kTF32 && a.bias) {
        const uint32_t* bsrc = static_cast<const uint32_t*>(a.bias);
        for (int c = threadIdx.x; c < a.Ndim / 2; c += kThreads) reinterpret_cast<uint32_t*>(s_bias)[c] = bsrc[c];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    const int NB = a.Ndim / BN;
    const int KS = a.ksplit;
    const int64_t a_row_bytes = (int64_t)a.Kdim * ES;
    const int KB = (int)(a_row_bytes / kKBytes);
    // unit u = (tile t, N block nb, tap group ks), u = (t * NB + nb) * KS + ks
    const int64_t per_tile = (int64_t)NB * KS;
    const int64_t units = a.num_tiles * per_tile;
    auto unit_taps = [&](int64_t uu) {
        const int64_t t = uu / per_tile;
        return tap_group(a.tile_mask[t], (int)(uu % KS), KS);
    };

    if (warp < 4) {
        // ------------------------------------------------------------ gather producer
        // Every gather thread runs the same unit loop and the same named barriers;
        // after a failed wait a thread only skips work, so no barrier is left short.
        // The neighbour lists of the next unit's tile arrive by one bulk copy while
        // the current unit is gathered (two buffers).
        const int p = threadIdx.x;
        const uint32_t tile_bytes = (uint32_t)C::kNbrTileBytes;
        uint32_t it = 0;
        bool ok = true;
        // Thread 0 claims unit q + 1 while unit q is gathered, publishes it in ring
        // slot (q + 1) % R for the other roles, hands it to the gather threads through
        // s_gu[(q + 1) & 1] (read after the named barrier that ends unit q, so the
        // loop ends for all 128 threads together), and copies its tile's neighbour
        // lists into the other buffer.
        auto claim_publish = [&](uint32_t qq, uint32_t nbuf) {
            const uint32_t slot = qq % kUnitRing;
            const bool free_slot = mbar_wait(uempty0 + 8 * slot, ((qq / kUnitRing) & 1u) ^ 1u, s_abort);
            // the first unit of every CTA is blockIdx.x (grid <= units); later ones are claimed
            const int64_t uu = !free_slot ? units
                               : qq == 0 ? (int64_t)blockIdx.x
                                         : (int64_t)gridDim.x + (int64_t)atomicAdd(a.unit_ctr, 1u);
            const int64_t pub = uu < units ? uu : -1;
            s_unit[slot] = pub;
            s_gu[qq & 1u] = pub;
            mbar_arrive(ufull0 + 8 * slot);
            if (pub >= 0) {
                mbar_arrive_expect_tx(nbar0 + 8 * nbuf, tile_bytes);
                bulk_g2s(smem_u32(s_nbr + nbuf * kBM * kTaps), a.sorted_nbr + (pub / per_tile) * kBM * kTaps,
                         tile_bytes, nbar0 + 8 * nbuf);
            }
        };
        if (p == 0) claim_publish(0, 0);
        named_bar_sync(1, 128);
        for (uint32_t idx = 0;; ++idx) {
            const int64_t u = s_gu[idx & 1u];
            if (u < 0) break;  // the same value in every gather thread
            const uint32_t buf = idx & 1u;
            const uint32_t tm = unit_taps(u);
            // buffer buf^1 was released by the named barrier that ended the previous unit
            if (p == 0) claim_publish(idx + 1, buf ^ 1u);
            // always wait for this unit's copy, so none is in flight when the block exits
            if (!mbar_wait_timed(nbar0 + 8 * buf, (idx >> 1) & 1u)) {
                ok = false;
                *s_abort = 1;
            }
            const uint32_t* nb_tile = s_nbr + buf * kBM * kTaps;
            const int ch = p & 7;
            for (int k = 0; k < kTaps && ok; ++k) {
                if (!((tm >> k) & 1u)) continue;
                // this thread's 8 source rows for tap k, read from shared memory once per tap
                // (all eight loads issue back to back) and reused by every K block
                const uint8_t* src[8];
                uint32_t src_bytes[8];
#pragma unroll
                for (int i2 = 0; i2 < 8; ++i2) {
                    const uint32_t j = nb_tile[(i2 * 16 + (p >> 3)) * kTaps + k];
                    src[i2] = a.A + (int64_t)(j != kNone ? j : 0u) * a_row_bytes + ch * 16;
                    src_bytes[i2] = j != kNone ? 16u : 0u;
                }
                for (int kb = 0; kb < KB; ++kb) {
                    const uint32_t stage = it % S, ph = (it / S) & 1u;
                    if (!mbar_wait(empty0 + 8 * stage, ph ^ 1u, s_abort)) {
                        ok = false;
                        *s_abort = 1;
                        break;
                    }
                    const uint32_t a_base = smem_u32(sA + stage * kABytes);
#pragma unroll
                    for (int i2 = 0; i2 < 8; ++i2) {
                        const int row = i2 * 16 + (p >> 3);
                        cp_async16(a_base + row * 128 + ((ch ^ (row & 7)) << 4), src[i2] + kb * kKBytes,
                                   src_bytes[i2]);
                    }
                    // arrives on the stage barrier when this thread's copies have landed
                    cp_async_arrive_noinc(full0 + 8 * stage);
                    ++it;
                }
            }
            named_bar_sync(1, 128);  // every gather thread is done with buffer buf
        }
        cp_async_wait_all();  // no copy of this thread is still writing shared memory
        if (!ok) atomicOr(a.err, kErrTimeout);
        // Before the block may exit, every stage's last fill must have landed, its
        // copy-completion arrivals included (already true unless a wait gave up).
        if (p == 0)
            for (uint32_t i = 0; i < S && i < it; ++i) {
                const uint32_t last = it - 1 - i;
                if (!mbar_wait_timed(full0 + 8 * (last % S), (last / S) & 1u)) atomicOr(a.err, kErrTimeout);
            }
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = DT == kTF32 ? idesc_tf32(BN) : idesc_f16(DT == kBF16, BN);
            uint32_t it = 0, ua = 0;
            bool ok = true;
            for (uint32_t qi = 0; ok; ++qi) {
                const int64_t u = read_unit_one(s_unit, ufull0, uempty0, qi, s_abort);
                if (u < 0) break;
                const uint32_t tm = unit_taps(u);
                if (tm == 0u) continue;  // an empty tap group (split units only): no accumulator used
                const uint32_t uc = ua++;
                const uint32_t buf = uc % NBUF;
                if (!mbar_wait(tempty0 + 8 * buf, ((uc / NBUF) & 1u) ^ 1u, s_abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem + buf * BN;
                uint32_t acc = 0;
                for (int k = 0; k < kTaps && ok; ++k) {
                    if (!((tm >> k) & 1u)) continue;
                    for (int kb = 0; kb < KB; ++kb) {
                        const uint32_t stage = it % S, ph = (it / S) & 1u;
                        if (!mbar_wait(full0 + 8 * stage, ph, s_abort)) { ok = false; break; }
                        // the A tile was written by cp.async (generic proxy); the MMA reads it
                        // through the async proxy
                        fence_proxy_async_smem();
                        tc_fence_after();
                        const uint32_t a_base = smem_u32(sA + stage * kABytes);
                        const uint32_t b_base = smem_u32(sB + stage * C::kBBytes);
                        // four MMAs per 128-byte K block: K = 16 (16-bit) or K = 8 (TF32),
                        // 32 bytes of each row apiece
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if constexpr (DT == kTF32)
                                mma_tf32(d_tmem, sw128_kmajor_desc(a_base + 32 * j),
                                         sw128_kmajor_desc(b_base + 32 * j), idesc, acc | (uint32_t)j);
                            else
                                mma_f16(d_tmem, sw128_kmajor_desc(a_base + 32 * j),
                                        sw128_kmajor_desc(b_base + 32 * j), idesc, acc | (uint32_t)j);
                        }
                        acc = 1;
                        mma_commit(empty0 + 8 * stage);
                        ++it;
                    }
                }
                if (ok) mma_commit(tfull0 + 8 * buf);
            }
            // all issued MMAs must finish before TMEM is released: time-bounded, ignores the abort flag
            mma_commit(done_bar);
            const bool drained = mbar_wait_timed(done_bar, 0);
            if (!ok || !drained) {
                *s_abort = 1;
                atomicOr(a.err, kErrTimeout);
            }
        }
        __syncwarp();
    } else if (warp <= 8) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const bool v8ok = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0;
        uint32_t ua = 0;
        bool ok = true;
        const int64_t rows_pad = a.num_tiles * kBM;
        for (uint32_t qi = 0;; ++qi) {
            const int64_t u = read_unit_warp(s_unit, ufull0, uempty0, qi, lane, s_abort);
            if (u < 0) break;
            const int64_t t = u / per_tile;
            const int nb = (int)((u % per_tile) / KS);
            const int ks = (int)(u % KS);
            // output row of this thread (its load overlaps the wait for the accumulator)
            const int64_t r_out = t * kBM + q * 32 + lane;
            const uint32_t v = KS == 1 && r_out < a.n ? a.sorted_idx[r_out] : kNone;
            const int col0 = nb * BN;
            // split units write fp32 partials for every row of the tile, in sorted order
            float* prow = KS > 1 ? a.partial + ((int64_t)ks * rows_pad + t * kBM + q * 32 + lane) * a.Ndim + col0
                                 : nullptr;
            if (KS > 1 && unit_taps(u) == 0u) {  // empty tap group: its partial is zero
                for (int c = 0; c < BN; c += 4)
                    *reinterpret_cast<float4*>(prow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                continue;
            }
            const uint32_t buf = ua % NBUF;
            ok = __all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * buf, (ua / NBUF) & 1u, s_abort));
            ++ua;
            if (!ok) break;  // warp-uniform
            tc_fence_after();
            if (KS > 1) {
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    uint32_t acc[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + buf * BN + c0, acc);
                    tmem_ld_wait();
                    float4* d4 = reinterpret_cast<float4*>(prow + c0);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        d4[i] = make_float4(__uint_as_float(acc[4 * i]), __uint_as_float(acc[4 * i + 1]),
                                            __uint_as_float(acc[4 * i + 2]), __uint_as_float(acc[4 * i + 3]));
                }
            } else {
                // one 128-byte output line per row at a time: 64 16-bit or 32 fp32 columns
                constexpr int kLine = 128 / ES;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += kLine) {
                    uint32_t z[32];
#pragma unroll
                    for (int part = 0; part < kLine / 32; ++part) {
                        uint32_t acc[32];
                        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + buf * BN + c0 + 32 * part, acc);
                        tmem_ld_wait();
                        pack_row32<DT>(z + part * 16, acc, s_bias, a.bias, col0 + c0 + 32 * part);
                    }
                    store_lines<ES>(a.out, a.Ndim, v, z, col0 + c0, lane, v8ok);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * buf);
        }
        if (!ok) {
            *s_abort = 1;
            atomicOr(a.err, kErrTimeout);
        }
    } else {
        // ------------------------------------------------------------ weight-tile loader
        if (lane == 0) {
            // One bulk copy per stage, in the gather threads' (unit, tap, K block) order;
            // its expect_tx arrival is the stage barrier's 129th.
            uint32_t it = 0;
            bool ok = true;
            for (uint32_t qi = 0; ok; ++qi) {
                const int64_t u = read_unit_one(s_unit, ufull0, uempty0, qi, s_abort);
                if (u < 0) break;
                const int nb = (int)((u % per_tile) / KS);
                const uint32_t tm = unit_taps(u);
                for (int k = 0; k < kTaps && ok; ++k) {
                    if (!((tm >> k) & 1u)) continue;
                    const uint8_t* bsrc = a.Bimg + ((int64_t)nb * kTaps + k) * KB * C::kBBytes;
                    for (int kb = 0; kb < KB; ++kb) {
                        const uint32_t stage = it % S, ph = (it / S) & 1u;
                        if (!mbar_wait(empty0 + 8 * stage, ph ^ 1u, s_abort)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full0 + 8 * stage, C::kBBytes);
                        bulk_g2s(smem_u32(sB + stage * C::kBBytes), bsrc + kb * C::kBBytes, C::kBBytes, full0 + 8 * stage);
                        ++it;
                    }
                }
            }
            if (!ok) {
                *s_abort = 1;
                atomicOr(a.err, kErrTimeout);
            }
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) tmem_dealloc(tmem, C::kTmemCols);
}

// ---------------------------------------------------------------------------
// Tile pairs (256 output columns): one unit = two consecutive 128-row tiles x
// one 256-column N block.  Each stage holds both tiles' gathered rows for one
// (tap, K block) and ONE weight tile, which feeds two M = 128 MMAs (one per
// tile, each into its own 256-column TMEM accumulator): per stage 64 KB of
// shared memory for 8.4 MFLOP instead of 48 KB for 4.2 MFLOP, so the weight
// tiles -- two thirds of the single-tile kernel's L2 reads -- are read once per
// pair.  Each tile still skips its own absent taps: a stage carries the rows of
// only the tiles whose mask has the tap, and the MMA thread issues only their
// MMAs, so no MMA runs on rows of a tap its tile does not use; only the weight
// tile is shared (read for the union of the two masks).
//   warps 0-3    gather (both tiles: 16 rows of 16 B per thread per stage)
//   warp 4       TMEM (all 512 columns) and the MMA-issuing thread
//   warps 5-8    epilogue of the first tile; warps 10-13 that of the second
//                (warp w reads TMEM lane quadrant w % 4), concurrently
//   warp 9       weight-tile loader
// The accumulators are not double-buffered (two tiles x 256 columns fill TMEM):
// the MMA thread starts a unit once the first tile's accumulator has been read
// out, and its first MMA into the second tile once that one has.
constexpr int kPairThreads = 448;  // 14 warps
constexpr int kPairReaders = 1 + 8 + 1;  // the MMA thread, 8 epilogue warps, the weight loader

struct PairCfg {
    static constexpr int S = 3;  // stages
    static constexpr int BN = 256;
    static constexpr int kBBytes = BN * kKBytes;                   // 32 KB
    static constexpr int kStageBytes = 2 * kABytes + kBBytes;      // 64 KB: tile 0 rows, tile 1 rows, weights
    static constexpr size_t kNbrBytes = (size_t)2 * kBM * kTaps * 4;
    // full x S, empty x S, tfull, tempty x 2, done, nbr, unit ring full and empty
    static constexpr int kNumBars = 2 * S + 5 + 2 * kUnitRing;
    static constexpr size_t kSmem = 1024 + (size_t)S * kStageBytes + kNbrBytes + 8 * kNumBars + 8 * (kUnitRing + 2) +
                                    16 + 2 * kMaxBiasCols;
};
static_assert(PairCfg::kSmem <= 232448, "tile-pair kernel exceeds the shared memory of one CTA");

template <int DT>
__global__ void __launch_bounds__(kPairThreads, 1) k_gather_gemm_pair(TcArgs a) {
    using C = PairCfg;
    constexpr int S = C::S, BN = C::BN;
    constexpr int ES = Elt<DT>::size;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sStage = smem;                                                     // [S][rows 0 | rows 1 | weights]
    uint32_t* s_nbr = reinterpret_cast<uint32_t*>(smem + (size_t)S * C::kStageBytes);  // [256][27]
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_nbr + 2 * kBM * kTaps);
    volatile int64_t* s_unit = reinterpret_cast<volatile int64_t*>(bars + C::kNumBars);
    volatile int64_t* s_gu = s_unit + kUnitRing;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + C::kNumBars + kUnitRing + 2);
    volatile uint32_t* s_abort = s_tmem + 1;
    uint8_t* s_bias = reinterpret_cast<uint8_t*>(s_tmem + 4);

    if (*a.nbr_status) return;  // bad neighbour map: write nothing (uniform over the block)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t tfull = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + 1);
    const uint32_t done_bar = smem_u32(bars + 2 * S + 3), nbar = smem_u32(bars + 2 * S + 4);
    const uint32_t ufull0 = smem_u32(bars + 2 * S + 5), uempty0 = ufull0 + 8 * kUnitRing;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kUnitRing; ++i) {
            mbar_init(ufull0 + 8 * i, 1);
            mbar_init(uempty0 + 8 * i, kPairReaders);
        }
        for (int i = 0; i < S; ++i) {
            mbar_init(full0 + 8 * i, 128 + 1);  // 128 gather threads + the weight-tile expect_tx
            mbar_init(empty0 + 8 * i, 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty0, 4);      // the four epilogue warps of tile 0
        mbar_init(tempty0 + 8, 4);  // ... of tile 1
        mbar_init(done_bar, 1);
        mbar_init(nbar, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(smem_u32(s_tmem), 2 * BN);
        tmem_relinquish();
    }
    if (DT != kTF32 && a.bias) {
        const uint32_t* bsrc = static_cast<const uint32_t*>(a.bias);
        for (int c = threadIdx.x; c < a.Ndim / 2; c += kPairThreads) reinterpret_cast<uint32_t*>(s_bias)[c] = bsrc[c];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    const int NB = a.Ndim / BN;
    const int64_t a_row_bytes = (int64_t)a.Kdim * ES;
    const int KB = (int)(a_row_bytes / kKBytes);
    // unit u = (tile pair tp, N block nb), u = tp * NB + nb; tiles 2tp and 2tp + 1
    const int64_t units = (a.num_tiles + 1) / 2 * NB;
    auto tile_taps = [&](int64_t t) { return t < a.num_tiles ? a.tile_mask[t] : 0u; };

    if (warp < 4) {
        // ------------------------------------------------------------ gather producer
        // As in the single-tile kernel, with one neighbour-list buffer (both tiles,
        // 27 KB): thread 0 copies the next unit's lists in once every gather thread
        // has finished the current unit.
        const int p = threadIdx.x;
        uint32_t it = 0;
        bool ok = true;
        auto claim_publish = [&](uint32_t qq) {
            const uint32_t slot = qq % kUnitRing;
            const bool free_slot = mbar_wait(uempty0 + 8 * slot, ((qq / kUnitRing) & 1u) ^ 1u, s_abort);
            const int64_t uu = !free_slot ? units
                               : qq == 0 ? (int64_t)blockIdx.x
                                         : (int64_t)gridDim.x + (int64_t)atomicAdd(a.unit_ctr, 1u);
            const int64_t pub = uu < units ? uu : -1;
            s_unit[slot] = pub;
            s_gu[qq & 1u] = pub;
            mbar_arrive(ufull0 + 8 * slot);
        };
        auto copy_nbr = [&](int64_t uu) {
            const int64_t t0 = uu / NB * 2;
            const uint32_t bytes = (uint32_t)((t0 + 1 < a.num_tiles ? 2 : 1) * kBM * kTaps * 4);
            mbar_arrive_expect_tx(nbar, bytes);
            bulk_g2s(smem_u32(s_nbr), a.sorted_nbr + t0 * kBM * kTaps, bytes, nbar);
        };
        if (p == 0) {
            claim_publish(0);
            if (s_gu[0] >= 0) copy_nbr(s_gu[0]);
        }
        named_bar_sync(1, 128);
        const int ch = p & 7;
        for (uint32_t idx = 0;; ++idx) {
            const int64_t u = s_gu[idx & 1u];
            if (u < 0) break;  // the same value in every gather thread
            const int64_t t0 = u / NB * 2;
            const uint32_t m0 = tile_taps(t0), m1 = tile_taps(t0 + 1);
            if (p == 0) claim_publish(idx + 1);
            // always wait for this unit's copy, so none is in flight when the block exits
            if (!mbar_wait_timed(nbar, idx & 1u)) {
                ok = false;
                *s_abort = 1;
            }
            for (int k = 0; k < kTaps && ok; ++k) {
                const bool h0 = (m0 >> k) & 1u, h1 = (m1 >> k) & 1u;
                if (!h0 && !h1) continue;
                // this thread's 8 source rows of each present tile for tap k
                const uint8_t* src[16];
                uint32_t src_bytes[16];
#pragma unroll
                for (int i2 = 0; i2 < 16; ++i2) {
                    const bool present = i2 < 8 ? h0 : h1;
                    const uint32_t j = present ? s_nbr[((i2 >> 3) * kBM + (i2 & 7) * 16 + (p >> 3)) * kTaps + k] : kNone;
                    src[i2] = a.A + (int64_t)(j != kNone ? j : 0u) * a_row_bytes + ch * 16;
                    src_bytes[i2] = j != kNone ? 16u : 0u;
                }
                for (int kb = 0; kb < KB; ++kb) {
                    const uint32_t stage = it % S, ph = (it / S) & 1u;
                    if (!mbar_wait(empty0 + 8 * stage, ph ^ 1u, s_abort)) {
                        ok = false;
                        *s_abort = 1;
                        break;
                    }
                    const uint32_t base = smem_u32(sStage + (size_t)stage * C::kStageBytes);
                    if (h0) {
#pragma unroll
                        for (int i2 = 0; i2 < 8; ++i2) {
                            const int row = i2 * 16 + (p >> 3);
                            cp_async16(base + row * 128 + ((ch ^ (row & 7)) << 4), src[i2] + kb * kKBytes,
                                       src_bytes[i2]);
                        }
                    }
                    if (h1) {
#pragma unroll
                        for (int i2 = 0; i2 < 8; ++i2) {
                            const int row = i2 * 16 + (p >> 3);
                            cp_async16(base + kABytes + row * 128 + ((ch ^ (row & 7)) << 4),
                                       src[8 + i2] + kb * kKBytes, src_bytes[8 + i2]);
                        }
                    }
                    cp_async_arrive_noinc(full0 + 8 * stage);
                    ++it;
                }
            }
            named_bar_sync(1, 128);  // every gather thread is done with the neighbour lists
            if (p == 0) {
                const int64_t nu = s_gu[(idx + 1) & 1u];
                if (nu >= 0) copy_nbr(nu);
            }
        }
        cp_async_wait_all();
        if (!ok) atomicOr(a.err, kErrTimeout);
        if (p == 0)
            for (uint32_t i = 0; i < S && i < it; ++i) {
                const uint32_t last = it - 1 - i;
                if (!mbar_wait_timed(full0 + 8 * (last % S), (last / S) & 1u)) atomicOr(a.err, kErrTimeout);
            }
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = DT == kTF32 ? idesc_tf32(BN) : idesc_f16(DT == kBF16, BN);
            uint32_t it = 0, uc = 0;
            bool ok = true;
            for (uint32_t qi = 0; ok; ++qi) {
                const int64_t u = read_unit_one(s_unit, ufull0, uempty0, qi, s_abort);
                if (u < 0) break;
                const int64_t t0 = u / NB * 2;
                const uint32_t m0 = tile_taps(t0), m1 = tile_taps(t0 + 1);
                // accumulator h is free once the epilogue has read out unit uc - 1's tile h
                const uint32_t par = (uc & 1u) ^ 1u;
                if (!mbar_wait(tempty0, par, s_abort)) { ok = false; break; }
                tc_fence_after();
                bool free1 = false;
                uint32_t acc0 = 0, acc1 = 0;
                for (int k = 0; k < kTaps && ok; ++k) {
                    const bool h0 = (m0 >> k) & 1u, h1 = (m1 >> k) & 1u;
                    if (!h0 && !h1) continue;
                    if (h1 && !free1) {
                        if (!mbar_wait(tempty0 + 8, par, s_abort)) { ok = false; break; }
                        tc_fence_after();
                        free1 = true;
                    }
                    for (int kb = 0; kb < KB; ++kb) {
                        const uint32_t stage = it % S, ph = (it / S) & 1u;
                        if (!mbar_wait(full0 + 8 * stage, ph, s_abort)) { ok = false; break; }
                        fence_proxy_async_smem();
                        tc_fence_after();
                        const uint32_t base = smem_u32(sStage + (size_t)stage * C::kStageBytes);
                        const uint32_t b_base = base + 2 * kABytes;
                        if (h0) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                if constexpr (DT == kTF32)
                                    mma_tf32(tmem, sw128_kmajor_desc(base + 32 * j), sw128_kmajor_desc(b_base + 32 * j),
                                             idesc, acc0 | (uint32_t)j);
                                else
                                    mma_f16(tmem, sw128_kmajor_desc(base + 32 * j), sw128_kmajor_desc(b_base + 32 * j),
                                            idesc, acc0 | (uint32_t)j);
                            }
                            acc0 = 1;
                        }
                        if (h1) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                if constexpr (DT == kTF32)
                                    mma_tf32(tmem + BN, sw128_kmajor_desc(base + kABytes + 32 * j),
                                             sw128_kmajor_desc(b_base + 32 * j), idesc, acc1 | (uint32_t)j);
                                else
                                    mma_f16(tmem + BN, sw128_kmajor_desc(base + kABytes + 32 * j),
                                            sw128_kmajor_desc(b_base + 32 * j), idesc, acc1 | (uint32_t)j);
                            }
                            acc1 = 1;
                        }
                        mma_commit(empty0 + 8 * stage);
                        ++it;
                    }
                }
                // tfull's next phase must not complete before the second tile's epilogue
                // warps have seen this one: wait for their previous read-out here at the latest
                if (ok && !free1 && !mbar_wait(tempty0 + 8, par, s_abort)) ok = false;
                if (ok) mma_commit(tfull);
                ++uc;
            }
            mma_commit(done_bar);
            const bool drained = mbar_wait_timed(done_bar, 0);
            if (!ok || !drained) {
                *s_abort = 1;
                atomicOr(a.err, kErrTimeout);
            }
        }
        __syncwarp();
    } else if (warp != 9) {
        // ------------------------------------------------------------ epilogue (tile h of the pair)
        const int h = warp >= 10 ? 1 : 0;
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const bool v8ok = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0;
        uint32_t uc = 0;
        bool ok = true;
        for (uint32_t qi = 0;; ++qi) {
            const int64_t u = read_unit_warp(s_unit, ufull0, uempty0, qi, lane, s_abort);
            if (u < 0) break;
            const int64_t t = u / NB * 2 + h;
            const int col0 = (int)(u % NB) * BN;
            const uint32_t mh = tile_taps(t);
            const int64_t r_out = t * kBM + q * 32 + lane;
            const uint32_t v = r_out < a.n ? a.sorted_idx[r_out] : kNone;
            ok = __all_sync(0xffffffffu, mbar_wait(tfull, uc & 1u, s_abort));
            ++uc;
            if (!ok) break;  // warp-uniform
            tc_fence_after();
            // one 128-byte output line per row at a time: 64 16-bit or 32 fp32 columns
            constexpr int kLine = 128 / ES;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += kLine) {
                uint32_t z[32];
#pragma unroll
                for (int part = 0; part < kLine / 32; ++part) {
                    uint32_t acc[32];
                    if (mh != 0u) {  // warp-uniform; a tile with no taps has a zero sum
                        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + h * BN + c0 + 32 * part, acc);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) acc[i] = 0u;
                    }
                    pack_row32<DT>(z + part * 16, acc, s_bias, a.bias, col0 + c0 + 32 * part);
                }
                store_lines<ES>(a.out, a.Ndim, v, z, col0 + c0, lane, v8ok);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * h);
        }
        if (!ok) {
            *s_abort = 1;
            atomicOr(a.err, kErrTimeout);
        }
    } else {
        // ------------------------------------------------------------ weight-tile loader
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (uint32_t qi = 0; ok; ++qi) {
                const int64_t u = read_unit_one(s_unit, ufull0, uempty0, qi, s_abort);
                if (u < 0) break;
                const int nb = (int)(u % NB);
                const int64_t t0 = u / NB * 2;
                const uint32_t mu = tile_taps(t0) | tile_taps(t0 + 1);
                for (int k = 0; k < kTaps && ok; ++k) {
                    if (!((mu >> k) & 1u)) continue;
                    const uint8_t* bsrc = a.Bimg + ((int64_t)nb * kTaps + k) * KB * C::kBBytes;
                    for (int kb = 0; kb < KB; ++kb) {
                        const uint32_t stage = it % S, ph = (it / S) & 1u;
                        if (!mbar_wait(empty0 + 8 * stage, ph ^ 1u, s_abort)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full0 + 8 * stage, C::kBBytes);
                        bulk_g2s(smem_u32(sStage + (size_t)stage * C::kStageBytes + 2 * kABytes), bsrc + kb * C::kBBytes,
                                 C::kBBytes, full0 + 8 * stage);
                        ++it;
                    }
                }
            }
            if (!ok) {
                *s_abort = 1;
                atomicOr(a.err, kErrTimeout);
            }
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) tmem_dealloc(tmem, 2 * BN);
}

// Repack W into the B-operand tiles the MMA reads: for tap k, N block nb and
// K block kb, a [BN rows][128 bytes of K] tile (64 16-bit or 32 fp32 K values),
// rows in the 128-byte swizzled layout (row n at (n/8)*1024 + (n%8)*128,
// 16-byte chunk c stored at chunk c ^ (n%8)).  fwd: row n = output channel,
// K = input channel, element W[k][kk][n].  dgrad: row n = input channel,
// K = output channel, element W[26-k][n][kk] (the flipped, transposed tap);
// mode 2 (input gradient of a strided / transposed map): element W[k][n][kk].
// One block = one tap, one K block and 32 consecutive rows n.
template <typename T>
__global__ void __launch_bounds__(256)
k_pack_weights(const T* __restrict__ W, int Cin, int Cout, int mode, int BN, uint8_t* __restrict__ img) {
    constexpr int KE = 128 / sizeof(T);  // K values per block row
    constexpr int PER_CHUNK = 16 / sizeof(T);
    __shared__ T tile[KE][33];
    const int k = blockIdx.x, kb = blockIdx.y, n0 = blockIdx.z * 32;
    const int Kdim = mode ? Cout : Cin;
    const int src_tap = mode == 1 ? 26 - k : k;
    const int KB = Kdim / KE;
    const int tid = threadIdx.x;
    for (int idx = tid; idx < KE * 32; idx += 256) {
        if (!mode) {
            const int kk = idx >> 5, n = idx & 31;
            tile[kk][n] = W[((int64_t)k * Cin + kb * KE + kk) * Cout + n0 + n];
        } else {
            const int n = idx / KE, kk = idx % KE;
            tile[kk][n] = W[((int64_t)src_tap * Cin + n0 + n) * Cout + kb * KE + kk];
        }
    }
    __syncthreads();
    for (int chk = tid; chk < 32 * 8; chk += 256) {
        const int n = chk >> 3, c = chk & 7;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if constexpr (sizeof(T) == 4)
                w[e] = __float_as_uint(tile[c * PER_CHUNK + e][n]);
            else
                w[e] = (uint32_t)tile[c * PER_CHUNK + 2 * e][n] | ((uint32_t)tile[c * PER_CHUNK + 2 * e + 1][n] << 16);
        }
        const int gn = n0 + n, nb = gn / BN, nl = gn - nb * BN;
        const int64_t base = (((int64_t)nb * kTaps + k) * KB + kb) * (int64_t)BN * 128;
        const int64_t off = base + (nl >> 3) * 1024 + (nl & 7) * 128 + ((c ^ (nl & 7)) << 4);
        *reinterpret_cast<uint4*>(img + off) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int BN, int DT>
int launch_tc(const TcArgs& a, cudaStream_t s) {
    using C = Cfg<BN>;
    auto kern = k_gather_gemm_tc<BN, DT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem) != cudaSuccess)
        return VG_ERR_CUDA;
    const int64_t units = a.num_tiles * (a.Ndim / BN) * a.ksplit;
    const int grid = (int)std::min<int64_t>(units, (int64_t)ctas_per_sm<BN>() * plan_sms(0));
    TcArgs b = a;
    b.unit_ctr = a.err + kGatherUnitCounter;
    // with no more units than CTAs every claim returns >= gridDim.x >= units (the end),
    // whatever the counter holds: no reset needed
    if (units > grid) cudaMemsetAsync(b.unit_ctr, 0, sizeof(uint32_t), s);
    kern<<<grid, kThreads, C::kSmem, s>>>(b);
    return VG_OK;
}

// Tile pairs at 256 output columns whenever the pairs alone give every SM a unit.
bool pair_tiles(int64_t num_tiles, int Ndim, int ksplit, int sms) {
    return ksplit == 1 && choose_bn(Ndim) == PairCfg::BN && (num_tiles + 1) / 2 * (Ndim / PairCfg::BN) >= sms;
}

template <int DT>
int launch_pair(const TcArgs& a, cudaStream_t s) {
    auto kern = k_gather_gemm_pair<DT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PairCfg::kSmem) != cudaSuccess)
        return VG_ERR_CUDA;
    const int64_t units = (a.num_tiles + 1) / 2 * (a.Ndim / PairCfg::BN);
    const int grid = (int)std::min<int64_t>(units, (int64_t)plan_sms(0));
    TcArgs b = a;
    b.unit_ctr = a.err + kGatherUnitCounter;
    if (units > grid) cudaMemsetAsync(b.unit_ctr, 0, sizeof(uint32_t), s);
    kern<<<grid, kPairThreads, PairCfg::kSmem, s>>>(b);
    return VG_OK;
}

// Forward / input-gradient with tap-group units: the fixed-order sum of the
// groups' fp32 partials (group 0 first), + bias, rounded once, written to the
// caller's row order through sorted_idx.
template <typename T>
__global__ void __launch_bounds__(256)
k_split_reduce(const float* __restrict__ partial, int ks_count, int64_t rows_pad, int64_t n, int Ndim,
               const uint32_t* __restrict__ sorted_idx, const T* __restrict__ bias, T* __restrict__ out,
               const uint32_t* __restrict__ nbr_status) {
    if (*nbr_status) return;
    const int c4n = Ndim / 4;
    const int64_t total = n * c4n;
    for (int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x; e < total; e += (int64_t)gridDim.x * 256) {
        const int64_t r = e / c4n;
        const int c = (int)(e - r * c4n) * 4;
        float4 acc = *reinterpret_cast<const float4*>(partial + r * Ndim + c);
        for (int g = 1; g < ks_count; ++g) {
            const float4 v = *reinterpret_cast<const float4*>(partial + ((int64_t)g * rows_pad + r) * Ndim + c);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        if (bias) {
            acc.x += to_f32(bias[c]);
            acc.y += to_f32(bias[c + 1]);
            acc.z += to_f32(bias[c + 2]);
            acc.w += to_f32(bias[c + 3]);
        }
        T* dst = out + (int64_t)sorted_idx[r] * Ndim + c;
        dst[0] = from_f32<T>(acc.x);
        dst[1] = from_f32<T>(acc.y);
        dst[2] = from_f32<T>(acc.z);
        dst[3] = from_f32<T>(acc.w);
    }
}

template <typename T>
void launch_split_reduce(const TcArgs& a, int sms, cudaStream_t s) {
    const int64_t total = a.n * (a.Ndim / 4);
    const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, 8 * (int64_t)sms));
    k_split_reduce<T><<<blocks, 256, 0, s>>>(a.partial, a.ksplit, a.num_tiles * kBM, a.n, a.Ndim, a.sorted_idx,
                                             static_cast<const T*>(a.bias), reinterpret_cast<T*>(a.out),
                                             a.nbr_status);
}

}  // namespace

// (Counted against the SM count, not the resident CTAs: at BN <= 128 two CTAs
// share an SM, and splitting units that already fill the SMs once was measured
// slower -- 25k voxels, C = 64: 0.0305 -> 0.045 ms.)
int tc_gather_splits(int64_t n, int Ndim, int sms) {
    const int64_t units = (n + kBM - 1) / kBM * (Ndim / choose_bn(Ndim));
    if (units == 0 || units >= sms) return 1;
    return (int)std::min<int64_t>(kMaxTapGroups, (sms + units - 1) / units);
}

int tc_supported(int dtype, int Cin, int Cout) {
    return (dtype == VG_F16 || dtype == VG_BF16) && Cin % 64 == 0 && Cout % 64 == 0 ? 1 : 0;
}

int tf32_supported(int dtype, int Cin, int Cout) {
    return dtype == VG_F32 && Cin % 32 == 0 && Cout % 32 == 0 ? 1 : 0;
}

size_t tc_packed_weight_bytes(int dtype, int Kdim, int Ndim) {
    return (size_t)kTaps * Kdim * Ndim * (dtype == VG_F32 ? 4 : 2);
}

int tc_pack_weights(const void* W, int dtype, int Cin, int Cout, int mode, int taps, void* packed,
                    const uint32_t* nbr_status, cudaStream_t s) {
    (void)nbr_status;
    const int Kdim = mode ? Cout : Cin, Ndim = mode ? Cin : Cout;
    const int ke = dtype == VG_F32 ? 32 : 64;
    // mode 1 reads tap 26 - k for image tap k: all 27 taps; otherwise the kernel's taps
    const dim3 grid(mode == 1 ? kTaps : taps, Kdim / ke, Ndim / 32);
    if (dtype == VG_F32)
        k_pack_weights<float><<<grid, 256, 0, s>>>(static_cast<const float*>(W), Cin, Cout, mode,
                                                   choose_bn(Ndim), static_cast<uint8_t*>(packed));
    else
        k_pack_weights<uint16_t><<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(W), Cin, Cout, mode,
                                                      choose_bn(Ndim), static_cast<uint8_t*>(packed));
    return VG_OK;
}

int tc_gather_pass(const GatherPass& p, const void* packed, cudaStream_t s) {
    if (p.n == 0) return VG_OK;
    if (p.dtype != VG_F32 && p.bias && p.Ndim > kMaxBiasCols) return VG_ERR_UNSUPPORTED;
    TcArgs a;
    a.sorted_idx = p.sorted_idx;
    a.tile_mask = p.tile_mask;
    a.sorted_nbr = p.sorted_nbr;
    a.nbr_status = p.nbr_status;
    a.n = p.n;
    a.num_tiles = (p.n + kBM - 1) / kBM;
    a.A = static_cast<const uint8_t*>(p.A);
    a.Kdim = p.Kdim;
    a.Bimg = static_cast<const uint8_t*>(packed);
    a.bias = p.bias;
    a.out = static_cast<uint8_t*>(p.out);
    a.Ndim = p.Ndim;
    a.ksplit = p.ksplit > 1 ? p.ksplit : 1;
    a.partial = p.partial;
    a.err = p.err;
    if (a.ksplit > 1 && !a.partial) return VG_ERR_INVALID_ARG;
    const int bn = choose_bn(p.Ndim);
    int st;
    if (pair_tiles(a.num_tiles, p.Ndim, a.ksplit, plan_sms(0))) {
        st = p.dtype == VG_F32    ? launch_pair<kTF32>(a, s)
             : p.dtype == VG_BF16 ? launch_pair<kBF16>(a, s)
                                  : launch_pair<kF16>(a, s);
    } else if (p.dtype == VG_F32) {
        switch (bn) {
            case 256: st = launch_tc<256, kTF32>(a, s); break;
            case 128: st = launch_tc<128, kTF32>(a, s); break;
            case 64: st = launch_tc<64, kTF32>(a, s); break;
            default: st = launch_tc<32, kTF32>(a, s); break;
        }
    } else {
        if (bn < 64) return VG_ERR_UNSUPPORTED;
        const bool bf16 = p.dtype == VG_BF16;
        switch (bn) {
            case 256: st = bf16 ? launch_tc<256, kBF16>(a, s) : launch_tc<256, kF16>(a, s); break;
            case 128: st = bf16 ? launch_tc<128, kBF16>(a, s) : launch_tc<128, kF16>(a, s); break;
            default: st = bf16 ? launch_tc<64, kBF16>(a, s) : launch_tc<64, kF16>(a, s); break;
        }
    }
    if (st != VG_OK || a.ksplit == 1) return st;
    const int sms = plan_sms(0);
    if (p.dtype == VG_F32) launch_split_reduce<float>(a, sms, s);
    else if (p.dtype == VG_BF16) launch_split_reduce<__nv_bfloat16>(a, sms, s);
    else launch_split_reduce<__half>(a, sms, s);
    return VG_OK;
}

// weight repack, gather GEMM (+ the split reduce when the pass is cut into tap groups)
int tc_fwd_launches(int ksplit) { return ksplit > 1 ? 3 : 2; }

}  // namespace vg
