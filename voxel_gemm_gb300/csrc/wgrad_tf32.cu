// TF32 tensor-core (tcgen05 kind::tf32) weight gradient for fp32 features, used
// when the caller allows TF32 (the pages' allow_tf32 switch, "From CUDA to
// Triton: Triton JIT and autotuning", §六 6.2; the split-K backward of
// "Contribution Tasks — JeffreyXiang/FlexGEMM", §二 key types table).
//
// dW[k][ci][co] = sum_r f[nbr[r][k]][ci] * dY[r][co] over the sorted rows r,
// split-K over chunks of the tile visiting order, fp32 partials per chunk, summed
// in a fixed order by k_reduce_splits (bitwise deterministic).
//
// Both MMA operands are kept K-major (K = voxel rows): the contraction runs over
// rows, while features and gradients are stored row-major, so the producer warps
// transpose on the way into shared memory.  Per stage of 32 rows, a lane loads
// four 16-byte pieces (4 channels) of four consecutive rows, transposes the 4x4
// block in registers and stores four 16-byte pieces (4 rows of one channel) into
// the 128-byte-swizzled K-major image; lanes are laid out so that those stores
// hit distinct bank groups.
//   A: M = 128 input channels of one tap (masked past Cin), K = 32 rows
//   B: N = BN output channels,                                K = 32 rows
// Warps 0-7 produce, warp 8 allocates TMEM and issues the MMAs (4 per stage,
// K = 8 each), warps 9-12 write the fp32 partials.  Every wait is bounded.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace vg {

namespace {

using namespace ptx;

constexpr int kProducerWarps = 8;  // (4 left one load latency per stage exposed: 2x slower)
constexpr int kMmaWarp = kProducerWarps;
constexpr int kThreads = (kProducerWarps + 1 + 4) * 32;
constexpr int kRows = 32;  // voxel rows per stage (one 128-byte K block of fp32)
constexpr int kBM = 128;   // input channels per unit

template <int BN>
struct TCfg {
    static constexpr int kABytes = kBM * 128;
    static constexpr int kBBytes = BN * 128;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int S = 196608 / kStageBytes < 8 ? 196608 / kStageBytes : 8;
    static constexpr int NBUF = 2;
    static constexpr int kTmemCols = NBUF * BN;
    static constexpr int kNumBars = 2 * S + 2 * NBUF + 1;
    static constexpr size_t kSmem = 1024 + (size_t)S * kStageBytes + 8 * kNumBars + 4 * S + 16;
};

struct T32Args {
    const uint32_t* sorted_idx;
    const uint32_t* tile_mask;
    const uint32_t* tile_order;
    const uint32_t* sorted_nbr;
    const uint32_t* nbr_status;
    int64_t n, num_tiles, tiles_per_chunk;
    int splits, taps;
    const float* f;
    const float* dy;
    int Cin, Cout;
    float* partial;  // [splits][27][Cin][Cout]
    uint32_t* err;
};

// Store the transpose of a 4x4 block: v[e] holds channels c..c+3 of row e; the
// image row of channel c + q gets (row 0..3) as one 16-byte piece at K chunk `kc`.
__device__ __forceinline__ void store_t4(uint8_t* img, int m0, int kc, const float4 (&v)[4]) {
    const float4 c0 = make_float4(v[0].x, v[1].x, v[2].x, v[3].x);
    const float4 c1 = make_float4(v[0].y, v[1].y, v[2].y, v[3].y);
    const float4 c2 = make_float4(v[0].z, v[1].z, v[2].z, v[3].z);
    const float4 c3 = make_float4(v[0].w, v[1].w, v[2].w, v[3].w);
    const float4 cs[4] = {c0, c1, c2, c3};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int m = m0 + q;
        *reinterpret_cast<float4*>(img + (m >> 3) * 1024 + (m & 7) * 128 + ((kc ^ (m & 7)) << 4)) = cs[q];
    }
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) k_wgrad_tf32(T32Args a) {
    using C = TCfg<BN>;
    constexpr int S = C::S;
    constexpr int NBUF = C::NBUF;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(stages + (size_t)S * C::kStageBytes);
    uint32_t* s_info = reinterpret_cast<uint32_t*>(bars + C::kNumBars);  // per stage: bit0 first, bit1 last
    uint32_t* s_tmem = s_info + S;
    volatile uint32_t* s_abort = s_tmem + 1;

    if (*a.nbr_status) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + NBUF);
    const uint32_t done_bar = smem_u32(bars + 2 * S + 2 * NBUF);
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full0 + 8 * i, kProducerWarps * 32);  // every producer thread
            mbar_init(empty0 + 8 * i, 1);   // one tcgen05.commit
        }
        for (int i = 0; i < NBUF; ++i) {
            mbar_init(tfull0 + 8 * i, 1);
            mbar_init(tempty0 + 8 * i, 4);
        }
        mbar_init(done_bar, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(s_tmem), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    const int MB = (a.Cin + kBM - 1) / kBM;
    const int NB = a.Cout / BN;
    const int64_t units = (int64_t)MB * a.taps * NB * a.splits;
    // unit u = mb + MB * (k + taps * (nb + NB * s))
    auto decode = [&](int64_t u, int& mb, int& k, int& nb, int64_t& s) {
        mb = (int)(u % MB);
        int64_t r = u / MB;
        k = (int)(r % a.taps);
        r /= a.taps;
        nb = (int)(r % NB);
        s = r / NB;
    };
    // the unit's tiles: positions [first, end) of the visiting order whose mask has
    // tap k; the first position always counts (so no unit is empty)
    auto next_active = [&](int64_t pos, int64_t first, int64_t end, int k) -> int64_t {
        for (; pos < end; ++pos)
            if (pos == first || ((a.tile_mask[a.tile_order[pos]] >> k) & 1u)) return pos;
        return -1;
    };

    if (warp < kProducerWarps) {
        // ------------------------------------------------------------ producers (transposing gather)
        const int p = threadIdx.x;
        const int rq = lane >> 2, cg = lane & 3;  // row quad (rows 4rq..4rq+3), channel group
        uint32_t it = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; u < units && ok; u += gridDim.x) {
            int mb, k, nb;
            int64_t s;
            decode(u, mb, k, nb, s);
            const int ci0 = mb * kBM, co0 = nb * BN;
            const int64_t first = s * a.tiles_per_chunk;
            const int64_t end = min(a.num_tiles, first + a.tiles_per_chunk);
            int64_t pos = next_active(first, first, end, k);
            bool first_stage = true;
            // Software pipeline: the row indices of a stage are loaded one stage ahead, and
            // a stage's data loads are all issued before its slot is waited for and before
            // any store (loads of independent rows in flight together; with the loads and
            // stores interleaved per 4x4 block the producers paced the pass, 0.03 of the
            // TF32 peak at C = 256).
            int64_t t = pos >= 0 ? a.tile_order[pos] : 0;
            int64_t npos = pos >= 0 ? next_active(pos + 1, first, end, k) : -1;
            int h = 0;
            uint32_t jn[4], in[4];  // this stage's neighbour rows (tap k) and dY rows
            auto load_idx = [&](int64_t tt, int hh, uint32_t (&jj)[4], uint32_t (&ii)[4]) {
                const int64_t rr = tt * 128 + hh * kRows + 4 * rq;  // < num_tiles * 128 always
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    jj[e] = a.sorted_nbr[(rr + e) * kTaps + k];
                    ii[e] = rr + e < a.n ? a.sorted_idx[rr + e] : kNone;
                }
            };
            if (pos >= 0) load_idx(t, 0, jn, in);
            while (pos >= 0 && ok) {
                // data of this stage
                constexpr int PW = kProducerWarps;
                constexpr int NAP = (kBM / 16 + PW - 1) / PW;  // A blocks of 16 channels per warp
                constexpr int NBP = (BN / 16 + PW - 1) / PW;   // B blocks per warp (at most)
                float4 va[NAP][4], vb[NBP][4];
#pragma unroll
                for (int P = 0; P < NAP; ++P) {
                    const int c = ci0 + (warp + PW * P) * 16 + cg * 4;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        va[P][e] = (jn[e] != kNone && c < a.Cin)
                                       ? __ldg(reinterpret_cast<const float4*>(a.f + (int64_t)jn[e] * a.Cin + c))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int P = 0; P < NBP; ++P) {
                    const int cl = (warp + PW * P) * 16 + cg * 4;
                    const bool blk = warp + PW * P < BN / 16;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        vb[P][e] = blk && in[e] != kNone
                                       ? __ldg(reinterpret_cast<const float4*>(a.dy + (int64_t)in[e] * a.Cout + co0 + cl))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                // the next stage's position and row indices
                const bool last = npos < 0 && h == 128 / kRows - 1;
                int64_t t_next = t, pos_next = pos, npos_next = npos;
                int h_next = h + 1;
                if (h_next == 128 / kRows) {
                    h_next = 0;
                    pos_next = npos;
                    if (pos_next >= 0) {
                        t_next = a.tile_order[pos_next];
                        npos_next = next_active(pos_next + 1, first, end, k);
                    }
                }
                if (!last) load_idx(t_next, h_next, jn, in);
                const uint32_t stage = it % S, ph = (it / S) & 1u;
                if (!mbar_wait(empty0 + 8 * stage, ph ^ 1u, s_abort)) {
                    ok = false;
                    *s_abort = 1;
                    break;
                }
                uint8_t* img_a = stages + (size_t)stage * C::kStageBytes;
                uint8_t* img_b = img_a + C::kABytes;
#pragma unroll
                for (int P = 0; P < NAP; ++P) store_t4(img_a, (warp + PW * P) * 16 + cg * 4, rq, va[P]);
#pragma unroll
                for (int P = 0; P < NBP; ++P)
                    if (warp + PW * P < BN / 16) store_t4(img_b, (warp + PW * P) * 16 + cg * 4, rq, vb[P]);
                if (p == 0) s_info[stage] = (first_stage ? 1u : 0u) | (last ? 2u : 0u);
                // (the MMA thread orders these generic-proxy stores before its async-proxy
                // reads with one proxy fence after the stage barrier, as for cp.async data)
                mbar_arrive(full0 + 8 * stage);
                ++it;
                first_stage = false;
                if (last) break;
                t = t_next;
                h = h_next;
                pos = pos_next;
                npos = npos_next;
            }
        }
        if (!ok) atomicOr(a.err, kErrTimeout);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_tf32(BN);
            uint32_t it = 0, ua = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; u < units && ok; u += gridDim.x, ++ua) {
                const uint32_t buf = ua % NBUF;
                if (!mbar_wait(tempty0 + 8 * buf, ((ua / NBUF) & 1u) ^ 1u, s_abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem + buf * BN;
                while (true) {
                    const uint32_t stage = it % S, ph = (it / S) & 1u;
                    if (!mbar_wait(full0 + 8 * stage, ph, s_abort)) { ok = false; break; }
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const uint32_t info = s_info[stage];
                    const uint32_t a_base = smem_u32(stages + (size_t)stage * C::kStageBytes);
                    const uint32_t b_base = a_base + C::kABytes;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_tf32(d_tmem, sw128_kmajor_desc(a_base + 32 * j), sw128_kmajor_desc(b_base + 32 * j),
                                 idesc, ((info & 1u) && j == 0) ? 0u : 1u);
                    mma_commit(empty0 + 8 * stage);
                    ++it;
                    if (info & 2u) break;
                }
                if (ok) mma_commit(tfull0 + 8 * buf);
            }
            mma_commit(done_bar);
            const bool drained = mbar_wait_timed(done_bar, 0);
            if (!ok || !drained) {
                *s_abort = 1;
                atomicOr(a.err, kErrTimeout);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue: fp32 partials
        const int q = warp & 3;
        const bool v8ok = (reinterpret_cast<uintptr_t>(a.partial) & 31u) == 0;
        uint32_t ua = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; u < units; u += gridDim.x, ++ua) {
            int mb, k, nb;
            int64_t s;
            decode(u, mb, k, nb, s);
            const uint32_t buf = ua % NBUF;
            ok = __all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * buf, (ua / NBUF) & 1u, s_abort));
            if (!ok) break;
            tc_fence_after();
            const int ci = mb * kBM + q * 32 + lane;
            float* dst = a.partial + ((s * kTaps + k) * a.Cin + ci) * (int64_t)a.Cout + nb * BN;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t acc[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + buf * BN + c0, acc);
                tmem_ld_wait();
                // 32 fp32 columns: one 128-byte line of this lane's row
                store_lines_quad(ci < a.Cin ? reinterpret_cast<uint8_t*>(dst + c0) : nullptr, acc, lane, v8ok);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * buf);
        }
        if (!ok) {
            *s_abort = 1;
            atomicOr(a.err, kErrTimeout);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
}

int tf32_bn(int cout) {
    if (cout % 256 == 0) return 256;
    if (cout % 128 == 0) return 128;
    if (cout % 64 == 0) return 64;
    return 32;
}

template <int BN>
int launch_tf32(const T32Args& a, int sms, cudaStream_t s) {
    using C = TCfg<BN>;
    auto kern = k_wgrad_tf32<BN>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem) != cudaSuccess)
        return VG_ERR_CUDA;
    const int64_t units = (int64_t)((a.Cin + kBM - 1) / kBM) * a.taps * (a.Cout / BN) * a.splits;
    const int grid = (int)std::min<int64_t>(units, sms);
    kern<<<grid, kThreads, C::kSmem, s>>>(a);
    return VG_OK;
}

}  // namespace

// Split-K chunks: about four units per SM, chunks of at most 256 tiles, at least
// 4 tiles per chunk, partial sums capped at 1 GiB (as the 16-bit kernel).
int tf32_wgrad_splits(int64_t n, int Cin, int Cout, int sms, int taps) {
    const int64_t T = std::max<int64_t>(1, (n + kTileRows - 1) / kTileRows);
    const int64_t per_split = (int64_t)((Cin + kBM - 1) / kBM) * taps * (Cout / tf32_bn(Cout));
    int64_t S = std::max<int64_t>(1, (4 * (int64_t)sms + per_split - 1) / per_split);
    S = std::max<int64_t>(S, (T + 255) / 256);
    const int64_t bytes_per_split = (int64_t)kTaps * Cin * Cout * 4;
    S = std::min<int64_t>(S, std::max<int64_t>(1, (int64_t(1) << 30) / bytes_per_split));
    S = std::min<int64_t>(S, std::max<int64_t>(1, T / 4));
    const int64_t tpc = (T + S - 1) / S;
    return (int)((T + tpc - 1) / tpc);
}

int tf32_wgrad(const WgradPass& p, cudaStream_t s) {
    if (p.n == 0) return VG_OK;
    if (p.dW) {
        T32Args a;
        a.sorted_idx = p.sorted_idx;
        a.tile_mask = p.tile_mask;
        a.tile_order = p.tile_order;
        a.sorted_nbr = p.sorted_nbr;
        a.nbr_status = p.nbr_status;
        a.n = p.n;
        a.num_tiles = (p.n + kTileRows - 1) / kTileRows;
        a.splits = p.splits;
        a.tiles_per_chunk = (a.num_tiles + p.splits - 1) / p.splits;
        a.taps = p.taps;
        a.f = static_cast<const float*>(p.f);
        a.dy = static_cast<const float*>(p.dy);
        a.Cin = p.Cin;
        a.Cout = p.Cout;
        a.partial = p.partial;
        a.err = p.err;
        int st;
        switch (tf32_bn(p.Cout)) {
            case 256: st = launch_tf32<256>(a, p.sms, s); break;
            case 128: st = launch_tf32<128>(a, p.sms, s); break;
            case 64: st = launch_tf32<64>(a, p.sms, s); break;
            default: st = launch_tf32<32>(a, p.sms, s); break;
        }
        if (st != VG_OK) return st;
        launch_reduce_splits(p.partial, p.splits, (int64_t)p.taps * p.Cin * p.Cout, (int64_t)kTaps * p.Cin * p.Cout,
                             p.dW, p.dtype, p.nbr_status, s);
    }
    if (p.db) launch_dbias(p.dy, p.n, p.Cout, p.sms, p.db, p.partial_db, p.dtype, p.nbr_status, s);
    return VG_OK;
}

}  // namespace vg
