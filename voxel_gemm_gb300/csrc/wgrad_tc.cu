// Tensor-core (tcgen05 / TMEM) weight gradient, split-K over the sorted rows.
//
// dW[k][ci][co] = sum_i f[nbr[i][k]][ci] * dY[i][co]: the backward of the
// masked implicit GEMM with Split-K ("Contribution Tasks — JeffreyXiang/FlexGEMM",
// §二 key types table: sparse_submanifold_conv_bwd_masked_implicit_gemm_splitk,
// split-K "reduces the accumulation bottleneck for large K"; here K is the
// voxel count).
//
// One MMA tile: D[128 x BN] in TMEM (two per work unit, sharing each dY stage),
// D[m][n] += sum over 64-row stages of
//   A[m][row] = f[nbr[row][tap(m)]][ci(m)]   (gathered feature rows)
//   B[n][row] = dY[row][co0 + n]
// Both operands are stored as rows of the sorted order, i.e. MN-major: a row
// holds 64 consecutive channels (128 B, swizzled).  M = 128 covers two 64-channel
// blocks, each a (tap, 64 channels) slot; slots are paired in tap-major order.
// A work unit = (M block, N block, row chunk); a row chunk is a range of the
// tile visiting order (the sorted row tiles regrouped by spatial region, so a
// chunk's gathers stay within a few regions of the grid), and a chunk's tiles
// whose tile mask has none of the unit's taps are skipped (their A rows would be zero).
// Each unit writes an fp32 partial [128 x BN] for its chunk; a second kernel sums
// the chunks in a fixed order (bitwise deterministic).
//
// Persistent CTAs, one per SM (two at narrow tiles, see WCfg below).
// Warp roles as in the forward kernel: warps 0-3 gather A with 16-byte cp.async
// (zero fill; each thread's copies arrive on the stage barrier by themselves),
// warp 4 issues tcgen05.mma, warps 5-8 store the partials.  B (dY) rows are
// consecutive sorted rows: for Cout >= 128 they are first copied into
// processing order as the B-operand image (one streaming pass, fused with the
// bias gradient's partial sums), so that each stage's B tile is one contiguous
// bulk copy (measured at C = 1024: 10.9 ms with four 2D tensor-map tile loads
// per stage); for Cout = 64 the gather threads fetch them with cp.async as well.
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace vg {

namespace {

using namespace ptx;


// Work units are handed out dynamically: thread 0 of the gather warps claims the
// next unit from a global counter and publishes it in a 4-slot ring that the
// gather, MMA and epilogue roles read in order (-1 ends the sequence).  A CTA
// whose units hold sparse taps (few active tiles) thus takes more units; with
// the fixed round-robin the busiest CTA had 18 % more tap-tiles than the mean
// (602k voxels, C = 1024).  Unit u = nb + NB * (mg + MG * chunk): the units
// claimed one after the other are the N blocks of one M group, which gather
// the same A rows while they are in L2 (measured at C = 1024: 11.77 ms, against
// 13.65 ms with the M groups of one N block next to each other).
constexpr int kUnitRing = 4;
// readers of each unit-ring slot: the gather warps, the MMA thread, the epilogue warps

// One CTA work unit holds MU M blocks (MU accumulators of 128 x BN side by side
// in TMEM, all sharing every dY stage) and streams stages of R sorted rows:
//   Cout = 64: MU = 7 (448 columns), R = 32;  Cout >= 128: MU = 2, R = 64.
// The larger MU, the fewer times dY is re-read (measured: 7 blocks at Cout = 64
// cut DRAM reads from 7.0 to about 2 GB at 4.9 M voxels; 4 blocks at Cout = 128
// were slower than 2).
// TWO = two CTAs per SM, each with half the stages and one accumulator buffer, so
// that one CTA's MMAs run while the other's epilogue or gather waits.  Always at
// Cout = 128 (measured at 319k voxels: 0.447 -> 0.384 ms); at Cout = 64 only when
// the MU = 7 units cannot fill the SMs, with MU = 3 (25k voxels: 0.061 -> 0.054 ms;
// at 4.9 M voxels MU = 3 re-reads dY more often and took 2.96 instead of 2.48 ms).
template <int BN, bool TWO>
struct WCfg {
    static constexpr int MU = BN == 64 ? (TWO ? 3 : 7) : 2;
    static constexpr int R = BN == 64 ? 32 : 64;           // rows per stage (K of the MMA)
    // gather warps: eight at 256 columns, where two M blocks share each 32 KB dY tile
    // (602k voxels, C = 1024: 10.62 ms with four, 10.35 with eight, 11.06 with
    // sixteen); four elsewhere (eight at C = 64, 4.9 M voxels: 2.17 -> 2.49 ms)
    static constexpr int GW = BN == 256 && !TWO ? 8 : 4;
    static constexpr int kThreads = (GW + 1 + 4) * 32;      // gather, MMA, epilogue warps
    static constexpr int kUnitReaders = GW + 1 + 4;
    static constexpr int RSTEP = GW * 4;                    // rows between one gather thread's rows
    static constexpr int RQ = R / RSTEP;                    // rows per gather thread
    static constexpr int kAccCols = MU * BN;
    static constexpr int NBUF = TWO ? 1 : (2 * kAccCols <= 512 ? 2 : 1);
    static constexpr int kTmemCols = NBUF * kAccCols <= 256 ? 256 : 512;
    static constexpr int kABytes = 2 * R * 128;             // two 64-channel blocks x R rows
    static constexpr int kBBytes = (BN / 64) * R * 128;
    static constexpr int kStageBytes = MU * kABytes + kBBytes;
    static constexpr int S = (TWO ? 98304 : 196608) / kStageBytes;  // 96 or 192 KB of stages
    // full[S], empty[S], tfull[2], tempty[2], done, unit ring full[4] and empty[4]
    static constexpr int kNumBars = 2 * S + 13;
    static constexpr size_t kSmem = 1024 + (size_t)S * kStageBytes + 8 * kNumBars + 8 * kUnitRing + 4 * S + 16;
    static_assert(!TWO || (kTmemCols <= 256 && 2 * kSmem <= 232448), "two CTAs must fit one SM");
};

struct WgArgs {
    const uint32_t* sorted_idx;
    const uint32_t* tile_mask;
    const uint32_t* tile_order;  // position -> tile
    const uint32_t* sorted_nbr;
    const uint32_t* nbr_status;
    int64_t n;
    int64_t num_tiles;
    int64_t tiles_per_chunk;
    int splits;
    const uint16_t* f;
    const uint16_t* dy;
    const uint16_t* dy_img;  // dY in processing order as the B-operand image (Cout >= 128)
    int Cin, Cout;
    int taps;        // taps of the kernel (27, or 8): (tap, channel block) slots of the M blocks
    float* partial;  // [splits][27][Cin][Cout]
    uint32_t* err;
    uint32_t* unit_ctr;  // next unit to claim (zero before the launch)
};

// Taps and channel offsets of M block m.  The 27 * (Cin/64) (tap, 64-channel
// block) slots, tap-major, are taken two at a time: slots 2m and 2m+1.  With
// Cin = 64 that pairs two taps; with Cin a multiple of 128 it is 128 channels of
// one tap; otherwise a pair may straddle two taps.
struct MUnit {
    int tap0, tap1;  // tap1 = -1: the second 64-channel block is unused (zero)
    int c0, c1;
};
__host__ __device__ __forceinline__ int num_munits(int Cin, int taps) { return (taps * (Cin / 64) + 1) / 2; }
__device__ __forceinline__ MUnit munit(int m, int Cin, int taps) {
    const int CB = Cin / 64;
    const int s0 = 2 * m, s1 = 2 * m + 1;
    MUnit r;
    if (s0 >= taps * CB) {  // past the last slot (a partial group of M blocks): all zero
        r.tap0 = r.tap1 = -1;
        r.c0 = r.c1 = 0;
        return r;
    }
    r.tap0 = s0 / CB;
    r.c0 = (s0 % CB) * 64;
    if (s1 < taps * CB) {
        r.tap1 = s1 / CB;
        r.c1 = (s1 % CB) * 64;
    } else {
        r.tap1 = -1;
        r.c1 = 0;
    }
    return r;
}

// Row metadata a gather thread needs for one stage (its RQ rows): the dY row
// and, for each of the unit's MU M blocks, the neighbour rows of its two taps.
template <int MU, int RQ>
struct Meta {
    uint32_t i[RQ], j0[MU][RQ], j1[MU][RQ];
};

// The dY row index is needed only when the gather threads fetch B themselves (WANT_I).
template <int MU, int RQ, int RSTEP, bool WANT_I>
__device__ __forceinline__ void load_meta(const WgArgs& a, const MUnit (&mu)[MU], int64_t row0, int p,
                                          Meta<MU, RQ>& m) {
#pragma unroll
    for (int q = 0; q < RQ; ++q) {
        const int64_t r = row0 + (p >> 3) + RSTEP * q;  // r < num_tiles * 128 always
        if (WANT_I) m.i[q] = r < a.n ? a.sorted_idx[r] : kNone;
#pragma unroll
        for (int u = 0; u < MU; ++u) {
            m.j0[u][q] = mu[u].tap0 >= 0 ? a.sorted_nbr[r * kTaps + mu[u].tap0] : kNone;
            m.j1[u][q] = mu[u].tap1 >= 0 ? a.sorted_nbr[r * kTaps + mu[u].tap1] : kNone;
        }
    }
}

// Walks the active tiles of one chunk (positions [base, end) of the tile visiting
// order), 32 positions per warp-wide load.
struct TileCursor {
    int64_t base, end;
    uint32_t bits;  // active positions in [base, base + 32) not yet returned
};
__device__ __forceinline__ uint32_t window_bits(const WgArgs& a, int64_t base, int64_t end, int64_t first,
                                                uint32_t umask, int lane) {
    const int64_t pos = base + lane;
    bool act = false;
    if (pos < end) act = (a.tile_mask[a.tile_order[pos]] & umask) != 0u || pos == first;
    return __ballot_sync(0xffffffffu, act);
}
// Tile index of the next active position (or -1); all lanes of the warp call it together.
__device__ __forceinline__ int64_t next_tile(const WgArgs& a, TileCursor& c, int64_t first, uint32_t umask,
                                             int lane) {
    while (c.bits == 0u) {
        c.base += 32;
        if (c.base >= c.end) return -1;
        c.bits = window_bits(a, c.base, c.end, first, umask, lane);
    }
    const int b = __ffs(c.bits) - 1;
    c.bits &= c.bits - 1u;
    return (int64_t)a.tile_order[c.base + b];
}

// Row r of dst = src[sorted_idx[r]] for r < n, zero rows up to rows_pad (16-bit
// rows of C values), stored as the B-operand image (dy_image_offset).
__global__ void __launch_bounds__(256)
k_sort_rows(const uint16_t* __restrict__ src, const uint32_t* __restrict__ sorted_idx, int64_t n, int64_t rows_pad,
            int C, const uint32_t* __restrict__ nbr_status, uint16_t* __restrict__ dst) {
    if (*nbr_status) return;
    const int cpr = C / 8;  // 16-byte chunks per row
    const int64_t total = rows_pad * cpr;
    for (int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x; e < total; e += (int64_t)gridDim.x * 256) {
        const int64_t r = e / cpr;
        const int c = (int)(e - r * cpr);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < n) v = reinterpret_cast<const uint4*>(src + (int64_t)sorted_idx[r] * C)[c];
        *reinterpret_cast<uint4*>(dst + dy_image_offset(r, c, C)) = v;
    }
}

// Warp-wide read of unit-ring slot `slot` (phase parity uph); lane 0 then releases
// the slot.  -1 when the sequence has ended or the wait gave up.
__device__ __forceinline__ int64_t read_unit(const volatile int64_t* s_unit, uint32_t ufull0, uint32_t uempty0,
                                             uint32_t slot, uint32_t uph, int lane, const volatile uint32_t* abort) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(ufull0 + 8 * slot, uph, abort));
    const int64_t u = ok ? s_unit[slot] : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(uempty0 + 8 * slot);
    return u;
}

template <int BN, bool BF16, bool TWO>
__global__ void __launch_bounds__(WCfg<BN, TWO>::kThreads, TWO ? 2 : 1) k_wgrad_tc(WgArgs a) {
    // B by one bulk copy from the dY image when the tile is wide (R = 64 rows)
    constexpr bool kImgB = BN >= 128;
    static_assert(!kImgB || WCfg<BN, TWO>::R == 64, "one image row group per stage");
    // row metadata two stages ahead with four gather warps (their threads carry twice
    // the rows), one stage ahead with two CTAs per SM (no registers for a third) and
    // with eight gather warps (measured at 602k voxels: C = 1024 10.44 -> 10.33 ms,
    // C = 256 0.970 -> 0.959 ms against two ahead; C = 64 at 4.9 M voxels with four
    // warps: 2.17 ms two ahead, 2.55 ms one ahead)
    using C = WCfg<BN, TWO>;
    constexpr bool kDeep = !TWO && C::GW == 4;
    constexpr int S = C::S;
    constexpr int MU = C::MU;
    constexpr int GW = C::GW;  // gather warps; then the MMA warp, then four epilogue warps
    constexpr int NBUF = C::NBUF;
    constexpr int R = C::R, RQ = C::RQ;
    constexpr int NBB = BN / 64;  // 64-column blocks of B
    constexpr int kABytes = C::kABytes;
    constexpr uint32_t kBlk = R * 128;  // bytes of one 64-channel block of R rows
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;  // stage g: MU A tiles, then the B tile
    uint64_t* bars = reinterpret_cast<uint64_t*>(stages + (size_t)S * C::kStageBytes);
    volatile int64_t* s_unit = reinterpret_cast<volatile int64_t*>(bars + C::kNumBars);  // unit ring
    uint32_t* s_info = reinterpret_cast<uint32_t*>(bars + C::kNumBars + kUnitRing);  // per stage: bit0 first, bit1 last
    uint32_t* s_tmem = s_info + S;
    volatile uint32_t* s_abort = s_tmem + 1;

    if (*a.nbr_status) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t tfull0 = smem_u32(bars + 2 * S), tempty0 = smem_u32(bars + 2 * S + 2);
    const uint32_t done_bar = smem_u32(bars + 2 * S + 4);
    const uint32_t ufull0 = smem_u32(bars + 2 * S + 5), uempty0 = smem_u32(bars + 2 * S + 5 + kUnitRing);
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full0 + 8 * i, GW * 32 + 1);  // the gather threads' copy arrivals + thread 0's info arrival
            mbar_init(empty0 + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull0 + 8 * i, 1);
            mbar_init(tempty0 + 8 * i, 4);
        }
        mbar_init(done_bar, 1);
        for (int i = 0; i < kUnitRing; ++i) {
            mbar_init(ufull0 + 8 * i, 1);             // thread 0's publication of the slot
            mbar_init(uempty0 + 8 * i, C::kUnitReaders);  // every reader of the slot
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == GW) {
        tmem_alloc(smem_u32(s_tmem), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    const int M = num_munits(a.Cin, a.taps);
    const int MG = (M + MU - 1) / MU;  // groups of MU M blocks
    const int NB = a.Cout / BN;
    const int64_t units = (int64_t)MG * NB * a.splits;

    if (warp < GW) {
        // ------------------------------------------------------------ gather producer
        const int p = threadIdx.x;
        const int ch = p & 7;
        uint32_t it = 0;
        bool ok = true;
        for (uint32_t q = 0; ok; ++q) {
            const uint32_t slot = q % kUnitRing, uph = (q / kUnitRing) & 1u;
            if (p == 0) {  // claim the next unit once every reader is done with the slot's last one
                const bool free_slot = mbar_wait(uempty0 + 8 * slot, uph ^ 1u, s_abort);
                // the first unit of every CTA is blockIdx.x (grid <= units); later ones are claimed
                const int64_t uu = !free_slot ? units
                                   : q == 0 ? (int64_t)blockIdx.x
                                            : (int64_t)gridDim.x + (int64_t)atomicAdd(a.unit_ctr, 1u);
                s_unit[slot] = uu < units ? uu : -1;
                mbar_arrive(ufull0 + 8 * slot);
            }
            const int64_t u = read_unit(s_unit, ufull0, uempty0, slot, uph, lane, s_abort);
            if (u < 0) break;
            const int nb = (int)(u % NB);  // the N blocks of one M group next to each other: they share A
            const int64_t rest = u / NB;
            const int mg = (int)(rest % MG);
            const int64_t s = rest / MG;
            MUnit mu[MU];
            uint32_t umask = 0;
#pragma unroll
            for (int v = 0; v < MU; ++v) {
                mu[v] = munit(mg * MU + v, a.Cin, a.taps);
                if (mu[v].tap0 >= 0) umask |= 1u << mu[v].tap0;
                if (mu[v].tap1 >= 0) umask |= 1u << mu[v].tap1;
            }
            const int64_t t_first = s * a.tiles_per_chunk;
            TileCursor cur;
            cur.base = t_first;
            cur.end = min(a.num_tiles, t_first + a.tiles_per_chunk);
            cur.bits = window_bits(a, cur.base, cur.end, t_first, umask, lane);
            // Row metadata is loaded ahead of the copies that use it (kDeep: two stages;
            // with four gather warps and one stage ahead the loads' latency set the pace:
            // the MMA thread waited for full stages 46 % of its time at C = 1024; two
            // ahead: C = 1024 11.92 -> 10.95 ms, C = 256 1.30 -> 1.18 ms).
            // (t0, h0): this stage's tile and R-row part; (t1, h1): the next stage's.
            auto advance = [&](int64_t t, int h, int64_t& tn, int& hn) {
                tn = t;
                hn = h + 1;
                if (hn == 128 / R) {
                    tn = next_tile(a, cur, t_first, umask, lane);
                    hn = 0;
                }
            };
            int64_t t0 = next_tile(a, cur, t_first, umask, lane);  // the first tile is always active
            int h0 = 0;
            Meta<MU, RQ> m0, m1, m2;
            bool null_stage = false;
            int64_t t1 = -1;
            int h1 = 0;
            if (t0 >= 0) {
                load_meta<MU, RQ, C::RSTEP, !kImgB>(a, mu, t0 * 128, p, m0);
                advance(t0, h0, t1, h1);
                if (kDeep && t1 >= 0) load_meta<MU, RQ, C::RSTEP, !kImgB>(a, mu, t1 * 128 + h1 * R, p, m1);
            } else {  // empty chunk (the host never makes one): one all-zero stage keeps roles in step
                null_stage = true;
                for (int q = 0; q < RQ; ++q) {
                    m0.i[q] = kNone;
                    for (int v = 0; v < MU; ++v) m0.j0[v][q] = m0.j1[v][q] = kNone;
                }
            }
            bool first = true;
            while (t0 >= 0 || null_stage) {
                null_stage = false;
                int64_t t2 = -1;
                int h2 = 0;
                if (t1 >= 0) advance(t1, h1, t2, h2);
                if constexpr (kDeep) {
                    if (t2 >= 0) load_meta<MU, RQ, C::RSTEP, !kImgB>(a, mu, t2 * 128 + h2 * R, p, m2);
                } else {
                    if (t1 >= 0) load_meta<MU, RQ, C::RSTEP, !kImgB>(a, mu, t1 * 128 + h1 * R, p, m1);
                }
                const int64_t t = t0, tn = t1;
                const int h = h0;
                const Meta<MU, RQ>& mc = m0;
                const uint32_t stage = it % S, ph = (it / S) & 1u;
                // warp-uniform decision: the tile cursor uses warp-wide ballots
                if (!__all_sync(0xffffffffu, mbar_wait(empty0 + 8 * stage, ph ^ 1u, s_abort))) {
                    ok = false;
                    *s_abort = 1;
                    break;
                }
                uint8_t* st = stages + (size_t)stage * C::kStageBytes;
                if (p == 0) {  // published by thread 0's own release arrival below
                    s_info[stage] = (first ? 1u : 0u) | (tn < 0 ? 2u : 0u);
                    if constexpr (kImgB) {
                        const uint32_t bytes = t >= 0 ? NBB * kBlk : 0u;
                        mbar_arrive_expect_tx(full0 + 8 * stage, bytes);
                        if (t >= 0)  // rows t * 128 + h * 64 .. + 63: row group 2t + h; channel blocks nb * NBB ..
                            bulk_g2s(smem_u32(st + MU * kABytes),
                                     a.dy_img + ((2 * t + h) * (a.Cout / 64) + nb * NBB) * (int64_t)(kBlk / 2), bytes,
                                     full0 + 8 * stage);
                    } else {
                        mbar_arrive(full0 + 8 * stage);
                    }
                }
#pragma unroll
                for (int v = 0; v < MU; ++v) {
                    const uint32_t a_base = smem_u32(st + v * kABytes);
#pragma unroll
                    for (int e = 0; e < 2 * RQ; ++e) {  // A: block e / RQ, row (p>>3) + RSTEP*(e % RQ)
                        const int q = e % RQ, blk = e / RQ;
                        const int row = (p >> 3) + C::RSTEP * q;
                        const uint32_t j = blk ? mc.j1[v][q] : mc.j0[v][q];
                        const int c = blk ? mu[v].c1 : mu[v].c0;
                        const uint16_t* src = a.f + (int64_t)(j != kNone ? j : 0u) * a.Cin + c + ch * 8;
                        cp_async16(a_base + blk * kBlk + (row >> 3) * 1024 + (row & 7) * 128 + ((ch ^ (row & 7)) << 4),
                                   src, j != kNone ? 16u : 0u);
                    }
                }
                const uint32_t b_base = smem_u32(st + MU * kABytes);
#pragma unroll
                for (int e = 0; e < (kImgB ? 0 : NBB * RQ); ++e) {  // B: block e / RQ, the same rows
                    const int q = e % RQ, blk = e / RQ;
                    const int row = (p >> 3) + C::RSTEP * q;
                    const uint32_t i = mc.i[q];
                    // rows with none of the unit's taps contribute nothing: skip their dY bytes
                    bool use = false;
#pragma unroll
                    for (int v = 0; v < MU; ++v) use |= mc.j0[v][q] != kNone || mc.j1[v][q] != kNone;
                    use = use && i != kNone;
                    const uint16_t* src = a.dy + (int64_t)(use ? i : 0u) * a.Cout + nb * BN + blk * 64 + ch * 8;
                    cp_async16(b_base + blk * kBlk + (row >> 3) * 1024 + (row & 7) * 128 + ((ch ^ (row & 7)) << 4),
                               src, use ? 16u : 0u);
                }
                cp_async_arrive_noinc(full0 + 8 * stage);  // fires when this thread's copies land
                ++it;
                first = false;
                t0 = t1;
                h0 = h1;
                m0 = m1;
                t1 = t2;
                h1 = h2;
                if constexpr (kDeep) m1 = m2;
            }
        }
        cp_async_wait_all();
        if (!ok) atomicOr(a.err, kErrTimeout);
    } else if (warp == GW) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_mn(BF16, BN);
            constexpr uint32_t lbo = kBlk;  // distance between 64-channel blocks
            uint32_t it = 0, ua = 0;
            bool ok = true;
            for (uint32_t q = 0; ok; ++q, ++ua) {
                const uint32_t slot = q % kUnitRing, uph = (q / kUnitRing) & 1u;
                if (!mbar_wait(ufull0 + 8 * slot, uph, s_abort)) { ok = false; break; }
                const int64_t u = s_unit[slot];
                mbar_arrive(uempty0 + 8 * slot);
                if (u < 0) break;
                const uint32_t buf = ua % NBUF;
                if (!mbar_wait(tempty0 + 8 * buf, ((ua / NBUF) & 1u) ^ 1u, s_abort)) { ok = false; break; }
                tc_fence_after();
                while (true) {
                    const uint32_t stage = it % S, ph = (it / S) & 1u;
                    if (!mbar_wait(full0 + 8 * stage, ph, s_abort)) { ok = false; break; }
                    fence_proxy_async_smem();  // cp.async (generic proxy) data read by the MMA (async proxy)
                    tc_fence_after();
                    const uint32_t info = s_info[stage];
                    const uint8_t* st = stages + (size_t)stage * C::kStageBytes;
                    const uint32_t b_base = smem_u32(st + MU * kABytes);
#pragma unroll
                    for (int v = 0; v < MU; ++v) {
                        const uint32_t a_base = smem_u32(st + v * kABytes);
                        const uint32_t d_tmem = tmem + buf * C::kAccCols + v * BN;
#pragma unroll
                        for (int j = 0; j < R / 16; ++j) {
                            mma_f16(d_tmem, sw128_mnmajor_desc(a_base + 2048 * j, lbo),
                                    sw128_mnmajor_desc(b_base + 2048 * j, lbo), idesc,
                                    ((info & 1u) && j == 0) ? 0u : 1u);
                        }
                    }
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
        for (uint32_t qi = 0;; ++qi, ++ua) {
            const int64_t u = read_unit(s_unit, ufull0, uempty0, qi % kUnitRing, (qi / kUnitRing) & 1u, lane, s_abort);
            if (u < 0) break;
            const int nb = (int)(u % NB);  // the N blocks of one M group next to each other: they share A
            const int64_t rest = u / NB;
            const int mg = (int)(rest % MG);
            const int64_t s = rest / MG;
            const uint32_t buf = ua % NBUF;
            ok = __all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * buf, (ua / NBUF) & 1u, s_abort));
            if (!ok) break;
            tc_fence_after();
            const int mrow = q * 32 + lane;  // M index: block mrow / 64, channel mrow % 64
            const int blk = mrow >> 6;
#pragma unroll 1
            for (int v = 0; v < MU; ++v) {
                const MUnit muv = munit(mg * MU + v, a.Cin, a.taps);
                const int tap = blk ? muv.tap1 : muv.tap0;
                const int ci = (blk ? muv.c1 : muv.c0) + (mrow & 63);
                float* dst = tap >= 0 ? a.partial + ((s * kTaps + tap) * a.Cin + ci) * (int64_t)a.Cout + nb * BN
                                      : nullptr;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    uint32_t acc[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + buf * C::kAccCols + v * BN + c0, acc);
                    tmem_ld_wait();
                    // 32 fp32 columns: one 128-byte line of this lane's row
                    store_lines_quad(dst ? reinterpret_cast<uint8_t*>(dst + c0) : nullptr, acc, lane, v8ok);
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
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == GW) tmem_dealloc(tmem, C::kTmemCols);
}

int wg_bn(int cout) {
    if (cout % 256 == 0) return 256;
    if (cout % 128 == 0) return 128;
    return 64;
}

template <int BN, bool BF16, bool TWO>
int launch_wgrad(const WgArgs& a, int sms, cudaStream_t s) {
    using C = WCfg<BN, TWO>;
    auto kern = k_wgrad_tc<BN, BF16, TWO>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem) != cudaSuccess)
        return VG_ERR_CUDA;
    if (BN >= 128 && !a.dy_img) return VG_ERR_INVALID_ARG;
    const int MG = (num_munits(a.Cin, a.taps) + C::MU - 1) / C::MU;
    const int64_t units = (int64_t)MG * (a.Cout / BN) * a.splits;
    const int grid = (int)std::min<int64_t>(units, (int64_t)(TWO ? 2 : 1) * sms);
    // with no more units than CTAs every claim returns >= gridDim.x >= units (the end),
    // whatever the counter holds: no reset needed
    if (units > grid) cudaMemsetAsync(a.unit_ctr, 0, sizeof(uint32_t), s);
    kern<<<grid, C::kThreads, C::kSmem, s>>>(a);
    return VG_OK;
}

// Split-K chunk count for M blocks of mu: about four work units per SM and
// chunks of at most 256 tiles (the units running side by side then stream the
// same rows through L2; measured at 602k voxels, C = 1024: 2 chunks 17.6 ms,
// 8 chunks 16.1 ms), at least 4 tiles per chunk (every chunk non-empty), partial
// sums capped at 768 MiB (at C = 1024: 6 chunks 13.79 ms, 4 chunks 13.89 ms,
// 9 chunks (1 GiB) 13.97 ms, 18 chunks 14.66 ms).
int64_t wgrad_splits_mu(int64_t n, int Cin, int Cout, int sms, int taps, int bn, int mu) {
    const int64_t T = std::max<int64_t>(1, (n + kTileRows - 1) / kTileRows);
    const int64_t MG = (num_munits(Cin, taps) + mu - 1) / mu;
    const int64_t per_split = MG * (Cout / bn);
    int64_t S = std::max<int64_t>(1, (4 * (int64_t)sms + per_split - 1) / per_split);
    S = std::max<int64_t>(S, (T + 255) / 256);
    if (bn == 256) {
        // Keep the rows of the chunks in flight (about sms / per_split of them side by
        // side) within 64 MiB, so that a chunk's units find its feature and dY rows in
        // L2 (measured at 602k voxels, C = 256: 23 chunks 1.13 ms with 32 % L2 hits and
        // 4.0 GB of DRAM reads, 46 chunks 0.99 ms, 74 chunks 0.99 ms; C = 512: 19 chunks
        // 2.98 ms, 27 chunks 2.92 ms)
        const int64_t in_flight = (sms + per_split - 1) / per_split;
        const int64_t chunk_bytes = in_flight * T * kTileRows * (int64_t)(Cin + Cout) * 2;
        S = std::max<int64_t>(S, (chunk_bytes + (int64_t(64) << 20) - 1) / (int64_t(64) << 20));
    }
    const int64_t bytes_per_split = (int64_t)kTaps * Cin * Cout * 4;
    S = std::min<int64_t>(S, std::max<int64_t>(1, (int64_t(3) << 28) / bytes_per_split));
    S = std::min<int64_t>(S, std::max<int64_t>(1, T / 4));
    const int64_t tpc = (T + S - 1) / S;
    return (T + tpc - 1) / tpc;
}

// Two CTAs per SM: always at 128 columns; at 64 columns when the MU = 7 units
// (M groups x chunks) number fewer than the SMs.
bool wgrad_two_cta(int64_t n, int Cin, int Cout, int sms, int taps) {
    const int bn = wg_bn(Cout);
    if (bn != 64) return bn == 128;
    const int64_t MG = (num_munits(Cin, taps) + WCfg<64, false>::MU - 1) / WCfg<64, false>::MU;
    return MG * (Cout / bn) * wgrad_splits_mu(n, Cin, Cout, sms, taps, bn, WCfg<64, false>::MU) < sms;
}

}  // namespace

int tc_wgrad_splits(int64_t n, int Cin, int Cout, int sms, int taps) {
    const int bn = wg_bn(Cout);
    const bool two = wgrad_two_cta(n, Cin, Cout, sms, taps);
    const int mu = bn == 64 ? (two ? WCfg<64, true>::MU : WCfg<64, false>::MU) : WCfg<256, false>::MU;
    return (int)wgrad_splits_mu(n, Cin, Cout, sms, taps, bn, mu);
}

size_t tc_wgrad_sorted_dy_bytes(int64_t n, int Cout) {
    if (wg_bn(Cout) < 128) return 0;
    const int64_t rows = (n + kTileRows - 1) / kTileRows * kTileRows;
    return (size_t)rows * Cout * 2;
}

int tc_wgrad(const WgradPass& p, cudaStream_t s) {
    if (p.n == 0) return VG_OK;
    bool db_done = false;
    if (p.dW) {
        WgArgs a;
        a.sorted_idx = p.sorted_idx;
        a.tile_mask = p.tile_mask;
        a.sorted_nbr = p.sorted_nbr;
        a.tile_order = p.tile_order;
        a.nbr_status = p.nbr_status;
        a.n = p.n;
        a.num_tiles = (p.n + kTileRows - 1) / kTileRows;
        a.splits = p.splits;
        a.tiles_per_chunk = (a.num_tiles + p.splits - 1) / p.splits;
        a.f = static_cast<const uint16_t*>(p.f);
        a.dy = static_cast<const uint16_t*>(p.dy);
        a.dy_img = static_cast<const uint16_t*>(p.dy_sorted);
        a.Cin = p.Cin;
        a.Cout = p.Cout;
        a.taps = p.taps;
        a.partial = p.partial;
        a.err = p.err;
        a.unit_ctr = p.err + kWgradUnitCounter;
        const bool bf16 = p.dtype == VG_BF16;
        const int bn = wg_bn(p.Cout);
        uint16_t* dys = static_cast<uint16_t*>(p.dy_sorted);
        if (bn >= 128) {
            if (!dys) return VG_ERR_INVALID_ARG;
            const int64_t rows_pad = a.num_tiles * kTileRows;
            if (p.db) {  // one read of dY: the copy into processing order and db's partial sums
                launch_dbias_sorted(p.dy, p.sorted_idx, p.n, rows_pad, p.Cout, p.sms, p.db, p.partial_db, dys,
                                    p.dtype, p.nbr_status, s);
                db_done = true;
            } else {
                const int64_t chunks = rows_pad * (p.Cout / 8);
                const unsigned blocks = (unsigned)std::min<int64_t>((chunks + 255) / 256, 16 * (int64_t)p.sms);
                k_sort_rows<<<blocks, 256, 0, s>>>(a.dy, p.sorted_idx, p.n, rows_pad, p.Cout, p.nbr_status, dys);
            }
        }
        int st;
        switch (bn) {
            case 256:
                st = bf16 ? launch_wgrad<256, true, false>(a, p.sms, s)
                          : launch_wgrad<256, false, false>(a, p.sms, s);
                break;
            case 128:
                st = bf16 ? launch_wgrad<128, true, true>(a, p.sms, s)
                          : launch_wgrad<128, false, true>(a, p.sms, s);
                break;
            default:
                if (wgrad_two_cta(p.n, p.Cin, p.Cout, p.sms, p.taps))
                    st = bf16 ? launch_wgrad<64, true, true>(a, p.sms, s)
                              : launch_wgrad<64, false, true>(a, p.sms, s);
                else
                    st = bf16 ? launch_wgrad<64, true, false>(a, p.sms, s)
                              : launch_wgrad<64, false, false>(a, p.sms, s);
                break;
        }
        if (st != VG_OK) return st;
        launch_reduce_splits(p.partial, p.splits, (int64_t)p.taps * p.Cin * p.Cout, (int64_t)kTaps * p.Cin * p.Cout,
                             p.dW, p.dtype, p.nbr_status, s);
    }
    if (p.db && !db_done) launch_dbias(p.dy, p.n, p.Cout, p.sms, p.db, p.partial_db, p.dtype, p.nbr_status, s);
    return VG_OK;
}

// dgrad (pack, gemm); Cout >= 128: dY into processing order with db's partial sums, wgrad gemm,
// split reduce, db reduce; Cout = 64: wgrad gemm, split reduce, db partials, db reduce
int tc_bwd_launches(int Cout) { return 2 + (wg_bn(Cout) >= 128 ? 3 + 1 : 2 + 2); }

}  // namespace vg
