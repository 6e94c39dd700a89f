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
// rows, while features and gradients are stored row-major.
//   B (dY): before the kernel, one streaming pass copies dY into processing order
//   as the B-operand image (tf32_dy_image_offset: per 32 sorted rows, each
//   channel's 32 values in a 128-byte swizzled row), fused with the bias
//   gradient's partial sums; a stage's B tile is then one contiguous bulk copy,
//   issued by a loader warp as soon as the stage's slot is free.
//   A (gathered features of one tap, 128 channels): the producer warps copy each
//   stage's 32 neighbour rows row-major into a staging ring with cp.async, several
//   stages ahead, then transpose each landed stage from shared memory into the
//   K-major image (4x4 blocks through registers; the staging rows are XOR-swizzled
//   so that both the copies and the transposing reads are free of bank conflicts).
//   A: M = 128 input channels of one tap (masked past Cin), K = 32 rows
//   B: N = BN output channels,                                K = 32 rows
// Warps 0-7 produce A, warp 8 allocates TMEM and issues the MMAs (4 per stage,
// K = 8 each), warps 9-12 write the fp32 partials, warp 13 loads B.  Units are
// taken N block first, so that the CTAs working side by side gather the same
// neighbour rows.  Every wait is bounded.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace vg {

namespace {

using namespace ptx;


constexpr int kProducerWarps = 8;
constexpr int kMmaWarp = kProducerWarps;       // warp 8
constexpr int kEpiWarp0 = kProducerWarps + 1;  // warps 9-12
constexpr int kLoaderWarp = kEpiWarp0 + 4;     // warp 13
constexpr int kThreads = (kLoaderWarp + 1) * 32;
constexpr int kProducers = kProducerWarps * 32;
constexpr int kRows = 32;  // voxel rows per stage (one 128-byte K block of fp32)
constexpr int kBM = 128;   // input channels per unit
constexpr int kStgBytes = kRows * kBM * 4;  // one staging slot: 32 rows x 128 channels, row-major (512 B rows)
constexpr int kUnitRingSlots = 4;

template <int BN>
struct TCfg {
    static constexpr int kABytes = kBM * 128;
    static constexpr int kBBytes = BN * 128;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int S = BN == 256 ? 3 : (BN == 128 ? 4 : 5);  // MMA operand stages
    static constexpr int D = BN == 256 ? 4 : 5;                     // staging slots (copies D - 1 stages ahead)
    static constexpr int NBUF = 2;
    static constexpr int kTmemCols = NBUF * BN;
    // full, empty, bfull; tfull, tempty; done; unit ring full and empty
    static constexpr int kNumBars = 3 * S + 2 * NBUF + 1 + 2 * kUnitRingSlots;
    static constexpr size_t kSmem = 1024 + (size_t)S * kStageBytes + (size_t)D * kStgBytes + 8 * kNumBars +
                                    8 * kUnitRingSlots + 4 * S + 16;
    static_assert(kSmem <= 232448, "TF32 weight-gradient stages exceed one CTA's shared memory");
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
    const float* dy_img;  // dY in processing order as the B-operand image (tf32_dy_image_offset)
    int Cin, Cout;
    float* partial;  // [splits][27][Cin][Cout]
    uint32_t* err;
    uint32_t* unit_ctr;  // next unit to claim (zero before the launch when units > grid)
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

// Byte offset, in a staging slot, of 16-byte chunk c (channels 4c..4c+3) of row r:
// chunk c ^ ((r / 4) % 8), so that the eight lanes of a transposing read (one
// chunk of row 4rq + e for rq = 0..7) cover all eight bank groups; a warp's copy
// of one row permutes the row's chunks.
__device__ __forceinline__ uint32_t stg_off(int r, int c) { return (uint32_t)(r * 512 + ((c ^ ((r >> 2) & 7)) << 4)); }

// Work units are handed out dynamically: the copy walker of producer warp 0
// claims the next unit from a global counter when it starts a unit and publishes
// it in a 4-slot ring (the CTA's first unit is blockIdx.x); every walker, the MMA
// thread and the epilogue warps read the ring in order (-1 ends the sequence).
// With the fixed round-robin the CTAs drifted apart over the chunks and L2 kept
// 22 % of the reads.
constexpr int kUnitRing = kUnitRingSlots;
constexpr int kUnitReaders = 2 * kProducerWarps + 1 + 1 + 4;  // producer walkers, loader, MMA thread, epilogue

struct Ring {
    volatile int64_t* slot;
    uint32_t full0, empty0;
    const volatile uint32_t* abort;
    uint32_t* ctr;
    int64_t units;
};

// Warp-wide read of ring entry qi (the whole warp calls it; lane 0 releases the
// slot).  timed: wait without looking at the abort flag (the producer warps must
// all see the same sequence; the claimer always publishes, -1 after a failure).
__device__ __forceinline__ int64_t ring_read(const Ring& R, uint32_t qi, int lane, bool timed) {
    const uint32_t slot = qi % kUnitRing, ph = (qi / kUnitRing) & 1u;
    const bool got = timed ? mbar_wait_timed(R.full0 + 8 * slot, ph) : mbar_wait(R.full0 + 8 * slot, ph, R.abort);
    const bool ok = __all_sync(0xffffffffu, got);
    const int64_t u = ok ? R.slot[slot] : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(R.empty0 + 8 * slot);
    return u;
}

// Single-thread read of ring entry qi (releases the slot).
__device__ __forceinline__ int64_t ring_read_one(const Ring& R, uint32_t qi) {
    const uint32_t slot = qi % kUnitRing;
    const int64_t u = mbar_wait(R.full0 + 8 * slot, (qi / kUnitRing) & 1u, R.abort) ? R.slot[slot] : -1;
    mbar_arrive(R.empty0 + 8 * slot);
    return u;
}

// Claim and publish ring entry qi (one thread).
__device__ __forceinline__ void ring_publish(const Ring& R, uint32_t qi) {
    const uint32_t slot = qi % kUnitRing;
    const bool free_slot = mbar_wait(R.empty0 + 8 * slot, ((qi / kUnitRing) & 1u) ^ 1u, R.abort);
    const int64_t uu = free_slot ? (int64_t)gridDim.x + (int64_t)atomicAdd(R.ctr, 1u) : R.units;
    R.slot[slot] = uu < R.units ? uu : -1;
    mbar_arrive(R.full0 + 8 * slot);
}

// Walk over the stages of the CTA's units: unit u = nb + NB * (mb + MB * (k + taps * s))
// (N blocks of one (M block, tap, chunk) next to each other), each unit the
// positions [first, end) of the tile visiting order whose tile mask has tap k (the
// first position always counts, so no unit is empty), four 32-row stages per tile.
// A whole warp walks together: the active positions are found 32 at a time (one
// load of tile id and mask per lane and a ballot), and the next active tile is
// looked up one tile ahead so that the last stage of a unit is known.
struct StageWalk {
    int64_t u, s, first, end, base;
    int64_t t, nt;      // this stage's tile; the unit's next active tile (-1: none)
    uint32_t bits;      // active positions in [base, base + 32) not yet taken
    uint32_t lane_tile; // tile id at position base + lane
    uint32_t qi;        // ring entry of the current unit
    int mb, k, nb, h;
    bool valid, first_stage, claims;
};

__device__ __forceinline__ void walk_window(StageWalk& w, const T32Args& a, int lane) {
    const int64_t pos = w.base + lane;
    bool act = false;
    w.lane_tile = 0;
    if (pos < w.end) {
        w.lane_tile = a.tile_order[pos];
        act = pos == w.first || ((a.tile_mask[w.lane_tile] >> w.k) & 1u);
    }
    w.bits = __ballot_sync(0xffffffffu, act);
}

// The unit's next active tile, or -1 (warp-uniform).
__device__ __forceinline__ int64_t walk_take(StageWalk& w, const T32Args& a, int lane) {
    while (w.bits == 0u) {
        w.base += 32;
        if (w.base >= w.end) return -1;
        walk_window(w, a, lane);
    }
    const int b = __ffs(w.bits) - 1;
    w.bits &= w.bits - 1u;
    return (int64_t)__shfl_sync(0xffffffffu, w.lane_tile, b);
}

// Start the unit of ring entry w.qi (the claiming walker first publishes the next one).
__device__ __forceinline__ void walk_unit(StageWalk& w, const T32Args& a, const Ring& R, int MB, int NB, int lane,
                                          bool timed) {
    w.u = ring_read(R, w.qi, lane, timed);
    w.valid = w.u >= 0;
    if (!w.valid) return;
    if (w.claims && lane == 0) ring_publish(R, w.qi + 1);
    w.nb = (int)(w.u % NB);
    int64_t r = w.u / NB;
    w.mb = (int)(r % MB);
    r /= MB;
    w.k = (int)(r % a.taps);
    w.s = r / a.taps;
    w.first = w.s * a.tiles_per_chunk;
    w.end = min(a.num_tiles, w.first + a.tiles_per_chunk);
    w.base = w.first;
    walk_window(w, a, lane);
    w.t = walk_take(w, a, lane);  // the first position always counts
    w.nt = walk_take(w, a, lane);
    w.h = 0;
    w.first_stage = true;
}

__device__ __forceinline__ bool walk_last(const StageWalk& w) { return w.h == 128 / kRows - 1 && w.nt < 0; }

__device__ __forceinline__ void walk_next(StageWalk& w, const T32Args& a, const Ring& R, int MB, int NB, int lane,
                                          bool timed) {
    w.first_stage = false;
    if (w.h + 1 < 128 / kRows) {
        ++w.h;
    } else if (w.nt >= 0) {
        w.t = w.nt;
        w.nt = walk_take(w, a, lane);
        w.h = 0;
    } else {
        ++w.qi;
        walk_unit(w, a, R, MB, NB, lane, timed);
    }
}

// bar.red.or over the named barrier: every participant gets the OR of the predicates.
__device__ __forceinline__ bool named_bar_any(uint32_t id, uint32_t threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) k_wgrad_tf32(T32Args a) {
    using C = TCfg<BN>;
    constexpr int S = C::S, D = C::D, NBUF = C::NBUF;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;                                     // [S][A image | B image]
    uint8_t* stg = smem + (size_t)S * C::kStageBytes;           // [D][32 rows x 512 B], row-major
    uint64_t* bars = reinterpret_cast<uint64_t*>(stg + (size_t)D * kStgBytes);
    volatile int64_t* s_unit = reinterpret_cast<volatile int64_t*>(bars + C::kNumBars);  // unit ring
    uint32_t* s_info = reinterpret_cast<uint32_t*>(bars + C::kNumBars + kUnitRing);  // per stage: bit0 first, bit1 last
    uint32_t* s_tmem = s_info + S;
    volatile uint32_t* s_abort = s_tmem + 1;

    if (*a.nbr_status) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // full: the producers' A image; bfull: the loader's B tile (transaction bytes)
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S), bfull0 = smem_u32(bars + 2 * S);
    const uint32_t tfull0 = smem_u32(bars + 3 * S), tempty0 = smem_u32(bars + 3 * S + NBUF);
    const uint32_t done_bar = smem_u32(bars + 3 * S + 2 * NBUF);
    const uint32_t ufull0 = smem_u32(bars + 3 * S + 2 * NBUF + 1), uempty0 = ufull0 + 8 * kUnitRing;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full0 + 8 * i, kProducers);  // every producer thread
            mbar_init(empty0 + 8 * i, 1);          // one tcgen05.commit
            mbar_init(bfull0 + 8 * i, 1);          // the loader's expect_tx
        }
        for (int i = 0; i < NBUF; ++i) {
            mbar_init(tfull0 + 8 * i, 1);
            mbar_init(tempty0 + 8 * i, 4);
        }
        mbar_init(done_bar, 1);
        for (int i = 0; i < kUnitRing; ++i) {
            mbar_init(ufull0 + 8 * i, 1);
            mbar_init(uempty0 + 8 * i, kUnitReaders);
        }
        *s_abort = 0;
        fence_mbar_init();
        s_unit[0] = (int64_t)blockIdx.x;  // the first unit of every CTA (grid <= units)
        mbar_arrive(ufull0);
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
    Ring R;
    R.slot = s_unit;
    R.full0 = ufull0;
    R.empty0 = uempty0;
    R.abort = s_abort;
    R.ctr = a.unit_ctr;
    R.units = units;

    if (warp < kProducerWarps) {
        // ------------------------------------------------------------ producers: copy, then transpose
        // Stage i: (1) this thread's copies of stage i have landed (cp.async groups
        // are committed one per stage, D - 1 stages ahead) and a barrier over the
        // producers makes everyone's visible -- and tells that everyone has finished
        // transposing stage i - 1, whose staging slot the copies of stage i + D - 1
        // then reuse; (2) transpose stage i into its operand slot once the MMAs of
        // stage i - S are done.  All producers walk the same stages and meet at the
        // same barriers; a failed wait ends the loop for all of them at the next one.
        const int p = threadIdx.x;
        const int rq = lane & 7, cg = lane >> 3;  // transpose: rows 4rq..4rq+3, channels 16 * warp + 4cg..
        bool ok = true;
        StageWalk wc, wt;  // copy walker (D - 1 stages ahead; warp 0's claims the units) and transpose walker
        wc.qi = wt.qi = 0;
        wc.claims = warp == 0;
        wt.claims = false;
        walk_unit(wc, a, R, MB, NB, lane, true);
        walk_unit(wt, a, R, MB, NB, lane, true);
        uint32_t jn[4];  // neighbour rows (tap k) of this warp's rows warp + 8q of the copy walker's stage
        auto load_idx = [&]() {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t r = wc.t * 128 + wc.h * kRows + warp + 8 * q;  // < num_tiles * 128 always
                jn[q] = wc.valid ? a.sorted_nbr[r * kTaps + wc.k] : kNone;
            }
        };
        auto issue = [&](uint32_t j) {  // the copies of stage j (the copy walker's), then advance it
            if (wc.valid) {
                const uint32_t base = smem_u32(stg + (size_t)(j % D) * kStgBytes);
                const int ch = wc.mb * kBM + 4 * lane;
                const bool cv = ch < a.Cin;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const bool v = cv && jn[q] != kNone;
                    const float* src = a.f + (int64_t)(v ? jn[q] : 0u) * a.Cin + (cv ? ch : 0);
                    cp_async16(base + stg_off(warp + 8 * q, lane), src, v ? 16u : 0u);
                }
                walk_next(wc, a, R, MB, NB, lane, true);
                load_idx();
            }
            cp_async_commit();
        };
        load_idx();
#pragma unroll 1
        for (uint32_t j = 0; j + 1 < D; ++j) issue(j);
        for (uint32_t i = 0; wt.valid; ++i) {
            cp_async_wait<D - 2>();
            if (named_bar_any(1, kProducers, !ok)) break;  // the same decision in every producer
            issue(i + D - 1);
            const uint32_t st = i % S, ph = (i / S) & 1u;
            if (mbar_wait(empty0 + 8 * st, ph ^ 1u, s_abort)) {
                const uint8_t* slot = stg + (size_t)(i % D) * kStgBytes;
                float4 v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    v[e] = *reinterpret_cast<const float4*>(slot + stg_off(4 * rq + e, 4 * warp + cg));
                store_t4(stages + (size_t)st * C::kStageBytes, 16 * warp + 4 * cg, rq, v);
                if (p == 0) s_info[st] = (wt.first_stage ? 1u : 0u) | (walk_last(wt) ? 2u : 0u);
                // (the MMA thread orders these generic-proxy stores before its async-proxy
                // reads with one proxy fence after the stage barrier)
                mbar_arrive(full0 + 8 * st);
            } else {  // leave at the next barrier, with the others (the walkers stay in step)
                ok = false;
                *s_abort = 1;
            }
            walk_next(wt, a, R, MB, NB, lane, true);
        }
        cp_async_wait_all();  // no copy of this thread is still writing shared memory
        if (!ok) atomicOr(a.err, kErrTimeout);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_tf32(BN);
            uint32_t it = 0;
            bool ok = true;
            for (uint32_t ua = 0; ok; ++ua) {
                if (ring_read_one(R, ua) < 0) break;
                const uint32_t buf = ua % NBUF;
                if (!mbar_wait(tempty0 + 8 * buf, ((ua / NBUF) & 1u) ^ 1u, s_abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem + buf * BN;
                while (true) {
                    const uint32_t stage = it % S, ph = (it / S) & 1u;
                    if (!mbar_wait(full0 + 8 * stage, ph, s_abort) || !mbar_wait(bfull0 + 8 * stage, ph, s_abort)) {
                        ok = false;
                        break;
                    }
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
    } else if (warp < kLoaderWarp) {
        // ------------------------------------------------------------ epilogue: fp32 partials
        const int q = warp & 3;
        const bool v8ok = (reinterpret_cast<uintptr_t>(a.partial) & 31u) == 0;
        bool ok = true;
        for (uint32_t ua = 0;; ++ua) {
            const int64_t u = ring_read(R, ua, lane, false);
            if (u < 0) break;
            const int nb = (int)(u % NB);
            int64_t r = u / NB;
            const int mb = (int)(r % MB);
            r /= MB;
            const int k = (int)(r % a.taps);
            const int64_t s = r / a.taps;
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
    } else {
        // ------------------------------------------------------------ B loader: one bulk copy per stage
        // (the whole warp walks the stages; lane 0 issues the copies)
        StageWalk wl;
        wl.qi = 0;
        wl.claims = false;
        walk_unit(wl, a, R, MB, NB, lane, false);
        uint32_t i = 0;
        bool ok = true;
        for (; wl.valid; ++i) {
            const uint32_t st = i % S, ph = (i / S) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(empty0 + 8 * st, ph ^ 1u, s_abort))) {
                ok = false;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(bfull0 + 8 * st, C::kBBytes);
                bulk_g2s(smem_u32(stages + (size_t)st * C::kStageBytes + C::kABytes),
                         a.dy_img + tf32_dy_image_offset(wl.t * 128 + wl.h * kRows, wl.nb * BN, a.Cout), C::kBBytes,
                         bfull0 + 8 * st);
            }
            walk_next(wl, a, R, MB, NB, lane, false);
        }
        if (lane == 0) {
            // before the block may exit, every issued copy must have landed
            for (uint32_t d = 0; d < S && d < i; ++d) {
                const uint32_t last = i - 1 - d;
                if (!mbar_wait_timed(bfull0 + 8 * (last % S), (last / S) & 1u)) ok = false;
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
    // with no more units than CTAs every claim returns >= gridDim.x >= units (the end),
    // whatever the counter holds: no reset needed
    if (units > grid) cudaMemsetAsync(a.unit_ctr, 0, sizeof(uint32_t), s);
    kern<<<grid, kThreads, C::kSmem, s>>>(a);
    return VG_OK;
}

}  // namespace

// Split-K chunks: about four units per SM, chunks of at most 256 tiles, at least
// 4 tiles per chunk, the rows of the chunks in flight (about sms / per_split of
// them side by side) within 32 MiB so that a chunk's units find its feature and
// dY rows in L2 (602k voxels, C = 256: 19 chunks 7.9 ms, 55 chunks 7.0 ms with
// the earlier register-staged producers; now 56 chunks 3.48 ms, 111 chunks
// 3.36 ms, 222 chunks 3.44 ms), partial sums capped at 1 GiB.
int tf32_wgrad_splits(int64_t n, int Cin, int Cout, int sms, int taps) {
    const int64_t T = std::max<int64_t>(1, (n + kTileRows - 1) / kTileRows);
    const int64_t per_split = (int64_t)((Cin + kBM - 1) / kBM) * taps * (Cout / tf32_bn(Cout));
    int64_t S = std::max<int64_t>(1, (4 * (int64_t)sms + per_split - 1) / per_split);
    S = std::max<int64_t>(S, (T + 255) / 256);
    const int64_t in_flight = (sms + per_split - 1) / per_split;
    const int64_t chunk_bytes = in_flight * T * kTileRows * (int64_t)(Cin + Cout) * 4;
    S = std::max<int64_t>(S, (chunk_bytes + (int64_t(32) << 20) - 1) / (int64_t(32) << 20));
    const int64_t bytes_per_split = (int64_t)kTaps * Cin * Cout * 4;
    S = std::min<int64_t>(S, std::max<int64_t>(1, (int64_t(1) << 30) / bytes_per_split));
    S = std::min<int64_t>(S, std::max<int64_t>(1, T / 4));
    const int64_t tpc = (T + S - 1) / S;
    return (int)((T + tpc - 1) / tpc);
}

size_t tf32_dy_image_bytes(int64_t n, int Cout) {
    const int64_t rows = (n + kTileRows - 1) / kTileRows * kTileRows;
    return (size_t)rows * Cout * 4;
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
        a.dy_img = static_cast<const float*>(p.dy_sorted);
        a.Cin = p.Cin;
        a.Cout = p.Cout;
        a.partial = p.partial;
        a.err = p.err;
        a.unit_ctr = p.err + kWgradUnitCounter;
        if (!a.dy_img) return VG_ERR_INVALID_ARG;
        // one read of dY: its B-operand image in processing order, and db's partial sums
        launch_dy_image_tf32(p.dy, p.sorted_idx, p.n, a.num_tiles * kTileRows, p.Cout, p.sms, p.db, p.partial_db,
                             p.dy_sorted, p.nbr_status, s);
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
    else if (p.db)
        launch_dbias(p.dy, p.n, p.Cout, p.sms, p.db, p.partial_db, p.dtype, p.nbr_status, s);
    return VG_OK;
}

}  // namespace vg
