// CUDA-core (FFMA) masked implicit GEMM: the fp32 path, and the path for
// 16-bit channel counts the tensor-core kernel does not tile (not multiples of 64).
//
// Forward / input gradient: "From CUDA to Triton: Triton JIT and autotuning",
// §六 6.2 (masked implicit GEMM over sorted rows, contraction V * Ci, taps
// that are empty for the whole tile are skipped).  Weight gradient: the
// split-K backward ("Contribution Tasks — JeffreyXiang/FlexGEMM", §二 key
// types table: sparse_submanifold_conv_bwd_masked_implicit_gemm_splitk).
#include "common.cuh"
#include "internal.h"

namespace vg {

namespace {

constexpr int BM = 64, BN = 64, BK = 32;

// Tile of BM sorted rows x BN output columns; 256 threads, 4x4 outputs each.
template <typename T>
__global__ void __launch_bounds__(256)
k_gather_gemm_simt(const uint32_t* __restrict__ sorted_idx, const uint32_t* __restrict__ nbr,
                   const uint32_t* __restrict__ nbr_status, int64_t n,
                   const T* __restrict__ A, int Kdim, const T* __restrict__ W, int flip,
                   int64_t sK, int64_t sN, const T* __restrict__ bias, T* __restrict__ out,
                   int Ndim) {
    __shared__ uint32_t s_rows[BM];
    __shared__ uint32_t s_nbr[BM][kTaps];
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    __shared__ uint32_t s_tmask;
    if (*nbr_status) return;
    const int tid = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * BM;
    const int n0 = blockIdx.y * BN;
    if (tid < BM) {
        const int64_t r = row0 + tid;
        s_rows[tid] = r < n ? sorted_idx[r] : kNone;
    }
    if (tid == 0) s_tmask = 0;
    __syncthreads();
    for (int idx = tid; idx < BM * kTaps; idx += 256) {
        const int rr = idx / kTaps, k = idx - rr * kTaps;
        const uint32_t v = s_rows[rr];
        s_nbr[rr][k] = v != kNone ? nbr[(int64_t)v * kTaps + k] : kNone;
    }
    __syncthreads();
    if (tid < BM) {
        uint32_t m = 0;
        for (int k = 0; k < kTaps; ++k) m |= (s_nbr[tid][k] != kNone ? 1u : 0u) << k;
        m = __reduce_or_sync(0xffffffffu, m);
        if ((tid & 31) == 0) atomicOr(&s_tmask, m);
    }
    __syncthreads();
    const uint32_t tmask = s_tmask;
    const int ty = tid >> 4, tx = tid & 15;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    const int64_t tap_stride = (int64_t)Kdim * Ndim;
    for (int k = 0; k < kTaps; ++k) {
        if (!((tmask >> k) & 1u)) continue;
        const T* Wk = W + (int64_t)(flip ? 26 - k : k) * tap_stride;
        for (int kk0 = 0; kk0 < Kdim; kk0 += BK) {
            {
                const int rr = tid >> 2, c0 = (tid & 3) * 8;
                const uint32_t j = s_nbr[rr][k];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int kk = kk0 + c0 + e;
                    As[c0 + e][rr] = (j != kNone && kk < Kdim) ? to_f32(A[(int64_t)j * Kdim + kk]) : 0.f;
                }
            }
            {
                const int kr = tid >> 3, c0 = (tid & 7) * 8;
                const int kk = kk0 + kr;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int nn = n0 + c0 + e;
                    Bs[kr][c0 + e] = (kk < Kdim && nn < Ndim) ? to_f32(Wk[kk * sK + nn * sN]) : 0.f;
                }
            }
            __syncthreads();
#pragma unroll 8
            for (int kk = 0; kk < BK; ++kk) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t v = s_rows[ty * 4 + i];
        if (v == kNone) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int nn = n0 + tx * 4 + j;
            if (nn < Ndim) {
                const float b = bias ? to_f32(bias[nn]) : 0.f;
                out[(int64_t)v * Ndim + nn] = from_f32<T>(acc[i][j] + b);
            }
        }
    }
}

constexpr int WR = 32;  // rows per step of the weight-gradient kernel

// Partial dW for (tap k, ci block, co block, row chunk s) -> partial[s][k][ci][co].
template <typename T>
__global__ void __launch_bounds__(256)
k_wgrad_simt(const uint32_t* __restrict__ sorted_idx, const uint32_t* __restrict__ nbr,
             const uint32_t* __restrict__ nbr_status, int64_t n, const T* __restrict__ f,
             const T* __restrict__ dy, int Cin, int Cout, int taps, int64_t rows_per_chunk,
             float* __restrict__ partial) {
    __shared__ float Fs[WR][BM + 4];
    __shared__ float Gs[WR][BN + 4];
    __shared__ uint32_t s_i[WR], s_j[WR];
    if (*nbr_status) return;
    const int tid = threadIdx.x;
    const int co0 = blockIdx.x * BN, ci0 = blockIdx.y * BM;
    const int k = blockIdx.z % taps;
    const int s = blockIdx.z / taps;
    const int64_t rb = (int64_t)s * rows_per_chunk;
    const int64_t re = min(n, rb + rows_per_chunk);
    const int ty = tid >> 4, tx = tid & 15;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int64_t r0 = rb; r0 < re; r0 += WR) {
        if (tid < WR) {
            const int64_t r = r0 + tid;
            const uint32_t v = r < re ? sorted_idx[r] : kNone;
            s_i[tid] = v;
            s_j[tid] = v != kNone ? nbr[(int64_t)v * kTaps + k] : kNone;
        }
        __syncthreads();
        const int any = __syncthreads_or(tid < WR && s_j[tid] != kNone);
        if (!any) continue;
        {
            const int rr = tid >> 3, c0 = (tid & 7) * 8;
            const uint32_t j = s_j[rr], i = s_i[rr];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int ci = ci0 + c0 + e, co = co0 + c0 + e;
                Fs[rr][c0 + e] = (j != kNone && ci < Cin) ? to_f32(f[(int64_t)j * Cin + ci]) : 0.f;
                Gs[rr][c0 + e] = (j != kNone && co < Cout) ? to_f32(dy[(int64_t)i * Cout + co]) : 0.f;
            }
        }
        __syncthreads();
#pragma unroll 8
        for (int rr = 0; rr < WR; ++rr) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = Fs[rr][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Gs[rr][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    float* P = partial + ((int64_t)s * kTaps + k) * Cin * Cout;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int ci = ci0 + ty * 4 + i;
        if (ci >= Cin) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int co = co0 + tx * 4 + j;
            if (co < Cout) P[(int64_t)ci * Cout + co] = acc[i][j];
        }
    }
}

}  // namespace

// Fixed-order sum of split-K partials (deterministic), then round to T.
template <typename T>
__global__ void k_reduce_splits(const float* __restrict__ partial, int splits, int64_t total, int64_t stride,
                                T* __restrict__ out, const uint32_t* __restrict__ nbr_status) {
    if (*nbr_status) return;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    float s = 0.f;
    for (int p = 0; p < splits; ++p) s += partial[(int64_t)p * stride + i];
    out[i] = from_f32<T>(s);
}

// The same sums for four consecutive outputs per thread (total and stride
// multiples of 4): 16-byte loads, four splits' loads issued before their adds,
// each output still summed from zero in split order (bit-identical results).
template <typename T>
__global__ void k_reduce_splits4(const float4* __restrict__ partial, int splits, int64_t total4, int64_t stride4,
                                 T* __restrict__ out, const uint32_t* __restrict__ nbr_status) {
    if (*nbr_status) return;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total4) return;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    int p = 0;
    for (; p + 3 < splits; p += 4) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = partial[(int64_t)(p + j) * stride4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            s.x += v[j].x;
            s.y += v[j].y;
            s.z += v[j].z;
            s.w += v[j].w;
        }
    }
    for (; p < splits; ++p) {
        const float4 v = partial[(int64_t)p * stride4 + i];
        s.x += v.x;
        s.y += v.y;
        s.z += v.z;
        s.w += v.w;
    }
    T* o = out + 4 * i;
    o[0] = from_f32<T>(s.x);
    o[1] = from_f32<T>(s.y);
    o[2] = from_f32<T>(s.z);
    o[3] = from_f32<T>(s.w);
}

// db partial sums: block b sums rows [b*rows, (b+1)*rows) of dy into
// partial_db[b][:].  Thread = (row lane, 8-column group); each thread sums its
// rows in order, then row lanes are combined in order: a fixed summation order.
// rows = n / (4 * SMs) rounded up to a multiple of 256, within [256, 4096]: about
// four blocks per SM keep enough rows in flight for the dY image copy (602k
// voxels: weight-gradient pass at C = 256 0.952 -> 0.909 ms, C = 1024 10.06-10.29
// -> 9.96 ms, TF32 C = 256 3.44 -> 3.19 ms against two blocks per SM).
inline int64_t dbias_rows(int64_t n, int sms) {
    int64_t r = (n / (4 * (int64_t)sms) + 255) / 256 * 256;
    return r < 256 ? 256 : (r > 4096 ? 4096 : r);
}

// Eight consecutive elements (16- or 32-byte aligned) as floats.
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = to_f32(e[q]);
}

template <typename T>
__global__ void __launch_bounds__(256)
k_dbias_partial(const T* __restrict__ dy, int64_t n, int Cout, int64_t rows, float* __restrict__ partial_db,
                const uint32_t* __restrict__ nbr_status) {
    __shared__ float red[256 * 8];
    if (*nbr_status) return;
    const int cg8 = Cout / 8;                      // 8-column groups
    const int lanes = cg8 >= 256 ? 1 : 256 / cg8;  // row lanes per block
    const int tid = threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.x * rows, r1 = min(n, r0 + rows);
    for (int g0 = 0; g0 < cg8; g0 += 256 / lanes) {
        const int rl = tid / (256 / lanes), g = g0 + tid % (256 / lanes);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (g < cg8) {
            // four rows per iteration, their loads issued together (the sums stay in row order)
            int64_t r = r0 + rl;
            for (; r + 3 * lanes < r1; r += 4 * lanes) {
                float v[4][8];
#pragma unroll
                for (int j = 0; j < 4; ++j) load8(dy + (r + j * lanes) * Cout + g * 8, v[j]);
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[q] += v[j][q];
            }
            for (; r < r1; r += lanes) {
                float v[8];
                load8(dy + r * Cout + g * 8, v);
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] += v[q];
            }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) red[tid * 8 + q] = acc[q];
        __syncthreads();
        const int width = 256 / lanes;  // column groups handled in this round
        for (int c = tid; c < width * 8; c += 256) {
            const int gg = g0 + c / 8;
            if (gg >= cg8) continue;
            float sum = 0.f;
            for (int l = 0; l < lanes; ++l) sum += red[(l * width + c / 8) * 8 + (c & 7)];
            partial_db[(int64_t)blockIdx.x * Cout + gg * 8 + (c & 7)] = sum;
        }
        __syncthreads();
    }
}

// The same partial sums read through the processing order, fused with the copy of
// dy into that order that the tensor-core weight gradient loads by bulk copies:
// row r of dst = dy[sorted_idx[r]] for r < n, zero rows up to rows_pad, stored
// as the B-operand image (dy_image_offset); block b sums
// the sorted rows [b*rows, (b+1)*rows) into partial_db[b][:] (fixed order as above).
// One read of dy serves both (16-bit types).
template <typename T>
__global__ void __launch_bounds__(256)
k_dbias_sorted(const T* __restrict__ dy, const uint32_t* __restrict__ sorted_idx, int64_t n, int64_t rows_pad,
               int Cout, int64_t rows, float* __restrict__ partial_db, T* __restrict__ dst,
               const uint32_t* __restrict__ nbr_status) {
    static_assert(sizeof(T) == 2, "16-bit rows");
    __shared__ float red[256 * 8];
    if (*nbr_status) return;
    const int cg8 = Cout / 8;
    const int lanes = cg8 >= 256 ? 1 : 256 / cg8;
    const int tid = threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.x * rows, r1 = min(n, r0 + rows);
    for (int g0 = 0; g0 < cg8; g0 += 256 / lanes) {
        const int rl = tid / (256 / lanes), g = g0 + tid % (256 / lanes);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (g < cg8) {
            // four rows per iteration, their loads issued together (the sums stay in row order)
            int64_t r = r0 + rl;
            for (; r + 3 * lanes < r1; r += 4 * lanes) {
                uint32_t src[4];
                uint4 u[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) src[j] = sorted_idx[r + j * lanes];
#pragma unroll
                for (int j = 0; j < 4; ++j) u[j] = *reinterpret_cast<const uint4*>(dy + (int64_t)src[j] * Cout + g * 8);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    *reinterpret_cast<uint4*>(dst + dy_image_offset(r + j * lanes, g, Cout)) = u[j];
                    const T* e = reinterpret_cast<const T*>(&u[j]);
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[q] += to_f32(e[q]);
                }
            }
            for (; r < r1; r += lanes) {
                const uint4 u = *reinterpret_cast<const uint4*>(dy + (int64_t)sorted_idx[r] * Cout + g * 8);
                *reinterpret_cast<uint4*>(dst + dy_image_offset(r, g, Cout)) = u;
                const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] += to_f32(e[q]);
            }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) red[tid * 8 + q] = acc[q];
        __syncthreads();
        const int width = 256 / lanes;
        for (int c = tid; c < width * 8; c += 256) {
            const int gg = g0 + c / 8;
            if (gg >= cg8) continue;
            float sum = 0.f;
            for (int l = 0; l < lanes; ++l) sum += red[(l * width + c / 8) * 8 + (c & 7)];
            partial_db[(int64_t)blockIdx.x * Cout + gg * 8 + (c & 7)] = sum;
        }
        __syncthreads();
    }
    if (blockIdx.x == gridDim.x - 1) {  // the padding rows of the sorted copy
        const int64_t chunks = (rows_pad - n) * cg8;
        for (int64_t e = tid; e < chunks; e += 256)
            *reinterpret_cast<uint4*>(dst + dy_image_offset(n + e / cg8, (int)(e % cg8), Cout)) =
                make_uint4(0u, 0u, 0u, 0u);
    }
}

// fp32 dy in processing order as the TF32 weight gradient's B-operand image
// (tf32_dy_image_offset), zero rows from n up to rows_pad.  Block b takes the
// sorted rows [b*rows, (b+1)*rows) in groups of 32, 32 channels at a time: each
// thread loads 4 channels of one row (a 32 x 32 tile through shared memory) and
// writes 4 rows of one channel (16 bytes of a 128-byte image row).  With
// partial_db, block b also sums its rows into partial_db[b][:] (fixed order: each
// thread over its row of every group, then the 32 threads of a channel in order).
__global__ void __launch_bounds__(256)
k_dy_image_tf32(const float* __restrict__ dy, const uint32_t* __restrict__ sorted_idx, int64_t n, int64_t rows_pad,
                int Cout, int64_t rows, float* __restrict__ partial_db, float* __restrict__ img,
                const uint32_t* __restrict__ nbr_status) {
    __shared__ float tile[32][33];
    __shared__ float red[32][33];
    if (*nbr_status) return;
    const int tid = threadIdx.x;
    const int lr = tid >> 3, lc = tid & 7;  // load: row lr of the group, channels 4lc..4lc+3
    const int wc = tid >> 3, wk = tid & 7;  // store: channel wc of the block, rows 4wk..4wk+3
    const int64_t r0 = (int64_t)blockIdx.x * rows, r1 = min(rows_pad, r0 + rows);
    for (int c0 = 0; c0 < Cout; c0 += 32) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int64_t g0 = r0; g0 < r1; g0 += 32) {
            const int64_t r = g0 + lr;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < n) v = *reinterpret_cast<const float4*>(dy + (int64_t)sorted_idx[r] * Cout + c0 + 4 * lc);
            acc[0] += v.x;
            acc[1] += v.y;
            acc[2] += v.z;
            acc[3] += v.w;
            __syncthreads();  // the previous group's tile has been read
            tile[lr][4 * lc] = v.x;
            tile[lr][4 * lc + 1] = v.y;
            tile[lr][4 * lc + 2] = v.z;
            tile[lr][4 * lc + 3] = v.w;
            __syncthreads();
            const float4 o = make_float4(tile[4 * wk][wc], tile[4 * wk + 1][wc], tile[4 * wk + 2][wc], tile[4 * wk + 3][wc]);
            *reinterpret_cast<float4*>(img + tf32_dy_image_offset(g0 + 4 * wk, c0 + wc, Cout)) = o;
        }
        if (partial_db) {
            red[lr][4 * lc] = acc[0];
            red[lr][4 * lc + 1] = acc[1];
            red[lr][4 * lc + 2] = acc[2];
            red[lr][4 * lc + 3] = acc[3];
            __syncthreads();
            if (tid < 32) {
                float sum = 0.f;
                for (int l = 0; l < 32; ++l) sum += red[l][tid];
                partial_db[(int64_t)blockIdx.x * Cout + c0 + tid] = sum;
            }
            __syncthreads();
        }
    }
}

template <typename T>
static int launch_gather(const GatherPass& p, cudaStream_t s) {
    const dim3 grid((unsigned)((p.n + BM - 1) / BM), (unsigned)((p.Ndim + BN - 1) / BN));
    // W offsets: fwd  W[k][kk][n]  -> sK = Cout, sN = 1
    //            dgrad W[26-k][n][kk] (mode 1) or W[k][n][kk] (mode 2) -> sK = 1, sN = Cout
    const int64_t sK = p.dgrad ? 1 : p.Cout;
    const int64_t sN = p.dgrad ? p.Cout : 1;
    k_gather_gemm_simt<T><<<grid, 256, 0, s>>>(p.sorted_idx, p.nbr, p.nbr_status, p.n,
                                               static_cast<const T*>(p.A), p.Kdim,
                                               static_cast<const T*>(p.W), p.dgrad == 1, sK, sN,
                                               static_cast<const T*>(p.bias), static_cast<T*>(p.out),
                                               p.Ndim);
    return VG_OK;
}

int simt_gather_pass(const GatherPass& p, cudaStream_t s) {
    if (p.n == 0) return VG_OK;
    switch (p.dtype) {
        case VG_F32: return launch_gather<float>(p, s);
        case VG_F16: return launch_gather<__half>(p, s);
        case VG_BF16: return launch_gather<__nv_bfloat16>(p, s);
    }
    return VG_ERR_INVALID_ARG;
}

int simt_wgrad_splits(int64_t n, int Cin, int Cout, int sms, int taps) {
    const int64_t tiles = (int64_t)taps * ((Cin + BM - 1) / BM) * ((Cout + BN - 1) / BN);
    int64_t s = (4 * (int64_t)sms + tiles - 1) / tiles;
    s = std::min<int64_t>(s, std::max<int64_t>(1, (n + 1023) / 1024));
    return (int)std::max<int64_t>(1, std::min<int64_t>(s, 64));
}

template <typename T>
static int launch_wgrad(const WgradPass& p, cudaStream_t s) {
    const int S = p.splits;
    const int64_t rpc = ((p.n + S - 1) / S + WR - 1) / WR * WR;
    const int64_t total = (int64_t)p.taps * p.Cin * p.Cout;
    if (p.dW) {
        const dim3 grid((unsigned)((p.Cout + BN - 1) / BN), (unsigned)((p.Cin + BM - 1) / BM),
                        (unsigned)(p.taps * S));
        k_wgrad_simt<T><<<grid, 256, 0, s>>>(p.sorted_idx, p.nbr, p.nbr_status, p.n,
                                             static_cast<const T*>(p.f), static_cast<const T*>(p.dy),
                                             p.Cin, p.Cout, p.taps, rpc, p.partial);
        launch_reduce_splits(p.partial, S, total, (int64_t)kTaps * p.Cin * p.Cout, p.dW, p.dtype, p.nbr_status, s);
    }
    if (p.db) launch_dbias(p.dy, p.n, p.Cout, p.sms, p.db, p.partial_db, p.dtype, p.nbr_status, s);
    return VG_OK;
}

int simt_wgrad(const WgradPass& p, cudaStream_t s) {
    if (p.n == 0) return VG_OK;  // zero-fill of empty outputs is done by the caller
    switch (p.dtype) {
        case VG_F32: return launch_wgrad<float>(p, s);
        case VG_F16: return launch_wgrad<__half>(p, s);
        case VG_BF16: return launch_wgrad<__nv_bfloat16>(p, s);
    }
    return VG_ERR_INVALID_ARG;
}

template <typename T>
static void reduce_t(const float* partial, int splits, int64_t total, int64_t stride, void* out,
                     const uint32_t* nbr_status, cudaStream_t s) {
    // Four outputs per thread where that still leaves millions of threads (602k voxels:
    // C = 1024 reduce 0.23 -> 0.12 ms per launch, weight-gradient pass 10.07-10.19 ->
    // 9.94-9.97 ms; C = 64 on 4.9 M voxels,
    // 110k outputs over many splits, 2.180 -> 2.198 ms, so small outputs stay scalar).
    // (partial is 256-byte aligned in the workspace)
    if (total % 4 == 0 && stride % 4 == 0 && total >= (int64_t(4) << 20)) {
        const int64_t t4 = total / 4;
        k_reduce_splits4<T><<<(unsigned)((t4 + 255) / 256), 256, 0, s>>>(
            reinterpret_cast<const float4*>(partial), splits, t4, stride / 4, static_cast<T*>(out), nbr_status);
        return;
    }
    k_reduce_splits<T><<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
        partial, splits, total, stride, static_cast<T*>(out), nbr_status);
}

void launch_reduce_splits(const float* partial, int splits, int64_t total, int64_t stride, void* out, int dtype,
                          const uint32_t* nbr_status, cudaStream_t s) {
    if (dtype == VG_F32) reduce_t<float>(partial, splits, total, stride, out, nbr_status, s);
    else if (dtype == VG_F16) reduce_t<__half>(partial, splits, total, stride, out, nbr_status, s);
    else reduce_t<__nv_bfloat16>(partial, splits, total, stride, out, nbr_status, s);
}

// db = the fixed-order sum of the R row-block partials: block = 32 columns,
// warp w sums partials w, w + 8, w + 16, ... in order, then the 8 warp sums are
// added in warp order (parallel over the partials, unlike k_reduce_splits,
// whose one thread per output walks all R of them: 77 us at R = 1200).
template <typename T>
__global__ void __launch_bounds__(256)
k_reduce_db(const float* __restrict__ partial, int R, int Cout, T* __restrict__ db,
            const uint32_t* __restrict__ nbr_status) {
    __shared__ float part[8][32];
    if (*nbr_status) return;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    float acc = 0.f;
    if (c < Cout)
        for (int p = w; p < R; p += 8) acc += partial[(int64_t)p * Cout + c];
    part[w][lane] = acc;
    __syncthreads();
    if (w == 0 && c < Cout) {
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) t += part[i][lane];
        db[c] = from_f32<T>(t);
    }
}

int dbias_blocks(int64_t n, int sms) {
    const int64_t r = dbias_rows(n, sms);
    return (int)std::max<int64_t>(1, (n + r - 1) / r);
}

template <typename T>
static void dbias_t(const void* dy, int64_t n, int Cout, int sms, void* db, float* partial_db,
                    const uint32_t* nbr_status, cudaStream_t s) {
    const int R = dbias_blocks(n, sms);
    k_dbias_partial<T><<<R, 256, 0, s>>>(static_cast<const T*>(dy), n, Cout, dbias_rows(n, sms), partial_db,
                                         nbr_status);
    k_reduce_db<T><<<(unsigned)((Cout + 31) / 32), 256, 0, s>>>(partial_db, R, Cout, static_cast<T*>(db), nbr_status);
}

void launch_dbias_sorted(const void* dy, const uint32_t* sorted_idx, int64_t n, int64_t rows_pad, int Cout,
                         int sms, void* db, float* partial_db, void* dy_sorted, int dtype,
                         const uint32_t* nbr_status, cudaStream_t s) {
    const int R = dbias_blocks(n, sms);
    const int64_t rows = dbias_rows(n, sms);
    const unsigned cb = (unsigned)((Cout + 31) / 32);
    if (dtype == VG_F16) {
        k_dbias_sorted<__half><<<R, 256, 0, s>>>(static_cast<const __half*>(dy), sorted_idx, n, rows_pad, Cout, rows,
                                                 partial_db, static_cast<__half*>(dy_sorted), nbr_status);
        k_reduce_db<__half><<<cb, 256, 0, s>>>(partial_db, R, Cout, static_cast<__half*>(db), nbr_status);
    } else {
        k_dbias_sorted<__nv_bfloat16><<<R, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(dy), sorted_idx, n,
                                                        rows_pad, Cout, rows, partial_db,
                                                        static_cast<__nv_bfloat16*>(dy_sorted), nbr_status);
        k_reduce_db<__nv_bfloat16><<<cb, 256, 0, s>>>(partial_db, R, Cout, static_cast<__nv_bfloat16*>(db),
                                                      nbr_status);
    }
}

void launch_dbias(const void* dy, int64_t n, int Cout, int sms, void* db, float* partial_db,
                  int dtype, const uint32_t* nbr_status, cudaStream_t s) {
    if (dtype == VG_F32) dbias_t<float>(dy, n, Cout, sms, db, partial_db, nbr_status, s);
    else if (dtype == VG_F16) dbias_t<__half>(dy, n, Cout, sms, db, partial_db, nbr_status, s);
    else dbias_t<__nv_bfloat16>(dy, n, Cout, sms, db, partial_db, nbr_status, s);
}

void launch_dy_image_tf32(const void* dy, const uint32_t* sorted_idx, int64_t n, int64_t rows_pad, int Cout, int sms,
                          void* db, float* partial_db, void* img, const uint32_t* nbr_status, cudaStream_t s) {
    const int R = dbias_blocks(n, sms);  // R * rows >= rows_pad (rows is a multiple of 256)
    k_dy_image_tf32<<<R, 256, 0, s>>>(static_cast<const float*>(dy), sorted_idx, n, rows_pad, Cout,
                                      dbias_rows(n, sms), db ? partial_db : nullptr, static_cast<float*>(img),
                                      nbr_status);
    if (db)
        k_reduce_db<float><<<(unsigned)((Cout + 31) / 32), 256, 0, s>>>(partial_db, R, Cout, static_cast<float*>(db),
                                                                       nbr_status);
}

// out[i] = sum over p = 0 .. nparts-1, in that order, of parts[p][i] (fp32 adds),
// rounded once to T: the rank-ordered gradient sum of data-parallel training.
template <typename T>
__global__ void __launch_bounds__(256)
k_sum_ordered(const T* __restrict__ parts, int nparts, int64_t count, T* __restrict__ out) {
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < count; i += (int64_t)gridDim.x * 256) {
        float s = to_f32(parts[i]);
        for (int p = 1; p < nparts; ++p) s += to_f32(parts[(int64_t)p * count + i]);
        out[i] = from_f32<T>(s);
    }
}

int launch_sum_ordered(const void* parts, int nparts, int64_t count, int dtype, void* out, int sms,
                       cudaStream_t s) {
    if (count == 0) return VG_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>((count + 255) / 256, 8 * (int64_t)sms);
    if (dtype == VG_F32)
        k_sum_ordered<float><<<blocks, 256, 0, s>>>(static_cast<const float*>(parts), nparts, count,
                                                    static_cast<float*>(out));
    else if (dtype == VG_F16)
        k_sum_ordered<__half><<<blocks, 256, 0, s>>>(static_cast<const __half*>(parts), nparts, count,
                                                     static_cast<__half*>(out));
    else
        k_sum_ordered<__nv_bfloat16><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(parts), nparts,
                                                             count, static_cast<__nv_bfloat16*>(out));
    return VG_OK;
}

int plan_sms(int requested) {
    if (requested > 0) return requested;
    constexpr int kMaxDev = 64;
    static int cached[kMaxDev];  // 0 = not looked up yet (benign race: same value)
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return kDefaultSms;
    }
    if (dev < kMaxDev && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return kDefaultSms;
    }
    if (dev < kMaxDev) cached[dev] = n;
    return n;
}

}  // namespace vg
