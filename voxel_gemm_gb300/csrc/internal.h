// Internal (C++ linkage) entry points shared by the library's translation units.
#pragma once
#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace vg {

struct NbrLayout;

// SM count the launch plans are sized for: `requested` if > 0, else the current
// device's (looked up once per device), else kDefaultSms when no device is
// available (host-only size queries on a machine without a GPU).
constexpr int kDefaultSms = 152;
int plan_sms(int requested);

int nbr_layout(int64_t N, int B, int X, int Y, int Z, unsigned flags, int sms, NbrLayout* L);
int nbr_sort_passes(const NbrLayout& l);
int nbr_build(const int32_t* coords, int64_t N, int B, int X, int Y, int Z, unsigned flags,
              void* ws, size_t ws_bytes, uint32_t* nbr, uint32_t* mask, cudaStream_t s);
int nbr_status(const void* ws, cudaStream_t s);

// Regular (strided / transposed) convolution map.  n_out < 0: the layout before
// the number of output sites is known (sizes for the largest possible count).
struct SparseLayout;
int sparse_layout(int64_t N, int B, int X, int Y, int Z, int K, int stride, unsigned flags, int sms,
                  int64_t n_out, SparseLayout* S);
int sparse_build(const int32_t* coords, int64_t N, int B, int X, int Y, int Z, int K, int stride, unsigned flags,
                 void* ws, size_t ws_bytes, int64_t* n_out_host, cudaStream_t s);

// Byte offset of sorted_idx / tile masks inside a neighbour-map workspace.
constexpr size_t kSortedIdxOffset = 256;
inline size_t tile_mask_offset(int64_t N) { return 256 + ((4 * (size_t)N + 255) / 256) * 256; }
inline size_t sorted_nbr_offset(int64_t N) {
    const size_t tiles = (size_t)((N + 127) / 128);
    return tile_mask_offset(N) + ((4 * tiles + 255) / 256) * 256;
}
// Tile visiting order of the weight gradient (tiles grouped by spatial region).
inline size_t tile_order_offset(int64_t N) {
    const size_t tiles = (size_t)((N + 127) / 128);
    return sorted_nbr_offset(N) + ((4 * 27 * 128 * tiles + 255) / 256) * 256;
}

// ---- convolution passes (all asynchronous on stream s) ----
// One "gather GEMM" pass over the sorted rows:
//   out[v][n] = bias[n] + sum_k sum_kk A[nbr[v][k]][kk] * Wk(k, kk, n)
// fwd:   A = feats (Kdim = Cin),  Ndim = Cout, Wk(k,kk,n) = W[k][kk][n]
// dgrad: A = dY    (Kdim = Cout), Ndim = Cin,  Wk(k,kk,n) = W[26-k][n][kk]
struct GatherPass {
    const uint32_t* sorted_idx;
    const uint32_t* tile_mask;   // per 128 sorted rows
    const uint32_t* nbr;
    const uint32_t* sorted_nbr;  // [tiles*128][27] neighbour lists in processing order
    const uint32_t* nbr_status;  // device word; non-zero = bad map, write nothing
    int64_t n;
    const void* A;
    int Kdim;
    const void* W;               // user weight [taps][Cin][Cout]
    int Cin, Cout;
    // 0 = forward (B_k = W_k^T), 1 = submanifold input gradient (B_k = W_{26-k}),
    // 2 = input gradient of a strided / transposed map (B_k = W_k, no flip)
    int dgrad;
    int taps = 27;               // taps of the kernel (27, or 8 for a 2x2x2 kernel)
    const void* bias;            // may be null
    void* out;
    int Ndim;
    int dtype;
    uint32_t* err;               // conv workspace error word
    // tensor-core path: tap groups per (tile, N block) (tc_gather_splits); > 1 needs
    // `partial`, [ksplit][ceil(n/128)*128][Ndim] fp32 of scratch
    int ksplit = 1;
    float* partial = nullptr;
};

int simt_gather_pass(const GatherPass& p, cudaStream_t s);

struct WgradPass {
    const uint32_t* sorted_idx;
    const uint32_t* tile_mask;
    const uint32_t* sorted_nbr;
    const uint32_t* tile_order;  // [tiles] visiting order: tiles grouped by spatial region
    const uint32_t* nbr;
    const uint32_t* mask;
    const uint32_t* nbr_status;
    int64_t n;
    const void* f;
    const void* dy;
    int Cin, Cout, dtype;
    void* dW;      // may be null
    void* db;      // may be null
    float* partial;     // [S][27][Cin][Cout]
    float* partial_db;  // [S][Cout]
    void* dy_sorted;    // tc_wgrad_sorted_dy_bytes (16-bit) or tf32_dy_image_bytes (TF32) bytes of scratch
    int splits;
    int sms;            // SM count of the plan (grid sizes, db row blocks)
    int taps = 27;      // dW has taps x Cin x Cout entries (partials keep a 27-tap stride)
    uint32_t* err;
};

int simt_wgrad_splits(int64_t n, int Cin, int Cout, int sms, int taps = 27);
int simt_wgrad(const WgradPass& p, cudaStream_t s);

// Deterministic fixed-order sum of split-K partials (split p at partial + p * stride)
// over the first `total` entries into out (dtype).
void launch_reduce_splits(const float* partial, int splits, int64_t total, int64_t stride, void* out, int dtype,
                          const uint32_t* nbr_status, cudaStream_t s);
// db = column sums of dy over dbias_blocks(n, sms) row blocks, reduced in a fixed order
// (partial_db holds dbias_blocks(n, sms) x Cout floats).
int dbias_blocks(int64_t n, int sms);
// The same db, read through the processing order while copying dy into it: row r
// of dy_sorted = dy[sorted_idx[r]] for r < n, zero rows up to rows_pad, stored as
// the weight gradient's B-operand image (dy_image_offset; 16-bit dtypes).
void launch_dbias_sorted(const void* dy, const uint32_t* sorted_idx, int64_t n, int64_t rows_pad, int Cout,
                         int sms, void* db, float* partial_db, void* dy_sorted, int dtype,
                         const uint32_t* nbr_status, cudaStream_t s);
void launch_dbias(const void* dy, int64_t n, int Cout, int sms, void* db, float* partial_db,
                  int dtype, const uint32_t* nbr_status, cudaStream_t s);
// fp32 dy in processing order as the TF32 weight gradient's B-operand image
// (tf32_dy_image_offset), rows n..rows_pad zero; with db non-null, fused with
// db's fixed-order partial sums over dbias_blocks(n, sms) row blocks and their reduce.
void launch_dy_image_tf32(const void* dy, const uint32_t* sorted_idx, int64_t n, int64_t rows_pad, int Cout, int sms,
                          void* db, float* partial_db, void* img, const uint32_t* nbr_status, cudaStream_t s);

// Space-filling-curve codes (curve 0 = z-order, 1 = Hilbert) of (b,x,y,z) rows and back.
int curve_encode(const int32_t* coords, int64_t n, int bits, int curve, uint64_t* codes, cudaStream_t s);
int curve_decode(const uint64_t* codes, int64_t n, int bits, int curve, int32_t* coords, cudaStream_t s);

// out = sum of parts[0..nparts) in index order with fp32 adds, rounded once (any dtype).
int launch_sum_ordered(const void* parts, int nparts, int64_t count, int dtype, void* out, int sms,
                       cudaStream_t s);

// ---- tensor-core (tcgen05) path, 16-bit types ----
int tc_supported(int dtype, int Cin, int Cout);
// fp32 features on the tensor cores as TF32 (forward and input gradient): Cin, Cout % 32 == 0
int tf32_supported(int dtype, int Cin, int Cout);
int tc_wgrad_splits(int64_t n, int Cin, int Cout, int sms, int taps = 27);
size_t tc_packed_weight_bytes(int dtype, int Kdim, int Ndim);
// Repack W ([taps][Cin][Cout]) into the swizzled shared-memory image of the B operand
// (mode 0: B_k = W_k^T, K = Cin;  1: B_k = W_{26-k}, K = Cout;  2: B_k = W_k, K = Cout).
int tc_pack_weights(const void* W, int dtype, int Cin, int Cout, int mode, int taps, void* packed,
                    const uint32_t* nbr_status, cudaStream_t s);
int tc_gather_pass(const GatherPass& p, const void* packed, cudaStream_t s);
int tc_wgrad(const WgradPass& p, cudaStream_t s);
// TF32 weight gradient (fp32 features, Cin and Cout multiples of 32): split-K chunks and the pass.
int tf32_wgrad_splits(int64_t n, int Cin, int Cout, int sms, int taps = 27);
size_t tf32_dy_image_bytes(int64_t n, int Cout);  // scratch for the TF32 weight gradient's dY image
int tf32_wgrad(const WgradPass& p, cudaStream_t s);
// Scratch of the weight gradient: dY rows copied into processing order (zero rows
// pad the last tile) when Cout takes the wide-N kernel, else 0 bytes.
size_t tc_wgrad_sorted_dy_bytes(int64_t n, int Cout);
// Tap groups per (tile, N block) of a forward or input-gradient pass: 1 when the
// (tile, N block) units already fill the SMs, else enough to about fill them
// (at most 6); each group adds n_pad * Ndim * 4 bytes of fp32 partials.
int tc_gather_splits(int64_t n, int Ndim, int sms);
int tc_fwd_launches(int ksplit);  // kernels per forward call on the tensor-core path
int tc_bwd_launches(int Cout);    // kernels per full backward call on the tensor-core path

}  // namespace vg
