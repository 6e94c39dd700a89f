/*
 * vg.h — C ABI of the GB300 (sm_103a) submanifold sparse 3D convolution library
 * (libvoxelgemm.so).
 *
 * The operator is the submanifold convolution of "Contribution Tasks —
 * JeffreyXiang/FlexGEMM", §一 (positioning) and §二 (architecture map; "how one
 * call flows through the modules"; key types and functions table):
 * sparse_submanifold_conv3d(feats, coords, shape, weight, bias) evaluates a
 * 3x3x3 convolution only at the active voxels, through a neighbour map that is
 * built once from a coordinate hash map and reused by the forward and the
 * backward pass (the page's neighbor_cache).  The kernel interface in "From
 * CUDA to Triton: Triton JIT and autotuning", §六 6.2 (signature of
 * sparse_submanifold_conv_fwd_masked_implicit_gemm_kernel) fixes V = 27 taps,
 * a uint32 neighbour table, a row order (sorted_idx) and a contraction over
 * V * Ci.
 *
 * Conventions used by every call below:
 *  - tap k <-> offset (dx,dy,dz) in {-1,0,1}^3 with k = 9(dx+1) + 3(dy+1) + (dz+1);
 *    k = 13 is the centre and o_{26-k} = -o_k.
 *  - nbr[i][k] = j when voxel j sits at coord_i + o_k in the same batch element,
 *    else VG_NONE; mask[i] bit k is set iff nbr[i][k] != VG_NONE.  A neighbour
 *    outside the grid is absent (no wrap, no padding).  Row indices are the
 *    caller's row order.
 *  - forward:  out[i][co] = bias[co] + sum_k sum_ci W[k][ci][co] * feats[nbr[i][k]][ci]
 *    input gradient:  dX[j] = sum over (i,k) with nbr[i][k] = j of W_k dY[i]
 *    weight gradient: dW[k][ci][co] = sum_i f[nbr[i][k]][ci] * dY[i][co];  db = sum_i dY[i]
 *  - Every pointer argument is a DEVICE pointer (cudaMalloc'd or equivalent),
 *    row-major and contiguous, owned by the caller; the library allocates no
 *    memory and keeps no global state.  `stream` is a cudaStream_t (NULL = the
 *    legacy default stream).  Calls are stream-ordered and asynchronous unless
 *    stated otherwise.
 *  - Argument errors are detected on the host before anything is launched and
 *    returned as a status code; nothing is written in that case.
 *  - Accumulation is fp32 on every path; outputs are rounded to the input
 *    dtype with round-to-nearest-even.
 *  - N < 2^31 rows.
 */
#ifndef VOXEL_GEMM_VG_H
#define VOXEL_GEMM_VG_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VG_API __attribute__((visibility("default")))
#else
#define VG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------------- */
#define VG_OK                       0
#define VG_ERR_INVALID_ARG          1  /* null pointer, bad size, misaligned pointer     */
#define VG_ERR_COORD_OUT_OF_RANGE   2  /* a coordinate outside [0,B)x[0,X)x[0,Y)x[0,Z)    */
#define VG_ERR_DUPLICATE_COORD      3  /* two rows with the same (b,x,y,z)               */
#define VG_ERR_HASH_FULL            4  /* the voxel hash table overflowed                */
#define VG_ERR_UNSUPPORTED          5  /* channel counts/dtype/flags this build does not run */
#define VG_ERR_WORKSPACE_TOO_SMALL  6  /* ws_bytes below the matching *_workspace_bytes() */
#define VG_ERR_CUDA                 7  /* a CUDA runtime call or launch failed           */
#define VG_ERR_DEVICE_TIMEOUT       8  /* a bounded device-side wait gave up (kernel returned early) */

/* ---- element types ---------------------------------------------------------------- */
#define VG_F32   0
#define VG_F16   1
#define VG_BF16  2

/* ---- flags -------------------------------------------------------------------------- */
#define VG_KEY32            0x1u   /* force 32-bit hash keys (needs B*X*Y*Z < 2^32)    */
#define VG_KEY64            0x2u   /* force 64-bit hash keys                            */
#define VG_ORDER_HILBERT    0x4u   /* row order from the Hilbert code instead of Morton  */
/* Map-build flags: how the probe finds a voxel's neighbours.  The hash table
 * is the pages' method.  The column index counts the voxels of every (b, x, y)
 * column, prefix-sums the counts, stores each column's voxels sorted by z, and
 * searches a voxel's 9 neighbouring columns for z - 1, z, z + 1; it needs
 * B*X*Y <= 2^28.  By default the column index is used when the hash table would
 * exceed 64 MiB (so would not stay in the GPU's L2) and B*X*Y <= 8 N + 2^20;
 * VG_MAP_HASH or VG_MAP_COLUMNS forces one (both: VG_ERR_INVALID_ARG;
 * VG_MAP_COLUMNS on a larger grid: VG_ERR_UNSUPPORTED).  The map, the row order
 * and the tiles are identical either way. */
#define VG_MAP_HASH         0x8u
#define VG_MAP_COLUMNS      0x40u
/* Testing aid: size the hash table below N so that the overflow path
 * (VG_ERR_HASH_FULL) can be exercised from the host. */
#define VG_TEST_SMALL_HASH  0x100u
/* Convolution flag: fp32 features may run on the tensor cores as TF32 (inputs
 * read with a 10-bit mantissa, products accumulated in fp32), as the pages'
 * allow_tf32 switch does ("From CUDA to Triton: Triton JIT and autotuning",
 * §六 6.2: allow_tf32 is part of the autotune key and of the kernel arguments).
 * Applies to fp32 with Cin and Cout multiples of 32 (forward, input gradient and
 * weight gradient); otherwise, and without the flag, fp32 runs on the exact FFMA
 * path. */
#define VG_ALLOW_TF32       0x10u
/* Convolution flag: on the tensor-core paths, keep one work unit per (128-row
 * tile, output-channel block) even when there are fewer such units than SMs.
 * By default a small problem (the pages' inference benchmark case: few voxels)
 * cuts each unit's taps into up to 6 groups that run on separate SMs and writes
 * fp32 partial sums, which a second kernel adds in group order (deterministic)
 * before the bias and the rounding; this flag turns that off, for comparisons.
 * Results agree within rounding either way. */
#define VG_NO_SMALL_N_SPLIT 0x20u

#define VG_NONE 0xFFFFFFFFu        /* missing neighbour in nbr                          */
#define VG_TILE_ROWS 128           /* rows per tile of the sorted order (tile masks)    */

/* Human-readable name of a status code (static string). */
VG_API const char* vg_strerror(int status);

/* Library version as 10000*major + 100*minor + patch. */
VG_API int vg_version(void);

/* ======================================================================================
 * Neighbour map (hash build, 27-tap probe, valid-tap mask, Morton row order, tile masks)
 * Follows the page's hashmap_insert_3d_idx_as_val + subm_neighbor_map +
 * migemm_neighmap_pp steps ("Contribution Tasks — JeffreyXiang/FlexGEMM", §二,
 * module table rows kernels.cuda.hash and kernels.cuda.spconv; init_hashmap picks
 * uint32 or uint64 keys by grid volume).  Reading taken: 64-bit keys iff
 * B*X*Y*Z >= 2^30, unless VG_KEY32/VG_KEY64 forces the width; the map itself is
 * identical either way, and identical again when a column index replaces the
 * hash table (VG_MAP_HASH).
 * ====================================================================================== */

/* Bytes of device workspace vg_nbrmap_build needs for these sizes and flags
 * (0 if the arguments are invalid).  The workspace is the neighbour cache: it
 * holds the hash table (or the column index), the sorted row order and the per-tile masks, and must
 * stay alive and unmodified while convolutions use the map. */
VG_API size_t vg_nbrmap_workspace_bytes(int64_t N, int B, int X, int Y, int Z, unsigned flags);

/* Build the neighbour map of N voxels.
 *   coords  [N][4] int32 (b,x,y,z), 16-byte aligned
 *   ws      workspace of >= vg_nbrmap_workspace_bytes(...) bytes, 256-byte aligned
 *   nbr     [N][27] uint32 output (original row order), mask [N] uint32 output
 * Asynchronous: argument errors are returned at once; data-dependent errors
 * (out-of-range or duplicate coordinates, hash overflow) are recorded on the
 * device in ws and returned by vg_nbrmap_status().  The convolution calls read
 * that record on the device and write nothing when the map is bad. */
VG_API int vg_nbrmap_build(const int32_t* coords, int64_t N, int B, int X, int Y, int Z,
                    unsigned flags, void* ws, size_t ws_bytes,
                    uint32_t* nbr, uint32_t* mask, void* stream);

/* Synchronises `stream` and returns the data-dependent status of the last build
 * into ws (VG_OK, VG_ERR_COORD_OUT_OF_RANGE, VG_ERR_DUPLICATE_COORD,
 * VG_ERR_HASH_FULL or VG_ERR_DEVICE_TIMEOUT when a bounded wait of the sort
 * gave up; the first in that order if several apply). */
VG_API int vg_nbrmap_status(const void* ws, void* stream);

/* Device pointers into a built workspace (no device access, no sync):
 *   sorted_idx [N] uint32 — row r of the processing order is voxel sorted_idx[r]
 *                (the page's sorted_idx).  Stable sort by the key
 *                ((m >> F) << (27 + G)) | (mask << G) | ((m & (2^F - 1)) >> (F - G)),
 *                where m = (b << 3L) | bit-interleave(x, y, z) is the Morton code
 *                (with VG_ORDER_HILBERT: m = (b << 3L) | Hilbert code of (x, y, z) with
 *                L bits, as vg_encode_seq computes it),
 *                L = ceil(log2(max(X,Y,Z))), F = min(3L, 30) and G = min(F, 6),
 *                lowered to 32 - 27 - (bits of m above F) when that makes the
 *                whole key fit 32 bits (4 radix passes instead of 5):
 *                batch element (or 1024^3-voxel Morton block of a larger grid),
 *                then the valid-tap mask, then the
 *                top G fine Morton bits (at most a 4x4x4 split of the block), then the
 *                input order (stable).
 *   tile_mask  [ceil(N/128)] uint32 — OR of mask over sorted rows [128t, 128t+128) */
VG_API const uint32_t* vg_nbrmap_sorted_idx(const void* ws);
VG_API const uint32_t* vg_nbrmap_tile_mask(const void* ws, int64_t N);
/*   sorted_nbr [ceil(N/128)*128][27] uint32 — sorted_nbr[r][k] = nbr[sorted_idx[r]][k],
 *                rows past N are VG_NONE (the map in processing order, so a tile's
 *                neighbour lists are one contiguous 13.5 KB block). */
VG_API const uint32_t* vg_nbrmap_sorted_nbr(const void* ws, int64_t N);

/* Host-only description of the build plan (no device work):
 *   info[0] = how neighbours are looked up: 0 hash table with 32-bit keys, 1 hash
 *   table with 64-bit keys, 2 column index (see VG_MAP_HASH); info[1] = significant bits of the
 *   sort key above, info[2] = radix-sort passes, info[3] = kernels launched by
 *   vg_nbrmap_build (memsets not counted).
 *   sm_count: SMs of the device the plan is for; 0 = the current device's (the
 *   launch grids and the workspace size follow the SM count; without any CUDA
 *   device, 0 plans for 152 SMs).  Returns VG_OK or VG_ERR_INVALID_ARG. */
VG_API int vg_nbrmap_describe(int64_t N, int B, int X, int Y, int Z, unsigned flags, int sm_count,
                              int info[4]);

/* ======================================================================================
 * Convolution (forward, input gradient, weight/bias gradient)
 * The masked implicit GEMM of "From CUDA to Triton: Triton JIT and autotuning",
 * §六 6.2 (kernel arguments input, weight, bias, neighbor, sorted_idx, output;
 * contraction V * Ci) and its backward ("Contribution Tasks — JeffreyXiang/FlexGEMM",
 * §二 call flow: the backward reuses the neighbour cache and returns feats.grad
 * and weight.grad).
 *   dtype: VG_F32 (fp32 FFMA path; with VG_ALLOW_TF32 and Cin, Cout multiples
 *          of 32 all three passes run on the tensor cores as TF32), VG_F16 or
 *          VG_BF16 (tensor-core path when Cin and Cout are
 *          multiples of 64, CUDA-core path otherwise).
 *   Cin and Cout must be multiples of 8 (VG_ERR_UNSUPPORTED otherwise); flags
 *   is 0 or a combination of VG_ALLOW_TF32 and VG_NO_SMALL_N_SPLIT (other bits:
 *   VG_ERR_UNSUPPORTED); the conv workspace size depends on the flags.
 *   feats [N][Cin], weight [27][Cin][Cout], bias [Cout] (or NULL), out [N][Cout],
 *   all of `dtype`, 16-byte aligned.
 *   nbr_ws/nbr/mask: a map built by vg_nbrmap_build for the same N.
 *   conv_ws: >= vg_conv_workspace_bytes(...) bytes, 256-byte aligned; holds the
 *   repacked weights, split-K partial sums, dY in processing order (16-bit
 *   tensor-core path with Cout >= 128, and TF32) and a device error record.  Calls that may overlap on
 *   the GPU (different streams) need their own conv_ws each; they may share
 *   nbr_ws/nbr/mask, which conv calls only read.
 * ====================================================================================== */

/* Bytes of conv workspace needed by vg_subm_conv3d_fwd/bwd for these sizes. */
VG_API size_t vg_conv_workspace_bytes(int64_t N, int Cin, int Cout, int dtype, unsigned flags);

/* Host-only description of the convolution plan (no device work):
 *   info[0] = 1 on the 16-bit tensor-core path, 2 when the fp32 passes run on the
 *   tensor cores as TF32, else 0, info[1] = split-K chunks of the weight
 *   gradient, info[2] = kernels launched by a forward call, info[3] = kernels
 *   launched by a backward call producing all three gradients (memsets not
 *   counted).  sm_count as in vg_nbrmap_describe (the split-K chunk count and
 *   the workspace size follow it; vg_conv_workspace_bytes and the conv calls
 *   use the current device's).  Returns VG_OK or the status vg_subm_conv3d_fwd
 *   would return for these sizes. */
VG_API int vg_conv_describe(int64_t N, int Cin, int Cout, int dtype, unsigned flags, int sm_count,
                            int info[4]);

VG_API int vg_subm_conv3d_fwd(const void* nbr_ws, const uint32_t* nbr, const uint32_t* mask, int64_t N,
                       int dtype, const void* feats, const void* weight, const void* bias,
                       void* out, int Cin, int Cout, unsigned flags,
                       void* conv_ws, size_t conv_ws_bytes, void* stream);

/* Backward.  grad_out [N][Cout]; outputs grad_feats [N][Cin], grad_weight
 * [27][Cin][Cout], grad_bias [Cout]; each output may be NULL to skip it.
 * grad_weight is reduced over split-K chunks in a fixed order (bitwise
 * deterministic run to run). */
VG_API int vg_subm_conv3d_bwd(const void* nbr_ws, const uint32_t* nbr, const uint32_t* mask, int64_t N,
                       int dtype, const void* grad_out, const void* feats, const void* weight,
                       void* grad_feats, void* grad_weight, void* grad_bias,
                       int Cin, int Cout, unsigned flags,
                       void* conv_ws, size_t conv_ws_bytes, void* stream);

/* Synchronises `stream` and returns VG_ERR_DEVICE_TIMEOUT if a kernel of the
 * most recent vg_subm_conv3d_fwd/bwd call on conv_ws gave up a bounded
 * device-side wait (its outputs are then incomplete), else VG_OK.  Every
 * fwd/bwd call clears this record when it starts. */
VG_API int vg_conv_status(void* conv_ws, void* stream);


/* ======================================================================================
 * Regular sparse convolution: strided (down-sampling) and transposed (up-sampling)
 * "Contribution Tasks — JeffreyXiang/FlexGEMM", §二 module table and key functions:
 * sparse_conv3d and kernels.cuda.spconv sparse_neighbor_map -- a convolution whose
 * output sites differ from its input sites.  The pages give no formula; the reading
 * taken is the convolution torch's dense conv3d computes on the densified grid, kept
 * at the output sites whose window holds an active input:
 *   kernel K in {2, 3} per axis (padding 0 for K = 2, 1 for K = 3), stride s in {1, 2};
 *   output grid Xo = (X + 2p - K) / s + 1 (floor), likewise Yo, Zo, same batch count;
 *   tap k = (tx*K + ty)*K + tz <-> offset d_k = (tx - p, ty - p, tz - p), taps = K^3;
 *   output site o is active iff an input sits at s*o + d_k for some k;
 *   output rows are numbered in ascending linear key ((b*Xo + x)*Yo + y)*Zo + z.
 * Strided forward:    out[o] = bias + sum_k W_k^T f[down[o][k]]         (f: input sites)
 * Transposed forward: out[j] = bias + sum_k W_k^T g[up[j][k]]           (g: output sites)
 *   (the dense equivalent is conv_transpose3d with the same K, s, p, output at the input sites)
 * W is [taps][Cin][Cout].  The backward passes run the same kernels as the
 * submanifold convolution (input gradient through the other map with W_k
 * transposed, weight gradient split-K with a fixed-order reduce).
 * ====================================================================================== */

/* A built regular-convolution map: host struct filled by vg_sparse_map_build.  Every
 * pointer points into the map workspace (device memory) and stays valid while it does. */
typedef struct {
    int64_t n_in;               /* input sites (rows of coords)                          */
    int64_t n_out;              /* output sites                                          */
    int kernel, stride, taps;   /* taps = kernel^3                                        */
    int out_grid[4];            /* B, Xo, Yo, Zo                                          */
    const void* side_in;        /* row order and tiles of the input sites (device)        */
    const void* side_out;       /* row order and tiles of the output sites (device)       */
    const uint32_t* down;       /* [n_out][27]: input row at stride*o + d_k, else VG_NONE */
    const uint32_t* down_mask;  /* [n_out]: bit k set iff down[o][k] is valid             */
    const uint32_t* up;         /* [n_in][27]: output row o with stride*o + d_k = coord   */
    const uint32_t* up_mask;    /* [n_in]                                                 */
    const int32_t* coords_out;  /* [n_out][4] (b, x, y, z) in the output grid             */
} vg_sparse_map;

/* Bytes of map workspace for N input sites (0 if the arguments are invalid); flags:
 * 0 or VG_ORDER_HILBERT.  Sized for the largest possible number of output sites. */
VG_API size_t vg_sparse_map_workspace_bytes(int64_t N, int B, int X, int Y, int Z, int kernel, int stride,
                                            unsigned flags);
/* Build the map of N input sites coords [N][4] (device, int32, 16-byte aligned) into
 * ws (device, 256-byte aligned).  SYNCHRONISES `stream`: the number of output sites
 * is data-dependent and returned in map->n_out.  Returns VG_OK, an argument error,
 * VG_ERR_COORD_OUT_OF_RANGE / VG_ERR_DUPLICATE_COORD for bad input sites (map->n_out
 * is then 0 and convolutions on the map write nothing), VG_ERR_HASH_FULL or
 * VG_ERR_DEVICE_TIMEOUT. */
VG_API int vg_sparse_map_build(const int32_t* coords, int64_t N, int B, int X, int Y, int Z, int kernel,
                               int stride, unsigned flags, void* ws, size_t ws_bytes, vg_sparse_map* map,
                               void* stream);
/* Conv workspace for a pass on `map` (transposed = 0: strided, input sites -> output
 * sites; 1: transposed, output sites -> input sites), as vg_conv_workspace_bytes. */
VG_API size_t vg_sparse_conv_workspace_bytes(const vg_sparse_map* map, int transposed, int Cin, int Cout,
                                             int dtype, unsigned flags);
/* Forward.  transposed = 0: feats [n_in][Cin] -> out [n_out][Cout];  transposed = 1:
 * feats [n_out][Cin] -> out [n_in][Cout].  Conventions, dtypes, flags and errors as
 * vg_subm_conv3d_fwd; asynchronous. */
VG_API int vg_sparse_conv3d_fwd(const vg_sparse_map* map, int transposed, int dtype, const void* feats,
                                const void* weight, const void* bias, void* out, int Cin, int Cout,
                                unsigned flags, void* conv_ws, size_t conv_ws_bytes, void* stream);
/* Backward: grad_out has the forward output's rows, grad_feats the forward input's;
 * grad_weight [taps][Cin][Cout], grad_bias [Cout]; each output may be NULL. */
VG_API int vg_sparse_conv3d_bwd(const vg_sparse_map* map, int transposed, int dtype, const void* grad_out,
                                const void* feats, const void* weight, void* grad_feats, void* grad_weight,
                                void* grad_bias, int Cin, int Cout, unsigned flags, void* conv_ws,
                                size_t conv_ws_bytes, void* stream);

/* ======================================================================================
 * Serialisation: space-filling-curve codes of voxel coordinates
 * "Contribution Tasks — JeffreyXiang/FlexGEMM", §二 module table (kernels.cuda.serialize:
 * z_order_encode/decode, hilbert_encode/decode) and the ops layer's
 * encode_seq/decode_seq(coords, shape, mode).  The pages give the names only; the
 * reading taken: code = (b << 3*bits) | curve(x, y, z) for x, y, z in [0, 2^bits).
 *   VG_CURVE_ZORDER:  bit j of x, y, z at bit 3j+2, 3j+1, 3j of the curve part.
 *   VG_CURVE_HILBERT: J. Skilling's Hilbert curve ("Programming the Hilbert curve",
 *                     AIP Conf. Proc. 707, 2004): consecutive codes are face
 *                     neighbours; its transposed index is interleaved like a z-order
 *                     code, x before y before z at each level.
 * The neighbour-map build can use either curve for its row order (VG_ORDER_HILBERT).
 * ====================================================================================== */
#define VG_CURVE_ZORDER  0
#define VG_CURVE_HILBERT 1

/* codes[i] (uint64, device) of coords[i] = (b,x,y,z) (int32 [N][4], device, 16-byte
 * aligned), bits in [0, 20].  A row whose x, y or z lies outside [0, 2^bits), or whose
 * b is negative or does not fit above the curve bits (b >= 2^(63 - 3*bits)), gets
 * the code 0xFFFFFFFFFFFFFFFF.  Asynchronous; VG_ERR_INVALID_ARG for bad sizes,
 * modes or pointers. */
VG_API int vg_encode_seq(const int32_t* coords, int64_t N, int bits, int mode, uint64_t* codes, void* stream);
/* The inverse: coords[i] = (b,x,y,z) of codes[i] (the bits above 3*bits are b). */
VG_API int vg_decode_seq(const uint64_t* codes, int64_t N, int bits, int mode, int32_t* coords, void* stream);

/* ======================================================================================
 * Data-parallel gradient exchange
 * The pages describe a single-GPU operator library and have no multi-GPU step.
 * When several processes each run the convolution on their own batch elements
 * with replicated weights, their weight and bias gradients must be summed; this
 * call is the arithmetic of that exchange, done in a fixed order so that every
 * process ends with the same bits run after run.  Moving the gradients between
 * processes (an all-gather) is the caller's.
 * ====================================================================================== */

/* out[i] = round(parts[0][i] + parts[1][i] + ... + parts[nparts-1][i]) with the
 * additions done in fp32 in index order (left to right) and one round-to-nearest-
 * even to `dtype` at the end.  parts: [nparts][count] contiguous, out: [count],
 * both of `dtype` and aligned to its size; out may not overlap parts.
 * Asynchronous on `stream`; VG_ERR_INVALID_ARG for nparts <= 0, count < 0, an
 * unknown dtype, or null/misaligned pointers. */
VG_API int vg_sum_ordered(const void* parts, int nparts, int64_t count, int dtype, void* out, void* stream);

/* ======================================================================================
 * Forward pass without a caller-provided workspace.
 * The paper has no counterpart to this call.  It is for callers that cannot
 * allocate device memory: plug-ins hosted by a runtime that owns all device memory
 * and forbids allocation after start-up, and hot paths that cannot afford the
 * device-wide synchronisation of cudaMalloc/cudaFree.
 * Arguments and output are those of vg_subm_conv3d_fwd without conv_ws: the scratch
 * (repacked weight tiles and the error word) is a fixed __device__ array of
 * 8 MiB + 256 B inside the library, which every GPU that loads the library holds
 * until the process exits.  The call runs the same kernels as vg_subm_conv3d_fwd
 * with VG_NO_SMALL_N_SPLIT (it has no room for split partial sums), so the
 * output is bit-identical to that call's.  A kernel that gives up a bounded wait
 * is reported by vg_subm_conv3d_fwd_noalloc_status(), not by this call's
 * return value (which covers argument and launch errors only).
 *  - Returns VG_ERR_WORKSPACE_TOO_SMALL when the repacked weights (27*Cin*Cout*2
 *    bytes on the tensor-core path: 16-bit dtype, Cin and Cout multiples of 64)
 *    exceed 8 MiB, e.g. Cin = Cout = 512.
 *  - Allocates nothing.  The first call on each device looks up the array's device
 *    address (cudaGetSymbolAddress) and keeps it once the lookup succeeds.
 *  - Every call uses the same array, which keeps the previous call's contents: calls
 *    that can overlap on the GPU (other streams, other host threads) race on it and
 *    must be serialised by the caller.
 * ====================================================================================== */
VG_API int vg_subm_conv3d_fwd_noalloc(const void* nbr_ws, const uint32_t* nbr, const uint32_t* mask,
                                      int64_t N, int dtype, const void* feats, const void* weight,
                                      const void* bias, void* out, int Cin, int Cout, unsigned flags,
                                      void* stream);

/* Device-side status of the most recent vg_subm_conv3d_fwd_noalloc call on the
 * current device.  The paper has no counterpart to this call either: it reads
 * the error word that the no-allocation forward keeps in its fixed array, so a
 * caller without a conv workspace can still learn that a kernel gave up a
 * bounded wait.  Synchronises `stream` (the stream of that call), then reads and
 * clears the word.  Returns VG_ERR_DEVICE_TIMEOUT if a kernel of that call gave
 * up (its output is then incomplete), VG_OK otherwise, VG_ERR_CUDA if the array's
 * address cannot be looked up or the copy fails.  Allocates nothing. */
VG_API int vg_subm_conv3d_fwd_noalloc_status(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* VOXEL_GEMM_VG_H */
