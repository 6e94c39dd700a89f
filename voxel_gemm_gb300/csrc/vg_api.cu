// extern "C" entry points declared in include/vg.h: argument checks, workspace
// layout, and the launch sequence of each call.  No memory is allocated here.
#include "common.cuh"
#include "internal.h"

namespace vg {

// Conv workspace layout for one (N, Cin, Cout, dtype) problem.
struct ConvPlan {
    int sms = 0;           // SM count the plan is sized for
    int tensor_core = 0;   // 16-bit tcgen05 path (all three passes)
    int tf32 = 0;          // fp32 forward and input gradient on tcgen05 as TF32 (VG_ALLOW_TF32)
    int ks_fwd = 1, ks_dgrad = 1;  // tap groups of the tensor-core forward / input gradient (small N)
    int splits = 1;        // split-K chunks of the weight gradient
    size_t off_err = 0, off_wfwd = 0, off_wbwd = 0, off_partial = 0, off_partial_db = 0, off_dys = 0;
    size_t off_gpart = 0, total = 0;
};

static size_t dtype_size(int dt) { return dt == VG_F32 ? 4 : 2; }

// n_fwd: rows the forward (and the weight gradient) produce / run over;
// n_dgrad: rows the input gradient produces; taps: 27 or 8.
static int conv_plan2(int64_t n_fwd, int64_t n_dgrad, int taps, int Cin, int Cout, int dtype, unsigned flags,
                      int sms, ConvPlan* P) {
    const int64_t N = n_fwd;
    if (N < 0 || N >= (int64_t(1) << 31) || n_dgrad < 0 || n_dgrad >= (int64_t(1) << 31) || Cin <= 0 || Cout <= 0)
        return VG_ERR_INVALID_ARG;
    if (dtype != VG_F32 && dtype != VG_F16 && dtype != VG_BF16) return VG_ERR_INVALID_ARG;
    if (flags & ~(VG_ALLOW_TF32 | VG_NO_SMALL_N_SPLIT)) return VG_ERR_UNSUPPORTED;
    if (Cin % 8 || Cout % 8) return VG_ERR_UNSUPPORTED;  // 16-byte rows for every dtype
    ConvPlan p;
    p.sms = plan_sms(sms);
    p.tensor_core = tc_supported(dtype, Cin, Cout);
    p.tf32 = (flags & VG_ALLOW_TF32) && tf32_supported(dtype, Cin, Cout) ? 1 : 0;
    const int packed = p.tensor_core || p.tf32;
    if (packed && !(flags & VG_NO_SMALL_N_SPLIT)) {
        p.ks_fwd = tc_gather_splits(N, Cout, p.sms);
        p.ks_dgrad = tc_gather_splits(n_dgrad, Cin, p.sms);
    }
    const size_t rows_pad = (size_t)((N + 127) / 128) * 128;
    const size_t rows_pad_d = (size_t)((n_dgrad + 127) / 128) * 128;
    const size_t gpart = std::max(p.ks_fwd > 1 ? (size_t)p.ks_fwd * rows_pad * Cout * 4 : 0,
                                  p.ks_dgrad > 1 ? (size_t)p.ks_dgrad * rows_pad_d * Cin * 4 : 0);
    p.splits = p.tensor_core ? tc_wgrad_splits(N, Cin, Cout, p.sms, taps)
               : p.tf32      ? tf32_wgrad_splits(N, Cin, Cout, p.sms, taps)
                             : simt_wgrad_splits(N, Cin, Cout, p.sms, taps);
    const size_t wbytes = (size_t)kTaps * Cin * Cout * dtype_size(dtype);
    size_t o = 0;
    p.off_err = o;         o += 256;
    p.off_wfwd = o;        o += packed ? align_up(tc_packed_weight_bytes(dtype, Cin, Cout), 256) : 0;
    p.off_wbwd = o;        o += packed ? align_up(tc_packed_weight_bytes(dtype, Cout, Cin), 256) : 0;
    p.off_partial = o;     o += align_up((size_t)p.splits * kTaps * Cin * Cout * 4, 256);
    p.off_partial_db = o;  o += align_up((size_t)dbias_blocks(N, p.sms) * Cout * 4, 256);
    p.off_dys = o;         o += p.tensor_core ? align_up(tc_wgrad_sorted_dy_bytes(N, Cout), 256)
                                : p.tf32      ? align_up(tf32_dy_image_bytes(N, Cout), 256)
                                              : 0;
    p.off_gpart = o;       o += align_up(gpart, 256);
    (void)wbytes;
    p.total = o;
    *P = p;
    return VG_OK;
}

static int conv_plan(int64_t N, int Cin, int Cout, int dtype, unsigned flags, int sms, ConvPlan* P) {
    return conv_plan2(N, N, kTaps, Cin, Cout, dtype, flags, sms, P);
}

static bool misaligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

// One side of a map: the rows a pass produces, with their row order, tiles and
// neighbour lists in processing order in `ws` (laid out like a neighbour-map
// workspace) and their neighbour table in the caller's row order.
struct Side {
    const char* ws;
    int64_t n;
    const uint32_t* nbr;
    const uint32_t* mask;
};

// One gather-GEMM pass over the rows of `sd`: out[r] = (bias) + sum_k B_k A[sd.nbr[r][k]],
// B from W by `mode` (0 forward, 1 submanifold input gradient, 2 input gradient of a
// strided / transposed map).
static int run_gather(const ConvPlan& p, const Side& sd, int mode, int taps, int ksplit, int dtype, const void* A,
                      int Kdim, const void* W, int Cin, int Cout, const void* bias, void* out, int Ndim,
                      uint32_t* err, char* ws, size_t off_packed, cudaStream_t s) {
    if (sd.n == 0) return VG_OK;
    GatherPass g;
    g.sorted_idx = reinterpret_cast<const uint32_t*>(sd.ws + kSortedIdxOffset);
    g.tile_mask = reinterpret_cast<const uint32_t*>(sd.ws + tile_mask_offset(sd.n));
    g.nbr = sd.nbr;
    g.sorted_nbr = reinterpret_cast<const uint32_t*>(sd.ws + sorted_nbr_offset(sd.n));
    g.nbr_status = reinterpret_cast<const uint32_t*>(sd.ws);
    g.n = sd.n;
    g.A = A;
    g.Kdim = Kdim;
    g.W = W;
    g.Cin = Cin;
    g.Cout = Cout;
    g.dgrad = mode;
    g.taps = taps;
    g.bias = bias;
    g.out = out;
    g.Ndim = Ndim;
    g.dtype = dtype;
    g.err = err;
    g.ksplit = ksplit;
    g.partial = reinterpret_cast<float*>(ws + p.off_gpart);
    if (p.tensor_core || p.tf32) {
        const int st = tc_pack_weights(W, dtype, Cin, Cout, mode, taps, ws + off_packed, g.nbr_status, s);
        if (st != VG_OK) return st;
        return tc_gather_pass(g, ws + off_packed, s);
    }
    return simt_gather_pass(g, s);
}

// Weight and bias gradient over the rows of `sd`: dW_k = sum_r f[sd.nbr[r][k]]^T dy[r], db = sum_r dy[r].
static int run_wgrad(const ConvPlan& p, const Side& sd, int taps, int dtype, const void* f, const void* dy,
                     void* dW, void* db, int Cin, int Cout, uint32_t* err, char* ws, cudaStream_t s) {
    WgradPass w;
    w.sorted_idx = reinterpret_cast<const uint32_t*>(sd.ws + kSortedIdxOffset);
    w.tile_mask = reinterpret_cast<const uint32_t*>(sd.ws + tile_mask_offset(sd.n));
    w.sorted_nbr = reinterpret_cast<const uint32_t*>(sd.ws + sorted_nbr_offset(sd.n));
    w.tile_order = reinterpret_cast<const uint32_t*>(sd.ws + tile_order_offset(sd.n));
    w.nbr = sd.nbr;
    w.mask = sd.mask;
    w.nbr_status = reinterpret_cast<const uint32_t*>(sd.ws);
    w.n = sd.n;
    w.f = f;
    w.dy = dy;
    w.Cin = Cin;
    w.Cout = Cout;
    w.dtype = dtype;
    w.dW = dW;
    w.db = db;
    w.partial = reinterpret_cast<float*>(ws + p.off_partial);
    w.partial_db = reinterpret_cast<float*>(ws + p.off_partial_db);
    w.dy_sorted = ws + p.off_dys;
    w.splits = p.splits;
    w.sms = p.sms;
    w.taps = taps;
    w.err = err;
    return p.tensor_core ? tc_wgrad(w, s) : (p.tf32 ? tf32_wgrad(w, s) : simt_wgrad(w, s));
}

static int check_common(const void* nbr_ws, const uint32_t* nbr, const uint32_t* mask, int64_t N,
                        void* conv_ws, size_t conv_ws_bytes, const ConvPlan& p) {
    if (!nbr_ws || misaligned(nbr_ws, 256)) return VG_ERR_INVALID_ARG;
    if (!conv_ws || misaligned(conv_ws, 256)) return VG_ERR_INVALID_ARG;
    if (conv_ws_bytes < p.total) return VG_ERR_WORKSPACE_TOO_SMALL;
    if (N > 0 && (!nbr || !mask || misaligned(nbr, 4) || misaligned(mask, 4))) return VG_ERR_INVALID_ARG;
    return VG_OK;
}

}  // namespace vg

using namespace vg;

extern "C" {

const char* vg_strerror(int status) {
    switch (status) {
        case VG_OK: return "ok";
        case VG_ERR_INVALID_ARG: return "invalid argument";
        case VG_ERR_COORD_OUT_OF_RANGE: return "coordinate out of range";
        case VG_ERR_DUPLICATE_COORD: return "duplicate coordinate";
        case VG_ERR_HASH_FULL: return "voxel hash table full";
        case VG_ERR_UNSUPPORTED: return "unsupported configuration";
        case VG_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case VG_ERR_CUDA: return "CUDA error";
        case VG_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

int vg_version(void) { return 100; }

size_t vg_nbrmap_workspace_bytes(int64_t N, int B, int X, int Y, int Z, unsigned flags) {
    NbrLayout l;
    return nbr_layout(N, B, X, Y, Z, flags, 0, &l) == VG_OK ? l.total : 0;
}

int vg_nbrmap_build(const int32_t* coords, int64_t N, int B, int X, int Y, int Z, unsigned flags,
                    void* ws, size_t ws_bytes, uint32_t* nbr, uint32_t* mask, void* stream) {
    return nbr_build(coords, N, B, X, Y, Z, flags, ws, ws_bytes, nbr, mask,
                     static_cast<cudaStream_t>(stream));
}

int vg_nbrmap_status(const void* ws, void* stream) {
    return nbr_status(ws, static_cast<cudaStream_t>(stream));
}

const uint32_t* vg_nbrmap_sorted_idx(const void* ws) {
    return ws ? reinterpret_cast<const uint32_t*>(static_cast<const char*>(ws) + kSortedIdxOffset) : nullptr;
}

const uint32_t* vg_nbrmap_sorted_nbr(const void* ws, int64_t N) {
    return ws ? reinterpret_cast<const uint32_t*>(static_cast<const char*>(ws) + sorted_nbr_offset(N)) : nullptr;
}

const uint32_t* vg_nbrmap_tile_mask(const void* ws, int64_t N) {
    return ws ? reinterpret_cast<const uint32_t*>(static_cast<const char*>(ws) + tile_mask_offset(N)) : nullptr;
}

int vg_nbrmap_describe(int64_t N, int B, int X, int Y, int Z, unsigned flags, int sm_count, int info[4]) {
    NbrLayout l;
    if (sm_count < 0) return VG_ERR_INVALID_ARG;
    const int st = nbr_layout(N, B, X, Y, Z, flags, sm_count, &l);
    if (st != VG_OK || !info) return st != VG_OK ? st : VG_ERR_INVALID_ARG;
    const int passes = nbr_sort_passes(l);
    info[0] = l.cols ? 2 : l.key64;
    info[1] = l.sort_bits;
    info[2] = passes;
    // hash: insert, probe, keys + digit counts; columns: count, scan, scatter, rank,
    // probe, keys + digit counts; then the passes, tile rows and the tile-order passes
    info[3] = N > 0 ? (l.cols ? 6 : 3) + passes + 1 + l.tile_passes : 0;
    return VG_OK;
}

int vg_conv_describe(int64_t N, int Cin, int Cout, int dtype, unsigned flags, int sm_count, int info[4]) {
    ConvPlan p;
    if (sm_count < 0) return VG_ERR_INVALID_ARG;
    const int st = conv_plan(N, Cin, Cout, dtype, flags, sm_count, &p);
    if (st != VG_OK || !info) return st != VG_OK ? st : VG_ERR_INVALID_ARG;
    info[0] = p.tensor_core ? 1 : (p.tf32 ? 2 : 0);
    info[1] = p.splits;
    const int dgrad_launches = p.tensor_core || p.tf32 ? tc_fwd_launches(p.ks_dgrad) : 1;
    info[2] = N > 0 ? (p.tensor_core || p.tf32 ? tc_fwd_launches(p.ks_fwd) : 1) : 0;
    // backward: input gradient, then dW (GEMM + split reduce; + the dY sort on the 16-bit
    // path when Cout >= 128) and db (partials + reduce)
    info[3] = N > 0 ? (p.tensor_core ? dgrad_launches - 2 + tc_bwd_launches(Cout) : dgrad_launches + 2 + 2) : 0;
    return VG_OK;
}

size_t vg_conv_workspace_bytes(int64_t N, int Cin, int Cout, int dtype, unsigned flags) {
    ConvPlan p;
    return conv_plan(N, Cin, Cout, dtype, flags, 0, &p) == VG_OK ? p.total : 0;
}

int vg_subm_conv3d_fwd(const void* nbr_ws, const uint32_t* nbr, const uint32_t* mask, int64_t N,
                       int dtype, const void* feats, const void* weight, const void* bias,
                       void* out, int Cin, int Cout, unsigned flags,
                       void* conv_ws, size_t conv_ws_bytes, void* stream) {
    ConvPlan p;
    int st = conv_plan(N, Cin, Cout, dtype, flags, 0, &p);
    if (st != VG_OK) return st;
    st = check_common(nbr_ws, nbr, mask, N, conv_ws, conv_ws_bytes, p);
    if (st != VG_OK) return st;
    if (!weight || misaligned(weight, 16) || (bias && misaligned(bias, 16))) return VG_ERR_INVALID_ARG;
    if (N > 0 && (!feats || !out || misaligned(feats, 16) || misaligned(out, 16))) return VG_ERR_INVALID_ARG;
    if (N == 0) return VG_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    char* ws = static_cast<char*>(conv_ws);
    cudaMemsetAsync(ws + p.off_err, 0, 4, s);  // the error record covers this call only
    const Side sd{static_cast<const char*>(nbr_ws), N, nbr, mask};
    st = run_gather(p, sd, 0, kTaps, p.ks_fwd, dtype, feats, Cin, weight, Cin, Cout, bias, out, Cout,
                    reinterpret_cast<uint32_t*>(ws + p.off_err), ws, p.off_wfwd, s);
    if (st != VG_OK) return st;
    return cudaGetLastError() == cudaSuccess ? VG_OK : VG_ERR_CUDA;
}

int vg_subm_conv3d_bwd(const void* nbr_ws, const uint32_t* nbr, const uint32_t* mask, int64_t N,
                       int dtype, const void* grad_out, const void* feats, const void* weight,
                       void* grad_feats, void* grad_weight, void* grad_bias,
                       int Cin, int Cout, unsigned flags,
                       void* conv_ws, size_t conv_ws_bytes, void* stream) {
    ConvPlan p;
    int st = conv_plan(N, Cin, Cout, dtype, flags, 0, &p);
    if (st != VG_OK) return st;
    st = check_common(nbr_ws, nbr, mask, N, conv_ws, conv_ws_bytes, p);
    if (st != VG_OK) return st;
    if ((grad_weight && misaligned(grad_weight, 16)) || (grad_bias && misaligned(grad_bias, 16)))
        return VG_ERR_INVALID_ARG;
    if (grad_feats && (!weight || misaligned(weight, 16))) return VG_ERR_INVALID_ARG;
    if (N > 0) {
        if (!grad_out || misaligned(grad_out, 16)) return VG_ERR_INVALID_ARG;
        if (grad_feats && misaligned(grad_feats, 16)) return VG_ERR_INVALID_ARG;
        if (grad_weight && (!feats || misaligned(feats, 16))) return VG_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    const size_t es = dtype_size(dtype);
    if (N == 0) {  // empty input: zero gradients for the parameters, nothing else
        if (grad_weight) cudaMemsetAsync(grad_weight, 0, (size_t)kTaps * Cin * Cout * es, s);
        if (grad_bias) cudaMemsetAsync(grad_bias, 0, (size_t)Cout * es, s);
        return cudaGetLastError() == cudaSuccess ? VG_OK : VG_ERR_CUDA;
    }
    char* ws = static_cast<char*>(conv_ws);
    cudaMemsetAsync(ws + p.off_err, 0, 4, s);  // the error record covers this call only
    uint32_t* err = reinterpret_cast<uint32_t*>(ws + p.off_err);
    const Side sd{static_cast<const char*>(nbr_ws), N, nbr, mask};
    if (grad_feats) {
        st = run_gather(p, sd, 1, kTaps, p.ks_dgrad, dtype, grad_out, Cout, weight, Cin, Cout, nullptr, grad_feats,
                        Cin, err, ws, p.off_wbwd, s);
        if (st != VG_OK) return st;
    }
    if (grad_weight || grad_bias) {
        st = run_wgrad(p, sd, kTaps, dtype, feats, grad_out, grad_weight, grad_bias, Cin, Cout, err, ws, s);
        if (st != VG_OK) return st;
    }
    return cudaGetLastError() == cudaSuccess ? VG_OK : VG_ERR_CUDA;
}

// ------------------------------------------------------------------ regular (strided / transposed) conv
size_t vg_sparse_map_workspace_bytes(int64_t N, int B, int X, int Y, int Z, int kernel, int stride,
                                     unsigned flags) {
    SparseLayout l;
    return sparse_layout(N, B, X, Y, Z, kernel, stride, flags, 0, -1, &l) == VG_OK ? l.total : 0;
}

int vg_sparse_map_build(const int32_t* coords, int64_t N, int B, int X, int Y, int Z, int kernel, int stride,
                        unsigned flags, void* ws, size_t ws_bytes, vg_sparse_map* map, void* stream) {
    if (!map) return VG_ERR_INVALID_ARG;
    int64_t n_out = 0;
    const int st = sparse_build(coords, N, B, X, Y, Z, kernel, stride, flags, ws, ws_bytes, &n_out,
                                static_cast<cudaStream_t>(stream));
    if (st != VG_OK && st != VG_ERR_DUPLICATE_COORD && st != VG_ERR_COORD_OUT_OF_RANGE && st != VG_ERR_HASH_FULL &&
        st != VG_ERR_DEVICE_TIMEOUT)
        return st;
    SparseLayout l;
    if (sparse_layout(N, B, X, Y, Z, kernel, stride, flags, 0, st == VG_OK ? n_out : 0, &l) != VG_OK)
        return VG_ERR_INVALID_ARG;
    const char* w = static_cast<const char*>(ws);
    map->n_in = N;
    map->n_out = st == VG_OK ? n_out : 0;
    map->kernel = kernel;
    map->stride = stride;
    map->taps = l.T;
    map->out_grid[0] = B;
    map->out_grid[1] = (int)l.Xo;
    map->out_grid[2] = (int)l.Yo;
    map->out_grid[3] = (int)l.Zo;
    map->side_in = w + l.off_side_i;
    map->side_out = w + l.off_side_o;
    map->down = reinterpret_cast<const uint32_t*>(w + l.off_nbr_down);
    map->down_mask = reinterpret_cast<const uint32_t*>(w + l.off_mask_down);
    map->up = reinterpret_cast<const uint32_t*>(w + l.off_nbr_up);
    map->up_mask = reinterpret_cast<const uint32_t*>(w + l.off_mask_up);
    map->coords_out = reinterpret_cast<const int32_t*>(w + l.off_coords_out);
    return st;
}

// The sides a pass runs over: the forward produces the rows of `fwd`, the input
// gradient those of `dgr`; the weight gradient runs over the forward's rows.
static int sparse_sides(const vg_sparse_map* m, int transposed, Side* fwd, Side* dgr) {
    if (!m || !m->side_in || !m->side_out || m->n_in < 0 || m->n_out < 0) return VG_ERR_INVALID_ARG;
    if (m->taps != 8 && m->taps != 27) return VG_ERR_INVALID_ARG;
    const Side in{static_cast<const char*>(m->side_in), m->n_in, m->up, m->up_mask};
    const Side out{static_cast<const char*>(m->side_out), m->n_out, m->down, m->down_mask};
    *fwd = transposed ? in : out;
    *dgr = transposed ? out : in;
    return VG_OK;
}

size_t vg_sparse_conv_workspace_bytes(const vg_sparse_map* map, int transposed, int Cin, int Cout, int dtype,
                                      unsigned flags) {
    Side f, d;
    if (sparse_sides(map, transposed, &f, &d) != VG_OK) return 0;
    ConvPlan p;
    return conv_plan2(f.n, d.n, map->taps, Cin, Cout, dtype, flags, 0, &p) == VG_OK ? p.total : 0;
}

int vg_sparse_conv3d_fwd(const vg_sparse_map* map, int transposed, int dtype, const void* feats, const void* weight,
                         const void* bias, void* out, int Cin, int Cout, unsigned flags, void* conv_ws,
                         size_t conv_ws_bytes, void* stream) {
    Side f, d;
    int st = sparse_sides(map, transposed, &f, &d);
    if (st != VG_OK) return st;
    ConvPlan p;
    st = conv_plan2(f.n, d.n, map->taps, Cin, Cout, dtype, flags, 0, &p);
    if (st != VG_OK) return st;
    if (!conv_ws || misaligned(conv_ws, 256)) return VG_ERR_INVALID_ARG;
    if (conv_ws_bytes < p.total) return VG_ERR_WORKSPACE_TOO_SMALL;
    if (!weight || misaligned(weight, 16) || (bias && misaligned(bias, 16))) return VG_ERR_INVALID_ARG;
    if (f.n > 0 && (!out || misaligned(out, 16))) return VG_ERR_INVALID_ARG;
    if (d.n > 0 && (!feats || misaligned(feats, 16))) return VG_ERR_INVALID_ARG;
    if (f.n == 0) return VG_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    char* ws = static_cast<char*>(conv_ws);
    cudaMemsetAsync(ws + p.off_err, 0, 4, s);
    st = run_gather(p, f, 0, map->taps, p.ks_fwd, dtype, feats, Cin, weight, Cin, Cout, bias, out, Cout,
                    reinterpret_cast<uint32_t*>(ws + p.off_err), ws, p.off_wfwd, s);
    if (st != VG_OK) return st;
    return cudaGetLastError() == cudaSuccess ? VG_OK : VG_ERR_CUDA;
}

int vg_sparse_conv3d_bwd(const vg_sparse_map* map, int transposed, int dtype, const void* grad_out,
                         const void* feats, const void* weight, void* grad_feats, void* grad_weight, void* grad_bias,
                         int Cin, int Cout, unsigned flags, void* conv_ws, size_t conv_ws_bytes, void* stream) {
    Side f, d;
    int st = sparse_sides(map, transposed, &f, &d);
    if (st != VG_OK) return st;
    ConvPlan p;
    st = conv_plan2(f.n, d.n, map->taps, Cin, Cout, dtype, flags, 0, &p);
    if (st != VG_OK) return st;
    if (!conv_ws || misaligned(conv_ws, 256)) return VG_ERR_INVALID_ARG;
    if (conv_ws_bytes < p.total) return VG_ERR_WORKSPACE_TOO_SMALL;
    if ((grad_weight && misaligned(grad_weight, 16)) || (grad_bias && misaligned(grad_bias, 16)))
        return VG_ERR_INVALID_ARG;
    if (grad_feats && (!weight || misaligned(weight, 16))) return VG_ERR_INVALID_ARG;
    if (f.n > 0 && (!grad_out || misaligned(grad_out, 16))) return VG_ERR_INVALID_ARG;
    if (d.n > 0 && grad_feats && misaligned(grad_feats, 16)) return VG_ERR_INVALID_ARG;
    if (d.n > 0 && grad_weight && (!feats || misaligned(feats, 16))) return VG_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    char* ws = static_cast<char*>(conv_ws);
    uint32_t* err = reinterpret_cast<uint32_t*>(ws + p.off_err);
    cudaMemsetAsync(ws + p.off_err, 0, 4, s);
    const size_t es = dtype_size(dtype);
    if (grad_feats && d.n > 0) {
        if (f.n == 0) {  // no output rows: the input gradient is zero
            cudaMemsetAsync(grad_feats, 0, (size_t)d.n * Cin * es, s);
        } else {
            st = run_gather(p, d, 2, map->taps, p.ks_dgrad, dtype, grad_out, Cout, weight, Cin, Cout, nullptr,
                            grad_feats, Cin, err, ws, p.off_wbwd, s);
            if (st != VG_OK) return st;
        }
    }
    if (f.n == 0) {
        if (grad_weight) cudaMemsetAsync(grad_weight, 0, (size_t)map->taps * Cin * Cout * es, s);
        if (grad_bias) cudaMemsetAsync(grad_bias, 0, (size_t)Cout * es, s);
    } else if (grad_weight || grad_bias) {
        st = run_wgrad(p, f, map->taps, dtype, feats, grad_out, grad_weight, grad_bias, Cin, Cout, err, ws, s);
        if (st != VG_OK) return st;
    }
    return cudaGetLastError() == cudaSuccess ? VG_OK : VG_ERR_CUDA;
}

int vg_encode_seq(const int32_t* coords, int64_t N, int bits, int mode, uint64_t* codes, void* stream) {
    if (N < 0 || bits < 0 || bits > 20 || (mode != VG_CURVE_ZORDER && mode != VG_CURVE_HILBERT))
        return VG_ERR_INVALID_ARG;
    if (N > 0 && (!coords || !codes || misaligned(coords, 16) || misaligned(codes, 8))) return VG_ERR_INVALID_ARG;
    cudaGetLastError();
    curve_encode(coords, N, bits, mode, codes, static_cast<cudaStream_t>(stream));
    return cudaGetLastError() == cudaSuccess ? VG_OK : VG_ERR_CUDA;
}

int vg_decode_seq(const uint64_t* codes, int64_t N, int bits, int mode, int32_t* coords, void* stream) {
    if (N < 0 || bits < 0 || bits > 20 || (mode != VG_CURVE_ZORDER && mode != VG_CURVE_HILBERT))
        return VG_ERR_INVALID_ARG;
    if (N > 0 && (!coords || !codes || misaligned(coords, 16) || misaligned(codes, 8))) return VG_ERR_INVALID_ARG;
    cudaGetLastError();
    curve_decode(codes, N, bits, mode, coords, static_cast<cudaStream_t>(stream));
    return cudaGetLastError() == cudaSuccess ? VG_OK : VG_ERR_CUDA;
}

int vg_sum_ordered(const void* parts, int nparts, int64_t count, int dtype, void* out, void* stream) {
    if (nparts <= 0 || count < 0) return VG_ERR_INVALID_ARG;
    if (dtype != VG_F32 && dtype != VG_F16 && dtype != VG_BF16) return VG_ERR_INVALID_ARG;
    if (count > 0 && (!parts || !out)) return VG_ERR_INVALID_ARG;
    const size_t es = dtype_size(dtype);
    if (misaligned(parts, es) || misaligned(out, es)) return VG_ERR_INVALID_ARG;
    cudaGetLastError();
    const int st = launch_sum_ordered(parts, nparts, count, dtype, out, plan_sms(0),
                                      static_cast<cudaStream_t>(stream));
    if (st != VG_OK) return st;
    return cudaGetLastError() == cudaSuccess ? VG_OK : VG_ERR_CUDA;
}

int vg_conv_status(void* conv_ws, void* stream) {
    if (!conv_ws) return VG_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t h = 0;
    if (cudaMemcpyAsync(&h, conv_ws, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return VG_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return VG_ERR_CUDA;
    if (cudaMemsetAsync(conv_ws, 0, sizeof(h), s) != cudaSuccess) return VG_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return VG_ERR_CUDA;
    return (h & kErrTimeout) ? VG_ERR_DEVICE_TIMEOUT : VG_OK;
}

}  // extern "C"
