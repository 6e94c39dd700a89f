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

static int conv_plan(int64_t N, int Cin, int Cout, int dtype, unsigned flags, int sms, ConvPlan* P) {
    if (N < 0 || N >= (int64_t(1) << 31) || Cin <= 0 || Cout <= 0) return VG_ERR_INVALID_ARG;
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
        p.ks_dgrad = tc_gather_splits(N, Cin, p.sms);
    }
    const size_t rows_pad = (size_t)((N + 127) / 128) * 128;
    const size_t gpart = std::max(p.ks_fwd > 1 ? (size_t)p.ks_fwd * rows_pad * Cout * 4 : 0,
                                  p.ks_dgrad > 1 ? (size_t)p.ks_dgrad * rows_pad * Cin * 4 : 0);
    p.splits = p.tensor_core ? tc_wgrad_splits(N, Cin, Cout, p.sms) : simt_wgrad_splits(N, Cin, Cout, p.sms);
    const size_t wbytes = (size_t)kTaps * Cin * Cout * dtype_size(dtype);
    size_t o = 0;
    p.off_err = o;         o += 256;
    p.off_wfwd = o;        o += packed ? align_up(tc_packed_weight_bytes(dtype, Cin, Cout), 256) : 0;
    p.off_wbwd = o;        o += packed ? align_up(tc_packed_weight_bytes(dtype, Cout, Cin), 256) : 0;
    p.off_partial = o;     o += align_up((size_t)p.splits * kTaps * Cin * Cout * 4, 256);
    p.off_partial_db = o;  o += align_up((size_t)dbias_blocks(N, p.sms) * Cout * 4, 256);
    p.off_dys = o;         o += p.tensor_core ? align_up(tc_wgrad_sorted_dy_bytes(N, Cout), 256) : 0;
    p.off_gpart = o;       o += align_up(gpart, 256);
    (void)wbytes;
    p.total = o;
    *P = p;
    return VG_OK;
}

static bool misaligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

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
    info[0] = l.key64;
    info[1] = l.sort_bits;
    info[2] = passes;
    // insert, probe, keys + digit counts, passes, tile rows, tile-order passes
    info[3] = N > 0 ? 4 + passes + l.tile_passes : 0;
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
    GatherPass g;
    g.sorted_idx = vg_nbrmap_sorted_idx(nbr_ws);
    g.tile_mask = vg_nbrmap_tile_mask(nbr_ws, N);
    g.nbr = nbr;
    g.sorted_nbr = vg_nbrmap_sorted_nbr(nbr_ws, N);
    g.nbr_status = static_cast<const uint32_t*>(nbr_ws);
    g.n = N;
    g.A = feats;
    g.Kdim = Cin;
    g.W = weight;
    g.Cin = Cin;
    g.Cout = Cout;
    g.dgrad = 0;
    g.bias = bias;
    g.out = out;
    g.Ndim = Cout;
    g.dtype = dtype;
    g.err = reinterpret_cast<uint32_t*>(ws + p.off_err);
    g.ksplit = p.ks_fwd;
    g.partial = reinterpret_cast<float*>(ws + p.off_gpart);
    if (p.tensor_core || p.tf32) {
        st = tc_pack_weights(weight, dtype, Cin, Cout, 0, ws + p.off_wfwd, g.nbr_status, s);
        if (st == VG_OK) st = tc_gather_pass(g, ws + p.off_wfwd, s);
    } else {
        st = simt_gather_pass(g, s);
    }
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
    const uint32_t* nbr_status = static_cast<const uint32_t*>(nbr_ws);
    uint32_t* err = reinterpret_cast<uint32_t*>(ws + p.off_err);
    if (grad_feats) {
        GatherPass g;
        g.sorted_idx = vg_nbrmap_sorted_idx(nbr_ws);
        g.tile_mask = vg_nbrmap_tile_mask(nbr_ws, N);
        g.nbr = nbr;
        g.sorted_nbr = vg_nbrmap_sorted_nbr(nbr_ws, N);
        g.nbr_status = nbr_status;
        g.n = N;
        g.A = grad_out;
        g.Kdim = Cout;
        g.W = weight;
        g.Cin = Cin;
        g.Cout = Cout;
        g.dgrad = 1;
        g.bias = nullptr;
        g.out = grad_feats;
        g.Ndim = Cin;
        g.dtype = dtype;
        g.err = err;
        g.ksplit = p.ks_dgrad;
        g.partial = reinterpret_cast<float*>(ws + p.off_gpart);
        if (p.tensor_core || p.tf32) {
            st = tc_pack_weights(weight, dtype, Cin, Cout, 1, ws + p.off_wbwd, nbr_status, s);
            if (st == VG_OK) st = tc_gather_pass(g, ws + p.off_wbwd, s);
        } else {
            st = simt_gather_pass(g, s);
        }
        if (st != VG_OK) return st;
    }
    if (grad_weight || grad_bias) {
        WgradPass w;
        w.sorted_idx = vg_nbrmap_sorted_idx(nbr_ws);
        w.tile_mask = vg_nbrmap_tile_mask(nbr_ws, N);
        w.sorted_nbr = vg_nbrmap_sorted_nbr(nbr_ws, N);
        w.tile_order = reinterpret_cast<const uint32_t*>(static_cast<const char*>(nbr_ws) + tile_order_offset(N));
        w.nbr = nbr;
        w.mask = mask;
        w.nbr_status = nbr_status;
        w.n = N;
        w.f = feats;
        w.dy = grad_out;
        w.Cin = Cin;
        w.Cout = Cout;
        w.dtype = dtype;
        w.dW = grad_weight;
        w.db = grad_bias;
        w.partial = reinterpret_cast<float*>(ws + p.off_partial);
        w.partial_db = reinterpret_cast<float*>(ws + p.off_partial_db);
        w.dy_sorted = ws + p.off_dys;
        w.splits = p.splits;
        w.sms = p.sms;
        w.err = err;
        st = p.tensor_core ? tc_wgrad(w, s) : simt_wgrad(w, s);
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
