/*
 * CPU oracle for submanifold sparse 3D convolution — TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, obviously-correct statement of what the GPU
 * library computes.  Only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark may load it; the product path never does.
 * It shares no code, header, table or helper with the CUDA sources.
 *
 * Sources (the web pages this method is described on):
 *  - "Contribution Tasks — JeffreyXiang/FlexGEMM", §一 (positioning) and §二
 *    (architecture map, "how one call flows through the modules", key types
 *    and functions table): the operator sparse_submanifold_conv3d(feats,
 *    coords, shape, weight, bias) computes outputs only at the active input
 *    sites; a neighbour map is built from a coordinate hash map
 *    (hashmap_insert_3d_idx_as_val, subm_neighbor_map) and reused by the
 *    forward and the backward pass (neighbor_cache).
 *  - "From CUDA to Triton: Triton JIT and autotuning", §六 6.2: the masked
 *    implicit GEMM kernel takes (input, weight, bias, neighbor, sorted_idx,
 *    output) with V = 27 taps, a uint32 neighbour table, and a contraction
 *    dimension of V * Ci.
 *
 * The pages do not write the sum out.  The reading taken here (the standard
 * submanifold convolution) is:
 *   tap k <-> offset o_k = (dx,dy,dz) in {-1,0,1}^3, k = 9(dx+1)+3(dy+1)+(dz+1)
 *   nbr[i][k] = j  if voxel j has coordinate coord_i + o_k in the same batch
 *               element, else 0xFFFFFFFF (outside the grid counts as absent)
 *   mask[i]   = sum_k [nbr[i][k] valid] * 2^k
 *   out[i][co]  = bias[co] + sum_k sum_ci W[k][ci][co] * f[nbr[i][k]][ci]
 *   dX[j][ci]   = sum over (i,k) with nbr[i][k] = j of sum_co W[k][ci][co] dY[i][co]
 *   dW[k][ci][co] = sum_i [nbr[i][k] valid] f[nbr[i][k]][ci] * dY[i][co]
 *   db[co]      = sum_i dY[i][co]
 * All floating point is accumulated in double precision from the (already
 * dtype-rounded) inputs.
 *
 * The neighbour lookup is a dictionary: a sorted array of (key, row) pairs
 * built with qsort and searched with bsearch from the C library.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_NONE 0xFFFFFFFFu

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_OUT_OF_RANGE = 2, ORACLE_DUPLICATE = 3,
       ORACLE_NO_MEMORY = 4 };

/* Tap index k -> offset (dx, dy, dz). */
static void tap_offset(int k, int* dx, int* dy, int* dz)
{
    *dx = k / 9 - 1;
    *dy = (k / 3) % 3 - 1;
    *dz = k % 3 - 1;
}

/* Linear address of (b,x,y,z) in a B x X x Y x Z grid. */
static uint64_t linear_key(int64_t b, int64_t x, int64_t y, int64_t z,
                           int64_t X, int64_t Y, int64_t Z)
{
    return (uint64_t)(((b * X + x) * Y + y) * Z + z);
}

typedef struct { uint64_t key; int64_t row; } dict_entry;

static int cmp_entry(const void* a, const void* b)
{
    const dict_entry* p = (const dict_entry*)a;
    const dict_entry* q = (const dict_entry*)b;
    if (p->key < q->key) return -1;
    if (p->key > q->key) return 1;
    return 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Neighbour map (the subm_neighbor_map step).  coords is [N][4] = (b,x,y,z).
 * Returns ORACLE_OUT_OF_RANGE if a coordinate lies outside [0,B)x[0,X)x[0,Y)x[0,Z),
 * ORACLE_DUPLICATE if two rows share a coordinate; nbr/mask are then unspecified.
 */
int oracle_nbrmap(const int32_t* coords, int64_t N, int B, int X, int Y, int Z,
                  uint32_t* nbr, uint32_t* mask)
{
    if (N < 0 || B <= 0 || X <= 0 || Y <= 0 || Z <= 0) return ORACLE_BAD_ARG;
    if (N == 0) return ORACLE_OK;
    for (int64_t i = 0; i < N; ++i) {
        const int32_t* c = coords + 4 * i;
        if (c[0] < 0 || c[0] >= B || c[1] < 0 || c[1] >= X ||
            c[2] < 0 || c[2] >= Y || c[3] < 0 || c[3] >= Z)
            return ORACLE_OUT_OF_RANGE;
    }
    dict_entry* dict = (dict_entry*)malloc((size_t)N * sizeof(dict_entry));
    if (!dict) return ORACLE_NO_MEMORY;
    for (int64_t i = 0; i < N; ++i) {
        const int32_t* c = coords + 4 * i;
        dict[i].key = linear_key(c[0], c[1], c[2], c[3], X, Y, Z);
        dict[i].row = i;
    }
    qsort(dict, (size_t)N, sizeof(dict_entry), cmp_entry);
    for (int64_t i = 1; i < N; ++i) {
        if (dict[i].key == dict[i - 1].key) {
            free(dict);
            return ORACLE_DUPLICATE;
        }
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N; ++i) {
        const int32_t* c = coords + 4 * i;
        uint32_t m = 0;
        for (int k = 0; k < 27; ++k) {
            int dx, dy, dz;
            tap_offset(k, &dx, &dy, &dz);
            int64_t x = (int64_t)c[1] + dx, y = (int64_t)c[2] + dy, z = (int64_t)c[3] + dz;
            uint32_t j = ORACLE_NONE;
            if (x >= 0 && x < X && y >= 0 && y < Y && z >= 0 && z < Z) {
                dict_entry probe;
                probe.key = linear_key(c[0], x, y, z, X, Y, Z);
                probe.row = 0;
                const dict_entry* hit = (const dict_entry*)bsearch(
                    &probe, dict, (size_t)N, sizeof(dict_entry), cmp_entry);
                if (hit) j = (uint32_t)hit->row;
            }
            nbr[i * 27 + k] = j;
            if (j != ORACLE_NONE) m |= 1u << k;
        }
        mask[i] = m;
    }
    free(dict);
    return ORACLE_OK;
}

/*
 * Forward: out[i][co] = bias[co] + sum_k sum_ci W[k][ci][co] * f[nbr[i][k]][ci]
 * for the R rows whose neighbour lists are given in nbr ([R][27], indices into
 * the Nf rows of f).  W is [27][Cin][Cout]; bias may be NULL (zero).
 */
void oracle_fwd(const uint32_t* nbr, int64_t R, const double* f, int64_t Nf,
                const double* W, const double* bias, int Cin, int Cout, double* out)
{
    (void)Nf;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < R; ++i) {
        double* o = out + i * Cout;
        for (int co = 0; co < Cout; ++co) o[co] = bias ? bias[co] : 0.0;
        for (int k = 0; k < 27; ++k) {
            uint32_t j = nbr[i * 27 + k];
            if (j == ORACLE_NONE) continue;
            const double* fj = f + (int64_t)j * Cin;
            for (int ci = 0; ci < Cin; ++ci) {
                const double a = fj[ci];
                const double* w = W + ((int64_t)k * Cin + ci) * Cout;
                for (int co = 0; co < Cout; ++co) o[co] += w[co] * a;
            }
        }
    }
}

/*
 * Input gradient by its definition (the adjoint of the forward): every valid
 * pair (i,k) with j = nbr[i][k] adds W_k dY[i] to dX[j].  nbr is [N][27] over
 * the N rows of dY and dX.  Sequential: the scatter is written out plainly.
 */
void oracle_dgrad_scatter(const uint32_t* nbr, int64_t N, const double* dY,
                          const double* W, int Cin, int Cout, double* dX)
{
    memset(dX, 0, (size_t)N * Cin * sizeof(double));
    for (int64_t i = 0; i < N; ++i) {
        const double* g = dY + i * Cout;
        for (int k = 0; k < 27; ++k) {
            uint32_t j = nbr[i * 27 + k];
            if (j == ORACLE_NONE) continue;
            double* d = dX + (int64_t)j * Cin;
            for (int ci = 0; ci < Cin; ++ci) {
                const double* w = W + ((int64_t)k * Cin + ci) * Cout;
                double s = 0.0;
                for (int co = 0; co < Cout; ++co) s += w[co] * g[co];
                d[ci] += s;
            }
        }
    }
}

/*
 * Input gradient for R chosen rows, gathered form: since o_{26-k} = -o_k,
 * nbr[i][k] = j holds exactly when nbr[j][26-k] = i, so
 *   dX[j][ci] = sum_k' sum_co W[26-k'][ci][co] * dY[nbr[j][k']][co].
 * nbr is [R][27] (indices into the rows of dY).  The tests check this form
 * against oracle_dgrad_scatter.
 */
void oracle_dgrad_rows(const uint32_t* nbr, int64_t R, const double* dY, int64_t Ny,
                       const double* W, int Cin, int Cout, double* dX)
{
    (void)Ny;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < R; ++r) {
        double* d = dX + r * Cin;
        for (int ci = 0; ci < Cin; ++ci) d[ci] = 0.0;
        for (int kp = 0; kp < 27; ++kp) {
            uint32_t i = nbr[r * 27 + kp];
            if (i == ORACLE_NONE) continue;
            const double* g = dY + (int64_t)i * Cout;
            const int k = 26 - kp;
            for (int ci = 0; ci < Cin; ++ci) {
                const double* w = W + ((int64_t)k * Cin + ci) * Cout;
                double s = 0.0;
                for (int co = 0; co < Cout; ++co) s += w[co] * g[co];
                d[ci] += s;
            }
        }
    }
}

/*
 * Weight and bias gradient:
 *   dW[k][ci][co] = sum_i [nbr[i][k] valid] f[nbr[i][k]][ci] * dY[i][co]
 *   db[co]        = sum_i dY[i][co]      (db may be NULL)
 * nbr is [N][27]; f has Nf rows; dY has N rows.  Parallel over taps only, so
 * every output entry is one plain sum in row order.
 */
void oracle_wgrad(const uint32_t* nbr, int64_t N, const double* f, int64_t Nf,
                  const double* dY, int Cin, int Cout, double* dW, double* db)
{
    (void)Nf;
#pragma omp parallel for schedule(dynamic, 1)
    for (int k = 0; k < 27; ++k) {
        double* w = dW + (int64_t)k * Cin * Cout;
        memset(w, 0, (size_t)Cin * Cout * sizeof(double));
        for (int64_t i = 0; i < N; ++i) {
            uint32_t j = nbr[i * 27 + k];
            if (j == ORACLE_NONE) continue;
            const double* fj = f + (int64_t)j * Cin;
            const double* g = dY + i * Cout;
            for (int ci = 0; ci < Cin; ++ci) {
                const double a = fj[ci];
                double* wr = w + (int64_t)ci * Cout;
                for (int co = 0; co < Cout; ++co) wr[co] += a * g[co];
            }
        }
    }
    if (db) {
        for (int co = 0; co < Cout; ++co) db[co] = 0.0;
        for (int64_t i = 0; i < N; ++i)
            for (int co = 0; co < Cout; ++co) db[co] += dY[i * Cout + co];
    }
}

/*
 * Space-filling-curve codes of voxel coordinates ("Contribution Tasks —
 * JeffreyXiang/FlexGEMM", §二 module table, kernels.cuda.serialize:
 * z_order_encode/decode and hilbert_encode/decode, with a CPU and a CUDA path;
 * ops.serialize encode_seq/decode_seq with mode 'z_order' or 'hilbert').  The
 * pages give the names only.  Readings taken: a code packs the batch index above
 * 3*bits curve bits, code = (b << 3*bits) | c(x, y, z), for coordinates in
 * [0, 2^bits).
 *  - z-order: bit j of x, y, z goes to bit 3j+2, 3j+1, 3j of c.
 *  - Hilbert: the curve of J. Skilling, "Programming the Hilbert curve" (AIP
 *    Conf. Proc. 707, 2004).  The coordinates are turned into the curve's
 *    "transposed" index -- from the top level down, each level's excess
 *    rotation/reflection is undone, then the words are Gray-coded -- and the
 *    transposed words are read out most significant level first, x before y
 *    before z, three bits per level.  Decoding runs those steps backwards.
 */
static uint64_t zorder_code(uint32_t x, uint32_t y, uint32_t z, int bits)
{
    uint64_t c = 0;
    for (int j = 0; j < bits; ++j) {
        c |= (uint64_t)((x >> j) & 1u) << (3 * j + 2);
        c |= (uint64_t)((y >> j) & 1u) << (3 * j + 1);
        c |= (uint64_t)((z >> j) & 1u) << (3 * j);
    }
    return c;
}

static void zorder_cell(uint64_t c, int bits, uint32_t* x, uint32_t* y, uint32_t* z)
{
    *x = *y = *z = 0;
    for (int j = 0; j < bits; ++j) {
        *x |= (uint32_t)((c >> (3 * j + 2)) & 1u) << j;
        *y |= (uint32_t)((c >> (3 * j + 1)) & 1u) << j;
        *z |= (uint32_t)((c >> (3 * j)) & 1u) << j;
    }
}

/* Skilling's AxesToTranspose for three axes. */
static void hilbert_to_transpose(uint32_t w[3], int bits)
{
    const uint32_t top = 1u << (bits - 1);
    for (uint32_t q = top; q > 1; q >>= 1) {          /* undo excess work, top level first */
        const uint32_t p = q - 1;
        for (int i = 0; i < 3; ++i) {
            if (w[i] & q) {
                w[0] ^= p;                             /* invert the low bits of axis 0 */
            } else {
                const uint32_t t = (w[0] ^ w[i]) & p;  /* exchange low bits of axes 0 and i */
                w[0] ^= t;
                w[i] ^= t;
            }
        }
    }
    for (int i = 1; i < 3; ++i) w[i] ^= w[i - 1];      /* Gray encode */
    uint32_t t = 0;
    for (uint32_t q = top; q > 1; q >>= 1)
        if (w[2] & q) t ^= q - 1;
    for (int i = 0; i < 3; ++i) w[i] ^= t;
}

/* Skilling's TransposeToAxes for three axes (the inverse of the above). */
static void hilbert_from_transpose(uint32_t w[3], int bits)
{
    const uint32_t end = 2u << (bits - 1);
    uint32_t t = w[2] >> 1;                            /* Gray decode */
    for (int i = 2; i > 0; --i) w[i] ^= w[i - 1];
    w[0] ^= t;
    for (uint32_t q = 2; q != end; q <<= 1) {          /* redo the work, bottom level first */
        const uint32_t p = q - 1;
        for (int i = 2; i >= 0; --i) {
            if (w[i] & q) {
                w[0] ^= p;
            } else {
                t = (w[0] ^ w[i]) & p;
                w[0] ^= t;
                w[i] ^= t;
            }
        }
    }
}

static uint64_t hilbert_code(uint32_t x, uint32_t y, uint32_t z, int bits)
{
    if (bits == 0) return 0;
    uint32_t w[3] = {x, y, z};
    hilbert_to_transpose(w, bits);
    uint64_t c = 0;
    for (int j = bits - 1; j >= 0; --j)
        for (int i = 0; i < 3; ++i) c = (c << 1) | ((w[i] >> j) & 1u);
    return c;
}

static void hilbert_cell(uint64_t c, int bits, uint32_t* x, uint32_t* y, uint32_t* z)
{
    uint32_t w[3] = {0, 0, 0};
    if (bits > 0) {
        int pos = 3 * bits - 1;                        /* bit of c being read, most significant first */
        for (int j = bits - 1; j >= 0; --j)
            for (int i = 0; i < 3; ++i, --pos) w[i] |= (uint32_t)((c >> pos) & 1u) << j;
        hilbert_from_transpose(w, bits);
    }
    *x = w[0];
    *y = w[1];
    *z = w[2];
}

/* codes[i] = (b << 3*bits) | curve(x, y, z) of coords[i] = (b, x, y, z); curve 0 =
 * z-order, 1 = Hilbert.  Returns ORACLE_BAD_ARG for bits outside [0, 20] or a
 * coordinate outside [0, 2^bits) (negative b included). */
int oracle_curve_encode(const int32_t* coords, int64_t N, int bits, int curve, uint64_t* codes)
{
    if (bits < 0 || bits > 20 || N < 0) return ORACLE_BAD_ARG;
    for (int64_t i = 0; i < N; ++i) {
        const int32_t* c = coords + 4 * i;
        if (c[0] < 0) return ORACLE_BAD_ARG;
        for (int a = 1; a < 4; ++a)
            if (c[a] < 0 || (int64_t)c[a] >= ((int64_t)1 << bits)) return ORACLE_BAD_ARG;
        const uint64_t h = curve ? hilbert_code((uint32_t)c[1], (uint32_t)c[2], (uint32_t)c[3], bits)
                                 : zorder_code((uint32_t)c[1], (uint32_t)c[2], (uint32_t)c[3], bits);
        codes[i] = ((uint64_t)c[0] << (3 * bits)) | h;
    }
    return ORACLE_OK;
}

/* The inverse: coords[i] = (b, x, y, z) of codes[i]. */
int oracle_curve_decode(const uint64_t* codes, int64_t N, int bits, int curve, int32_t* coords)
{
    if (bits < 0 || bits > 20 || N < 0) return ORACLE_BAD_ARG;
    for (int64_t i = 0; i < N; ++i) {
        const uint64_t low = bits ? codes[i] & ((((uint64_t)1) << (3 * bits)) - 1) : 0;
        uint32_t x, y, z;
        if (curve) hilbert_cell(low, bits, &x, &y, &z);
        else zorder_cell(low, bits, &x, &y, &z);
        coords[4 * i + 0] = (int32_t)(codes[i] >> (3 * bits));
        coords[4 * i + 1] = (int32_t)x;
        coords[4 * i + 2] = (int32_t)y;
        coords[4 * i + 3] = (int32_t)z;
    }
    return ORACLE_OK;
}

/*
 * Input gradient by its definition with separate row counts: the R rows of
 * dY (lists nbr [R][27]) scatter W_k dY[i] into the Nx rows of dX.  The regular
 * (strided / transposed) convolution below uses it, where the rows of dY and
 * the rows of dX are different voxel sets.
 */
void oracle_dgrad_scatter_to(const uint32_t* nbr, int64_t R, const double* dY, const double* W,
                             int Cin, int Cout, int64_t Nx, double* dX)
{
    memset(dX, 0, (size_t)Nx * Cin * sizeof(double));
    for (int64_t i = 0; i < R; ++i) {
        const double* g = dY + i * Cout;
        for (int k = 0; k < 27; ++k) {
            uint32_t j = nbr[i * 27 + k];
            if (j == ORACLE_NONE) continue;
            double* d = dX + (int64_t)j * Cin;
            for (int ci = 0; ci < Cin; ++ci) {
                const double* w = W + ((int64_t)k * Cin + ci) * Cout;
                double s = 0.0;
                for (int co = 0; co < Cout; ++co) s += w[co] * g[co];
                d[ci] += s;
            }
        }
    }
}

/*
 * Regular (non-submanifold) sparse convolution map: "Contribution Tasks —
 * JeffreyXiang/FlexGEMM", §二 module table and key functions (sparse_conv3d,
 * kernels.cuda.spconv sparse_neighbor_map): the output sites differ from the
 * input sites (strided down-sampling, and its transposed up-sampling).  The
 * pages give no formula; the reading taken is the convolution that
 * torch.nn.functional.conv3d computes on the densified grid, with kernel K per
 * axis (K = 3: padding 1, taps t - 1 for t in {0,1,2}; K = 2: padding 0, taps
 * t in {0,1}) and stride s, evaluated only at the output sites whose window
 * holds at least one active input:
 *   output grid: Xo = (X + 2p - K) / s + 1 (floor), likewise Yo, Zo, same batch
 *   tap k = (tx*K + ty)*K + tz  <->  offset d = (tx - p, ty - p, tz - p)
 *   o is active  iff  some input sits at s*o + d_k
 *   down[o][k] = input row at s*o + d_k (or NONE); columns k >= K^3 are NONE
 *   up[j][k]   = output row o with s*o + d_k = coord_j (or NONE)
 * Output rows are numbered in ascending linear key ((b*Xo + x)*Yo + y)*Zo + z.
 * The strided convolution is then out[o] = bias + sum_k W_k^T f[down[o][k]];
 * its input gradient scatters along down (oracle_dgrad_scatter_to) and its
 * weight gradient is oracle_wgrad over down.  The transposed convolution maps
 * the output sites back to the input sites: out[j] = bias + sum_k W_k^T
 * g[up[j][k]] (torch conv_transpose3d with the same K, s, p).
 * coords_out must hold N * K^3 rows, down N * K^3 rows of 27, up N rows of 27.
 * Returns ORACLE_BAD_ARG for K not in {2,3}, s not in {1,2} or a grid with no
 * output cell, ORACLE_OUT_OF_RANGE / ORACLE_DUPLICATE as oracle_nbrmap.
 */
typedef struct { uint64_t key; int32_t b, x, y, z; } cand_entry;

static int cmp_cand(const void* a, const void* b)
{
    const uint64_t ka = ((const cand_entry*)a)->key, kb = ((const cand_entry*)b)->key;
    return ka < kb ? -1 : (ka > kb ? 1 : 0);
}

int oracle_sparse_map(const int32_t* coords, int64_t N, int B, int X, int Y, int Z, int K, int s,
                      int64_t* N_out, int32_t* coords_out, uint32_t* down, uint32_t* up)
{
    if (N < 0 || B <= 0 || X <= 0 || Y <= 0 || Z <= 0) return ORACLE_BAD_ARG;
    if ((K != 2 && K != 3) || (s != 1 && s != 2)) return ORACLE_BAD_ARG;
    const int p = K == 3 ? 1 : 0;
    const int64_t Xo = (X + 2 * p - K) / s + 1, Yo = (Y + 2 * p - K) / s + 1, Zo = (Z + 2 * p - K) / s + 1;
    if (X + 2 * p < K || Y + 2 * p < K || Z + 2 * p < K) return ORACLE_BAD_ARG;
    const int T = K * K * K;
    *N_out = 0;
    if (N == 0) return ORACLE_OK;
    /* the input sites, as a dictionary (also rejects bad or repeated coordinates) */
    uint32_t* nbr_sub = (uint32_t*)malloc((size_t)N * 27 * sizeof(uint32_t));
    uint32_t* mask_sub = (uint32_t*)malloc((size_t)N * sizeof(uint32_t));
    dict_entry* din = (dict_entry*)malloc((size_t)N * sizeof(dict_entry));
    cand_entry* cand = (cand_entry*)malloc((size_t)N * T * sizeof(cand_entry));
    if (!nbr_sub || !mask_sub || !din || !cand) {
        free(nbr_sub); free(mask_sub); free(din); free(cand);
        return ORACLE_NO_MEMORY;
    }
    int rc = oracle_nbrmap(coords, N, B, X, Y, Z, nbr_sub, mask_sub);
    free(nbr_sub);
    free(mask_sub);
    if (rc != ORACLE_OK) {
        free(din); free(cand);
        return rc;
    }
    for (int64_t i = 0; i < N; ++i) {
        const int32_t* c = coords + 4 * i;
        din[i].key = linear_key(c[0], c[1], c[2], c[3], X, Y, Z);
        din[i].row = i;
    }
    qsort(din, (size_t)N, sizeof(dict_entry), cmp_entry);
    /* every output whose window holds an input: o = (c - d_k) / s where divisible */
    int64_t nc = 0;
    for (int64_t i = 0; i < N; ++i) {
        const int32_t* c = coords + 4 * i;
        for (int k = 0; k < T; ++k) {
            const int d[3] = {k / (K * K) - p, (k / K) % K - p, k % K - p};
            int64_t o[3];
            int ok = 1;
            for (int a = 0; a < 3; ++a) {
                const int64_t v = (int64_t)c[1 + a] - d[a];
                const int64_t lim = a == 0 ? Xo : (a == 1 ? Yo : Zo);
                if (v < 0 || v % s != 0 || v / s >= lim) ok = 0;
                o[a] = ok ? v / s : 0;
            }
            if (!ok) continue;
            cand[nc].key = linear_key(c[0], o[0], o[1], o[2], Xo, Yo, Zo);
            cand[nc].b = c[0];
            cand[nc].x = (int32_t)o[0];
            cand[nc].y = (int32_t)o[1];
            cand[nc].z = (int32_t)o[2];
            ++nc;
        }
    }
    qsort(cand, (size_t)nc, sizeof(cand_entry), cmp_cand);
    int64_t no = 0;
    for (int64_t i = 0; i < nc; ++i) {
        if (no > 0 && cand[i].key == cand[no - 1].key) continue;
        cand[no++] = cand[i];
    }
    for (int64_t o = 0; o < no; ++o) {
        coords_out[4 * o + 0] = cand[o].b;
        coords_out[4 * o + 1] = cand[o].x;
        coords_out[4 * o + 2] = cand[o].y;
        coords_out[4 * o + 3] = cand[o].z;
    }
    /* down: the input row at s*o + d_k */
    for (int64_t o = 0; o < no; ++o) {
        for (int k = 0; k < 27; ++k) {
            uint32_t j = ORACLE_NONE;
            if (k < T) {
                const int64_t x = (int64_t)s * cand[o].x + k / (K * K) - p;
                const int64_t y = (int64_t)s * cand[o].y + (k / K) % K - p;
                const int64_t z = (int64_t)s * cand[o].z + k % K - p;
                if (x >= 0 && x < X && y >= 0 && y < Y && z >= 0 && z < Z) {
                    dict_entry probe;
                    probe.key = linear_key(cand[o].b, x, y, z, X, Y, Z);
                    probe.row = 0;
                    const dict_entry* hit = (const dict_entry*)bsearch(&probe, din, (size_t)N,
                                                                       sizeof(dict_entry), cmp_entry);
                    if (hit) j = (uint32_t)hit->row;
                }
            }
            down[o * 27 + k] = j;
        }
    }
    /* up: the output row o with s*o + d_k = coord_j (the outputs are sorted by key) */
    for (int64_t i = 0; i < N; ++i) {
        const int32_t* c = coords + 4 * i;
        for (int k = 0; k < 27; ++k) {
            uint32_t oi = ORACLE_NONE;
            if (k < T) {
                const int d[3] = {k / (K * K) - p, (k / K) % K - p, k % K - p};
                int64_t o[3];
                int ok = 1;
                for (int a = 0; a < 3; ++a) {
                    const int64_t v = (int64_t)c[1 + a] - d[a];
                    const int64_t lim = a == 0 ? Xo : (a == 1 ? Yo : Zo);
                    if (v < 0 || v % s != 0 || v / s >= lim) ok = 0;
                    o[a] = ok ? v / s : 0;
                }
                if (ok) {
                    cand_entry probe;
                    probe.key = linear_key(c[0], o[0], o[1], o[2], Xo, Yo, Zo);
                    const cand_entry* hit = (const cand_entry*)bsearch(&probe, cand, (size_t)no,
                                                                       sizeof(cand_entry), cmp_cand);
                    if (hit) oi = (uint32_t)(hit - cand);
                }
            }
            up[i * 27 + k] = oi;
        }
    }
    *N_out = no;
    free(din);
    free(cand);
    return ORACLE_OK;
}
