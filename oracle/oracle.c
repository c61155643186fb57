/*
 * oracle.c -- plain CPU oracle for the tile-wise mixed-precision CG hot path.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg load this library. The GPU library neither links nor calls it,
 * and the two share no source, header, table or helper.
 *
 * Everything here is single-threaded, written for a reader to check by eye, and
 * computed in IEEE binary64 unless the method fixes another format. Build with
 * -ffp-contract=off so that no a*b+c is ever fused: every product and every sum is
 * rounded on its own, on every host.
 *
 * The method is the one of "EvoCG: Self-Evolving Precision Control for Faster
 * Conjugate Gradient" (arXiv 2611.04469), cited below as "EvoCG" with the section,
 * equation or figure each function restates.
 *
 * Readings of points the paper leaves open (also listed in the design notes):
 *  - Rounding to FP32/BF16 is IEEE round-to-nearest-even, taken once, directly from
 *    the FP64 value (BF16 is never reached through FP32). No flush-to-zero.
 *  - The per-column quantisation factor of EvoCG §3.3.2 is a power of two,
 *    s_j = 2^e_j with e_j = floor(log2 max_i |a_ij|) clamped to [-100, 100]
 *    (e_j = 0 for an empty column). The FP32/BF16 value streams hold
 *    RN(a_ij / s_j); the FP64 stream holds a_ij itself.
 *  - A low-precision tile multiplies RN(a_ij / s_j) by RN(x_j) (the x entry rounded
 *    to the tile's own format) and scales the product by s_j. Both factors have at
 *    most 24 significant bits, so the FP64 product is exact.
 *  - Tiles are square, T x T (R = C = T), as the workloads fix them. Inside a tile the
 *    layout is EvoCG's CSC (§3.3.2, Fig. 4(b)): colPtr of length T+1 relative to the
 *    tile's first entry, rowIdx relative to the row block's first row, entries of a
 *    column in ascending row. Padding of a column to even length with the sentinel
 *    row index T ("R" in Fig. 4(b)) and zero values is a build parameter, pad = 2
 *    (the paper) or pad = 1 (no padding). The N/C entries of Fig. 4(a) are read as
 *    placeholders: there is no padding of the tile list.
 *  - The reuse interval K* (EvoCG §3.4) is the largest of 1, 2, 4, ... for which fewer than
 *    10% of the upward transitions in a per-iteration decision log would be delayed, a
 *    transition at iteration k being delayed when the decision of iteration K*floor(k/K)
 *    has a lower precision than iteration k's.
 *
 * Parity pins live in tests/test_oracle_*.py. The MLP controller is pinned only
 * through special cases and invariances (its weights are seeded, not trained):
 * parity partially pinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status codes, same meaning as the GPU library's (the values are restated here,
 * not shared). */
enum { ORA_OK = 0, ORA_EINVAL = 1, ORA_ENOMEM = 2, ORA_ENOTCONV = 4, ORA_EBREAKDOWN = 5 };

/* Precision codes of EvoCG Eq. 9: 0 = FP64, 1 = FP32, 2 = BF16. */
enum { P_FP64 = 0, P_FP32 = 1, P_BF16 = 2 };

/* ------------------------------------------------------------------------ */
/* Rounding (IEEE 754 round-to-nearest, ties-to-even).                       */
/* ------------------------------------------------------------------------ */

/* Round x to a binary format with `frac_bits` stored fraction bits and normal
 * exponents [emin, emax]: the result is returned as an FP64 value that the
 * target format holds exactly. The quantum of the binade of x (or of the
 * subnormal range) is 2^q; x / 2^q is rounded to the nearest integer with
 * ties to even (nearbyint under the default rounding mode), then scaled back.
 * Magnitudes that round above the largest finite value become infinities. */
double ora_round_to_format(double x, int frac_bits, int emin, int emax)
{
    if (isnan(x) || isinf(x) || x == 0.0)
        return x;
    int e2;
    frexp(fabs(x), &e2);          /* |x| = f * 2^e2, f in [0.5, 1) */
    int lead = e2 - 1;            /* exponent of the leading bit */
    if (lead < emin)
        lead = emin;              /* subnormal range: fixed quantum */
    int q = lead - frac_bits;
    double r = nearbyint(ldexp(x, -q));
    double y = ldexp(r, q);
    double maxfinite = ldexp(2.0 - ldexp(1.0, -frac_bits), emax);
    if (fabs(y) > maxfinite)
        y = copysign(INFINITY, x);
    return y;
}

double ora_round_f32(double x) { return ora_round_to_format(x, 23, -126, 127); }
double ora_round_bf16(double x) { return ora_round_to_format(x, 7, -126, 127); }

/* Storage encodings of rounded values. */
static float f32_of(double x) { return (float)ora_round_f32(x); }  /* exact cast */
static uint16_t bf16_bits_of(double x)
{
    float f = (float)ora_round_bf16(x);  /* a BF16 value is exactly an FP32 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);          /* its low 16 bits are zero */
}

void ora_round_f32_array(int64_t n, const double *x, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f32_of(x[i]);
}
void ora_round_bf16_array(int64_t n, const double *x, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_bits_of(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Plain CSR SpMV in FP64 (EvoCG §2.1: the SpMV of the CG recurrence).       */
/* ------------------------------------------------------------------------ */
void ora_csr_spmv(int64_t n, const int64_t *rp, const int32_t *ci, const double *v,
                  const double *x, double *y)
{
    for (int64_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (int64_t k = rp[i]; k < rp[i + 1]; ++k) s += v[k] * x[ci[k]];
        y[i] = s;
    }
}

/* Check the CSR input: monotone row pointers, columns in range and strictly
 * ascending within each row, finite values. */
int ora_csr_check(int64_t n, const int64_t *rp, const int32_t *ci, const double *v)
{
    if (n < 0 || rp[0] != 0) return ORA_EINVAL;
    for (int64_t i = 0; i < n; ++i) {
        if (rp[i + 1] < rp[i]) return ORA_EINVAL;
        for (int64_t k = rp[i]; k < rp[i + 1]; ++k) {
            if (ci[k] < 0 || ci[k] >= n) return ORA_EINVAL;
            if (k > rp[i] && ci[k] <= ci[k - 1]) return ORA_EINVAL;
            if (!isfinite(v[k])) return ORA_EINVAL;
        }
    }
    return ORA_OK;
}

/* ------------------------------------------------------------------------ */
/* Column quantisation exponents (EvoCG §3.3.2: one factor per column,       */
/* shared by FP32 and BF16).                                                 */
/* ------------------------------------------------------------------------ */
void ora_col_exp(int64_t n, const int64_t *rp, const int32_t *ci, const double *v, int8_t *e)
{
    double *mx = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
    for (int64_t i = 0; i < n; ++i)
        for (int64_t k = rp[i]; k < rp[i + 1]; ++k)
            if (fabs(v[k]) > mx[ci[k]]) mx[ci[k]] = fabs(v[k]);
    for (int64_t j = 0; j < n; ++j) {
        int ex = 0;
        if (mx[j] > 0.0) {
            int e2;
            frexp(mx[j], &e2);
            ex = e2 - 1;           /* floor(log2(max |a_ij|)) */
            if (ex < -100) ex = -100;
            if (ex > 100) ex = 100;
        }
        e[j] = (int8_t)ex;
    }
    free(mx);
}

/* ------------------------------------------------------------------------ */
/* Tile-CSC layout (EvoCG §3.3.1 and Fig. 4(a): CSR over row blocks of       */
/* tiles; §3.3.2 and Fig. 4(b): each tile stored as CSC, three value streams */
/* over one set of indices, columns padded to even length with a sentinel    */
/* row index).                                                               */
/* ------------------------------------------------------------------------ */

/* One stored entry of a row block: its global column, its row within the block, and
 * its index in the CSR arrays. */
typedef struct {
    int32_t col;
    int32_t lrow;
    int64_t k;
} ora_entry;

/* Column-major order inside a row block: by column, then by row. */
static int entry_col_row(const void *a, const void *b)
{
    const ora_entry *x = (const ora_entry *)a, *y = (const ora_entry *)b;
    if (x->col != y->col) return x->col < y->col ? -1 : 1;
    return (x->lrow > y->lrow) - (x->lrow < y->lrow);
}

/* The entries of row block rb (rows rb*T .. rb*T + T - 1), sorted column-major into
 * buf; returns how many there are. */
static int64_t row_block_entries(int64_t n, const int64_t *rp, const int32_t *ci, int T,
                                 int64_t rb, ora_entry *buf)
{
    int64_t r0 = rb * T, r1 = (r0 + T < n) ? r0 + T : n, m = 0;
    for (int64_t i = r0; i < r1; ++i)
        for (int64_t k = rp[i]; k < rp[i + 1]; ++k) {
            buf[m].col = ci[k];
            buf[m].lrow = (int32_t)(i - r0);
            buf[m].k = k;
            m++;
        }
    qsort(buf, (size_t)m, sizeof(ora_entry), entry_col_row);
    return m;
}

/* Largest number of entries of one row block (the size of the sort buffer). */
static int64_t max_row_block_entries(int64_t n, const int64_t *rp, int T)
{
    int64_t best = 0;
    for (int64_t r0 = 0; r0 < n; r0 += T) {
        int64_t r1 = (r0 + T < n) ? r0 + T : n;
        if (rp[r1] - rp[r0] > best) best = rp[r1] - rp[r0];
    }
    return best;
}

/* Entries a column of c stored entries occupies: c, rounded up to a multiple of pad
 * (pad = 2 is the paper's padding to a multiple of two; pad = 1 stores no padding). */
static int64_t padded(int64_t c, int pad) { return (c + pad - 1) / pad * pad; }

/* Count the nonempty T x T tiles, the stored entries, and the entries of the padded
 * streams (stored entries plus sentinels). */
int ora_tile_csc_count(int64_t n, const int64_t *rp, const int32_t *ci, int T, int pad,
                       int64_t *ntiles_out, int64_t *nnz_out, int64_t *nnzp_out)
{
    if (T < 1 || T > 64 || n < 0 || (pad != 1 && pad != 2)) return ORA_EINVAL;
    int64_t nrb = (n + T - 1) / T, ntiles = 0, nnzp = 0;
    ora_entry *buf = (ora_entry *)malloc(sizeof(ora_entry) * (size_t)(max_row_block_entries(n, rp, T) + 1));
    if (!buf) return ORA_ENOMEM;
    for (int64_t rb = 0; rb < nrb; ++rb) {
        int64_t m = row_block_entries(n, rp, ci, T, rb, buf);
        for (int64_t e = 0; e < m;) {
            int64_t cb = buf[e].col / T;
            ntiles++;
            while (e < m && buf[e].col / T == cb) {      /* the columns of tile (rb, cb) */
                int64_t c0 = e;
                while (e < m && buf[e].col == buf[c0].col) e++;
                nnzp += padded(e - c0, pad);
            }
        }
    }
    free(buf);
    *ntiles_out = ntiles;
    *nnz_out = (n > 0) ? rp[n] : 0;
    *nnzp_out = nnzp;
    return ORA_OK;
}

/* Fill the Tile-CSC layout.
 * Inter-tile level (EvoCG §3.3.1, Fig. 4(a)): row block rb holds tiles
 * tileRowPtr[rb] .. tileRowPtr[rb+1]-1, listed in ascending column block tileColIdx.
 * Intra-tile level (EvoCG §3.3.2, Fig. 4(b)): tile t's entries start at tileNnzOff[t] in
 * the padded streams (tileNnzOff has ntiles+1 entries); colPtr[t*(T+1) + c] .. [c+1] is
 * the range of local column c relative to that start (colPtr[t*(T+1)] = 0); inside a
 * column the entries are in ascending row and rowIdx holds each entry's row relative to
 * the row block's first row. With pad = 2 a column with an odd count gets one more
 * entry: rowIdx = T (the sentinel row index R of Fig. 4(b), one past the last row) and
 * +0 in all three value streams. v64 holds a_ij; v32 and v16 hold a_ij / s_j rounded
 * once to FP32 / BF16, with s_j = 2^colExp[j]. */
int ora_tile_csc_build(int64_t n, const int64_t *rp, const int32_t *ci, const double *v, int T,
                       int pad, int64_t *tileRowPtr, int32_t *tileColIdx, int64_t *tileNnzOff,
                       uint16_t *colPtr, uint8_t *rowIdx, double *v64, float *v32, uint16_t *v16,
                       int8_t *colExp)
{
    if (T < 1 || T > 64 || n < 0 || (pad != 1 && pad != 2)) return ORA_EINVAL;
    ora_col_exp(n, rp, ci, v, colExp);
    int64_t nrb = (n + T - 1) / T, t = 0, pos = 0;
    ora_entry *buf = (ora_entry *)malloc(sizeof(ora_entry) * (size_t)(max_row_block_entries(n, rp, T) + 1));
    if (!buf) return ORA_ENOMEM;
    tileRowPtr[0] = 0;
    for (int64_t rb = 0; rb < nrb; ++rb) {
        int64_t m = row_block_entries(n, rp, ci, T, rb, buf);
        for (int64_t e = 0; e < m;) {
            int64_t cb = buf[e].col / T;
            uint16_t *cp = colPtr + t * (T + 1);
            tileColIdx[t] = (int32_t)cb;
            tileNnzOff[t] = pos;
            int64_t local = 0;              /* entries of this tile so far, pads included */
            int64_t next_col = 0;           /* local columns below it have their pointer set */
            while (e < m && buf[e].col / T == cb) {
                int64_t c = buf[e].col - cb * T;
                for (; next_col <= c; ++next_col) cp[next_col] = (uint16_t)local;
                int64_t c0 = e;
                while (e < m && buf[e].col == buf[c0].col) {
                    int64_t k = buf[e].k;
                    int ec = colExp[ci[k]];
                    rowIdx[pos + local] = (uint8_t)buf[e].lrow;
                    v64[pos + local] = v[k];
                    v32[pos + local] = f32_of(ldexp(v[k], -ec));
                    v16[pos + local] = bf16_bits_of(ldexp(v[k], -ec));
                    local++;
                    e++;
                }
                if (padded(e - c0, pad) > e - c0) {   /* sentinel-marked zero */
                    rowIdx[pos + local] = (uint8_t)T;
                    v64[pos + local] = 0.0;
                    v32[pos + local] = 0.0f;
                    v16[pos + local] = 0;
                    local++;
                }
            }
            for (; next_col <= T; ++next_col) cp[next_col] = (uint16_t)local;
            pos += local;
            t++;
        }
        tileRowPtr[rb + 1] = t;
    }
    tileNnzOff[t] = pos;
    free(buf);
    return ORA_OK;
}

/* Index of the tile (rb, cb) in the tile list, or -1. */
static int64_t find_tile(const int64_t *tileRowPtr, const int32_t *tileColIdx, int64_t rb, int64_t cb)
{
    /* binary search: the column blocks of a row block are ascending */
    int64_t lo = tileRowPtr[rb], hi = tileRowPtr[rb + 1];
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        if (tileColIdx[mid] < cb) lo = mid + 1; else hi = mid;
    }
    return (lo < tileRowPtr[rb + 1] && tileColIdx[lo] == cb) ? lo : -1;
}

/* ------------------------------------------------------------------------ */
/* Mixed-precision SpMV, the emulated operator of EvoCG Eq. 2 / Eq. 5:       */
/* y = (A + E(a)) x, where E(a) is exactly the rounding of each tile's       */
/* values, and of the x entries the tile reads, to the tile's format.        */
/* Computed from the CSR input, not from any tile layout: the tile list only */
/* names which format each (row block, column block) uses.                   */
/* ------------------------------------------------------------------------ */
void ora_mixed_spmv(int64_t n, const int64_t *rp, const int32_t *ci, const double *v, int T,
                    const int8_t *colExp, const int64_t *tileRowPtr, const int32_t *tileColIdx,
                    const uint8_t *tilePrec, const double *x, double *y)
{
    for (int64_t i = 0; i < n; ++i) {
        int64_t rb = i / T;
        double s = 0.0;
        for (int64_t k = rp[i]; k < rp[i + 1]; ++k) {
            int64_t j = ci[k];
            int prec = tilePrec ? tilePrec[find_tile(tileRowPtr, tileColIdx, rb, j / T)] : P_FP64;
            double term;
            if (prec == P_FP64) {
                term = v[k] * x[j];
            } else {
                int ej = colExp[j];
                double a_t, x_t;
                if (prec == P_FP32) {
                    a_t = ora_round_f32(ldexp(v[k], -ej));
                    x_t = ora_round_f32(x[j]);
                } else {
                    a_t = ora_round_bf16(ldexp(v[k], -ej));
                    x_t = ora_round_bf16(x[j]);
                }
                term = ldexp(a_t * x_t, ej);  /* exact: <= 48 significant bits */
            }
            s += term;
        }
        y[i] = s;
    }
}

/* ------------------------------------------------------------------------ */
/* Precision controllers. Both decide per column block i (the segment        */
/* p[iC : (i+1)C - 1] with C = T, EvoCG Eq. 8-10).                           */
/* ------------------------------------------------------------------------ */

/* Residual-threshold rule (EvoCG §4.7): m_i = max_j |p_i[j]|; BF16 when
 * m_i < 0.1*eps, FP32 when 0.1*eps <= m_i < eps, FP64 otherwise. A partial last
 * segment takes the entries that exist. */
void ora_ctrl_threshold(int64_t n, int T, const double *p, double eps, uint8_t *cbPrec)
{
    int64_t ncb = (n + T - 1) / T;
    double lo = 0.1 * eps;
    for (int64_t i = 0; i < ncb; ++i) {
        double m = 0.0;
        for (int64_t j = i * T; j < (i + 1) * T && j < n; ++j) {
            double a = fabs(p[j]);
            if (isnan(a) || a > m) m = a;  /* a NaN entry makes the maximum NaN */
        }
        /* NaN fails both tests and keeps FP64 */
        cbPrec[i] = (m < lo) ? P_BF16 : (m < eps) ? P_FP32 : P_FP64;
    }
}

/* Policy MLP (EvoCG §3.2.3 with hidden sizes [64, 64] from §4.1): input
 * phi = p_i / max(||p_i||_2, delta) (Eq. 8; a partial last segment is padded
 * with zeros), two ReLU layers, a 3-way head; the action is the argmax of the
 * logits, the lowest code (highest precision) on a tie. Weights are row-major
 * (out, in) FP32; the arithmetic here is FP64. logits may be NULL. */
void ora_ctrl_mlp(int64_t n, int T, const double *p, int H1, int H2,
                  const float *W1, const float *b1, const float *W2, const float *b2,
                  const float *W3, const float *b3, double delta, uint8_t *cbPrec,
                  double *logits)
{
    int64_t ncb = (n + T - 1) / T;
    double *phi = (double *)malloc(sizeof(double) * (size_t)T);
    double *h1 = (double *)malloc(sizeof(double) * (size_t)H1);
    double *h2 = (double *)malloc(sizeof(double) * (size_t)H2);
    for (int64_t i = 0; i < ncb; ++i) {
        double ss = 0.0;
        for (int c = 0; c < T; ++c) {
            int64_t j = i * T + c;
            phi[c] = (j < n) ? p[j] : 0.0;
            ss += phi[c] * phi[c];
        }
        double nrm = sqrt(ss);
        double den = (nrm > delta) ? nrm : delta;
        for (int c = 0; c < T; ++c) phi[c] = phi[c] / den;
        for (int o = 0; o < H1; ++o) {
            double s = (double)b1[o];
            for (int c = 0; c < T; ++c) s += (double)W1[o * T + c] * phi[c];
            h1[o] = s > 0.0 ? s : 0.0;
        }
        for (int o = 0; o < H2; ++o) {
            double s = (double)b2[o];
            for (int c = 0; c < H1; ++c) s += (double)W2[o * H1 + c] * h1[c];
            h2[o] = s > 0.0 ? s : 0.0;
        }
        double z[3];
        for (int o = 0; o < 3; ++o) {
            double s = (double)b3[o];
            for (int c = 0; c < H2; ++c) s += (double)W3[o * H2 + c] * h2[c];
            z[o] = s;
        }
        int best = 0;
        for (int o = 1; o < 3; ++o)
            if (z[o] > z[best]) best = o;
        cbPrec[i] = (uint8_t)best;
        if (logits)
            for (int o = 0; o < 3; ++o) logits[i * 3 + o] = z[o];
    }
    free(phi); free(h1); free(h2);
}

/* ------------------------------------------------------------------------ */
/* CG / Jacobi-PCG with a precision map (EvoCG §2.1 Fig. 1, the SOVR lines   */
/* of Algorithm 1, §4.1 solver protocol, §4.6 Jacobi-PCG).                   */
/* ------------------------------------------------------------------------ */

typedef struct {
    int ctrl;            /* 0 = static map (tileMap, or all FP64 when NULL), 1 = threshold,
                            2 = MLP, 3 = replay: iteration k uses row k of `replay` (the last
                            row past its end), a column-block map per row */
    const uint8_t *tileMap;
    double eps;          /* threshold rule */
    int kstar;           /* controller interval, >= 1 */
    int H1, H2;
    const float *W1, *b1, *W2, *b2, *W3, *b3;
    double delta;
    const uint8_t *replay;   /* replayRows x ncb column-block codes (ctrl 3) */
    int64_t replayRows;
    uint8_t *logOut;         /* NULL, or logRows x ncb: row k = the column-block map in force
                                at iteration k of the controlled phase (ctrl 1, 2, 3) */
    int64_t logRows;
} ora_ctrl_t;

static double dot(int64_t n, const double *a, const double *b)
{
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

/* ||b - A x||_2 / ||b||_2 with plain CSR FP64 (the FP64 true-residual check of
 * EvoCG §4.3). */
double ora_true_residual(int64_t n, const int64_t *rp, const int32_t *ci, const double *v,
                         const double *b, const double *x)
{
    double *ax = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    ora_csr_spmv(n, rp, ci, v, x, ax);
    double num = 0.0, den = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double d = b[i] - ax[i];
        num += d * d;
        den += b[i] * b[i];
    }
    free(ax);
    return den > 0.0 ? sqrt(num) / sqrt(den) : sqrt(num);
}

/*
 * Solve A x = b from x0 = 0. Per iteration k (Hestenes-Stiefel order):
 *   controller on p_k when k mod kstar == 0 (Algorithm 1 decides before the SpMV),
 *   q = A~(map) p, sigma = p.q (breakdown if not finite and positive),
 *   alpha = rho / sigma, x += alpha p, r -= alpha q,
 *   hist[k+1] = ||r||_2 / ||r_0||_2, stop when <= rtol (recursive residual, §4.1),
 *   z = D^-1 r (Jacobi) or r, rho' = r.z, beta = rho'/rho, p = z + beta p.
 * With finish_fp64, a recursive convergence is followed by an FP64 true-residual
 * check; if it is above rtol, the solve continues from r = b - A x with every
 * tile in FP64 (the counter of iterations runs on). hist needs maxit+1 entries.
 * out[0] = iterations, out[1] = iterations at the first recursive convergence
 * (or -1), out[2] = restarts; fout[0] = final recursive relative residual,
 * fout[1] = FP64 true relative residual; prec_nnz[3] sums the stored entries
 * processed per precision over all SpMVs.
 */
int ora_cg(int64_t n, const int64_t *rp, const int32_t *ci, const double *v, int T,
           const int64_t *tileRowPtr, const int32_t *tileColIdx, const int8_t *colExp,
           const double *b, double *x, double rtol, int maxit, int jacobi,
           const ora_ctrl_t *ctrl, int finish_fp64, double *hist, int64_t *out,
           double *fout, int64_t *prec_nnz)
{
    int64_t nrb = (n + T - 1) / T, ncb = nrb;
    int64_t ntiles = tileRowPtr[nrb];
    size_t nb = sizeof(double) * (size_t)(n > 0 ? n : 1);
    double *r = (double *)malloc(nb), *z = (double *)malloc(nb), *p = (double *)malloc(nb);
    double *q = (double *)malloc(nb), *dinv = (double *)malloc(nb);
    uint8_t *map = (uint8_t *)malloc((size_t)(ntiles > 0 ? ntiles : 1));
    uint8_t *cbp = (uint8_t *)malloc((size_t)(ncb > 0 ? ncb : 1));
    int64_t *tnnz = (int64_t *)malloc(sizeof(int64_t) * (size_t)(ntiles > 0 ? ntiles : 1));
    int status = ORA_OK;
    out[0] = 0; out[1] = -1; out[2] = 0;
    prec_nnz[0] = prec_nnz[1] = prec_nnz[2] = 0;

    /* stored entries of each tile, for the precision census */
    for (int64_t t = 0; t < ntiles; ++t) tnnz[t] = 0;
    for (int64_t i = 0; i < n; ++i)
        for (int64_t k = rp[i]; k < rp[i + 1]; ++k)
            tnnz[find_tile(tileRowPtr, tileColIdx, i / T, ci[k] / T)]++;

    for (int64_t i = 0; i < n; ++i) {
        dinv[i] = 1.0;
        if (jacobi) {
            double d = 0.0;
            for (int64_t k = rp[i]; k < rp[i + 1]; ++k)
                if (ci[k] == i) d = v[k];
            if (!(d > 0.0)) { status = ORA_EINVAL; goto done; }
            dinv[i] = 1.0 / d;
        }
    }
    for (int64_t t = 0; t < ntiles; ++t)
        map[t] = (ctrl->ctrl == 0 && ctrl->tileMap) ? ctrl->tileMap[t] : P_FP64;

    for (int64_t i = 0; i < n; ++i) { x[i] = 0.0; r[i] = b[i]; }
    int allfp64 = 0, k = 0;
    double nr0 = sqrt(dot(n, r, r));
    hist[0] = 1.0;
    if (nr0 == 0.0) { fout[0] = 0.0; goto check; }

    for (;;) {  /* one pass per (re)start */
        for (int64_t i = 0; i < n; ++i) z[i] = jacobi ? dinv[i] * r[i] : r[i];
        for (int64_t i = 0; i < n; ++i) p[i] = z[i];
        double rho = dot(n, r, z);
        int converged = 0;
        while (k < maxit) {
            if (!allfp64 && ctrl->ctrl == 3) {
                int64_t row = k < ctrl->replayRows ? k : ctrl->replayRows - 1;
                for (int64_t cb = 0; cb < ncb; ++cb) cbp[cb] = ctrl->replay[row * ncb + cb];
                for (int64_t t = 0; t < ntiles; ++t) map[t] = cbp[tileColIdx[t]];
            } else if (!allfp64 && ctrl->ctrl != 0 && k % ctrl->kstar == 0) {
                if (ctrl->ctrl == 1)
                    ora_ctrl_threshold(n, T, p, ctrl->eps, cbp);
                else
                    ora_ctrl_mlp(n, T, p, ctrl->H1, ctrl->H2, ctrl->W1, ctrl->b1, ctrl->W2,
                                 ctrl->b2, ctrl->W3, ctrl->b3, ctrl->delta, cbp, NULL);
                for (int64_t t = 0; t < ntiles; ++t) map[t] = cbp[tileColIdx[t]];
            }
            if (!allfp64 && ctrl->ctrl != 0 && ctrl->logOut && k < ctrl->logRows)
                for (int64_t cb = 0; cb < ncb; ++cb) ctrl->logOut[k * ncb + cb] = cbp[cb];
            for (int64_t t = 0; t < ntiles; ++t) prec_nnz[map[t]] += tnnz[t];
            ora_mixed_spmv(n, rp, ci, v, T, colExp, tileRowPtr, tileColIdx, map, p, q);
            double sigma = dot(n, p, q);
            if (!(sigma > 0.0) || !isfinite(sigma)) { status = ORA_EBREAKDOWN; goto check; }
            double alpha = rho / sigma;
            for (int64_t i = 0; i < n; ++i) x[i] += alpha * p[i];
            for (int64_t i = 0; i < n; ++i) r[i] -= alpha * q[i];
            double rr = dot(n, r, r);
            k++;
            hist[k] = sqrt(rr) / nr0;
            fout[0] = hist[k];
            if (hist[k] <= rtol) { converged = 1; break; }
            for (int64_t i = 0; i < n; ++i) z[i] = jacobi ? dinv[i] * r[i] : r[i];
            double rho_new = dot(n, r, z);
            double beta = rho_new / rho;
            rho = rho_new;
            for (int64_t i = 0; i < n; ++i) p[i] = z[i] + beta * p[i];
        }
        if (!converged) { status = ORA_ENOTCONV; break; }
        if (out[1] < 0) out[1] = k;
        if (!finish_fp64) break;
        if (ora_true_residual(n, rp, ci, v, b, x) <= rtol) break;
        /* restart from the true residual with every tile in FP64 */
        allfp64 = 1;
        out[2]++;
        for (int64_t t = 0; t < ntiles; ++t) map[t] = P_FP64;
        ora_csr_spmv(n, rp, ci, v, x, q);
        for (int64_t i = 0; i < n; ++i) r[i] = b[i] - q[i];
        if (out[2] > 8) { status = ORA_ENOTCONV; break; }
    }
check:
    out[0] = k;
    fout[1] = ora_true_residual(n, rp, ci, v, b, x);
done:
    free(r); free(z); free(p); free(q); free(dinv); free(map); free(cbp); free(tnnz);
    return status;
}

/* Flat-argument wrapper of ora_cg for foreign-function callers. */
int ora_cg_flat(int64_t n, const int64_t *rp, const int32_t *ci, const double *v, int T,
                const int64_t *tileRowPtr, const int32_t *tileColIdx, const int8_t *colExp,
                const double *b, double *x, double rtol, int maxit, int jacobi,
                int ctrl_kind, const uint8_t *tileMap, double eps, int kstar,
                int H1, int H2, const float *W1, const float *b1, const float *W2,
                const float *b2, const float *W3, const float *b3, double delta,
                int finish_fp64, double *hist, int64_t *out, double *fout, int64_t *prec_nnz,
                const uint8_t *replay, int64_t replayRows, uint8_t *logOut, int64_t logRows)
{
    ora_ctrl_t c;
    c.ctrl = ctrl_kind; c.tileMap = tileMap; c.eps = eps; c.kstar = kstar > 0 ? kstar : 1;
    c.H1 = H1; c.H2 = H2; c.W1 = W1; c.b1 = b1; c.W2 = W2; c.b2 = b2; c.W3 = W3; c.b3 = b3;
    c.delta = delta;
    c.replay = replay; c.replayRows = replayRows; c.logOut = logOut; c.logRows = logRows;
    if (ctrl_kind == 3 && (!replay || replayRows < 1)) return ORA_EINVAL;
    return ora_cg(n, rp, ci, v, T, tileRowPtr, tileColIdx, colExp, b, x, rtol, maxit, jacobi,
                  &c, finish_fp64, hist, out, fout, prec_nnz);
}

/* ------------------------------------------------------------------------ */
/* Reuse interval K* (EvoCG §3.4, interval reuse scheduling).                */
/* ------------------------------------------------------------------------ */

/* For each candidate interval K = 1, 2, 4, ... (up to the largest power of two not above
 * `rows`), count over every column block i and iteration k >= 1 the upward transitions
 * (the block's code at k below its code at k-1: a higher precision) and, among them, those
 * that reusing every K-th decision would delay: the decision in force at k is the one of
 * iteration K*floor(k/K), and the transition is delayed when that decision's code is above
 * the code at k. frac[K index] = delayed / upward (0 with no upward transition); *kstar =
 * the largest K with frac below `limit` (1 if none is). Returns the number of candidates. */
int ora_kstar_select(const uint8_t *log, int64_t rows, int64_t ncb, double limit,
                     int *kstar, double *frac, int max_frac)
{
    int nc = 0;
    *kstar = 1;
    int64_t top = rows > 0 ? rows : 1;
    for (int64_t K = 1; K <= top; K *= 2) {
        int64_t up = 0, delayed = 0;
        for (int64_t i = 0; i < ncb; ++i) {
            for (int64_t k = 1; k < rows; ++k) {
                int before = log[(k - 1) * ncb + i];
                int now = log[k * ncb + i];
                if (now >= before) continue;          /* not an upward transition */
                up++;
                int64_t start = k - (k % K);          /* the window's decision iteration */
                if (log[start * ncb + i] > now) delayed++;
            }
        }
        double f = (up == 0) ? 0.0 : (double)delayed / (double)up;
        if (nc < max_frac) frac[nc] = f;
        nc++;
        if (f < limit && K > *kstar) *kstar = (int)K;
    }
    return nc;
}
