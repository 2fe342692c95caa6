/*
 * qlora_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU implementation of the QLoRA-adapted
 * linear layer, in fp64.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library; the product path
 * never does.  It shares no code, header or table with the CUDA library.
 *
 * Sources (web pages this follows):
 *  - "Introducing Unsloth: LLM 训练提速 30 倍", section 手动 Autograd:
 *      Q = X(W_q + A_q B_q) with W frozen and only A, B trained; the
 *      backward needs the derivatives w.r.t. A, B and the input; the
 *      chain product is bracketed through the skinny rank-r factors.
 *  - "利用 Unsloth 和 NVIDIA 硬件加速 LLM 训练", section 1 (4-bit):
 *      the 4-bit weight is dequantised to 16-bit at compute time.
 *  - "UnSloth极速微调", hardware/precision paragraphs: bf16 rather than fp16.
 *  - "Unsloth如何实现2倍速训练", section 2.2: frozen weights get no gradient.
 *
 * Notation (row-major everywhere):
 *   X  [M,K]     activations            dY [M,N]  upstream gradient
 *   W  [N,K]     frozen, 4-bit: idx (two codes per byte, even k in the low
 *                nibble), one fp32 absmax per 64 consecutive elements of the
 *                row-major flattening, a 16-entry fp32 codebook
 *   A  [K,R]     R = nseg*r   (segment j uses columns j*r .. j*r+r-1)
 *   B  [r,N]     column n belongs to segment seg(n) (seg_n[] widths)
 *   s            LoRA scale
 *
 *   deq(W)[n,k] = bf16( fp32( codebook[idx[n,k]] * absmax[(n*K+k)/64] ) )
 *   XA[m,J]  = sum_k X[m,k] A[k,J]
 *   Y[m,n]   = sum_k X[m,k] Wd[n,k] + s * sum_c XA[m, seg(n)*r+c] B[c,n]
 *   G[m,J]   = sum_{n in segment J/r} dY[m,n] B[J%r, n]
 *   dX[m,k]  = sum_n dY[m,n] Wd[n,k] + s * sum_J G[m,J] A[k,J]
 *   dA[k,J]  = s * sum_m X[m,k] G[m,J]
 *   dB[c,n]  = s * sum_m XA[m, seg(n)*r+c] dY[m,n]
 *
 * Every sum runs in ascending index order in double precision.  The linear
 * functions take their operands as double arrays (the caller converts the
 * bf16 inputs exactly) and compute only the requested output indices, so that
 * full-size problems can be checked on a sample.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Rounding                                                                  */
/* ------------------------------------------------------------------------ */

/* fp32 -> bf16, round to nearest, ties to even, from the bit pattern.
 * Keeps the sign of zero; an fp32 value whose rounding exceeds the bf16 range
 * becomes +-inf (the carry runs into the exponent); NaN keeps a quiet NaN. */
uint16_t oracle_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);           /* NaN stays NaN */
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Dequantisation ("4-bit dequantised to 16-bit at compute time")            */
/* ------------------------------------------------------------------------ */

/* code of element (n,k): byte (n*K+k)/2 of the packed array, low nibble for
 * even k, high nibble for odd k. */
static unsigned code_at(const uint8_t *idx, int64_t K, int64_t n, int64_t k)
{
    uint8_t byte = idx[(n * K + k) / 2];
    return (k % 2 == 0) ? (byte & 0x0fu) : (byte >> 4);
}

/* out_f32 (nullable) [N,K]: the fp32 product; out_bf16 (nullable) [N,K]: its
 * bf16 rounding.  The product of two fp32 numbers is exact in double (24+24
 * significant bits), so converting it to float is the correctly rounded fp32
 * multiply. */
void oracle_dequant(const uint8_t *idx, const float *absmax, const float *codebook,
                    int64_t N, int64_t K, int64_t block,
                    float *out_f32, uint16_t *out_bf16)
{
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            int64_t e = n * K + k;
            double p = (double)codebook[code_at(idx, K, n, k)] * (double)absmax[e / block];
            float w32 = (float)p;
            if (out_f32) out_f32[e] = w32;
            if (out_bf16) out_bf16[e] = oracle_bf16_rne(w32);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Quantisation: the stored form the path starts from (the pages load the    */
/* model with load_in_4bit=True -- "利用 Unsloth 和 NVIDIA 硬件加速 LLM 训练",  */
/* section 代码实战; the 4-bit format itself is the reading in the header)    */
/* ------------------------------------------------------------------------ */

/* w [N,K] fp32 -> idx [N,K/2] (two codes per byte, even k in the low nibble)
 * and absmax [N*K/block].  For each block of `block` consecutive elements of
 * the row-major flattening: absmax = max |w| over the block; each element
 * takes the code i that minimises |t - codebook[i]|, t = w / absmax computed
 * as a double division (t = 0 when absmax is 0), each distance a double
 * subtraction; the first (lowest) such i wins a tie.  The codebook need not
 * be sorted.  Inputs are finite. */
void oracle_quantize(const float *w, int64_t N, int64_t K, int64_t block, const float *codebook,
                     uint8_t *idx, float *absmax)
{
    memset(idx, 0, (size_t)(N * K / 2));
    for (int64_t b = 0; b < N * K / block; ++b) {
        float a = 0.0f;
        for (int64_t e = b * block; e < (b + 1) * block; ++e) {
            float v = w[e] < 0.0f ? -w[e] : w[e];
            if (v > a) a = v;
        }
        absmax[b] = a;
        for (int64_t e = b * block; e < (b + 1) * block; ++e) {
            double t = (a == 0.0f) ? 0.0 : (double)w[e] / (double)a;
            unsigned best = 0;
            double dbest = 0.0;
            for (unsigned i = 0; i < 16; ++i) {
                double d = t - (double)codebook[i];
                if (d < 0.0) d = -d;
                if (i == 0 || d < dbest) {
                    best = i;
                    dbest = d;
                }
            }
            idx[e / 2] |= (uint8_t)((e % 2 == 0) ? best : (best << 4));
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Segment bookkeeping (several adapters side by side over N, e.g. fused QKV) */
/* ------------------------------------------------------------------------ */

static int64_t seg_of(const int64_t *seg_n, int64_t nseg, int64_t n)
{
    int64_t off = 0;
    for (int64_t j = 0; j < nseg; ++j) {
        if (n < off + seg_n[j]) return j;
        off += seg_n[j];
    }
    return nseg - 1;  /* unreachable for valid n */
}

static int64_t seg_begin(const int64_t *seg_n, int64_t j)
{
    int64_t off = 0;
    for (int64_t i = 0; i < j; ++i) off += seg_n[i];
    return off;
}

/* XA[m,J] = sum_k X[m,k] A[k,J] */
static double xa_elem(const double *X, const double *A, int64_t K, int64_t R,
                      int64_t m, int64_t J)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += X[m * K + k] * A[k * R + J];
    return acc;
}

/* G[m,J] = sum over the columns n of segment J/r of dY[m,n] B[J%r,n] */
static double g_elem(const double *dY, const double *B, int64_t N, int64_t r,
                     const int64_t *seg_n, int64_t m, int64_t J)
{
    int64_t j = J / r, c = J % r;
    int64_t n0 = seg_begin(seg_n, j), n1 = n0 + seg_n[j];
    double acc = 0.0;
    for (int64_t n = n0; n < n1; ++n) acc += dY[m * N + n] * B[c * N + n];
    return acc;
}

/* ------------------------------------------------------------------------ */
/* Forward: rows[] of XA and Y                                                */
/* ------------------------------------------------------------------------ */

/* XA_out [nrows, R], Y_out [nrows, N]; row i holds output row rows[i]. */
void oracle_forward_rows(const double *X, const double *Wd, const double *A, const double *B,
                         int64_t M, int64_t N, int64_t K, int64_t r, int64_t nseg,
                         const int64_t *seg_n, double s,
                         const int64_t *rows, int64_t nrows,
                         double *XA_out, double *Y_out)
{
    int64_t R = nseg * r;
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows[i];
        double *xa = XA_out + i * R;
        for (int64_t J = 0; J < R; ++J) xa[J] = xa_elem(X, A, K, R, m, J);
        for (int64_t n = 0; n < N; ++n) {
            double base = 0.0;
            for (int64_t k = 0; k < K; ++k) base += X[m * K + k] * Wd[n * K + k];
            int64_t j = seg_of(seg_n, nseg, n);
            double lora = 0.0;
            for (int64_t c = 0; c < r; ++c) lora += xa[j * r + c] * B[c * N + n];
            Y_out[i * N + n] = base + s * lora;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Backward                                                                   */
/* ------------------------------------------------------------------------ */

/* G_out [nrows, R], dX_out [nrows, K] for the requested rows. */
void oracle_backward_dx_rows(const double *dY, const double *Wd, const double *A, const double *B,
                             int64_t M, int64_t N, int64_t K, int64_t r, int64_t nseg,
                             const int64_t *seg_n, double s,
                             const int64_t *rows, int64_t nrows,
                             double *G_out, double *dX_out)
{
    int64_t R = nseg * r;
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows[i];
        double *g = G_out + i * R;
        for (int64_t J = 0; J < R; ++J) g[J] = g_elem(dY, B, N, r, seg_n, m, J);
        for (int64_t k = 0; k < K; ++k) {
            double base = 0.0;
            for (int64_t n = 0; n < N; ++n) base += dY[m * N + n] * Wd[n * K + k];
            double lora = 0.0;
            for (int64_t J = 0; J < R; ++J) lora += g[J] * A[k * R + J];
            dX_out[i * K + k] = base + s * lora;
        }
    }
}

/* dA at (kidx[a], Jidx[b]) -> dA_out[a*nJ + b], summing over all M rows. */
void oracle_backward_da(const double *X, const double *dY, const double *B,
                        int64_t M, int64_t N, int64_t K, int64_t r, int64_t nseg,
                        const int64_t *seg_n, double s,
                        const int64_t *kidx, int64_t nk, const int64_t *Jidx, int64_t nJ,
                        double *dA_out)
{
    (void)nseg;
    double *gcol = (double *)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1));
    for (int64_t b = 0; b < nJ; ++b) {
        int64_t J = Jidx[b];
#pragma omp parallel for schedule(static)
        for (int64_t m = 0; m < M; ++m) gcol[m] = g_elem(dY, B, N, r, seg_n, m, J);
#pragma omp parallel for schedule(static)
        for (int64_t a = 0; a < nk; ++a) {
            int64_t k = kidx[a];
            double acc = 0.0;
            for (int64_t m = 0; m < M; ++m) acc += X[m * K + k] * gcol[m];
            dA_out[a * nJ + b] = s * acc;
        }
    }
    free(gcol);
}

/* dB at (cidx[a], nidx[b]) -> dB_out[a*nn + b], summing over all M rows. */
void oracle_backward_db(const double *X, const double *dY, const double *A,
                        int64_t M, int64_t N, int64_t K, int64_t r, int64_t nseg,
                        const int64_t *seg_n, double s,
                        const int64_t *cidx, int64_t nc, const int64_t *nidx, int64_t nn,
                        double *dB_out)
{
    int64_t R = nseg * r;
    /* XA columns, computed once per (segment, c) actually used */
    double *xacol = (double *)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1));
    for (int64_t a = 0; a < nc; ++a) {
        int64_t c = cidx[a];
        for (int64_t j = 0; j < nseg; ++j) {
            int used = 0;
            for (int64_t b = 0; b < nn; ++b)
                if (seg_of(seg_n, nseg, nidx[b]) == j) { used = 1; break; }
            if (!used) continue;
            int64_t J = j * r + c;
#pragma omp parallel for schedule(static)
            for (int64_t m = 0; m < M; ++m) xacol[m] = xa_elem(X, A, K, R, m, J);
#pragma omp parallel for schedule(static)
            for (int64_t b = 0; b < nn; ++b) {
                int64_t n = nidx[b];
                if (seg_of(seg_n, nseg, n) != j) continue;
                double acc = 0.0;
                for (int64_t m = 0; m < M; ++m) acc += xacol[m] * dY[m * N + n];
                dB_out[a * nn + b] = s * acc;
            }
        }
    }
    free(xacol);
}

/* Number of worker threads the OpenMP runtime will use (1 without OpenMP),
 * and a way to change it (the benchmark also times the oracle on one core). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
void oracle_set_num_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
#else
int oracle_num_threads(void) { return 1; }
void oracle_set_num_threads(int n) { (void)n; }
#endif
