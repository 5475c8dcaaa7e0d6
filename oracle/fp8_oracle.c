/* fp8_oracle.c -- fp64 CPU oracle of the FP8 forward with incoherent
 * processing (test infrastructure only; never linked into the CUDA library).
 *
 * "Trois idées pour FA3" (marketmaker.cc), point 3: naive FP8 attention is
 * ruined by outlier coordinates; FA3 rotates the query and key vectors at
 * random before quantising them block by block, which spreads an outlier's
 * magnitude over all coordinates, and the page reports a 2.6x lower error than
 * naive FP8.  The page fixes neither the rotation, the block, the scale rule
 * nor how the probabilities are quantised; the readings taken here are:
 *
 *   rotation   Q^ = Q D H / d and K^ = K D H, with H the d x d Sylvester
 *              Hadamard matrix (H_ab = (-1)^popcount(a & b), H H^T = d I) and
 *              D = diag(signs), signs in {-1, +1} drawn by the caller; then
 *              Q^ K^^T = Q D H H^T D K^T / d = Q K^T exactly.  V is not rotated.
 *   blocks     one scale per block of `block` consecutive rows of Q^, K^ and V
 *              of one head (128 for the kernel; block >= N is one scale per
 *              head, the "naive" per-tensor scaling the comparison uses).
 *   scale      the smallest power of two sigma with amax / sigma <= 448 (the
 *              largest finite e4m3 value); sigma = 1 for an all-zero block.
 *   codes      e4m3 (sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 *              infinities, 448 the largest finite value) of x / sigma, rounded
 *              to nearest with ties to even, saturating at +-448.  The value
 *              quantised is x rounded to fp32, the precision the kernel takes
 *              the same decision in.
 *   forward    the online recurrence of "L'algorithme Flash Attention" over
 *              key blocks of 128, on the decoded operands:
 *                s_ij  = scale sigma_q sigma_k (q8_i . k8_j)
 *                m_new = max(m, max_j s_ij)
 *                P~_ij = exp(s_ij - m_new), quantised as e4m3(256 P~_ij)
 *                        (again from its fp32 value) for the P~ V product
 *                l     = l e^(m - m_new) + sum_j P~_ij  (the unquantised P~)
 *                O     = O e^(m - m_new) + sigma_v,j sum_j (Pq_ij / 256) v8_j
 *              and at the end O / l and LSE = m + ln l, as in the exact path.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* e4m3 from its definition.  Finite magnitudes: subnormals m 2^-9 (m = 1..7) */
/* and normals (1 + m/8) 2^(e-7) for e = 1..15, except e = 15, m = 7 (NaN).    */
/* ------------------------------------------------------------------------ */
static double e4m3_value(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(8.0 + m, e - 10); /* (1 + m/8) 2^(e-7) */
    return s ? -v : v;
}

/* round to nearest, ties to even, of a non-negative x to an integer */
static double rne(double x)
{
    double f = floor(x), r = x - f;
    if (r > 0.5)
        return f + 1.0;
    if (r < 0.5)
        return f;
    return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

static uint8_t e4m3_code(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t s = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0)
        return s | 0x7E; /* saturate to the largest finite value */
    int ex;
    frexp(a, &ex); /* a = f 2^ex, f in [0.5, 1): the leading power is 2^(ex-1) */
    int lead = ex - 1;
    if (a == 0.0 || lead < -6) {
        /* subnormal quantum 2^-9; a count of 8 is the smallest normal */
        int q = (int)rne(ldexp(a, 9));
        if (q >= 8)
            return s | (uint8_t)(1 << 3);
        return s | (uint8_t)q;
    }
    int q = (int)rne(ldexp(a, 3 - lead)); /* in [8, 16] */
    if (q == 16) {
        q = 8;
        ++lead;
    }
    if (lead > 8 || (lead == 8 && q > 14))
        return s | 0x7E;
    return s | (uint8_t)(((lead + 7) << 3) | (q - 8));
}

void orc_e4m3_encode(long long n, const double *x, uint8_t *code)
{
    for (long long i = 0; i < n; ++i)
        code[i] = e4m3_code(x[i]);
}

void orc_e4m3_decode(long long n, const uint8_t *code, double *x)
{
    for (long long i = 0; i < n; ++i)
        x[i] = e4m3_value(code[i]);
}

/* Smallest power of two sigma with amax / sigma <= 448 (1 when amax = 0). */
static double block_scale(double amax)
{
    if (!(amax > 0.0))
        return 1.0;
    int ex;
    frexp(amax / 448.0, &ex); /* amax / 448 = f 2^ex with f in [0.5, 1) */
    double sigma = ldexp(1.0, ex);
    /* f 2^ex <= 2^ex always; step down while the next smaller power still fits */
    while (amax / (sigma * 0.5) <= 448.0)
        sigma *= 0.5;
    while (amax / sigma > 448.0)
        sigma *= 2.0;
    return sigma;
}

double orc_fp8_block_scale(double amax) { return block_scale(amax); }

/* Sylvester Hadamard entry (-1)^popcount(a & b). */
static double hadamard(int a, int b)
{
    unsigned v = (unsigned)(a & b);
    int par = 0;
    while (v) {
        par ^= 1;
        v &= v - 1;
    }
    return par ? -1.0 : 1.0;
}

/* out[r] = x[r] D H * post (rows of d), the direct matrix product. */
void orc_hadamard_rotate(long long rows, int d, const double *x, const double *signs,
                         double post, double *out)
{
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < rows; ++r) {
        const double *xr = x + r * d;
        double *o = out + r * d;
        for (int c = 0; c < d; ++c) {
            double t = 0.0;
            for (int k = 0; k < d; ++k)
                t += xr[k] * signs[k] * hadamard(k, c);
            o[c] = t * post;
        }
    }
}

/* Quantise rows [0, N) of one head of x ([N][d], already fp32-valued) in
 * blocks of `block` rows: codes row-major [N][d] (or transposed [d][ld]
 * when trans != 0) and one scale per block. */
static void quant_head(int N, int d, const double *x, int block, int trans, long long ld,
                       uint8_t *codes, double *scales)
{
    int T = (N + block - 1) / block;
    for (int t = 0; t < T; ++t) {
        int r0 = t * block, r1 = r0 + block < N ? r0 + block : N;
        double amax = 0.0;
        for (int r = r0; r < r1; ++r)
            for (int c = 0; c < d; ++c)
                if (fabs(x[(size_t)r * d + c]) > amax)
                    amax = fabs(x[(size_t)r * d + c]);
        double sigma = block_scale(amax);
        scales[t] = sigma;
        for (int r = r0; r < r1; ++r)
            for (int c = 0; c < d; ++c) {
                uint8_t q = e4m3_code(x[(size_t)r * d + c] / sigma);
                if (trans)
                    codes[(size_t)c * ld + r] = q;
                else
                    codes[(size_t)r * d + c] = q;
            }
    }
}

/* Rotation (signs != NULL) and block quantisation of Q, K, V ([B*H][N][d],
 * fp64 holding the inputs' values).  Outputs: q8, k8 [B*H][N][d]; vt8
 * [B*H][d][ld] (V transposed, columns [N, ld) zero); sq, sk, sv
 * [B*H][ceil(N / block)]. */
void orc_fp8_quantize(int BH, int N, int d, const double *Q, const double *K, const double *V,
                      const double *signs, int block, long long ld, uint8_t *q8, uint8_t *k8,
                      uint8_t *vt8, double *sq, double *sk, double *sv)
{
    int T = (N + block - 1) / block;
    memset(vt8, 0, (size_t)BH * d * ld);
#pragma omp parallel
    {
        double *xq = (double *)malloc(sizeof(double) * (size_t)N * d);
        double *xk = (double *)malloc(sizeof(double) * (size_t)N * d);
        double *xv = (double *)malloc(sizeof(double) * (size_t)N * d);
#pragma omp for schedule(dynamic, 1)
        for (int bh = 0; bh < BH; ++bh) {
            size_t base = (size_t)bh * N * d;
            if (signs) {
                orc_hadamard_rotate(N, d, Q + base, signs, 1.0 / d, xq);
                orc_hadamard_rotate(N, d, K + base, signs, 1.0, xk);
            } else {
                memcpy(xq, Q + base, sizeof(double) * (size_t)N * d);
                memcpy(xk, K + base, sizeof(double) * (size_t)N * d);
            }
            memcpy(xv, V + base, sizeof(double) * (size_t)N * d);
            for (size_t i = 0; i < (size_t)N * d; ++i) { /* the kernel's precision */
                xq[i] = (double)(float)xq[i];
                xk[i] = (double)(float)xk[i];
                xv[i] = (double)(float)xv[i];
            }
            quant_head(N, d, xq, block, 0, 0, q8 + base, sq + (size_t)bh * T);
            quant_head(N, d, xk, block, 0, 0, k8 + base, sk + (size_t)bh * T);
            quant_head(N, d, xv, block, 1, ld, vt8 + (size_t)bh * d * ld, sv + (size_t)bh * T);
        }
        free(xq);
        free(xk);
        free(xv);
    }
}

/* The forward on FP8 operands (see the header).  Key blocks of 128 keys; the
 * scales cover blocks of `block` rows (128 for the kernel's codes).  mask:
 * [T][T] over mask_block tokens, shared by every head, or NULL. */
void orc_fp8_fwd(int BH, int N, int d, const uint8_t *q8, const uint8_t *k8, const uint8_t *vt8,
                 long long ld, const double *sq, const double *sk, const double *sv, int block,
                 double scale, int causal, const unsigned char *mask, int mask_block, double *O,
                 double *LSE)
{
    const int Bc = 128;
    const int T = (N + block - 1) / block;
    const int Tm = mask ? (N + mask_block - 1) / mask_block : 0;
    /* the operands' values, decoded once */
    double *kd = (double *)malloc(sizeof(double) * (size_t)BH * N * d);
    double *vd = (double *)malloc(sizeof(double) * (size_t)BH * N * d); /* [bh][j][c] */
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < (long long)BH * N; ++r) {
        int bh = (int)(r / N), j = (int)(r % N);
        for (int c = 0; c < d; ++c) {
            kd[(size_t)r * d + c] = e4m3_value(k8[(size_t)r * d + c]);
            vd[(size_t)r * d + c] = e4m3_value(vt8[((size_t)bh * d + c) * ld + j]);
        }
    }
#pragma omp parallel
    {
        double *qd = (double *)malloc(sizeof(double) * d);
        double *s = (double *)malloc(sizeof(double) * Bc);
        double *acc = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(dynamic, 16)
        for (long long job = 0; job < (long long)BH * N; ++job) {
            int bh = (int)(job / N), i = (int)(job % N);
            const double *kh = kd + (size_t)bh * N * d, *vh = vd + (size_t)bh * N * d;
            for (int c = 0; c < d; ++c)
                qd[c] = e4m3_value(q8[((size_t)bh * N + i) * d + c]);
            double m = -INFINITY, l = 0.0;
            for (int c = 0; c < d; ++c)
                acc[c] = 0.0;
            for (int j0 = 0; j0 < N; j0 += Bc) {
                int j1 = j0 + Bc < N ? j0 + Bc : N;
                double mt = -INFINITY;
                for (int j = j0; j < j1; ++j) {
                    int ok = !(causal && j > i);
                    if (ok && mask)
                        ok = mask[(size_t)(i / mask_block) * Tm + j / mask_block] != 0;
                    double v = -INFINITY;
                    if (ok) {
                        double t = 0.0;
                        for (int c = 0; c < d; ++c)
                            t += qd[c] * kh[(size_t)j * d + c];
                        v = scale * sq[(size_t)bh * T + i / block] * sk[(size_t)bh * T + j / block] * t;
                    }
                    s[j - j0] = v;
                    if (v > mt)
                        mt = v;
                }
                if (mt == -INFINITY)
                    continue; /* no allowed key in this block: nothing changes */
                double mn = m > mt ? m : mt;
                double alpha = (m == -INFINITY) ? 0.0 : exp(m - mn);
                l *= alpha;
                for (int c = 0; c < d; ++c)
                    acc[c] *= alpha;
                for (int j = j0; j < j1; ++j) {
                    if (s[j - j0] == -INFINITY)
                        continue;
                    double p = exp(s[j - j0] - mn);
                    l += p;
                    double pq = e4m3_value(e4m3_code(256.0 * (double)(float)p)) / 256.0;
                    double w = pq * sv[(size_t)bh * T + j / block];
                    for (int c = 0; c < d; ++c)
                        acc[c] += w * vh[(size_t)j * d + c];
                }
                m = mn;
            }
            double *o = O + ((size_t)bh * N + i) * d;
            for (int c = 0; c < d; ++c)
                o[c] = l > 0 ? acc[c] / l : 0.0;
            LSE[(size_t)bh * N + i] = l > 0 ? m + log(l) : -INFINITY;
        }
        free(qd);
        free(s);
        free(acc);
    }
    free(kd);
    free(vd);
}
