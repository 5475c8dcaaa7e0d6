/*
 * attn_oracle.c -- a plain, slow fp64 CPU statement of exact scaled-dot-product
 * attention, forward and backward.
 *
 * TEST INFRASTRUCTURE.  This is the oracle that the CUDA kernels are checked
 * against.  Only the test suite, the smoke entry point and the bench's CPU
 * baseline leg may build, load or call it.  It shares no code, header, helper,
 * table or constant with the CUDA library, and it never receives a value that
 * the CUDA library produced.
 *
 * What it computes (the pages' own statement of the problem):
 *   "Pourquoi l'attention est liée à la mémoire" (marketmaker.cc, "Un contexte
 *   d'une journée complète bat-il un contexte de dix minutes ?") defines the
 *   operation as softmax(Q K^T / sqrt(d_k)) V; "Problema e motivação" of the
 *   FlashAttention reading guide (xyznot.com, arXiv 2205.14135) writes it as
 *   S = QK^T, P = softmax(S), O = PV.  The caller passes the score scale
 *   (1/sqrt(d) in every workload); it multiplies QK^T before the softmax.
 *
 * Layout: every tensor is [B][H][N][d], contiguous, double precision.
 * LSE is [B][H][N].  The allowed key set of query row i of head (b,h) is
 *     A_i = { j < N : (!causal || j <= i) && (mask == 0 || M_bh[i/mb][j/mb] != 0) }
 * where M_bh is that head's block mask ("Extensão: Block-Sparse FlashAttention"
 * of the reading guide) stored row-major with ceil(N/mb) columns, and the causal
 * rule hides keys in the future of the query ("Le masquage causal est l'endroit
 * où le trading bénéficie d'une remise", marketmaker.cc).
 *
 * Readings taken where the pages are silent:
 *   - the saved per-row statistic is LSE_i = m_i + ln(l_i) in natural log and
 *     scaled-score units (the pages keep the pair (m, l); LSE carries the same
 *     information);
 *   - a row whose allowed set is empty has O_i = 0 and LSE_i = -inf, and it
 *     contributes nothing to any gradient;
 *   - the backward formulas are the derivative of the definition (the pages only
 *     say that S and P are recomputed from Q, K, V and the saved statistics);
 *   - dropout ("Fusão de Kernels" among the "Ideias centrais" of the reading
 *     guide fuses it into the same kernel; the integration code of "L'intégration
 *     est de huit lignes", marketmaker.cc, passes dropout_p to the attention
 *     call) acts on the attention weights after the softmax: each weight P_ij is
 *     kept with probability 1 - p and scaled by 1/(1 - p), or set to 0.  The
 *     statistics m, l and LSE stay those of the undropped softmax.  The pages
 *     name no random-number generator; the keep decisions come from the
 *     counter-based generator Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
 *     "Parallel random numbers: as easy as 1, 2, 3", SC 2011), so that a
 *     backward pass regenerates them instead of storing them: for head bh,
 *     query row i and key j, Philox4x32-10 with counter (floor(j / 8), i, bh,
 *     offset) and key (seed mod 2^32, floor(seed / 2^32)) gives four words;
 *     word floor((j mod 8) / 2), its low 16 bits for even j and its high 16
 *     bits for odd j, keeps the weight when it is at least t = floor(p * 2^16).
 *     A weight is then kept with probability 1 - t / 2^16 (p to within 2^-16)
 *     and scaled by 2^16 / (2^16 - t), the inverse of that probability.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Philox4x32-10, written from its definition in Salmon et al. (SC 2011): a    */
/* counter of four 32-bit words and a key of two go through ten rounds of      */
/*   (x0, x1, x2, x3) -> (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1,  */
/*                        lo(M0 x0))                                           */
/* with M0 = 0xD2511F53, M1 = 0xCD9E8D57 and hi/lo the halves of the 64-bit    */
/* product; the key is bumped by the Weyl constants (0x9E3779B9, 0xBB67AE85)   */
/* before every round but the first.                                           */
/* ------------------------------------------------------------------------ */
static void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)x0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ x1 ^ k0, n2 = hi0 ^ x3 ^ k1;
        x0 = n0;
        x1 = lo1;
        x2 = n2;
        x3 = lo0;
    }
    out[0] = x0;
    out[1] = x1;
    out[2] = x2;
    out[3] = x3;
}

void orc_philox4x32_10(const uint32_t *ctr, const uint32_t *key, uint32_t *out)
{
    philox4x32_10(ctr, key, out);
}

/* Dropout of one call: off when p == 0. */
typedef struct {
    int on;
    uint32_t t;     /* keep when the 16-bit half is >= t = floor(p * 2^16) */
    double z;       /* 2^16 / (2^16 - t) */
    uint32_t key[2];
    uint32_t offset;
} drop_cfg;

static drop_cfg make_drop(double p, unsigned long long seed, unsigned int offset)
{
    drop_cfg g;
    g.on = p > 0.0;
    double t = floor(p * 65536.0);
    g.t = t >= 65535.0 ? 65535u : (uint32_t)t;
    g.z = g.on ? 65536.0 / (65536.0 - (double)g.t) : 1.0;
    g.key[0] = (uint32_t)(seed & 0xFFFFFFFFull);
    g.key[1] = (uint32_t)(seed >> 32);
    g.offset = offset;
    return g;
}

typedef struct {
    int N, d;
    double scale;
    int causal;
    const unsigned char *mask; /* this head's block mask, or NULL */
    int mask_block;            /* tokens per mask entry */
    int mask_cols;             /* ceil(N / mask_block) */
    drop_cfg drop;
    int bh;                    /* b * H + h, part of the dropout counter */
} head_cfg;

/* The 16-bit draw of weight (i, j) of head bh. */
static uint32_t drop_draw(const drop_cfg *g, int bh, int i, int j)
{
    uint32_t ctr[4] = {(uint32_t)j >> 3, (uint32_t)i, (uint32_t)bh, g->offset};
    uint32_t w[4];
    philox4x32_10(ctr, g->key, w);
    uint32_t word = w[(j & 7) >> 1];
    return (j & 1) ? (word >> 16) : (word & 0xFFFFu);
}

/* The factor dropout applies to weight (i, j) of this head: 1 without dropout,
 * else 2^16 / (2^16 - t) or 0. */
static double drop_factor(const head_cfg *c, int i, int j)
{
    if (!c->drop.on)
        return 1.0;
    return drop_draw(&c->drop, c->bh, i, j) >= c->drop.t ? c->drop.z : 0.0;
}

/* Keep decisions of every (b, h, i, j) as bytes [B][H][N][N] (1 = kept). */
void orc_dropout_keep(int B, int H, int N, double p, unsigned long long seed,
                      unsigned int offset, unsigned char *keep)
{
    drop_cfg g = make_drop(p, seed, offset);
    const long long rows = (long long)B * H * N;
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < rows; ++r) {
        int bh = (int)(r / N), i = (int)(r % N);
        for (int j = 0; j < N; ++j)
            keep[(size_t)r * N + j] = (unsigned char)(!g.on || drop_draw(&g, bh, i, j) >= g.t);
    }
}

static head_cfg make_cfg(int N, int d, double scale, int causal,
                         const unsigned char *mask_h, int mask_block)
{
    head_cfg c;
    c.drop = make_drop(0.0, 0, 0);
    c.bh = 0;
    c.N = N;
    c.d = d;
    c.scale = scale;
    c.causal = causal;
    c.mask = mask_h;
    c.mask_block = mask_block > 0 ? mask_block : 1;
    c.mask_cols = (N + c.mask_block - 1) / c.mask_block;
    return c;
}

/* Is key j in the allowed set of query row i? */
static int allowed(const head_cfg *c, int i, int j)
{
    if (c->causal && j > i)
        return 0;
    if (c->mask) {
        size_t at = (size_t)(i / c->mask_block) * (size_t)c->mask_cols +
                    (size_t)(j / c->mask_block);
        if (!c->mask[at])
            return 0;
    }
    return 1;
}

static double dot(const double *a, const double *b, int d)
{
    double acc = 0.0;
    for (int k = 0; k < d; ++k)
        acc += a[k] * b[k];
    return acc;
}

/* ------------------------------------------------------------------------ */
/* Forward: the direct two-pass softmax of one query row.                     */
/*   s_j = scale * q_i . k_j          (j in A_i)                               */
/*   m   = max_j s_j                                                           */
/*   l   = sum_j exp(s_j - m)                                                  */
/*   O_i = sum_j exp(s_j - m) / l * z_ij * v_j   (z: the dropout factor)       */
/*   LSE = m + ln l                                                            */
/* s is caller scratch of N doubles.                                           */
/* ------------------------------------------------------------------------ */
static void fwd_row(const head_cfg *c, const double *Qh, const double *Kh,
                    const double *Vh, int i, double *s, double *o, double *lse)
{
    const int N = c->N, d = c->d;
    const double *q = Qh + (size_t)i * d;
    double m = -INFINITY;
    for (int j = 0; j < N; ++j) {
        if (!allowed(c, i, j))
            continue;
        s[j] = c->scale * dot(q, Kh + (size_t)j * d, d);
        if (s[j] > m)
            m = s[j];
    }
    for (int k = 0; k < d; ++k)
        o[k] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int j = 0; j < N; ++j)
        if (allowed(c, i, j))
            l += exp(s[j] - m);
    for (int j = 0; j < N; ++j) {
        if (!allowed(c, i, j))
            continue;
        double w = exp(s[j] - m) / l * drop_factor(c, i, j);
        const double *v = Vh + (size_t)j * d;
        for (int k = 0; k < d; ++k)
            o[k] += w * v[k];
    }
    *lse = m + log(l);
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static const unsigned char *head_mask(const unsigned char *mask, long long sb,
                                      long long sh, int b, int h)
{
    if (!mask)
        return NULL;
    return mask + (ptrdiff_t)b * sb + (ptrdiff_t)h * sh;
}

/* Whole-tensor forward.  mask may be NULL; sb/sh are the mask's batch and head
 * strides in elements (0 broadcasts one mask over that axis). */
void orc_fwd(int B, int H, int N, int d, const double *Q, const double *K,
             const double *V, double scale, int causal,
             const unsigned char *mask, int mask_block, long long sb,
             long long sh, double *O, double *LSE, double drop_p,
             unsigned long long seed, unsigned int offset)
{
    const drop_cfg g = make_drop(drop_p, seed, offset);
    const long long rows = (long long)B * H * N;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 16)
        for (long long r = 0; r < rows; ++r) {
            int bh = (int)(r / N), i = (int)(r % N);
            int b = bh / H, h = bh % H;
            head_cfg c = make_cfg(N, d, scale, causal,
                                  head_mask(mask, sb, sh, b, h), mask_block);
            c.drop = g;
            c.bh = bh;
            size_t base = (size_t)bh * N * d;
            fwd_row(&c, Q + base, K + base, V + base, i, s,
                    O + base + (size_t)i * d, LSE + (size_t)bh * N + i);
        }
        free(s);
    }
}

/* Forward of selected query rows of one head (the head's tensors are [N][d];
 * bh is the head's index b * H + h, used by dropout only).
 * O_rows is [nrows][d], LSE_rows is [nrows]. */
void orc_fwd_rows(int N, int d, const double *Qh, const double *Kh,
                  const double *Vh, double scale, int causal,
                  const unsigned char *mask_h, int mask_block, int nrows,
                  const int *rows, double *O_rows, double *LSE_rows, double drop_p,
                  unsigned long long seed, unsigned int offset, int bh)
{
    head_cfg c = make_cfg(N, d, scale, causal, mask_h, mask_block);
    c.drop = make_drop(drop_p, seed, offset);
    c.bh = bh;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 4)
        for (int t = 0; t < nrows; ++t)
            fwd_row(&c, Qh, Kh, Vh, rows[t], s, O_rows + (size_t)t * d,
                    LSE_rows + t);
        free(s);
    }
}

/* ------------------------------------------------------------------------ */
/* Blockwise online forward, in the order of "L'algorithme Flash Attention"    */
/* (marketmaker.cc) and "Método" / "Rastreamento Incremental do Softmax" of    */
/* the reading guide: queries in blocks of Br rows, keys and values in blocks  */
/* of Bc rows; per key block the local max m~, P~ = exp(S - m~) and l~ =       */
/* rowsum(P~); then the running statistics merge as                            */
/*     m_new = max(m, m~),  l_new = e^(m - m_new) l + e^(m~ - m_new) l~        */
/* and the output block is either renormalised at every step                   */
/*     O <- (l e^(m - m_new) O + e^(m~ - m_new) P~ V) / l_new                  */
/* (norm_at_end = 0, the FA1 form) or kept unnormalised and divided by the     */
/* running sum once at the end (norm_at_end = 1, the deferred form of          */
/* "FA2 : parallélisme" and of the PyTorch loop on the Ultralytics page).      */
/* A merge factor whose exponent is (-inf) - (-inf) is taken as 0: a block     */
/* with no allowed key contributes nothing.  Br and Bc may be any positive     */
/* sizes, including ones that do not divide N.  REAL is float or double.       */
/* ------------------------------------------------------------------------ */
#define DEFINE_BLOCKWISE(NAME, REAL, EXP, LOG)                                  \
void NAME(int B, int H, int N, int d, const REAL *Q, const REAL *K,            \
          const REAL *V, REAL scale, int causal, const unsigned char *mask,    \
          int mask_block, long long sb, long long sh, int Br, int Bc,          \
          int norm_at_end, REAL *O, REAL *LSE)                                 \
{                                                                              \
    const REAL NEG_INF = (REAL)(-INFINITY);                                    \
    const int Tr = (N + Br - 1) / Br;                                          \
    const long long jobs = (long long)B * H * Tr;                              \
    _Pragma("omp parallel")                                                    \
    {                                                                          \
        REAL *S = (REAL *)malloc(sizeof(REAL) * (size_t)Br * Bc);              \
        REAL *acc = (REAL *)malloc(sizeof(REAL) * (size_t)d);                  \
        REAL *m = (REAL *)malloc(sizeof(REAL) * (size_t)Br);                   \
        REAL *l = (REAL *)malloc(sizeof(REAL) * (size_t)Br);                   \
        _Pragma("omp for schedule(dynamic, 1)")                                \
        for (long long job = 0; job < jobs; ++job) {                           \
            int bh = (int)(job / Tr), ib = (int)(job % Tr);                    \
            int b = bh / H, h = bh % H;                                        \
            head_cfg c = make_cfg(N, d, (double)scale, causal,                 \
                                  head_mask(mask, sb, sh, b, h), mask_block);  \
            size_t base = (size_t)bh * N * d;                                  \
            const REAL *Qh = Q + base, *Kh = K + base, *Vh = V + base;         \
            REAL *Oh = O + base;                                               \
            int i0 = ib * Br, i1 = i0 + Br < N ? i0 + Br : N;                  \
            for (int i = i0; i < i1; ++i) {                                    \
                m[i - i0] = NEG_INF;                                           \
                l[i - i0] = 0;                                                 \
                for (int k = 0; k < d; ++k)                                    \
                    Oh[(size_t)i * d + k] = 0;                                 \
            }                                                                  \
            for (int j0 = 0; j0 < N; j0 += Bc) {                               \
                int j1 = j0 + Bc < N ? j0 + Bc : N;                            \
                /* S_ij = scale * Q_i K_j^T, hidden entries -inf */            \
                for (int i = i0; i < i1; ++i)                                  \
                    for (int j = j0; j < j1; ++j) {                            \
                        REAL sv = NEG_INF;                                     \
                        if (allowed(&c, i, j)) {                               \
                            REAL t = 0;                                        \
                            for (int k = 0; k < d; ++k)                        \
                                t += Qh[(size_t)i * d + k] *                   \
                                     Kh[(size_t)j * d + k];                    \
                            sv = scale * t;                                    \
                        }                                                      \
                        S[(size_t)(i - i0) * Bc + (j - j0)] = sv;              \
                    }                                                          \
                for (int i = i0; i < i1; ++i) {                                \
                    REAL *Srow = S + (size_t)(i - i0) * Bc;                    \
                    REAL mt = NEG_INF, lt = 0;                                 \
                    for (int j = j0; j < j1; ++j)                              \
                        if (Srow[j - j0] > mt)                                 \
                            mt = Srow[j - j0];                                 \
                    /* P~ = exp(S - m~), l~ = rowsum(P~), acc = P~ V_j */      \
                    for (int k = 0; k < d; ++k)                                \
                        acc[k] = 0;                                            \
                    if (mt != NEG_INF) {                                       \
                        for (int j = j0; j < j1; ++j) {                        \
                            REAL p = EXP(Srow[j - j0] - mt);                   \
                            lt += p;                                           \
                            for (int k = 0; k < d; ++k)                        \
                                acc[k] += p * Vh[(size_t)j * d + k];           \
                        }                                                      \
                    }                                                          \
                    REAL mo = m[i - i0], lo = l[i - i0];                       \
                    REAL mn = mo > mt ? mo : mt;                               \
                    REAL a = mo == NEG_INF ? (REAL)0 : EXP(mo - mn);           \
                    REAL bt = mt == NEG_INF ? (REAL)0 : EXP(mt - mn);          \
                    REAL ln = a * lo + bt * lt;                                \
                    REAL *o = Oh + (size_t)i * d;                              \
                    if (norm_at_end) {                                         \
                        for (int k = 0; k < d; ++k)                            \
                            o[k] = a * o[k] + bt * acc[k];                     \
                    } else if (ln > 0) {                                       \
                        for (int k = 0; k < d; ++k)                            \
                            o[k] = (lo * a * o[k]) / ln + (bt * acc[k]) / ln;  \
                    }                                                          \
                    m[i - i0] = mn;                                            \
                    l[i - i0] = ln;                                            \
                }                                                              \
            }                                                                  \
            for (int i = i0; i < i1; ++i) {                                    \
                REAL li = l[i - i0];                                           \
                REAL *o = Oh + (size_t)i * d;                                  \
                if (norm_at_end && li > 0)                                     \
                    for (int k = 0; k < d; ++k)                                \
                        o[k] = o[k] / li;                                      \
                LSE[(size_t)bh * N + i] =                                      \
                    li > 0 ? m[i - i0] + LOG(li) : NEG_INF;                    \
            }                                                                  \
        }                                                                      \
        free(S);                                                               \
        free(acc);                                                             \
        free(m);                                                               \
        free(l);                                                               \
    }                                                                          \
}

DEFINE_BLOCKWISE(orc_fwd_blockwise_f64, double, exp, log)
DEFINE_BLOCKWISE(orc_fwd_blockwise_f32, float, expf, logf)

/* ------------------------------------------------------------------------ */
/* Backward from the definition (the pages give no formulas; these are the     */
/* derivative of O = softmax(scale * Q K^T) V with respect to Q, K and V for   */
/* the loss whose gradient at O is dO):                                        */
/*   P_ij  = exp(s_ij - LSE_i)                (0 when j is not in A_i)         */
/*   dV_j  = sum_i P_ij z_ij dO_i             (z: the dropout factor, 1        */
/*   dP_ij = dO_i . v_j                        without dropout)                */
/*   D_i   = sum_j P_ij z_ij dP_ij            (= dO_i . O_i)                   */
/*   dS_ij = P_ij (z_ij dP_ij - D_i)                                           */
/*   dQ_i  = scale * sum_j dS_ij k_j                                           */
/*   dK_j  = scale * sum_i dS_ij q_i                                           */
/* Pass 1 walks query rows (LSE_i, D_i and dQ_i); pass 2 walks key rows (dK_j  */
/* and dV_j), recomputing P and dP from the row statistics of pass 1.          */
/* ------------------------------------------------------------------------ */

/* Pass 1 for query row i: LSE_i, D_i and, when dq != NULL, dQ_i. */
static void bwd_row_stats(const head_cfg *c, const double *Qh, const double *Kh,
                          const double *Vh, const double *dOh, int i, double *s,
                          double *lse_out, double *D_out, double *dq)
{
    const int N = c->N, d = c->d;
    const double *q = Qh + (size_t)i * d, *g = dOh + (size_t)i * d;
    double m = -INFINITY;
    for (int j = 0; j < N; ++j) {
        if (!allowed(c, i, j))
            continue;
        s[j] = c->scale * dot(q, Kh + (size_t)j * d, d);
        if (s[j] > m)
            m = s[j];
    }
    if (dq)
        for (int k = 0; k < d; ++k)
            dq[k] = 0.0;
    if (m == -INFINITY) {
        *lse_out = -INFINITY;
        *D_out = 0.0;
        return;
    }
    double l = 0.0;
    for (int j = 0; j < N; ++j)
        if (allowed(c, i, j))
            l += exp(s[j] - m);
    double lse = m + log(l);
    double D = 0.0;
    for (int j = 0; j < N; ++j) {
        if (!allowed(c, i, j))
            continue;
        double P = exp(s[j] - lse);
        double dP = dot(g, Vh + (size_t)j * d, d);
        D += P * drop_factor(c, i, j) * dP;
    }
    *lse_out = lse;
    *D_out = D;
    if (!dq)
        return;
    for (int j = 0; j < N; ++j) {
        if (!allowed(c, i, j))
            continue;
        double P = exp(s[j] - lse);
        double dP = dot(g, Vh + (size_t)j * d, d);
        double dS = P * (drop_factor(c, i, j) * dP - D);
        const double *kr = Kh + (size_t)j * d;
        for (int k = 0; k < d; ++k)
            dq[k] += c->scale * dS * kr[k];
    }
}

/* Pass 2 for key row j: dK_j and dV_j from the row statistics LSE, D. */
static void bwd_key_row(const head_cfg *c, const double *Qh, const double *Kh,
                        const double *Vh, const double *dOh, const double *LSE,
                        const double *Dv, int j, double *dk, double *dv)
{
    const int N = c->N, d = c->d;
    const double *kr = Kh + (size_t)j * d, *vr = Vh + (size_t)j * d;
    for (int k = 0; k < d; ++k) {
        dk[k] = 0.0;
        dv[k] = 0.0;
    }
    for (int i = 0; i < N; ++i) {
        if (!allowed(c, i, j) || LSE[i] == -INFINITY)
            continue;
        const double *q = Qh + (size_t)i * d, *g = dOh + (size_t)i * d;
        double sij = c->scale * dot(q, kr, d);
        double P = exp(sij - LSE[i]);
        double z = drop_factor(c, i, j);
        double dP = dot(g, vr, d);
        double dS = P * (z * dP - Dv[i]);
        for (int k = 0; k < d; ++k) {
            dv[k] += P * z * g[k];
            dk[k] += c->scale * dS * q[k];
        }
    }
}

void orc_bwd(int B, int H, int N, int d, const double *Q, const double *K,
             const double *V, const double *dO, double scale, int causal,
             const unsigned char *mask, int mask_block, long long sb,
             long long sh, double *dQ, double *dK, double *dV, double drop_p,
             unsigned long long seed, unsigned int offset)
{
    const drop_cfg g = make_drop(drop_p, seed, offset);
    const long long rows = (long long)B * H * N;
    double *LSE = (double *)malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1));
    double *Dv = (double *)malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1));
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 16)
        for (long long r = 0; r < rows; ++r) {
            int bh = (int)(r / N), i = (int)(r % N);
            head_cfg c = make_cfg(N, d, scale, causal,
                                  head_mask(mask, sb, sh, bh / H, bh % H),
                                  mask_block);
            c.drop = g;
            c.bh = bh;
            size_t base = (size_t)bh * N * d;
            bwd_row_stats(&c, Q + base, K + base, V + base, dO + base, i, s,
                          LSE + r, Dv + r, dQ + base + (size_t)i * d);
        }
        free(s);
    }
#pragma omp parallel for schedule(dynamic, 16)
    for (long long r = 0; r < rows; ++r) {
        int bh = (int)(r / N), j = (int)(r % N);
        head_cfg c = make_cfg(N, d, scale, causal,
                              head_mask(mask, sb, sh, bh / H, bh % H),
                              mask_block);
        c.drop = g;
        c.bh = bh;
        size_t base = (size_t)bh * N * d;
        bwd_key_row(&c, Q + base, K + base, V + base, dO + base,
                    LSE + (size_t)bh * N, Dv + (size_t)bh * N, j,
                    dK + base + (size_t)j * d, dV + base + (size_t)j * d);
    }
    free(LSE);
    free(Dv);
}

/* Backward outputs of selected rows of one head: dQ for the query rows qrows
 * and dK, dV for the key rows krows.  The row statistics of every query row of
 * the head are computed first (they are needed by any key row). */
void orc_bwd_rows(int N, int d, const double *Qh, const double *Kh,
                  const double *Vh, const double *dOh, double scale, int causal,
                  const unsigned char *mask_h, int mask_block, int nq,
                  const int *qrows, double *dQ_rows, int nk, const int *krows,
                  double *dK_rows, double *dV_rows, double drop_p,
                  unsigned long long seed, unsigned int offset, int bh)
{
    head_cfg c = make_cfg(N, d, scale, causal, mask_h, mask_block);
    c.drop = make_drop(drop_p, seed, offset);
    c.bh = bh;
    double *LSE = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double *Dv = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    int need_all = nk > 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (need_all) {
#pragma omp for schedule(dynamic, 16)
            for (int i = 0; i < N; ++i)
                bwd_row_stats(&c, Qh, Kh, Vh, dOh, i, s, LSE + i, Dv + i, NULL);
        }
#pragma omp for schedule(dynamic, 1)
        for (int t = 0; t < nq; ++t) {
            double lse, D;
            bwd_row_stats(&c, Qh, Kh, Vh, dOh, qrows[t], s, &lse, &D,
                          dQ_rows + (size_t)t * d);
        }
#pragma omp for schedule(dynamic, 1)
        for (int t = 0; t < nk; ++t)
            bwd_key_row(&c, Qh, Kh, Vh, dOh, LSE, Dv, krows[t],
                        dK_rows + (size_t)t * d, dV_rows + (size_t)t * d);
        free(s);
    }
    free(LSE);
    free(Dv);
}
