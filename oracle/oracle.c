/*
 * oracle.c -- plain, slow, float64 CPU definition of the CSA + HCA hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
 * its Python binding) may link, load or call this file.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark use it.
 *
 * It shares no code, header, table or helper with the CUDA path.  Every value
 * is taken in double precision; the caller converts stored bf16/f32 inputs to
 * double exactly before calling in.
 *
 * Sources (web pages on DeepSeek-V4; cited by title and section):
 *  [P2]  "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section
 *        "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)": CSA merges m consecutive KV
 *        entries into one, each query attends only its top-k compressed
 *        entries, plus a sliding-window branch; HCA merges m' >> m entries and
 *        attends densely with no selection.
 *  [P2q] same page, section "오픈소스 MoE 인프라: MegaMoE와 TileLang": the indexer
 *        QK path is stored in FP4 (MXFP4), dequantised to FP8 without loss.
 *  [P3]  "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를 저렴하게", sections
 *        "Compressed Sparse Attention (CSA)" (compress per block, indexer
 *        finds relevant blocks, attend only the top candidates, keep recent
 *        tokens in a sliding window), "Heavily Compressed Attention (HCA)"
 *        (attend all compressed entries) and "KV Cache 관리" (compressed
 *        cache, sliding-window cache, tail of not-yet-compressed tokens).
 *  [P1]  "EP 95. DeepSeek-V4 논문 읽기 — 노정석", section IDEAS: KV cache
 *        compressed to 1/4, a lightning indexer picks the top-k; MQA.
 *
 * Where the pages leave a step open, the reading taken is the one fixed in
 * the project's specification: softmax pooling with one scalar logit per raw
 * token, indexer score sum_h w_h * ReLU(q_h . k), lowest index wins ties,
 * OCP MX v1.0 block scaling for MXFP4.
 *
 * Threading: the batched entry points run independent rows in an OpenMP
 * parallel-for; each row's arithmetic is the plain sequential definition.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- rounding */

/* Round a double to the nearest bfloat16 value (ties to even), returned as a
 * double.  bfloat16 has 8 significant bits and the float32 exponent range
 * (normal >= 2^-126, subnormal quantum 2^-133, largest finite 0x1.FEp127). */
double orc_round_bf16(double x)
{
    if (x != x || x == 0.0 || isinf(x)) return x;
    double ax = fabs(x);
    int e;
    frexp(ax, &e);                 /* ax = f * 2^e, f in [0.5, 1) */
    int q = e - 8;                 /* quantum exponent for 8 significant bits */
    if (q < -133) q = -133;        /* subnormal range */
    double r = ldexp(nearbyint(ldexp(ax, -q)), q);   /* default mode: ties-to-even */
    if (r > 0x1.FEp127) r = INFINITY;
    return x < 0 ? -r : r;
}

/* Round a double to the nearest float32 (ties to even): the C conversion. */
double orc_round_f32(double x) { return (double)(float)x; }

/* ------------------------------------------------------- a1: compression */

/* Compress nblk blocks of m rows each.  Row i of block b is X[(b*m+i)*d ..],
 * with pooling logit z[b*m+i].  Block output:
 *     Xc[b] = sum_i softmax(z_block)_i * X[b*m+i]
 * (softmax pooling within the block; the pages say only "m entries into one",
 * [P2] and [P3] step 1).  round_mode: 0 = keep double, 1 = round each output
 * to float32, 2 = round each output to bfloat16 (the cache storage type). */
void orc_compress(int64_t nblk, int m, int d, const double *X, const double *z,
                  int round_mode, double *Xc)
{
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblk; ++b) {
        const double *zb = z + b * m;
        double mu = zb[0];
        for (int i = 1; i < m; ++i) if (zb[i] > mu) mu = zb[i];
        double den = 0.0;
        for (int i = 0; i < m; ++i) den += exp(zb[i] - mu);
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int i = 0; i < m; ++i)
                acc += (exp(zb[i] - mu) / den) * X[(b * m + i) * (int64_t)d + c];
            if (round_mode == 1) acc = orc_round_f32(acc);
            else if (round_mode == 2) acc = orc_round_bf16(acc);
            Xc[b * (int64_t)d + c] = acc;
        }
    }
}

/* ---------------------------------------------------- a2: indexer scores */

/* Per-channel softmax pooling: the compressor variant with one logit per raw
 * token AND channel ([P3] "Compressed Sparse Attention (CSA)" step 1, m
 * consecutive entries merged into one; the pages do not say whether the
 * merge weights are shared by all channels -- this is the variant where they
 * are not).  For block b and channel c, with the block's m logits of that
 * channel,
 *   Xc[b, c] = sum_i softmax_i(z[b*m+i, c]) * X[b*m+i, c].
 * Layouts: X, z [nblk*m, d] (row = raw position, column = channel);
 * Xc [nblk, d].  round_mode as orc_compress. */
void orc_compress_channels(int64_t nblk, int m, int d, const double *X, const double *z,
                           int round_mode, double *Xc)
{
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblk; ++b) {
        for (int c = 0; c < d; ++c) {
            double mu = z[(b * m) * (int64_t)d + c];
            for (int i = 1; i < m; ++i) {
                const double zi = z[(b * m + i) * (int64_t)d + c];
                if (zi > mu) mu = zi;
            }
            double den = 0.0;
            for (int i = 0; i < m; ++i) den += exp(z[(b * m + i) * (int64_t)d + c] - mu);
            double acc = 0.0;
            for (int i = 0; i < m; ++i)
                acc += (exp(z[(b * m + i) * (int64_t)d + c] - mu) / den) *
                       X[(b * m + i) * (int64_t)d + c];
            if (round_mode == 1) acc = orc_round_f32(acc);
            else if (round_mode == 2) acc = orc_round_bf16(acc);
            Xc[b * (int64_t)d + c] = acc;
        }
    }
}

/* Lightning-indexer score of every visible compressed entry for each query row
 * ([P3] step 2, [P1] IDEAS):
 *     s[r, j] = sum_h w[r,h] * max(0, q_I[r,h,:] . Ik_c[seq[r], j, :])
 * for 0 <= j < nvis[r]; entries j >= nvis[r] are set to -INFINITY.
 * Ik has layout [nseq, ncap, dI]; s has layout [rows, ncap]. */
void orc_index_scores(int64_t rows, int HI, int dI, const double *qI,
                      const double *w, const double *Ik, int64_t ncap,
                      const int64_t *seq, const int64_t *nvis, double *s)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        const double *kbase = Ik + seq[r] * ncap * dI;
        for (int64_t j = 0; j < ncap; ++j) {
            if (j >= nvis[r]) { s[r * ncap + j] = -INFINITY; continue; }
            double acc = 0.0;
            for (int h = 0; h < HI; ++h) {
                double dot = 0.0;
                for (int c = 0; c < dI; ++c)
                    dot += qI[(r * HI + h) * (int64_t)dI + c] * kbase[j * dI + c];
                acc += w[r * HI + h] * (dot > 0.0 ? dot : 0.0);
            }
            s[r * ncap + j] = acc;
        }
    }
}

/* ------------------------------------------------------------ a3: top-k */

typedef struct { double s; int64_t j; } orc_cand;

/* Order: higher score first; on equal scores the lower index first. */
static int orc_cand_cmp(const void *a, const void *b)
{
    const orc_cand *x = (const orc_cand *)a, *y = (const orc_cand *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int orc_int_cmp(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* Per-row top-k ([P2]: each query keeps its k highest compressed entries;
 * [P3] step 3).  Candidates are j in [0, n[r]) with score s[r*ld + j].
 * Selects min(k, n[r]) entries ordered by (score desc, index asc), then writes
 * them in ascending index order to idx[r*k ..], padding with -1.
 * Scores compare as numbers, so -0.0 equals +0.0.  Returns the number of rows
 * holding a NaN candidate score (such rows are written as all -1). */
int64_t orc_topk(int64_t rows, int64_t ld, const double *s, const int64_t *n,
                 int k, int32_t *idx)
{
    int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+:bad)
    for (int64_t r = 0; r < rows; ++r) {
        int32_t *out = idx + r * (int64_t)k;
        for (int i = 0; i < k; ++i) out[i] = -1;
        int64_t nr = n[r];
        int nan_row = 0;
        for (int64_t j = 0; j < nr; ++j)
            if (s[r * ld + j] != s[r * ld + j]) nan_row = 1;
        if (nan_row) { bad += 1; continue; }
        if (nr <= 0 || k <= 0) continue;
        orc_cand *c = (orc_cand *)malloc((size_t)nr * sizeof(orc_cand));
        for (int64_t j = 0; j < nr; ++j) {
            c[j].s = s[r * ld + j];
            c[j].j = j;
        }
        qsort(c, (size_t)nr, sizeof(orc_cand), orc_cand_cmp);
        int64_t take = nr < k ? nr : k;
        for (int64_t i = 0; i < take; ++i) out[i] = (int32_t)c[i].j;
        qsort(out, (size_t)take, sizeof(int32_t), orc_int_cmp);
        free(c);
    }
    return bad;
}

/* ------------------------------------------------------- a4/a5: attention */

/* Multi-query attention of each row over an explicit key multiset.
 * Row r has H query heads q[r,h,:] and the keys K[o], values V[o] for
 * off[r] <= o < off[r+1] (shared by all heads: one KV head, [P1] IDEAS).
 *     l_o   = scale * q[r,h,:] . K[o,:]
 *     LSE   = mu + log sum_o exp(l_o - mu),   mu = max_o l_o   (natural log)
 *     O     = sum_o exp(l_o - LSE) * V[o,:]
 * An empty key set gives O = 0 and LSE = -INFINITY.  For CSA the multiset is
 * the selected compressed rows plus the window rows ([P2], [P3] steps 3-4);
 * for HCA it is every visible compressed row plus the window ([P3] HCA). */
void orc_attend(int64_t rows, int H, int d, double scale, const double *q,
                const int64_t *off, const double *K, const double *V,
                double *O, double *lse)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t o0 = off[r], o1 = off[r + 1];
        double *lg = (double *)malloc((size_t)((o1 - o0) > 0 ? (o1 - o0) : 1) * sizeof(double));
        for (int h = 0; h < H; ++h) {
            const double *qh = q + (r * H + h) * (int64_t)d;
            double *oh = O + (r * H + h) * (int64_t)d;
            for (int c = 0; c < d; ++c) oh[c] = 0.0;
            if (o1 <= o0) { lse[r * H + h] = -INFINITY; continue; }
            double mu = -INFINITY;
            for (int64_t o = o0; o < o1; ++o) {
                double dot = 0.0;
                for (int c = 0; c < d; ++c) dot += qh[c] * K[o * d + c];
                lg[o - o0] = scale * dot;
                if (lg[o - o0] > mu) mu = lg[o - o0];
            }
            double sum = 0.0;
            for (int64_t o = o0; o < o1; ++o) sum += exp(lg[o - o0] - mu);
            double L = mu + log(sum);
            for (int64_t o = o0; o < o1; ++o) {
                double p = exp(lg[o - o0] - L);
                for (int c = 0; c < d; ++c) oh[c] += p * V[o * d + c];
            }
            lse[r * H + h] = L;
        }
        free(lg);
    }
}

/* ------------------------------------------------------------- a6: merge */

/* Exact merge of attention partials over disjoint key sets (the branches and
 * splits of the multi-branch design in [P2] and [P1] IDEAS):
 *     LSE = log sum_i exp(LSE_i),   O = sum_i exp(LSE_i - LSE) * O_i
 * Parts with LSE_i = -INFINITY contribute nothing; if all are -INFINITY the
 * result is O = 0, LSE = -INFINITY.  Layouts: O_parts [nparts, rows, d],
 * lse_parts [nparts, rows]. */
void orc_merge(int nparts, int64_t rows, int d, const double *O_parts,
               const double *lse_parts, double *O, double *lse)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double mu = -INFINITY;
        for (int i = 0; i < nparts; ++i)
            if (lse_parts[i * rows + r] > mu) mu = lse_parts[i * rows + r];
        for (int c = 0; c < d; ++c) O[r * d + c] = 0.0;
        if (mu == -INFINITY) { lse[r] = -INFINITY; continue; }
        double sum = 0.0;
        for (int i = 0; i < nparts; ++i) sum += exp(lse_parts[i * rows + r] - mu);
        double L = mu + log(sum);
        for (int i = 0; i < nparts; ++i) {
            double a = exp(lse_parts[i * rows + r] - L);
            for (int c = 0; c < d; ++c) O[r * d + c] += a * O_parts[(i * rows + r) * d + c];
        }
        lse[r] = L;
    }
}

/* ------------------------------------------------------------ a7: MXFP4 */

/* e2m1 magnitudes by 3-bit code (OCP Microscaling Formats v1.0, FP4 E2M1):
 * exponent bits 2..1 (bias 1), mantissa bit 0; code 1 is the subnormal 0.5. */
static double orc_e2m1_value(int code3)
{
    int e = (code3 >> 1) & 3, mbit = code3 & 1;
    if (e == 0) return 0.5 * mbit;
    return ldexp(1.0 + 0.5 * mbit, e - 1);
}

/* Nearest e2m1 code (3-bit magnitude) to |v|, ties to the even code,
 * saturating at 6.  Searches the eight grid values. */
static int orc_e2m1_round(double av)
{
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c < 8; ++c) {
        double dd = fabs(av - orc_e2m1_value(c));
        if (dd < bd || (dd == bd && (c & 1) == 0)) { bd = dd; best = c; }
    }
    return best;
}

/* MXFP4 quantisation of nblk blocks of 32 values ([P2q]; block rule from OCP
 * MX v1.0): shared exponent e = floor(log2(max |x|)) - 2 (2 = largest e2m1
 * exponent), clamped to [-127, 127]; an all-zero block gets e = -127.  Each
 * element is x / 2^e rounded to the nearest e2m1 value (ties to even code,
 * saturating at +-6).  A negative element whose magnitude rounds to zero is
 * stored as +0.  Output: codes[b*16 + i] holds element 2i in its low nibble and
 * element 2i+1 in its high nibble; scales[b] = e + 127 (e8m0). */
void orc_mxfp4_quantize(int64_t nblk, const double *x, uint8_t *codes, uint8_t *scales)
{
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblk; ++b) {
        const double *xb = x + b * 32;
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) if (fabs(xb[i]) > amax) amax = fabs(xb[i]);
        int e;
        if (amax == 0.0) {
            e = -127;
        } else {
            int fe;
            frexp(amax, &fe);          /* amax in [2^(fe-1), 2^fe) */
            e = (fe - 1) - 2;
            if (e < -127) e = -127;
            if (e > 127) e = 127;
        }
        scales[b] = (uint8_t)(e + 127);
        for (int i = 0; i < 32; i += 2) {
            int nib[2];
            for (int t = 0; t < 2; ++t) {
                double v = ldexp(xb[i + t], -e);
                int mag = orc_e2m1_round(fabs(v));
                nib[t] = (v < 0 && mag != 0) ? (8 | mag) : mag;
            }
            codes[b * 16 + i / 2] = (uint8_t)(nib[0] | (nib[1] << 4));
        }
    }
}

/* Exact dequantisation: value = e2m1(code) * 2^(scale - 127). */
void orc_mxfp4_dequantize(int64_t nblk, const uint8_t *codes, const uint8_t *scales, double *x)
{
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblk; ++b) {
        int e = (int)scales[b] - 127;
        for (int i = 0; i < 32; ++i) {
            int nib = (codes[b * 16 + i / 2] >> ((i & 1) * 4)) & 15;
            double v = ldexp(orc_e2m1_value(nib & 7), e);
            x[b * 32 + i] = (nib & 8) ? -v : v;
        }
    }
}

/* ------------------------------------------------------------- backward */

/* Gradient of orc_attend for one loss L with dL/dO = dO, the key multiset of
 * every row held fixed (the top-k selection is not differentiable -- "EP 95.
 * DeepSeek-V4 논문 읽기 — 노정석", IDEAS -- so it is a constant mask here).
 * With l_o = scale * q_h . K_o, P_o = exp(l_o - LSE_h) (LSE as in orc_attend):
 *     dV_o += sum_h P_o * dO_h
 *     dP_o  = dO_h . V_o,      D_h = sum_o P_o * dP_o
 *     dl_o  = P_o * (dP_o - D_h)
 *     dq_h  = scale * sum_o dl_o * K_o
 *     dK_o += scale * sum_h dl_o * q_h
 * dK, dV [off[rows], d] are per entry of the multisets (the caller adds the
 * entries that name the same cache or ring row); dq [rows, H, d].  A row with
 * no keys gets dq = 0. */
void orc_attend_backward(int64_t rows, int H, int d, double scale, const double *q,
                         const int64_t *off, const double *K, const double *V,
                         const double *dO, double *dq, double *dK, double *dV)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t o0 = off[r], o1 = off[r + 1], n = o1 - o0;
        for (int64_t o = o0; o < o1; ++o)
            for (int c = 0; c < d; ++c) { dK[o * d + c] = 0.0; dV[o * d + c] = 0.0; }
        double *p = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
        double *dp = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
        for (int h = 0; h < H; ++h) {
            const double *qh = q + (r * H + h) * (int64_t)d;
            const double *gh = dO + (r * H + h) * (int64_t)d;
            double *dqh = dq + (r * H + h) * (int64_t)d;
            for (int c = 0; c < d; ++c) dqh[c] = 0.0;
            if (n <= 0) continue;
            double mu = -INFINITY;
            for (int64_t o = o0; o < o1; ++o) {
                double dot = 0.0;
                for (int c = 0; c < d; ++c) dot += qh[c] * K[o * d + c];
                p[o - o0] = scale * dot;
                if (p[o - o0] > mu) mu = p[o - o0];
            }
            double sum = 0.0;
            for (int64_t i = 0; i < n; ++i) sum += exp(p[i] - mu);
            double L = mu + log(sum);
            double D = 0.0;
            for (int64_t o = o0; o < o1; ++o) {
                double pr = exp(p[o - o0] - L);
                p[o - o0] = pr;
                double g = 0.0;
                for (int c = 0; c < d; ++c) g += gh[c] * V[o * d + c];
                dp[o - o0] = g;
                D += pr * g;
            }
            for (int64_t o = o0; o < o1; ++o) {
                double pr = p[o - o0];
                double dl = pr * (dp[o - o0] - D);
                for (int c = 0; c < d; ++c) {
                    dV[o * d + c] += pr * gh[c];
                    dqh[c] += scale * dl * K[o * d + c];
                    dK[o * d + c] += scale * dl * qh[c];
                }
            }
        }
        free(p);
        free(dp);
    }
}

/* Gradient of orc_compress for dL/dXc = dXc, the storage rounding taken as
 * the identity.  With a = softmax(z_block) and the unrounded pooled row
 * Xc = sum_i a_i X_i:
 *     dX_i  = a_i * dXc                        (written)
 *     dz_i += a_i * (X_i - Xc) . dXc           (added: arrays pooled with the
 *                                               same logits add their parts)
 * Layouts as orc_compress: X, dX [nblk*m, d], z, dz [nblk*m], dXc [nblk, d]. */
void orc_compress_backward(int64_t nblk, int m, int d, const double *X, const double *z,
                           const double *dXc, double *dX, double *dz)
{
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < nblk; ++b) {
        const double *zb = z + b * m;
        double mu = zb[0];
        for (int i = 1; i < m; ++i) if (zb[i] > mu) mu = zb[i];
        double den = 0.0;
        for (int i = 0; i < m; ++i) den += exp(zb[i] - mu);
        const double *g = dXc + b * (int64_t)d;
        for (int i = 0; i < m; ++i) {
            double a = exp(zb[i] - mu) / den;
            const double *xi = X + (b * m + i) * (int64_t)d;
            double *dxi = dX + (b * m + i) * (int64_t)d;
            double t = 0.0;
            for (int c = 0; c < d; ++c) {
                double xc = 0.0;
                for (int l = 0; l < m; ++l)
                    xc += (exp(zb[l] - mu) / den) * X[(b * m + l) * (int64_t)d + c];
                dxi[c] = a * g[c];
                t += (xi[c] - xc) * g[c];
            }
            dz[b * m + i] += a * t;
        }
    }
}
