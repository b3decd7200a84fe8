/*
 * tl_oracle.c -- plain, slow, obviously correct CPU oracle for the ternary
 * projection linears.  TEST INFRASTRUCTURE ONLY: the test suite, the smoke
 * check and the benchmark's CPU-baseline leg call it; the library under
 * bit_matvec_ternary_b300/ never links, loads or calls it, and it shares no
 * source with that library.
 *
 * What it computes (Neutrino-1 pages):
 *   - every projection weight is one of {-1, 0, +1} ("Neutrino-1: quantization
 *     is a training decision", "What's actually ternary"; wpnews "Not
 *     Quantization - Trained Ternary");
 *   - a linear's output is the signed sum of its inputs times a scale
 *     ("state times scale", same blog, "What's actually ternary"), with one
 *     scale per output row and per-row row sums ("Neutrino-1 8B" model page,
 *     "Architecture": per-row metadata holds "row dimensions, scales, and row
 *     sums");
 *   - weights stay packed and are decoded inside the matrix kernel (model
 *     page, "Overview"); the packing is the library's own TL2P v2 layout,
 *     because the pages' format is unpublished (wiki "Neutrino-1", "What is
 *     actually new").  The layout is restated in tl2p_position() below.
 *
 * Definition: y[n,m] = scale[m] * sum_k w[m,k] * x[n,k].
 *   mode A: x is bf16, the sum is taken in double (exact for these inputs up
 *           to at most one rounding), y = (float)(sum * scale) in double.
 *   mode B: x is quantised per token to int8 q with scale s and zero point z,
 *           acc = sum_k w*q in exact integers,
 *           y = ((float)(acc - z*rowsum) * s) * scale, two fp32 products.
 * The pages say nothing about activation quantisation; the quantiser below is
 * the plain per-token asymmetric reading (range widened to include 0, round
 * half to even), and the symmetric one for prefill.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -pthread -shared
 * -fPIC (see build.py in this folder).  No intrinsics, no vector code.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <pthread.h>

/* ------------------------------------------------------------------ */
/* TL2P v2 layout                                                       */
/* ------------------------------------------------------------------ */
/*
 * Logical W[M][K], padded with zero weights to Mp = ceil(M/16)*16 rows and
 * Kp = ceil(K/128)*128 columns.  A tile is 16 rows x 128 columns = 512 bytes
 * = 128 uint32 words; tile (r, b) (row tile r, column block b) starts at word
 * (r * Kp/128 + b) * 128, so the 16-row panel r is contiguous along K.
 * Inside a tile the 128 words belong to 32 "lanes" of 4 words each: lane
 * L = 4*g + t owns words 4L..4L+3.  For a weight at tile-local row i (0..15)
 * and column c (0..127):
 *     g = i % 8,  h = i / 8           (row g or row g+8)
 *     s = c / 16, cc = c % 16         (16-column step inside the tile)
 *     u = cc / 8, t = (cc % 8) / 2, e = cc % 2
 *     lane L = 4*g + t, word j = 2*u + h  (0..3)
 * Its 2-bit field starts at bit 2*s + 16*e and holds 1 - w as an unsigned
 * number:  00 -> +1,  01 -> 0,  10 -> -1,  11 -> never written (decodes to
 * 0 and is counted as invalid).  Padding positions hold 01.
 */
static void tl2p_position(int64_t m, int64_t k, int64_t Kp,
                          int64_t *word_index, int *lo_bit)
{
    int64_t r = m / 16, i = m % 16;
    int64_t b = k / 128, c = k % 128;
    int g = (int)(i % 8), h = (int)(i / 8);
    int s = (int)(c / 16), cc = (int)(c % 16);
    int u = cc / 8, t = (cc % 8) / 2, e = cc % 2;
    int lane = 4 * g + t;
    int j = 2 * u + h;
    int64_t tile = r * (Kp / 128) + b;
    *word_index = (tile * 32 + lane) * 4 + j;
    *lo_bit = 2 * s + 16 * e;
}

static int64_t pad16(int64_t M) { return (M + 15) / 16 * 16; }
static int64_t pad128(int64_t K) { return (K + 127) / 128 * 128; }

int64_t oracle_tl2p_words(int64_t M, int64_t K)
{
    if (M <= 0 || K <= 0) return 0;
    return pad16(M) * pad128(K) / 16;
}

/* Pack W (int8, row-major M x K) into P.  Returns the number of entries of W
 * outside {-1, 0, 1}; P is fully written (padding = zero weights) only when
 * that is 0. */
int64_t oracle_pack(const int8_t *W, int64_t M, int64_t K, uint32_t *P)
{
    int64_t bad = 0;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            int8_t v = W[m * K + k];
            if (v < -1 || v > 1) ++bad;
        }
    if (bad) return bad;
    int64_t words = oracle_tl2p_words(M, K);
    for (int64_t i = 0; i < words; ++i) P[i] = 0x55555555u;   /* every field 01 */
    int64_t Kp = pad128(K);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            int v = W[m * K + k];
            int64_t wi; int lb;
            tl2p_position(m, k, Kp, &wi, &lb);
            P[wi] &= ~((uint32_t)3u << lb);
            P[wi] |= (uint32_t)(1 - v) << lb;
        }
    return 0;
}

/* Decode one weight.  *invalid is incremented for the field 11. */
static int oracle_weight(const uint32_t *P, int64_t m, int64_t k, int64_t Kp,
                         int64_t *invalid)
{
    int64_t wi; int lb;
    tl2p_position(m, k, Kp, &wi, &lb);
    int f = (int)((P[wi] >> lb) & 3u);
    if (f == 3) {
        if (invalid) ++*invalid;
        return 0;
    }
    return 1 - f;
}

/* Unpack the logical M x K block.  Returns the count of invalid codes seen in
 * the whole padded matrix plus the count of non-zero padding weights (both
 * must be 0 for a well-formed matrix). */
int64_t oracle_unpack(const uint32_t *P, int64_t M, int64_t K, int8_t *W)
{
    int64_t Mp = pad16(M), Kp = pad128(K), bad = 0;
    for (int64_t m = 0; m < Mp; ++m)
        for (int64_t k = 0; k < Kp; ++k) {
            int v = oracle_weight(P, m, k, Kp, &bad);
            if (m < M && k < K) W[m * K + k] = (int8_t)v;
            else if (v != 0) ++bad;
        }
    return bad;
}

/* rowsum[m] = sum_k w[m,k] (the per-row metadata next to the scale). */
void oracle_rowsum(const uint32_t *P, int64_t M, int64_t K, int32_t *rowsum)
{
    int64_t Kp = pad128(K);
    for (int64_t m = 0; m < M; ++m) {
        int64_t acc = 0;
        for (int64_t k = 0; k < K; ++k) acc += oracle_weight(P, m, k, Kp, NULL);
        rowsum[m] = (int32_t)acc;
    }
}

/* ------------------------------------------------------------------ */
/* bf16 helpers                                                          */
/* ------------------------------------------------------------------ */
static float bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even; NaN stays NaN. */
uint16_t oracle_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void oracle_bf16_rne_array(const float *in, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_rne(in[i]);
}

/* ------------------------------------------------------------------ */
/* Per-token activation quantisation (fp32, round half to even).        */
/* ------------------------------------------------------------------ */
/* asymmetric: lo = min(0, min x), hi = max(0, max x), s = (hi - lo) / 255,
 *             z = -128 - rint(lo / s), q = clamp(rint(x / s) + z, -128, 127);
 *             hi == lo == 0 gives s = 1, z = 0, q = 0.
 * symmetric:  a = max |x|, s = a / 127 (s = 1 when a == 0), z = 0,
 *             q = clamp(rint(x / s), -127, 127). */
void oracle_quant(const uint16_t *X, int64_t N, int64_t K, int symmetric,
                  int8_t *Q, float *s_out, int32_t *z_out)
{
    for (int64_t n = 0; n < N; ++n) {
        const uint16_t *x = X + n * K;
        float s;
        int32_t z;
        if (symmetric) {
            float a = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                float v = fabsf(bf16_to_float(x[k]));
                if (v > a) a = v;
            }
            s = (a == 0.0f) ? 1.0f : a / 127.0f;
            z = 0;
            for (int64_t k = 0; k < K; ++k) {
                float r = rintf(bf16_to_float(x[k]) / s);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                Q[n * K + k] = (int8_t)r;
            }
        } else {
            float lo = 0.0f, hi = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                float v = bf16_to_float(x[k]);
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            if (hi == lo) {           /* both 0: every x is 0 */
                s = 1.0f;
                z = 0;
            } else {
                s = (hi - lo) / 255.0f;
                z = -128 - (int32_t)rintf(lo / s);
            }
            for (int64_t k = 0; k < K; ++k) {
                float r = rintf(bf16_to_float(x[k]) / s) + (float)z;
                if (r > 127.0f) r = 127.0f;
                if (r < -128.0f) r = -128.0f;
                Q[n * K + k] = (int8_t)r;
            }
        }
        s_out[n] = s;
        z_out[n] = z;
    }
}

/* ------------------------------------------------------------------ */
/* The linears                                                          */
/* ------------------------------------------------------------------ */
/* Rows [m0, m1) of mode A.  S (optional, N x M doubles) receives the exact
 * signed sums before scaling. */
static void linear_a_rows(const uint32_t *P, const float *scale, int64_t M,
                          int64_t K, const uint16_t *X, int64_t N, float *Y,
                          double *S, int64_t m0, int64_t m1)
{
    int64_t Kp = pad128(K);
    int8_t *w = (int8_t *)malloc((size_t)(K > 0 ? K : 1));
    for (int64_t m = m0; m < m1; ++m) {
        for (int64_t k = 0; k < K; ++k) w[k] = (int8_t)oracle_weight(P, m, k, Kp, NULL);
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)w[k] * (double)bf16_to_float(X[n * K + k]);
            if (S) S[n * M + m] = acc;
            Y[n * M + m] = (float)(acc * (double)scale[m]);
        }
    }
    free(w);
}

void oracle_linear_a(const uint32_t *P, const float *scale, int64_t M, int64_t K,
                     const uint16_t *X, int64_t N, float *Y, double *S)
{
    linear_a_rows(P, scale, M, K, X, N, Y, S, 0, M);
}

static void linear_b_rows(const uint32_t *P, const float *scale,
                          const int32_t *rowsum, int64_t M, int64_t K,
                          const int8_t *Q, const float *s, const int32_t *z,
                          int64_t N, int32_t *ACC, float *Y, int64_t m0, int64_t m1)
{
    int64_t Kp = pad128(K);
    int8_t *w = (int8_t *)malloc((size_t)(K > 0 ? K : 1));
    for (int64_t m = m0; m < m1; ++m) {
        for (int64_t k = 0; k < K; ++k) w[k] = (int8_t)oracle_weight(P, m, k, Kp, NULL);
        for (int64_t n = 0; n < N; ++n) {
            int64_t acc = 0;
            for (int64_t k = 0; k < K; ++k) acc += (int64_t)w[k] * (int64_t)Q[n * K + k];
            if (ACC) ACC[n * M + m] = (int32_t)acc;
            int64_t corrected = acc - (int64_t)z[n] * (int64_t)rowsum[m];
            float t = (float)corrected * s[n];
            Y[n * M + m] = t * scale[m];
        }
    }
    free(w);
}

void oracle_linear_b(const uint32_t *P, const float *scale, const int32_t *rowsum,
                     int64_t M, int64_t K, const int8_t *Q, const float *s,
                     const int32_t *z, int64_t N, int32_t *ACC, float *Y)
{
    linear_b_rows(P, scale, rowsum, M, K, Q, s, z, N, ACC, Y, 0, M);
}

/* ------------------------------------------------------------------ */
/* Threaded drivers, used only to time the oracle on all host cores.    */
/* Rows are split into contiguous ranges, one per thread; the arithmetic */
/* per row is exactly the single-thread code above.                       */
/* ------------------------------------------------------------------ */
typedef struct {
    int mode;
    const uint32_t *P; const float *scale; const int32_t *rowsum;
    int64_t M, K, N;
    const uint16_t *X; const int8_t *Q; const float *s; const int32_t *z;
    float *Y; int32_t *ACC;
    int64_t m0, m1;
} job_t;

static void *job_run(void *arg)
{
    job_t *j = (job_t *)arg;
    if (j->mode == 0)
        linear_a_rows(j->P, j->scale, j->M, j->K, j->X, j->N, j->Y, NULL, j->m0, j->m1);
    else
        linear_b_rows(j->P, j->scale, j->rowsum, j->M, j->K, j->Q, j->s, j->z,
                      j->N, j->ACC, j->Y, j->m0, j->m1);
    return NULL;
}

static void run_threads(job_t proto, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    job_t jobs[256];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = proto;
        jobs[i].m0 = proto.M * i / nthreads;
        jobs[i].m1 = proto.M * (i + 1) / nthreads;
        pthread_create(&th[i], NULL, job_run, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
}

void oracle_linear_a_mt(const uint32_t *P, const float *scale, int64_t M, int64_t K,
                        const uint16_t *X, int64_t N, float *Y, int nthreads)
{
    job_t j = {0};
    j.mode = 0; j.P = P; j.scale = scale; j.M = M; j.K = K; j.N = N; j.X = X; j.Y = Y;
    run_threads(j, nthreads);
}

void oracle_linear_b_mt(const uint32_t *P, const float *scale, const int32_t *rowsum,
                        int64_t M, int64_t K, const int8_t *Q, const float *s,
                        const int32_t *z, int64_t N, float *Y, int nthreads)
{
    job_t j = {0};
    j.mode = 1; j.P = P; j.scale = scale; j.rowsum = rowsum; j.M = M; j.K = K;
    j.N = N; j.Q = Q; j.s = s; j.z = z; j.Y = Y;
    run_threads(j, nthreads);
}

/* ------------------------------------------------------------------ */
/* int8 output head and embedding                                       */
/* ------------------------------------------------------------------ */
/*
 * The projections are ternary, but the embedding table and the output head
 * stay int8 with one higher-precision scale per row (blog "Neutrino-1:
 * quantization is a training decision", "What's actually ternary"; the model
 * page "Neutrino-1 8B", "Architecture", lists them as two untied int8 tensors
 * of vocabulary x hidden, one scale per row).  Greedy decoding -- and the
 * draft/verify gate, which accepts a drafted token only when it equals the
 * verifier's own argmax -- reads the head's argmax.
 *
 * Head, on activations quantised per token exactly as for the linears
 * (oracle_quant: q, s, z):
 *   acc[n,v]   = sum_d H[v,d] * q[n,d]                (exact integers)
 *   rowsum[v]  = sum_d H[v,d]
 *   logit[n,v] = ((float)(acc - z[n] * rowsum[v]) * s[n]) * scale[v]
 *                (the integer rounded once to fp32, then two fp32 products)
 *   token[n]   = the smallest v whose logit is the largest; best[n] = that logit.
 * Embedding: x[n,d] = bf16 of the fp32 product E[t,d] * scale[t], t = tokens[n].
 */
void oracle_head(const int8_t *H, const float *scale, int64_t V, int64_t D,
                 const int8_t *Q, const float *s, const int32_t *z, int64_t N,
                 int32_t *ACC, float *logits, int32_t *token, float *best)
{
    for (int64_t n = 0; n < N; ++n) {
        int64_t best_i = -1;
        float best_y = 0.0f;
        for (int64_t v = 0; v < V; ++v) {
            int64_t acc = 0, rs = 0;
            for (int64_t d = 0; d < D; ++d) {
                acc += (int64_t)H[v * D + d] * (int64_t)Q[n * D + d];
                rs += (int64_t)H[v * D + d];
            }
            int64_t corrected = acc - (int64_t)z[n] * rs;
            float per_token = (float)corrected * s[n];
            float y = per_token * scale[v];
            if (ACC) ACC[n * V + v] = (int32_t)acc;
            if (logits) logits[n * V + v] = y;
            if (best_i < 0 || y > best_y) {
                best_i = v;
                best_y = y;
            }
        }
        token[n] = (int32_t)best_i;
        best[n] = best_y;
    }
}

void oracle_embed(const int8_t *E, const float *scale, int64_t V, int64_t D,
                  const int32_t *tokens, int64_t N, uint16_t *X)
{
    for (int64_t n = 0; n < N; ++n) {
        int64_t t = tokens[n];
        for (int64_t d = 0; d < D; ++d) {
            float y = (float)E[t * D + d] * scale[t];
            X[n * D + d] = oracle_bf16_rne(y);
        }
        (void)V;
    }
}

/* ------------------------------------------------------------------ */
/* Neighbours of the linears: RMSNorm and SwiGLU                        */
/* ------------------------------------------------------------------ */
/*
 * Each decoder layer normalises its input with RMSNorm (eps 1e-6) before
 * the q/k/v and gate/up projections, and its feed-forward is SwiGLU
 * (model page "Neutrino-1 8B", "Architecture": Qwen3 geometry).  In double,
 * straight from the definitions:
 *   rmsnorm: y[n,k] = x[n,k] * gamma[k] / sqrt(mean_k x[n,k]^2 + eps)
 *   swiglu:  h[n,m] = silu(g[n,m]) * u[n,m],  silu(g) = g / (1 + exp(-g))
 */
void oracle_rmsnorm(const uint16_t *X, const uint16_t *gamma, double eps, int64_t N,
                    int64_t K, double *Y)
{
    for (int64_t n = 0; n < N; ++n) {
        const uint16_t *row = X + n * K;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double x = (double)bf16_to_float(row[k]);
            ss += x * x;
        }
        double r = 1.0 / sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; ++k)
            Y[n * K + k] = (double)bf16_to_float(row[k]) * r * (double)bf16_to_float(gamma[k]);
    }
}

void oracle_swiglu(const uint16_t *G, const uint16_t *U, int64_t N, int64_t M, double *H)
{
    for (int64_t i = 0; i < N * M; ++i) {
        double g = (double)bf16_to_float(G[i]);
        double u = (double)bf16_to_float(U[i]);
        H[i] = g / (1.0 + exp(-g)) * u;
    }
}

/* ------------------------------------------------------------------ */
/* Block-wise scales and the absmean ternariser                         */
/* ------------------------------------------------------------------ */
/*
 * The blog ("Neutrino-1: quantization is a training decision", "What's
 * actually ternary") describes each block of weights carrying its own
 * higher-precision scale, the ternary code being round(clamp(w / scale,
 * -1, 1)) with scale the block's mean absolute value.  Reading: a block is
 * 128 consecutive columns of one row (the last block of a row may be
 * shorter); the mean is taken in double over the block's real columns and
 * stored as fp32; the code is rint(clamp(w / scale, -1, 1)) with that fp32
 * scale, in double, ties to even; a block of zeros gets scale 0 and codes 0.
 *   y[n,m] = sum_b scale[m,b] * sum_{k in b} w[m,k] * x[n,k]
 * taken in double and rounded once to fp32.
 */
#define TL_BLOCK 128

void oracle_absmean_ternarize(const float *W, int64_t M, int64_t K, int8_t *T, float *bscale)
{
    int64_t KB = (K + TL_BLOCK - 1) / TL_BLOCK;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < KB; ++b) {
            int64_t k0 = b * TL_BLOCK, k1 = k0 + TL_BLOCK < K ? k0 + TL_BLOCK : K;
            double sum = 0.0;
            for (int64_t k = k0; k < k1; ++k) sum += fabs((double)W[m * K + k]);
            float scale = (float)(sum / (double)(k1 - k0));
            bscale[m * KB + b] = scale;
            for (int64_t k = k0; k < k1; ++k) {
                double r = scale > 0.0f ? (double)W[m * K + k] / (double)scale : 0.0;
                if (r > 1.0) r = 1.0;
                if (r < -1.0) r = -1.0;
                T[m * K + k] = (int8_t)rint(r);
            }
        }
}

void oracle_linear_blockscale(const uint32_t *P, const float *bscale, int64_t M, int64_t K,
                              const uint16_t *X, int64_t N, float *Y)
{
    int64_t Kp = pad128(K), KB = (K + TL_BLOCK - 1) / TL_BLOCK;
    int8_t *w = (int8_t *)malloc((size_t)(K > 0 ? K : 1));
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t k = 0; k < K; ++k) w[k] = (int8_t)oracle_weight(P, m, k, Kp, NULL);
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t *xn = X + n * K;
            double y = 0.0;
            for (int64_t b = 0; b < KB; ++b) {
                int64_t k0 = b * TL_BLOCK, k1 = k0 + TL_BLOCK < K ? k0 + TL_BLOCK : K;
                double s = 0.0;
                for (int64_t k = k0; k < k1; ++k) s += (double)w[k] * (double)bf16_to_float(xn[k]);
                y += (double)bscale[m * KB + b] * s;
            }
            Y[n * M + m] = (float)y;
        }
    }
    free(w);
}
