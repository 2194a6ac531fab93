/*
 * oracle.c -- CPU oracle for fine-grained FP8 (E4M3) quantisation and the
 * block-scaled GEMM with FP32 promotion.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plainly written
 * definition that the CUDA library is checked against.  Only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark load it; the product
 * path never does.  It shares no code, header, table or constant with the
 * CUDA sources.
 *
 * Sources (web pages on DeepSeek-V3):
 *   [V3-report]  "DeepSeek-V3 技术报告：从 671B MoE 到低成本训练系统"
 *                (xutianle.me), §6 FP8 混合精度, §6.1 细粒度量化如何处理异常值,
 *                §6.2 更高精度累加是 FP8 能训练稳定的关键.
 *   [infra]      51itzy.com infra commentary on DeepSeek-V3, FP8 paragraphs.
 *   [evolution]  "deepseek-evolution" post, 技术突破一：FP8 混合精度训练.
 *
 * What the pages fix: E4M3 for every GEMM input ([infra]; [V3-report] §6),
 * one scale per 1x128 activation tile and per 128x128 weight block, computed
 * online from the current tensor ([V3-report] §6.1), and promotion of the
 * tensor-core partial sum to FP32 after every 128 FP8 products
 * ([V3-report] §6.2).  Readings taken where they are silent (each one is
 * listed with its reason in the design notes):
 *   - E4M3 is the OCP "FN" flavour: bias 7, no infinities, max finite 448.
 *   - scale = amax / 448 as an IEEE single-precision divide; amax == 0 gives
 *     scale 1.0.
 *   - codes = E4M3(x / scale) with an IEEE single-precision divide, rounded to
 *     nearest, ties to the even code, saturating at +-448, sign kept (so -0
 *     and negative values that round to zero give 0x80).
 *   - promotion happens at each 128-wide K chunk (the same 128 as the
 *     scaling group): acc = fmaf(fl32(sa*sb), fl32(P_chunk), acc), with the
 *     chunk partial P_chunk summed exactly in double.
 *
 * Build: plain C99, no -ffast-math, -ffp-contract=off (no silent FMA).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* E4M3 format (OCP FP8 E4M3FN): 1 sign bit, 4 exponent bits (bias 7),      */
/* 3 mantissa bits; exponent field 0 is subnormal; S.1111.111 is NaN;       */
/* there is no infinity.                                                    */
/* ------------------------------------------------------------------------ */

double orc_e4m3_decode(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = (double)m * ldexp(1.0, -9);              /* m/8 * 2^(1-7) */
    else
        v = (1.0 + (double)m / 8.0) * ldexp(1.0, e - 7);
    return sign ? -v : v;
}

/* The 127 non-negative finite magnitudes, code c -> decode(c), c = 0..126.
 * Filled from the decoder above; ascending in c. */
static double MAG[127];
static double DEC[256];
static pthread_once_t tables_once = PTHREAD_ONCE_INIT;

static void build_tables(void)
{
    for (int c = 0; c < 127; ++c)
        MAG[c] = orc_e4m3_decode((uint8_t)c);
    for (int c = 0; c < 256; ++c)
        DEC[c] = orc_e4m3_decode((uint8_t)c);
}

static void ensure_tables(void) { pthread_once(&tables_once, build_tables); }

/* Round a single-precision value to the nearest E4M3 value: scan the sorted
 * magnitudes for the bracket [MAG[c], MAG[c+1]), pick the nearer end, and on
 * an exact tie the code whose last (mantissa) bit is 0.  Magnitudes at or
 * above 448 saturate to 448 (code 0x7E).  The sign bit is always carried. */
uint8_t orc_e4m3_encode(float y)
{
    ensure_tables();
    if (isnan(y))
        return signbit(y) ? 0xFF : 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int c = 0;
    while (c < 125 && MAG[c + 1] <= a)
        ++c;
    /* now MAG[c] <= a < MAG[c+1] (c+1 <= 126) */
    double lo = MAG[c], hi = MAG[c + 1];
    /* a - lo versus hi - a, compared exactly as 2a versus lo + hi */
    double twice = 2.0 * a, mid2 = lo + hi;
    int pick;
    if (twice < mid2)
        pick = c;
    else if (twice > mid2)
        pick = c + 1;
    else
        pick = (c % 2 == 0) ? c : c + 1;
    return (uint8_t)(sign | pick);
}

/* BF16 -> FP32 is exact: the BF16 bits are the top half of the FP32 bits. */
static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* FP32 -> BF16, round to nearest even (output rounding of the GEMM). */
uint16_t orc_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if (isnan(f))
        return (uint16_t)((u >> 16) | 0x40);
    uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1;
    return (uint16_t)upper;
}

/* Tile scale: amax / 448 in single precision; an all-zero tile gets 1.0. */
float orc_tile_scale(float amax)
{
    if (amax == 0.0f)
        return 1.0f;
    return amax / 448.0f;
}

/* ------------------------------------------------------------------------ */
/* Row-parallel driver: runs body(ctx, i) for i in [0, n) on nthreads.       */
/* Each index is handled by exactly one thread; no arithmetic is shared.     */
/* ------------------------------------------------------------------------ */
typedef void (*row_fn)(void *ctx, int64_t i);
typedef struct {
    row_fn fn;
    void *ctx;
    int64_t n;
    int t, nt;
} job_t;

static void *job_main(void *p)
{
    job_t *j = (job_t *)p;
    for (int64_t i = j->t; i < j->n; i += j->nt)
        j->fn(j->ctx, i);
    return NULL;
}

static void parallel_for(int64_t n, int nthreads, row_fn fn, void *ctx)
{
    ensure_tables();
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if (n < nthreads)
        nthreads = (int)(n > 0 ? n : 1);
    pthread_t th[256];
    job_t jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].n = n;
        jobs[t].t = t;
        jobs[t].nt = nthreads;
    }
    for (int t = 1; t < nthreads; ++t)
        pthread_create(&th[t], NULL, job_main, &jobs[t]);
    job_main(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------------ */
/* 1x128 tiles along the contiguous dimension (activations, [V3-report]     */
/* §6.1: one scale per token per 128 channels).                              */
/* x: BF16 bits [M][ldx]; q: codes [M][ldq]; s: FP32 [K/128][lds].          */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint16_t *x;
    int64_t M, K, ldx;
    uint8_t *q;
    int64_t ldq;
    float *s;
    int64_t lds;
} q1_ctx;

static void q1_row(void *p, int64_t m)
{
    q1_ctx *c = (q1_ctx *)p;
    for (int64_t kb = 0; kb < c->K / 128; ++kb) {
        const uint16_t *xt = c->x + m * c->ldx + kb * 128;
        float amax = 0.0f;
        for (int k = 0; k < 128; ++k) {
            float a = fabsf(bf16_to_f32(xt[k]));
            if (a > amax)
                amax = a;
        }
        float sc = orc_tile_scale(amax);
        c->s[kb * c->lds + m] = sc;
        for (int k = 0; k < 128; ++k)
            c->q[m * c->ldq + kb * 128 + k] = orc_e4m3_encode(bf16_to_f32(xt[k]) / sc);
    }
}

void orc_quant_1x128_rows(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                          uint8_t *q, int64_t ldq, float *s, int64_t lds, int nthreads)
{
    q1_ctx c = {x, M, K, ldx, q, ldq, s, lds};
    parallel_for(M, nthreads, q1_row, &c);
}

/* ------------------------------------------------------------------------ */
/* 1x128 tiles along the strided dimension (the token dimension of a        */
/* weight-gradient operand): x is BF16 [T][ldx] with C channels; each tile  */
/* is 128 consecutive tokens of one channel.  Output is transposed so that  */
/* the token dimension is contiguous: q [C][ldq] (T codes per row),         */
/* s [T/128][lds] (C scales per row).                                       */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint16_t *x;
    int64_t T, C, ldx;
    uint8_t *q;
    int64_t ldq;
    float *s;
    int64_t lds;
} q2_ctx;

static void q2_chan(void *p, int64_t ch)
{
    q2_ctx *c = (q2_ctx *)p;
    for (int64_t tb = 0; tb < c->T / 128; ++tb) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float a = fabsf(bf16_to_f32(c->x[(tb * 128 + i) * c->ldx + ch]));
            if (a > amax)
                amax = a;
        }
        float sc = orc_tile_scale(amax);
        c->s[tb * c->lds + ch] = sc;
        for (int i = 0; i < 128; ++i) {
            float v = bf16_to_f32(c->x[(tb * 128 + i) * c->ldx + ch]);
            c->q[ch * c->ldq + tb * 128 + i] = orc_e4m3_encode(v / sc);
        }
    }
}

void orc_quant_1x128_cols(const uint16_t *x, int64_t T, int64_t C, int64_t ldx,
                          uint8_t *q, int64_t ldq, float *s, int64_t lds, int nthreads)
{
    q2_ctx c = {x, T, C, ldx, q, ldq, s, lds};
    parallel_for(C, nthreads, q2_chan, &c);
}

/* ------------------------------------------------------------------------ */
/* 128x128 blocks (weights, [V3-report] §6.1).  w: BF16 [N][ldw];            */
/* q: codes [N][ldq]; s: FP32 [ceil(N/128)][lds].  A partial edge block uses */
/* only the rows that exist.                                                */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint16_t *w;
    int64_t N, K, ldw;
    uint8_t *q;
    int64_t ldq;
    float *s;
    int64_t lds;
} q3_ctx;

static void q3_blockrow(void *p, int64_t nb)
{
    q3_ctx *c = (q3_ctx *)p;
    int64_t r0 = nb * 128;
    int64_t r1 = r0 + 128 < c->N ? r0 + 128 : c->N;
    for (int64_t kb = 0; kb < c->K / 128; ++kb) {
        float amax = 0.0f;
        for (int64_t r = r0; r < r1; ++r)
            for (int k = 0; k < 128; ++k) {
                float a = fabsf(bf16_to_f32(c->w[r * c->ldw + kb * 128 + k]));
                if (a > amax)
                    amax = a;
            }
        float sc = orc_tile_scale(amax);
        c->s[nb * c->lds + kb] = sc;
        for (int64_t r = r0; r < r1; ++r)
            for (int k = 0; k < 128; ++k)
                c->q[r * c->ldq + kb * 128 + k] =
                    orc_e4m3_encode(bf16_to_f32(c->w[r * c->ldw + kb * 128 + k]) / sc);
    }
}

void orc_quant_128x128(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                       uint8_t *q, int64_t ldq, float *s, int64_t lds, int nthreads)
{
    q3_ctx c = {w, N, K, ldw, q, ldq, s, lds};
    parallel_for((N + 127) / 128, nthreads, q3_blockrow, &c);
}

/* ------------------------------------------------------------------------ */
/* Block-scaled GEMM, C = A * B^T ([V3-report] §6, §6.2).                    */
/*   A codes [M][lda], sa [K/128][ldsa] (one scale per row per K chunk).    */
/*   B codes [N][ldb];                                                      */
/*     b_mode 0: sb [ceil(N/128)][ldsb], one scale per 128x128 block;        */
/*     b_mode 1: sb [K/128][ldsb], one scale per row n per K chunk.          */
/* For each output (m, n): acc = 0 (FP32); for each 128-wide K chunk kb the  */
/* chunk partial P = sum of decoded products is formed exactly in double,    */
/* rounded to FP32, and promoted: acc = fmaf(fl32(sa*sb), fl32(P), acc).     */
/* Only the rows listed in rows[0..nrows) are computed; out is FP32           */
/* [nrows][N].                                                              */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint8_t *A;
    int64_t lda;
    const float *sa;
    int64_t ldsa;
    const uint8_t *B;
    int64_t ldb;
    const float *sb;
    int64_t ldsb;
    int b_mode;
    int64_t N, K;
    const int64_t *rows;
    float *out;
} g_ctx;

static void g_row(void *p, int64_t r)
{
    g_ctx *c = (g_ctx *)p;
    int64_t m = c->rows[r];
    const uint8_t *a = c->A + m * c->lda;
    for (int64_t n = 0; n < c->N; ++n) {
        const uint8_t *b = c->B + n * c->ldb;
        float acc = 0.0f;
        for (int64_t kb = 0; kb < c->K / 128; ++kb) {
            double P = 0.0;
            for (int k = 0; k < 128; ++k)
                P += DEC[a[kb * 128 + k]] * DEC[b[kb * 128 + k]];
            float P32 = (float)P;
            float s_a = c->sa[kb * c->ldsa + m];
            float s_b = (c->b_mode == 0) ? c->sb[(n / 128) * c->ldsb + kb]
                                         : c->sb[kb * c->ldsb + n];
            float sc = s_a * s_b;
            acc = fmaf(sc, P32, acc);
        }
        c->out[r * c->N + n] = acc;
    }
}

void orc_gemm_blockscaled(const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa,
                          const uint8_t *B, int64_t ldb, const float *sb, int64_t ldsb,
                          int b_mode, int64_t N, int64_t K,
                          const int64_t *rows, int64_t nrows, float *out, int nthreads)
{
    g_ctx c = {A, lda, sa, ldsa, B, ldb, sb, ldsb, b_mode, N, K, rows, out};
    parallel_for(nrows, nthreads, g_row, &c);
}

/* Round an FP32 buffer to BF16 bits (RNE). */
void orc_bf16_round_buffer(const float *x, uint16_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        y[i] = orc_bf16_rne(x[i]);
}

/* Encode a buffer of FP32 values (used to compare encoders exhaustively). */
typedef struct {
    const float *x;
    uint8_t *q;
    int64_t n, chunk;
} enc_ctx;

static void enc_chunk(void *p, int64_t ci)
{
    enc_ctx *c = (enc_ctx *)p;
    int64_t i0 = ci * c->chunk, i1 = i0 + c->chunk < c->n ? i0 + c->chunk : c->n;
    for (int64_t i = i0; i < i1; ++i)
        c->q[i] = orc_e4m3_encode(c->x[i]);
}

void orc_e4m3_encode_buffer(const float *x, uint8_t *q, int64_t n, int nthreads)
{
    enc_ctx c = {x, q, n, 1 << 16};
    parallel_for((n + c.chunk - 1) / c.chunk, nthreads, enc_chunk, &c);
}

/* Encode every FP32 bit pattern in [lo, lo + n) (as uint32 values). */
typedef struct {
    uint64_t lo;
    uint8_t *q;
    int64_t n, chunk;
} encp_ctx;

static void encp_chunk(void *p, int64_t ci)
{
    encp_ctx *c = (encp_ctx *)p;
    int64_t i0 = ci * c->chunk, i1 = i0 + c->chunk < c->n ? i0 + c->chunk : c->n;
    for (int64_t i = i0; i < i1; ++i) {
        uint32_t u = (uint32_t)(c->lo + (uint64_t)i);
        float f;
        memcpy(&f, &u, 4);
        c->q[i] = orc_e4m3_encode(f);
    }
}

void orc_e4m3_encode_patterns(uint64_t lo, int64_t n, uint8_t *q, int nthreads)
{
    encp_ctx c = {lo, q, n, 1 << 16};
    parallel_for((n + c.chunk - 1) / c.chunk, nthreads, encp_chunk, &c);
}

/* ======================================================================== */
/* The MoE chain ([V3-report] §2 DeepSeekMoE: 256 routed experts, 8 per     */
/* token, SwiGLU experts; §4 无辅助损失负载均衡: sigmoid affinity to each    */
/* expert's centroid, selection by affinity + bias, gate from the affinity  */
/* normalised over the selected experts).                                   */
/* ======================================================================== */

/* Affinity logits l[t][e] = u_t . c_e, the token-centroid product inside  */
/* the sigmoid of [V3-report] §4, in double: every product of a BF16 and an */
/* FP32 value is exact in double (8 + 24 significant bits), and the sum of  */
/* D of them in double is within D * 2^-53 * sum |u c| of the exact value,  */
/* far below any FP32 evaluation.  No summation order of a GPU kernel is    */
/* adopted.  x: BF16 [T][ldx] (D used); c: FP32 [E][ldc]; l: double [T][E].*/
typedef struct {
    const uint16_t *x;
    int64_t D, ldx;
    const float *c;
    int64_t ldc, E;
    double *l;
} rl_ctx;

static void rl_token(void *p, int64_t t)
{
    rl_ctx *c = (rl_ctx *)p;
    const uint16_t *u = c->x + t * c->ldx;
    for (int64_t e = 0; e < c->E; ++e) {
        const float *ce = c->c + e * c->ldc;
        double acc = 0.0;
        for (int64_t k = 0; k < c->D; ++k)
            acc += (double)bf16_to_f32(u[k]) * (double)ce[k];
        c->l[t * c->E + e] = acc;
    }
}

void orc_route_logits(const uint16_t *x, int64_t T, int64_t D, int64_t ldx,
                      const float *c, int64_t ldc, int64_t E, double *l, int nthreads)
{
    rl_ctx ctx = {x, D, ldx, c, ldc, E, l};
    parallel_for(T, nthreads, rl_token, &ctx);
}

/* Gates of a given selection: fl32(s_e / sum of the chosen s) with        */
/* s_e = 1 / (1 + exp(-l_e)), the sum taken over the chosen experts in the  */
/* order listed, in double ([V3-report] §4: the gate is the affinity        */
/* normalised over the selected experts).                                   */
void orc_route_gates(const double *l, int64_t T, int64_t E, const int32_t *sel, int topk, float *gate)
{
    for (int64_t t = 0; t < T; ++t) {
        double sum = 0.0;
        for (int j = 0; j < topk; ++j)
            sum += 1.0 / (1.0 + exp(-l[t * E + sel[t * topk + j]]));
        for (int j = 0; j < topk; ++j)
            gate[t * topk + j] = (float)((1.0 / (1.0 + exp(-l[t * E + sel[t * topk + j]]))) / sum);
    }
}

/* Selection: affinity s_e = 1 / (1 + exp(-l_e)) and key_e = s_e + b_e in   */
/* double; the top-k keys win, a tie going to the lower expert index.  The  */
/* chosen experts are listed in increasing index order; their gates are     */
/* those of orc_route_gates.                                                */
void orc_route_select(const double *l, int64_t T, int64_t E, const float *bias, int topk,
                      int32_t *sel, float *gate)
{
    double *key = (double *)malloc((size_t)E * sizeof(double));
    char *taken = (char *)malloc((size_t)E);
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) {
            key[e] = 1.0 / (1.0 + exp(-l[t * E + e])) + (double)bias[e];
            taken[e] = 0;
        }
        for (int j = 0; j < topk; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || key[e] > key[best]))
                    best = e;
            if (best < 0)
                break; /* topk > E: every expert is chosen */
            taken[best] = 1;
        }
        int j = 0;
        for (int64_t e = 0; e < E; ++e)
            if (taken[e])
                sel[t * topk + j++] = (int32_t)e;
    }
    orc_route_gates(l, T, E, sel, topk, gate);
    free(key);
    free(taken);
}

/* Grouping: rows of expert e are offsets[e] .. offsets[e+1]-1, holding the */
/* tokens that chose e in increasing token order.  token_of_row[r] is the   */
/* token of row r; row_of[t*topk + j] is the row of token t's j-th expert.  */
void orc_route_permute(const int32_t *sel, int64_t T, int topk, int64_t E,
                       int32_t *offsets, int32_t *token_of_row, int32_t *row_of)
{
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) {
        int32_t n = 0;
        for (int64_t i = 0; i < T * topk; ++i)
            n += (sel[i] == e);
        offsets[e + 1] = offsets[e] + n;
    }
    for (int64_t e = 0; e < E; ++e) {
        int32_t r = offsets[e];
        for (int64_t t = 0; t < T; ++t)
            for (int j = 0; j < topk; ++j)
                if (sel[t * topk + j] == e) {
                    token_of_row[r] = (int32_t)t;
                    row_of[t * topk + j] = r;
                    ++r;
                }
    }
}

/* SwiGLU of one expert's up-projection and its 1x128 quantisation: from    */
/* the FP32 accumulators gate g = acc[r][i] and up u = acc[r][Nh + i],      */
/* h = g / (1 + exp(-g)) * u in double, rounded once to FP32; then the      */
/* 1x128 tiles of h as for activations: amax over |h| (FP32), scale =       */
/* amax / 448 (IEEE single), codes = E4M3(fl32(h / scale)).                 */
/* acc: FP32 [R][ldacc] (2*Nh used); q: [R][ldq]; s: FP32 [Nh/128][lds].    */
typedef struct {
    const float *acc;
    int64_t Nh, ldacc;
    uint8_t *q;
    int64_t ldq;
    float *s;
    int64_t lds;
} sw_ctx;

static void sw_row(void *p, int64_t r)
{
    sw_ctx *c = (sw_ctx *)p;
    const float *a = c->acc + r * c->ldacc;
    float h[128];
    for (int64_t kb = 0; kb < c->Nh / 128; ++kb) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            double g = a[kb * 128 + i], u = a[c->Nh + kb * 128 + i];
            h[i] = (float)(g / (1.0 + exp(-g)) * u);
            float m = fabsf(h[i]);
            if (m > amax)
                amax = m;
        }
        float sc = orc_tile_scale(amax);
        c->s[kb * c->lds + r] = sc;
        for (int i = 0; i < 128; ++i)
            c->q[r * c->ldq + kb * 128 + i] = orc_e4m3_encode(h[i] / sc);
    }
}

void orc_swiglu_quant(const float *acc, int64_t R, int64_t Nh, int64_t ldacc,
                      uint8_t *q, int64_t ldq, float *s, int64_t lds, int nthreads)
{
    sw_ctx c = {acc, Nh, ldacc, q, ldq, s, lds};
    parallel_for(R, nthreads, sw_row, &c);
}

/* Combine: y[t][n] = sum_j gate[t][j] * Y[row_of[t][j]][n], one FP32 fused */
/* multiply-add per expert in the listed (increasing expert) order, from    */
/* the BF16 expert outputs; the result rounded to BF16 (RNE).               */
typedef struct {
    const uint16_t *Y;
    int64_t ldy, N;
    const int32_t *row_of;
    const float *gate;
    int topk;
    uint16_t *out;
    int64_t ldo;
} cb_ctx;

static void cb_token(void *p, int64_t t)
{
    cb_ctx *c = (cb_ctx *)p;
    for (int64_t n = 0; n < c->N; ++n) {
        float acc = 0.0f;
        for (int j = 0; j < c->topk; ++j)
            acc = fmaf(c->gate[t * c->topk + j],
                       bf16_to_f32(c->Y[(int64_t)c->row_of[t * c->topk + j] * c->ldy + n]), acc);
        c->out[t * c->ldo + n] = orc_bf16_rne(acc);
    }
}

void orc_moe_combine(const uint16_t *Y, int64_t ldy, int64_t N, const int32_t *row_of,
                     const float *gate, int64_t T, int topk, uint16_t *out, int64_t ldo,
                     int nthreads)
{
    cb_ctx c = {Y, ldy, N, row_of, gate, topk, out, ldo};
    parallel_for(T, nthreads, cb_token, &c);
}

/* ======================================================================== */
/* Power-of-two (UE8M0) scales: the variant whose scales the tensor cores'  */
/* block-scaled MMA can apply in hardware.  The scale of a tile is 2^e, e   */
/* the smallest integer with amax <= 448 * 2^e (so no code saturates), kept */
/* within UE8M0's range (e >= -127); an all-zero tile has e = 0.  Codes are */
/* E4M3(x * 2^-e): the scaling itself is exact.                             */
/* ======================================================================== */
int orc_pow2_exponent(float amax)
{
    if (amax == 0.0f)
        return 0;
    int e = ilogb(amax) - 9; /* 448 * 2^e = 0.875 * 2^(ilogb+0) < amax: too small */
    while ((double)amax > ldexp(448.0, e))
        ++e;
    return e < -127 ? -127 : e;
}

static uint8_t pow2_code(float x, int e) { return orc_e4m3_encode((float)ldexp((double)x, -e)); }

static void q1p_row(void *p, int64_t m)
{
    q1_ctx *c = (q1_ctx *)p;
    for (int64_t kb = 0; kb < c->K / 128; ++kb) {
        const uint16_t *xt = c->x + m * c->ldx + kb * 128;
        float amax = 0.0f;
        for (int k = 0; k < 128; ++k) {
            float a = fabsf(bf16_to_f32(xt[k]));
            if (a > amax)
                amax = a;
        }
        int e = orc_pow2_exponent(amax);
        c->s[kb * c->lds + m] = (float)ldexp(1.0, e);
        for (int k = 0; k < 128; ++k)
            c->q[m * c->ldq + kb * 128 + k] = pow2_code(bf16_to_f32(xt[k]), e);
    }
}

void orc_quant_1x128_rows_pow2(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                               uint8_t *q, int64_t ldq, float *s, int64_t lds, int nthreads)
{
    q1_ctx c = {x, M, K, ldx, q, ldq, s, lds};
    parallel_for(M, nthreads, q1p_row, &c);
}

static void q3p_blockrow(void *p, int64_t nb)
{
    q3_ctx *c = (q3_ctx *)p;
    int64_t r0 = nb * 128;
    int64_t r1 = r0 + 128 < c->N ? r0 + 128 : c->N;
    for (int64_t kb = 0; kb < c->K / 128; ++kb) {
        float amax = 0.0f;
        for (int64_t r = r0; r < r1; ++r)
            for (int k = 0; k < 128; ++k) {
                float a = fabsf(bf16_to_f32(c->w[r * c->ldw + kb * 128 + k]));
                if (a > amax)
                    amax = a;
            }
        int e = orc_pow2_exponent(amax);
        c->s[nb * c->lds + kb] = (float)ldexp(1.0, e);
        for (int64_t r = r0; r < r1; ++r)
            for (int k = 0; k < 128; ++k)
                c->q[r * c->ldq + kb * 128 + k] = pow2_code(bf16_to_f32(c->w[r * c->ldw + kb * 128 + k]), e);
    }
}

void orc_quant_128x128_pow2(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                            uint8_t *q, int64_t ldq, float *s, int64_t lds, int nthreads)
{
    q3_ctx c = {w, N, K, ldw, q, ldq, s, lds};
    parallel_for((N + 127) / 128, nthreads, q3p_blockrow, &c);
}

/* The product of the scaled codes summed in double over all of K, then     */
/* rounded once to FP32: C[m][n] = fl32(sum_kb sa*sb * sum_k dec*dec).      */
/* With power-of-two scales every term is exact in double, so this is the   */
/* value a block-scaled tensor-core product approximates (it accumulates in */
/* FP32 inside the MMA instead of promoting per chunk).                     */
static void ge_row(void *p, int64_t r)
{
    g_ctx *c = (g_ctx *)p;
    int64_t m = c->rows[r];
    const uint8_t *a = c->A + m * c->lda;
    for (int64_t n = 0; n < c->N; ++n) {
        const uint8_t *b = c->B + n * c->ldb;
        double acc = 0.0;
        for (int64_t kb = 0; kb < c->K / 128; ++kb) {
            double P = 0.0;
            for (int k = 0; k < 128; ++k)
                P += DEC[a[kb * 128 + k]] * DEC[b[kb * 128 + k]];
            double s_a = c->sa[kb * c->ldsa + m];
            double s_b = (c->b_mode == 0) ? c->sb[(n / 128) * c->ldsb + kb] : c->sb[kb * c->ldsb + n];
            acc += s_a * s_b * P;
        }
        c->out[r * c->N + n] = (float)acc;
    }
}

void orc_gemm_exact_sum(const uint8_t *A, int64_t lda, const float *sa, int64_t ldsa,
                        const uint8_t *B, int64_t ldb, const float *sb, int64_t ldsb,
                        int b_mode, int64_t N, int64_t K,
                        const int64_t *rows, int64_t nrows, float *out, int nthreads)
{
    g_ctx c = {A, lda, sa, ldsa, B, ldb, sb, ldsb, b_mode, N, K, rows, out};
    parallel_for(nrows, nthreads, ge_row, &c);
}
