/*
 * Oracle for the compressed-KV attention path of a DeepSeek-V4-style engine.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package's
 * smoke check and the benchmark's CPU-baseline leg may load this library.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * Plain, slow, literal C99: one token at a time, dot products and softmax
 * sums in double, results rounded to float where the engine stores floats
 * (the per-layer cache holds float arrays: "Metal グラフと圧縮 KV の実装を読む" §2).
 * Build: gcc -O2 -std=c99 -fopenmp -ffp-contract=off (no fast-math, so that the
 * fp32 indexer chain below is evaluated exactly as written).
 *
 * Sources (page title, section):
 *   [P2] "Metal グラフと圧縮 KV の実装を読む" (DwarfStar/ds4 series, part 3)
 *   [P1] "【#4】ds4.c を読み解く" (disk KV cache, DSV4 payload)
 * Readings where the pages are open are marked READING and listed in the
 * design notes; they are shared with the CUDA path by specification only.
 *
 * Parity status: every function below is pinned by a CPU test (closed forms,
 * invariants, brute force or a library routine), see tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t d_model, head_dim, n_rot, idx_head_dim, n_heads, ratio, swa, top_k;
    int32_t comp_cap, idx_cap;
    int32_t bf16;          /* weights and hidden stored as bfloat16 (uint16) */
    float rms_eps;
    float attn_scale;
    double rope_base;
    int32_t idx_heads;     /* indexer query heads of the multi-head score (0 or 1: one query vector) */
    int32_t idx_qat;       /* 1: the indexer rows and queries take the Hadamard + FP4 round trip */
} orc_cfg;

typedef struct {
    const void *wkv, *wgate;   /* [coff*Dl][d_model] */
    const float *ape;          /* [ratio][coff*Dl] */
    const float *norm;         /* [Dl] RMSNorm gain, NULL = ones */
} orc_lane_w;

typedef struct {
    float *comp;               /* [cap][Dl] appended compressed rows */
    float *state_kv;           /* [coff*ratio][coff*Dl] frontier */
    float *state_score;        /* same shape */
    float *prequant;           /* [cap][Dl] row before the FP8 round trip, may be NULL */
} orc_lane_s;

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * Layer routing, ring capacity, chunk size
 * ------------------------------------------------------------------------- */

/* [P2] §1, ds4_expected_layer_compress_ratio: Flash layers 0-1 uncompressed,
 * Pro layers 0-1 ratio 128; from layer 2 on, even layers ratio 4, odd 128.
 * variant 0 = Flash, 1 = Pro. */
int orc_layer_ratio(int variant, int il) {
    if (il < 2) return variant == 0 ? 0 : 128;
    return (il % 2 == 0) ? 4 : 128;
}

/* [P2] §2, ds4_default_raw_cap: the raw ring holds DS4_N_SWA = 128 rows,
 * clamped to the context size. */
int orc_raw_cap(int ctx_size) {
    int cap = 128;
    if (cap > ctx_size) cap = ctx_size;
    return cap;
}

/* [P2] §3, ds4_default_prefill_cap_for_prompt: an environment override wins;
 * otherwise prompts longer than 4096 tokens run in 4096-token chunks.
 * READING: a prompt of at most 4096 tokens runs in one pass (the page elides
 * that branch). */
int orc_prefill_chunk(int prompt_len, int env_chunk) {
    if (env_chunk > 0) return env_chunk;
    if (prompt_len > 4096) return 4096;
    return prompt_len;
}

/* READING (C-5): theta_i = base^(-2i/n_rot), computed in double and rounded
 * to float; [P2] §8 names the base but not the frequency formula. */
void orc_inv_freq(double base, int n_rot, float *out) {
    for (int i = 0; i < n_rot / 2; i++)
        out[i] = (float)pow(base, -2.0 * (double)i / (double)n_rot);
}

/* ---------------------------------------------------------------------------
 * Element access
 * ------------------------------------------------------------------------- */

static double elem(const void *base, int bf16, size_t i) {
    if (!bf16) return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------------------
 * A1. Projections.  [P2] §4: wkv makes the KV candidate, wgate the score;
 * [P2] §5: both are coff*head_dim wide (coff = 2 on ratio-4 layers).
 * out[t][n] = float( sum_k W[n][k] * h[t][k] ), the sum in double.
 * ------------------------------------------------------------------------- */
void orc_project(const void *W, const void *h, int bf16, int T, int K, int N, float *out) {
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        for (int n = 0; n < N; n++) {
            double s = 0.0;
            for (int k = 0; k < K; k++)
                s += elem(W, bf16, (size_t)n * K + k) * elem(h, bf16, (size_t)t * K + k);
            out[(size_t)t * N + n] = (float)s;
        }
    }
}

/* ---------------------------------------------------------------------------
 * A7. FP8 E4M3 round trip.  [P2] §9: the attention compressed row goes through
 * an E4M3 quantise/dequantise of its non-RoPE part; the RoPE tail is left as is.
 * READING (C-6): OCP E4M3FN (bias 7, max 448, no infinities), round to nearest
 * with ties to even, saturating; one power-of-two scale per 64-element block,
 * the smallest 2^e with amax <= 448 * 2^e (e = 0 for an all-zero block).
 * ------------------------------------------------------------------------- */

/* Value of the non-negative E4M3FN code c (0x00..0x7E). */
static double e4m3_value(int c) {
    int E = c >> 3, m = c & 7;
    if (E == 0) return ldexp((double)m, -9);          /* subnormal: m * 2^-9 */
    return ldexp(1.0 + (double)m / 8.0, E - 7);
}

/* Nearest E4M3FN value to y, ties to the even code, saturating to +-448. */
float orc_e4m3_rne(float y) {
    double a = fabs((double)y);
    double r;
    if (a >= 448.0) {
        r = 448.0;
    } else {
        int lo = 0;                                     /* largest code with value <= a */
        for (int c = 0; c <= 0x7E; c++)
            if (e4m3_value(c) <= a) lo = c;
        double vlo = e4m3_value(lo), vhi = e4m3_value(lo + 1);
        double dlo = a - vlo, dhi = vhi - a;
        if (dlo < dhi) r = vlo;
        else if (dhi < dlo) r = vhi;
        else r = ((lo & 1) == 0) ? vlo : vhi;
    }
    return (float)(signbit(y) ? -r : r);
}

/* Smallest integer e with amax <= 448 * 2^e; 0 when amax == 0. */
int orc_fp8_scale_exp(float amax) {
    if (!(amax > 0.0f)) return 0;
    int e = 0;
    while ((double)amax > ldexp(448.0, e)) e++;
    while ((double)amax <= ldexp(448.0, e - 1)) e--;
    return e;
}

void orc_fp8_roundtrip(float *row, int n_nope) {
    for (int b0 = 0; b0 < n_nope; b0 += 64) {
        int b1 = b0 + 64 < n_nope ? b0 + 64 : n_nope;
        float amax = 0.0f;
        for (int j = b0; j < b1; j++) {
            float a = fabsf(row[j]);
            if (a > amax) amax = a;
        }
        int e = orc_fp8_scale_exp(amax);
        for (int j = b0; j < b1; j++) {
            double y = ldexp((double)row[j], -e);       /* exact */
            row[j] = (float)ldexp((double)orc_e4m3_rne((float)y), e);
        }
    }
}

/* ---------------------------------------------------------------------------
 * Indexer QAT round trip.  "Metal グラフと圧縮 KV の実装を読む" §9: the indexer row
 * (and, the page says, the indexer query) goes through a Hadamard transform of
 * order 128 and an FP4 activation-quantisation round trip instead of the FP8
 * one, so that the top-k selection follows the model's graph.
 * READING R-16: the orthonormal Sylvester Hadamard transform y = H x / sqrt(n),
 * H[i][j] = (-1)^popcount(i & j), evaluated as the fast Walsh-Hadamard
 * transform in binary32 (stages h = 1, 2, 4, ..., n/2; stage h replaces each
 * pair (x[j], x[j + h]) with j & h == 0 by (x[j] + x[j + h], x[j] - x[j + h]))
 * followed by one binary32 multiply by binary32(1 / sqrt(n)).  The evaluation
 * order is part of the reading because the FP4 rounding that follows decides
 * codes from these binary32 values.
 * READING R-17: OCP E2M1 (values 0, 0.5, 1, 1.5, 2, 3, 4, 6), round to nearest
 * with ties to the even code, saturating at +-6; one power-of-two scale per
 * block of 32 consecutive values, the smallest 2^e with amax <= 6 * 2^e (e = 0
 * for an all-zero block); value = e2m1(x / 2^e) * 2^e.
 * ------------------------------------------------------------------------- */
void orc_hadamard(float *x, int n) {
    for (int h = 1; h < n; h <<= 1) {
        for (int j = 0; j < n; j++) {
            if (j & h) continue;
            float a = x[j], b = x[j + h];
            x[j] = a + b;
            x[j + h] = a - b;
        }
    }
    const float c = (float)(1.0 / sqrt((double)n));
    for (int j = 0; j < n; j++) x[j] = x[j] * c;
}

/* Value of the non-negative E2M1 code c (0..7): exponent bits c >> 1 (bias 1),
 * mantissa bit c & 1; code 1 is the subnormal 0.5. */
static double e2m1_value(int c) {
    int E = c >> 1, m = c & 1;
    if (E == 0) return 0.5 * (double)m;
    return ldexp(1.0 + 0.5 * (double)m, E - 1);
}

/* Nearest E2M1 value to y, ties to the even code, saturating to +-6. */
float orc_e2m1_rne(float y) {
    double a = fabs((double)y);
    double r;
    if (a >= 6.0) {
        r = 6.0;
    } else {
        int lo = 0;                                     /* largest code with value <= a */
        for (int c = 0; c <= 7; c++)
            if (e2m1_value(c) <= a) lo = c;
        double vlo = e2m1_value(lo), vhi = e2m1_value(lo + 1);
        double dlo = a - vlo, dhi = vhi - a;
        if (dlo < dhi) r = vlo;
        else if (dhi < dlo) r = vhi;
        else r = ((lo & 1) == 0) ? vlo : vhi;
    }
    return (float)(signbit(y) ? -r : r);
}

/* Smallest integer e with amax <= 6 * 2^e; 0 when amax == 0. */
int orc_fp4_scale_exp(float amax) {
    if (!(amax > 0.0f)) return 0;
    int e = 0;
    while ((double)amax > ldexp(6.0, e)) e++;
    while ((double)amax <= ldexp(6.0, e - 1)) e--;
    return e;
}

void orc_fp4_roundtrip(float *x, int n) {
    for (int b0 = 0; b0 < n; b0 += 32) {
        int b1 = b0 + 32 < n ? b0 + 32 : n;
        float amax = 0.0f;
        for (int j = b0; j < b1; j++) {
            float a = fabsf(x[j]);
            if (a > amax) amax = a;
        }
        int e = orc_fp4_scale_exp(amax);
        for (int j = b0; j < b1; j++) {
            double y = ldexp((double)x[j], -e);         /* exact */
            x[j] = (float)ldexp((double)orc_e2m1_rne((float)y), e);
        }
    }
}

/* The round trip of one indexer row or query head: Hadamard, then FP4. */
void orc_indexer_qat(float *x, int n) {
    orc_hadamard(x, n);
    orc_fp4_roundtrip(x, n);
}

/* ---------------------------------------------------------------------------
 * A6. Tail RoPE.  [P2] §8, rope_tail_ext_inplace: only the last n_rot dims of
 * a head rotate (n_nope = head_dim - n_rot untouched).
 * READING (C-5): pairs (2i, 2i+1) of the tail; angle = float(p * inv_freq[i])
 * as one float multiply; rotation (x0 + i x1) e^{i angle}, in double.
 * ------------------------------------------------------------------------- */
void orc_rope_tail(double *x, int head_dim, int n_rot, uint64_t p, const float *inv_freq) {
    double *tail = x + (head_dim - n_rot);
    for (int i = 0; i < n_rot / 2; i++) {
        float ang = (float)p * inv_freq[i];
        double c = cos((double)ang), s = sin((double)ang);
        double x0 = tail[2 * i], x1 = tail[2 * i + 1];
        tail[2 * i] = x0 * c - x1 * s;
        tail[2 * i + 1] = x0 * s + x1 * c;
    }
}

/* A5. RMSNorm over the whole row: y = x / sqrt(mean(x^2) + eps) * gain
 * ([P2] §4 lists the normalisation step; READING C-4: eps from the config,
 * gain = the lane's norm tensor, ones when absent). */
void orc_rmsnorm(double *x, int n, const float *gain, float eps) {
    double ss = 0.0;
    for (int j = 0; j < n; j++) ss += x[j] * x[j];
    double inv = 1.0 / sqrt(ss / (double)n + (double)eps);
    for (int j = 0; j < n; j++) x[j] = x[j] * inv * (gain ? (double)gain[j] : 1.0);
}

/* ---------------------------------------------------------------------------
 * A2-A8. Compressor, one token of one lane.  [P2] §4 compressor_decode_one:
 * store kv and score+APE into the frontier; at a ratio boundary softmax-pool,
 * RMSNorm, tail RoPE, FP8 (attention lane) and append; [P2] §5: ratio-4 lanes
 * keep 8 rows (two 4-row halves), write row 4 + pos%4, pool at (pos+1)%4 == 0,
 * then move rows 4..7 to rows 0..3.
 *
 * READINGS: C-1 APE row = pos % ratio; C-3 the ratio-4 pool takes, per output
 * column j, rows 0..3 at column j and rows 4..7 at column Dl + j (8 candidates);
 * C-5 a compressed row c carries position c * ratio.
 * lane_is_attn selects the FP8 round trip; the indexer lane's QAT round trip
 * is the identity here (C-7).
 * ------------------------------------------------------------------------- */
void orc_compress_token(const orc_cfg *cfg, int lane_is_attn, const float *ape, const float *gain,
                        const float *inv_freq, orc_lane_s st, const float *kv, const float *score,
                        uint64_t pos) {
    const int r = cfg->ratio;
    const int Dl = lane_is_attn ? cfg->head_dim : cfg->idx_head_dim;
    const int coff = (r == 4) ? 2 : 1;
    const int W = coff * Dl;
    const int row = (r == 4) ? 4 + (int)(pos % 4) : (int)(pos % (uint64_t)r);
    const int in_win = (int)(pos % (uint64_t)r);

    /* store (kernel_dsv4_compressor_store_one): state_kv = kv, state_score = score + ape */
    for (int j = 0; j < W; j++) {
        st.state_kv[(size_t)row * W + j] = kv[j];
        st.state_score[(size_t)row * W + j] = score[j] + ape[(size_t)in_win * W + j];
    }
    if ((pos + 1) % (uint64_t)r != 0) return;

    /* pool (compressor_pool_decode_state): per column, max, exp weights, weighted mean */
    const uint64_t c = pos / (uint64_t)r;
    double *x = (double *)malloc(sizeof(double) * (size_t)Dl);
    const int n_cand = (r == 4) ? 8 : r;
    for (int j = 0; j < Dl; j++) {
        double m = -INFINITY;
        for (int q = 0; q < n_cand; q++) {
            int col = (r == 4 && q >= 4) ? Dl + j : j;
            double s = (double)st.state_score[(size_t)q * W + col];
            if (s > m) m = s;
        }
        double denom = 0.0, sum = 0.0;
        for (int q = 0; q < n_cand; q++) {
            int col = (r == 4 && q >= 4) ? Dl + j : j;
            double w = exp((double)st.state_score[(size_t)q * W + col] - m);
            denom += w;
            sum += w * (double)st.state_kv[(size_t)q * W + col];
        }
        x[j] = denom > 0.0 ? sum / denom : 0.0;
    }
    orc_rmsnorm(x, Dl, gain, cfg->rms_eps);
    orc_rope_tail(x, Dl, cfg->n_rot, c * (uint64_t)r, inv_freq);
    float *out = st.comp + (size_t)c * Dl;
    for (int j = 0; j < Dl; j++) out[j] = (float)x[j];
    if (st.prequant) memcpy(st.prequant + (size_t)c * Dl, out, sizeof(float) * (size_t)Dl);
    if (lane_is_attn) orc_fp8_roundtrip(out, Dl - cfg->n_rot);
    else if (cfg->idx_qat) orc_indexer_qat(out, Dl);
    free(x);

    /* ratio-4 shift (kernel_dsv4_ratio4_shift_f32): rows 4..7 -> rows 0..3 */
    if (r == 4) {
        for (size_t g = 0; g < (size_t)4 * W; g++) {
            st.state_kv[g] = st.state_kv[(size_t)4 * W + g];
            st.state_score[g] = st.state_score[(size_t)4 * W + g];
        }
    }
}

/* READING (C-2): a fresh frontier holds kv = 0 and score = -inf, so rows no
 * token has written carry no weight in the pool. */
void orc_state_init_lane(const orc_cfg *cfg, int lane_is_attn, orc_lane_s st) {
    const int r = cfg->ratio;
    const int Dl = lane_is_attn ? cfg->head_dim : cfg->idx_head_dim;
    const int coff = (r == 4) ? 2 : 1;
    size_t n = (size_t)coff * r * coff * Dl;
    for (size_t i = 0; i < n; i++) {
        st.state_kv[i] = 0.0f;
        st.state_score[i] = -INFINITY;
    }
}

/* A1-A8 over T tokens at absolute positions pos0 .. pos0+T-1 of one sequence.
 * [P2] §3: chunking keeps absolute-position boundaries, so this literal token
 * loop is the definition for any chunk split.  kvbuf is caller scratch of
 * T * 2 * coff * max(D, d) floats. */
void orc_compress(const orc_cfg *cfg, const orc_lane_w *aw, const orc_lane_w *iw,
                  orc_lane_s as, orc_lane_s is, const void *hidden, int T, uint64_t pos0,
                  float *kvbuf) {
    const int r = cfg->ratio;
    if (r == 0 || T <= 0) return;
    const int coff = (r == 4) ? 2 : 1;
    float *inv_freq = (float *)malloc(sizeof(float) * (size_t)(cfg->n_rot / 2 + 1));
    orc_inv_freq(cfg->rope_base, cfg->n_rot, inv_freq);
    for (int lane = 0; lane < (r == 4 ? 2 : 1); lane++) {
        const orc_lane_w *w = lane == 0 ? aw : iw;
        orc_lane_s st = lane == 0 ? as : is;
        const int Dl = lane == 0 ? cfg->head_dim : cfg->idx_head_dim;
        const int W = coff * Dl;
        float *kv = kvbuf, *sc = kvbuf + (size_t)T * W;
        orc_project(w->wkv, hidden, cfg->bf16, T, cfg->d_model, W, kv);
        orc_project(w->wgate, hidden, cfg->bf16, T, cfg->d_model, W, sc);
        for (int t = 0; t < T; t++)
            orc_compress_token(cfg, lane == 0, w->ape, w->norm, inv_freq, st,
                               kv + (size_t)t * W, sc + (size_t)t * W, pos0 + (uint64_t)t);
    }
    free(inv_freq);
}

/* ---------------------------------------------------------------------------
 * A9-A10. Indexer score and top-k ([P2] §6 and §7).
 * READING (C-8): score = dot(q_idx, index_comp_kv row) as the float chain
 * s = fmaf(q[i], row[i], s), i = 0 .. d-1.
 * READING (C-9): a query at position t sees rows c < (t+1)/4; it keeps the k
 * largest scores (ties: lower index first, -0 == +0), listed by ascending
 * index and padded with -1 (the attention loop stops at the first index
 * >= visible, so the list is ascending).
 * ------------------------------------------------------------------------- */
float orc_index_score(const float *q, const float *row, int d) {
    float s = 0.0f;
    for (int i = 0; i < d; i++) s = fmaf(q[i], row[i], s);
    return s;
}

typedef struct { float s; int32_t i; } orc_si;

static int cmp_score_desc(const void *a, const void *b) {
    const orc_si *x = (const orc_si *)a, *y = (const orc_si *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->i > y->i) - (x->i < y->i);
}

static int cmp_int_asc(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

void orc_topk(const float *scores, int visible, int k, int32_t *out) {
    orc_si *v = (orc_si *)malloc(sizeof(orc_si) * (size_t)(visible > 0 ? visible : 1));
    for (int c = 0; c < visible; c++) { v[c].s = scores[c]; v[c].i = c; }
    qsort(v, (size_t)visible, sizeof(orc_si), cmp_score_desc);
    int n = visible < k ? visible : k;
    for (int i = 0; i < n; i++) out[i] = v[i].i;
    qsort(out, (size_t)n, sizeof(int32_t), cmp_int_asc);
    for (int i = n; i < k; i++) out[i] = -1;
    free(v);
}

/* n queries of one sequence at positions pos[j]; rows = that sequence's
 * index_comp_kv.  scores_out (may be NULL) gets [n][score_stride]. */
void orc_indexer_topk(const orc_cfg *cfg, const float *idx_comp, const float *q_idx,
                      const uint64_t *pos, int n, int32_t *topk, float *scores_out,
                      int64_t score_stride) {
    const int d = cfg->idx_head_dim, k = cfg->top_k;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < n; j++) {
        int visible = (int)((pos[j] + 1) / 4);
        float *s = (float *)malloc(sizeof(float) * (size_t)(visible > 0 ? visible : 1));
        for (int c = 0; c < visible; c++)
            s[c] = orc_index_score(q_idx + (size_t)j * d, idx_comp + (size_t)c * d, d);
        orc_topk(s, visible, k, topk + (size_t)j * k);
        if (scores_out)
            for (int c = 0; c < visible; c++) scores_out[(size_t)j * score_stride + c] = s[c];
        free(s);
    }
}

/* ---------------------------------------------------------------------------
 * Multi-head indexer score ("Metal グラフと圧縮 KV の実装を読む" §6: 64 indexer heads
 * of width 128 score each compressed row, four heads at a time).
 * READING R-15: the heads' dot products with the row, each the in-order binary32
 * fmaf chain of R-8, are clamped at zero (ReLU) and summed with per-query head
 * weights w as one more in-order fmaf chain over the heads:
 *   s = 0; for j = 0 .. heads-1: s = fmaf(w[j], max(dot_j, 0), s).
 * q holds the heads' query vectors after the round trip, [heads][d].
 * ------------------------------------------------------------------------- */
float orc_index_score_heads(const float *q, const float *w, const float *row, int d, int heads) {
    float s = 0.0f;
    for (int j = 0; j < heads; j++) {
        float dj = orc_index_score(q + (size_t)j * d, row, d);
        s = fmaf(w[j], dj > 0.0f ? dj : 0.0f, s);
    }
    return s;
}

/* n queries of one sequence at positions pos[j]: q_raw [n][heads][d] (before the
 * round trip; it is applied here when cfg->idx_qat), w [n][heads]; rows = that
 * sequence's index_comp_kv; top-k as orc_indexer_topk. */
void orc_indexer_topk_heads(const orc_cfg *cfg, const float *idx_comp, const float *q_raw, const float *w,
                            const uint64_t *pos, int n, int32_t *topk, float *scores_out, int64_t score_stride) {
    const int d = cfg->idx_head_dim, k = cfg->top_k, H = cfg->idx_heads;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < n; j++) {
        float *q = (float *)malloc(sizeof(float) * (size_t)H * d);
        memcpy(q, q_raw + (size_t)j * H * d, sizeof(float) * (size_t)H * d);
        if (cfg->idx_qat)
            for (int h = 0; h < H; h++) orc_indexer_qat(q + (size_t)h * d, d);
        int visible = (int)((pos[j] + 1) / 4);
        float *s = (float *)malloc(sizeof(float) * (size_t)(visible > 0 ? visible : 1));
        for (int c = 0; c < visible; c++)
            s[c] = orc_index_score_heads(q, w + (size_t)j * H, idx_comp + (size_t)c * d, d, H);
        orc_topk(s, visible, k, topk + (size_t)j * k);
        if (scores_out)
            for (int c = 0; c < visible; c++) scores_out[(size_t)j * score_stride + c] = s[c];
        free(s);
        free(q);
    }
}

/* ---------------------------------------------------------------------------
 * A11. Sparse SWA attention ([P2] §7, kernel_dsv4_indexed_mixed_attention):
 * per query position t and head h, one softmax over the raw rows at positions
 * [max(0, t+1-swa), t] and the compressed rows; ratio 4: the indexer's list,
 * skipping idx < 0 and stopping at idx >= visible; ratio 128: every visible
 * row (READING); ratio 0: raw rows only.
 * READING (C-10/C-11): K = V = the stored row, logit = (q . x) * attn_scale,
 * no sink, no de-duplication.  Raw rows of positions before pos0 come from
 * the ring (slot p % swa), the rest from raw_new.
 * ------------------------------------------------------------------------- */
void orc_attention(const orc_cfg *cfg, const float *ring, const float *comp, const float *q,
                   const float *raw_new, const int32_t *topk, uint64_t pos0, int T, float *out) {
    const int D = cfg->head_dim, H = cfg->n_heads, S = cfg->swa, r = cfg->ratio;
    const int k = cfg->top_k;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int jt = 0; jt < T; jt++) {
        const uint64_t t = pos0 + (uint64_t)jt;
        const uint64_t first = (t + 1 > (uint64_t)S) ? t + 1 - (uint64_t)S : 0;
        int cap = (int)(t - first + 1) + (r == 4 ? k : (r == 128 ? (int)((t + 1) / 128) : 0));
        const float **rows = (const float **)malloc(sizeof(float *) * (size_t)cap);
        int n = 0;
        for (uint64_t p = first; p <= t; p++)
            rows[n++] = (p >= pos0) ? raw_new + (size_t)(p - pos0) * D : ring + (size_t)(p % (uint64_t)S) * D;
        if (r == 4) {
            const uint64_t visible = (t + 1) / 4;
            for (int i = 0; i < k; i++) {
                int32_t idx = topk[(size_t)jt * k + i];
                if (idx < 0) continue;
                if ((uint64_t)idx >= visible) break;
                rows[n++] = comp + (size_t)idx * D;
            }
        } else if (r == 128) {
            const uint64_t visible = (t + 1) / 128;
            for (uint64_t c = 0; c < visible; c++) rows[n++] = comp + (size_t)c * D;
        }
        double *logit = (double *)malloc(sizeof(double) * (size_t)n);
        double *acc = (double *)malloc(sizeof(double) * (size_t)D);
        for (int h = 0; h < H; h++) {
            const float *qh = q + ((size_t)jt * H + h) * D;
            double m = -INFINITY;
            for (int i = 0; i < n; i++) {
                double s = 0.0;
                for (int dd = 0; dd < D; dd++) s += (double)qh[dd] * (double)rows[i][dd];
                logit[i] = s * (double)cfg->attn_scale;
                if (logit[i] > m) m = logit[i];
            }
            double denom = 0.0;
            for (int dd = 0; dd < D; dd++) acc[dd] = 0.0;
            for (int i = 0; i < n; i++) {
                double w = exp(logit[i] - m);
                denom += w;
                for (int dd = 0; dd < D; dd++) acc[dd] += w * (double)rows[i][dd];
            }
            float *o = out + ((size_t)jt * H + h) * D;
            for (int dd = 0; dd < D; dd++) o[dd] = (float)(acc[dd] / denom);
        }
        free(acc);
        free(logit);
        free(rows);
    }
}

/* A12. Ring commit: after the attention of positions pos0 .. pos0+T-1, slot
 * p % swa holds raw row p for the last min(T, swa) of them ([P2] §2 raw_kv is
 * a sliding window of the most recent rows). */
void orc_ring_commit(const orc_cfg *cfg, float *ring, const float *raw_new, uint64_t pos0, int T) {
    const int D = cfg->head_dim, S = cfg->swa;
    uint64_t end = pos0 + (uint64_t)T;
    uint64_t start = (end > (uint64_t)S && end - (uint64_t)S > pos0) ? end - (uint64_t)S : pos0;
    for (uint64_t p = start; p < end; p++)
        memcpy(ring + (size_t)(p % (uint64_t)S) * D, raw_new + (size_t)(p - pos0) * D, sizeof(float) * (size_t)D);
}

/* ---------------------------------------------------------------------------
 * A15. Checkpoint gather ([P1] §5 payload body order, §6 raw ring in logical
 * position order, §7 frontier tensors), for one sequence after pos tokens:
 *   raw rows of positions pos-n_live .. pos-1 (n_live = min(pos, swa)),
 *   attn_comp_kv rows 0 .. pos/ratio - 1, attn_state_kv, attn_state_score,
 *   and on ratio-4 layers index_comp_kv rows 0 .. pos/4 - 1, index_state_kv,
 *   index_state_score.
 * ------------------------------------------------------------------------- */
int64_t orc_checkpoint_floats(const orc_cfg *cfg, uint64_t pos) {
    const int D = cfg->head_dim, d = cfg->idx_head_dim, r = cfg->ratio, S = cfg->swa;
    int64_t n_live = (int64_t)(pos < (uint64_t)S ? pos : (uint64_t)S);
    int64_t total = n_live * D;
    if (r != 0) {
        const int coff = (r == 4) ? 2 : 1;
        total += (int64_t)(pos / (uint64_t)r) * D + 2 * (int64_t)(coff * r) * (coff * D);
    }
    if (r == 4) total += (int64_t)(pos / 4) * d + 2 * (int64_t)8 * (2 * d);
    return total;
}

int64_t orc_checkpoint_gather(const orc_cfg *cfg, const float *ring, orc_lane_s as, orc_lane_s is,
                              uint64_t pos, float *dst) {
    const int D = cfg->head_dim, d = cfg->idx_head_dim, r = cfg->ratio, S = cfg->swa;
    int64_t o = 0;
    uint64_t n_live = pos < (uint64_t)S ? pos : (uint64_t)S;
    for (uint64_t p = pos - n_live; p < pos; p++) {
        memcpy(dst + o, ring + (size_t)(p % (uint64_t)S) * D, sizeof(float) * (size_t)D);
        o += D;
    }
    if (r != 0) {
        const int coff = (r == 4) ? 2 : 1;
        size_t nc = (size_t)(pos / (uint64_t)r) * D, nf = (size_t)(coff * r) * (coff * D);
        memcpy(dst + o, as.comp, sizeof(float) * nc); o += (int64_t)nc;
        memcpy(dst + o, as.state_kv, sizeof(float) * nf); o += (int64_t)nf;
        memcpy(dst + o, as.state_score, sizeof(float) * nf); o += (int64_t)nf;
    }
    if (r == 4) {
        size_t nc = (size_t)(pos / 4) * d, nf = (size_t)8 * (2 * d);
        memcpy(dst + o, is.comp, sizeof(float) * nc); o += (int64_t)nc;
        memcpy(dst + o, is.state_kv, sizeof(float) * nf); o += (int64_t)nf;
        memcpy(dst + o, is.state_score, sizeof(float) * nf); o += (int64_t)nf;
    }
    return o;
}

/* Restore ("【#4】ds4.c を読み解く" §6-§7): the same body read back into the
 * state -- raw rows in logical order to slot p % swa, then the compressed rows
 * and frontier tensors of each lane.  Returns the number of floats read. */
int64_t orc_checkpoint_scatter(const orc_cfg *cfg, float *ring, orc_lane_s as, orc_lane_s is, uint64_t pos,
                               const float *src) {
    const int D = cfg->head_dim, d = cfg->idx_head_dim, r = cfg->ratio, S = cfg->swa;
    int64_t o = 0;
    uint64_t n_live = pos < (uint64_t)S ? pos : (uint64_t)S;
    for (uint64_t p = pos - n_live; p < pos; p++) {
        memcpy(ring + (size_t)(p % (uint64_t)S) * D, src + o, sizeof(float) * (size_t)D);
        o += D;
    }
    if (r != 0) {
        const int coff = (r == 4) ? 2 : 1;
        size_t nc = (size_t)(pos / (uint64_t)r) * D, nf = (size_t)(coff * r) * (coff * D);
        memcpy(as.comp, src + o, sizeof(float) * nc); o += (int64_t)nc;
        memcpy(as.state_kv, src + o, sizeof(float) * nf); o += (int64_t)nf;
        memcpy(as.state_score, src + o, sizeof(float) * nf); o += (int64_t)nf;
    }
    if (r == 4) {
        size_t nc = (size_t)(pos / 4) * d, nf = (size_t)8 * (2 * d);
        memcpy(is.comp, src + o, sizeof(float) * nc); o += (int64_t)nc;
        memcpy(is.state_kv, src + o, sizeof(float) * nf); o += (int64_t)nf;
        memcpy(is.state_score, src + o, sizeof(float) * nf); o += (int64_t)nf;
    }
    return o;
}

/* ---------------------------------------------------------------------------
 * DSV4 session payload of a layer stack ("【#4】ds4.c を読み解く" §5).
 * Header: 13 u32 fields in the page's table order -- magic "DSV4" (the bytes
 * 'D','S','V','4' read as a little-endian u32), payload version 2, then the 11
 * fields of `fields` (saved context size, prefill chunk size, raw KV ring
 * capacity, raw sliding-window length, compressed KV capacity, checkpoint
 * token count, layer count, raw/head KV dimension, indexer head dimension,
 * vocabulary size, live raw rows).  Body, in the page's order: u32 token ids
 * [token_count], f32 logits [vocab_size], u32 compressed attention row counts
 * [layer_count], u32 ratio-4 indexer row counts [layer_count], then per layer
 * the raw SWA rows (logical order, §6), the attention compressed rows, the
 * compressor frontier (§7), the indexer compressed rows and the indexer
 * frontier (ratio-4 layers) -- READING: the page's list is written once per
 * layer, layer by layer, which is the single-layer checkpoint body above.
 * The checkpoint position is the token count.  Returns the bytes written.
 * ------------------------------------------------------------------------- */
static void put_u32(uint8_t *dst, int64_t *o, uint32_t v) {
    dst[*o + 0] = (uint8_t)(v & 0xFFu);
    dst[*o + 1] = (uint8_t)((v >> 8) & 0xFFu);
    dst[*o + 2] = (uint8_t)((v >> 16) & 0xFFu);
    dst[*o + 3] = (uint8_t)((v >> 24) & 0xFFu);
    *o += 4;
}

static uint32_t get_u32(const uint8_t *src, int64_t *o) {
    uint32_t v = (uint32_t)src[*o] | ((uint32_t)src[*o + 1] << 8) | ((uint32_t)src[*o + 2] << 16) |
                 ((uint32_t)src[*o + 3] << 24);
    *o += 4;
    return v;
}

static void put_f32(uint8_t *dst, int64_t *o, float f) {
    uint32_t v;
    memcpy(&v, &f, sizeof v);
    put_u32(dst, o, v);
}

static float get_f32(const uint8_t *src, int64_t *o) {
    uint32_t v = get_u32(src, o);
    float f;
    memcpy(&f, &v, sizeof f);
    return f;
}

int64_t orc_payload_write(const uint32_t *fields, int n_layers, const orc_cfg *cfgs, float *const *rings,
                          const orc_lane_s *attn, const orc_lane_s *idx, const uint32_t *tokens,
                          const float *logits, uint8_t *dst) {
    const uint32_t magic = (uint32_t)'D' | ((uint32_t)'S' << 8) | ((uint32_t)'V' << 16) | ((uint32_t)'4' << 24);
    const uint32_t token_count = fields[5], vocab = fields[9];
    const uint64_t pos = token_count;
    int64_t o = 0;
    put_u32(dst, &o, magic);
    put_u32(dst, &o, 2u);
    for (int i = 0; i < 11; i++) put_u32(dst, &o, fields[i]);
    for (uint32_t i = 0; i < token_count; i++) put_u32(dst, &o, tokens[i]);
    for (uint32_t i = 0; i < vocab; i++) put_f32(dst, &o, logits[i]);
    for (int l = 0; l < n_layers; l++) put_u32(dst, &o, cfgs[l].ratio ? (uint32_t)(pos / (uint64_t)cfgs[l].ratio) : 0u);
    for (int l = 0; l < n_layers; l++) put_u32(dst, &o, cfgs[l].ratio == 4 ? (uint32_t)(pos / 4) : 0u);
    for (int l = 0; l < n_layers; l++) {
        int64_t n = orc_checkpoint_floats(&cfgs[l], pos);
        float *body = (float *)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
        orc_checkpoint_gather(&cfgs[l], rings[l], attn[l], idx[l], pos, body);
        for (int64_t i = 0; i < n; i++) put_f32(dst, &o, body[i]);
        free(body);
    }
    return o;
}

/* The inverse: the 11 fields after magic and version into fields_out, the
 * token ids and logits out, each layer's body scattered into its state.
 * Returns the bytes read, or -1 when the magic or the version differ. */
int64_t orc_payload_read(const uint8_t *src, int n_layers, const orc_cfg *cfgs, float *const *rings,
                         const orc_lane_s *attn, const orc_lane_s *idx, uint32_t *fields_out,
                         uint32_t *tokens_out, float *logits_out) {
    const uint32_t magic = (uint32_t)'D' | ((uint32_t)'S' << 8) | ((uint32_t)'V' << 16) | ((uint32_t)'4' << 24);
    int64_t o = 0;
    if (get_u32(src, &o) != magic) return -1;
    if (get_u32(src, &o) != 2u) return -1;
    for (int i = 0; i < 11; i++) fields_out[i] = get_u32(src, &o);
    const uint32_t token_count = fields_out[5], vocab = fields_out[9];
    const uint64_t pos = token_count;
    for (uint32_t i = 0; i < token_count; i++) tokens_out[i] = get_u32(src, &o);
    for (uint32_t i = 0; i < vocab; i++) logits_out[i] = get_f32(src, &o);
    o += 8 * (int64_t)n_layers;                     /* the two count arrays follow from pos */
    for (int l = 0; l < n_layers; l++) {
        int64_t n = orc_checkpoint_floats(&cfgs[l], pos);
        float *body = (float *)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
        for (int64_t i = 0; i < n; i++) body[i] = get_f32(src, &o);
        orc_checkpoint_scatter(&cfgs[l], rings[l], attn[l], idx[l], pos, body);
        free(body);
    }
    return o;
}
