/*
 * pqe_oracle.c -- CPU oracle of the paged, quantized MoE expert layer.
 *
 * TEST INFRASTRUCTURE. This is a plain, slow, deliberately unoptimised CPU
 * statement of what the expert layer computes. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the product library
 * never does. It shares no source, header, table or constant generator with
 * the CUDA library: every format below is re-derived here from its definition.
 *
 * Sources (web pages; section given after the page title):
 *   [EP]  vllm-expert-pager article (rand.pepabo.com, 2026-09-18): sections
 *         はじめに, プラグインの仕組み (エキスパート重みの階層ページング,
 *         重みの圧縮), 評価 (表1-表4).
 *   [PW]  "PagedWeight Efficient MoE LLM Serving" commentary (spectral-agent.com):
 *         技術的に面白い点.
 *   [MG]  MoE-Gen summary (aibr.jp): 3.中核となる技術的要素 (module-based batching).
 *   [OCP-FP8] OCP 8-bit floating point specification (E4M3, bias 7).
 *   [OCP-MX]  OCP Microscaling formats specification v1.0 (E2M1, E8M0, k=32).
 *
 * Where the pages leave a step open, the reading taken is stated at the
 * function. Floating point is fp64 except the router logits, which the layer
 * defines in fp32 with a fixed reduction order so that the top-k decision is
 * reproducible (see orc_router_logits).
 *
 * Parity-unpinned: none of the functions below is without a pin; the pins
 * live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 [OCP-FP8]: sign 1, exponent 4 (bias 7), mantissa 3; no infinity;  */
/* S.1111.111 is NaN; largest finite 448 = 1.75 * 2^8; subnormal step 2^-9.   */
/* ------------------------------------------------------------------------ */

EXPORT double orc_e4m3_value(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* the 256 decoded values, filled once from orc_e4m3_value (a cache, same values) */
static double e4m3_table[256];
static int e4m3_table_ready = 0;

static double e4m3_cached(uint8_t b)
{
    if (!e4m3_table_ready) {
#pragma omp critical(orc_e4m3_table)
        {
            if (!e4m3_table_ready) {
                for (int i = 0; i < 256; ++i) e4m3_table[i] = orc_e4m3_value((uint8_t)i);
                e4m3_table_ready = 1;
            }
        }
    }
    return e4m3_table[b];
}

/* Codes 0x00..0x7E hold the non-negative finite values in increasing order.
 * Round |v| to the nearest of them; on an exact tie take the even code (its
 * mantissa LSB is 0: round half to even); beyond 448 saturate to 448. */
static uint8_t e4m3_magnitude_code(double a)
{
    int lo = 0, hi = 0x7E;
    if (a >= e4m3_cached(0x7E)) return 0x7E;
    /* largest code with value <= a */
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (e4m3_cached((uint8_t)mid) <= a) lo = mid; else hi = mid - 1;
    }
    {
        double below = e4m3_cached((uint8_t)lo);
        double above = e4m3_cached((uint8_t)(lo + 1));
        double dlo = a - below, dhi = above - a;
        if (dlo < dhi) return (uint8_t)lo;
        if (dhi < dlo) return (uint8_t)(lo + 1);
        return (lo & 1) ? (uint8_t)(lo + 1) : (uint8_t)lo;
    }
}

EXPORT uint8_t orc_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    return sign | e4m3_magnitude_code(fabs((double)v));
}

/* Per-row FP8 weight quantisation: E4M3 codes with one fp32 scale per row.
 * Reading: s = amax/448 in fp32 (s = 1 for an all-zero
 * row); code = RNE_e4m3(w / s) with the quotient taken in fp32; dequant is
 * e4m3(code) * s. */
EXPORT void orc_quant_e4m3_rows(const float *w, int rows, int cols, uint8_t *q, float *scale)
{
    for (int r = 0; r < rows; ++r) {
        const float *wr = w + (size_t)r * cols;
        float amax = 0.0f, s;
        for (int c = 0; c < cols; ++c) {
            float a = fabsf(wr[c]);
            if (a > amax) amax = a;
        }
        s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
        scale[r] = s;
        for (int c = 0; c < cols; ++c) {
            volatile float quotient = wr[c] / s; /* fp32 quotient, as specified */
            q[(size_t)r * cols + c] = orc_e4m3_encode(quotient);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* MXFP4 [OCP-MX]: E2M1 elements {0, .5, 1, 1.5, 2, 3, 4, 6} with sign, and   */
/* one E8M0 scale 2^(byte-127) per block of 32 elements along a row.         */
/* ------------------------------------------------------------------------ */

EXPORT double orc_e2m1_value(uint8_t nib)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[nib & 7];
    return (nib & 8) ? -v : v;
}

EXPORT double orc_e8m0_value(uint8_t b)
{
    return ldexp(1.0, (int)b - 127); /* 0xFF (NaN) is never produced here */
}

static uint8_t e2m1_magnitude_code(double a)
{
    int lo = 0;
    if (a >= 6.0) return 7;
    while (lo < 7 && orc_e2m1_value((uint8_t)(lo + 1)) <= a) ++lo;
    {
        double dlo = a - orc_e2m1_value((uint8_t)lo);
        double dhi = orc_e2m1_value((uint8_t)(lo + 1)) - a;
        if (dlo < dhi) return (uint8_t)lo;
        if (dhi < dlo) return (uint8_t)(lo + 1);
        return (lo & 1) ? (uint8_t)(lo + 1) : (uint8_t)lo;
    }
}

EXPORT uint8_t orc_e2m1_encode(float v)
{
    return (signbit(v) ? 8 : 0) | e2m1_magnitude_code(fabs((double)v));
}

/* 4-bit page of an FP8 expert matrix [PW: lower bit-width pages]. The master
 * copy stays FP8 ([EP] 位置づけ keeps the vendor FP8), so the 4-bit copy is
 * derived from the dequantised FP8 values v = fp32(e4m3(q)) * s (fp32 product).
 * Per block of 32 along the row: amax; E = floor(log2 amax); shared scale
 * X = 2^(E - 2) stored as E8M0 byte E - 2 + 127 (clamped to [0, 254]); an
 * all-zero block stores byte 0. Elements: RNE_e2m1(v / X) saturating to 6,
 * quotient in fp32. Output nibbles: two per byte, low nibble = even column. */
EXPORT void orc_quant_mxfp4_rows(const uint8_t *q8, const float *s8, int rows, int cols,
                                 uint8_t *q4, uint8_t *e8m0)
{
    int nblk = cols / 32;
    memset(q4, 0, (size_t)rows * cols / 2);
    for (int r = 0; r < rows; ++r) {
        for (int b = 0; b < nblk; ++b) {
            float v[32], amax = 0.0f;
            uint8_t sb;
            for (int i = 0; i < 32; ++i) {
                volatile float prod = (float)orc_e4m3_value(q8[(size_t)r * cols + b * 32 + i]) * s8[r];
                v[i] = prod;
                if (fabsf(v[i]) > amax) amax = fabsf(v[i]);
            }
            if (amax == 0.0f) {
                sb = 0;
            } else {
                int ex;
                int E;
                frexp((double)amax, &ex); /* amax = f * 2^ex, f in [0.5, 1) */
                E = ex - 1;
                E = E - 2 + 127;
                sb = (uint8_t)(E < 0 ? 0 : (E > 254 ? 254 : E));
            }
            e8m0[(size_t)r * nblk + b] = sb;
            for (int i = 0; i < 32; ++i) {
                float X = (float)orc_e8m0_value(sb);
                volatile float quotient = v[i] / X;
                uint8_t code = orc_e2m1_encode(quotient);
                size_t idx = (size_t)r * cols + b * 32 + i;
                q4[idx / 2] |= (idx & 1) ? (uint8_t)(code << 4) : code;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Router [EP 階層ページング, MG §3]: the pages only say each token picks a   */
/* few experts. Reading (plain MoE top-k, as in the Qwen FP8 MoE models the   */
/* [EP] plugin targets): logits -> top-k by logit (ties to the lower id,      */
/* ordered by logit desc then id asc) -> softmax over the k picked.          */
/* ------------------------------------------------------------------------ */

/* logits[t,e] = sum_h x[t,h] * W_r[e,h] in fp32. The sum order is part of the
 * definition so that the top-k decision is reproducible bit for bit: 32
 * partial sums p_l (l = 0..31), p_l accumulating h = l, l+32, l+64, ... in
 * ascending h with a correctly rounded fused multiply-add from 0; then a
 * pairwise tree: p_l += p_{l+16} (l < 16), p_l += p_{l+8} (l < 8), then +4,
 * +2, +1; the result is p_0. x holds bf16 bit patterns. */
EXPORT void orc_router_logits(const uint16_t *x_bf16, const float *w_r, int T, int H, int E,
                              float *logits)
{
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            float p[32];
            for (int l = 0; l < 32; ++l) {
                float acc = 0.0f;
                for (int h = l; h < H; h += 32) {
                    uint32_t bits = (uint32_t)x_bf16[(size_t)t * H + h] << 16;
                    float xv;
                    memcpy(&xv, &bits, 4);
                    acc = fmaf(xv, w_r[(size_t)e * H + h], acc);
                }
                p[l] = acc;
            }
            for (int off = 16; off >= 1; off /= 2)
                for (int l = 0; l < off; ++l) p[l] = p[l] + p[l + off];
            logits[(size_t)t * E + e] = p[0];
        }
    }
}

/* Top-k with gates. Selection: k rounds, each taking the largest remaining
 * logit, the lower expert id on an exact tie. gates: g_j = exp(l_j - l_0) /
 * sum_i exp(l_i - l_0) over the k picked, in fp64 (equal to the full softmax
 * over E renormalised to the k picked). Logits must be finite. */
EXPORT void orc_topk_gates(const float *logits, int T, int E, int k, int32_t *ids, double *gates)
{
    char *taken = (char *)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        double denom = 0.0;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e; /* strict '>' keeps the lower id */
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        for (int j = 0; j < k; ++j)
            denom += exp((double)l[ids[(size_t)t * k + j]] - (double)l[ids[(size_t)t * k]]);
        for (int j = 0; j < k; ++j)
            gates[(size_t)t * k + j] =
                exp((double)l[ids[(size_t)t * k + j]] - (double)l[ids[(size_t)t * k]]) / denom;
    }
    free(taken);
}

/* ------------------------------------------------------------------------ */
/* Token-to-expert permutation [MG §3 module-based batching]: group the T*k   */
/* assignments by expert so that each expert sees one contiguous batch.      */
/* Definition (stable counting sort on the flat index f = t*k + j):          */
/*   counts[e] = #{f : ids[f] = e}; offsets = exclusive prefix sum (E+1);     */
/*   within expert e, assignments keep ascending f; perm_src[p] = f of the    */
/*   assignment at batch position p; inv[f] = p.                             */
/* ------------------------------------------------------------------------ */

EXPORT void orc_permute(const int32_t *ids, int T, int k, int E, int32_t *counts,
                        int32_t *offsets, int32_t *perm_src, int32_t *inv)
{
    int A = T * k;
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int f = 0; f < A; ++f) counts[ids[f]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    for (int e = 0; e <= E; ++e) next[e] = offsets[e];
    for (int f = 0; f < A; ++f) {
        int p = next[ids[f]]++;
        perm_src[p] = f;
        inv[f] = p;
    }
    free(next);
}

/* ------------------------------------------------------------------------ */
/* Per-layer VRAM slot pool with LRU [EP 階層ページング]: each layer owns S   */
/* slots, one expert per slot, managed LRU; a missing expert is copied in;   */
/* when one step needs more experts than slots, the layer switches to a      */
/* working buffer that holds what is needed.                                 */
/* Readings (the pages say only "LRU"):                                      */
/*  1. U = {e : counts[e] > 0}.                                              */
/*  2. |U| > S: working-buffer step. Slot state is left untouched (no        */
/*     eviction, no recency update). Resident experts are read in place from */
/*     their slots; every non-resident e in U gets working-buffer entry w =  */
/*     its rank among those, in ascending id; page_table[e] = S + w.         */
/*  3. |U| <= S: each hit refreshes last_use = step. Misses, in ascending id, */
/*     take the lowest-index empty slot, else the slot with the smallest     */
/*     last_use whose expert is not in U (ties: lowest slot index); the slot */
/*     gets the expert and last_use = step.                                  */
/*  4. page_table[e] = slot (or S + w) for e in U, -1 otherwise. The step    */
/*     counter advances by one per call.                                     */
/* The miss list holds (expert, destination index) in ascending expert id.   */
/* ------------------------------------------------------------------------ */

typedef struct {
    int E, S;
    int64_t step;
    int32_t *slot_expert; /* [S], -1 = empty */
    int64_t *last_use;    /* [S] */
} orc_lru;

EXPORT orc_lru *orc_lru_create(int E, int S)
{
    orc_lru *st = (orc_lru *)calloc(1, sizeof(orc_lru));
    st->E = E;
    st->S = S;
    st->slot_expert = (int32_t *)malloc(sizeof(int32_t) * (size_t)S);
    st->last_use = (int64_t *)malloc(sizeof(int64_t) * (size_t)S);
    for (int s = 0; s < S; ++s) {
        st->slot_expert[s] = -1;
        st->last_use[s] = -1;
    }
    return st;
}

EXPORT void orc_lru_destroy(orc_lru *st)
{
    if (!st) return;
    free(st->slot_expert);
    free(st->last_use);
    free(st);
}

EXPORT void orc_lru_state(const orc_lru *st, int32_t *slot_expert, int64_t *last_use, int64_t *step)
{
    memcpy(slot_expert, st->slot_expert, sizeof(int32_t) * (size_t)st->S);
    memcpy(last_use, st->last_use, sizeof(int64_t) * (size_t)st->S);
    *step = st->step;
}

/* Forgetting an expert's resident copy (its page changed, e.g. a new bit
 * width): its slot becomes empty, as at the start. */
EXPORT void orc_lru_invalidate(orc_lru *st, int e)
{
    for (int s = 0; s < st->S; ++s) {
        if (st->slot_expert[s] == e) {
            st->slot_expert[s] = -1;
            st->last_use[s] = -1;
        }
    }
}

static int lru_slot_of(const orc_lru *st, int e)
{
    for (int s = 0; s < st->S; ++s)
        if (st->slot_expert[s] == e) return s;
    return -1;
}

/* returns 1 for a working-buffer step, 0 otherwise */
EXPORT int orc_lru_step(orc_lru *st, const int32_t *counts, int32_t *page_table,
                        int32_t *miss_expert, int32_t *miss_dest, int32_t *n_miss)
{
    int E = st->E, S = st->S, nu = 0, wb = 0;
    int64_t now = st->step;
    char *in_u = (char *)calloc((size_t)E, 1);
    *n_miss = 0;
    for (int e = 0; e < E; ++e) {
        page_table[e] = -1;
        if (counts[e] > 0) {
            in_u[e] = 1;
            ++nu;
        }
    }
    if (nu > S) {
        int w = 0;
        wb = 1;
        for (int e = 0; e < E; ++e) {
            int s;
            if (!in_u[e]) continue;
            s = lru_slot_of(st, e);
            if (s >= 0) {
                page_table[e] = s;
            } else {
                page_table[e] = S + w;
                miss_expert[*n_miss] = e;
                miss_dest[*n_miss] = S + w;
                ++*n_miss;
                ++w;
            }
        }
    } else {
        for (int e = 0; e < E; ++e) {
            int s;
            if (!in_u[e]) continue;
            s = lru_slot_of(st, e);
            if (s >= 0) {
                st->last_use[s] = now;
                page_table[e] = s;
            }
        }
        for (int e = 0; e < E; ++e) {
            int victim = -1;
            if (!in_u[e] || page_table[e] >= 0) continue;
            for (int s = 0; s < S && victim < 0; ++s)
                if (st->slot_expert[s] < 0) victim = s;
            if (victim < 0) {
                for (int s = 0; s < S; ++s) {
                    if (in_u[st->slot_expert[s]]) continue;
                    if (victim < 0 || st->last_use[s] < st->last_use[victim]) victim = s;
                }
            }
            st->slot_expert[victim] = e;
            st->last_use[victim] = now;
            page_table[e] = victim;
            miss_expert[*n_miss] = e;
            miss_dest[*n_miss] = victim;
            ++*n_miss;
        }
    }
    st->step = now + 1;
    free(in_u);
    return wb;
}

/* ------------------------------------------------------------------------ */
/* Expert FFN and combine. Per assignment (t, j) with e = ids[t,j]:          */
/*   u = W13_e x_t   (W13 rows 0..I-1 are the gate projection, rows I..2I-1  */
/*                    the up projection: the packed "w13_weight" that [EP]   */
/*                    評価 names for vLLM's FP8 MoE)                          */
/*   h = SiLU(u_gate) * u_up,  SiLU(z) = z / (1 + exp(-z))                   */
/*   o = W2_e h       ("w2_weight", [H, I])                                  */
/*   y_t = sum_j g[t,j] * o_(t,j)                                            */
/* in fp64 from the dequantised weights; x is bf16 (exact in fp64). No       */
/* activation quantisation.                                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
    int32_t fmt;        /* 0: e4m3 + fp32 row scale; 1: e2m1 + e8m0 per 32 */
    int32_t pad;
    const uint8_t *w13; /* fmt 0: [2I*H] codes; fmt 1: [2I*H/2] nibble pairs */
    const void *s13;    /* fmt 0: float [2I]; fmt 1: uint8 [2I*H/32] */
    const uint8_t *w2;  /* fmt 0: [H*I]; fmt 1: [H*I/2] */
    const void *s2;     /* fmt 0: float [H]; fmt 1: uint8 [H*I/32] */
} orc_expert;

/* dequantised weight element (r, c) of a [rows, cols] matrix */
static double weight_at(int fmt, const uint8_t *w, const void *s, int cols, int r, int c)
{
    size_t idx = (size_t)r * cols + c;
    if (fmt == 0) return e4m3_cached(w[idx]) * (double)((const float *)s)[r];
    {
        uint8_t byte = w[idx / 2];
        uint8_t nib = (idx & 1) ? (byte >> 4) : (byte & 15);
        uint8_t sc = ((const uint8_t *)s)[(size_t)r * (cols / 32) + c / 32];
        return orc_e2m1_value(nib) * orc_e8m0_value(sc);
    }
}

/* y[n, H] for the tokens listed in token_list[n] (all T when token_list is
 * NULL). gates may come from orc_topk_gates or from elsewhere. */
EXPORT void orc_moe_ffn(const uint16_t *x_bf16, int T, int H, int I, int k, const int32_t *ids,
                        const double *gates, const orc_expert *experts, const int32_t *token_list,
                        int n_list, double *y)
{
    int n = token_list ? n_list : T;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < n; ++i) {
        int t = token_list ? token_list[i] : i;
        double *x = (double *)malloc(sizeof(double) * (size_t)H);
        double *u = (double *)malloc(sizeof(double) * (size_t)(2 * I));
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
        double *yt = y + (size_t)i * H;
        for (int c = 0; c < H; ++c) {
            uint32_t bits = (uint32_t)x_bf16[(size_t)t * H + c] << 16;
            float xv;
            memcpy(&xv, &bits, 4);
            x[c] = xv;
            yt[c] = 0.0;
        }
        for (int j = 0; j < k; ++j) {
            const orc_expert *ex = &experts[ids[(size_t)t * k + j]];
            double g = gates[(size_t)t * k + j];
            for (int r = 0; r < 2 * I; ++r) {
                double acc = 0.0;
                for (int c = 0; c < H; ++c) acc += weight_at(ex->fmt, ex->w13, ex->s13, H, r, c) * x[c];
                u[r] = acc;
            }
            for (int c = 0; c < I; ++c) h[c] = u[c] / (1.0 + exp(-u[c])) * u[I + c];
            for (int r = 0; r < H; ++r) {
                double acc = 0.0;
                for (int c = 0; c < I; ++c) acc += weight_at(ex->fmt, ex->w2, ex->s2, I, r, c) * h[c];
                yt[r] += g * acc;
            }
        }
        free(x);
        free(u);
        free(h);
    }
}

EXPORT int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

EXPORT void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Lossless compression of FP8 pages [EP 重みの圧縮]: per row of each expert  */
/* weight matrix, the exponent field is Huffman-coded and the rest is kept   */
/* raw; decoding happens on the GPU right after the host-to-device copy, and */
/* the code table stays resident in VRAM ([EP] 表4 discussion).              */
/* The pages fix nothing else. Format read here (one code per matrix):       */
/*  - symbol of byte b = (b >> 3) & 15 (the E4M3 exponent field);            */
/*    raw nibble = (b >> 7) << 3 | (b & 7) (sign, mantissa);                  */
/*  - code lengths: optimal prefix code over the matrix's symbol histogram   */
/*    with lengths <= LMAX = 12, by package-merge (Larmore & Hirschberg,     */
/*    1990); a single occurring symbol gets length 1; absent symbols get 0;  */
/*  - canonical codes: symbols sorted by (length, symbol) get consecutive    */
/*    code values, the code growing by one and shifting left at each new     */
/*    length (as in DEFLATE, RFC 1951 §3.2.2);                               */
/*  - each row is its own bitstream; rows start on 32-bit word boundaries;   */
/*    the stream is a sequence of uint32 words, bit i of a row is bit        */
/*    31 - (i % 32) of its word i / 32 (most significant bit first);          */
/*  - each row is cut into chunks of G = 64 symbols; chunk_bit[r][c] (uint16)*/
/*    is the bit offset of chunk c inside row r's stream;                    */
/*  - row_word[r] (uint32, R+1 entries) is the first word of row r;          */
/*  - nibbles[r][c/2]: two raw nibbles per byte, low nibble = even column.   */
/* Package-merge tie rule: items are kept sorted by weight; at equal weight  */
/* an original symbol item comes before a package, symbols among themselves  */
/* by ascending symbol, packages by creation order.                          */
/* ------------------------------------------------------------------------ */

#define HUF_NSYM 16
#define HUF_G 64

typedef struct {
    uint64_t weight;
    int is_pkg;
    int order;                 /* symbol id, or creation index of a package */
    unsigned char cnt[HUF_NSYM];
} pm_item;

static int pm_before(const pm_item *a, const pm_item *b)
{
    if (a->weight != b->weight) return a->weight < b->weight;
    if (a->is_pkg != b->is_pkg) return a->is_pkg < b->is_pkg;
    return a->order < b->order;
}

/* code lengths from frequencies; returns 0, or -1 if n symbols do not fit */
EXPORT int orc_huff_lengths(const uint64_t *freq, int lmax, uint8_t *len)
{
    pm_item leaves[HUF_NSYM], list[4 * HUF_NSYM], merged[4 * HUF_NSYM], pk[2 * HUF_NSYM];
    int n = 0, nl = 0, pkg_counter = 0;
    memset(len, 0, HUF_NSYM);
    for (int s = 0; s < HUF_NSYM; ++s) {
        if (!freq[s]) continue;
        memset(&leaves[n], 0, sizeof(pm_item));
        leaves[n].weight = freq[s];
        leaves[n].order = s;
        leaves[n].cnt[s] = 1;
        ++n;
    }
    if (n == 0) return 0;
    if (n == 1) {
        for (int s = 0; s < HUF_NSYM; ++s)
            if (freq[s]) len[s] = 1;
        return 0;
    }
    if ((1 << lmax) < n) return -1;
    /* sort leaves by (weight, symbol) */
    for (int i = 1; i < n; ++i)
        for (int j = i; j > 0 && pm_before(&leaves[j], &leaves[j - 1]); --j) {
            pm_item tmp = leaves[j];
            leaves[j] = leaves[j - 1];
            leaves[j - 1] = tmp;
        }
    /* deepest level: the leaves alone */
    for (int i = 0; i < n; ++i) list[i] = leaves[i];
    nl = n;
    for (int level = lmax - 1; level >= 1; --level) {
        int np = 0, a = 0, b = 0, m = 0;
        for (int i = 0; i + 1 < nl; i += 2) {
            memset(&pk[np], 0, sizeof(pm_item));
            pk[np].weight = list[i].weight + list[i + 1].weight;
            pk[np].is_pkg = 1;
            pk[np].order = pkg_counter++;
            for (int s = 0; s < HUF_NSYM; ++s)
                pk[np].cnt[s] = (unsigned char)(list[i].cnt[s] + list[i + 1].cnt[s]);
            ++np;
        }
        while (a < n || b < np) {
            if (b >= np || (a < n && pm_before(&leaves[a], &pk[b]))) merged[m++] = leaves[a++];
            else merged[m++] = pk[b++];
        }
        for (int i = 0; i < m; ++i) list[i] = merged[i];
        nl = m;
    }
    for (int i = 0; i < 2 * n - 2; ++i)
        for (int s = 0; s < HUF_NSYM; ++s) len[s] = (uint8_t)(len[s] + list[i].cnt[s]);
    return 0;
}

/* canonical code values from lengths */
EXPORT void orc_huff_codes(const uint8_t *len, uint32_t *code)
{
    uint32_t next = 0;
    int prev_len = 0;
    for (int l = 1; l <= 31; ++l) {
        for (int s = 0; s < HUF_NSYM; ++s) {
            if (len[s] != l) continue;
            next <<= (l - prev_len);
            prev_len = l;
            code[s] = next++;
        }
    }
    for (int s = 0; s < HUF_NSYM; ++s)
        if (!len[s]) code[s] = 0;
}

/* words needed by row r's stream, from the lengths */
static uint32_t row_bits(const uint8_t *q, int cols, const uint8_t *len)
{
    uint32_t bits = 0;
    for (int c = 0; c < cols; ++c) bits += len[(q[c] >> 3) & 15];
    return bits;
}

/* Encode a [rows, cols] FP8 matrix (cols a multiple of HUF_G).
 * Outputs: len[16]; row_word[rows+1]; chunk_bit[rows*cols/64];
 * nibbles[rows*cols/2]; words[] (size row_word[rows], pass words=NULL to size).
 * Returns the word count, or -1 if the code cannot be built. */
EXPORT int64_t orc_huff_encode(const uint8_t *q, int rows, int cols, int lmax, uint8_t *len,
                               uint32_t *row_word, uint16_t *chunk_bit, uint8_t *nibbles,
                               uint32_t *words)
{
    uint64_t freq[HUF_NSYM] = {0};
    uint32_t code[HUF_NSYM];
    int nchunk = cols / HUF_G;
    for (size_t i = 0; i < (size_t)rows * cols; ++i) freq[(q[i] >> 3) & 15]++;
    if (orc_huff_lengths(freq, lmax, len) != 0) return -1;
    orc_huff_codes(len, code);
    row_word[0] = 0;
    for (int r = 0; r < rows; ++r) {
        uint32_t nb = row_bits(q + (size_t)r * cols, cols, len);
        row_word[r + 1] = row_word[r] + (nb + 31) / 32;
    }
    if (!words) return row_word[rows];
    for (int r = 0; r < rows; ++r) {
        const uint8_t *qr = q + (size_t)r * cols;
        uint32_t *wr = words + row_word[r];
        uint32_t bit = 0;
        for (uint32_t w = row_word[r]; w < row_word[r + 1]; ++w) words[w] = 0;
        for (int c = 0; c < cols; ++c) {
            int sym = (qr[c] >> 3) & 15;
            if (c % HUF_G == 0) chunk_bit[(size_t)r * nchunk + c / HUF_G] = (uint16_t)bit;
            for (int i = len[sym] - 1; i >= 0; --i) {
                if ((code[sym] >> i) & 1) wr[bit / 32] |= 1u << (31 - bit % 32);
                ++bit;
            }
        }
        for (int c = 0; c < cols; c += 2) {
            uint8_t b0 = qr[c], b1 = qr[c + 1];
            uint8_t n0 = (uint8_t)(((b0 >> 7) << 3) | (b0 & 7));
            uint8_t n1 = (uint8_t)(((b1 >> 7) << 3) | (b1 & 7));
            nibbles[((size_t)r * cols + c) / 2] = (uint8_t)(n0 | (n1 << 4));
        }
    }
    return row_word[rows];
}

/* Decode back to FP8 bytes by walking the canonical code bit by bit.
 * Returns 0, or -2 when the stream is corrupt (a bit string that is no
 * code, or a read past the row's last word). */
EXPORT int orc_huff_decode(const uint8_t *len, const uint32_t *row_word, const uint16_t *chunk_bit,
                           const uint8_t *nibbles, const uint32_t *words, int rows, int cols,
                           uint8_t *q)
{
    uint32_t code[HUF_NSYM];
    int nchunk = cols / HUF_G;
    orc_huff_codes(len, code);
    for (int r = 0; r < rows; ++r) {
        uint32_t nbits = (row_word[r + 1] - row_word[r]) * 32;
        const uint32_t *wr = words + row_word[r];
        for (int ch = 0; ch < nchunk; ++ch) {
            uint32_t bit = chunk_bit[(size_t)r * nchunk + ch];
            for (int c = ch * HUF_G; c < (ch + 1) * HUF_G; ++c) {
                uint32_t acc = 0;
                int l = 0, sym = -1;
                while (sym < 0) {
                    if (bit >= nbits || l >= 31) return -2;
                    acc = (acc << 1) | ((wr[bit / 32] >> (31 - bit % 32)) & 1);
                    ++bit;
                    ++l;
                    for (int s = 0; s < HUF_NSYM; ++s)
                        if (len[s] == l && code[s] == acc) sym = s;
                }
                {
                    size_t idx = (size_t)r * cols + c;
                    uint8_t nib = (idx & 1) ? (nibbles[idx / 2] >> 4) : (nibbles[idx / 2] & 15);
                    q[idx] = (uint8_t)(((nib >> 3) << 7) | (sym << 3) | (nib & 7));
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Per-expert bit-width from importance [PW 技術的に面白い点: the router's    */
/* choice estimates each expert's importance; important experts keep more     */
/* bits]. Reading: importance m_e is an exponential moving average of the    */
/* gate mass the expert receives per token,                                  */
/*   m_e <- alpha * m_e + (1 - alpha) * (sum_{t,j: ids=e} g[t,j]) / T,       */
/* the sum taken in ascending (t, j) in fp64 from the fp32 gates. Every       */
/* `every` steps (after the update of steps every-1, 2*every-1, ...) the      */
/* experts are ranked by m (descending; ties to the lower id) and the top    */
/* n_hi keep FP8 (tag 0), the rest get 4-bit pages (tag 1).                  */
/* ------------------------------------------------------------------------ */

EXPORT void orc_rank_formats(const double *m, int E, int n_hi, uint8_t *fmt)
{
    char *done = (char *)calloc((size_t)E, 1);
    for (int e = 0; e < E; ++e) fmt[e] = 1;
    for (int r = 0; r < n_hi && r < E; ++r) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (done[e]) continue;
            if (best < 0 || m[e] > m[best]) best = e;
        }
        done[best] = 1;
        fmt[best] = 0;
    }
    free(done);
}

/* Quality-aware ranking (the PagedWeight feedback loop, a reading): expert e's
 * score is its importance m[e] times q[e], the relative output error its 4-bit
 * page shows on sampled tokens; the top n_hi scores keep FP8 (ties: lower id). */
EXPORT void orc_rank_formats_quality(const double *m, const double *q, int E, int n_hi, uint8_t *fmt)
{
    double *score = (double *)malloc((size_t)E * sizeof(double));
    for (int e = 0; e < E; ++e) score[e] = m[e] * q[e];
    orc_rank_formats(score, E, n_hi, fmt);
    free(score);
}

/* returns 1 when the formats were re-ranked at this step */
EXPORT int orc_importance_step(double *m, const int32_t *ids, const float *gates, int T, int k,
                               int E, double alpha, int64_t step, int every, int n_hi, uint8_t *fmt)
{
    double *mass = (double *)calloc((size_t)E, sizeof(double));
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) mass[ids[(size_t)t * k + j]] += (double)gates[(size_t)t * k + j];
    for (int e = 0; e < E; ++e) m[e] = alpha * m[e] + (1.0 - alpha) * (mass[e] / (double)T);
    free(mass);
    if ((step + 1) % every == 0) {
        orc_rank_formats(m, E, n_hi, fmt);
        return 1;
    }
    return 0;
}
