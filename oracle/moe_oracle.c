/*
 * Block-coreset sparse MoE FFN -- CPU ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain definition that the
 * CUDA path is checked against.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load it; the product path never does.  It
 * shares no code, header, table or constant with the CUDA sources.
 *
 * What it computes, and where each step comes from:
 *
 *  - Model card "Clover-35B-A3B-Preview -- CMF", intro: an MoE with 256 experts,
 *    top-8, plus one shared expert; text is written in 32-token blocks, each
 *    resolved by repeated denoising passes over the whole block.
 *  - Same page, Usage: the block's experts are restricted to the set that
 *    carries 90% of the block's routing; block size 8, 16 or 32.
 *  - InfiniLM PR #604, Summary: preview passes use "block coreset routing";
 *    Notes: a full-route replay (coreset disabled) on commit.
 *
 * The pages leave the arithmetic open.  The readings taken here:
 *
 *  1. Router logit z[r,e] = sum_h x[r,h] * Wr[e,h] (+ bias[b,e]) in fp32, in a
 *     FIXED order so that top-k indices can be compared bit for bit: h is cut
 *     into stripes of 256; "lane" p (0..31) owns elements 8p..8p+7 of every
 *     stripe and sums its products in ascending h; the 32 partial sums are then
 *     combined by the xor butterfly t_p = s_p + s_(p^o), o = 16,8,4,2,1.  A
 *     bf16*bf16 product is exact in fp32 (16 significant bits).  The logit is
 *     finally z + 0.0f, which turns -0 into +0.
 *  2. Top-k: experts ordered by (z descending, id ascending); NaN ranks last.
 *  3. Weights: softmax restricted to the k selected logits (the full-softmax
 *     denominator cancels when the top-k weights are renormalised):
 *     a_j = exp_c(z_j - z_max), S = a_0 + ... + a_(k-1) in rank order,
 *     w_j = a_j / S.  exp_c is a Cody-Waite reduction (ln 2 split into a
 *     12-significant-bit head and a tail) with a degree-7 Taylor polynomial
 *     evaluated by Horner's rule in fmaf, scaled by 2^n through the exponent.
 *  3b. Probability mass (the other reading of "90% of its routing", InfiniLM
 *     PR #604, Summary; model card, Usage): the mass of slot j is the
 *     unnormalised probability p_j = a_j / D of the full softmax over all E
 *     experts, D = sum over every expert e of exp_c(z_e - z_max) in a fixed
 *     order: "lane" p (0..31) sums the experts e = p, p + 32, p + 64, ... in
 *     ascending e, and the 32 lane sums are combined by the same xor
 *     butterfly as the logits (o = 16, 8, 4, 2, 1).  Only the coreset mass
 *     changes; the renormalised weights still come from w.
 *  4. Block mass: q = trunc(w * 2^32) (or trunc(p * 2^32) under 3b) as an exact
 *     integer; Q_e = sum of q over the block's rows that selected e;
 *     T = sum_e Q_e.
 *  5. Coreset: tau >= 1 keeps every touched expert and leaves w unchanged.
 *     Otherwise theta = ceil(tau * T) computed exactly (tau is the fp32 value
 *     M * 2^-s), experts ordered by (Q descending, id ascending), and the
 *     coreset is the shortest prefix whose mass reaches theta.  An expert
 *     budget B > 0 (InfiniLM PR #604, Summary, names it without defining it)
 *     keeps at most the first B experts of that order; when it drops an
 *     expert with tau >= 1, the rows are renormalised as in 6.
 *  6. Renormalise: per row, s' = sum of surviving w_j in rank order (fp32),
 *     w'_j = w_j / s', 0 for dropped j; a row with s' == 0 keeps only the
 *     shared expert and is counted as empty.
 *  8. Quantised experts (model card, Files: 8-bit and 4-bit expert files; the
 *     page gives no codec).  Reading: along a weight row's input dimension,
 *     blocks of 32 weights share one bf16 scale d; the weight is stored as a
 *     signed integer q (int8, or a 4-bit two's-complement nibble, two per byte,
 *     the even element in the low nibble) and stands for q * d rounded once to
 *     bf16 (round to nearest, ties to even; q * d itself is exact in fp32).  The
 *     scales are stored block-major: d[block][row].  The FFN of step 7 then runs
 *     on those bf16 weights.
 *  7. Expert FFN in fp64: E_e(x) = Wd_e (silu(Wg_e x) * (Wu_e x)); the shared
 *     expert S is the same form; y_r = S(x_r) + sum_j w'_j E_(e_j)(x_r), with j
 *     in rank order, over surviving j only.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 *        (contraction off: every fp32 operation above is a separate IEEE
 *        operation unless written as fmaf).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG (-1)

/* ------------------------------------------------------------------------- */
/* scalar helpers                                                            */

static float bf16_to_float(uint16_t v) {
    uint32_t u = (uint32_t)v << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t float_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

static float bits_float(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Order-preserving 32-bit key of a float: larger float -> larger key; every
 * NaN maps to 0, below -inf. */
static uint32_t order_key(float f) {
    if (f != f) return 0u;
    uint32_t u = float_bits(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

/* exp_c(t) for t <= 0 (reading 3).  Cody-Waite: n = rint(t / ln 2),
 * r = t - n ln2 with ln 2 = LN2_HI + LN2_LO, LN2_HI = 2839 / 4096 (12
 * significant bits, so n * LN2_HI is exact for |n| <= 2^12).  Then
 * e^r = sum_{k<=7} r^k / k! and e^t = e^r * 2^n. */
float moe_oracle_exp_c(float t) {
    const float LOG2E = 1.44269504088896341f;                       /* 1 / ln 2 */
    const float LN2_HI = 0.693115234375f;                           /* 2839/4096 */
    const float LN2_LO = (float)(0.69314718055994530942 - 0.693115234375);
    const float C[8] = {1.0f, 1.0f, 0.5f, (float)(1.0 / 6.0), (float)(1.0 / 24.0),
                        (float)(1.0 / 120.0), (float)(1.0 / 720.0), (float)(1.0 / 5040.0)};
    if (t != t) return 0.0f;
    if (t < -87.0f) return 0.0f;
    float n = rintf(t * LOG2E);
    float r = fmaf(-n, LN2_HI, t);
    r = fmaf(-n, LN2_LO, r);
    float p = C[7];
    for (int i = 6; i >= 0; --i) p = fmaf(p, r, C[i]);
    int ni = (int)n;                      /* in [-126, 0] for t in [-87, 0] */
    float scale = bits_float((uint32_t)(ni + 127) << 23);
    return p * scale;
}

/* Reading 1: one router logit in the fixed lane/stripe order. */
float moe_oracle_logit(const uint16_t* xr, const uint16_t* we, int H) {
    float s[32];
    for (int p = 0; p < 32; ++p) {
        float acc = 0.0f;
        for (int stripe = 0; stripe < H; stripe += 256)
            for (int t = 0; t < 8; ++t) {
                int h = stripe + 8 * p + t;
                float prod = bf16_to_float(xr[h]) * bf16_to_float(we[h]);
                acc = acc + prod;
            }
        s[p] = acc;
    }
    for (int o = 16; o >= 1; o >>= 1) {
        float t[32];
        for (int p = 0; p < 32; ++p) t[p] = s[p] + s[p ^ o];
        memcpy(s, t, sizeof s);
    }
    return s[0];
}

/* ------------------------------------------------------------------------- */
/* routing: logits, top-k, weights                                           */

typedef struct {
    const uint16_t* x;
    const uint16_t* wr;
    const float* bias;
    const int32_t* block_of_row;
    int R, H, E, k;
    int32_t* topk_idx;
    float* topk_w;
    float* topk_p;      /* [R, k] probability mass (reading 3b) or NULL */
    float* logits;      /* [R, E] or NULL */
    int r0, r1;
    long nonfinite;
} route_job;

static void route_rows(route_job* J) {
    float* z = (float*)malloc(sizeof(float) * (size_t)J->E);
    unsigned char* taken = (unsigned char*)malloc((size_t)J->E);
    for (int r = J->r0; r < J->r1; ++r) {
        const uint16_t* xr = J->x + (size_t)r * J->H;
        for (int e = 0; e < J->E; ++e) {
            float v = moe_oracle_logit(xr, J->wr + (size_t)e * J->H, J->H);
            if (J->bias) v = v + J->bias[(size_t)J->block_of_row[r] * J->E + e];
            v = v + 0.0f;
            if (!isfinite(v)) J->nonfinite++;
            z[e] = v;
            if (J->logits) J->logits[(size_t)r * J->E + e] = v;
        }
        /* top-k by (z desc, id asc); NaN last */
        memset(taken, 0, (size_t)J->E);
        int32_t* idx = J->topk_idx + (size_t)r * J->k;
        for (int j = 0; j < J->k; ++j) {
            int best = -1;
            uint32_t bk = 0;
            for (int e = 0; e < J->E; ++e) {
                if (taken[e]) continue;
                uint32_t key = order_key(z[e]);
                if (best < 0 || key > bk) { best = e; bk = key; }
            }
            taken[best] = 1;
            idx[j] = best;
        }
        /* weights: softmax over the selected k, in rank order */
        float m = z[idx[0]];
        float a[64];
        float S = 0.0f;
        for (int j = 0; j < J->k; ++j) {
            a[j] = moe_oracle_exp_c(z[idx[j]] - m);
            S = S + a[j];
        }
        float* w = J->topk_w + (size_t)r * J->k;
        for (int j = 0; j < J->k; ++j) w[j] = a[j] / S;
        if (J->topk_p) {
            /* reading 3b: the full-softmax denominator in the lane order */
            float d[32];
            for (int p = 0; p < 32; ++p) {
                float acc = 0.0f;
                for (int e = p; e < J->E; e += 32) acc = acc + moe_oracle_exp_c(z[e] - m);
                d[p] = acc;
            }
            for (int o = 16; o >= 1; o >>= 1) {
                float t[32];
                for (int p = 0; p < 32; ++p) t[p] = d[p] + d[p ^ o];
                memcpy(d, t, sizeof d);
            }
            float* pj = J->topk_p + (size_t)r * J->k;
            for (int j = 0; j < J->k; ++j) pj[j] = a[j] / d[0];
        }
    }
    free(z);
    free(taken);
}

static void* route_thread(void* p) {
    route_rows((route_job*)p);
    return NULL;
}

static int check_offsets(const int32_t* off, int nb, int R) {
    if (nb < 0 || !off || off[0] != 0 || off[nb] != R) return 0;
    for (int b = 0; b < nb; ++b)
        if (off[b + 1] < off[b]) return 0;
    return 1;
}

/* Route every row.  bias: [nb, E] fp32 or NULL.  topk_p: [R, k] probability
 * mass of reading 3b, or NULL.  logits: [R, E] or NULL.
 * Returns the number of non-finite logits (>= 0) or ORC_ERR_ARG. */
long moe_oracle_route(const uint16_t* x, const uint16_t* wr, const float* bias,
                      const int32_t* block_offsets, int nb, int R, int H, int E, int k,
                      int32_t* topk_idx, float* topk_w, float* topk_p, float* logits,
                      int nthreads) {
    if (!x || !wr || !topk_idx || !topk_w || H <= 0 || H % 256 || E <= 0 || k <= 0 ||
        k > E || k > 64 || R < 0 || !check_offsets(block_offsets, nb, R))
        return ORC_ERR_ARG;
    int32_t* bor = (int32_t*)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
    for (int b = 0; b < nb; ++b)
        for (int r = block_offsets[b]; r < block_offsets[b + 1]; ++r) bor[r] = b;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > R) nthreads = R > 0 ? R : 1;
    route_job* jobs = (route_job*)calloc((size_t)nthreads, sizeof(route_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        route_job j = {x, wr, bias, bor, R, H, E, k, topk_idx, topk_w, topk_p, logits,
                       (int)((long)R * t / nthreads), (int)((long)R * (t + 1) / nthreads), 0};
        jobs[t] = j;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, route_thread, &jobs[t]);
    route_rows(&jobs[0]);
    long nf = jobs[0].nonfinite;
    for (int t = 1; t < nthreads; ++t) {
        pthread_join(th[t], NULL);
        nf += jobs[t].nonfinite;
    }
    free(jobs);
    free(th);
    free(bor);
    return nf;
}

/* ------------------------------------------------------------------------- */
/* coreset                                                                   */

typedef unsigned __int128 u128;

/* theta = ceil(tau * T) exactly, for 0 < tau < 1 (reading 5). */
static uint64_t mass_threshold(float tau, uint64_t T) {
    uint32_t u = float_bits(tau);
    uint32_t ex = (u >> 23) & 0xFFu;
    uint64_t M = (ex == 0) ? (u & 0x7FFFFFu) : ((u & 0x7FFFFFu) | 0x800000u);
    int s = (ex == 0) ? 149 : 150 - (int)ex;   /* tau = M * 2^-s, s >= 24 */
    u128 prod = (u128)M * (u128)T;
    if (prod == 0) return 0;
    if (s >= 128) return 1;
    u128 q = prod >> s;
    if ((q << s) != prod) q += 1;
    return (uint64_t)q;
}

/* Every block of rows.  Outputs keep bits [E/32 words], core size, w_renorm
 * and the number of empty rows per block.  topk_mass: [R, k] masses of the
 * slots (reading 3b), or NULL for the weights w themselves (reading 4). */
long moe_oracle_coreset(const int32_t* block_offsets, int nb, int R, int E, int k,
                        const int32_t* topk_idx, const float* topk_w,
                        const float* topk_mass, float tau,
                        uint32_t* keep, int32_t* core_size, float* w_renorm,
                        int32_t* n_empty, int max_experts) {
    if (!topk_idx || !topk_w || !keep || !core_size || !w_renorm || E <= 0 || k <= 0 ||
        k > E || !check_offsets(block_offsets, nb, R) || !(tau > 0.0f))
        return ORC_ERR_ARG;
    int words = (E + 31) / 32;
    uint64_t* Q = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)E);
    unsigned char* touched = (unsigned char*)malloc((size_t)E);
    unsigned char* in_core = (unsigned char*)malloc((size_t)E);
    int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    long bad = 0;
    for (int b = 0; b < nb; ++b) {
        int r0 = block_offsets[b], r1 = block_offsets[b + 1];
        memset(Q, 0, sizeof(uint64_t) * (size_t)E);
        memset(touched, 0, (size_t)E);
        memset(in_core, 0, (size_t)E);
        for (int r = r0; r < r1; ++r)
            for (int j = 0; j < k; ++j) {
                int e = topk_idx[(size_t)r * k + j];
                if (e < 0 || e >= E) { bad++; continue; }
                touched[e] = 1;
                /* the mass of the slot: w, or p under reading 3b */
                float wj = (topk_mass ? topk_mass : topk_w)[(size_t)r * k + j];
                /* a mass is in [0, 1]; anything else (NaN) carries no mass */
                if (wj >= 0.0f && wj <= 1.0f) Q[e] += (uint64_t)ldexpf(wj, 32);
            }
        int nt = 0;
        uint64_t T = 0;
        for (int e = 0; e < E; ++e)
            if (touched[e]) { order[nt++] = e; T += Q[e]; }
        /* expert budget (InfiniLM PR #604, Summary: "expert-budget"; reading:
         * at most max_experts of the block's experts are kept, the first ones of
         * the same order; max_experts <= 0: no budget) */
        const int cap = (max_experts > 0 && max_experts < nt) ? max_experts : nt;
        /* rows keep their weights bit for bit only when nothing is dropped */
        const int renorm = tau < 1.0f || cap < nt;
        int c;
        if (!renorm) {
            c = nt;
            for (int i = 0; i < nt; ++i) in_core[order[i]] = 1;
        } else {
            /* insertion sort by (Q desc, id asc); order[] starts in id order */
            for (int i = 1; i < nt; ++i) {
                int e = order[i], p = i - 1;
                while (p >= 0 && Q[order[p]] < Q[e]) { order[p + 1] = order[p]; --p; }
                order[p + 1] = e;
            }
            if (tau >= 1.0f) {
                c = cap;
            } else {
                uint64_t theta = mass_threshold(tau, T);
                uint64_t run = 0;
                c = 0;
                while (c < cap && run < theta) { run += Q[order[c]]; ++c; }
            }
            for (int i = 0; i < c; ++i) in_core[order[i]] = 1;
        }
        core_size[b] = c;
        for (int wd = 0; wd < words; ++wd) {
            uint32_t bits = 0;
            for (int i = 0; i < 32 && wd * 32 + i < E; ++i)
                if (in_core[wd * 32 + i]) bits |= 1u << i;
            keep[(size_t)b * words + wd] = bits;
        }
        int empty = 0;
        for (int r = r0; r < r1; ++r) {
            const int32_t* idx = topk_idx + (size_t)r * k;
            const float* w = topk_w + (size_t)r * k;
            float* wo = w_renorm + (size_t)r * k;
            if (!renorm) {
                for (int j = 0; j < k; ++j) wo[j] = w[j];
                continue;
            }
            float s = 0.0f;
            for (int j = 0; j < k; ++j)
                if (idx[j] >= 0 && idx[j] < E && in_core[idx[j]]) s = s + w[j];
            if (s == 0.0f) {
                for (int j = 0; j < k; ++j) wo[j] = 0.0f;
                empty++;
                continue;
            }
            for (int j = 0; j < k; ++j)
                wo[j] = (idx[j] >= 0 && idx[j] < E && in_core[idx[j]]) ? w[j] / s : 0.0f;
        }
        if (n_empty) n_empty[b] = empty;
    }
    free(Q);
    free(touched);
    free(in_core);
    free(order);
    return bad;
}

/* ------------------------------------------------------------------------- */
/* quantised weights (reading 8)                                             */

/* fp32 -> bf16 bits, round to nearest, ties to even (NaN stays NaN). */
static uint16_t float_to_bf16_rne(float f) {
    uint32_t u = float_bits(f);
    if ((u & 0x7F800000u) == 0x7F800000u)
        return (uint16_t)((u >> 16) | ((u & 0x7FFFFFu) ? 0x40u : 0u));
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* One weight matrix [rows, K] back to bf16 bits: q is int8 [rows, K] (bits 8)
 * or packed nibbles uint8 [rows, K / 2] (bits 4); d is bf16 [K / 32, rows].
 * Returns 0, or ORC_ERR_ARG. */
int moe_oracle_dequant(const void* q, const uint16_t* d, int bits, int rows, int K,
                       uint16_t* out) {
    if (!q || !d || !out || rows <= 0 || K <= 0 || K % 32 || (bits != 8 && bits != 4))
        return ORC_ERR_ARG;
    for (int r = 0; r < rows; ++r)
        for (int k = 0; k < K; ++k) {
            int qv;
            if (bits == 8) {
                qv = (int)((const int8_t*)q)[(size_t)r * K + k];
            } else {
                uint8_t byte = ((const uint8_t*)q)[(size_t)r * (K / 2) + k / 2];
                int nib = (k & 1) ? (byte >> 4) : (byte & 0xF);
                qv = nib >= 8 ? nib - 16 : nib;
            }
            float scale = bf16_to_float(d[(size_t)(k / 32) * rows + r]);
            out[(size_t)r * K + k] = float_to_bf16_rne((float)qv * scale);
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* FFN (fp64)                                                                */

/* SwiGLU expert on one row: out[H] = Wd (silu(Wg x) * (Wu x)), all fp64.
 * Wg, Wu: [I, H]; Wd: [H, I]. */
void moe_oracle_expert_ffn(const uint16_t* xr, const uint16_t* wg, const uint16_t* wu,
                           const uint16_t* wd, int H, int I, double* out) {
    double* hbuf = (double*)malloc(sizeof(double) * (size_t)I);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        const uint16_t* gi = wg + (size_t)i * H;
        const uint16_t* ui = wu + (size_t)i * H;
        for (int h = 0; h < H; ++h) {
            double xv = (double)bf16_to_float(xr[h]);
            g += xv * (double)bf16_to_float(gi[h]);
            u += xv * (double)bf16_to_float(ui[h]);
        }
        hbuf[i] = g / (1.0 + exp(-g)) * u;
    }
    for (int h = 0; h < H; ++h) {
        const uint16_t* dh = wd + (size_t)h * I;
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += (double)bf16_to_float(dh[i]) * hbuf[i];
        out[h] = acc;
    }
    free(hbuf);
}

typedef struct {
    const uint16_t* x;
    const uint16_t* const* wg;
    const uint16_t* const* wu;
    const uint16_t* const* wd;
    const uint16_t *sg, *su, *sd;
    const int32_t* topk_idx;
    const float* w_renorm;
    const uint32_t* keep;
    const int32_t* block_of_row;
    int H, E, k, I, Is, words;
    double* y;
    int r0, r1;
    int missing;
} fwd_job;

static void forward_rows(fwd_job* J) {
    double* o = (double*)malloc(sizeof(double) * (size_t)J->H);
    for (int r = J->r0; r < J->r1; ++r) {
        const uint16_t* xr = J->x + (size_t)r * J->H;
        double* yr = J->y + (size_t)r * J->H;
        moe_oracle_expert_ffn(xr, J->sg, J->su, J->sd, J->H, J->Is, yr);
        int b = J->block_of_row[r];
        for (int j = 0; j < J->k; ++j) {
            int e = J->topk_idx[(size_t)r * J->k + j];
            if (e < 0 || e >= J->E) continue;
            if (!((J->keep[(size_t)b * J->words + e / 32] >> (e % 32)) & 1u)) continue;
            if (!J->wg[e] || !J->wu[e] || !J->wd[e]) { J->missing = 1; continue; }
            double wj = (double)J->w_renorm[(size_t)r * J->k + j];
            moe_oracle_expert_ffn(xr, J->wg[e], J->wu[e], J->wd[e], J->H, J->I, o);
            for (int h = 0; h < J->H; ++h) yr[h] += wj * o[h];
        }
    }
    free(o);
}

static void* forward_thread(void* p) {
    forward_rows((fwd_job*)p);
    return NULL;
}

/* y[R, H] (fp64) = shared(x) + sum over surviving (r, j) of w_renorm * expert(x).
 * wg/wu/wd are tables of E per-expert pointers (NULL for an expert that no
 * surviving pair uses).  Returns 0, ORC_ERR_ARG, or -2 if a needed expert
 * pointer was NULL. */
int moe_oracle_forward(const uint16_t* x, const int32_t* block_offsets, int nb, int R, int H,
                       int E, int k, int I, int Is, const uint16_t* const* wg,
                       const uint16_t* const* wu, const uint16_t* const* wd,
                       const uint16_t* sg, const uint16_t* su, const uint16_t* sd,
                       const int32_t* topk_idx, const float* w_renorm, const uint32_t* keep,
                       double* y, int nthreads) {
    if (!x || !wg || !wu || !wd || !sg || !su || !sd || !topk_idx || !w_renorm || !keep ||
        !y || H <= 0 || E <= 0 || k <= 0 || I <= 0 || Is <= 0 ||
        !check_offsets(block_offsets, nb, R))
        return ORC_ERR_ARG;
    int32_t* bor = (int32_t*)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
    for (int b = 0; b < nb; ++b)
        for (int r = block_offsets[b]; r < block_offsets[b + 1]; ++r) bor[r] = b;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > R) nthreads = R > 0 ? R : 1;
    fwd_job* jobs = (fwd_job*)calloc((size_t)nthreads, sizeof(fwd_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        fwd_job j = {x, wg, wu, wd, sg, su, sd, topk_idx, w_renorm, keep, bor,
                     H, E, k, I, Is, (E + 31) / 32, y,
                     (int)((long)R * t / nthreads), (int)((long)R * (t + 1) / nthreads), 0};
        jobs[t] = j;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, forward_thread, &jobs[t]);
    forward_rows(&jobs[0]);
    int missing = jobs[0].missing;
    for (int t = 1; t < nthreads; ++t) {
        pthread_join(th[t], NULL);
        missing |= jobs[t].missing;
    }
    free(jobs);
    free(th);
    free(bor);
    return missing ? -2 : ORC_OK;
}
