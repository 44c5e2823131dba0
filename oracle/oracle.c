/*
 * oracle.c -- plain, slow, single-threaded CPU reference of the OEA MoE
 * decode layer.  TEST INFRASTRUCTURE ONLY: the library's product path never
 * links, loads or calls this file; only the tests, the smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code with the CUDA path.
 *
 * What it computes, with the passage each step follows:
 *
 *   Page "Opportunistic Expert Activation (OEA)" (zhaifeiyue.github.io,
 *   papers/2511.02237), sections 1-4 and 7:
 *     - router scores and per-token top-k over N experts (section 2, Q1/Q2)
 *     - OEA phase 1: baseline of the token's top-n_i experts,
 *       n_i = min(k0, t_i), t_i an adaptive top-p count (section 2, Q2)
 *     - batch union S_base of the baselines, T = |S_base| (section 2, Q2)
 *     - OEA phase 2: walk the token's own ranked list and add an expert
 *       only if it is in S_base (section 3, the "e_ij in S_base" gate),
 *       at most k^max experts, ranks at most maxP (sections 4-5, 7)
 *     - kept router scores renormalised (section 2, Q2)
 *     - per-expert load cnt_e and the invariants cnt_e <= B, T <= N,
 *       sum cnt_e = B*k for plain top-k (section 4, check 3)
 *     - padding tokens select no expert (section 7, implementation detail 1)
 *   The expert FFN is the SwiGLU form of the Qwen3 MoE experts the page
 *   measures: y = W_down (silu(W_gate x) * (W_up x)).
 *   The INT4 group-wise weight format is the low-precision expert version
 *   of the DynaExq page (hotelren.com/news/4921287, section 3.2,
 *   "precision tiers"): symmetric 4-bit codes, one bf16 scale per group.
 *
 * Precision: floating point sums are carried in fp64.  Decisions that turn
 * floats into integers (the top-p count t_i) are taken in fp32, the
 * precision in which the GPU takes them; ranking compares the fp32 logits
 * exactly.  Ties in the ranking go to the lower expert id.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_TOPK 0
#define ORACLE_OEA 1

/* logits[i][e] = sum_c x[i][c] * w_router[e][c] + bias[e]
 * fp64 accumulation in ascending c.  Inputs are fp32 arrays (bf16 values are
 * exactly representable); bias may be NULL. */
void oracle_router_logits(const float *x, const float *w_router, const float *bias,
                          int B, int N, int d, double *logits)
{
    for (int i = 0; i < B; ++i)
        for (int e = 0; e < N; ++e) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += (double)x[(size_t)i * d + c] * (double)w_router[(size_t)e * d + c];
            if (bias)
                acc += (double)bias[e];
            logits[(size_t)i * N + e] = acc;
        }
}

/* a ranks before b: larger logit, or equal logit and smaller id */
static int ranks_before(float la, int a, float lb, int b)
{
    return la > lb || (la == lb && a < b);
}

/* order[0..N) = expert ids sorted by (logit desc, id asc); insertion sort */
static void rank_experts(const float *l, int N, int *order)
{
    for (int e = 0; e < N; ++e) {
        int j = e;
        while (j > 0 && ranks_before(l[e], e, l[order[j - 1]], order[j - 1])) {
            order[j] = order[j - 1];
            --j;
        }
        order[j] = e;
    }
}

/* Adaptive top-p count t_i: the smallest t with sum_{j<=t} P_(j) >= p, where
 * P is the softmax over all N logits taken in ranked order.  p >= 1 means
 * top-p is off and t_i = N.  fp32, sums in ascending expert id. */
static int top_p_count(const float *l, const int *order, int N, float p)
{
    if (p >= 1.0f)
        return N;
    float m = l[order[0]];
    float Z = 0.0f;
    for (int e = 0; e < N; ++e)
        Z += expf(l[e] - m);
    float prefix = 0.0f;
    for (int t = 1; t <= N; ++t) {
        prefix += expf(l[order[t - 1]] - m) / Z;
        if (prefix >= p)
            return t;
    }
    return N;
}

/*
 * Batch-size-dependent k0 (OEA page, section 7, implementation detail 2):
 * piggybacking adds nothing for a single token and OEA belongs only to
 * non-trivial batches, so a batch with at most one real token routes by
 * plain top-k (k0 = k, top-p off: *p is set to 1); smaller batches take
 * the larger, safer k0 = ceil(5k/8) and batches of 16 or more tokens the
 * aggressive k0 = ceil(3k/8).  For k = 8 these are the page's two settings,
 * k0 = 5 and k0 = 3, whose results the page reports at B = 16 (section 5,
 * Figs. 2-3, Table 3).
 */
int oracle_policy_k0(int B_valid, int k, float *p)
{
    if (B_valid <= 1) {
        *p = 1.0f;
        return k;
    }
    if (B_valid < 16)
        return (5 * k + 7) / 8;
    return (3 * k + 7) / 8;
}

/*
 * Routing for one batch.
 *   logits   [B][N] fp32 (row i of token i)
 *   mode     ORACLE_TOPK or ORACLE_OEA
 *   k        top-k of the plain router (slots per token when mode is top-k)
 *   k0, p    OEA baseline cap and top-p threshold (p >= 1: top-p off);
 *            k0 <= 0 takes k0 (and possibly p) from oracle_policy_k0
 *   maxP     deepest rank phase 2 may take an expert from (>= N: no limit)
 *   kmax     experts per token after phase 2 (slots per token in OEA mode)
 *   B_valid  tokens i >= B_valid are padding and select nothing
 *   nbase_in [B] or NULL (OEA only): phase 1 takes n_i = nbase_in[i]
 *            (1..k0) for every real token instead of computing t_i; for
 *            comparing with a router whose fp32 prefix sums land on the
 *            other side of p for a token whose prefix lies at p
 * Outputs (kslots = k for top-k, kmax for OEA):
 *   idx   [B][kslots] expert ids in ranked order, -1 in unused slots
 *   w     [B][kslots] renormalised weights, 0 in unused slots
 *   nbase [B]         n_i (k for top-k; 0 for padding tokens)
 *   T                 number of distinct experts selected by the batch
 *   counts [N], offsets [N+1] (exclusive scan of counts in expert order)
 *   active [N]        experts with counts > 0 in ascending id, first T valid
 *   perm  [sum counts] token*kslots+slot, grouped by expert (ascending id),
 *                      tokens ascending within an expert
 * Returns 0, or -1 on invalid arguments.
 */
int oracle_route(const float *logits, int B, int N, int mode, int k, int k0,
                 float p, int maxP, int kmax, int B_valid, const int *nbase_in,
                 int *idx, double *w, int *nbase, int *T, int *counts,
                 int *offsets, int *active, int *perm)
{
    if (B < 0 || N < 1 || k < 1 || k > N || B_valid < 0 || B_valid > B)
        return -1;
    if (mode == ORACLE_OEA && k0 <= 0)
        k0 = oracle_policy_k0(B_valid, k, &p);
    if (mode == ORACLE_OEA && (k0 < 1 || k0 > k || kmax < k0 || kmax > N ||
                               maxP < 1 || !(p > 0.0f)))
        return -1;
    if (mode != ORACLE_TOPK && mode != ORACLE_OEA)
        return -1;
    if (mode == ORACLE_OEA && nbase_in)
        for (int i = 0; i < B_valid; ++i)
            if (nbase_in[i] < 1 || nbase_in[i] > k0)
                return -1;
    const int kslots = (mode == ORACLE_TOPK) ? k : kmax;

    int *order = malloc(sizeof(int) * (size_t)N * (B > 0 ? B : 1));
    char *in_base = calloc((size_t)N, 1);
    char *sel = calloc((size_t)N * (B > 0 ? B : 1), 1);   /* sel[i][e] */
    int *slot_of = malloc(sizeof(int) * (size_t)N * (B > 0 ? B : 1));

    for (int i = 0; i < B; ++i)
        rank_experts(logits + (size_t)i * N, N, order + (size_t)i * N);

    for (size_t q = 0; q < (size_t)B * kslots; ++q) {
        idx[q] = -1;
        w[q] = 0.0;
    }

    if (mode == ORACLE_TOPK) {
        for (int i = 0; i < B; ++i) {
            nbase[i] = (i < B_valid) ? k : 0;
            for (int j = 0; j < nbase[i]; ++j)
                idx[(size_t)i * kslots + j] = order[(size_t)i * N + j];
        }
    } else {
        /* Phase 1: n_i = min(k0, t_i); baseline = the token's top-n_i. */
        for (int i = 0; i < B; ++i) {
            if (i >= B_valid) {
                nbase[i] = 0;
                continue;
            }
            const float *l = logits + (size_t)i * N;
            const int *o = order + (size_t)i * N;
            if (nbase_in) {
                nbase[i] = nbase_in[i];
            } else {
                int t = top_p_count(l, o, N, p);
                nbase[i] = t < k0 ? t : k0;
            }
            for (int j = 0; j < nbase[i]; ++j)
                in_base[o[j]] = 1;             /* S_base = union of baselines */
        }
        /* Phase 2: walk ranks nbase+1 .. maxP, keep experts already in S_base. */
        const int depth = maxP < N ? maxP : N;
        for (int i = 0; i < B; ++i) {
            const int *o = order + (size_t)i * N;
            int cnt = 0;
            for (int j = 0; j < nbase[i]; ++j)
                idx[(size_t)i * kslots + cnt++] = o[j];
            if (i >= B_valid)
                continue;
            for (int j = nbase[i]; j < depth && cnt < kmax; ++j)
                if (in_base[o[j]])
                    idx[(size_t)i * kslots + cnt++] = o[j];
        }
    }

    /* Renormalise the kept scores: softmax over the kept logits (fp64). */
    for (int i = 0; i < B; ++i) {
        const float *l = logits + (size_t)i * N;
        int *ii = idx + (size_t)i * kslots;
        double *ww = w + (size_t)i * kslots;
        if (ii[0] < 0)
            continue;
        double m = (double)l[ii[0]];
        double Z = 0.0;
        for (int j = 0; j < kslots && ii[j] >= 0; ++j)
            Z += exp((double)l[ii[j]] - m);
        for (int j = 0; j < kslots && ii[j] >= 0; ++j)
            ww[j] = exp((double)l[ii[j]] - m) / Z;
    }

    /* Per-expert loads, the active list and the grouping by expert. */
    for (int i = 0; i < B; ++i)
        for (int j = 0; j < kslots; ++j) {
            int e = idx[(size_t)i * kslots + j];
            if (e >= 0) {
                sel[(size_t)i * N + e] = 1;
                slot_of[(size_t)i * N + e] = j;
            }
        }
    int t_count = 0, pos = 0;
    for (int e = 0; e < N; ++e) {
        counts[e] = 0;
        offsets[e] = pos;
        for (int i = 0; i < B; ++i)
            if (sel[(size_t)i * N + e]) {
                perm[pos++] = i * kslots + slot_of[(size_t)i * N + e];
                counts[e]++;
            }
        if (counts[e] > 0)
            active[t_count++] = e;
    }
    offsets[N] = pos;
    for (int a = t_count; a < N; ++a)
        active[a] = -1;
    *T = t_count;

    free(order);
    free(in_base);
    free(sel);
    free(slot_of);
    return 0;
}

static double silu(double z)
{
    return z / (1.0 + exp(-z));
}

/* One expert on one token, fp64:
 *   g = W_gate x, u = W_up x   (W_gate, W_up: [F][d])
 *   h = silu(g) * u
 *   y = W_down h               (W_down: [d][F]) */
void oracle_expert_ffn(const float *x, const float *w_gate, const float *w_up,
                       const float *w_down, int d, int F, double *y)
{
    double *h = malloc(sizeof(double) * (size_t)F);
    for (int f = 0; f < F; ++f) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < d; ++c) {
            g += (double)w_gate[(size_t)f * d + c] * (double)x[c];
            u += (double)w_up[(size_t)f * d + c] * (double)x[c];
        }
        h[f] = silu(g) * u;
    }
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int f = 0; f < F; ++f)
            acc += (double)w_down[(size_t)j * F + f] * h[f];
        y[j] = acc;
    }
    free(h);
}

/* Whole expert stage + weighted combine for a batch whose routing is given:
 *   out[i] = sum over slots j (in slot order) of w[i][j] * FFN_{idx[i][j]}(x_i)
 * Expert e's matrices are the e-th [F][d] / [d][F] blocks of the arrays. */
void oracle_moe_experts(const float *x, const float *w_gate, const float *w_up,
                        const float *w_down, int B, int d, int F, int kslots,
                        const int *idx, const double *w, double *out)
{
    double *y = malloc(sizeof(double) * (size_t)d);
    const size_t esz = (size_t)F * d;
    for (int i = 0; i < B; ++i) {
        double *o = out + (size_t)i * d;
        for (int c = 0; c < d; ++c)
            o[c] = 0.0;
        for (int j = 0; j < kslots; ++j) {
            int e = idx[(size_t)i * kslots + j];
            if (e < 0)
                continue;
            oracle_expert_ffn(x + (size_t)i * d, w_gate + e * esz, w_up + e * esz,
                              w_down + e * esz, d, F, y);
            for (int c = 0; c < d; ++c)
                o[c] += w[(size_t)i * kslots + j] * y[c];
        }
    }
    free(y);
}

/* INT4 group-wise dequantisation of one packed matrix [rows][cols]:
 * w[r][c] = q[r][c] * s[r][c / 128], symmetric codes q in -7..7.
 * Packed format (chunks of rb rows x 128 columns -- one scale group -- in
 * row-block-major then column-group order; each chunk = rb*64 code bytes
 * then rb bf16 scales): within a chunk row r, local column c is the nibble
 * at bit 4*((c%8)/2) + 16*(c%2) of the little-endian 32-bit word c/8 of
 * the row's 64 bytes, stored as q + 8; the row's scale of the group
 * follows all code bytes, at r*2 bytes. */
void oracle_dequant_int4(const uint8_t *packed, int rows, int cols, int rb, float *out)
{
    const int nkb = cols / 128;
    const size_t chunk = (size_t)rb * 64 + (size_t)rb * 2;
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c) {
            const int rbi = r / rb, rr = r % rb, kb = c / 128, cl = c % 128;
            const uint8_t *ch = packed + ((size_t)rbi * nkb + kb) * chunk;
            const uint8_t *wp = ch + (size_t)rr * 64 + (size_t)(cl / 8) * 4;
            uint32_t word = (uint32_t)wp[0] | ((uint32_t)wp[1] << 8) | ((uint32_t)wp[2] << 16) |
                            ((uint32_t)wp[3] << 24);
            const int o = cl % 8;
            const int bit = 4 * (o / 2) + 16 * (o % 2);
            const int q = (int)((word >> bit) & 0xFu) - 8;
            const uint8_t *sp = ch + (size_t)rb * 64 + (size_t)rr * 2;   /* this row's group scale */
            uint32_t sb = ((uint32_t)sp[0] | ((uint32_t)sp[1] << 8)) << 16;
            float sc;
            memcpy(&sc, &sb, sizeof sc);
            out[(size_t)r * cols + c] = (float)q * sc;
        }
}

/*
 * Hotness and the high-precision set (DynaExq page, section 2.5 / 3.5):
 *   - EMA hotness per expert over update intervals:
 *       S_e <- alpha * S_e + (1 - alpha) * c_e,
 *     c_e = the times the router selected expert e in the interval;
 *   - the high-precision set has a fixed size (the layer's budget);
 *   - hysteresis: an expert outside the set is promoted only if its score
 *     exceeds the score of the lowest-ranked expert inside the set by the
 *     margin, and an expert inside is demoted only if its score is below
 *     that of the highest-ranked expert outside by the same margin.
 * With a fixed set size, every promotion pairs with a demotion: the best
 * outsider (highest score, ties to the lower id) replaces the weakest
 * insider (lowest score, ties to the higher id) while the outsider's score
 * exceeds the insider's by more than the margin.
 */
void oracle_ema_update(double *S, const double *c, int N, double alpha)
{
    for (int e = 0; e < N; ++e)
        S[e] = alpha * S[e] + (1.0 - alpha) * c[e];
}

/* in_hot[N] (0/1) is updated in place; promote[] / demote[] receive the
 * swaps in the order they are made; returns their number. */
int oracle_hot_select(const double *S, int N, double margin, unsigned char *in_hot,
                      int *promote, int *demote)
{
    int n = 0;
    for (;;) {
        int o = -1, i = -1;
        for (int e = 0; e < N; ++e) {
            if (!in_hot[e] && (o < 0 || S[e] > S[o]))
                o = e;                        /* first maximum: the lower id */
            if (in_hot[e] && (i < 0 || S[e] <= S[i]))
                i = e;                        /* last minimum: the higher id */
        }
        if (o < 0 || i < 0 || !(S[o] > S[i] + margin))
            return n;
        in_hot[o] = 1;
        in_hot[i] = 0;
        promote[n] = o;
        demote[n] = i;
        ++n;
    }
}
