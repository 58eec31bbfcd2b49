/*
 * spec_oracle.c -- plain, slow, fp64 CPU oracle for the speculative-decoding
 * verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline
 * leg use it.  It shares no code, header, table or constant generator with the
 * CUDA path in speculative_decoding_verification_36_gb300/csrc/.
 *
 * Every step follows the method as the source pages state it, in their order
 * and notation, and is written for a reader to check by eye: no blocking, no
 * fusion, no reordering.  Citations name the page and its section:
 *
 *   [P1] "Speculative Decoding & Draft Model Topologies: Slashing Enterprise LLM
 *        Latency by 3.5x in 2026", sec. 2 "Mathematical Foundation: Speculative
 *        Verification & Rejection Sampling" (acceptance probability
 *        alpha = min(1, p(x)/q(x)), draw u ~ U(0,1), discard on rejection, the
 *        residual max(0, p - q) / sum max(0, p - q)); sec. 4 (token tree, 2D
 *        tree mask, longest accepted path).
 *   [P2] "Speculative Decoding for LLM Inference: How Draft-and-Verify
 *        Accelerates Token Generation", sections "The draft-and-verify loop"
 *        (longest accepted prefix, resample on rejection, bonus token when all
 *        are accepted) and "The correctness guarantee" (min(1, p/q),
 *        norm(max(0, p - q))).
 *   [P3] "Speculative Decoding at Scale: Latency Reduction in Distributed LLM
 *        Serving", sequence diagram (accept matching tokens + 1 bonus token)
 *        and sec. 1 (relu(P - Q) / sum relu(P - Q)).
 *   [P4] "Speculative Decoding in Production: How Small Draft Models & Medusa
 *        Heads Deliver 2x-3x LLM Speedups Without Accuracy Loss", sec. 2
 *        (P_accept = min(1, p/q); p >= q always accepted) and sec. 4 (SpecInfer
 *        tree of top-2 candidates verified with a 2D causal mask).
 *
 * Where the pages are silent the oracle takes these readings (all of them are
 * also listed, with reasons, in the design notes):
 *   - p = softmax(z_target / tau), q = softmax(z_draft / tau), the same tau for
 *     both; tau == 0 selects greedy verification.
 *   - accept iff p(x) >= q(x) or u * q(x) < p(x)   (strict "<"; [P1] writes
 *     "u <= alpha"; with u on a grid of 2^-52 the two differ with
 *     probability at most 2^-52 per draw).
 *   - uniforms come from Philox-4x64-10 with key (seed, 0x5350454356455249)
 *     and counter (sequence b, position, stream, 0); stream 0 is the
 *     acceptance draw, stream 1 the resampling draw.  The first output word r
 *     maps to u = (2 * (r >> 12) + 1) * 2^-53, an odd multiple of 2^-53 in
 *     (0, 1), exact in fp64: the 52 top bits of r, so that a token of
 *     probability p is drawn with probability p to within 2^-52 (the method
 *     draws u from U(0, 1): [P1] sec. 2, [P2] "The correctness guarantee").
 *   - the replacement / bonus token is drawn by inverse CDF in vocabulary
 *     order: the smallest j with C_j > w * Z, C_j = sum_{v <= j} r(v).
 *   - greedy ties go to the lowest token id.
 *   - tree: row 0 is the root, row i + 1 is node i, parents precede children;
 *     the deepest accepted node wins, ties to the lowest node index.
 *   - bad data (NaN or +inf logit, all -inf row, token id outside [0, V),
 *     parent index not in [-1, i)) marks the sequence: n = -1 and all outputs
 *     of that sequence are -1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_DTYPE_F32 0
#define ORC_DTYPE_BF16 1

/* ------------------------------------------------------------------------ */
/* Philox-4x64-10 counter-based generator, written from its published        */
/* definition: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy */
/* as 1, 2, 3", SC'11.  Ten rounds; each round multiplies words 0 and 2 by   */
/* the two round multipliers, xors the high halves with the other two words  */
/* and the key, and the key is bumped by the two Weyl constants between      */
/* rounds.                                                                   */
/* ------------------------------------------------------------------------ */
static void philox_mulhilo(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo)
{
    unsigned __int128 prod = (unsigned __int128)a * (unsigned __int128)b;
    *hi = (uint64_t)(prod >> 64);
    *lo = (uint64_t)prod;
}

void oracle_philox4x64_10(const uint64_t ctr_in[4], const uint64_t key_in[2], uint64_t out[4])
{
    const uint64_t mult0 = 0xD2E7470EE14C6C93ULL;
    const uint64_t mult1 = 0xCA5A826395121157ULL;
    const uint64_t weyl0 = 0x9E3779B97F4A7C15ULL;
    const uint64_t weyl1 = 0xBB67AE8584CAA73BULL;
    uint64_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
    uint64_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t hi0, lo0, hi1, lo1;
        if (round > 0) {
            k0 += weyl0;
            k1 += weyl1;
        }
        philox_mulhilo(mult0, x0, &hi0, &lo0);
        philox_mulhilo(mult1, x2, &hi1, &lo1);
        uint64_t y0 = hi1 ^ x1 ^ k0;
        uint64_t y1 = lo1;
        uint64_t y2 = hi0 ^ x3 ^ k1;
        uint64_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* The uniform draw u ~ U(0,1) for (seed, sequence b, position, stream). */
double oracle_uniform(uint64_t seed, uint64_t b, uint64_t position, uint64_t stream)
{
    const uint64_t key[2] = {seed, 0x5350454356455249ULL};
    const uint64_t ctr[4] = {b, position, stream, 0};
    uint64_t out[4];
    oracle_philox4x64_10(ctr, key, out);
    const uint64_t top52 = out[0] >> 12;
    return (double)(2 * top52 + 1) * ldexp(1.0, -53);
}

/* ------------------------------------------------------------------------ */
/* logits                                                                    */
/* ------------------------------------------------------------------------ */
static double logit_at(const void *base, int dtype, size_t i)
{
    if (dtype == ORC_DTYPE_F32)
        return (double)((const float *)base)[i];
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* A row is usable when it has no NaN, no +inf and at least one finite entry. */
static int row_is_bad(const void *row, int dtype, int V)
{
    int any_finite_or_neg = 0;
    for (int v = 0; v < V; ++v) {
        double z = logit_at(row, dtype, (size_t)v);
        if (isnan(z) || z == INFINITY)
            return 1;
        if (z != -INFINITY)
            any_finite_or_neg = 1;
    }
    return !any_finite_or_neg;
}

/*
 * Temperature softmax of one row: p[v] = exp(z_v / tau - m) / s with
 * m = max_v z_v / tau and s = sum_v exp(z_v / tau - m).  ([P1] sec. 2 and
 * [P2] "The correctness guarantee": p and q are the two models' probabilities.)
 */
static void softmax_row(const void *row, int dtype, int V, double tau, double *p,
                        double *m_out, double *s_out)
{
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double x = logit_at(row, dtype, (size_t)v) / tau;
        if (x > m)
            m = x;
    }
    double s = 0.0;
    for (int v = 0; v < V; ++v) {
        double e = exp(logit_at(row, dtype, (size_t)v) / tau - m);
        p[v] = e;
        s += e;
    }
    for (int v = 0; v < V; ++v)
        p[v] = p[v] / s;
    *m_out = m;
    *s_out = s;
}

/* Inverse CDF in vocabulary order: the smallest j with C_j > theta, where C_j
 * is the running sum of r.  When rounding leaves no such j, the largest j with
 * r(j) > 0.  Also reports the distance from theta to the nearest C. */
static int inverse_cdf(const double *r, int V, double theta, double *dist_out)
{
    double c_prev = 0.0, c = 0.0;
    for (int j = 0; j < V; ++j) {
        c_prev = c;
        c = c + r[j];
        if (c > theta) {
            double d0 = theta - c_prev, d1 = c - theta;
            *dist_out = d0 < d1 ? d0 : d1;
            return j;
        }
    }
    for (int j = V - 1; j >= 0; --j) {
        if (r[j] > 0.0) {
            *dist_out = 0.0;
            return j;
        }
    }
    *dist_out = 0.0;
    return 0;
}

/*
 * Speculative-sampling verification of B independent sequences.
 *
 * target: B x (K+1) x V logits, sequence b at target + b * t_stride_b elements;
 * draft:  B x K x V logits, sequence b at draft + b * d_stride_b elements
 *         (a stride of 0 broadcasts one sequence to every b);
 * tokens: B x K drafted ids (row stride K);
 * seq_ids: optional B sequence numbers used as the Philox sequence counter
 *         (NULL: the batch index b), so that a subset of a batch can be
 *         verified with the uniforms the whole batch would draw;
 * out_tokens: B x (K+1), out_n: B.
 *
 * Optional diagnostics (each may be NULL):
 *   row_logmax, row_sum: B x (2K+1), target rows 0..K then draft rows 0..K-1;
 *                        the max of z / tau and sum exp(z / tau - max);
 *   px, qx, u, acc_margin: B x K, p_i(x_i), q_i(x_i), the acceptance draw and
 *                        |u - min(1, p/q)| (NaN for positions not examined);
 *   resid_mass, theta, w, sample_margin: B; Z = sum of the unnormalised
 *                        replacement weights, w * Z, w, and the distance from
 *                        w * Z to the nearest cumulative sum divided by Z;
 *   degenerate: B, 1 when a rejection left Z == 0 and p_n was used instead.
 *
 * Returns 0; sequences with bad data get n = -1 and -1 everywhere.
 */
/*
 * used_rows_only selects the early-exit reading of the bad-data rule: only
 * the rows the result depends on are checked, in position order -- target
 * and draft rows 0..n and the drafted tokens x_0..x_n, plus target row K when
 * all K drafts are accepted.  A bad position stops the scan and marks the
 * sequence bad; rows after the first rejection never matter.  Otherwise (the
 * default) every row and every drafted token is checked before anything else.
 */
int oracle_spec_verify(const void *target, const void *draft, int dtype,
                       long long t_stride_b, long long d_stride_b,
                       const int32_t *tokens, long long tok_stride_b,
                       int B, int K, int V, double tau, uint64_t seed,
                       const long long *seq_ids, int used_rows_only,
                       int32_t *out_tokens, int32_t *out_n,
                       double *row_logmax, double *row_sum,
                       double *px_out, double *qx_out, double *u_out, double *acc_margin,
                       double *resid_mass, double *theta_out, double *w_out,
                       double *sample_margin, int32_t *degenerate)
{
    const size_t esz = dtype == ORC_DTYPE_F32 ? 4 : 2;
    const int R = 2 * K + 1;
    double *probs = (double *)malloc(sizeof(double) * (size_t)R * (size_t)V);
    double *r = (double *)malloc(sizeof(double) * (size_t)V);
    int *rowbad = (int *)malloc(sizeof(int) * (size_t)R);
    if (!probs || !r || !rowbad) {
        free(probs);
        free(r);
        free(rowbad);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        const char *tb = (const char *)target + (size_t)((long long)b * t_stride_b) * esz;
        const char *db = (const char *)draft + (size_t)((long long)b * d_stride_b) * esz;
        const int32_t *x = tokens + (long long)b * tok_stride_b;
        const uint64_t seq = seq_ids ? (uint64_t)seq_ids[b] : (uint64_t)b;
        int32_t *out = out_tokens + (size_t)b * (size_t)(K + 1);
        for (int j = 0; j <= K; ++j)
            out[j] = -1;
        for (int i = 0; i < K && px_out; ++i) {
            px_out[(size_t)b * K + i] = NAN;
            qx_out[(size_t)b * K + i] = NAN;
        }
        for (int i = 0; i < K && acc_margin; ++i)
            acc_margin[(size_t)b * K + i] = NAN;
        for (int i = 0; i < K && u_out; ++i)
            u_out[(size_t)b * K + i] = NAN;
        if (resid_mass) resid_mass[b] = NAN;
        if (theta_out) theta_out[b] = NAN;
        if (w_out) w_out[b] = NAN;
        if (sample_margin) sample_margin[b] = NAN;
        if (degenerate) degenerate[b] = 0;

        /* bad data: any unusable row or an out-of-range drafted token */
        int bad = 0;
        for (int rr = 0; rr < R; ++rr) {
            const char *row = rr <= K ? tb + (size_t)rr * V * esz : db + (size_t)(rr - K - 1) * V * esz;
            rowbad[rr] = row_is_bad(row, dtype, V);
            if (!used_rows_only)
                bad = bad || rowbad[rr];
        }
        for (int i = 0; i < K && !bad && !used_rows_only; ++i)
            bad = x[i] < 0 || x[i] >= V;
        if (bad) {
            out_n[b] = -1;
            continue;
        }

        /* step 1: temperature softmax of every target row and draft row
         * (an unusable row is only ever used when it makes the sequence bad) */
        for (int rr = 0; rr < R; ++rr) {
            const char *row = rr <= K ? tb + (size_t)rr * V * esz : db + (size_t)(rr - K - 1) * V * esz;
            double m = NAN, s = NAN;
            if (!rowbad[rr])
                softmax_row(row, dtype, V, tau, probs + (size_t)rr * V, &m, &s);
            if (row_logmax) row_logmax[(size_t)b * R + rr] = m;
            if (row_sum) row_sum[(size_t)b * R + rr] = s;
        }
        const double *p_rows = probs;                        /* p_0 .. p_K */
        const double *q_rows = probs + (size_t)(K + 1) * V;  /* q_0 .. q_{K-1} */

        /* steps 2-4: gather p(x_i), q(x_i); accept with probability
         * min(1, p/q); stop at the first rejection */
        int n = K;
        for (int i = 0; i < K; ++i) {
            if (used_rows_only && (rowbad[i] || rowbad[K + 1 + i] || x[i] < 0 || x[i] >= V)) {
                bad = 1;
                break;
            }
            double p = p_rows[(size_t)i * V + x[i]];
            double q = q_rows[(size_t)i * V + x[i]];
            double u = oracle_uniform(seed, seq, (uint64_t)i, 0);
            double alpha = q > 0.0 ? fmin(1.0, p / q) : 1.0;
            if (px_out) {
                px_out[(size_t)b * K + i] = p;
                qx_out[(size_t)b * K + i] = q;
            }
            if (u_out) u_out[(size_t)b * K + i] = u;
            if (acc_margin) acc_margin[(size_t)b * K + i] = fabs(u - alpha);
            int accept = (p >= q) || (u * q < p);
            if (!accept) {
                n = i;
                break;
            }
            out[i] = x[i];
        }

        if (used_rows_only && !bad && n == K && rowbad[K])
            bad = 1;
        if (bad) {
            for (int j = 0; j <= K; ++j)
                out[j] = -1;
            out_n[b] = -1;
            continue;
        }

        /* step 5: the replacement distribution max(0, p_n - q_n) after a
         * rejection, or the bonus distribution p_K when all K were accepted */
        double Z = 0.0;
        if (n < K) {
            for (int v = 0; v < V; ++v) {
                double d = p_rows[(size_t)n * V + v] - q_rows[(size_t)n * V + v];
                r[v] = d > 0.0 ? d : 0.0;
                Z += r[v];
            }
            if (Z == 0.0) {
                if (degenerate) degenerate[b] = 1;
                for (int v = 0; v < V; ++v) {
                    r[v] = p_rows[(size_t)n * V + v];
                    Z += r[v];
                }
            }
        } else {
            for (int v = 0; v < V; ++v) {
                r[v] = p_rows[(size_t)K * V + v];
                Z += r[v];
            }
        }

        /* step 6: inverse-CDF draw with the stream-1 uniform */
        double w = oracle_uniform(seed, seq, (uint64_t)n, 1);
        double theta = w * Z;
        double dist;
        int j = inverse_cdf(r, V, theta, &dist);
        out[n] = j;
        out_n[b] = n;
        if (resid_mass) resid_mass[b] = Z;
        if (theta_out) theta_out[b] = theta;
        if (w_out) w_out[b] = w;
        if (sample_margin) sample_margin[b] = dist / Z;
    }
    free(probs);
    free(r);
    free(rowbad);
    return 0;
}

/* First index of the maximum of a row (lowest id wins ties). */
static int row_argmax(const void *row, int dtype, int V)
{
    int best = 0;
    double best_z = logit_at(row, dtype, 0);
    for (int v = 1; v < V; ++v) {
        double z = logit_at(row, dtype, (size_t)v);
        if (z > best_z) {
            best_z = z;
            best = v;
        }
    }
    return best;
}

/*
 * Greedy verification (tau == 0): accept drafted tokens while they equal the
 * target argmax ([P3] "accept matching tokens ... + 1 bonus token", "reject
 * mismatched"); the token after the accepted prefix is the argmax of that
 * target row, which is the bonus token when all K match.
 * Layouts as in oracle_spec_verify; draft logits are not read.
 */
/*
 * used_rows_only: the early-exit reading, as for the sampled verify above --
 * positions are examined in order and only what the result uses is checked:
 * target row i (NaN / +inf / no finite maximum), then x_i outside [0, V), then
 * x_i against the argmax of row i; the first mismatch is n, and target row K
 * is checked only when all K drafts match.  A bad position stops the scan and
 * marks the sequence bad.  row_argmax_out then holds the argmax of rows 0..n
 * and -1 after n.
 */
int oracle_spec_verify_greedy(const void *target, int dtype, long long t_stride_b,
                              const int32_t *tokens, long long tok_stride_b,
                              int B, int K, int V, int used_rows_only,
                              int32_t *out_tokens, int32_t *out_n, int32_t *row_argmax_out)
{
    const size_t esz = dtype == ORC_DTYPE_F32 ? 4 : 2;
    for (int b = 0; b < B; ++b) {
        const char *tb = (const char *)target + (size_t)((long long)b * t_stride_b) * esz;
        const int32_t *x = tokens + (long long)b * tok_stride_b;
        int32_t *out = out_tokens + (size_t)b * (size_t)(K + 1);
        for (int j = 0; j <= K; ++j)
            out[j] = -1;
        if (used_rows_only) {
            int n = K, bad = 0, last = -1;
            for (int i = 0; i <= K; ++i) {
                const char *row = tb + (size_t)i * V * esz;
                if (row_is_bad(row, dtype, V)) {
                    bad = 1;
                    break;
                }
                const int a = row_argmax(row, dtype, V);
                if (row_argmax_out) row_argmax_out[(size_t)b * (K + 1) + i] = a;
                last = i;
                if (i == K)
                    break;
                if (x[i] < 0 || x[i] >= V) {
                    bad = 1;
                    break;
                }
                if (x[i] != a) {
                    n = i;
                    break;
                }
            }
            for (int rr = last + 1; rr <= K && row_argmax_out; ++rr)
                row_argmax_out[(size_t)b * (K + 1) + rr] = -1;
            if (bad) {
                out_n[b] = -1;
                continue;
            }
            for (int i = 0; i < n; ++i)
                out[i] = x[i];
            out[n] = row_argmax(tb + (size_t)n * V * esz, dtype, V);
            out_n[b] = n;
            continue;
        }
        int bad = 0;
        for (int rr = 0; rr <= K && !bad; ++rr)
            bad = row_is_bad(tb + (size_t)rr * V * esz, dtype, V);
        for (int i = 0; i < K && !bad; ++i)
            bad = x[i] < 0 || x[i] >= V;
        if (bad) {
            out_n[b] = -1;
            for (int rr = 0; rr <= K && row_argmax_out; ++rr)
                row_argmax_out[(size_t)b * (K + 1) + rr] = -1;
            continue;
        }
        int n = K;
        for (int rr = 0; rr <= K; ++rr) {
            int a = row_argmax(tb + (size_t)rr * V * esz, dtype, V);
            if (row_argmax_out) row_argmax_out[(size_t)b * (K + 1) + rr] = a;
        }
        for (int i = 0; i < K; ++i) {
            int a = row_argmax(tb + (size_t)i * V * esz, dtype, V);
            if (x[i] != a) {
                n = i;
                break;
            }
            out[i] = x[i];
        }
        out[n] = row_argmax(tb + (size_t)n * V * esz, dtype, V);
        out_n[b] = n;
    }
    return 0;
}

/*
 * Greedy verification of a candidate tree ([P1] sec. 4: all nodes verified in
 * one pass, the longest accepted path is selected; [P4] sec. 4: a SpecInfer
 * tree of top-2 candidates under a 2D causal mask).
 *
 * target: B x (N+1) x V; row 0 is the root's next-token row, row i+1 belongs
 * to node i.  tree_tokens, parent_idx: B x N; parent -1 is the root.
 * Node i is accepted when every node on its root path carries the argmax of
 * its parent's row.  Outputs: out_path B x (N+1) token ids (the accepted path
 * from the root's child down, then the bonus argmax of the deepest accepted
 * node's row, -1 padding), out_len B (path length + 1), out_mask
 * B x N x ceil(N/32) words with bit j of row i set iff j == i or j is an
 * ancestor of i.  Everything is computed by explicit ancestor walks.
 *
 * used_rows_only: the early-exit reading -- only what the result depends on
 * is checked.  Every parent index (the mask depends on all of them), the
 * root's row, the token of every node whose parent is accepted (it is
 * compared with the parent's argmax) and the row of every accepted node (its
 * argmax judges its children, or is the bonus token) are checked; the rows
 * and tokens under a rejected node are never examined.
 */
int oracle_tree_verify_greedy(const void *target, int dtype, const int32_t *tree_tokens,
                              const int32_t *parent_idx, int B, int N, int V, int used_rows_only,
                              int32_t *out_path, int32_t *out_len, uint32_t *out_mask)
{
    const size_t esz = dtype == ORC_DTYPE_F32 ? 4 : 2;
    const int W = (N + 31) / 32;
    int *g = (int *)malloc(sizeof(int) * (size_t)(N + 1));
    int *acc = (int *)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
    int *depth = (int *)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
    int *walk = (int *)malloc(sizeof(int) * (size_t)(N + 1));
    if (!g || !acc || !depth || !walk) {
        free(g); free(acc); free(depth); free(walk);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        const char *tb = (const char *)target + (size_t)b * (size_t)(N + 1) * V * esz;
        const int32_t *tok = tree_tokens + (size_t)b * N;
        const int32_t *par = parent_idx + (size_t)b * N;
        int32_t *path = out_path + (size_t)b * (size_t)(N + 1);
        uint32_t *mask = out_mask + (size_t)b * (size_t)N * W;
        for (int j = 0; j <= N; ++j)
            path[j] = -1;
        for (size_t w = 0; w < (size_t)N * W; ++w)
            mask[w] = 0;
        int bad = 0;
        if (used_rows_only) {
            /* top-down: a node's row is examined only once the node is accepted */
            for (int i = 0; i < N && !bad; ++i)
                bad = par[i] < -1 || par[i] >= i;
            if (!bad)
                bad = row_is_bad(tb, dtype, V);
            if (!bad)
                g[0] = row_argmax(tb, dtype, V);
            for (int i = 0; i < N && !bad; ++i) {
                const int p = par[i];
                if (p >= 0 && !acc[p]) {
                    acc[i] = 0;
                    continue;
                }
                if (tok[i] < 0 || tok[i] >= V) {
                    bad = 1;
                    break;
                }
                acc[i] = tok[i] == g[p + 1];
                if (acc[i]) {
                    const char *row = tb + (size_t)(i + 1) * V * esz;
                    bad = row_is_bad(row, dtype, V);
                    if (!bad)
                        g[i + 1] = row_argmax(row, dtype, V);
                }
            }
            if (bad) {
                out_len[b] = -1;
                continue;
            }
        } else {
            for (int rr = 0; rr <= N && !bad; ++rr)
                bad = row_is_bad(tb + (size_t)rr * V * esz, dtype, V);
            for (int i = 0; i < N && !bad; ++i)
                bad = par[i] < -1 || par[i] >= i || tok[i] < 0 || tok[i] >= V;
            if (bad) {
                out_len[b] = -1;
                continue;
            }
            for (int rr = 0; rr <= N; ++rr)
                g[rr] = row_argmax(tb + (size_t)rr * V * esz, dtype, V);
        }
        /* acceptance and depth of every node by walking its ancestors (with
         * used_rows_only a node is accepted only after its parent is, so
         * every g the walk reads was computed) */
        for (int i = 0; i < N; ++i) {
            int ok = 1, d = 0;
            for (int node = i; node != -1; node = par[node]) {
                int prow = par[node] + 1; /* parent -1 (root) uses row 0 */
                if (used_rows_only ? !acc[node] : tok[node] != g[prow])
                    ok = 0;
                d += 1;
            }
            acc[i] = ok;
            depth[i] = d;
        }
        int best = -1, best_depth = 0;
        for (int i = 0; i < N; ++i)
            if (acc[i] && depth[i] > best_depth) {
                best = i;
                best_depth = depth[i];
            }
        /* path tokens root -> best, then the bonus token */
        int len = 0;
        for (int node = best; node != -1; node = par[node])
            walk[len++] = node;
        for (int k = 0; k < len; ++k)
            path[k] = tok[walk[len - 1 - k]];
        path[len] = g[best + 1];
        out_len[b] = len + 1;
        /* ancestor mask */
        for (int i = 0; i < N; ++i)
            for (int node = i; node != -1; node = par[node])
                mask[(size_t)i * W + (size_t)(node / 32)] |= 1u << (node % 32);
    }
    free(g); free(acc); free(depth); free(walk);
    return 0;
}

/*
 * Acceptance statistics over a batch of verify outputs
 *   [P2] "How much speedup to expect": the per-position acceptance rate alpha
 *   and the expected number of tokens per draft-and-verify iteration.
 * hist[j] = number of sequences with n_accepted == j (j = 0..K); hist[K+1]
 * counts the rest (bad sequences, n = -1, or values outside [0, K]).
 * alpha[i] = #(n > i) / #(n >= i) over the counted sequences: of the sequences
 * whose position i was tested, the fraction that accepted it (NaN when none
 * reached position i).  *mean_tokens = mean of n + 1 over the counted
 * sequences (NaN when there are none).
 */
void oracle_acceptance_stats(const int32_t *n_accepted, int B, int K, uint64_t *hist,
                             double *alpha, double *mean_tokens)
{
    for (int j = 0; j <= K + 1; ++j)
        hist[j] = 0;
    for (int b = 0; b < B; ++b) {
        int n = n_accepted[b];
        if (n >= 0 && n <= K)
            hist[n] += 1;
        else
            hist[K + 1] += 1;
    }
    for (int i = 0; i < K; ++i) {
        uint64_t reached = 0, accepted = 0;
        for (int j = i; j <= K; ++j)
            reached += hist[j];
        for (int j = i + 1; j <= K; ++j)
            accepted += hist[j];
        alpha[i] = reached ? (double)accepted / (double)reached : NAN;
    }
    uint64_t count = 0;
    double total = 0.0;
    for (int j = 0; j <= K; ++j) {
        count += hist[j];
        total += (double)hist[j] * (double)(j + 1);
    }
    *mean_tokens = count ? total / (double)count : NAN;
}

/*
 * Entropy (nats) of p = softmax(z / tau) for each of `rows` rows of V logits
 *   [P3] "Speculative Decoding at Scale: Latency Reduction in Distributed LLM
 *   Serving", sec. 3 "Engineering Recommendations" (speculation depth chosen
 *   from how uncertain the distribution is); the entropy H = -sum_v p(v) ln p(v)
 *   is the plain measure of that uncertainty.
 * Terms with p(v) == 0 contribute 0.  A row with a NaN or +inf logit or no
 * finite logit gets NaN.
 */
void oracle_row_entropy(const void *logits, int dtype, long long rows, int V, double tau,
                        double *out)
{
    double *p = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    for (long long r = 0; r < rows; ++r) {
        const char *row = (const char *)logits + (size_t)r * (size_t)V * (dtype == ORC_DTYPE_F32 ? 4 : 2);
        if (row_is_bad(row, dtype, V)) {
            out[r] = NAN;
            continue;
        }
        double m, ssum;
        softmax_row(row, dtype, V, tau, p, &m, &ssum);
        double h = 0.0;
        for (int v = 0; v < V; ++v)
            if (p[v] > 0.0)
                h -= p[v] * log(p[v]);
        out[r] = h;
    }
    free(p);
}

/*
 * Suggested draft length for each sequence's next iteration, from the entropy
 * of the target distributions this iteration consulted
 *   [P3] "Speculative Decoding at Scale: Latency Reduction in Distributed LLM
 *   Serving", sec. 3 "Engineering Recommendations" (speculation depth tuning:
 *   a shorter draft where the text is uncertain, a longer one where it is
 *   predictable); [P2] "How much speedup to expect" (the draft length trades
 *   tokens per iteration against wasted work on rejections).
 * The page gives no formula; the rule here is the plain reading of it:
 *   Hbar_b = (1 / (n_b + 1)) * sum_{i=0..n_b} H(p_{b,i}),
 * the mean entropy (nats) of target rows 0..n_b -- the rows whose verdicts
 * (acceptances, then the rejection or the bonus) made this iteration's
 * tokens -- and
 *   K_next = clamp(K + 1, k_min, k_max)  when Hbar_b < h_lo,
 *            clamp(K - 1, k_min, k_max)  when Hbar_b > h_hi,
 *            clamp(K,     k_min, k_max)  otherwise (also for a NaN mean).
 * target_entropy: B x (K+1), row i of sequence b = H(p_{b,i}); n: B (-1 marks a
 * bad sequence, which gets K_next = -1 and a NaN mean).  The caller
 * guarantees 0 <= k_min <= k_max and h_lo <= h_hi.
 */
void oracle_adaptive_k(const double *target_entropy, const int32_t *n, int B, int K, double h_lo,
                       double h_hi, int k_min, int k_max, int32_t *out_k, double *out_hmean)
{
    for (int b = 0; b < B; ++b) {
        const int nb = n[b];
        if (nb < 0 || nb > K) {
            out_k[b] = -1;
            out_hmean[b] = NAN;
            continue;
        }
        double sum = 0.0;
        for (int i = 0; i <= nb; ++i)
            sum += target_entropy[(size_t)b * (size_t)(K + 1) + (size_t)i];
        const double hbar = sum / (double)(nb + 1);
        int k = K;
        if (hbar < h_lo)
            k = K + 1;
        else if (hbar > h_hi)
            k = K - 1;
        if (k < k_min)
            k = k_min;
        if (k > k_max)
            k = k_max;
        out_k[b] = k;
        out_hmean[b] = hbar;
    }
}

/*
 * Stochastic (temperature > 0) verification of a token tree per sequence.
 *   [P4] sec. 4 "Tree-Based Speculative Verification & Custom 2D Attention
 *   Masks" (a tree of candidates verified in one target pass, the longest
 *   accepted path kept) with the acceptance rule and residual of [P1] sec. 2 /
 *   [P2] "The correctness guarantee", applied node by node: the children of the
 *   current node are tried in index order, each against the current target
 *   distribution P; a rejected child replaces P by norm(max(0, P - Q)) before the
 *   next sibling is tried.  When no child is accepted (or the node is a leaf) one
 *   token is drawn from the current P.
 *
 * target, draft: B x (N+1) x V; row 0 is the root, row i+1 node i.  At node u,
 *   P = softmax(target row u / tau) and Q = softmax(draft row u / tau), Q being
 *   the distribution u's children were drawn from.
 * tree_tokens, parents: B x N; parents[i] in [-1, i) (-1: the root).
 * Draws: child c's acceptance uniform uses counter (b, c, 0, 0); the final draw
 *   at the stopping node uses (b, row of the node, 1, 0).
 * out_path: B x (N+1): accepted tokens root to leaf, then the drawn token, -1
 *   after; out_len: B, the number of entries written (depth + 1).
 * boundary (may be NULL): B x (N+1), entry [b][j] 1 when a draw that decided
 *   path entry j (the acceptance tests of the children of the node at depth
 *   j, or the final draw when the walk stops there) lies within 1e-6 of its
 *   decision boundary (|u - min(1, P(x)/Q(x))|, or the distance of w * Z to
 *   the nearest cumulative sum relative to Z); a diagnostic only.
 * Bad data (any bad row of the sequence, a token outside [0, V), a parent not in
 * [-1, i)) gives out_len = -1 and -1 everywhere.  Returns 0, or -1 if memory
 * could not be allocated.
 */
int oracle_tree_verify_sampling(const void *target, const void *draft, int dtype,
                                const int32_t *tree_tokens, const int32_t *parents, int B, int N,
                                int V, double tau, uint64_t seed, int32_t *out_path,
                                int32_t *out_len, int32_t *boundary)
{
    const size_t esz = dtype == ORC_DTYPE_F32 ? 4 : 2;
    const size_t rowb = (size_t)V * esz;
    double *P = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    double *Q = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    double *R = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    if (!P || !Q || !R) {
        free(P); free(Q); free(R);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        const char *T = (const char *)target + (size_t)b * (size_t)(N + 1) * rowb;
        const char *D = (const char *)draft + (size_t)b * (size_t)(N + 1) * rowb;
        const int32_t *tok = tree_tokens + (size_t)b * N;
        const int32_t *par = parents + (size_t)b * N;
        int32_t *path = out_path + (size_t)b * (N + 1);
        for (int j = 0; j <= N; ++j)
            path[j] = -1;
        int32_t *bnd = boundary ? boundary + (size_t)b * (N + 1) : NULL;
        if (bnd)
            for (int j = 0; j <= N; ++j)
                bnd[j] = 0;
        int bad = 0;
        for (int r = 0; r <= N; ++r)
            if (row_is_bad(T + r * rowb, dtype, V) || row_is_bad(D + r * rowb, dtype, V))
                bad = 1;
        for (int i = 0; i < N; ++i)
            if (tok[i] < 0 || tok[i] >= V || par[i] < -1 || par[i] >= i)
                bad = 1;
        if (bad) {
            out_len[b] = -1;
            continue;
        }
        int u = -1, len = 0;
        double m, s;
        softmax_row(T, dtype, V, tau, P, &m, &s);
        softmax_row(D, dtype, V, tau, Q, &m, &s);
        for (;;) {
            int accepted = -1;
            for (int c = 0; c < N; ++c) {
                if (par[c] != u)
                    continue;
                const int x = tok[c];
                const double r = oracle_uniform(seed, (uint64_t)b, (uint64_t)c, 0);
                const int ok = P[x] >= Q[x] || r * Q[x] < P[x];
                if (bnd && Q[x] > 0.0) {
                    double a = P[x] / Q[x];
                    if (a > 1.0)
                        a = 1.0;
                    if (fabs(r - a) < 1e-6)
                        bnd[len] = 1;
                }
                if (ok) {
                    accepted = c;
                    break;
                }
                /* rejected: P <- norm(max(0, P - Q)) for the next sibling */
                double z = 0.0;
                for (int v = 0; v < V; ++v) {
                    R[v] = P[v] > Q[v] ? P[v] - Q[v] : 0.0;
                    z += R[v];
                }
                if (z > 0.0)
                    for (int v = 0; v < V; ++v)
                        P[v] = R[v] / z;
            }
            if (accepted < 0)
                break;
            path[len++] = tok[accepted];
            u = accepted;
            softmax_row(T + (size_t)(u + 1) * rowb, dtype, V, tau, P, &m, &s);
            softmax_row(D + (size_t)(u + 1) * rowb, dtype, V, tau, Q, &m, &s);
        }
        double z = 0.0;
        for (int v = 0; v < V; ++v)
            z += P[v];
        const double w = oracle_uniform(seed, (uint64_t)b, (uint64_t)(u + 1), 1);
        double dist;
        const int32_t drawn = inverse_cdf(P, V, w * z, &dist);
        if (bnd && dist < 1e-6 * z)
            bnd[len] = 1;
        path[len++] = drawn;
        out_len[b] = len;
    }
    free(P); free(Q); free(R);
    return 0;
}

/*
 * N-gram (prompt-lookup) drafting
 *   [P2] "Speculative Decoding for LLM Inference: How Draft-and-Verify
 *   Accelerates Token Generation", sections "The variant landscape" and
 *   "Support in production systems", and the FAQ "Do all variants require a
 *   separate draft model?": candidate continuations are copied from the prompt
 *   or the output so far through an n-gram lookup, with no drafter weights.
 * Reading (the pages fix no rule): for each sequence b with history
 * tokens[b][0 .. L-1], try the match length m = n_max, n_max - 1, ..., n_min.
 * For the first m that occurs, take the latest earlier occurrence of the last
 * m tokens: the largest end e (exclusive, e <= L - 1, so at least one token
 * follows it) with tokens[e - m .. e - 1] == tokens[L - m .. L - 1].  The
 * drafts are the tokens that follow it, tokens[e .. e + d - 1] with
 * d = min(K, L - e).  Outputs: drafts [B, K] (-1 past d), n_drafts [B] = d
 * (0 when nothing matches), match_len [B] = m (0 when nothing matches).  A
 * length outside [0, stride] marks the sequence bad: n_drafts = match_len = -1
 * and every draft -1.  Token values are compared and copied as given.
 */
int oracle_ngram_draft(const int32_t *tokens, long long stride, const int32_t *lengths, int B, int n_min,
                       int n_max, int K, int32_t *drafts, int32_t *n_drafts, int32_t *match_len)
{
    for (int b = 0; b < B; ++b) {
        const int32_t *h = tokens + (long long)b * stride;
        const long long L = lengths[b];
        for (int i = 0; i < K; ++i)
            drafts[(long long)b * K + i] = -1;
        if (L < 0 || L > stride) {
            n_drafts[b] = -1;
            match_len[b] = -1;
            continue;
        }
        n_drafts[b] = 0;
        match_len[b] = 0;
        long long found_e = -1;
        int found_m = 0;
        for (int m = n_max; m >= n_min && found_e < 0; --m) {
            if (L < (long long)m + 1)
                continue;  /* no room for the suffix and one earlier token */
            for (long long e = L - 1; e >= m; --e) {
                int same = 1;
                for (int t = 0; t < m; ++t) {
                    if (h[e - m + t] != h[L - m + t]) {
                        same = 0;
                        break;
                    }
                }
                if (same) {
                    found_e = e;
                    found_m = m;
                    break;
                }
            }
        }
        if (found_e < 0)
            continue;
        long long d = L - found_e;
        if (d > K)
            d = K;
        for (long long i = 0; i < d; ++i)
            drafts[(long long)b * K + i] = h[found_e + i];
        n_drafts[b] = (int32_t)d;
        match_len[b] = found_m;
    }
    return 0;
}
