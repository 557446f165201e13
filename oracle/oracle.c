/*
 * oracle.c - plain, slow reference of the speculative-decoding verify step,
 * written in C and double precision.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's
 * CPU-baseline / reference arm are the only code allowed to load this library.
 * The CUDA library and its Python binding never call it, include it or share
 * any code with it.
 *
 * Sources (page title, section):
 *  [Maga]      "Inference-4" (brunomaga.github.io), "Draft-model speculative
 *              decoding": the step reads the target distribution at the K draft
 *              positions plus one more after the last draft; drafts are checked
 *              left to right; greedy rule, sampling rule, residual, bonus; and
 *              the greedy loop listing (argmax, match prefix, commit drafts[:n]
 *              followed by predictions[n]).
 *  [Monigatti] "Speculative decoding" (leoniemonigatti.com blog), "Rejection
 *              sampling": accept with probability min(1, p/q) where p is the
 *              target and q the draft; the residual norm(max(0, p - q)); bonus
 *              token when every draft is accepted.
 *  [Patel]     "Speculative decoding" (denimpatel.github.io interactive
 *              course), "Why this is not approximate": same rule, residual
 *              proportional to max(0, p - q), renormalised.
 *  [Atomic]    "What is speculative decoding?" (atomic.chat guide), "How
 *              speculative decoding works": p(x) >= q(x) is always accepted;
 *              verification stops at the first rejection.
 *  [SC11]      Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
 *              as 1, 2, 3", SC'11: the Philox4x32-10 counter-based generator.
 *
 * Notation: P_t is the target distribution, P_d the draft distribution (the
 * pages disagree on which is called p and which q; the rule itself is the
 * same everywhere: accept x with probability min(1, P_t(x) / P_d(x))).
 *
 * Readings where the pages are silent (each one is also listed in the design
 * notes):
 *  - Both distributions are softmax(logits / T) at the call's temperature T;
 *    greedy mode ignores T and compares raw logits.
 *  - The accept test is the strict u * P_d(x) < P_t(x) with
 *    u = (w0 >> 8) * 2^-24 from Philox, which accepts with probability
 *    min(1, P_t(x)/P_d(x)) up to the 2^-24 grid of u, and needs no division.
 *  - argmax breaks ties toward the lowest index (the first occurrence, as
 *    torch.argmax does in the greedy listing).
 *  - Inverse CDF in index order 0..V-1: the token is the smallest k whose
 *    cumulative mass exceeds t = u2 * (total mass).
 *  - A residual that sums to zero after a rejection (possible only through
 *    rounding) falls back to a draw from P_t of the same row.
 *  - A sequence is invalid (n_accepted = -1, every token -1) when a draft
 *    token lies outside [0, V) or when a row the step reads has no finite
 *    maximum (all -inf, or +inf / NaN present at the maximum).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };
enum { ORC_GREEDY = 0, ORC_SAMPLE = 1 };

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 [SC11]: ten rounds of the Philox S-box on a 4x32-bit counter */
/* with a 2x32-bit key; the key is bumped by the Weyl constants between       */
/* rounds.                                                                   */
/* ------------------------------------------------------------------------- */
static const uint32_t PHILOX_M0 = 0xD2511F53u;
static const uint32_t PHILOX_M1 = 0xCD9E8D57u;
static const uint32_t PHILOX_W0 = 0x9E3779B9u;
static const uint32_t PHILOX_W1 = 0xBB67AE85u;

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                          uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t prod0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The draw for sequence id `seq` at draft position `pos`: counter
 * (pos, seq_lo, seq_hi, 0), key (seed_lo, seed_hi). Word 0 gives the accept
 * uniform u, word 1 the uniform u2 of the residual or bonus draw. Both are
 * the top 24 bits scaled by 2^-24, so they are exact in float and double. */
static void draw_uniforms(uint64_t seed, uint64_t seq, uint32_t pos,
                          double* u, double* u2) {
    uint32_t ctr[4] = {pos, (uint32_t)seq, (uint32_t)(seq >> 32), 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    *u = (double)(w[0] >> 8) * (1.0 / 16777216.0);
    *u2 = (double)(w[1] >> 8) * (1.0 / 16777216.0);
}

void oracle_philox_uniforms(uint64_t seed, const uint64_t* seq_ids, int n_seq,
                            int n_pos, double* out_u, double* out_u2) {
    for (int b = 0; b < n_seq; ++b)
        for (int p = 0; p < n_pos; ++p)
            draw_uniforms(seed, seq_ids[b], (uint32_t)p,
                          &out_u[(size_t)b * n_pos + p],
                          &out_u2[(size_t)b * n_pos + p]);
}

/* ------------------------------------------------------------------------- */
/* Row access: fp32, bf16 (widened exactly: its bits are the top half of a    */
/* float) or fp64 logits, rows of V contiguous elements.                      */
/* ------------------------------------------------------------------------- */
static double logit_at(const void* base, int dtype, size_t i) {
    if (dtype == ORC_F32) return (double)((const float*)base)[i];
    if (dtype == ORC_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return ((const double*)base)[i];
}

/* Largest logit of a row and its lowest index. */
static double row_max(const void* base, int dtype, size_t row_off, int V,
                      int* argmax) {
    double best = logit_at(base, dtype, row_off);
    int idx = 0;
    for (int v = 1; v < V; ++v) {
        double l = logit_at(base, dtype, row_off + (size_t)v);
        if (l > best) {  /* strict: a tie keeps the earlier index */
            best = l;
            idx = v;
        }
    }
    if (argmax) *argmax = idx;
    return best;
}

/* A row is usable when its maximum is a finite number and no element is NaN
 * or +inf. */
static int row_valid(const void* base, int dtype, size_t row_off, int V) {
    int any_finite = 0;
    for (int v = 0; v < V; ++v) {
        double l = logit_at(base, dtype, row_off + (size_t)v);
        if (isnan(l) || (isinf(l) && l > 0)) return 0;
        if (isfinite(l)) any_finite = 1;
    }
    return any_finite;
}

/* Softmax at temperature T: P(v) = exp((l_v - m)/T) / sum_w exp((l_w - m)/T)
 * with m the row maximum; the sum runs sequentially over v = 0..V-1. */
static void row_softmax(const void* base, int dtype, size_t row_off, int V,
                        double T, double* P) {
    double m = row_max(base, dtype, row_off, V, NULL);
    double S = 0.0;
    for (int v = 0; v < V; ++v) {
        double e = exp((logit_at(base, dtype, row_off + (size_t)v) - m) / T);
        P[v] = e;
        S += e;
    }
    for (int v = 0; v < V; ++v) P[v] /= S;
}

/* Inverse CDF in index order: the smallest k with sum_{v<=k} r_v > t, where
 * t = u2 * sum_v r_v. Writes the distances from t down to the lower and up to
 * the upper edge of the chosen token's interval (in the units of r) to
 * edges[0], edges[1], and the smaller of the two to *margin. */
static int inverse_cdf(const double* r, int V, double u2, double* total_out,
                       double* margin, double edges[2]) {
    double total = 0.0;
    for (int v = 0; v < V; ++v) total += r[v];
    double t = u2 * total;
    double cum = 0.0;
    int last_positive = -1;
    for (int v = 0; v < V; ++v) {
        double prev = cum;
        cum += r[v];
        if (r[v] > 0.0) last_positive = v;
        if (cum > t) {
            double d0 = t - prev, d1 = cum - t;
            *margin = d0 < d1 ? d0 : d1;
            edges[0] = d0;
            edges[1] = d1;
            *total_out = total;
            return v;
        }
    }
    /* Only reachable through rounding: take the last token with mass. */
    *margin = 0.0;
    edges[0] = edges[1] = 0.0;
    *total_out = total;
    return last_positive;
}

/* Per-sequence results besides the committed tokens. */
typedef struct {
    double accept_margin; /* min over tested positions of |u*P_d - P_t| / P_d */
    double draw_margin;   /* distance of t to the chosen interval's edges     */
    double draw_edges[2]; /* t's distances to the lower and the upper edge    */
    double residual_mass; /* sum of the distribution the final draw used      */
    int fallback;         /* 1 when a zero residual fell back to P_t          */
} seq_extra;

/* Verify one sequence with the uniforms given explicitly.
 *   tgt: the K+1 target rows, drf: the K draft rows (unused when greedy),
 *   x: K draft tokens, u[0..K-1]: accept uniforms, u2[0..K]: draw uniforms.
 * Output: tokens[0..K] = x_0..x_{j-1}, then the correction or bonus token,
 * then -1; returns j = number of accepted drafts, or -1 if invalid. */
static int verify_sequence(const void* tgt, size_t tgt_off, const void* drf,
                           size_t drf_off, int dtype_t, int dtype_d,
                           const int32_t* x, int K, int V, int mode, double T,
                           const double* u, const double* u2, int32_t* tokens,
                           double* p_t_at_x, double* p_d_at_x, seq_extra* ex,
                           double* Pt, double* Pd, double* r) {
    ex->accept_margin = INFINITY;
    ex->draw_margin = INFINITY;
    ex->draw_edges[0] = ex->draw_edges[1] = NAN;
    ex->residual_mass = NAN;
    ex->fallback = 0;
    for (int i = 0; i <= K; ++i) tokens[i] = -1;
    for (int i = 0; i < K; ++i) {
        if (p_t_at_x) p_t_at_x[i] = NAN;
        if (p_d_at_x) p_d_at_x[i] = NAN;
    }

    /* Validity: every draft token in range, every row the step reads usable. */
    for (int i = 0; i < K; ++i)
        if (x[i] < 0 || x[i] >= V) return -1;
    for (int i = 0; i <= K; ++i)
        if (!row_valid(tgt, dtype_t, tgt_off + (size_t)i * V, V)) return -1;
    if (mode == ORC_SAMPLE)
        for (int i = 0; i < K; ++i)
            if (!row_valid(drf, dtype_d, drf_off + (size_t)i * V, V)) return -1;

    if (mode == ORC_GREEDY) {
        /* [Maga] greedy rule: accept while the draft equals the target's most
         * likely token; at the first mismatch emit the target's token; if all
         * K match, emit the target's token after the last draft (bonus). */
        int j = 0, a = 0;
        for (; j < K; ++j) {
            row_max(tgt, dtype_t, tgt_off + (size_t)j * V, V, &a);
            if (x[j] != a) break;
        }
        row_max(tgt, dtype_t, tgt_off + (size_t)j * V, V, &a);
        for (int i = 0; i < j; ++i) tokens[i] = x[i];
        tokens[j] = a;
        return j;
    }

    /* Sampling [Maga], [Monigatti], [Patel], [Atomic]: check drafts left to
     * right; accept x_i with probability min(1, P_t(x_i)/P_d(x_i)); stop at
     * the first rejection. */
    int j = K;
    for (int i = 0; i < K; ++i) {
        row_softmax(tgt, dtype_t, tgt_off + (size_t)i * V, V, T, Pt);
        row_softmax(drf, dtype_d, drf_off + (size_t)i * V, V, T, Pd);
        double pt = Pt[x[i]], pd = Pd[x[i]];
        if (p_t_at_x) p_t_at_x[i] = pt;
        if (p_d_at_x) p_d_at_x[i] = pd;
        double m = pd > 0.0 ? fabs(u[i] * pd - pt) / pd : (pt > 0.0 ? INFINITY : 0.0);
        if (m < ex->accept_margin) ex->accept_margin = m;
        if (!(u[i] * pd < pt)) {
            j = i;
            break;
        }
    }

    int token;
    double total = 0.0, margin = 0.0;
    if (j < K) {
        /* Rejection at j: draw from norm(max(0, P_t - P_d)) of row j (Pt and
         * Pd still hold row j). */
        for (int v = 0; v < V; ++v) {
            double d = Pt[v] - Pd[v];
            r[v] = d > 0.0 ? d : 0.0;
        }
        double s = 0.0;
        for (int v = 0; v < V; ++v) s += r[v];
        if (!(s > 0.0)) {
            ex->fallback = 1;
            for (int v = 0; v < V; ++v) r[v] = Pt[v];
        }
        token = inverse_cdf(r, V, u2[j], &total, &margin, ex->draw_edges);
    } else {
        /* All K accepted: the bonus token comes from P_t of row K. */
        row_softmax(tgt, dtype_t, tgt_off + (size_t)K * V, V, T, Pt);
        token = inverse_cdf(Pt, V, u2[K], &total, &margin, ex->draw_edges);
    }
    ex->draw_margin = margin;
    ex->residual_mass = total;
    for (int i = 0; i < j; ++i) tokens[i] = x[i];
    tokens[j] = token;
    return j;
}

/* Batch entry point, sequences [b_begin, b_end).
 *   target [B, K+1, V] (dtype_t), draft [B, K, V] (dtype_d; may be NULL when
 *   every sequence is greedy), draft_tokens [B, K], modes [B] (0 greedy,
 *   1 sample). Uniforms come either from `uniforms` (u [B, K+1] then
 *   u2 [B, K+1], when non-NULL) or from Philox with `seed` and the sequence
 *   ids seq_ids [B] (NULL means id = b).
 *   Outputs: out_tokens [B, K+1], out_n_accepted [B]; optional (NULL to
 *   skip): out_p_target / out_p_draft [B, K], out_residual_mass [B],
 *   out_accept_margin [B], out_draw_margin [B], out_fallback [B],
 *   out_draw_edges [B, 2] (t's distances to the chosen interval's lower and
 *   upper edges; NaN for greedy or invalid sequences).
 * Returns 0, or -1 if a work buffer could not be allocated. */
int oracle_verify(const void* target, const void* draft,
                  const int32_t* draft_tokens, int B, int K, int V,
                  int dtype_t, int dtype_d, double temperature,
                  const int32_t* modes, uint64_t seed, const uint64_t* seq_ids,
                  const double* uniforms, int b_begin, int b_end,
                  int32_t* out_tokens, int32_t* out_n_accepted,
                  double* out_p_target, double* out_p_draft,
                  double* out_residual_mass, double* out_accept_margin,
                  double* out_draw_margin, int32_t* out_fallback,
                  const int32_t* draft_lens, double* out_draw_edges) {
    double* Pt = (double*)malloc(sizeof(double) * (size_t)V);
    double* Pd = (double*)malloc(sizeof(double) * (size_t)V);
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    double* u = (double*)malloc(sizeof(double) * (size_t)(K + 1));
    double* u2 = (double*)malloc(sizeof(double) * (size_t)(K + 1));
    if (!Pt || !Pd || !r || !u || !u2) {
        free(Pt); free(Pd); free(r); free(u); free(u2);
        return -1;
    }
    for (int b = b_begin; b < b_end; ++b) {
        if (uniforms) {
            for (int p = 0; p <= K; ++p) {
                u[p] = uniforms[(size_t)b * (K + 1) + p];
                u2[p] = uniforms[(size_t)B * (K + 1) + (size_t)b * (K + 1) + p];
            }
        } else {
            uint64_t id = seq_ids ? seq_ids[b] : (uint64_t)b;
            for (int p = 0; p <= K; ++p) draw_uniforms(seed, id, (uint32_t)p, &u[p], &u2[p]);
        }
        seq_extra ex;
        int mode = modes ? modes[b] : ORC_SAMPLE;
        /* A sequence may verify fewer drafts than the layout holds: its own
         * draft length Kb reads target rows 0..Kb and draft rows 0..Kb-1 of
         * its block (continuous batching); positions past Kb emit -1. */
        const int Kb = draft_lens ? draft_lens[b] : K;
        int32_t* tok_b = out_tokens + (size_t)b * (K + 1);
        for (int i = 0; i <= K; ++i) tok_b[i] = -1;
        for (int i = 0; i < K; ++i) {
            if (out_p_target) out_p_target[(size_t)b * K + i] = NAN;
            if (out_p_draft) out_p_draft[(size_t)b * K + i] = NAN;
        }
        int j;
        if (Kb < 0 || Kb > K) {
            j = -1;
            ex.accept_margin = INFINITY;
            ex.draw_margin = INFINITY;
            ex.draw_edges[0] = ex.draw_edges[1] = NAN;
            ex.residual_mass = NAN;
            ex.fallback = 0;
        } else {
            j = verify_sequence(
                target, (size_t)b * (K + 1) * V, draft, (size_t)b * K * V, dtype_t,
                dtype_d, draft_tokens + (size_t)b * K, Kb, V, mode, temperature, u, u2,
                tok_b, out_p_target ? out_p_target + (size_t)b * K : NULL,
                out_p_draft ? out_p_draft + (size_t)b * K : NULL, &ex, Pt, Pd, r);
        }
        out_n_accepted[b] = j;
        if (out_residual_mass) out_residual_mass[b] = ex.residual_mass;
        if (out_accept_margin) out_accept_margin[b] = ex.accept_margin;
        if (out_draw_margin) out_draw_margin[b] = ex.draw_margin;
        if (out_fallback) out_fallback[b] = ex.fallback;
        if (out_draw_edges) {
            out_draw_edges[2 * (size_t)b] = ex.draw_edges[0];
            out_draw_edges[2 * (size_t)b + 1] = ex.draw_edges[1];
        }
    }
    free(Pt); free(Pd); free(r); free(u); free(u2);
    return 0;
}

/* Greedy tree verification ("Inference-4", section "Medusa": the candidate
 * continuations form a tree, all of them are verified in one forward pass,
 * and the longest accepted path is kept). Node 0 is the root (the last
 * committed token); node i > 0 carries token tokens[i] and has parent
 * parents[i] < i; target row i is the target's distribution after the prefix
 * that ends at node i. With the greedy rule a node is accepted when its
 * parent is and its token is the argmax of its parent's row. The kept path
 * ends at the deepest accepted node (lowest index among equally deep ones);
 * the output is the path's tokens followed by the argmax of that node's row.
 * Layout: target [B, N, V], tokens and parents [B, N]; outputs tokens [B, N]
 * (-1 padded), n_accepted [B] (the path length, -1 for an invalid sequence:
 * a parent outside [0, i), a token outside [0, V) on a tested node, or a row
 * without a finite maximum) and last_node [B]. */
int oracle_verify_tree(const void* target, int dtype, const int32_t* tokens,
                       const int32_t* parents, int B, int N, int V,
                       int b_begin, int b_end, int32_t* out_tokens,
                       int32_t* out_n_accepted, int32_t* out_last_node) {
    int* am = (int*)malloc(sizeof(int) * (size_t)N);
    int* acc = (int*)malloc(sizeof(int) * (size_t)N);
    int* depth = (int*)malloc(sizeof(int) * (size_t)N);
    if (!am || !acc || !depth) {
        free(am); free(acc); free(depth);
        return -1;
    }
    for (int b = b_begin; b < b_end; ++b) {
        const int32_t* tok = tokens + (size_t)b * N;
        const int32_t* par = parents + (size_t)b * N;
        int32_t* out = out_tokens + (size_t)b * N;
        for (int i = 0; i < N; ++i) out[i] = -1;
        out_n_accepted[b] = -1;
        out_last_node[b] = -1;
        int ok = 1;
        for (int i = 1; i < N; ++i)
            if (par[i] < 0 || par[i] >= i) ok = 0;
        for (int i = 0; i < N && ok; ++i) {
            size_t off = ((size_t)b * N + i) * V;
            if (!row_valid(target, dtype, off, V)) ok = 0;
            else row_max(target, dtype, off, V, &am[i]);
        }
        if (!ok) continue;
        acc[0] = 1;
        depth[0] = 0;
        for (int i = 1; i < N; ++i) {
            depth[i] = depth[par[i]] + 1;
            acc[i] = 0;
            if (acc[par[i]]) {
                /* a tested node: its token is compared with its parent's argmax */
                if (tok[i] < 0 || tok[i] >= V) ok = 0;
                acc[i] = tok[i] == am[par[i]];
            }
        }
        if (!ok) continue;
        int best = 0;
        for (int i = 1; i < N; ++i)
            if (acc[i] && depth[i] > depth[best]) best = i;
        const int n = depth[best];
        for (int i = best, k = n - 1; i != 0; i = par[i], --k) out[k] = tok[i];
        out[n] = am[best];
        out_n_accepted[b] = n;
        out_last_node[b] = best;
    }
    free(am); free(acc); free(depth);
    return 0;
}

/* Prompt lookup drafting ("Inference-4", section "Prompt lookup decoding"):
 * the drafts are the tokens that followed the most recent earlier occurrence
 * of the sequence's last n-gram, trying n = max_ngram first and shorter
 * n-grams after; no drafts when none of them occurred before. For each n with
 * n < L: the candidate windows are the n-grams starting at s = 0 .. L-1-n (they
 * end before the last token); the most recent match has the largest s; the
 * drafts are tokens s+n .. s+n+n_drafts-1, cut at the end of the sequence.
 * Layout: tokens [B, L_max] with lengths [B]; out_drafts [B, n_drafts]
 * (-1 padded), out_n_drafts [B] (-1 for a length outside [0, L_max]). */
void oracle_prompt_lookup(const int32_t* tokens, const int32_t* lengths, int B,
                          int L_max, int max_ngram, int n_drafts, int b_begin,
                          int b_end, int32_t* out_drafts, int32_t* out_n_drafts) {
    for (int b = b_begin; b < b_end; ++b) {
        const int32_t* seq = tokens + (size_t)b * L_max;
        int32_t* out = out_drafts + (size_t)b * n_drafts;
        const int L = lengths[b];
        for (int i = 0; i < n_drafts; ++i) out[i] = -1;
        if (L < 0 || L > L_max) {
            out_n_drafts[b] = -1;
            continue;
        }
        out_n_drafts[b] = 0;
        for (int n = max_ngram; n >= 1; --n) {
            if (L <= n) continue;
            int found = -1;
            for (int st = L - 1 - n; st >= 0 && found < 0; --st) {
                int same = 1;
                for (int t = 0; t < n && same; ++t)
                    if (seq[st + t] != seq[L - n + t]) same = 0;
                if (same) found = st;
            }
            if (found >= 0) {
                int c = 0;
                for (int i = found + n; i < L && c < n_drafts; ++i) out[c++] = seq[i];
                out_n_drafts[b] = c;
                break;
            }
        }
    }
}

/* Logits of the fused LM-head variant: logits[m, v] = sum_k hidden[m, k] *
 * W[k, v] over bf16 inputs widened exactly, accumulated in double in k order.
 * hidden [M, d] and W [d, V] are raw bf16 bits; rows [m_begin, m_end) only. */
void oracle_lmhead_logits(const uint16_t* hidden, const uint16_t* W, int M,
                          int d, int V, int m_begin, int m_end, double* out) {
    double* h = (double*)malloc(sizeof(double) * (size_t)d);
    if (!h) return;
    for (int m = m_begin; m < m_end; ++m) {
        for (int k = 0; k < d; ++k) h[k] = logit_at(hidden, ORC_BF16, (size_t)m * d + k);
        double* row = out + (size_t)(m - m_begin) * V;
        for (int v = 0; v < V; ++v) row[v] = 0.0;
        for (int k = 0; k < d; ++k) {
            double hk = h[k];
            const uint16_t* wrow = W + (size_t)k * V;
            for (int v = 0; v < V; ++v) row[v] += hk * logit_at(wrow, ORC_BF16, (size_t)v);
        }
    }
    (void)M;
    free(h);
}
