/*
 * spec_verify_ref.c -- CPU oracle (fp64) for batched speculative-sampling verification.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py, never by the CUDA library.  It
 * shares no code with the CUDA path.  Plain, slow and written to be checked
 * by eye against the pages:
 *
 *  [LEV]  "Fast Inference from Transformers via Speculative Decoding" (paper
 *         review page), section "Speculative Sampling", Algorithm 1
 *         SpeculativeDecodingStep, and section "Method: Speculative Decoding"
 *         (temperature / top-k / nucleus / argmax all become standard sampling
 *         from an adjusted distribution; argmax zeroes the non-max entries).
 *  [SUR]  "投机解码（Speculative Decoding）" survey page, section 2 (lossless
 *         acceptance rule, residual p' = norm(max(0, p - q))), section 4
 *         (speculative_step pseudocode: left-to-right, stop at first rejection,
 *         bonus from p_{gamma+1}).
 *  [AGW]  "Speculative decoding: the art of guessing well", section 投机采样
 *         (alpha = sum_x min(p, q); the `verify` listing: accept iff
 *         uniform < min(1, p/q); first rejection = argmin(append(accepted, False));
 *         q_{gamma+1} treated as zero so the residual becomes p_{gamma+1}).
 *  [PHX]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *         1, 2, 3", SC'11 -- the Philox4x32-10 block function.
 *  [AGW-G] "Speculative decoding: the art of guessing well", section 共享噪声的
 *         采样 (Gumbel-max, shared noise, the `gumbel_verify` listing) -- the
 *         shared-noise functions at the end of this file.
 *  [LEN]  the same review page, section Lenience: a parameter l in [0, 1]
 *         multiplies q(x) in the acceptance test; no token is then emitted with
 *         more than 1/l times its probability, and the acceptance rate rises.
 *  [STR]  "SpecTr: Fast Speculative Decoding via Optimal Transport" page,
 *         section K-SEQ (eqs. (4)-(7), the residual distribution) -- the K-SEQ
 *         functions at the end of this file (the page's p and q swapped).
 *
 * Readings taken where the pages are silent (each resolves a point the pages leave open):
 *  - normalisation order: temperature, softmax, top-k, renormalise, top-p,
 *    renormalise; ties in top-k / top-p / argmax go to the lower token id;
 *    the top-p set is the shortest descending prefix whose mass reaches top_p
 *    (the crossing token is kept);
 *  - acceptance is the strict test u * q(x) < p(x) (no division), so a draft
 *    token with q(x) = 0 is accepted iff p(x) > 0;
 *  - the residual / bonus draw is an inverse CDF in ascending token id with
 *    v = u * Z, Z = sum_x max(0, p - q); if Z <= 0 the draw falls back to p;
 *  - randomness: u = U(seed, b, pos, draw), draw 0 = acceptance at pos,
 *    draw 1 = residual/bonus at pos, pos 1-based.
 */
#include "spec_verify_ref.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 [PHX].  Parity: pinned only statistically (uniformity,       */
/* independence and bijectivity tests) and by agreement with the separately   */
/* written device copy; no published known-answer vector is stored here.      */
/* ------------------------------------------------------------------------- */

#define PHX_M0 0xD2511F53u /* round multipliers [PHX] */
#define PHX_M1 0xCD9E8D57u
#define PHX_W0 0x9E3779B9u /* Weyl key increments [PHX]: golden ratio, sqrt(3)-1 */
#define PHX_W1 0xBB67AE85u

void svr_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { /* the key is bumped before every round but the first */
            k0 += PHX_W0;
            k1 += PHX_W1;
        }
        uint64_t prod0 = (uint64_t)PHX_M0 * (uint64_t)x0;
        uint64_t prod1 = (uint64_t)PHX_M1 * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0;
        x1 = y1;
        x2 = y2;
        x3 = y3;
    }
    out[0] = x0;
    out[1] = x1;
    out[2] = x2;
    out[3] = x3;
}

/* u = ((w0 >> 8) + 1/2) * 2^-24: strictly inside (0,1) and exact in fp64. */
double svr_uniform(uint64_t seed, uint32_t b, uint32_t pos, uint32_t draw) {
    uint32_t ctr[4] = {b, pos, draw, 0u};
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    svr_philox4x32_10(ctr, key, out);
    return ((double)(out[0] >> 8) + 0.5) / 16777216.0;
}

void svr_philox_uniforms(uint64_t seed, int B, int G, double* u_accept, double* u_resid) {
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < G; ++i) u_accept[(size_t)b * G + i] = svr_uniform(seed, (uint32_t)b, (uint32_t)(i + 1), 0u);
        for (int j = 0; j <= G; ++j)
            u_resid[(size_t)b * (G + 1) + j] = svr_uniform(seed, (uint32_t)b, (uint32_t)(j + 1), 1u);
    }
}

/* ------------------------------------------------------------------------- */
/* Inputs                                                                     */
/* ------------------------------------------------------------------------- */

/* exact value of one stored logit, widened to double */
static double logit_value(const void* base, int dtype, size_t idx) {
    if (dtype == SVR_DTYPE_F32) return (double)((const float*)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16; /* bf16 = top half of an fp32 */
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------- */
/* Normalisation [LEV "Method": temperature / top-k / nucleus / argmax are all  */
/* standard sampling from an adjusted distribution].                          */
/* Parity: pinned by the softmax identity, argmax special case, brute force   */
/* over all subsets for V <= 8, and the identity cases top_k = V, top_p = 1.  */
/* ------------------------------------------------------------------------- */

typedef struct {
    double p;
    int id;
} ranked_t;

/* descending probability, ascending token id on ties */
static int ranked_cmp(const void* a, const void* b) {
    const ranked_t* x = (const ranked_t*)a;
    const ranked_t* y = (const ranked_t*)b;
    if (x->p > y->p) return -1;
    if (x->p < y->p) return 1;
    return (x->id < y->id) ? -1 : (x->id > y->id);
}

int svr_normalise(const double* logits, int V, double T, int top_k, double top_p, double* probs,
                  double* filter_margin) {
    double margin = INFINITY;

    /* the largest finite-or-minus-infinity logit; lowest id on ties */
    int arg = -1;
    for (int x = 0; x < V; ++x)
        if (arg < 0 || logits[x] > logits[arg]) arg = x;
    if (arg < 0 || !(logits[arg] > -INFINITY)) return -1;

    if (T == 0.0) { /* argmax: zero the non-max entries and renormalise */
        for (int x = 0; x < V; ++x) probs[x] = 0.0;
        probs[arg] = 1.0;
        if (filter_margin) *filter_margin = margin;
        return 0;
    }

    /* temperature then softmax */
    double m = logits[arg] / T;
    double S = 0.0;
    for (int x = 0; x < V; ++x) {
        probs[x] = exp(logits[x] / T - m);
        S += probs[x];
    }
    for (int x = 0; x < V; ++x) probs[x] /= S;

    int use_k = (top_k > 0 && top_k < V);
    int use_p = (top_p < 1.0);
    if (use_k || use_p) {
        ranked_t* order = (ranked_t*)malloc(sizeof(ranked_t) * (size_t)V);
        for (int x = 0; x < V; ++x) {
            order[x].p = probs[x];
            order[x].id = x;
        }
        qsort(order, (size_t)V, sizeof(ranked_t), ranked_cmp);

        if (use_k) { /* keep the k largest, renormalise */
            double pk = order[top_k - 1].p, pn = order[top_k].p;
            if (pn > 0.0 && pk > pn) margin = fmin(margin, (pk - pn) / pk);
            double Sk = 0.0;
            for (int r = 0; r < V; ++r) {
                if (r < top_k)
                    Sk += order[r].p;
                else
                    order[r].p = 0.0;
            }
            for (int r = 0; r < top_k; ++r) order[r].p /= Sk;
        }
        if (use_p) { /* shortest descending prefix with mass >= top_p, crossing token kept */
            int keep = V;
            double cum = 0.0, before = 0.0;
            for (int r = 0; r < V; ++r) {
                if (order[r].p <= 0.0) {
                    keep = r; /* mass exhausted by rounding before reaching top_p */
                    break;
                }
                before = cum;
                cum += order[r].p;
                if (cum >= top_p) {
                    keep = r + 1;
                    margin = fmin(margin, fmin(cum - top_p, top_p - before));
                    if (r + 1 < V && order[r + 1].p > 0.0 && order[r].p > order[r + 1].p)
                        margin = fmin(margin, (order[r].p - order[r + 1].p) / order[r].p);
                    break;
                }
            }
            double Sp = 0.0;
            for (int r = 0; r < V; ++r) {
                if (r < keep)
                    Sp += order[r].p;
                else
                    order[r].p = 0.0;
            }
            for (int r = 0; r < keep; ++r) order[r].p /= Sp;
        }
        for (int r = 0; r < V; ++r) probs[order[r].id] = order[r].p;
        free(order);
    }
    if (filter_margin) *filter_margin = margin;
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Residual / bonus draw [LEV Algorithm 1 steps 4-5; AGW `verify`]:           */
/* r = max(0, p - q) (q := 0 for the bonus), inverse CDF in ascending id.      */
/* Parity: pinned by the worked example of the SpecTr page (residual          */
/* (0, .5, .5)), exact enumeration and chi-square of the output marginal.     */
/* ------------------------------------------------------------------------- */

static int residual_draw(const double* p, const double* q, int V, double u, double* margin_out) {
    double Z = 0.0;
    for (int x = 0; x < V; ++x) {
        double r = p[x] - (q ? q[x] : 0.0);
        if (r > 0.0) Z += r;
    }
    int fallback = !(Z > 0.0); /* p <= q everywhere: cannot follow a rejection exactly; use p */
    if (fallback) {
        Z = 0.0;
        for (int x = 0; x < V; ++x) Z += p[x];
    }
    double v = u * Z;
    double cum = 0.0, before = 0.0;
    int token = -1, last_pos = -1;
    for (int x = 0; x < V; ++x) {
        double r = fallback ? p[x] : p[x] - (q ? q[x] : 0.0);
        if (!(r > 0.0)) continue;
        last_pos = x;
        before = cum;
        cum += r;
        if (cum > v) {
            token = x;
            break;
        }
    }
    double margin;
    if (token < 0) { /* v beyond the accumulated total by rounding: last token with mass */
        token = last_pos;
        margin = 0.0;
    } else {
        margin = fmin(v - before, cum - v) / Z;
    }
    if (Z < 1e-12) margin = 0.0; /* residual made of rounding noise: no stable answer */
    if (margin_out) *margin_out = margin;
    return token;
}

/* ------------------------------------------------------------------------- */
/* Batched verification [LEV Algorithm 1; SUR section 4; AGW `verify`].       */
/* ------------------------------------------------------------------------- */

/* Acceptance mass of one token under lenience l [LEN]: q(x) * P(u l q(x) < p(x)) with
 * u uniform on (0, 1), i.e. q(x) when l q(x) <= p(x) and p(x) > 0, else p(x) / l (which
 * is 0 when p(x) = 0).  With l = 1 this is min(p(x), q(x)) [AGW 投机采样]. */
static double accept_mass(double p, double q, double l) {
    if (l * q <= p) return p > 0.0 ? q : 0.0;
    return p / l; /* here l q > p >= 0, so l > 0 */
}

int svr_verify(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
               const int32_t* num_draft, const float* temperature, const int32_t* top_k,
               const float* top_p, const double* u_accept, const double* u_resid, int B, int G, int V,
               int32_t* accepted_len, int32_t* out_tokens, double* alpha, int32_t* pos_accept,
               int32_t* pos_token, double* p_out, double* q_out, uint32_t* status,
               double* accept_margin, double* resid_margin, double* filter_margin) {
    return svr_verify_ex(target, draft, dtype, draft_tokens, num_draft, temperature, top_k, top_p, NULL, u_accept,
                         u_resid, B, G, V, accepted_len, out_tokens, alpha, pos_accept, pos_token, p_out, q_out,
                         status, accept_margin, resid_margin, filter_margin);
}

int svr_verify_ex(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                  const int32_t* num_draft, const float* temperature, const int32_t* top_k,
                  const float* top_p, const float* lenience, const double* u_accept, const double* u_resid,
                  int B, int G, int V, int32_t* accepted_len, int32_t* out_tokens, double* alpha,
                  int32_t* pos_accept, int32_t* pos_token, double* p_out, double* q_out, uint32_t* status,
                  double* accept_margin, double* resid_margin, double* filter_margin) {
    if (B < 0 || G < 1 || V < 1) return -1;
    if (dtype != SVR_DTYPE_F32 && dtype != SVR_DTYPE_BF16) return -1;
    if (B > 0 && (!target || !draft || !draft_tokens || !temperature || !u_accept || !u_resid ||
                  !accepted_len || !out_tokens || !alpha))
        return -1;
    int all_positions = (pos_accept || pos_token || accept_margin || resid_margin);

    double* logits = (double*)malloc(sizeof(double) * (size_t)V);
    double* P = (double*)malloc(sizeof(double) * (size_t)V * (size_t)(G + 1)); /* p_1..p_{G+1} */
    double* Q = (double*)malloc(sizeof(double) * (size_t)V * (size_t)G);       /* q_1..q_G */

    for (int b = 0; b < B; ++b) {
        uint32_t st = 0;
        int gamma = num_draft ? num_draft[b] : G;
        double T = (double)temperature[b];
        int k = top_k ? top_k[b] : 0;
        double tp = top_p ? (double)top_p[b] : 1.0;
        double len = lenience ? (double)lenience[b] : 1.0;
        if (!(T >= 0.0) || isinf(T)) st |= SVR_ST_BAD_TEMPERATURE;
        if (k < 0) st |= SVR_ST_BAD_TOP_K;
        if (!(tp > 0.0 && tp <= 1.0)) st |= SVR_ST_BAD_TOP_P;
        if (!(len >= 0.0 && len <= 1.0)) st |= SVR_ST_BAD_LENIENCE;
        if (gamma < 1 || gamma > G) st |= SVR_ST_BAD_NUM_DRAFT;
        if (!(st & SVR_ST_BAD_NUM_DRAFT))
            for (int i = 0; i < gamma; ++i) {
                int32_t x = draft_tokens[(size_t)b * G + i];
                if (x < 0 || x >= V) st |= SVR_ST_BAD_DRAFT_TOKEN;
            }

        /* normalise the rows in use: target rows 0..gamma, draft rows 0..gamma-1 */
        if (!st) {
            for (int row = 0; row < 2 * gamma + 1 && !st; ++row) {
                int is_target = row <= gamma;
                int r = is_target ? row : row - gamma - 1;
                const void* src = is_target ? target : draft;
                size_t base = is_target ? ((size_t)b * (G + 1) + r) * (size_t)V : ((size_t)b * G + r) * (size_t)V;
                for (int x = 0; x < V; ++x) {
                    logits[x] = logit_value(src, dtype, base + x);
                    if (isnan(logits[x]) || logits[x] == INFINITY) st |= SVR_ST_NONFINITE;
                }
                if (st) break;
                double fm = INFINITY;
                double* dst = is_target ? P + (size_t)r * V : Q + (size_t)r * V;
                if (svr_normalise(logits, V, T, k, tp, dst, &fm) != 0) st |= SVR_ST_NONFINITE;
                if (filter_margin) filter_margin[(size_t)b * (2 * G + 1) + (is_target ? r : G + 1 + r)] = fm;
            }
        }
        if (status) status[b] = st;

        /* defaults: nothing accepted, no token, zero alpha, undefined positions */
        accepted_len[b] = 0;
        for (int j = 0; j <= G; ++j) out_tokens[(size_t)b * (G + 1) + j] = -1;
        for (int i = 0; i < G; ++i) alpha[(size_t)b * G + i] = 0.0;
        if (pos_accept)
            for (int i = 0; i < G; ++i) pos_accept[(size_t)b * G + i] = -1;
        if (pos_token)
            for (int j = 0; j <= G; ++j) pos_token[(size_t)b * (G + 1) + j] = -1;
        if (accept_margin)
            for (int i = 0; i < G; ++i) accept_margin[(size_t)b * G + i] = NAN;
        if (resid_margin)
            for (int j = 0; j <= G; ++j) resid_margin[(size_t)b * (G + 1) + j] = NAN;
        if (filter_margin && st)
            for (int r = 0; r < 2 * G + 1; ++r) filter_margin[(size_t)b * (2 * G + 1) + r] = NAN;
        if (p_out) memset(p_out + (size_t)b * (G + 1) * V, 0, sizeof(double) * (size_t)(G + 1) * V);
        if (q_out) memset(q_out + (size_t)b * G * V, 0, sizeof(double) * (size_t)G * V);
        if (st) continue;

        if (p_out) memcpy(p_out + (size_t)b * (G + 1) * V, P, sizeof(double) * (size_t)(gamma + 1) * V);
        if (q_out) memcpy(q_out + (size_t)b * G * V, Q, sizeof(double) * (size_t)gamma * V);

        /* per-position acceptance rate alpha_i = sum_x min(p_i(x), q_i(x)) [AGW 投机采样];
         * under lenience l, sum_x q_i(x) P(accept | x) [LEN] */
        for (int i = 0; i < gamma; ++i) {
            double a = 0.0;
            for (int x = 0; x < V; ++x) a += accept_mass(P[(size_t)i * V + x], Q[(size_t)i * V + x], len);
            alpha[(size_t)b * G + i] = a;
        }

        /* acceptance test left to right, stop at the first rejection [LEV Alg. 1 step 3];
         * lenience multiplies q(x) in the test [LEN] */
        int n = gamma;
        for (int i = 0; i < gamma; ++i) {
            int x = draft_tokens[(size_t)b * G + i];
            double px = P[(size_t)i * V + x], qx = Q[(size_t)i * V + x];
            double u = u_accept[(size_t)b * G + i];
            double lq = len * qx;
            int accept = (u * lq < px);
            if (accept_margin) accept_margin[(size_t)b * G + i] = (lq > 0.0) ? fabs(u - px / lq) : INFINITY;
            if (pos_accept) pos_accept[(size_t)b * G + i] = accept;
            if (!accept && n == gamma) {
                n = i;
                if (!all_positions) break;
            }
        }

        /* residual at position n+1, or the bonus from p_{gamma+1} [LEV Alg. 1 steps 4-5] */
        for (int j = 0; j <= gamma; ++j) {
            if (!all_positions && j != n) continue;
            const double* pj = P + (size_t)j * V;
            const double* qj = (j < gamma) ? Q + (size_t)j * V : NULL; /* q_{gamma+1} := 0 */
            double rm = 0.0;
            int tok = residual_draw(pj, qj, V, u_resid[(size_t)b * (G + 1) + j], &rm);
            if (pos_token) pos_token[(size_t)b * (G + 1) + j] = tok;
            if (resid_margin) resid_margin[(size_t)b * (G + 1) + j] = rm;
            if (j == n) {
                for (int i = 0; i < n; ++i) out_tokens[(size_t)b * (G + 1) + i] = draft_tokens[(size_t)b * G + i];
                out_tokens[(size_t)b * (G + 1) + n] = tok;
                accepted_len[b] = n;
            }
        }
    }
    free(logits);
    free(P);
    free(Q);
    return 0;
}

int svr_verify_seeded(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                      const int32_t* num_draft, const float* temperature, const int32_t* top_k,
                      const float* top_p, uint64_t seed, int B, int G, int V, int32_t* accepted_len,
                      int32_t* out_tokens, double* alpha, int32_t* pos_accept, int32_t* pos_token,
                      double* p_out, double* q_out, uint32_t* status, double* accept_margin,
                      double* resid_margin, double* filter_margin) {
    return svr_verify_ex_seeded(target, draft, dtype, draft_tokens, num_draft, temperature, top_k, top_p, NULL,
                                seed, B, G, V, accepted_len, out_tokens, alpha, pos_accept, pos_token, p_out,
                                q_out, status, accept_margin, resid_margin, filter_margin);
}

int svr_verify_ex_seeded(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                         const int32_t* num_draft, const float* temperature, const int32_t* top_k,
                         const float* top_p, const float* lenience, uint64_t seed, int B, int G, int V,
                         int32_t* accepted_len, int32_t* out_tokens, double* alpha, int32_t* pos_accept,
                         int32_t* pos_token, double* p_out, double* q_out, uint32_t* status,
                         double* accept_margin, double* resid_margin, double* filter_margin) {
    if (B < 0 || G < 1) return -1;
    double* ua = (double*)malloc(sizeof(double) * (size_t)(B > 0 ? B : 1) * (size_t)G);
    double* ur = (double*)malloc(sizeof(double) * (size_t)(B > 0 ? B : 1) * (size_t)(G + 1));
    svr_philox_uniforms(seed, B, G, ua, ur);
    int rc = svr_verify_ex(target, draft, dtype, draft_tokens, num_draft, temperature, top_k, top_p, lenience,
                           ua, ur, B, G, V, accepted_len, out_tokens, alpha, pos_accept, pos_token, p_out, q_out,
                           status, accept_margin, resid_margin, filter_margin);
    free(ua);
    free(ur);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Gumbel-coupled (shared-noise) verification [AGW, section 共享噪声的采样].    */
/*                                                                           */
/* Sampling from softmax(l) is argmax_i(l_i + g_i) with g_i = -log(-log u_i)  */
/* (the Gumbel-max trick).  The drafter and the target share the noise g_k of */
/* each position k: the drafter proposes argmax_i(log q_k(i) + g_k,i), the    */
/* target takes argmax_i(log p_k(i) + g_k,i), and the round keeps the longest */
/* prefix where the two agree plus the target's token at the first            */
/* disagreement (all gamma agree: the target's token at gamma + 1).  p and q  */
/* are the rows normalised as in svr_normalise (temperature, top-k, top-p);   */
/* tokens outside the kept set have log p = -inf and are never chosen.        */
/*                                                                           */
/* Readings where the page is silent: the noise of token i at position k of  */
/* sequence b is u = Philox4x32-10(counter (b, k, 2, i >> 2), key seed), word */
/* i & 3, on the same 24-bit grid as svr_uniform (draw 2: disjoint from the   */
/* acceptance and residual draws 0 and 1); argmax ties go to the lower id;    */
/* T = 0 is the plain argmax of the logits (no noise).                        */
/* Parity: pinned by the Gumbel-max law, drafter invariance, the page's       */
/* closed form for the match probability and its lower bound, and the greedy  */
/* special case (tests/test_gumbel_oracle.py).                                */
/* ------------------------------------------------------------------------- */

double svr_gumbel_uniform(uint64_t seed, uint32_t b, uint32_t pos, uint32_t token) {
    uint32_t ctr[4] = {b, pos, 2u, token >> 2};
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    svr_philox4x32_10(ctr, key, out);
    return ((double)(out[token & 3u] >> 8) + 0.5) / 16777216.0;
}

/* argmax_i(log probs[i] + g_i) over probs[i] > 0, ties to the lower id;
 * *gap = best score - second best score (INFINITY if one candidate). */
static int gumbel_argmax(const double* probs, int V, int noisy, uint64_t seed, uint32_t b, uint32_t pos,
                         double* gap) {
    int best = -1;
    double s1 = -INFINITY, s2 = -INFINITY;
    for (int i = 0; i < V; ++i) {
        if (!(probs[i] > 0.0)) continue;
        double s = log(probs[i]);
        if (noisy) s += -log(-log(svr_gumbel_uniform(seed, b, pos, (uint32_t)i)));
        if (best < 0 || s > s1) {
            s2 = s1;
            s1 = s;
            best = i;
        } else if (s > s2) {
            s2 = s;
        }
    }
    *gap = s1 - s2;
    return best;
}

/* validation and normalisation of one row (the rules of svr_verify); returns the status bits */
static uint32_t gumbel_row(const void* logits_base, int dtype, size_t base, int V, double T, int k, double tp,
                           double* logits, double* probs) {
    for (int x = 0; x < V; ++x) {
        logits[x] = logit_value(logits_base, dtype, base + x);
        if (isnan(logits[x]) || logits[x] == INFINITY) return SVR_ST_NONFINITE;
    }
    return svr_normalise(logits, V, T, k, tp, probs, NULL) != 0 ? SVR_ST_NONFINITE : 0u;
}

static uint32_t gumbel_params(int gamma, int G, double T, int k, double tp) {
    uint32_t st = 0;
    if (!(T >= 0.0) || isinf(T)) st |= SVR_ST_BAD_TEMPERATURE;
    if (k < 0) st |= SVR_ST_BAD_TOP_K;
    if (!(tp > 0.0 && tp <= 1.0)) st |= SVR_ST_BAD_TOP_P;
    if (gamma < 1 || gamma > G) st |= SVR_ST_BAD_NUM_DRAFT;
    return st;
}

int svr_gumbel_verify(const void* target, int dtype, const int32_t* draft_tokens, const int32_t* num_draft,
                      const float* temperature, const int32_t* top_k, const float* top_p, uint64_t seed, int B,
                      int G, int V, int32_t* accepted_len, int32_t* out_tokens, int32_t* target_tokens,
                      double* margin, uint32_t* status) {
    if (B < 0 || G < 1 || G > SVR_MAX_G || V < 1) return -1;
    if (dtype != SVR_DTYPE_F32 && dtype != SVR_DTYPE_BF16) return -1;
    if (B > 0 && (!target || !draft_tokens || !temperature || !accepted_len || !out_tokens)) return -1;
    double* logits = (double*)malloc(sizeof(double) * (size_t)V);
    double* probs = (double*)malloc(sizeof(double) * (size_t)V);
    for (int b = 0; b < B; ++b) {
        int gamma = num_draft ? num_draft[b] : G;
        double T = (double)temperature[b];
        int k = top_k ? top_k[b] : 0;
        double tp = top_p ? (double)top_p[b] : 1.0;
        uint32_t st = gumbel_params(gamma, G, T, k, tp);
        if (!(st & SVR_ST_BAD_NUM_DRAFT))
            for (int i = 0; i < gamma; ++i) {
                int32_t x = draft_tokens[(size_t)b * G + i];
                if (x < 0 || x >= V) st |= SVR_ST_BAD_DRAFT_TOKEN;
            }
        accepted_len[b] = 0;
        for (int j = 0; j <= G; ++j) {
            out_tokens[(size_t)b * (G + 1) + j] = -1;
            if (target_tokens) target_tokens[(size_t)b * (G + 1) + j] = -1;
            if (margin) margin[(size_t)b * (G + 1) + j] = NAN;
        }
        /* the target's own noise-driven token at every position 1..gamma+1 */
        int32_t tt[SVR_MAX_G + 1];
        for (int j = 0; j <= gamma && !st; ++j) {
            st |= gumbel_row(target, dtype, ((size_t)b * (G + 1) + j) * (size_t)V, V, T, k, tp, logits, probs);
            if (st) break;
            double gap = INFINITY;
            tt[j] = gumbel_argmax(probs, V, T > 0.0, seed, (uint32_t)b, (uint32_t)(j + 1), &gap);
            if (target_tokens) target_tokens[(size_t)b * (G + 1) + j] = tt[j];
            if (margin) margin[(size_t)b * (G + 1) + j] = gap;
        }
        if (status) status[b] = st;
        if (st) {
            if (target_tokens)
                for (int j = 0; j <= G; ++j) target_tokens[(size_t)b * (G + 1) + j] = -1;
            continue;
        }
        /* the longest prefix where the draft equals the target's choice, then the target's token */
        int n = 0;
        while (n < gamma && draft_tokens[(size_t)b * G + n] == tt[n]) ++n;
        accepted_len[b] = n;
        for (int i = 0; i < n; ++i) out_tokens[(size_t)b * (G + 1) + i] = draft_tokens[(size_t)b * G + i];
        out_tokens[(size_t)b * (G + 1) + n] = tt[n];
    }
    free(logits);
    free(probs);
    return 0;
}

int svr_gumbel_draft(const void* draft, int dtype, const int32_t* num_draft, const float* temperature,
                     const int32_t* top_k, const float* top_p, uint64_t seed, int B, int G, int V,
                     int32_t* draft_tokens) {
    if (B < 0 || G < 1 || V < 1) return -1;
    if (dtype != SVR_DTYPE_F32 && dtype != SVR_DTYPE_BF16) return -1;
    if (B > 0 && (!draft || !temperature || !draft_tokens)) return -1;
    double* logits = (double*)malloc(sizeof(double) * (size_t)V);
    double* probs = (double*)malloc(sizeof(double) * (size_t)V);
    for (int b = 0; b < B; ++b) {
        int gamma = num_draft ? num_draft[b] : G;
        double T = (double)temperature[b];
        int k = top_k ? top_k[b] : 0;
        double tp = top_p ? (double)top_p[b] : 1.0;
        uint32_t st = gumbel_params(gamma, G, T, k, tp);
        for (int i = 0; i < G; ++i) {
            int32_t x = 0; /* padding and invalid rows: token 0 */
            if (!st && i < gamma) {
                if (gumbel_row(draft, dtype, ((size_t)b * G + i) * (size_t)V, V, T, k, tp, logits, probs) == 0u) {
                    double gap;
                    x = gumbel_argmax(probs, V, T > 0.0, seed, (uint32_t)b, (uint32_t)(i + 1), &gap);
                }
            }
            draft_tokens[(size_t)b * G + i] = x;
        }
    }
    free(logits);
    free(probs);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* K-SEQ multi-candidate verification, one position ["SpecTr: Fast           */
/* Speculative Decoding via Optimal Transport" page, section K-SEQ, eqs.      */
/* (4)-(7) and the residual distribution].  The page names the draft p and    */
/* the target q; here, as everywhere in this oracle, p is the TARGET and q the */
/* DRAFT.  With k candidates X_1..X_k drawn independently from q:             */
/*   m_rho(x) = min(q(x), p(x) / rho)         (the mass one try gives to x)    */
/*   beta(rho) = sum_x m_rho(x)                                              */
/*   candidate i is accepted iff u_i * rho * q(X_i) < p(X_i), i.e. with       */
/*   probability min(1, p / (rho q)), tried in order, the first accepted wins */
/*   P_A = 1 - (1 - beta)^k, A_rho(x) = (P_A / beta) m_rho(x)                 */
/*   all rejected: draw from the residual p - A_rho (normalised by 1 - P_A),  */
/*   by inverse CDF in ascending token id with v = u_res * sum(p - A_rho).    */
/* rho* is the root in [1, k] of 1 - (1 - beta(rho))^k = rho beta(rho) (the   */
/* left side minus the right is non-increasing in rho); bisection, keeping    */
/* the end where the left side <= the right, so the residual is nonnegative.  */
/* Special cases from the page: beta = 0 -> nothing is accepted (A = 0) and   */
/* the residual is p itself; P_A = 1 -> the residual branch is never reached   */
/* (numerically: a residual with no mass falls back to p).                    */
/* Readings where the page is silent: strict acceptance u * rho * q < p as in */
/* the single-candidate rule; residual order and uniform as in residual_draw */
/* Parity: pinned by the output law (exact enumeration and chi-square), k = 1 */
/* equal to the single-candidate rule, the page's counterexample to the naive */
/* rule, A_rho* = min(rho* q, p) >= min(q, p), and the page's fixed-rho closed */
/* form (tests/test_kseq_oracle.py).                                          */
/* ------------------------------------------------------------------------- */

double svr_kseq_beta(const double* p, const double* q, int V, double rho) {
    double s = 0.0;
    for (int x = 0; x < V; ++x) s += fmin(q[x], p[x] / rho);
    return s;
}

double svr_kseq_rho(const double* p, const double* q, int V, int k) {
    double lo = 1.0, hi = (double)k;
    /* f(rho) = 1 - (1 - beta)^k - rho * beta; f(1) >= 0 >= f(k) */
    for (int it = 0; it < 200 && hi - lo > 1e-15 * hi; ++it) {
        double mid = 0.5 * (lo + hi);
        double be = svr_kseq_beta(p, q, V, mid);
        double f = 1.0 - pow(1.0 - be, (double)k) - mid * be;
        if (f > 0.0)
            lo = mid;
        else
            hi = mid;
    }
    return hi;
}

/* direct acceptance mass A_rho(x) for rho = rho*(p, q, k); returns P_A */
double svr_kseq_direct(const double* p, const double* q, int V, int k, double* A, double* rho_out) {
    double rho = svr_kseq_rho(p, q, V, k);
    double be = svr_kseq_beta(p, q, V, rho);
    double pa = be > 0.0 ? 1.0 - pow(1.0 - be, (double)k) : 0.0;
    for (int x = 0; x < V; ++x) A[x] = be > 0.0 ? pa / be * fmin(q[x], p[x] / rho) : 0.0;
    if (rho_out) *rho_out = rho;
    return pa;
}

int svr_kseq_step(const double* p, const double* q, int V, int k, const int32_t* cand, const double* u,
                  double u_res, int32_t* accepted_index) {
    double rho = svr_kseq_rho(p, q, V, k);
    *accepted_index = -1;
    for (int i = 0; i < k; ++i) {
        int32_t x = cand[i];
        if (u[i] * rho * q[x] < p[x]) {
            *accepted_index = i;
            return x;
        }
    }
    /* all rejected: residual p - A_rho*, in ascending token id */
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    double* A = (double*)malloc(sizeof(double) * (size_t)V);
    svr_kseq_direct(p, q, V, k, A, NULL);
    double Z = 0.0;
    for (int x = 0; x < V; ++x) {
        r[x] = fmax(p[x] - A[x], 0.0);
        Z += r[x];
    }
    if (!(Z > 0.0)) { /* no residual mass (P_A = 1 up to rounding): fall back to p */
        Z = 0.0;
        for (int x = 0; x < V; ++x) {
            r[x] = p[x];
            Z += r[x];
        }
    }
    double v = u_res * Z, cum = 0.0;
    int token = -1, last = -1;
    for (int x = 0; x < V; ++x) {
        if (!(r[x] > 0.0)) continue;
        last = x;
        cum += r[x];
        if (cum > v) {
            token = x;
            break;
        }
    }
    free(r);
    free(A);
    return token >= 0 ? token : last;
}

/* Batched K-SEQ verification of one position per row [SpecTr page, K-SEQ].  Row b:
 * target logits [V] and draft logits [V] normalised as in svr_normalise, k_b =
 * num_cand[b] candidates cand[b, 0..k_b-1] (tried in that order), uniforms
 * u_i = svr_uniform(seed, b, 1, 3 + i) for candidate i (draws 3..3+K-1, below the
 * input-generation domain 16+) and u_res = svr_uniform(seed, b, 1, 1).  out_token[b]
 * is the emitted token, accepted[b] the index of the accepted candidate or -1
 * (residual), status[b] the usual bits (a candidate outside [0, V) is
 * SVR_ST_BAD_DRAFT_TOKEN, k_b outside [1, K] SVR_ST_BAD_NUM_DRAFT). */
int svr_kseq_verify(const void* target, const void* draft, int dtype, const int32_t* cand, const int32_t* num_cand,
                    const float* temperature, const int32_t* top_k, const float* top_p, uint64_t seed, int B, int K,
                    int V, int32_t* out_token, int32_t* accepted, uint32_t* status) {
    if (B < 0 || K < 1 || K > 13 || V < 1) return -1;
    if (dtype != SVR_DTYPE_F32 && dtype != SVR_DTYPE_BF16) return -1;
    if (B > 0 && (!target || !draft || !cand || !temperature || !out_token || !accepted)) return -1;
    double* logits = (double*)malloc(sizeof(double) * (size_t)V);
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    for (int b = 0; b < B; ++b) {
        int k = num_cand ? num_cand[b] : K;
        double T = (double)temperature[b];
        int tk = top_k ? top_k[b] : 0;
        double tp = top_p ? (double)top_p[b] : 1.0;
        uint32_t st = gumbel_params(k, K, T, tk, tp); /* the same parameter rules (k plays gamma's part) */
        if (!(st & SVR_ST_BAD_NUM_DRAFT))
            for (int i = 0; i < k; ++i) {
                int32_t x = cand[(size_t)b * K + i];
                if (x < 0 || x >= V) st |= SVR_ST_BAD_DRAFT_TOKEN;
            }
        if (!st) st |= gumbel_row(target, dtype, (size_t)b * V, V, T, tk, tp, logits, p);
        if (!st) st |= gumbel_row(draft, dtype, (size_t)b * V, V, T, tk, tp, logits, q);
        if (status) status[b] = st;
        out_token[b] = -1;
        accepted[b] = -1;
        if (st) continue;
        double u[13];
        for (int i = 0; i < k; ++i) u[i] = svr_uniform(seed, (uint32_t)b, 1u, 3u + (uint32_t)i);
        int32_t idx = -1;
        out_token[b] = svr_kseq_step(p, q, V, k, cand + (size_t)b * K, u, svr_uniform(seed, (uint32_t)b, 1u, 1u),
                                     &idx);
        accepted[b] = idx;
    }
    free(logits);
    free(p);
    free(q);
    return 0;
}

/* One SpecTr round for one sequence [STR, section SpecTr]: K draft sequences of
 * length L (tok[K][L]), the target rows at every candidate's prefix of length
 * l = 0..L (target [K][L+1][V] logits) and the draft rows at lengths 0..L-1 (draft
 * [K][L][V]); rows of candidates that share a prefix must be equal (the first alive
 * candidate's are used).  At each position: K-SEQ over the alive candidates' next
 * tokens (duplicates kept, in candidate order), uniforms U(seed, b, l+1, 3+i) and
 * U(seed, b, l+1, 1); the emitted token Y keeps the candidates whose token equals
 * it; none left ends the round; after all L positions matched, a bonus token is
 * drawn from the target row at length L by inverse CDF with U(seed, b, L+1, 1).
 * Writes the emitted tokens to out[0..n-1] (n <= L+1) and returns n (-1 on a bad
 * row: a non-finite logit, a token outside [0, V), bad T / top-k / top-p). */
int svr_spectr_round(const void* target, const void* draft, int dtype, const int32_t* tok, int K, int L, int V,
                     float temperature, int top_k, float top_p, uint64_t seed, uint32_t b, int32_t* out) {
    if (K < 1 || K > 13 || L < 1 || V < 1) return -1;
    double T = (double)temperature, tp = (double)top_p;
    if (gumbel_params(1, 1, T, top_k, tp)) return -1;
    for (int j = 0; j < K; ++j)
        for (int l = 0; l < L; ++l)
            if (tok[(size_t)j * L + l] < 0 || tok[(size_t)j * L + l] >= V) return -1;
    double* logits = (double*)malloc(sizeof(double) * (size_t)V);
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    int alive[13], na = K, n = 0, rc = 0;
    for (int j = 0; j < K; ++j) alive[j] = j;
    for (int l = 0;; ++l) {
        const int j0 = alive[0];
        if (l == L) { /* every position matched: the bonus token from the target row at length L */
            if (gumbel_row(target, dtype, ((size_t)j0 * (L + 1) + L) * (size_t)V, V, T, top_k, tp, logits, p)) {
                rc = -1;
                break;
            }
            double v = svr_uniform(seed, b, (uint32_t)(L + 1), 1u), cum = 0.0;
            int y = -1, last = -1;
            for (int x = 0; x < V; ++x) {
                if (!(p[x] > 0.0)) continue;
                last = x;
                cum += p[x];
                if (cum > v) {
                    y = x;
                    break;
                }
            }
            out[n++] = y >= 0 ? y : last;
            break;
        }
        if (gumbel_row(target, dtype, ((size_t)j0 * (L + 1) + l) * (size_t)V, V, T, top_k, tp, logits, p) ||
            gumbel_row(draft, dtype, ((size_t)j0 * L + l) * (size_t)V, V, T, top_k, tp, logits, q)) {
            rc = -1;
            break;
        }
        int32_t cand[13];
        double u[13];
        for (int i = 0; i < na; ++i) {
            cand[i] = tok[(size_t)alive[i] * L + l];
            u[i] = svr_uniform(seed, b, (uint32_t)(l + 1), 3u + (uint32_t)i);
        }
        int32_t idx;
        const int y = svr_kseq_step(p, q, V, na, cand, u, svr_uniform(seed, b, (uint32_t)(l + 1), 1u), &idx);
        out[n++] = y;
        int m = 0;
        for (int i = 0; i < na; ++i)
            if (tok[(size_t)alive[i] * L + l] == y) alive[m++] = alive[i];
        na = m;
        if (na == 0) break;
    }
    free(logits);
    free(p);
    free(q);
    return rc ? -1 : n;
}
