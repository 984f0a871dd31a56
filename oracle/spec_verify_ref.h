/*
 * spec_verify_ref.h -- CPU oracle for batched speculative-sampling verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load or call this code.  The
 * product path (the CUDA library) never links, loads or calls it, and this
 * oracle shares no code, header, constant table or helper with it.
 *
 * Everything here is plain, slow, fp64 C written from the pages:
 *   - "Fast Inference from Transformers via Speculative Decoding" review pages
 *     (Algorithm 1 "SpeculativeDecodingStep"; section "Speculative Sampling"),
 *   - the speculative-decoding survey page, section 4 (speculative_step),
 *   - "Speculative decoding: the art of guessing well", section 投机采样
 *     (the `verify` listing: bonus token via q_{gamma+1} := 0).
 * The Philox4x32-10 generator follows Salmon, Moraes, Dror and Shaw,
 * "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11).  Two adjacent
 * methods follow at the end: shared-noise (Gumbel-coupled) verification
 * ("the art of guessing well", section 共享噪声的采样) and K-SEQ
 * multi-candidate verification ("SpecTr" page, section K-SEQ).
 *
 * Parity status of each function is given in its comment in the .c file.
 */
#ifndef SPEC_VERIFY_REF_H
#define SPEC_VERIFY_REF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* logits storage types accepted by the oracle */
#define SVR_DTYPE_F32 0
#define SVR_DTYPE_BF16 1

/* per-sequence status bits (same values as the library's contract) */
#define SVR_ST_BAD_TEMPERATURE 0x01u
#define SVR_ST_BAD_TOP_K 0x02u
#define SVR_ST_BAD_TOP_P 0x04u
#define SVR_ST_BAD_NUM_DRAFT 0x08u
#define SVR_ST_BAD_DRAFT_TOKEN 0x10u
#define SVR_ST_NONFINITE 0x20u
#define SVR_ST_BAD_LENIENCE 0x80u

/* Philox4x32-10 block function: ctr[4], key[2] -> out[4]. */
void svr_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* Uniform in (0,1) on the 24-bit grid from counter (b, pos, draw, 0) and key = seed. */
double svr_uniform(uint64_t seed, uint32_t b, uint32_t pos, uint32_t draw);

/* Fill u_accept[B*G] (draw 0, pos = 1..G) and u_resid[B*(G+1)] (draw 1, pos = 1..G+1). */
void svr_philox_uniforms(uint64_t seed, int B, int G, double* u_accept, double* u_resid);

/* Normalise one row of logits into probabilities (temperature, then top-k, then top-p).
 * T == 0 gives the one-hot argmax (lowest id on ties).  top_k <= 0 or >= V: off.
 * top_p >= 1: off.  Returns 0, or -1 if the row has no finite maximum.
 * filter_margin (may be NULL) receives the smallest margin of the filter decisions. */
int svr_normalise(const double* logits, int V, double T, int top_k, double top_p, double* probs,
                  double* filter_margin);

/* The verification step for a batch, with the uniforms passed in.
 *
 * target: [B, G+1, V] logits, draft: [B, G, V] logits (dtype SVR_DTYPE_*)
 * draft_tokens [B, G]; num_draft [B] (NULL = all G); temperature [B];
 * top_k [B] (NULL = off); top_p [B] (NULL = off).
 * u_accept [B, G]: uniform for the acceptance test at position i (1-based i = index+1)
 * u_resid [B, G+1]: uniform for the residual / bonus draw at position j.
 *
 * Outputs: accepted_len [B], out_tokens [B, G+1], alpha [B, G].
 * Optional outputs (NULL to skip):
 *   pos_accept [B, G]   acceptance decision at every position 1..gamma_b (-1 beyond)
 *   pos_token  [B, G+1] residual/bonus token that position j would emit (-1 beyond)
 *   p_out [B, G+1, V], q_out [B, G, V]  normalised probabilities (0 beyond gamma_b)
 *   status [B]          SVR_ST_* bits
 *   accept_margin [B, G]  |u - p/q| of each acceptance decision (+inf if q(x) = 0)
 *   resid_margin [B, G+1] distance of v/Z to the nearest CDF edge of the chosen token
 *   filter_margin [B, 2G+1] smallest filter-boundary margin per row
 *                           (target rows 0..G, then draft rows 0..G-1)
 * When any of pos_accept / pos_token / accept_margin / resid_margin is given, every
 * position is evaluated; the main outputs are unchanged by that.
 * Returns 0, or a negative value on a bad argument. */
int svr_verify(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
               const int32_t* num_draft, const float* temperature, const int32_t* top_k,
               const float* top_p, const double* u_accept, const double* u_resid, int B, int G, int V,
               int32_t* accepted_len, int32_t* out_tokens, double* alpha, int32_t* pos_accept,
               int32_t* pos_token, double* p_out, double* q_out, uint32_t* status,
               double* accept_margin, double* resid_margin, double* filter_margin);

/* svr_verify with a per-sequence lenience l_b in [0, 1] ("Fast Inference from
 * Transformers via Speculative Decoding" review page, section Lenience: q(x) is
 * multiplied by l in the acceptance test).  lenience [B] (NULL = 1 everywhere,
 * which is svr_verify exactly):
 *   accept x_i iff u * l * q_i(x_i) < p_i(x_i)   (accept_margin |u - p/(l q)|, +inf if l q = 0)
 *   alpha_i = sum_x q_i(x) * P(accept | x) = sum_x min(q_i(x), p_i(x) / l)
 *             (x with p(x) > 0 and l q(x) <= p(x) always pass; l = 0 accepts exactly the
 *             tokens with p(x) > 0)
 *   the residual / bonus draw is unchanged: norm(max(0, p - q)), q_{gamma+1} := 0.
 * A lenience that is NaN or outside [0, 1] gives SVR_ST_BAD_LENIENCE. */
int svr_verify_ex(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                  const int32_t* num_draft, const float* temperature, const int32_t* top_k,
                  const float* top_p, const float* lenience, const double* u_accept, const double* u_resid,
                  int B, int G, int V, int32_t* accepted_len, int32_t* out_tokens, double* alpha,
                  int32_t* pos_accept, int32_t* pos_token, double* p_out, double* q_out, uint32_t* status,
                  double* accept_margin, double* resid_margin, double* filter_margin);

/* Same, drawing the uniforms from the Philox stream keyed by (seed, b, pos, draw). */
int svr_verify_seeded(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                      const int32_t* num_draft, const float* temperature, const int32_t* top_k,
                      const float* top_p, uint64_t seed, int B, int G, int V, int32_t* accepted_len,
                      int32_t* out_tokens, double* alpha, int32_t* pos_accept, int32_t* pos_token,
                      double* p_out, double* q_out, uint32_t* status, double* accept_margin,
                      double* resid_margin, double* filter_margin);

/* svr_verify_ex with the Philox uniforms of svr_verify_seeded. */
int svr_verify_ex_seeded(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                         const int32_t* num_draft, const float* temperature, const int32_t* top_k,
                         const float* top_p, const float* lenience, uint64_t seed, int B, int G, int V,
                         int32_t* accepted_len, int32_t* out_tokens, double* alpha, int32_t* pos_accept,
                         int32_t* pos_token, double* p_out, double* q_out, uint32_t* status,
                         double* accept_margin, double* resid_margin, double* filter_margin);

/* Gumbel-coupled (shared-noise) verification ("Speculative decoding: the art
 * of guessing well", section 共享噪声的采样).  The noise of token i at 1-based
 * position k of sequence b is g = -log(-log u), u = svr_gumbel_uniform(seed, b,
 * k, i): Philox4x32-10 with counter (b, k, 2, i >> 2) and key seed, word i & 3,
 * on the 24-bit grid.  Rows are normalised as in svr_normalise. */
#define SVR_MAX_G 32
double svr_gumbel_uniform(uint64_t seed, uint32_t b, uint32_t pos, uint32_t token);

/* Verification: target [B, G+1, V] logits, the drafter's tokens [B, G].  For each
 * sequence the target's token t_k = argmax_i(log p_k(i) + g_k,i) at k = 1..gamma_b+1
 * (T = 0: argmax of the logits), n = the first k with draft_k != t_k (gamma_b if
 * none), out = draft_1..draft_n, t_{n+1}, then -1.  target_tokens [B, G+1] (or
 * NULL) receives every t_k (-1 beyond gamma_b + 1), margin [B, G+1] (or NULL) the
 * gap between the best and the second-best score at each position.  status as
 * in svr_verify.  Returns 0, or -1 on bad sizes / pointers (G <= SVR_MAX_G). */
int svr_gumbel_verify(const void* target, int dtype, const int32_t* draft_tokens, const int32_t* num_draft,
                      const float* temperature, const int32_t* top_k, const float* top_p, uint64_t seed, int B,
                      int G, int V, int32_t* accepted_len, int32_t* out_tokens, int32_t* target_tokens,
                      double* margin, uint32_t* status);

/* The coupled drafter: draft_tokens[b, k-1] = argmax_i(log q_k(i) + g_k,i) for
 * k = 1..gamma_b with the same noise (0 for padding and invalid rows). */
int svr_gumbel_draft(const void* draft, int dtype, const int32_t* num_draft, const float* temperature,
                     const int32_t* top_k, const float* top_p, uint64_t seed, int B, int G, int V,
                     int32_t* draft_tokens);

/* K-SEQ multi-candidate verification at one position ("SpecTr: Fast Speculative
 * Decoding via Optimal Transport", section K-SEQ).  p: target probabilities [V],
 * q: draft probabilities [V] (normalised rows), k candidates drawn from q.
 *   svr_kseq_beta    beta(rho) = sum_x min(q(x), p(x) / rho)
 *   svr_kseq_rho     rho* in [1, k]: 1 - (1 - beta)^k = rho beta (bisection)
 *   svr_kseq_direct  A_rho*(x) = (P_A / beta) min(q(x), p(x) / rho*) into A[V];
 *                    returns P_A = 1 - (1 - beta)^k (0 if beta = 0)
 *   svr_kseq_step    the emitted token: the first candidate i with
 *                    u[i] * rho* * q(cand[i]) < p(cand[i]) (its index in
 *                    *accepted_index), else the residual p - A_rho* drawn by
 *                    inverse CDF in ascending id with v = u_res * sum (index -1). */
double svr_kseq_beta(const double* p, const double* q, int V, double rho);
double svr_kseq_rho(const double* p, const double* q, int V, int k);
double svr_kseq_direct(const double* p, const double* q, int V, int k, double* A, double* rho_out);
int svr_kseq_step(const double* p, const double* q, int V, int k, const int32_t* cand, const double* u,
                  double u_res, int32_t* accepted_index);

/* Batched K-SEQ at one position per row: target / draft logits [B, V], candidates
 * [B, K] (K <= 13), num_cand [B] or NULL (all K); uniforms svr_uniform(seed, b, 1,
 * 3 + i) per candidate and svr_uniform(seed, b, 1, 1) for the residual.  Outputs:
 * out_token [B], accepted [B] (candidate index or -1), status [B] (or NULL). */
int svr_kseq_verify(const void* target, const void* draft, int dtype, const int32_t* cand, const int32_t* num_cand,
                    const float* temperature, const int32_t* top_k, const float* top_p, uint64_t seed, int B, int K,
                    int V, int32_t* out_token, int32_t* accepted, uint32_t* status);

/* One SpecTr round for sequence b ("SpecTr" page, section SpecTr): K draft sequences
 * tok [K, L], target rows at every candidate's prefix [K, L+1, V], draft rows [K, L, V];
 * K-SEQ at each position over the alive candidates (uniforms U(seed, b, l+1, 3+i) and
 * U(seed, b, l+1, 1)), candidates whose token equals the emitted one stay alive, the
 * round ends when none do, or after L matched positions with a bonus token from the
 * target row at length L (U(seed, b, L+1, 1)).  Emitted tokens into out [L+1]; returns
 * their count, or -1 for a bad row.  K <= 13. */
int svr_spectr_round(const void* target, const void* draft, int dtype, const int32_t* tok, int K, int L, int V,
                     float temperature, int top_k, float top_p, uint64_t seed, uint32_t b, int32_t* out);

#ifdef __cplusplus
}
#endif

#endif
