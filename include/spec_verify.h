/*
 * spec_verify.h -- C ABI of the GB300 batched speculative-sampling verification library.
 *
 * What one call computes (per sequence b of a batch, all on the GPU, no host sync):
 *   1. normalise the target rows p_1..p_{gamma_b+1} and the draft rows q_1..q_{gamma_b}
 *      the same way: temperature, softmax, top-k, renormalise, top-p, renormalise
 *      ("Fast Inference from Transformers via Speculative Decoding" review page,
 *      section "Method: Speculative Decoding": temperature / top-k / nucleus /
 *      argmax are standard sampling from an adjusted distribution; argmax zeroes
 *      the non-max entries);
 *   2. alpha_i = sum_x min(p_i(x), q_i(x)) for i = 1..gamma_b
 *      ("Speculative decoding: the art of guessing well", section 投机采样);
 *   3. accept draft token x_i iff u_i * q_i(x_i) < p_i(x_i), u_i = U(seed, b, i, 0)
 *      (same page, the `verify` listing: uniform < min(1, p/q));
 *   4. n_b = number of draft tokens before the first rejection
 *      (review page, Algorithm 1 SpeculativeDecodingStep, step 3);
 *   5. one more token t drawn from norm(max(0, p_{n+1} - q_{n+1})) with
 *      q_{gamma_b+1} := 0 (the bonus token when every draft was accepted) by an
 *      inverse CDF in ascending token id with v = U(seed, b, n+1, 1) * Z
 *      (Algorithm 1 steps 4-5; the `verify` listing's "treat it as zero").
 * U(seed, b, pos, draw) = ((w >> 8) + 0.5) * 2^-24 with w = word 0 of
 * Philox4x32-10(counter = (b, pos, draw, 0), key = (lo32(seed), hi32(seed))).
 * Temperature 0 means greedy: p, q are one-hot at the argmax (lowest id on ties),
 * so a draft token is accepted iff it is the target's argmax.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers unless the name says host.  The
 *    caller owns every buffer; the library allocates nothing and keeps no
 *    state between calls beyond the caller's workspace (spec_verify_static
 *    excepted: it uses a fixed buffer of the library's own).
 *  - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 *    stream) and never synchronise with the host (spec_verify_host excepted).
 *  - Argument errors return a negative SV_E* status before anything is
 *    enqueued.  A failed launch returns SV_ECUDA.  Problems in the device-side
 *    data of one sequence (bad per-row parameters, non-finite logits, draft
 *    tokens out of range) never fail the call: that sequence gets
 *    accepted_len = 0, out_tokens = -1, alpha = 0 and its SV_ROW_* bits in
 *    row_status.
 *  - Layouts are row-major, vocabulary innermost.  Logit arrays must start on
 *    a 16-byte boundary.
 *  - Results are deterministic for a given seed; callers advance the seed
 *    every round.
 *  - Calls on the same workspace must not overlap on the GPU.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

typedef enum {
    SV_OK = 0,
    SV_EINVAL = -1,       /* a bad argument (null pointer, bad size, misaligned logits) */
    SV_EUNSUPPORTED = -2, /* unsupported combination (e.g. dtype) */
    SV_ECUDA = -3,        /* a CUDA launch or runtime call failed */
    SV_ETOO_LARGE = -4,   /* V, gamma_max or B beyond the supported maximum */
    SV_EWORKSPACE = -5,   /* workspace missing or smaller than spec_verify_workspace_size() */
    SV_ESCRATCH = -6      /* spec_verify_static: the shape needs more than SV_STATIC_SCRATCH_BYTES */
} sv_status;

/* per-sequence bits written to row_status */
#define SV_ROW_BAD_TEMPERATURE 0x01u /* temperature negative, NaN or infinite */
#define SV_ROW_BAD_TOP_K 0x02u       /* top_k < 0 */
#define SV_ROW_BAD_TOP_P 0x04u       /* top_p NaN, <= 0 or > 1 */
#define SV_ROW_BAD_NUM_DRAFT 0x08u   /* num_draft outside [1, gamma_max] */
#define SV_ROW_BAD_DRAFT_TOKEN 0x10u /* a draft token outside [0, V) */
#define SV_ROW_NONFINITE 0x20u       /* NaN or +inf logit, or a row with no finite logit */
#define SV_ROW_INTERNAL 0x40u        /* a device-side wait gave up (internal error); outputs are defaults */
#define SV_ROW_BAD_LENIENCE 0x80u    /* lenience NaN or outside [0, 1] (spec_verify_ex) */

/* supported maxima */
#define SV_MAX_GAMMA 32
#define SV_MAX_VOCAB 262144
#define SV_MAX_BATCH 16777216
#define SV_MAX_KSEQ 13 /* candidates per row of spec_verify_kseq */

/*
 * Bytes of device workspace one call needs for this shape (a pure host
 * function: no CUDA call).  The workspace may be reused by consecutive calls
 * on one stream; it needs no initialisation.  Returns 0 for invalid shapes.
 */
size_t spec_verify_workspace_size(int B, int gamma_max, int V, int dtype);

/*
 * The batched verification step.
 *
 * target_logits [B, gamma_max+1, V]  dtype logits of the target model (row i = p_{i+1})
 * draft_logits  [B, gamma_max, V]    dtype logits of the drafter (row i = q_{i+1})
 * dtype                              SV_F32 or SV_BF16, both logit arrays
 * draft_tokens  [B, gamma_max] int32 x_1..x_gamma; entries past gamma_b are ignored
 * num_draft     [B] int32            gamma_b in [1, gamma_max], or NULL = all gamma_max
 * temperature   [B] float            >= 0; 0 = greedy
 * top_k         [B] int32            0 or >= V = off; NULL = off everywhere
 * top_p         [B] float            in (0, 1], 1 = off; NULL = off everywhere
 * seed                               Philox key for this call
 * accepted_len  [B] int32 out        n_b in [0, gamma_b]; the round emits n_b + 1 tokens
 * out_tokens    [B, gamma_max+1] int32 out  x_1..x_n, then the residual/bonus token, then -1
 * alpha         [B, gamma_max] float out    alpha_i for i <= gamma_b, 0 beyond
 * p_out         [B, gamma_max+1, V] float out or NULL: normalised target probabilities
 * q_out         [B, gamma_max, V] float out or NULL: normalised draft probabilities
 *               (debug outputs; rows past gamma_b are written as zeros)
 * row_status    [B] uint32 out or NULL: SV_ROW_* bits, 0 = fine
 * workspace, workspace_bytes         device scratch of spec_verify_workspace_size() bytes
 * stream                             cudaStream_t
 */
int spec_verify(const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_tokens,
                const int32_t* num_draft, const float* temperature, const int32_t* top_k, const float* top_p,
                uint64_t seed, int B, int gamma_max, int V, int32_t* accepted_len, int32_t* out_tokens,
                float* alpha, float* p_out, float* q_out, uint32_t* row_status, void* workspace,
                size_t workspace_bytes, void* stream);

/* Path selection for spec_verify_ex (testing and measurement). */
typedef enum {
    SV_PATH_AUTO = 0,  /* greedy and top_k <= SV_STREAM_MAX_TOP_K rows: streaming top-k path; rows with no
                          top-k (with or without top-p): whole-row path; top_k > SV_STREAM_MAX_TOP_K: dense
                          cluster path (which also finishes whole-row units whose nucleus cut holds more
                          than 256 tied logits) */
    SV_PATH_DENSE = 1  /* every row through the dense (whole-row, cluster) path */
} sv_path;

#define SV_STREAM_MAX_TOP_K 256

/*
 * Extra, optional outputs and controls.  Zero-initialise, set struct_size =
 * sizeof(sv_options), fill what you need.
 *   pos_accept [B, gamma_max] int32: acceptance decision at every position
 *              1..gamma_b, evaluated even after the first rejection (-1 beyond)
 *   pos_token  [B, gamma_max+1] int32: the residual/bonus token each position
 *              j would emit if the round stopped there (-1 beyond gamma_b+1)
 *   path       sv_path
 *   ev_stream  two cudaEvent_t (or NULL) recorded on `stream` immediately
 *              before and after the streaming top-k kernel
 *   ev_dense   the same around the dense cluster kernel (top-k > 256)
 *   ev_free    the same around the whole-row kernel of rows with no top-k
 *              (its per-unit tail kernel follows, outside the events)
 *   ev_gumbel  the same around the one-pass kernel of spec_verify_gumbel's rows
 *              with no filter (temperature only); not recorded by other calls
 *   lenience   [B] float or NULL (1 everywhere): the lenient acceptance test of
 *              the review page's section Lenience -- draft token x_i is accepted
 *              iff u_i * l_b * q_i(x_i) < p_i(x_i), so no token is emitted with
 *              more than 1/l_b times its probability under p, and alpha_i becomes
 *              the acceptance probability sum_x min(q_i(x), p_i(x) / l_b).  The
 *              residual draw is unchanged.  l_b = 1 is the exact rule; NaN or a
 *              value outside [0, 1] gives SV_ROW_BAD_LENIENCE.
 *   wait_limit_ns  limit of each device-side wait on another warp or on a copy
 *              (0 = the default, 2 s; below 1000 a wait gives up after one try,
 *              since the device timer ticks about once a microsecond).  A wait that runs out makes the call mark
 *              SV_ROW_INTERNAL on the sequences of the kernel that gave up and of
 *              the paths whose kernels run after it in the same call (their
 *              outputs are the defaults of an invalid sequence); the context stays
 *              usable and the next call is unaffected.  For tests of that path;
 *              production callers leave it 0.
 */
typedef struct {
    uint32_t struct_size;
    int32_t* pos_accept;
    int32_t* pos_token;
    int32_t path;
    void* ev_stream[2];
    void* ev_dense[2];
    void* ev_free[2];
    const float* lenience;
    uint64_t wait_limit_ns;
    void* ev_gumbel[2];
} sv_options;

int spec_verify_ex(const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_tokens,
                   const int32_t* num_draft, const float* temperature, const int32_t* top_k, const float* top_p,
                   uint64_t seed, int B, int gamma_max, int V, int32_t* accepted_len, int32_t* out_tokens,
                   float* alpha, float* p_out, float* q_out, uint32_t* row_status, void* workspace,
                   size_t workspace_bytes, void* stream, const sv_options* options);

/*
 * Bytes of device staging that spec_verify_host needs (inputs and outputs
 * copied through it) plus the workspace; a pure host function.
 */
size_t spec_verify_host_staging_size(int B, int gamma_max, int V, int dtype, int has_num_draft, int has_top_k,
                                     int has_top_p);

/*
 * End-to-end form: the same computation on HOST buffers (pinned memory gives
 * asynchronous copies).  Inputs are copied to `device_staging` with one
 * cudaMemcpyAsync per array, spec_verify runs, the three outputs are copied
 * back, and the call returns after cudaStreamSynchronize(stream).
 * device_staging: device buffer of spec_verify_host_staging_size() bytes,
 * 256-byte aligned.  Optional host arrays may be NULL as in spec_verify.
 */
int spec_verify_host(const void* host_target_logits, const void* host_draft_logits, int dtype,
                     const int32_t* host_draft_tokens, const int32_t* host_num_draft,
                     const float* host_temperature, const int32_t* host_top_k, const float* host_top_p,
                     uint64_t seed, int B, int gamma_max, int V, int32_t* host_accepted_len,
                     int32_t* host_out_tokens, float* host_alpha, void* device_staging, size_t staging_bytes,
                     void* stream);

/*
 * The same step as spec_verify with no workspace argument and no allocation:
 * the scratch is a fixed device buffer of SV_STATIC_SCRATCH_BYTES owned by the
 * library (the pages have no counterpart; this is a deployment form).
 *
 * For callers that cannot allocate device memory between decode steps: a
 * plain C/C++ host with no caching allocator to own a workspace, or a loop
 * that must not call cudaMalloc / cudaFree (cudaFree waits for the whole
 * device, stalling every other stream).
 *
 * Arguments, outputs and errors are those of spec_verify, plus:
 *  - SV_ESCRATCH, before anything is enqueued, when
 *    spec_verify_workspace_size(B, gamma_max, V, dtype) > SV_STATIC_SCRATCH_BYTES
 *    (8 MiB; that query tells a caller beforehand whether a shape fits -- decode
 *    batches of a few dozen sequences at 128k-152k vocabularies do); beyond it,
 *    use spec_verify with a workspace;
 *  - SV_ECUDA if the buffer's address cannot be looked up.
 * The first call on each device looks the buffer's address up, once per CUDA
 * context (so again after cudaDeviceReset); make that call outside any stream
 * capture.  All calls on a device share the one
 * buffer: calls that may overlap on the GPU race and must be ordered (one
 * stream, or events).  Nothing has to be cleared between calls.
 */
#define SV_STATIC_SCRATCH_BYTES (8u << 20)

int spec_verify_static(const void* target_logits, const void* draft_logits, int dtype,
                       const int32_t* draft_tokens, const int32_t* num_draft, const float* temperature,
                       const int32_t* top_k, const float* top_p, uint64_t seed, int B, int gamma_max, int V,
                       int32_t* accepted_len, int32_t* out_tokens, float* alpha, float* p_out, float* q_out,
                       uint32_t* row_status, void* stream);

/*
 * Shared-noise (Gumbel-coupled) verification ("Speculative decoding: the art of
 * guessing well", section 共享噪声的采样, the gumbel_verify listing and the
 * Gumbel-max identity: sampling from softmax(l) is argmax(l + g) with g Gumbel).
 * The drafter and the target use the same noise g_k at each position k, so the
 * target's own sample there is t_k = argmax_i(log p_k(i) + g_k,i); the round keeps
 * the longest prefix of draft tokens equal to t_1, t_2, ..., then emits the target's
 * token at the first difference (t_{gamma_b+1} when every draft token matched).
 * The emitted tokens are exactly the target's own samples, whatever the drafter.
 *
 * p_k is the target row k normalised as in spec_verify (temperature, top-k, top-p;
 * log p = -inf outside the kept set); argmax ties go to the lower token id;
 * temperature 0 is the plain argmax of the logits (no noise).  The noise of token i
 * at 1-based position k of sequence b is g = -ln(-ln u), u = ((w >> 8) + 1/2) 2^-24,
 * w = word (i & 3) of Philox4x32-10(counter = (b, k, 2, i >> 2), key = (lo32(seed),
 * hi32(seed))) -- draw 2, apart from the draws 0 and 1 of spec_verify.  A drafter
 * sharing the noise proposes argmax_i(log q_k(i) + g_k,i) with the same g.
 *
 * target_logits [B, gamma_max+1, V] dtype     (no draft logits are needed)
 * draft_tokens, num_draft, temperature, top_k, top_p, seed, B, gamma_max, V: as spec_verify
 * accepted_len  [B] int32 out                 n_b: draft tokens before the first difference
 * out_tokens    [B, gamma_max+1] int32 out    x_1..x_n, t_{n+1}, then -1
 * target_tokens [B, gamma_max+1] int32 out or NULL: t_k for k <= gamma_b + 1 (-1 beyond)
 * row_status    [B] uint32 out or NULL        SV_ROW_* bits (lenience does not apply)
 * workspace     spec_verify_workspace_size() bytes for the same shape and dtype
 * options       NULL or sv_options: path, pos_accept (draft k equals t_k), wait_limit_ns
 *               and the events are honoured; lenience is ignored
 * Rows with neither top-k nor top-p (temperature > 0) take one pass: log p differs
 * from l / T by a constant of the row, so t_k = argmax_i(l_i / T + g_k,i) needs no
 * maximum or sum; the batch's rows are cut into equal parts, one per CTA.
 * Errors and asynchrony as spec_verify.
 */
int spec_verify_gumbel(const void* target_logits, int dtype, const int32_t* draft_tokens, const int32_t* num_draft,
                       const float* temperature, const int32_t* top_k, const float* top_p, uint64_t seed, int B,
                       int gamma_max, int V, int32_t* accepted_len, int32_t* out_tokens, int32_t* target_tokens,
                       uint32_t* row_status, void* workspace, size_t workspace_bytes, void* stream,
                       const sv_options* options);

/*
 * K-SEQ multi-candidate verification of one position per row ("SpecTr: Fast
 * Speculative Decoding via Optimal Transport" page, section K-SEQ, eqs. (4)-(7)
 * and the residual distribution; that page names the draft p and the target q,
 * here p is the target and q the draft).  Row b holds k_b candidates X_i drawn
 * independently from the drafter's q.  With beta(rho) = sum_x min(q(x), p(x)/rho)
 * and rho* the root in [1, k] of 1 - (1 - beta)^k = rho beta, candidate i (in the
 * given order) is accepted iff u_i rho* q(X_i) < p(X_i); the first accepted one is
 * emitted; if none is, a token is drawn from the residual p - A with
 * A(x) = (P_A / beta) min(q(x), p(x)/rho*), P_A = 1 - (1 - beta)^k, by the inverse
 * CDF in ascending token id (no residual mass: from p itself).  The output law is
 * exactly p.  Uniforms: u_i = U(seed, b, 1, 3 + i), the residual's U(seed, b, 1, 1)
 * (U as for spec_verify).  p and q are normalised as in spec_verify.
 *
 * target_logits  [B, V] dtype, draft_logits [B, V] dtype
 * candidates     [B, K] int32 in [0, V); entries past k_b are ignored
 * num_candidates [B] int32 k_b in [1, K], or NULL = all K (K <= SV_MAX_KSEQ)
 * temperature, top_k, top_p: as spec_verify
 * out_token      [B] int32 out: the emitted token (-1 for an invalid row)
 * accepted       [B] int32 out: the index of the accepted candidate, or -1 (residual)
 * row_status     [B] uint32 out or NULL: SV_ROW_* bits (SV_ROW_BAD_NUM_DRAFT for k_b,
 *                SV_ROW_BAD_DRAFT_TOKEN for a candidate outside [0, V))
 * workspace      spec_verify_kseq_workspace_size() bytes
 * options        NULL or sv_options: path (SV_PATH_DENSE sends every row to the cluster
 *                kernel), ev_stream and ev_dense (the events around the streaming and
 *                cluster kernels) and wait_limit_ns are honoured; the rest is ignored
 * Rows with 1 <= top_k <= SV_STREAM_MAX_TOP_K, or temperature 0, are supported on
 * their kept lists: the streaming top-k kernel selects both rows' candidates and
 * one warp solves rho* and draws over those lists.  Other rows are each one unit
 * of the cluster kernel (the rows are held on chip while rho* is found).  Errors
 * and asynchrony as spec_verify.
 */
size_t spec_verify_kseq_workspace_size(int B, int K, int V, int dtype);
int spec_verify_kseq(const void* target_logits, const void* draft_logits, int dtype, const int32_t* candidates,
                     const int32_t* num_candidates, const float* temperature, const int32_t* top_k,
                     const float* top_p, uint64_t seed, int B, int K, int V, int32_t* out_token, int32_t* accepted,
                     uint32_t* row_status, void* workspace, size_t workspace_bytes, void* stream,
                     const sv_options* options);

/* A static English description of a status code. */
const char* spec_verify_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
