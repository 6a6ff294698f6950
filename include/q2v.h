/*
 * q2v.h -- C ABI of libq2v, the GB300 (sm_103a) target-verifier step of lossless p/q
 * speculative decoding.
 *
 * The verifier of a speculative-decoding cycle runs the target model over K+1 rows
 * (one committed row and K draft rows) and then accepts or replaces the drafts
 * ("Optimizing DeepSeek-V4-Flash on a single NVIDIA GB10/GX10 with DSpark speculative
 * decoding", page 1, opening post, "Current results": the verifier takes about 148 ms
 * of a 169 ms cycle at about 5 target rows; page 2, the verifier-bottleneck reply: the
 * verify executes attention, routed MoE, projections and the vocabulary head over the
 * K+1 rows).  This library provides the two hot parts of that step:
 *
 *   q2_tiny_gemm     Y = A W^T for 1..64 activation rows against Q2B32 weights
 *                    (dense projections and the vocabulary head);
 *   q2_moe_grouped   the routed-expert FFN over the same rows (device routing,
 *                    fused gate+up+SiLU, down projection, weighted combine);
 *   pq_verify        the exact p/q rejection-sampling verify over target and draft
 *                    logits.
 *
 * Q2B32 weight format (a stand-in for the 2-bit GGUF formats that the pages name but
 * do not define): blocks of 32 consecutive weights of one row along K, 12 bytes each:
 * bytes 0..7 hold the 32 two-bit unsigned codes q, four per byte, low bits first
 * (code j in byte j/4, bits 2(j%4)..2(j%4)+1); bytes 8..9 an fp16 scale d; bytes
 * 10..11 an fp16 offset m (little-endian).  w = d*q + m.  A matrix with N rows and K
 * columns is N*(K/32) blocks, row-major over N, the K/32 blocks of a row contiguous.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library never
 *    allocates, frees or synchronises on the enqueue path; every call only enqueues
 *    kernels on `stream` and returns.
 *  - Workspace: each call takes a caller-owned device workspace of at least the size
 *    its *_workspace() query returns (16-byte aligned).  The first 256 bytes hold a
 *    device status word shared by all calls on that workspace; each call initialises
 *    the rest of the scratch it uses.  Calls that share a workspace must be ordered
 *    on one stream.
 *  - Errors found on the host (bad sizes, NULL or misaligned pointers, too small a
 *    workspace) are returned before anything is enqueued.  Errors found on the device
 *    (a draft token out of range, a weight scale outside the exact range) are recorded
 *    in the workspace's status word; the affected outputs are then unspecified.  Read
 *    and clear the word with q2_get_device_status().  No kernel traps, asserts or
 *    waits without a bound.
 */
#ifndef Q2V_H
#define Q2V_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t); 0 is the legacy default stream. */
typedef struct CUstream_st *q2_stream_t;

typedef enum {
    Q2_OK = 0,
    Q2_ERR_INVALID_ARG = 1, /* a size, count, pointer or temperature is invalid           */
    Q2_ERR_ALIGNMENT = 2,   /* a pointer or leading dimension breaks the alignment rules   */
    Q2_ERR_UNSUPPORTED = 3, /* valid, but outside the sizes this build implements          */
    Q2_ERR_WORKSPACE = 4,   /* workspace NULL, misaligned or smaller than the query        */
    Q2_ERR_CUDA = 5,        /* a CUDA runtime call (launch, attribute, copy) failed        */
    Q2_ERR_TIMEOUT = 6,     /* a bounded device-side wait gave up                          */
    Q2_ERR_BAD_TOKEN = 7,   /* device: a draft token is outside [0, V)                     */
    Q2_ERR_RANGE = 8,       /* device: a Q2B32 scale |d| >= 64 or infinite (outside the exact path) */
    Q2_ERR_BAD_TEMPERATURE = 9 /* device: a per-session temperature is negative or not finite */
} q2_status;

#define Q2_WORKSPACE_HEADER_BYTES 256

/* ------------------------------------------------------------------ tiny GEMM */

/* Workspace bytes for q2_tiny_gemm with these sizes (>= Q2_WORKSPACE_HEADER_BYTES). */
size_t q2_tiny_gemm_workspace(int M, int N, int K);

/*
 * Y[m][n] = sum_k A[m][k] * w[n][k]  for m < M, n < N   (Y = A W^T, fp32 out).
 *
 * The projection matmuls and the vocabulary head that the K+1-row verify runs (page 2 of
 * the thread above, verifier-bottleneck reply) with the tiny-batch matmul shapes of
 * post #1 (K+1 = 1..5 rows per session; up to 12 sessions batched in the cohort
 * post #20 describes).
 *
 *   W    Q2B32 weights of an [N,K] matrix: N*(K/32)*12 bytes, 16-byte aligned.
 *   N    output features, 1 <= N.          K   reduction length, K % 32 == 0, 32 <= K <= 8192.
 *   A    bf16 activations [M][lda] (row-major), 16-byte aligned, lda >= K, lda % 8 == 0.
 *   M    activation rows, 1 <= M <= 64.
 *   Y    fp32 output [M][ldy], ldy >= N, 4-byte aligned.  Fully overwritten for n < N.
 *   ws   workspace of q2_tiny_gemm_workspace(M,N,K) bytes (the size depends on M and K only).
 * The kernel (mma.sync, or tcgen05 for K % 128 == 0 with more rows) is chosen from the shape
 * and the device; both give the same bound below.  Accumulation is fp32; each product uses q*d rounded once to fp16 and the offset m
 * exactly, and activations converted to fp16 under an exact per-row power-of-two scale, so
 * |Y - exact| stays far below 2e-3 * sum_k |a_k w_k|.  Scales must satisfy |d| < 64 (real
 * 2-bit block scales are orders of magnitude smaller).
 * Device errors: Q2_ERR_RANGE if a block has |d| >= 64 (infinity included; a NaN scale is not
 * flagged and propagates to the outputs it touches).
 */
q2_status q2_tiny_gemm(const void *W, int N, int K, const uint16_t *A, int M, int lda,
                       float *Y, int ldy, void *ws, size_t ws_bytes, q2_stream_t stream);

/* ------------------------------------------------------------------ routed MoE */

/* Workspace bytes for q2_moe_grouped with these sizes. */
size_t q2_moe_grouped_workspace(int M, int E, int topk, int H, int F);

#define Q2_MOE_RENORMALIZE 1u /* divide the selected gate probabilities by their sum */

/*
 * Routed-expert FFN over M rows (the routed-expert part of the K+1-row verify; the fused
 * router, fused gate+up+SwiGLU decode and expert deduplication listed in "1x Spark tuned
 * DSpark for DeepSeek-V4-Flash ...", reply on the decode arc, and in "ds4-on-spark",
 * section "What the fork adds", where each active expert's gate/up weights are read once
 * for all rows routed to it):
 *
 *   prob[r] = softmax(router_logits[r][0..E));  top-`topk` experts by probability,
 *   ties to the lower expert index;  g = the selected probabilities (renormalised to
 *   sum 1 only when flags has Q2_MOE_RENORMALIZE);
 *   h = silu(x Wg_e^T) * (x Wu_e^T)  (silu(z) = z / (1 + e^-z)),   out = h Wd_e^T;
 *   Y[r] = sum over the selected slots, in descending-probability order, of g * out.
 *
 * Each active expert's weights are read once for all rows routed to it.
 *   Wg, Wu  Q2B32 [E][F rows][H/32 blocks];  Wd  Q2B32 [E][H rows][F/32 blocks]; 16-B aligned.
 *   E <= 256 experts, 1 <= topk <= min(E, 16), H and F multiples of 32, 32 <= H, F <= 8192.
 *   X       bf16 [M][H], 16-byte aligned, 1 <= M <= 64.
 *   router_logits fp32 [M][E].
 *   Y       fp32 [M][H] (overwritten).
 *   topk_ids_out int32 [M][topk], topk_w_out fp32 [M][topk]: optional (NULL to skip).
 *   flags   0 or Q2_MOE_RENORMALIZE.
 * Device errors: Q2_ERR_RANGE as for q2_tiny_gemm.
 */
q2_status q2_moe_grouped(const void *Wg, const void *Wu, const void *Wd, int E, int H, int F,
                         int topk, unsigned flags, const uint16_t *X, int M,
                         const float *router_logits, float *Y, int32_t *topk_ids_out,
                         float *topk_w_out, void *ws, size_t ws_bytes, q2_stream_t stream);

/* ------------------------------------------------------------------ p/q verify */

/* Workspace bytes for pq_verify with these sizes. */
size_t pq_verify_workspace(int S, int k, int V);

/*
 * Exact p/q rejection-sampling verify for S independent sessions of k drafts each
 * ("Optimizing DeepSeek-V4-Flash ...", page 1, opening post: drafts are sampled from
 * q, the target defines p, accepted tokens follow min(1, p(x)/q(x)), rejected drafts
 * are replaced from the positive residual distribution; posts #12 and #20 describe the
 * correction as exact; "1x Spark tuned DSpark ...", deep-dive, "On losslessness":
 * the verify rows are the only token source, drawn with the request's own sampler).
 *
 * For session s:  p_i = softmax(target[s][i] / T) (i = 0..k),  q_i = softmax(draft[s][i] / T)
 * (i < k).  For i = 0..k-1 with x_i = draft_tokens[s][i]: accept iff q_i(x_i) == 0 or
 * u_acc[s][i] < p_i(x_i) / q_i(x_i); stop at the first rejection j.  If j < k, draw y
 * from max(0, p_j - q_j) normalised (from p_j if that mass is zero); if all k are
 * accepted, draw the extra token y from p_k.  A draw takes the smallest token y (in
 * ascending index) whose cumulative mass exceeds u_fin[s] times the total.
 *
 *   target_logits fp32 [S][k+1][V];  draft_logits fp32 [S][k][V] (NULL allowed when k == 0);
 *                 both 16-byte aligned.
 *   draft_tokens  int32 [S][k], each must lie in [0, V) (else device Q2_ERR_BAD_TOKEN).
 *   u_acc fp32 [S][k], u_fin fp32 [S]: uniforms in [0, 1), supplied by the caller's
 *                 per-session RNG.
 *   S >= 1, 0 <= k <= 16, 1 <= V <= 2^28, temperature > 0 and finite.
 *   n_accepted    int32 [S]: j, in [0, k].
 *   out_tokens    int32 [S][k+1]: x_0..x_{j-1}, y, then -1.
 *   probs_out     optional fp32 [S][2k+1][V]: rows p_0..p_k then q_0..q_{k-1} (for tests).
 * Arithmetic is fp32, with compensated (two-sum) fp32 cross-chunk and cross-segment sums;
 * tokens equal the exact (fp64) result except when a uniform lies within about 1e-6 of a
 * decision boundary.
 */
q2_status pq_verify(const float *target_logits, const float *draft_logits,
                    const int32_t *draft_tokens, const float *u_acc, const float *u_fin,
                    int S, int k, int V, float temperature, int32_t *n_accepted,
                    int32_t *out_tokens, float *probs_out, void *ws, size_t ws_bytes,
                    q2_stream_t stream);

/*
 * pq_verify with one temperature per session, and the greedy verify.
 *   temperatures  fp32 [S] in device memory, 4-byte aligned: T_s for session s (p and q of a
 *                 session share it, as in pq_verify).  T_s = 0 selects the greedy verify for
 *                 that session (the T -> 0 limit, bit-exact decoding: "1x Spark tuned DSpark
 *                 ...", the reply on the decode arc; "Optimizing DeepSeek-V4-Flash ...", post
 *                 #20): draft x_i is accepted iff it is argmax p_i, the token after the first
 *                 rejection j (or the extra token, j = k) is argmax p_j, ties going to the lower
 *                 token index; the draft logits' values and the uniforms are then not used, and
 *                 probs_out rows are one-hot at each row's argmax.
 * Every other argument is as for pq_verify, and required as there (greedy sessions ignore
 * their uniforms and draft logits).  Device errors: as pq_verify, plus Q2_ERR_BAD_TEMPERATURE for a
 * negative, NaN or infinite T_s (that session gets n_accepted = -1 and tokens -1; the others are
 * unaffected).  The workspace is pq_verify_workspace(S, k, V).
 */
q2_status pq_verify_ex(const float *target_logits, const float *draft_logits,
                       const int32_t *draft_tokens, const float *u_acc, const float *u_fin,
                       int S, int k, int V, const float *temperatures, int32_t *n_accepted,
                       int32_t *out_tokens, float *probs_out, void *ws, size_t ws_bytes,
                       q2_stream_t stream);

/*
 * pq_verify without a workspace, for callers that cannot allocate device memory: e.g. a
 * decode loop inside a host framework whose memory pool already owns the device, so it has
 * no buffer to lend and must not call cudaMalloc (which can stall the device, or fail under
 * a reserved pool).  The pages have no counterpart of this entry point; it is a library
 * convenience.
 *
 * Arguments and results are those of pq_verify, minus ws/ws_bytes.  The scratch is a fixed
 * 2 MiB array in device memory that the library holds on every device that loads it, until
 * the process exits; nothing is allocated.  Host-detectable errors return before anything is
 * enqueued: the argument errors of pq_verify, and Q2_ERR_UNSUPPORTED for sizes whose
 * pq_verify_workspace(S, k, V) exceeds 2 MiB (at k = 4 drafts and V = 129,280, up to S = 15
 * sessions fit; S = 16 does not).  Each call looks up the array's address on the current
 * device (a host-side query; the first lookup on a device may load the library's device code
 * there, so make the first call on each device before any stream capture).  Every call shares
 * the one array and clears its status word; calls that may overlap on the GPU (other streams,
 * other host threads) race on it and must be ordered by the caller.  Device-detected errors
 * show in the outputs: a session with a draft token outside [0, V) gets n_accepted = -1.
 */
q2_status pq_verify_noalloc(const float *target_logits, const float *draft_logits,
                            const int32_t *draft_tokens, const float *u_acc, const float *u_fin,
                            int S, int k, int V, float temperature, int32_t *n_accepted,
                            int32_t *out_tokens, float *probs_out, q2_stream_t stream);

/* ------------------------------------------------------------------ vocabulary head + verify */

/* Workspace bytes for q2_lm_head_verify with these sizes (either choice of flags). */
size_t q2_lm_head_verify_workspace(int S, int k, int V, int K);

/*
 * The vocabulary head of the K+1-row verify followed by the p/q verify over its logits, with
 * the GEMM's epilogue fused with the verify's softmax statistics ("Optimizing DeepSeek-V4-Flash
 * ...", page 2, verifier-bottleneck reply: the vocabulary head is part of the K+1-row verify;
 * post #1, paragraph after the analyzer output: fused operations cut the memory traffic
 * between steps).
 *   target_logits[s][i][:] = A[s*(k+1) + i] W^T   (as q2_tiny_gemm, N = V), written to the
 *                 caller's fp32 [S][k+1][V] buffer (16-byte aligned), then
 *   the verify of pq_verify_ex (temperatures non-NULL: device fp32 [S], 0 = greedy) or of
 *   pq_verify (temperatures NULL: one temperature > 0 for every session) over those logits.
 *   W Q2B32 [V rows][K], A bf16 [S*(k+1)][lda]; 1 <= S*(k+1) <= 64; alignment, K and the
 *   verify's other arguments as for q2_tiny_gemm and pq_verify.
 * flags: Q2_LM_HEAD_FUSE_STATS -- when 17 <= S*(k+1) <= 64, K % 128 == 0 and V > 4096, the
 * tcgen05 GEMM's epilogue also reduces each target row's logits to (max, sum of exponentials)
 * partials, one per CTA, and the verify's statistics pass then reads only the draft logits.
 * Without the flag (the faster choice on GB300, where the statistics pass over the just-written,
 * L2-resident logits costs less than the epilogue's cross-lane reductions) the same kernels run
 * unfused.  The
 * results are those of q2_tiny_gemm followed by pq_verify(_ex) up to floating-point summation
 * order.  Device errors: those of both calls, in one status word.
 */
#define Q2_LM_HEAD_FUSE_STATS 1u
q2_status q2_lm_head_verify(const void *W, int V, int K, const uint16_t *A, int lda,
                            const float *draft_logits, const int32_t *draft_tokens,
                            const float *u_acc, const float *u_fin, int S, int k,
                            const float *temperatures, float temperature, unsigned flags,
                            float *target_logits, int32_t *n_accepted, int32_t *out_tokens,
                            float *probs_out, void *ws, size_t ws_bytes, q2_stream_t stream);

/* ------------------------------------------------------------------ yield quench (host) */

/* Per-session state of the terminal yield-quench controller ("ds4-on-spark" README, "The
 * break-even law"; "1x Spark tuned DSpark ...", "The break-even law, and why speculation
 * can't hurt you here"): the running regret in plain decode steps, the steps counted, and
 * whether speculation has been switched off for the rest of the request. */
typedef struct {
    double regret;
    int steps;
    int quenched;
} q2_quench_state;

/* Host memory, S entries: zero regret, no steps, not quenched.  Q2_ERR_INVALID_ARG for a NULL
 * state or S < 1. */
q2_status q2_quench_init(q2_quench_state *state, int S);

/* One verify step for S sessions (host code; n_accepted is the verify's output copied to the
 * host).  A session that is not quenched and has n_accepted[s] >= 0 adds
 * guard - (n_accepted[s] + 1) (one verify costs `guard` plain steps and commits
 * n_accepted + 1 tokens; 2.16 is the pages' calibration) to its regret and is quenched,
 * terminally, once the regret exceeds `threshold` (about 4 plain-step times).  Sessions with
 * n_accepted < 0 (a device error) are skipped.  Returns the number of sessions quenched by
 * this step, or -1 for invalid arguments (NULL pointers, S < 1, non-finite guard/threshold). */
int q2_quench_update(q2_quench_state *state, int S, const int32_t *n_accepted, double guard,
                     double threshold);

/* ------------------------------------------------------------------ measurement hook */

/* Kernels that q2_set_probe can bracket. */
typedef enum {
    Q2_PROBE_NONE = 0,
    Q2_PROBE_MOE_GATE_UP = 1, /* q2_moe_grouped: the gate+up grouped dequant GEMM          */
    Q2_PROBE_MOE_DOWN = 2,    /* q2_moe_grouped: the down grouped dequant GEMM             */
    Q2_PROBE_GEMM = 3,        /* q2_tiny_gemm: the dequant GEMM kernel (not the prep)      */
    Q2_PROBE_PQ_STATS = 4,    /* pq_verify: the per-row softmax statistics kernel          */
    Q2_PROBE_PQ_VERIFY = 5    /* pq_verify: the accept-scan and draw kernel                */
} q2_probe_kernel;

/* Timing hook for measurement harnesses; the verifier method has no counterpart.  From this
 * call on, every call that launches the kernel named by `kernel` records `ev_begin` on the
 * call's stream just before that launch and `ev_end` just after it, so that the caller can
 * read the kernel's own duration with cudaEventElapsedTime.  Under stream capture the two
 * records become external event nodes of the graph (cudaEventRecordExternal).
 *   ev_begin, ev_end: cudaEvent_t handles (passed as void *) created by the caller with
 *                     timing enabled; the library keeps them until the next q2_set_probe.
 *   kernel = Q2_PROBE_NONE turns the hook off (the events may then be NULL).
 * Errors: Q2_ERR_INVALID_ARG for an unknown kernel or a NULL event.  Process-wide state,
 * not thread-safe; a recording failure makes the bracketed call return Q2_ERR_CUDA. */
q2_status q2_set_probe(int kernel, void *ev_begin, void *ev_end);

/* Read-only HBM bandwidth probe for measurement harnesses; the verifier method has no
 * counterpart (the "ds4-on-spark" README, section "Roofline", measures copy and read-only
 * bandwidth the same way on GB10).  Enqueues on `stream` one kernel that reads every byte of
 * `buf` once (16-byte loads, L1 bypassed, evict-first in L2) and writes nothing, except *sink
 * when the folded value of the data happens to equal a fixed constant; time it with events
 * around the call.  The caller owns both buffers.
 *   buf   device memory, 16-byte aligned, `bytes` > 0 and a multiple of 16.
 *   sink  device memory, 4 bytes, 4-byte aligned.
 * Errors: Q2_ERR_INVALID_ARG, Q2_ERR_ALIGNMENT, Q2_ERR_CUDA (launch failure). */
q2_status q2_hbm_read_probe(const void *buf, size_t bytes, unsigned int *sink, q2_stream_t stream);

/* ------------------------------------------------------------------ status */

/* Synchronise `stream`, read the device status word of workspace `ws`, clear it, and
 * return it (Q2_OK if no device error was recorded since the last read). */
q2_status q2_get_device_status(const void *ws, q2_stream_t stream);

/* ------------------------------------------------------------------ failure detection */

/* Self-test of device-side failure detection; the verifier method has no counterpart.  Every
 * wait inside the library's kernels is bounded: the tcgen05 GEMM's roles wait on mbarriers for
 * at most 1 s, then record Q2_ERR_TIMEOUT and wind down.  This call exercises that give-up
 * path without a GPU fault.  It launches one CTA on `stream` in which one thread performs the
 * same bounded mbarrier wait on a barrier that nothing completes.  After 1 s the wait gives
 * up, Q2_ERR_TIMEOUT goes into the status word of `ws`, the kernel returns, and the context
 * stays usable, so the next q2_get_device_status(ws) returns Q2_ERR_TIMEOUT.
 *   ws  device workspace of at least Q2_WORKSPACE_HEADER_BYTES, 16-byte aligned; only its
 *       status word is written.
 * Errors: Q2_ERR_WORKSPACE for a NULL, misaligned or too small workspace; Q2_ERR_CUDA if the
 * launch fails. */
q2_status q2_selftest_wait_timeout(void *ws, size_t ws_bytes, q2_stream_t stream);

/* Static description of a status code. */
const char *q2_status_string(q2_status status);

/* Library version: major*10000 + minor*100 + patch. */
int q2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* Q2V_H */
