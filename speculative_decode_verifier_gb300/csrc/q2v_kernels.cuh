// q2v_kernels.cuh -- launch interfaces between the C ABI (q2v_api.cu) and the kernels.
#pragma once

#include "q2v_common.cuh"
#include "q2v_mma_core.cuh"

namespace q2v {

// Host-side caches of per-device launch state (a kernel's dynamic shared-memory opt-in and its
// occupancy are properties of a device) are indexed by the current device's ordinal; an
// ordinal beyond the cache (-1 here) is served without caching.
constexpr int kCacheDevices = 64;
inline int cache_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kCacheDevices) return -1;
    return d;
}

// ------------------------------------------------------------------ GEMM

cudaError_t launch_prep_bf16(const uint16_t *src, int ld, const int *rows, int R, int K, const PrepPtrs &P,
                             const PrepLayout &L, cudaStream_t s);
cudaError_t launch_gemm_small(const void *W, int N, int K, const PrepPtrs &P, const PrepLayout &L, int M,
                              float *Y, int ldy, unsigned int *status, cudaStream_t s);
// The streaming variant for M <= 8 against many weight rows (q2v_gemm.cu): persistent CTAs with
// per-warp weight rings; K % 256 == 0 and N % 16 == 0 (stream_gemm_usable).
bool stream_gemm_usable(int M, int N, int K);
bool stream_gemm_preferred(int M, int N, int K, int sms);
cudaError_t launch_gemm_stream(const void *W, int N, int K, const PrepPtrs &P, const PrepLayout &L, int M, float *Y,
                               int ldy, unsigned int *status, int num_sms, cudaStream_t s);

// ------------------------------------------------------------------ p/q verify

constexpr int kMaxDrafts = 16;
constexpr int kMaxRows = 2 * kMaxDrafts + 1;
constexpr int kWarpTierMaxV = 4096;   // sessions with V at most this use one warp each
constexpr int kChunkAlign = 128;      // chunk lengths are multiples of this (float4 x 32 lanes)
constexpr int kMaxChunks = 1024;      // chunks per session (workspace sizing bound)
constexpr int kSegsPerChunk = 8;      // warp segments per chunk (one per warp of the verify CTA)

struct PqArgs {
    const float *target;
    const float *draft;
    const int32_t *drafts;
    const float *u_acc;
    const float *u_fin;
    int S, k, V;
    float beta;     // log2(e) / T (every session, when temps is null)
    const float *temps;  // [S] per-session temperatures, nullable: 0 = greedy
    int32_t *n_acc;
    int32_t *tokens;
    float *probs;
    unsigned int *status;
};

struct PqSplit {
    int C;               // chunks per session
    int L;               // chunk length (multiple of kChunkAlign)
    float *stats;        // [S][2k+1][C] float2 (max, sum)
    float *mass;         // [S][C][8] draw mass of each warp segment of each chunk
    float *pmass;        // [S][C][8] p_j mass of each segment (zero-residual fallback)
    unsigned int *tickets;  // [S]
    float2 *xin;         // [S][k] (target, draft) logit at each draft token, gathered by kernel 1
    // Target rows' partials made elsewhere (the fused vocabulary-head GEMM), nullable:
    // [S][k+1][Ct] float2, one per 128-token tile.  When set, the statistics kernel only
    // streams the draft rows and the combine reads the target rows from here.
    const float *tstats;
    int Ct;
};

cudaError_t launch_pq_verify(const PqArgs &a, const PqSplit &sp, bool warp_tier, int num_sms, cudaStream_t st);
// pq_verify's host-side argument checks alone (q2v_api.cu): Q2_OK or the status pq_verify would
// return for these arguments before enqueueing anything.
q2_status pq_verify_precheck(const float *target_logits, const float *draft_logits, const int32_t *draft_tokens,
                             const float *u_acc, const float *u_fin, int S, int k, int V, float temperature,
                             int32_t *n_accepted, int32_t *out_tokens, float *probs_out);

// ------------------------------------------------------------------ routed MoE

constexpr int kMaxKSplits = 8;  // K splits of the grouped GEMM units (workspace sizing bound)

struct MoeArgs {
    const uint8_t *Wg, *Wu, *Wd;
    int E, H, F, topk, M;
    unsigned flags;
    const uint16_t *X;
    const float *router;
    float *Y;
    int32_t *ids_out;
    float *w_out;
    unsigned int *status;
};

struct MoeWs {
    int *counts;      // [E]
    int *offsets;     // [E+1]
    int *active;      // [E] expert ids with count > 0, ascending; active_n at active[E]
    int *pair_row;    // [M*topk] activation row of each expert-grouped pair
    int *pair_of;     // [M*topk] grouped position of (row, slot)
    int *slot_of;     // [M*topk] (row, slot) index r*topk + t of each grouped position
    float *gate_w;    // [M*topk] gate weight of (row, slot)
    float *h;         // [KS][2][M*topk][F] fp32 gate and up partial sums per K split
    float *out;       // [KS][M*topk][H] fp32 down projection partial sums per K split, by (row, slot)
    PrepPtrs prepX;   // prepared X rows (K = H)
    PrepPtrs prepH;   // prepared h rows (K = F)
};

cudaError_t launch_moe(const MoeArgs &a, const MoeWs &w, int num_sms, cudaStream_t s);

// q2_tiny_gemm on the tcgen05 tensor cores (q2v_umma.cu), for 1 <= M <= 64 and K % 128 == 0
// (the weight rows then start on 16-byte boundaries, as TMA needs).  umma_gemm_usable says
// whether a shape can take that path; umma_gemm_preferred picks the faster path for a shape on
// `sms` SMs: tcgen05 above 16 rows, and at 5..16 rows once there are enough 128-row tiles per
// SM.  The crossovers, measured on GB300 at K = 4096, are about 108 weight rows per SM at 9..16
// activation rows (where the mma.sync kernel needs two 8-row slices) and 216 at 5..8 rows; at
// fewer rows, or fewer weight rows, the mma.sync kernel is the faster one.
bool umma_gemm_usable(int M, int K);
bool umma_gemm_preferred(int M, int N, int K, int sms);
// The prep writes the activation operand image into a workspace region of umma_gemm_ws_bytes.
size_t umma_gemm_ws_bytes(int M, int K);
cudaError_t launch_prep_umma(const uint16_t *A, int lda, int M, int K, void *ws_region, cudaStream_t s);

// Fusion of the vocabulary-head GEMM with the verify's softmax statistics: activation row m
// is row m % k1 of session m / k1; the epilogue merges, over the 128-token tiles its CTA
// computes, each row's (max, sum 2^((y - max) beta_s)) partial of the logits it stores
// (greedy sessions: (max, first argmax as int bits)) and writes one partial per row per CTA
// to tstats [S][k1][grid].  tstats null: a plain GEMM.
struct UmFuse {
    float *tstats;
    const float *temps;  // [S] per-session temperatures (0 = greedy), nullable: beta for all
    float beta;          // log2(e) / T when temps is null
    int k1;              // rows per session (k + 1)
};
cudaError_t launch_gemm_umma(const void *W, int N, int K, int M, const void *ws_region, float *Y, int ldy,
                             unsigned int *status, int num_sms, cudaStream_t s, const UmFuse &fuse);
// The tcgen05 GEMM's grid (one persistent CTA per SM, at most one per 128-row tile); the fused
// statistics are one partial per CTA.
inline int umma_gemm_grid(int N, int num_sms) { return N < 1 ? 1 : (cdiv(N, 128) < num_sms ? cdiv(N, 128) : num_sms); }

// One CTA whose bounded mbarrier wait runs out and records Q2_ERR_TIMEOUT in *status
// (q2_selftest_wait_timeout, q2v_umma.cu).
cudaError_t launch_wait_selftest(unsigned int *status, cudaStream_t s);

// Measurement hook (q2_set_probe): records the caller's begin (end = 0) or end (end = 1)
// event on s when `kernel` is the bracketed one; a no-op otherwise.
enum ProbeKernel : int { kProbeMoeGateUp = 1, kProbeMoeDown = 2, kProbeGemm = 3, kProbePqStats = 4, kProbePqVerify = 5 };
cudaError_t probe_mark(int kernel, int end, cudaStream_t s);

// launch(), bracketed by the probe events of `kernel`.
template <typename F>
cudaError_t probed(int kernel, cudaStream_t s, F &&launch) {
    cudaError_t e = probe_mark(kernel, 0, s);
    if (e != cudaSuccess) return e;
    e = launch();
    if (e != cudaSuccess) return e;
    return probe_mark(kernel, 1, s);
}

}  // namespace q2v
