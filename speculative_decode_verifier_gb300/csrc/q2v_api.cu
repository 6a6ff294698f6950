// q2v_api.cu -- the extern "C" boundary of libq2v: argument checks, workspace carving
// and kernel dispatch.  Nothing here allocates, frees or synchronises except
// q2_get_device_status, whose job is to read the device status word.
#include <math.h>
#include <stdio.h>

#include "q2v_kernels.cuh"

using namespace q2v;

namespace {

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];  // cached SM count per device (0 = unknown)

int device_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    if (g_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

unsigned int *status_word(void *ws) { return &static_cast<WsHeader *>(ws)->status; }

// Sequential carve of 256-byte-aligned regions after the header.
struct Carver {
    char *base;
    size_t off;
    explicit Carver(void *ws) : base(static_cast<char *>(ws)), off(Q2_WORKSPACE_HEADER_BYTES) {}
    void *take(size_t bytes) {
        void *p = base ? base + off : nullptr;
        off += align_up(bytes, 256);
        return p;
    }
};

q2_status check_ws(void *ws, size_t ws_bytes, size_t need) {
    if (!ws || !aligned(ws, 16) || ws_bytes < need) return Q2_ERR_WORKSPACE;
    return Q2_OK;
}

q2_status cuda_status(cudaError_t e) { return e == cudaSuccess ? Q2_OK : Q2_ERR_CUDA; }

// ---------------------------------------------------------------- tiny GEMM sizes

bool gemm_k_ok(int K) { return K >= kBlockK && K % kBlockK == 0 && K <= kMaxTileWarps * kTileBlocks * kBlockK; }

// Either path's needs (which path runs depends on N and the device), so a workspace sized
// once fits every call with these M and K.
size_t gemm_ws_bytes(int M, int K) {
    Carver c(nullptr);
    const size_t prep = PrepLayout(K).bytes(M);
    c.take(umma_gemm_usable(M, K) ? std::max(umma_gemm_ws_bytes(M, K), prep) : prep);
    return c.off;
}

// ---------------------------------------------------------------- pq_verify sizes

int pq_cmax(int V) { return std::min(cdiv(V, kChunkAlign), kMaxChunks); }

struct PqCarve {
    float *stats;
    float *mass, *pmass;
    unsigned int *tickets;
    float2 *xin;
    size_t bytes;
};

PqCarve pq_carve_from(Carver &c, int S, int k, int V) {
    const size_t off0 = c.off;
    PqCarve r{};
    const size_t R = 2 * (size_t)k + 1, C = pq_cmax(V);
    r.stats = static_cast<float *>(c.take((size_t)S * R * C * 2 * sizeof(float)));
    r.mass = static_cast<float *>(c.take((size_t)S * C * kSegsPerChunk * sizeof(float)));
    r.pmass = static_cast<float *>(c.take((size_t)S * C * kSegsPerChunk * sizeof(float)));
    r.tickets = static_cast<unsigned int *>(c.take((size_t)S * sizeof(unsigned int)));
    r.xin = static_cast<float2 *>(c.take((size_t)S * std::max(k, 1) * sizeof(float2)));
    r.bytes = c.off - off0 + Q2_WORKSPACE_HEADER_BYTES;  // as a workspace of its own
    return r;
}

PqCarve pq_carve(void *ws, int S, int k, int V) {
    Carver c(ws);
    return pq_carve_from(c, S, k, V);
}

// ---------------------------------------------------------------- MoE sizes

struct MoeCarve {
    MoeWs w;
    size_t bytes;
};

MoeCarve moe_carve(void *ws, int M, int E, int topk, int H, int F) {
    Carver c(ws);
    MoeCarve r{};
    const size_t P = (size_t)M * topk;
    r.w.counts = static_cast<int *>(c.take((size_t)E * sizeof(int)));
    r.w.offsets = static_cast<int *>(c.take((size_t)(E + 1) * sizeof(int)));
    r.w.active = static_cast<int *>(c.take((size_t)(E + 1) * sizeof(int)));
    r.w.pair_row = static_cast<int *>(c.take(P * sizeof(int)));
    r.w.pair_of = static_cast<int *>(c.take(P * sizeof(int)));
    r.w.slot_of = static_cast<int *>(c.take(P * sizeof(int)));
    r.w.gate_w = static_cast<float *>(c.take(P * sizeof(float)));
    r.w.h = static_cast<float *>(c.take((size_t)kMaxKSplits * 2 * P * (size_t)F * sizeof(float)));
    r.w.out = static_cast<float *>(c.take((size_t)kMaxKSplits * P * (size_t)H * sizeof(float)));
    const PrepLayout LX(H), LH(F);
    void *px = c.take(LX.bytes(M));
    void *ph = c.take(LH.bytes((int)P));
    if (ws) {
        r.w.prepX = PrepPtrs::carve(px, LX, M);
        r.w.prepH = PrepPtrs::carve(ph, LH, (int)P);
    }
    r.bytes = c.off;
    return r;
}

}  // namespace

// ------------------------------------------------------------------ measurement hook

namespace {
int g_probe_kernel = 0;
cudaEvent_t g_probe_ev[2] = {nullptr, nullptr};
}  // namespace

cudaError_t q2v::probe_mark(int kernel, int end, cudaStream_t s) {
    if (g_probe_kernel == 0 || kernel != g_probe_kernel) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    if (cs == cudaStreamCaptureStatusActive)
        return cudaEventRecordWithFlags(g_probe_ev[end], s, cudaEventRecordExternal);
    return cudaEventRecord(g_probe_ev[end], s);
}

namespace {
q2_status pq_verify_impl(const float *target_logits, const float *draft_logits, const int32_t *draft_tokens,
                         const float *u_acc, const float *u_fin, int S, int k, int V, float temperature,
                         const float *temps, int32_t *n_accepted, int32_t *out_tokens, float *probs_out, void *ws,
                         size_t ws_bytes, q2_stream_t stream);
q2_status pq_check_args(const float *target_logits, const float *draft_logits, const int32_t *draft_tokens,
                        const float *u_acc, const float *u_fin, int S, int k, int V, int32_t *n_accepted,
                        int32_t *out_tokens, float *probs_out);
void pq_setup(PqArgs &a, PqSplit &sp, Carver &c, const float *target_logits, const float *draft_logits,
              const int32_t *draft_tokens, const float *u_acc, const float *u_fin, int S, int k, int V,
              float temperature, const float *temps, int32_t *n_accepted, int32_t *out_tokens, float *probs_out,
              unsigned int *status, int sms);
}  // namespace

extern "C" {

int q2_version(void) { return Q2V_VERSION; }

q2_status q2_set_probe(int kernel, void *ev_begin, void *ev_end) {
    if (kernel < Q2_PROBE_NONE || kernel > Q2_PROBE_PQ_VERIFY) return Q2_ERR_INVALID_ARG;
    if (kernel != Q2_PROBE_NONE && (!ev_begin || !ev_end)) return Q2_ERR_INVALID_ARG;
    g_probe_kernel = kernel;
    g_probe_ev[0] = static_cast<cudaEvent_t>(ev_begin);
    g_probe_ev[1] = static_cast<cudaEvent_t>(ev_end);
    return Q2_OK;
}

const char *q2_status_string(q2_status s) {
    switch (s) {
        case Q2_OK: return "ok";
        case Q2_ERR_INVALID_ARG: return "invalid argument";
        case Q2_ERR_ALIGNMENT: return "misaligned pointer or leading dimension";
        case Q2_ERR_UNSUPPORTED: return "unsupported size";
        case Q2_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case Q2_ERR_CUDA: return "CUDA runtime error";
        case Q2_ERR_TIMEOUT: return "device wait timed out";
        case Q2_ERR_BAD_TOKEN: return "draft token out of range";
        case Q2_ERR_RANGE: return "Q2B32 scale outside the exact range";
        case Q2_ERR_BAD_TEMPERATURE: return "per-session temperature negative or not finite";
    }
    return "unknown status";
}

q2_status q2_selftest_wait_timeout(void *ws, size_t ws_bytes, q2_stream_t stream) {
    const q2_status wst = check_ws(ws, ws_bytes, Q2_WORKSPACE_HEADER_BYTES);
    if (wst != Q2_OK) return wst;
    return cuda_status(launch_wait_selftest(status_word(ws), reinterpret_cast<cudaStream_t>(stream)));
}

q2_status q2_get_device_status(const void *ws, q2_stream_t stream) {
    if (!ws || !aligned(ws, 16)) return Q2_ERR_WORKSPACE;
    unsigned int st = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&st, ws, sizeof(st), cudaMemcpyDeviceToHost, s) != cudaSuccess) return Q2_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return Q2_ERR_CUDA;
    if (st != 0) {
        if (cudaMemsetAsync(const_cast<void *>(ws), 0, sizeof(st), s) != cudaSuccess) return Q2_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return Q2_ERR_CUDA;
    }
    return static_cast<q2_status>(st);
}

// ---------------------------------------------------------------- tiny GEMM

size_t q2_tiny_gemm_workspace(int M, int N, int K) {
    (void)N;
    if (M < 1 || M > 64 || !gemm_k_ok(K)) return Q2_WORKSPACE_HEADER_BYTES;
    return gemm_ws_bytes(M, K);
}

q2_status q2_tiny_gemm(const void *W, int N, int K, const uint16_t *A, int M, int lda, float *Y, int ldy,
                       void *ws, size_t ws_bytes, q2_stream_t stream) {
    if (!W || !A || !Y || N < 1 || M < 1 || K < kBlockK || K % kBlockK != 0 || lda < K || ldy < N)
        return Q2_ERR_INVALID_ARG;
    if (M > 64 || !gemm_k_ok(K)) return Q2_ERR_UNSUPPORTED;
    if (!aligned(W, 16) || !aligned(A, 16) || lda % 8 != 0 || !aligned(Y, 4)) return Q2_ERR_ALIGNMENT;
    const q2_status wst = check_ws(ws, ws_bytes, gemm_ws_bytes(M, K));
    if (wst != Q2_OK) return wst;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    Carver c(ws);
    const int sms = device_sms();
    if (stream_gemm_preferred(M, N, K, sms)) {  // few activation rows, many weight rows
        const PrepLayout L(K);
        const PrepPtrs P = PrepPtrs::carve(c.take(L.bytes(M)), L, M);
        if (launch_prep_bf16(A, lda, nullptr, M, K, P, L, s) != cudaSuccess) return Q2_ERR_CUDA;
        return cuda_status(probed(kProbeGemm, s, [&] {
            return launch_gemm_stream(W, N, K, P, L, M, Y, ldy, status_word(ws), sms, s);
        }));
    }
    if (umma_gemm_preferred(M, N, K, sms)) {
        void *img = c.take(umma_gemm_ws_bytes(M, K));
        if (launch_prep_umma(A, lda, M, K, img, s) != cudaSuccess) return Q2_ERR_CUDA;
        return cuda_status(probed(kProbeGemm, s, [&] {
            return launch_gemm_umma(W, N, K, M, img, Y, ldy, status_word(ws), sms, s, UmFuse{});
        }));
    }
    const PrepLayout L(K);
    const PrepPtrs P = PrepPtrs::carve(c.take(L.bytes(M)), L, M);
    const cudaError_t e = launch_prep_bf16(A, lda, nullptr, M, K, P, L, s);
    if (e != cudaSuccess) return Q2_ERR_CUDA;
    return cuda_status(
        probed(kProbeGemm, s, [&] { return launch_gemm_small(W, N, K, P, L, M, Y, ldy, status_word(ws), s); }));
}

// ---------------------------------------------------------------- routed MoE

size_t q2_moe_grouped_workspace(int M, int E, int topk, int H, int F) {
    if (M < 1 || M > 64 || E < 1 || E > 256 || topk < 1 || topk > 16 || topk > E || !gemm_k_ok(H) ||
        !gemm_k_ok(F))
        return Q2_WORKSPACE_HEADER_BYTES;
    return moe_carve(nullptr, M, E, topk, H, F).bytes;
}

q2_status q2_moe_grouped(const void *Wg, const void *Wu, const void *Wd, int E, int H, int F, int topk,
                         unsigned flags, const uint16_t *X, int M, const float *router_logits, float *Y,
                         int32_t *topk_ids_out, float *topk_w_out, void *ws, size_t ws_bytes,
                         q2_stream_t stream) {
    if (!Wg || !Wu || !Wd || !X || !router_logits || !Y || E < 1 || topk < 1 || topk > E || M < 1 || H < kBlockK ||
        F < kBlockK || H % kBlockK != 0 || F % kBlockK != 0 || (flags & ~Q2_MOE_RENORMALIZE) != 0)
        return Q2_ERR_INVALID_ARG;
    if (M > 64 || E > 256 || topk > 16 || !gemm_k_ok(H) || !gemm_k_ok(F)) return Q2_ERR_UNSUPPORTED;
    if (!aligned(Wg, 16) || !aligned(Wu, 16) || !aligned(Wd, 16) || !aligned(X, 16) || !aligned(router_logits, 4) ||
        !aligned(Y, 4) || !aligned(topk_ids_out, 4) || !aligned(topk_w_out, 4))
        return Q2_ERR_ALIGNMENT;
    const MoeCarve need = moe_carve(nullptr, M, E, topk, H, F);
    const q2_status wst = check_ws(ws, ws_bytes, need.bytes);
    if (wst != Q2_OK) return wst;
    MoeArgs a;
    a.Wg = static_cast<const uint8_t *>(Wg);
    a.Wu = static_cast<const uint8_t *>(Wu);
    a.Wd = static_cast<const uint8_t *>(Wd);
    a.E = E; a.H = H; a.F = F; a.topk = topk; a.M = M; a.flags = flags;
    a.X = X;
    a.router = router_logits;
    a.Y = Y;
    a.ids_out = topk_ids_out;
    a.w_out = topk_w_out;
    a.status = status_word(ws);
    const MoeCarve mc = moe_carve(ws, M, E, topk, H, F);
    return cuda_status(launch_moe(a, mc.w, device_sms(), reinterpret_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- p/q verify

size_t pq_verify_workspace(int S, int k, int V) {
    if (S < 1 || k < 0 || k > kMaxDrafts || V < 1 || V > (1 << 28)) return Q2_WORKSPACE_HEADER_BYTES;
    if (V <= kWarpTierMaxV) return Q2_WORKSPACE_HEADER_BYTES;
    return pq_carve(nullptr, S, k, V).bytes;
}

q2_status pq_verify(const float *target_logits, const float *draft_logits, const int32_t *draft_tokens,
                    const float *u_acc, const float *u_fin, int S, int k, int V, float temperature,
                    int32_t *n_accepted, int32_t *out_tokens, float *probs_out, void *ws, size_t ws_bytes,
                    q2_stream_t stream) {
    if (!(temperature > 0.0f) || !isfinite(temperature)) return Q2_ERR_INVALID_ARG;
    return pq_verify_impl(target_logits, draft_logits, draft_tokens, u_acc, u_fin, S, k, V, temperature, nullptr,
                          n_accepted, out_tokens, probs_out, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- fused vocabulary head + verify

size_t q2_lm_head_verify_workspace(int S, int k, int V, int K) {
    const long long M = (long long)S * (k + 1);
    if (S < 1 || k < 0 || k > kMaxDrafts || V < 1 || V > (1 << 28) || M > 64 || !gemm_k_ok(K))
        return Q2_WORKSPACE_HEADER_BYTES;
    // either GEMM path's regions (the path depends on the shape and the device), then the verify's
    Carver a(nullptr), b(nullptr);
    if (umma_gemm_usable((int)M, K)) {
        a.take(umma_gemm_ws_bytes((int)M, K));
        a.take((size_t)M * umma_gemm_grid(V, device_sms()) * sizeof(float2));
        if (V > kWarpTierMaxV) pq_carve_from(a, S, k, V);
    }
    b.take(PrepLayout(K).bytes((int)M));
    if (V > kWarpTierMaxV) pq_carve_from(b, S, k, V);
    return std::max(a.off, b.off);
}

q2_status q2_lm_head_verify(const void *W, int V, int K, const uint16_t *A, int lda, const float *draft_logits,
                            const int32_t *draft_tokens, const float *u_acc, const float *u_fin, int S, int k,
                            const float *temperatures, float temperature, unsigned flags, float *target_logits,
                            int32_t *n_accepted, int32_t *out_tokens, float *probs_out, void *ws, size_t ws_bytes,
                            q2_stream_t stream) {
    if (!W || !A || K < kBlockK || K % kBlockK != 0 || lda < K) return Q2_ERR_INVALID_ARG;
    if (!temperatures && (!(temperature > 0.0f) || !isfinite(temperature))) return Q2_ERR_INVALID_ARG;
    const q2_status ast = pq_check_args(target_logits, draft_logits, draft_tokens, u_acc, u_fin, S, k, V,
                                        n_accepted, out_tokens, probs_out);
    if (ast != Q2_OK) return ast;
    const long long M = (long long)S * (k + 1);
    if (M > 64 || !gemm_k_ok(K)) return Q2_ERR_UNSUPPORTED;
    if (!aligned(W, 16) || !aligned(A, 16) || lda % 8 != 0 || (temperatures && !aligned(temperatures, 4)))
        return Q2_ERR_ALIGNMENT;
    const q2_status wst = check_ws(ws, ws_bytes, q2_lm_head_verify_workspace(S, k, V, K));
    if (wst != Q2_OK) return wst;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int sms = device_sms();
    unsigned int *status = status_word(ws);
    if (flags & ~Q2_LM_HEAD_FUSE_STATS) return Q2_ERR_INVALID_ARG;
    const bool streamed = stream_gemm_preferred((int)M, V, K, sms);
    const bool umma = !streamed && umma_gemm_preferred((int)M, V, K, sms);
    const bool fused = (flags & Q2_LM_HEAD_FUSE_STATS) && umma && V > kWarpTierMaxV;
    Carver c(ws);
    // 1. target logits = A W^T (rows s*(k+1) + i), with the target rows' softmax partials
    //    taken in the tcgen05 epilogue when fused
    cudaError_t e;
    float *tstats = nullptr;
    const int Ct = umma_gemm_grid(V, sms);
    if (umma) {
        void *img = c.take(umma_gemm_ws_bytes((int)M, K));
        // the partials region is carved either way, so the workspace size does not depend on flags
        float *tregion = static_cast<float *>(c.take((size_t)M * Ct * sizeof(float2)));
        if (fused) tstats = tregion;
        e = launch_prep_umma(A, lda, (int)M, K, img, s);
        if (e != cudaSuccess) return Q2_ERR_CUDA;
        UmFuse fz{};
        if (fused) {
            fz.tstats = tstats;
            fz.temps = temperatures;
            fz.beta = temperatures ? 0.0f : (float)(1.4426950408889634 / (double)temperature);
            fz.k1 = k + 1;
        }
        e = probed(kProbeGemm, s, [&] {
            return launch_gemm_umma(W, V, K, (int)M, img, target_logits, V, status, sms, s, fz);
        });
    } else {
        const PrepLayout L(K);
        const PrepPtrs P = PrepPtrs::carve(c.take(L.bytes((int)M)), L, (int)M);
        e = launch_prep_bf16(A, lda, nullptr, (int)M, K, P, L, s);
        if (e != cudaSuccess) return Q2_ERR_CUDA;
        e = probed(kProbeGemm, s, [&] {
            return streamed ? launch_gemm_stream(W, V, K, P, L, (int)M, target_logits, V, status, sms, s)
                          : launch_gemm_small(W, V, K, P, L, (int)M, target_logits, V, status, s);
        });
    }
    if (e != cudaSuccess) return Q2_ERR_CUDA;
    // 2. the verify over those logits
    PqArgs a;
    PqSplit sp;
    pq_setup(a, sp, c, target_logits, draft_logits, draft_tokens, u_acc, u_fin, S, k, V,
             temperatures ? 1.0f : temperature, temperatures, n_accepted, out_tokens, probs_out, status, sms);
    if (fused) {
        sp.tstats = tstats;
        sp.Ct = Ct;
    }
    return cuda_status(launch_pq_verify(a, sp, V <= kWarpTierMaxV, sms, s));
}

}  // extern "C"

// The host-side checks pq_verify makes before it enqueues anything (temperature, pointers,
// sizes, alignment), for callers that must reject bad arguments before touching the stream.
q2_status q2v::pq_verify_precheck(const float *target_logits, const float *draft_logits,
                                  const int32_t *draft_tokens, const float *u_acc, const float *u_fin, int S,
                                  int k, int V, float temperature, int32_t *n_accepted, int32_t *out_tokens,
                                  float *probs_out) {
    if (!(temperature > 0.0f) || !isfinite(temperature)) return Q2_ERR_INVALID_ARG;
    return pq_check_args(target_logits, draft_logits, draft_tokens, u_acc, u_fin, S, k, V, n_accepted,
                         out_tokens, probs_out);
}

extern "C" {

q2_status pq_verify_ex(const float *target_logits, const float *draft_logits, const int32_t *draft_tokens,
                       const float *u_acc, const float *u_fin, int S, int k, int V, const float *temperatures,
                       int32_t *n_accepted, int32_t *out_tokens, float *probs_out, void *ws, size_t ws_bytes,
                       q2_stream_t stream) {
    if (!temperatures) return Q2_ERR_INVALID_ARG;
    if (!aligned(temperatures, 4)) return Q2_ERR_ALIGNMENT;
    return pq_verify_impl(target_logits, draft_logits, draft_tokens, u_acc, u_fin, S, k, V, 1.0f, temperatures,
                          n_accepted, out_tokens, probs_out, ws, ws_bytes, stream);
}

}  // extern "C"

namespace {
// Checks of the verify's own arguments (shared by pq_verify, pq_verify_ex and the fused
// vocabulary-head verify).
q2_status pq_check_args(const float *target_logits, const float *draft_logits, const int32_t *draft_tokens,
                        const float *u_acc, const float *u_fin, int S, int k, int V, int32_t *n_accepted,
                        int32_t *out_tokens, float *probs_out) {
    if (S < 1 || k < 0 || V < 1 || !target_logits || !u_fin || !n_accepted || !out_tokens)
        return Q2_ERR_INVALID_ARG;
    if (k > 0 && (!draft_logits || !draft_tokens || !u_acc)) return Q2_ERR_INVALID_ARG;
    if (k > kMaxDrafts || V > (1 << 28)) return Q2_ERR_UNSUPPORTED;
    if (!aligned(target_logits, 16) || (k > 0 && !aligned(draft_logits, 16)) || !aligned(draft_tokens, 4) ||
        !aligned(u_acc, 4) || !aligned(u_fin, 4) || !aligned(n_accepted, 4) || !aligned(out_tokens, 4) ||
        !aligned(probs_out, 4))
        return Q2_ERR_ALIGNMENT;
    if (V > kWarpTierMaxV && S > 65535) return Q2_ERR_UNSUPPORTED;  // sessions map to grid.y
    return Q2_OK;
}

// Fill the verify's launch arguments; the split tier's scratch continues the carve c.
void pq_setup(PqArgs &a, PqSplit &sp, Carver &c, const float *target_logits, const float *draft_logits,
              const int32_t *draft_tokens, const float *u_acc, const float *u_fin, int S, int k, int V,
              float temperature, const float *temps, int32_t *n_accepted, int32_t *out_tokens, float *probs_out,
              unsigned int *status, int sms) {
    a.target = target_logits;
    a.draft = draft_logits;
    a.drafts = draft_tokens;
    a.u_acc = u_acc;
    a.u_fin = u_fin;
    a.S = S; a.k = k; a.V = V;
    a.beta = (float)(1.4426950408889634 / (double)temperature);
    a.temps = temps;
    a.n_acc = n_accepted;
    a.tokens = out_tokens;
    a.probs = probs_out;
    a.status = status;
    sp = PqSplit{};
    if (V > kWarpTierMaxV) {
        const PqCarve pc = pq_carve_from(c, S, k, V);
        int C = std::max(1, std::min(cdiv(2 * sms, S), pq_cmax(V)));
        const int L = (int)align_up((size_t)cdiv(V, C), kChunkAlign);
        C = cdiv(V, L);
        sp.C = C;
        sp.L = L;
        sp.xin = pc.xin;
        sp.stats = pc.stats;
        sp.mass = pc.mass;
        sp.pmass = pc.pmass;
        sp.tickets = pc.tickets;
    }
}

q2_status pq_verify_impl(const float *target_logits, const float *draft_logits, const int32_t *draft_tokens,
                         const float *u_acc, const float *u_fin, int S, int k, int V, float temperature,
                         const float *temps, int32_t *n_accepted, int32_t *out_tokens, float *probs_out, void *ws,
                         size_t ws_bytes, q2_stream_t stream) {
    const q2_status ast = pq_check_args(target_logits, draft_logits, draft_tokens, u_acc, u_fin, S, k, V,
                                        n_accepted, out_tokens, probs_out);
    if (ast != Q2_OK) return ast;
    const bool warp_tier = V <= kWarpTierMaxV;
    const size_t need = warp_tier ? (size_t)Q2_WORKSPACE_HEADER_BYTES : pq_carve(nullptr, S, k, V).bytes;
    const q2_status wst = check_ws(ws, ws_bytes, need);
    if (wst != Q2_OK) return wst;
    PqArgs a;
    PqSplit sp;
    const int sms = device_sms();
    Carver c(ws);
    pq_setup(a, sp, c, target_logits, draft_logits, draft_tokens, u_acc, u_fin, S, k, V, temperature, temps,
             n_accepted, out_tokens, probs_out, status_word(ws), sms);
    return cuda_status(launch_pq_verify(a, sp, warp_tier, sms, reinterpret_cast<cudaStream_t>(stream)));
}
}  // namespace
