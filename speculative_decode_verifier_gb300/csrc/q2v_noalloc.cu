// q2v_noalloc.cu -- pq_verify for callers that cannot allocate device memory.
//
// Some callers of the verifier cannot hand the library a workspace: for instance a decode
// loop embedded in a host framework whose own pool already owns the device's memory, so it
// has no spare buffer to lend and must not call cudaMalloc (which can stall the whole device
// and, under a reserved pool, simply fail).  For them pq_verify_noalloc runs the ordinary
// pq_verify with its scratch in a fixed array that the library itself places in device
// memory when it is loaded.  It allocates nothing, at set-up or per call.
#include "q2v_kernels.cuh"

namespace {

// The fixed scratch.  Every device that loads the library holds these bytes until the
// process exits.  In host code `g_pq_scratch` only names the symbol: its device address is
// obtained with cudaGetSymbolAddress (once per device) and that address is what the kernels
// receive.
constexpr size_t kNoAllocScratchBytes = (size_t)2 << 20;  // 2 MiB
static __device__ __align__(256) unsigned char g_pq_scratch[kNoAllocScratchBytes];

constexpr int kMaxNoAllocDevices = 64;
void *g_scratch_addr[kMaxNoAllocDevices];  // device address of g_pq_scratch, per device

}  // namespace

extern "C" q2_status pq_verify_noalloc(const float *target_logits, const float *draft_logits,
                                       const int32_t *draft_tokens, const float *u_acc, const float *u_fin,
                                       int S, int k, int V, float temperature, int32_t *n_accepted,
                                       int32_t *out_tokens, float *probs_out, q2_stream_t stream) {
    // the same scratch layout pq_verify uses; sizes it cannot hold are refused up front
    const size_t need = pq_verify_workspace(S, k, V);
    if (need > kNoAllocScratchBytes) return Q2_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxNoAllocDevices) return Q2_ERR_CUDA;
    if (g_scratch_addr[dev] == nullptr) {
        // one-time set-up on this device (with this device current)
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pq_scratch) != cudaSuccess || p == nullptr) return Q2_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    void *ws = g_scratch_addr[dev];
    // the array keeps the previous call's contents: the status word must start at zero (the
    // kernels reset their own counters and overwrite every partial they read)
    if (cudaMemsetAsync(ws, 0, Q2_WORKSPACE_HEADER_BYTES, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return Q2_ERR_CUDA;
    return pq_verify(target_logits, draft_logits, draft_tokens, u_acc, u_fin, S, k, V, temperature, n_accepted,
                     out_tokens, probs_out, ws, kNoAllocScratchBytes, stream);
}
