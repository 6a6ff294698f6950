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
// process exits.  In host code `g_pq_scratch` only names the symbol: its device address on
// the current device is obtained with cudaGetSymbolAddress, and that address is what the
// kernels receive.
constexpr size_t kNoAllocScratchBytes = (size_t)2 << 20;  // 2 MiB
static __device__ __align__(256) unsigned char g_pq_scratch[kNoAllocScratchBytes];

}  // namespace

extern "C" q2_status pq_verify_noalloc(const float *target_logits, const float *draft_logits,
                                       const int32_t *draft_tokens, const float *u_acc, const float *u_fin,
                                       int S, int k, int V, float temperature, int32_t *n_accepted,
                                       int32_t *out_tokens, float *probs_out, q2_stream_t stream) {
    // everything the host can reject is rejected before any work is enqueued: the arguments
    // as pq_verify checks them, then sizes whose scratch (the layout pq_verify uses) would not
    // fit the fixed array
    const q2_status ast = q2v::pq_verify_precheck(target_logits, draft_logits, draft_tokens, u_acc, u_fin, S, k,
                                                  V, temperature, n_accepted, out_tokens, probs_out);
    if (ast != Q2_OK) return ast;
    if (pq_verify_workspace(S, k, V) > kNoAllocScratchBytes) return Q2_ERR_UNSUPPORTED;
    // the array's address on the current device, looked up on every call (a host-side query),
    // so no cached address is shared between host threads or outlives a device reset
    void *ws = nullptr;
    if (cudaGetSymbolAddress(&ws, g_pq_scratch) != cudaSuccess || ws == nullptr) return Q2_ERR_CUDA;
    // the array keeps the previous call's contents: the status word must start at zero (the
    // kernels reset their own counters and overwrite every partial they read)
    if (cudaMemsetAsync(ws, 0, Q2_WORKSPACE_HEADER_BYTES, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return Q2_ERR_CUDA;
    return pq_verify(target_logits, draft_logits, draft_tokens, u_acc, u_fin, S, k, V, temperature, n_accepted,
                     out_tokens, probs_out, ws, kNoAllocScratchBytes, stream);
}
