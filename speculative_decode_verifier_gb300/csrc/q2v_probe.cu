// q2v_probe.cu -- read-only HBM bandwidth probe (a measurement hook, not part of the verify).
//
// Every kernel of the verifier step is a read stream (weights, logits) with almost no writes,
// so its roofline is the read bandwidth of HBM rather than the copy bandwidth (read + write).
// This kernel streams a caller's buffer once with 16-byte loads that bypass L1 and are marked
// evict-first in L2, every thread keeping 8 loads in flight, over a grid of 4 CTAs of 512
// threads per SM; the loaded words are folded into one value that is stored only if it equals
// an arbitrary constant, so the loads cannot be dropped and nothing else is written.  The
// "ds4-on-spark" README, section "Roofline", measures the same pair (copy and read-only) on
// GB10.
#include "q2v_kernels.cuh"

namespace q2v {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeUnroll = 8;

__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint4 *__restrict__ p, size_t n16,
                                                                   unsigned int *sink) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    unsigned int acc = 0u;
    for (; i + (kProbeUnroll - 1) * stride < n16; i += kProbeUnroll * stride) {
        uint4 v[kProbeUnroll];
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u) v[u] = __ldcs(p + i + u * stride);
#pragma unroll
        for (int u = 0; u < kProbeUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = __ldcs(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (acc == 0x2545F491u) *sink = acc;
}

}  // namespace
}  // namespace q2v

extern "C" q2_status q2_hbm_read_probe(const void *buf, size_t bytes, unsigned int *sink, q2_stream_t stream) {
    if (!buf || !sink || bytes == 0 || bytes % 16 != 0) return Q2_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(buf) % 16 != 0 || reinterpret_cast<uintptr_t>(sink) % 4 != 0)
        return Q2_ERR_ALIGNMENT;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return Q2_ERR_CUDA;
    q2v::read_probe_kernel<<<4 * sms, q2v::kProbeThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(buf), bytes / 16, sink);
    return cudaGetLastError() == cudaSuccess ? Q2_OK : Q2_ERR_CUDA;
}
