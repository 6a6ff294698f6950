// q2v_gemm.cu -- activation prep and the small-M Q2B32 dequant GEMM (Y = A W^T).
//
// The "projections and the vocabulary head" of the K+1-row verify ("Optimizing
// DeepSeek-V4-Flash on a single NVIDIA GB10/GX10 with DSpark speculative decoding",
// page 2, verifier-bottleneck reply) at the tiny-batch shapes of the opening post
// (about 5 target rows per verify).  The pages' own kernels were tiny-batch HMMA
// matmuls for GB10; this is a new design for sm_103a (see q2v_mma_core.cuh).
#include "q2v_kernels.cuh"
#include "q2v_mma_core.cuh"

namespace q2v {

// One CTA per activation row: per-row exponent, permuted f16x2 pair slots, hi/lo block
// sums.  src rows: bf16 bits or fp32, row r of the prep is source row rows[r] (or r).
template <bool F32>
__global__ void __launch_bounds__(256) prep_act_kernel(const void *__restrict__ src, int ld,
                                                       const int *__restrict__ rows, int R, int K,
                                                       PrepPtrs P, PrepLayout L) {
    const int r = blockIdx.x;
    if (r >= R) return;
    const int srow = rows ? rows[r] : r;
    const int tid = threadIdx.x;
    __shared__ float red[8];
    __shared__ int sexp;
    auto at = [&](int k) -> float {
        if (F32) return reinterpret_cast<const float *>(src)[(size_t)srow * ld + k];
        const uint16_t b = reinterpret_cast<const uint16_t *>(src)[(size_t)srow * ld + k];
        return __uint_as_float((uint32_t)b << 16);
    };
    float mx = 0.0f;
    if (srow >= 0)
        for (int k = tid; k < K; k += blockDim.x) mx = fmaxf(mx, fabsf(at(k)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    if (tid == 0) {
        float m = 0.0f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
        sexp = act_exponent(m);
        P.exps[r] = sexp;
    }
    __syncthreads();
    const int e = sexp;
    uint32_t *act = P.act + (size_t)r * L.act_words_per_row();
    for (int j = tid; j < L.nbp * 16; j += blockDim.x) {
        const int b = j >> 4, p = j & 15;
        uint32_t v = 0;
        if (srow >= 0 && b < L.nb) {
            const int k0 = b * kBlockK + 16 * (p >> 3) + (p & 7);
            v = pack_half2(__float2half_rn(ldexpf(at(k0), -e)), __float2half_rn(ldexpf(at(k0 + 8), -e)));
        }
        act[j] = v;
    }
    __half *sh = reinterpret_cast<__half *>(P.shi + (size_t)r * L.sum_words_per_row());
    __half *sl = reinterpret_cast<__half *>(P.slo + (size_t)r * L.sum_words_per_row());
    for (int b = tid; b < L.nbp; b += blockDim.x) {
        float s = 0.0f;
        if (srow >= 0 && b < L.nb)
            for (int kk = 0; kk < kBlockK; ++kk)
                s += __half2float(__float2half_rn(ldexpf(at(b * kBlockK + kk), -e)));
        const __half hi = __float2half_rn(s);
        sh[b] = hi;
        sl[b] = __float2half_rn(s - __half2float(hi));
    }
}

void launch_prep(const void *src, bool src_f32, int ld, const int *rows, int R, int K, const PrepPtrs &P,
                 const PrepLayout &L, cudaStream_t s) {
    if (R <= 0) return;
    if (src_f32)
        prep_act_kernel<true><<<R, 256, 0, s>>>(src, ld, rows, R, K, P, L);
    else
        prep_act_kernel<false><<<R, 256, 0, s>>>(src, ld, rows, R, K, P, L);
}

// Dense small-M GEMM: CTA = 16 weight rows, one warp per K tile; the activation rows are
// processed in slices of 8 with the weight tile kept in registers across slices.
template <bool ALIGN8>
__global__ void __launch_bounds__(1024) q2_gemm_mma_kernel(const uint8_t *__restrict__ W, int N, int K,
                                                           PrepPtrs P, PrepLayout L, int M,
                                                           float *__restrict__ Y, int ldy,
                                                           unsigned int *status) {
    __shared__ float red[kMaxTileWarps * kRowsPerCta * 8];
    const int n0 = blockIdx.x * kRowsPerCta;
    const int rows_valid = min(kRowsPerCta, N - n0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const size_t row_bytes = (size_t)L.nb * kBlockBytes;
    TileRegs wr;
    load_tile<ALIGN8>(wr, W + (size_t)n0 * row_bytes, row_bytes, rows_valid, L.nb, warp, lane);
    bool range_bad = false;
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mc = min(8, M - m0);
        ActRegs ar;
        const int col = lane >> 2;
        load_act(ar, P, L, col < mc ? m0 + col : -1, warp, lane);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        compute_tile(wr, ar, acc, range_bad);
        store_fragments(red + warp * kRowsPerCta * 8, acc, lane);
        __syncthreads();
        for (int j = threadIdx.x; j < kRowsPerCta * mc; j += blockDim.x) {
            const int r = j % kRowsPerCta, m = j / kRowsPerCta;
            float s = 0.0f;
            for (int w = 0; w < nwarps; ++w) s += red[w * kRowsPerCta * 8 + r * 8 + m];
            if (r < rows_valid) Y[(size_t)(m0 + m) * ldy + n0 + r] = ldexpf(s, P.exps[m0 + m]);
        }
        __syncthreads();
    }
    if (range_bad) set_status(status, Q2_ERR_RANGE);
}

cudaError_t launch_gemm_small(const void *W, int N, int K, const PrepPtrs &P, const PrepLayout &L, int M,
                              float *Y, int ldy, unsigned int *status, cudaStream_t s) {
    const int grid = cdiv(N, kRowsPerCta);
    const int block = 32 * L.ntk;
    if ((L.nb % 2) == 0)
        q2_gemm_mma_kernel<true><<<grid, block, 0, s>>>(static_cast<const uint8_t *>(W), N, K, P, L, M, Y, ldy,
                                                        status);
    else
        q2_gemm_mma_kernel<false><<<grid, block, 0, s>>>(static_cast<const uint8_t *>(W), N, K, P, L, M, Y, ldy,
                                                         status);
    return cudaGetLastError();
}

}  // namespace q2v
