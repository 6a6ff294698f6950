// q2v_gemm.cu -- activation prep and the small-M Q2B32 dequant GEMM (Y = A W^T).
//
// The projection matmuls and the vocabulary head of the K+1-row verify ("Optimizing
// DeepSeek-V4-Flash on a single NVIDIA GB10/GX10 with DSpark speculative decoding",
// page 2, verifier-bottleneck reply) at the tiny-batch shapes of the opening post
// (about 5 target rows per verify).  The pages' own kernels were tiny-batch HMMA
// matmuls for GB10; this is a new design for sm_103a (see q2v_mma_core.cuh).
#include "q2v_kernels.cuh"
#include "q2v_mma_core.cuh"

namespace q2v {

// One CTA per activation row (prep_row_bf16, q2v_mma_core.cuh).
__global__ void __launch_bounds__(256) prep_bf16_kernel(const uint16_t *__restrict__ src, int ld,
                                                        const int *__restrict__ rows, int R, int K,
                                                        PrepPtrs P, PrepLayout L) {
    __shared__ float scratch[32];
    pdl_wait();
    pdl_trigger();
    prep_row_bf16(src, ld, rows ? rows[blockIdx.x] : (int)blockIdx.x, (int)blockIdx.x, P, L, scratch);
}

cudaError_t launch_prep_bf16(const uint16_t *src, int ld, const int *rows, int R, int K, const PrepPtrs &P,
                             const PrepLayout &L, cudaStream_t s) {
    return launch_pdl(prep_bf16_kernel, dim3(R), dim3(256), s, src, ld, rows, R, K, P, L);
}

// Dense small-M GEMM: CTA = 16 weight rows and ceil(tiles/2) warps (<= 16); warp w owns K
// tiles w and w + nwarps, both requested before the programmatic wait (they do not depend
// on the prep kernel), so the weight stream overlaps the prep and the launch.  The prepared
// activation rows are then staged in shared memory, 8 at a time, with the weight tiles
// kept in registers across slices.  Partial sums of the K split are reduced across warps
// in warp order.
constexpr int kGemmWarps = 16;
constexpr int kMaxTilesPerWarp = kMaxTileWarps / kGemmWarps;

template <bool ALIGN8>
__global__ void __launch_bounds__(kGemmWarps * 32) q2_gemm_mma_kernel(const uint8_t *__restrict__ W, int N, int K,
                                                                         PrepPtrs P, PrepLayout L, int M, int ncols,
                                                                         float *__restrict__ Y, int ldy,
                                                                         unsigned int *status) {
    extern __shared__ __align__(16) uint32_t sm_act[];
    __shared__ float red[kGemmWarps * kRowsPerCta * 8];
    __shared__ int s_rows[8];
    const int n0 = blockIdx.x * kRowsPerCta;
    const int rows_valid = min(kRowsPerCta, N - n0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const size_t row_bytes = (size_t)L.nb * kBlockBytes;
    static_assert(kMaxTilesPerWarp == 2, "two weight tiles per warp");
    TileRegs wr0, wr1;
    load_tile<ALIGN8>(wr0, W + (size_t)n0 * row_bytes, row_bytes, rows_valid, L.nb, warp, lane);
    if (warp + nwarps < L.ntk)
        load_tile<ALIGN8>(wr1, W + (size_t)n0 * row_bytes, row_bytes, rows_valid, L.nb, warp + nwarps, lane);
    pdl_wait();
    pdl_trigger();
    const SmemAct SA(L, ncols);
    uint32_t scale_max = 0u;  // running max of |d|, |m| (f16x2)
    for (int m0 = 0; m0 < M; m0 += 8) {
        const int mc = min(8, M - m0);
        if (threadIdx.x < 8) s_rows[threadIdx.x] = m0 + threadIdx.x;
        __syncthreads();
        stage_act(sm_act, SA, P, L, s_rows, mc);
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        // one tile at a time (not unrolled), so the two tiles' register lifetimes stay apart
#pragma unroll 1
        for (int i = 0; i < kMaxTilesPerWarp; ++i) {
            const int tile = warp + i * nwarps;
            if (tile < L.ntk) {
                TileRegs cur;
#pragma unroll
                for (int q = 0; q < 12; ++q)
                    (&cur.w[0][0][0])[q] = i ? (&wr1.w[0][0][0])[q] : (&wr0.w[0][0][0])[q];
                compute_tile_smem(cur, sm_act, SA, mc, tile, lane, acc, scale_max);
            }
        }
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
    if (scale_mag_out_of_range(scale_max)) set_status(status, Q2_ERR_RANGE);
}

// Dense small-M GEMM with the activation prep fused in, for M <= 8 (one MMA column slice).
// CTA = 16 weight rows and ceil(tiles/2) warps; warp w owns K tiles w and w + nwarps, whose
// weights it requests before the programmatic wait.  After the wait each warp reads only its
// own slice of A (the 16 Q2B32 blocks of its two tiles, for every activation row) straight from
// global memory and writes it, prepared, into a private staged operand in shared memory: a
// per-(row, warp) power-of-two exponent (from the row's largest magnitude in the slice), the
// permuted f16x2 pair slots pre-scaled by 4^-(code position), and the hi + lo block sums.  No
// prep kernel, no CTA-wide staging: the only dependent round trip after the wait is the warp's
// own activation load.  The warps' partial sums are reduced in warp order, each scaled by its
// own exponent.
template <bool ALIGN8>
__global__ void __launch_bounds__(kGemmWarps * 32) q2_gemm_fused_kernel(const uint8_t *__restrict__ W, int N, int K,
                                                                           const uint16_t *__restrict__ A, int lda,
                                                                           int M, float *__restrict__ Y, int ldy,
                                                                           unsigned int *status) {
    extern __shared__ __align__(16) uint32_t sm_act[];
    __shared__ float red[kGemmWarps * kRowsPerCta * 8];
    __shared__ int s_exp[kGemmWarps][8];
    const PrepLayout L(K);
    const int n0 = blockIdx.x * kRowsPerCta;
    const int rows_valid = min(kRowsPerCta, N - n0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const size_t row_bytes = (size_t)L.nb * kBlockBytes;
    static_assert(kMaxTilesPerWarp == 2, "two weight tiles per warp");
    TileRegs wr0, wr1;
    load_tile<ALIGN8>(wr0, W + (size_t)n0 * row_bytes, row_bytes, rows_valid, L.nb, warp, lane);
    if (warp + nwarps < L.ntk)
        load_tile<ALIGN8>(wr1, W + (size_t)n0 * row_bytes, row_bytes, rows_valid, L.nb, warp + nwarps, lane);
    pdl_wait();
    pdl_trigger();
    // this warp's staged operand: 16 local blocks (local tile i = global tile warp + i * nwarps)
    const PrepLayout LW(2 * kTileBlocks * kBlockK);
    const SmemAct SA(LW, M);
    uint32_t *wsm = sm_act + (size_t)warp * SA.words();
    // lanes 16h .. 16h+15 of round q prepare the 16 local blocks of activation row 2q + h; every
    // round's loads go out before any is used
    constexpr int kRounds = kFusedMaxM / 2;
    uint4 raw[kRounds][4];
#pragma unroll
    for (int q = 0; q < kRounds; ++q) {
        const int row = 2 * q + (lane >> 4), lb = lane & 15;
        const int gb = (warp + (lb >> 3) * nwarps) * kTileBlocks + (lb & 7);
        const bool valid = row < M && gb < L.nb;
        const uint4 *p = reinterpret_cast<const uint4 *>(A + (size_t)(valid ? row : 0) * lda +
                                                         (size_t)(valid ? gb : 0) * kBlockK);
#pragma unroll
        for (int j = 0; j < 4; ++j) raw[q][j] = valid ? __ldg(p + j) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < kRounds; ++q) {
        if (2 * q >= M) break;
        const int row = 2 * q + (lane >> 4), lb = lane & 15;
        const uint32_t w[16] = {raw[q][0].x, raw[q][0].y, raw[q][0].z, raw[q][0].w, raw[q][1].x, raw[q][1].y,
                                raw[q][1].z, raw[q][1].w, raw[q][2].x, raw[q][2].y, raw[q][2].z, raw[q][2].w,
                                raw[q][3].x, raw[q][3].y, raw[q][3].z, raw[q][3].w};
        float mx = bf16x2_maxabs(w);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const int e = act_exponent(mx);
        if (row < M) {
            prep_store_block_smem(w, e, wsm, SA, row, lb);
            if (lb == 0) s_exp[warp][row] = e;
        }
    }
    __syncwarp();
    uint32_t scale_max = 0u;  // running max of |d|, |m| (f16x2)
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    compute_tile_smem(wr0, wsm, SA, M, 0, lane, acc, scale_max);
    if (warp + nwarps < L.ntk) compute_tile_smem(wr1, wsm, SA, M, 1, lane, acc, scale_max);
    store_fragments(red + warp * kRowsPerCta * 8, acc, lane);
    __syncthreads();
    for (int j = threadIdx.x; j < kRowsPerCta * M; j += blockDim.x) {
        const int r = j % kRowsPerCta, m = j / kRowsPerCta;
        float s = 0.0f;
        for (int w = 0; w < nwarps; ++w) {
            const int e = s_exp[w][m];
            const float x = red[w * kRowsPerCta * 8 + r * 8 + m];
            // x * 2^e: one exact multiply when 2^e is a normal fp32 number
            s += (e >= -126 && e <= 127) ? x * exp2i(e) : ldexpf(x, e);
        }
        if (r < rows_valid) Y[(size_t)m * ldy + n0 + r] = s;
    }
    if (scale_mag_out_of_range(scale_max)) set_status(status, Q2_ERR_RANGE);
}

namespace {
size_t g_gemm_smem[kCacheDevices][2];  // dynamic shared memory each variant was configured for, per device
size_t g_fused_smem[kCacheDevices][2];

template <bool A8>
cudaError_t launch_fused_variant(const uint8_t *w, int N, int K, const uint16_t *A, int lda, int M, float *Y,
                                 int ldy, unsigned int *status, cudaStream_t s) {
    auto kern = q2_gemm_fused_kernel<A8>;
    const PrepLayout L(K);
    const int nwarps = cdiv(L.ntk, kMaxTilesPerWarp);
    const size_t smem = (size_t)nwarps * SmemAct(PrepLayout(2 * kTileBlocks * kBlockK), M).bytes();
    const int dv = cache_device();
    if (dv < 0 || g_fused_smem[dv][A8] < smem) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dv >= 0) g_fused_smem[dv][A8] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cdiv(N, kRowsPerCta));
    cfg.blockDim = dim3(32 * nwarps);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, w, N, K, A, lda, M, Y, ldy, status);
}

template <bool A8>
cudaError_t launch_gemm_variant(const uint8_t *w, int N, int K, const PrepPtrs &P, const PrepLayout &L, int M,
                                float *Y, int ldy, unsigned int *status, cudaStream_t s) {
    auto kern = q2_gemm_mma_kernel<A8>;
    const int ncols = min(8, M);
    const size_t smem = SmemAct(L, ncols).bytes();
    const int dv = cache_device();
    if (dv < 0 || g_gemm_smem[dv][A8] < smem) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dv >= 0) g_gemm_smem[dv][A8] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cdiv(N, kRowsPerCta));
    cfg.blockDim = dim3(32 * cdiv(L.ntk, kMaxTilesPerWarp));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, w, N, K, P, L, M, ncols, Y, ldy, status);
}
}  // namespace

cudaError_t launch_gemm_fused(const void *W, int N, int K, const uint16_t *A, int lda, int M, float *Y, int ldy,
                              unsigned int *status, cudaStream_t s) {
    const uint8_t *w = static_cast<const uint8_t *>(W);
    if ((PrepLayout(K).nb % 2) == 0) return launch_fused_variant<true>(w, N, K, A, lda, M, Y, ldy, status, s);
    return launch_fused_variant<false>(w, N, K, A, lda, M, Y, ldy, status, s);
}

cudaError_t launch_gemm_small(const void *W, int N, int K, const PrepPtrs &P, const PrepLayout &L, int M,
                              float *Y, int ldy, unsigned int *status, cudaStream_t s) {
    const uint8_t *w = static_cast<const uint8_t *>(W);
    if ((L.nb % 2) == 0) return launch_gemm_variant<true>(w, N, K, P, L, M, Y, ldy, status, s);
    return launch_gemm_variant<false>(w, N, K, P, L, M, Y, ldy, status, s);
}

}  // namespace q2v
