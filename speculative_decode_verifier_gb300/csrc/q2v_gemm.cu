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

// Small M (<= 8) against many weight rows: a persistent grid (one CTA of 24 warps per SM), the
// prepared activation rows staged in shared memory once per CTA, and the CTA's contiguous range
// of 16-row units (all of K) split evenly over its warps by tiles, each warp streaming its
// 16 x 256 weight tiles through its own 3-deep cp.async ring and decoding them with the same
// exact mma.sync tile decode (the MoE stream kernels' arrangement, for one matrix).  Measured on
// the M=5 x 129,280 x 4,096 head (head GEMM + verify, us): even split 77.0, strided units 80.2;
// with strided units, 16 warps and 4-tile rings or two CTAs of 8 warps were slower still.  The
// first ring tiles are requested before the programmatic wait (the weights do not depend on the
// previous kernel); the staged activations after it.  Requires K % 256 == 0 and N % 16 == 0.
constexpr int kStreamRing = 3;
constexpr int kStreamWarps = 24;
constexpr bool kStreamEven = true;

__global__ void __launch_bounds__(kStreamWarps * 32, 1)
    q2_gemm_stream_kernel(const uint8_t *__restrict__ W, int N, int K, PrepPtrs P, PrepLayout L, int M,
                          float *__restrict__ Y, int ldy, unsigned int *status) {
    extern __shared__ __align__(16) uint32_t sm_dyn[];
    __shared__ int s_rows[8], s_exps[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const SmemAct SA(L, M);
    uint32_t *sm_act = sm_dyn;
    uint32_t *ring = sm_dyn + SA.words() + (size_t)warp * kStreamRing * kTileWords;
    const size_t row_bytes = (size_t)L.nb * kBlockBytes;
    const int units = N / kRowsPerCta;
    const int q = cdiv(units, gridDim.x);
    const int u0 = blockIdx.x * q, u1 = min(units, u0 + q);
    auto unit_w = [&](int u) { return W + (size_t)u * kRowsPerCta * row_bytes; };
    TileCursor<kStreamEven, decltype(unit_w)> pc;
    pc.begin(u0, u1, L.ntk, kStreamWarps, warp, unit_w);
#pragma unroll
    for (int sidx = 0; sidx < kStreamRing - 1; ++sidx)
        pc.produce(ring + sidx * kTileWords, row_bytes, L.ntk, kStreamWarps, lane, unit_w);
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x < 8) {
        s_rows[threadIdx.x] = threadIdx.x < M ? (int)threadIdx.x : 0;
        s_exps[threadIdx.x] = threadIdx.x < M ? P.exps[threadIdx.x] : 0;
    }
    __syncthreads();
    stage_act_issue(sm_act, SA, P, L, s_rows, M);  // the newest group: wait for every group
    cp_async_wait<0>();
    __syncthreads();
    uint32_t scale_max = 0u;  // running max of |d|, |m| (f16x2)
    auto cols = [&](int) { return make_int2(M, 0); };
    // rows g, g+8 of the unit, activation rows 2t, 2t+1
    auto store = [&](int u, int2, const float *v) {
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            const int m = 2 * t + (qq & 1), n = u * kRowsPerCta + g + 8 * (qq >> 1);
            if (m < M) Y[(size_t)m * ldy + n] = ldexpf(v[qq], s_exps[m]);
        }
    };
    float *part = reinterpret_cast<float *>(sm_dyn + SA.words() + (size_t)kStreamWarps * kStreamRing * kTileWords);
    stream_warp_tiles<kStreamRing, kStreamEven>(pc, ring, sm_act, SA, part, u0, u1, L.ntk, row_bytes, kStreamWarps, warp, lane,
                                   unit_w, cols, store, scale_max);
    if (scale_mag_out_of_range(scale_max)) set_status(status, Q2_ERR_RANGE);
}

size_t stream_smem_bytes(int M, int K) {
    return SmemAct(PrepLayout(K), M).bytes() + (size_t)kStreamWarps * (kStreamRing * kTileWords + 128) * 4;
}

bool stream_gemm_usable(int M, int N, int K) {
    return M >= 1 && M <= 8 && K % (kTileBlocks * kBlockK) == 0 && N % kRowsPerCta == 0 &&
           stream_smem_bytes(M, K) <= (size_t)220 * 1024;
}

// The streaming kernel pays off once the persistent grid has about 16 rows for each of 16
// warps per SM (N >= 16 x 16 x SMs: 38,912 rows on 152 SMs); at fewer rows the per-CTA kernel or
// the tcgen05 kernel is used.
bool stream_gemm_preferred(int M, int N, int K, int sms) {
    return stream_gemm_usable(M, N, K) && (long long)N >= (long long)kRowsPerCta * 16 * sms;
}

namespace {
size_t g_stream_smem_cfg[kCacheDevices];
}  // namespace

cudaError_t launch_gemm_stream(const void *W, int N, int K, const PrepPtrs &P, const PrepLayout &L, int M, float *Y,
                               int ldy, unsigned int *status, int num_sms, cudaStream_t s) {
    auto kern = q2_gemm_stream_kernel;
    const size_t smem = stream_smem_bytes(M, K);
    const int dv = cache_device();
    if (dv < 0 || g_stream_smem_cfg[dv] < smem) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dv >= 0) g_stream_smem_cfg[dv] = smem;
    }
    const int units = N / kRowsPerCta;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(max(1, min(units, num_sms)));
    cfg.blockDim = dim3(kStreamWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint8_t *>(W), N, K, P, L, M, Y, ldy, status);
}

namespace {
size_t g_gemm_smem[kCacheDevices][2];  // dynamic shared memory each variant was configured for, per device

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

cudaError_t launch_gemm_small(const void *W, int N, int K, const PrepPtrs &P, const PrepLayout &L, int M,
                              float *Y, int ldy, unsigned int *status, cudaStream_t s) {
    const uint8_t *w = static_cast<const uint8_t *>(W);
    if ((L.nb % 2) == 0) return launch_gemm_variant<true>(w, N, K, P, L, M, Y, ldy, status, s);
    return launch_gemm_variant<false>(w, N, K, P, L, M, Y, ldy, status, s);
}

}  // namespace q2v
