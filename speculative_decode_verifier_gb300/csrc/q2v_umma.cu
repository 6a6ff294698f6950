// q2v_umma.cu -- the Q2B32 dequant GEMM on the fifth-generation tensor cores (tcgen05), for
// the wider verify batches: more than 16 activation rows, such as 12 sessions x (k+1) = 60
// rows against the vocabulary head, and 5..16 rows against many weight rows, such as one
// session's vocabulary head (the vocabulary head is one of the matmuls of the K+1-row verify,
// "Optimizing DeepSeek-V4-Flash on a single NVIDIA GB10/GX10 with DSpark speculative
// decoding", page 2, verifier-bottleneck reply).  At 60 rows the contraction is as heavy as
// the weight stream (about 250 flop per weight byte), so both the tensor cores and HBM have to
// run flat out, overlapped.
//
// One persistent CTA per SM walks 128-row weight tiles.  Per tile, the K dimension goes by
// in stages of 4 Q2B32 blocks (128 k):
//   * TMA warp: one 2-D tensor copy per stage brings the tile's raw Q2B32 bytes
//     (128 rows x 48 B) into a deep shared-memory ring (the weights do not depend on the
//     previous kernel, so this warp starts before the programmatic wait);
//   * B warp: brings each prepared activation stage (the B operand, laid out by
//     prep_umma_kernel) into a shared-memory ring with 16-byte cp.async copies (small and
//     L2-resident, so they stay off the TMA engine that streams the weights);
//   * 8 dequant warps, in two groups that take the stages in turn: each thread decodes one
//     weight row of the stage with the exact lop3 + f16x2 fma decode and writes it straight
//     from registers into tensor memory (tcgen05.st) as the MMA's A operand; the blocks'
//     offsets m go to a small shared-memory tile;
//   * MMA thread: per stage 8 tcgen05.mma (M=128, N=NPAD, K=16) with A read from TMEM plus
//     one with A = the m tile against the activation block sums, into a TMEM accumulator;
//     two tiles share each activation stage, and accumulators are double-buffered;
//   * 4 epilogue warps: tcgen05.ld the finished accumulators, undo the per-row activation
//     exponent and store Y.
// Keeping A in TMEM leaves only the 2 KB activation operand to be read from shared memory
// per MMA.  Every wait is bounded: on a time-out the CTA records Q2_ERR_TIMEOUT, lets the
// copies and MMAs it issued land, frees its TMEM and returns.
#include <cuda.h>

#include "q2v_kernels.cuh"
#include "q2v_mma_core.cuh"

namespace q2v {

namespace {

constexpr int kUmRows = 128;                                     // weight rows per tile (UMMA M)
constexpr int kUmBlocks = 4;                                     // Q2B32 blocks per stage
constexpr int kUmKg = 18;                                        // 16-byte k-groups per B stage
constexpr int kUmDataMmas = 8;                                   // K=16 MMAs on the weights per stage
constexpr int kUmKgBytes = (kUmRows / 8) * 128;                  // one k-group of a 128-row tile
constexpr int kUmMTile = 2 * kUmKgBytes;                         // m k-group + zero k-group: 4,096 B
constexpr int kUmACols = kUmBlocks * 16;                         // TMEM columns of one A stage (64)
constexpr int kUmRawSpan = 4;                                    // stages per raw copy
constexpr int kUmStageRaw = kUmBlocks * kBlockBytes;             // 48 raw bytes of a row per stage
constexpr int kUmRawRow = kUmRawSpan * kUmStageRaw;              // 192 B of each row per raw copy
constexpr int kUmRawStage = kUmRows * kUmRawRow;                 // 24,576 B
constexpr int kUmAStages = 4;                                    // A stages in TMEM (+ m tiles)
constexpr int kUmBStages = 4;                                    // activation (B) stages
constexpr int kUmBLag = 2;                                       // B stages in flight before signalling
constexpr int kUmRawStages = 5;                                  // raw copies in flight
constexpr int kUmGroup = 2;                                      // weight tiles sharing a B stage
constexpr int kUmAccStride = 64;                                 // TMEM columns per accumulator
constexpr int kUmAccBase = kUmAStages * kUmACols;                // accumulators after the A stages
constexpr uint32_t kUmCols = 512;                                // all of TMEM: one CTA per SM
constexpr int kUmEpiWarps = 4;
constexpr int kUmTmaWarp = 4;
constexpr int kUmBWarp = 5;
constexpr int kUmMmaWarp = 6;                                    // MMA thread of the group's tile 0 (+1: tile 1)
constexpr int kUmDeqWarp0 = kUmMmaWarp + kUmGroup;
constexpr int kUmDeqGroups = 2;                                  // groups take the stages in turn
constexpr int kUmDeqWarps = 4 * kUmDeqGroups;                   // a group: one warp per TMEM lane quarter
constexpr int kUmThreads = (kUmDeqWarp0 + kUmDeqWarps) * 32;    // 512
constexpr uint64_t kUmWaitNs = 1000000000ull;                    // 1 s per wait, then give up

static_assert(kUmAccBase + 2 * kUmGroup * kUmAccStride <= (int)kUmCols, "TMEM holds 512 columns");
static_assert(kUmGroup == 2, "one MMA-issuing warp per tile of a group");
// A stages are slotted by activation stage: slot (gb % 2) * kUmGroup + t holds tile t of
// activation stage gb, and is free again once b_empty of stage gb completes (each MMA thread
// commits that barrier after its MMAs of the stage), so one commit per stage and thread
// releases both the activation stage and its A stages.
static_assert(kUmAStages == 2 * kUmGroup, "two activation stages of A stages");

__host__ __device__ constexpr int um_bstage(int npad) { return kUmKg * (npad / 8) * 128; }

struct UmShared {
    uint64_t raw_full[kUmRawStages];
    uint64_t raw_empty[kUmRawStages];
    uint64_t ab_full[kUmAStages];    // the dequant warps have written A (TMEM) and the m tile
    uint64_t b_full[kUmBStages];     // the activation stage has landed
    uint64_t b_empty[kUmBStages];    // the MMAs reading the B stage are done
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    uint32_t abort_flag;
    int exps[64];
    // fused verify statistics: per-column (activation row) beta and mode, and the epilogue
    // warps' partials of the current tile
    float col_beta[64];
    int col_mode[64];
    float2 part[kUmEpiWarps][64];
    float2 run[64];  // this CTA's running partial of each row over its tiles
};

__host__ __device__ constexpr size_t um_smem_bytes(int npad) {
    return 1024 + (size_t)kUmBStages * um_bstage(npad) + (size_t)kUmAStages * kUmMTile +
           (size_t)kUmRawStages * kUmRawStage + sizeof(UmShared);
}

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Wait for the phase of `parity` to complete.  False if another role gave up first or this
// wait ran out of time (then it records the time-out and tells the other roles to stop).
__device__ __forceinline__ bool um_wait(uint64_t *bar, uint32_t parity, volatile uint32_t *abort_flag,
                                        unsigned int *status) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > kUmWaitNs) {
            *abort_flag = 1u;
            set_status(status, Q2_ERR_TIMEOUT);
            return false;
        }
    }
}

// um_wait by every lane of a warp, with one outcome for the whole warp.
__device__ __forceinline__ bool um_wait_warp(uint64_t *bar, uint32_t parity, volatile uint32_t *abort_flag,
                                             unsigned int *status) {
    const bool ok = um_wait(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

// Bounded wait used when winding down: copies and MMAs already issued complete by
// themselves, so this only waits for them to land.
__device__ __forceinline__ void um_drain(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    while (!mbar_try(bar, parity) && global_ns() - t0 < kUmWaitNs) {
    }
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// UMMA shared-memory descriptor, canonical K-major layout without swizzle: 8-row x 16-byte
// core matrices stored as 128 contiguous bytes; `lbo` = byte distance between core
// matrices adjacent in K, `sbo` = between core matrices adjacent in M (or N).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
           (1ull << 46);  // descriptor version 1 (bits 46-48 = 0b001), base offset 0, no swizzle
}

// Instruction descriptor, kind::f16: f32 accumulator, f16 A and B, both K-major.
template <int NPAD>
__device__ __forceinline__ constexpr uint32_t umma_idesc() {
    return (1u << 4) | ((uint32_t)(NPAD >> 3) << 17) | ((uint32_t)(kUmRows >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Same, with A read from tensor memory (a_tmem = its first column, lane 0).
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// This thread's TMEM lane, 32 consecutive columns from taddr: r[i] -> column i.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ float um_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ bool um_better_arg(float m2, int i2, float m1, int i1) {
    return m2 > m1 || (m2 == m1 && i2 < i1);
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

// ---------------------------------------------------------------- activation prep

// B operand image of the activations, one contiguous stage after another.  Stage s (Q2B32
// blocks 4s..4s+3) holds 18 k-groups; k-group g, activation row m sits at byte
//   s * um_bstage(NPAD) + g * (NPAD/8) * 128 + (m / 8) * 128 + (m % 8) * 16.
// k-groups 4j..4j+3 are block 4s+j's 16 f16x2 pair slots (the order and scaling of
// prep_store_block); k-group 16 holds the blocks' activation sums, hi parts in slots 0..3
// and lo parts in slots 4..7 (they meet the blocks' m in the A operand); k-group 17 is zero.
// Rows m >= M and blocks past K hold zeros.  One CTA per row m < NPAD, one thread per block.
__global__ void __launch_bounds__(256) prep_umma_kernel(const uint16_t *__restrict__ src, int ld, int M, int nb,
                                                        int nst, int npad, uint8_t *__restrict__ img,
                                                        int *__restrict__ exps) {
    __shared__ float scratch[32];
    pdl_wait();
    pdl_trigger();
    const int m = blockIdx.x;
    const int b = threadIdx.x;
    const bool live = b < nb && m < M;
    float v[32];
    float mx = 0.0f;
    if (live) {
        const uint4 *p = reinterpret_cast<const uint4 *>(src + (size_t)m * ld + (size_t)b * kBlockK);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 q = __ldg(p + j);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[8 * j + 2 * i] = __uint_as_float(w[i] << 16);
                v[8 * j + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) mx = fmaxf(mx, fabsf(v[j]));
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.0f;
    }
    const int e = act_exponent(block_max_nonneg(mx, scratch));
    if (b == 0 && m < 64) exps[m] = m < M ? e : 0;
    if (b >= nst * kUmBlocks) return;
    // pair slots and the block sum exactly as prep_store_block forms them
    uint32_t words[16];
    __half hs[32];
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        hs[j] = __float2half_rn(ldexpf(v[j], -e - 2 * (j & 3)));
        s += __half2float(__float2half_rn(ldexpf(v[j], -e)));
    }
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        const int k0 = 16 * (p >> 3) + (p & 7);
        words[p] = pack_half2(hs[k0], hs[k0 + 8]);
    }
    const int st = b / kUmBlocks, bl = b % kUmBlocks;
    const size_t kg_bytes = (size_t)(npad / 8) * 128;
    uint8_t *base = img + (size_t)st * um_bstage(npad) + (size_t)(m >> 3) * 128 + (size_t)(m & 7) * 16;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4 *>(base + (size_t)(4 * bl + j) * kg_bytes) =
            make_uint4(words[4 * j], words[4 * j + 1], words[4 * j + 2], words[4 * j + 3]);
    const __half hi = __float2half_rn(s);
    const __half lo = __float2half_rn(s - __half2float(hi));
    __half *sums = reinterpret_cast<__half *>(base + 16 * kg_bytes);
    sums[bl] = hi;
    sums[4 + bl] = lo;
    if (bl == 0) *reinterpret_cast<uint4 *>(base + 17 * kg_bytes) = make_uint4(0u, 0u, 0u, 0u);
}

// ---------------------------------------------------------------- the GEMM

// Decode one weight row of a stage (4 Q2B32 blocks = 48 raw bytes) into 64 f16x2 words, word
// 16*b + p = pair slot p of block b (the order prep_store_block gives the activations).
__device__ __forceinline__ void um_decode_blocks(const uint32_t *raw, uint32_t *w, uint32_t &scale_max) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const uint32_t c0 = raw[3 * b], c1 = raw[3 * b + 1], dm = raw[3 * b + 2];
        scale_max = scale_mag_max(scale_max, dm);
        uint32_t d2, nd;
        scale_pair(dm, d2, nd);
        const uint32_t h0 = c0 >> 8, h1 = c1 >> 8;
        uint32_t *o = w + 16 * b;
        o[0] = dequant_pos<0>(c0, d2, nd);
        o[1] = dequant_pos<2>(c0, d2, nd);
        o[2] = dequant_pos<4>(c0, d2, nd);
        o[3] = dequant_pos<6>(c0, d2, nd);
        o[4] = dequant_pos<0>(h0, d2, nd);
        o[5] = dequant_pos<2>(h0, d2, nd);
        o[6] = dequant_pos<4>(h0, d2, nd);
        o[7] = dequant_pos<6>(h0, d2, nd);
        o[8] = dequant_pos<0>(c1, d2, nd);
        o[9] = dequant_pos<2>(c1, d2, nd);
        o[10] = dequant_pos<4>(c1, d2, nd);
        o[11] = dequant_pos<6>(c1, d2, nd);
        o[12] = dequant_pos<0>(h1, d2, nd);
        o[13] = dequant_pos<2>(h1, d2, nd);
        o[14] = dequant_pos<4>(h1, d2, nd);
        o[15] = dequant_pos<6>(h1, d2, nd);
    }
}

// A CTA's tiles are blockIdx.x, blockIdx.x + gridDim.x, ...; they are processed in groups of
// up to kUmGroup tiles that share each activation stage: for every stage s the group's tiles
// are multiplied one after another, each into its own TMEM accumulator.
template <int NPAD>
__global__ void __launch_bounds__(kUmThreads, 1)
    q2_gemm_umma_kernel(const __grid_constant__ CUtensorMap wmap, int N, int nst, const uint8_t *__restrict__ bimg,
                        const int *__restrict__ exps, int M, float *__restrict__ Y, int ldy,
                        unsigned int *status, UmFuse fz) {
    constexpr int kB = um_bstage(NPAD);
    extern __shared__ uint8_t um_smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(um_smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sB = sm;
    uint8_t *sM = sB + kUmBStages * kB;
    uint8_t *sR = sM + kUmAStages * kUmMTile;
    UmShared *sh = reinterpret_cast<UmShared *>(sR + kUmRawStages * kUmRawStage);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = cdiv(N, kUmRows);
    const int my_tiles = blockIdx.x < ntiles ? cdiv(ntiles - (int)blockIdx.x, (int)gridDim.x) : 0;
    const int ngroups = cdiv(my_tiles, kUmGroup);

    // ---- set-up: barriers, the zero k-group of every m tile, TMEM
    if (threadIdx.x == 0) {
        for (int i = 0; i < kUmRawStages; ++i) {
            mbar_init(&sh->raw_full[i], 1);
            mbar_init(&sh->raw_empty[i], 4 * kUmRawSpan);  // 4 warps x kUmRawSpan uses
        }
        for (int i = 0; i < kUmAStages; ++i) {
            mbar_init(&sh->ab_full[i], 4);
        }
        for (int i = 0; i < kUmBStages; ++i) {
            mbar_init(&sh->b_full[i], 1);  // the B warp, once its copies have landed
            mbar_init(&sh->b_empty[i], kUmGroup);  // one commit per MMA thread
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh->acc_full[i], kUmGroup);
            mbar_init(&sh->acc_empty[i], kUmEpiWarps);
        }
        mbar_init(&sh->drain, kUmGroup);
        sh->abort_flag = 0u;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < kUmAStages * (kUmKgBytes / 16); i += blockDim.x) {
        const int a = i / (kUmKgBytes / 16), j = i % (kUmKgBytes / 16);
        *reinterpret_cast<uint4 *>(sM + (size_t)a * kUmMTile + kUmKgBytes + j * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_async_smem();
    if (warp == kUmMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         smem_u32(&sh->tmem_base)),
                     "r"(kUmCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    volatile uint32_t *abort_flag = &sh->abort_flag;

    if (warp == kUmTmaWarp) {
        // ---- raw weight stages, in the order the dequant warps consume them (independent of
        // the previous kernel: no programmatic wait)
        if (lane == 0) {
            uint32_t g = 0;
            bool ok = true;
            const int nsup = cdiv(nst, kUmRawSpan);
            for (int q = 0; ok && q < ngroups; ++q) {
                const int t0 = q * kUmGroup, tn = min(kUmGroup, my_tiles - t0);
                for (int S = 0; ok && S < nsup; ++S) {
                    for (int t = 0; t < tn; ++t) {
                        const uint32_t r = g % kUmRawStages;
                        if (!um_wait(&sh->raw_empty[r], ((g / kUmRawStages) & 1u) ^ 1u, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_tx(&sh->raw_full[r], kUmRawStage);
                        tma_load_2d(sR + (size_t)r * kUmRawStage, &wmap, S * kUmRawRow,
                                    ((int)blockIdx.x + (t0 + t) * (int)gridDim.x) * kUmRows, &sh->raw_full[r]);
                        ++g;
                    }
                }
            }
            // every copy issued lands before the CTA can exit
            for (uint32_t i = g > (uint32_t)kUmRawStages ? g - kUmRawStages : 0u; i < g; ++i)
                um_drain(&sh->raw_full[i % kUmRawStages], (i / kUmRawStages) & 1u);
        }
    } else if (warp == kUmBWarp) {
        // ---- activation stages (written by the prep kernel: after the programmatic wait).
        // They are small and L2-resident, so they go by cp.async on the load/store path rather
        // than queueing behind the weight stream's TMA copies.  A stage is signalled once it
        // has landed, kUmBLag stages behind the newest copy (kUmBLag < kUmBStages, so the MMA
        // always has the stage it waits for signalled before this warp waits on it in turn).
        pdl_wait();
        constexpr int kChunks = kB / 16;
        uint32_t g = 0, done = 0;
        bool ok = true;
        auto signal_oldest = [&](bool all) {
            if (all)
                asm volatile("cp.async.wait_group 0;\n" ::: "memory");
            else
                asm volatile("cp.async.wait_group %0;\n" ::"n"(kUmBLag) : "memory");
            fence_async_smem();  // cp.async wrote through the generic proxy; the MMA reads via the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh->b_full[done % kUmBStages]);
            ++done;
        };
        for (int q = 0; ok && q < ngroups; ++q) {
            for (int s = 0; s < nst; ++s) {
                const uint32_t b = g % kUmBStages;
                if (!um_wait_warp(&sh->b_empty[b], ((g / kUmBStages) & 1u) ^ 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                const uint32_t dst = smem_u32(sB + (size_t)b * kB);
                const uint8_t *src = bimg + (size_t)s * kB;
                for (int c = lane; c < kChunks; c += 32)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst + 16u * c), "l"(src + 16 * c)
                                 : "memory");
                asm volatile("cp.async.commit_group;\n" ::: "memory");
                ++g;
                if (g - done > (uint32_t)kUmBLag) signal_oldest(false);
            }
        }
        // every copy issued lands (and is signalled) before the warp leaves
        while (done < g) signal_oldest(true);
    } else if (warp >= kUmMmaWarp && warp < kUmMmaWarp + kUmGroup) {
        // ---- MMA issue: one thread per tile slot of a group (tile t of every group), so
        // that one thread's commit and barrier round trips overlap the other's issue.  Both
        // commit every B stage and every group, with or without a tile of their own.
        if (lane == 0) {
            const int me = warp - kUmMmaWarp;
            constexpr uint32_t idesc = umma_idesc<NPAD>();
            // descriptors of slot 0, k-step 0; a descriptor's low field is the start address
            // / 16 (below 2^14 anywhere in shared memory), so other slots and k-steps are
            // plain additions
            const uint64_t bdesc0 = umma_desc(smem_u32(sB), (NPAD / 8) * 128, 128);
            const uint64_t mdesc0 = umma_desc(smem_u32(sM), kUmKgBytes, 128);
            constexpr uint64_t kBStep = (2 * (NPAD / 8) * 128) >> 4;
            uint32_t gb = 0;
            bool ok = true;
            for (int q = 0; ok && q < ngroups; ++q) {
                const int tn = min(kUmGroup, my_tiles - q * kUmGroup);
                const uint32_t buf = (uint32_t)q & 1u;
                if (!um_wait(&sh->acc_empty[buf], (((uint32_t)q >> 1) & 1u) ^ 1u, abort_flag, status)) break;
                tc_fence_after();
                const uint32_t d = tmem + kUmAccBase + (buf * kUmGroup + (uint32_t)me) * kUmAccStride;
                for (int s = 0; ok && s < nst; ++s, ++gb) {
                    // both threads wait for the B stage, a thread without a tile too: its
                    // release of the B slot must not run ahead of the stage (b_empty counts
                    // one arrival per thread per stage)
                    const uint32_t b = gb % kUmBStages;
                    if (!um_wait(&sh->b_full[b], (gb / kUmBStages) & 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    if (me < tn) {
                        const uint32_t a = (gb & 1u) * kUmGroup + (uint32_t)me;  // this thread's A stage
                        if (!um_wait(&sh->ab_full[a], (gb >> 1) & 1u, abort_flag, status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t bd = bdesc0 + (uint64_t)((b * (uint32_t)kB) >> 4);
                        const uint32_t ta = tmem + a * kUmACols;
                        umma_f16_ts(d, ta, bd, idesc, s != 0);
#pragma unroll
                        for (int j = 1; j < kUmDataMmas; ++j) umma_f16_ts(d, ta + 8 * j, bd + j * kBStep, idesc, 1u);
                        // the blocks' offsets: m (A, shared memory) x the blocks' activation sums
                        umma_f16(d, mdesc0 + (uint64_t)((a * (uint32_t)kUmMTile) >> 4), bd + kUmDataMmas * kBStep,
                                 idesc, 1u);
                    }
                    umma_commit(&sh->b_empty[b]);
                }
                if (!ok) break;
                umma_commit(&sh->acc_full[buf]);
            }
            // no MMA may still be running when the CTA frees TMEM or exits
            umma_commit(&sh->drain);
            um_drain(&sh->drain, 0u);
        }
    } else if (warp >= kUmDeqWarp0) {
        // ---- dequant: thread = one weight row of the stage; A goes to TMEM, m to the m tile
        const int grp = (warp - kUmDeqWarp0) / 4;
        const int quarter = warp & 3;  // this warp's TMEM lanes: 32 * quarter ..
        const int row = 32 * quarter + lane;
        uint32_t scale_max = 0u;  // running max of |d|, |m| (f16x2)
        const int nsup = cdiv(nst, kUmRawSpan);
        uint32_t g = 0, gb = 0, rq = 0;  // A stages and activation stages so far; raw copies before q
        bool ok = true;
        for (int q = 0; ok && q < ngroups; ++q) {
            const int tn = min(kUmGroup, my_tiles - q * kUmGroup);
            for (int s = 0; ok && s < nst; ++s, ++gb) {
                for (int t = 0; t < tn; ++t, ++g) {
                    if ((int)(g % kUmDeqGroups) != grp) continue;
                    // raw copy of (tile t, stages 4 (s/4) ..): released after its last use
                    const uint32_t gr = rq + (uint32_t)((s / kUmRawSpan) * tn + t);
                    const uint32_t r = gr % kUmRawStages, a = (gb & 1u) * kUmGroup + (uint32_t)t;
                    const int first = s - s % kUmRawSpan;
                    const int uses = min(kUmRawSpan, nst - first);
                    const uint32_t release = (s == first + uses - 1) ? 1u + (uint32_t)(kUmRawSpan - uses) : 1u;
                    // the slot's previous user, activation stage gb - 2, must be done (its b_empty)
                    const uint32_t gp = gb - 2u;
                    if (!um_wait_warp(&sh->raw_full[r], (gr / kUmRawStages) & 1u, abort_flag, status) ||
                        (gb >= 2u && !um_wait_warp(&sh->b_empty[gp % kUmBStages], (gp / kUmBStages) & 1u, abort_flag,
                                                   status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the row's 48 raw bytes of stage s
                    const uint4 *src = reinterpret_cast<const uint4 *>(sR + (size_t)r * kUmRawStage + row * kUmRawRow +
                                                                       (s % kUmRawSpan) * kUmStageRaw);
                    uint32_t raw[12];
#pragma unroll
                    for (int i = 0; i < 3; ++i) {
                        const uint4 v = src[i];
                        raw[4 * i] = v.x;
                        raw[4 * i + 1] = v.y;
                        raw[4 * i + 2] = v.z;
                        raw[4 * i + 3] = v.w;
                    }
                    const uint32_t taddr = tmem + ((uint32_t)(32 * quarter) << 16) + a * kUmACols;
                    uint32_t w[32];
                    um_decode_blocks(raw, w, scale_max);
                    tmem_st32(taddr, w);
                    um_decode_blocks(raw + 6, w, scale_max);
                    tmem_st32(taddr + 32, w);
                    // m tile, k-group 16: slots 0..3 and 4..7 both hold the 4 blocks' m
                    const uint32_t m01 = (raw[2] >> 16) | (raw[5] & 0xFFFF0000u);
                    const uint32_t m23 = (raw[8] >> 16) | (raw[11] & 0xFFFF0000u);
                    *reinterpret_cast<uint4 *>(sM + (size_t)a * kUmMTile + (row >> 3) * 128 + (row & 7) * 16) =
                        make_uint4(m01, m23, m01, m23);
                    tmem_wait_st();
                    fence_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&sh->ab_full[a]);
                        mbar_arrive_n(&sh->raw_empty[r], release);
                    }
                }
            }
            rq += (uint32_t)(nsup * tn);
        }
        if (scale_mag_out_of_range(scale_max)) set_status(status, Q2_ERR_RANGE);
    } else {
        // ---- epilogue: TMEM -> registers -> Y (warp w reads TMEM lanes 32w..32w+31), and when
        // fused, each row's softmax (or argmax) partial over the tile's 128 tokens
        pdl_wait();
        pdl_trigger();
        if (threadIdx.x < 64) {
            const int m = threadIdx.x;
            sh->exps[m] = m < M ? exps[m] : 0;
            if (fz.tstats && m < M) {
                const float T = fz.temps ? fz.temps[m / fz.k1] : 0.0f;
                int mode = 1;
                float beta = fz.beta;
                if (fz.temps) {
                    mode = (T == 0.0f) ? 0 : ((T > 0.0f && T < INFINITY) ? 1 : -1);
                    beta = mode == 1 ? (float)(1.4426950408889634 / (double)T) : 0.0f;
                }
                sh->col_mode[m] = mode;
                sh->col_beta[m] = beta;
                sh->run[m] = make_float2(-INFINITY, mode == 0 ? __int_as_float(0x7FFFFFFF) : 0.0f);
            }
        }
        asm volatile("bar.sync 1, %0;\n" ::"n"(kUmEpiWarps * 32) : "memory");
        for (int q = 0; q < ngroups; ++q) {
            const int t0 = q * kUmGroup, tn = min(kUmGroup, my_tiles - t0);
            const uint32_t buf = (uint32_t)q & 1u;
            if (!um_wait_warp(&sh->acc_full[buf], ((uint32_t)q >> 1) & 1u, abort_flag, status)) break;
            tc_fence_after();
            for (int t = 0; t < tn; ++t) {
                float v[NPAD];
                const uint32_t col = kUmAccBase + (buf * kUmGroup + (uint32_t)t) * kUmAccStride;
#pragma unroll
                for (int c = 0; c < NPAD / 16; ++c)
                    tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + col + (uint32_t)(c * 16), v + 16 * c);
                tmem_wait_ld();
                const int tile = (int)blockIdx.x + (t0 + t) * (int)gridDim.x;
                const int n = tile * kUmRows + warp * 32 + lane;
#pragma unroll
                for (int m = 0; m < NPAD; ++m) v[m] = ldexpf(v[m], sh->exps[m]);
                if (n < N) {
#pragma unroll
                    for (int m = 0; m < NPAD; ++m)
                        if (m < M) Y[(size_t)m * ldy + n] = v[m];
                }
                if (fz.tstats) {
                    // per row (column m): this warp's (max, first argmax) over its 32 tokens, then
                    // for sampling rows the sum of 2^((y - max) beta); 8 columns at a time, so
                    // their shuffle chains overlap
#pragma unroll
                    for (int g0 = 0; g0 < NPAD; g0 += 8) {
                        if (g0 >= M) break;
                        float mx[8], zz[8];
                        int ix[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            mx[c] = (n < N && g0 + c < M) ? v[g0 + c] : -INFINITY;
                            ix[c] = n < N ? n : 0x7FFFFFFF;
                        }
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                const float m2 = __shfl_xor_sync(0xffffffffu, mx[c], o);
                                const int i2 = __shfl_xor_sync(0xffffffffu, ix[c], o);
                                if (um_better_arg(m2, i2, mx[c], ix[c])) {
                                    mx[c] = m2;
                                    ix[c] = i2;
                                }
                            }
                        }
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const float y = (n < N && g0 + c < M) ? v[g0 + c] : -INFINITY;
                            zz[c] = (y > -INFINITY) ? um_ex2((y - mx[c]) * sh->col_beta[g0 + c < M ? g0 + c : 0]) : 0.0f;
                        }
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                            for (int c = 0; c < 8; ++c) zz[c] += __shfl_xor_sync(0xffffffffu, zz[c], o);
                        }
                        if (lane == 0) {
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                const int m = g0 + c;
                                if (m < M)
                                    sh->part[warp][m] = sh->col_mode[m] == 0 ? make_float2(mx[c], __int_as_float(ix[c]))
                                                                             : make_float2(mx[c], zz[c]);
                            }
                        }
                    }
                    asm volatile("bar.sync 1, %0;\n" ::"n"(kUmEpiWarps * 32) : "memory");
                    if (threadIdx.x < M) {
                        // merge the four warps' partials of this tile into the CTA's running one
                        const int m = threadIdx.x, mode = sh->col_mode[m];
                        float2 r = sh->run[m];
                        if (mode == 1) {
                            const float beta = sh->col_beta[m];
                            float mx = r.x;
                            for (int w = 0; w < kUmEpiWarps; ++w) mx = fmaxf(mx, sh->part[w][m].x);
                            float z = (r.x > -INFINITY) ? r.y * um_ex2((r.x - mx) * beta) : 0.0f;
                            for (int w = 0; w < kUmEpiWarps; ++w) {
                                const float2 pw = sh->part[w][m];
                                if (pw.x > -INFINITY) z += pw.y * um_ex2((pw.x - mx) * beta);
                            }
                            r = make_float2(mx, z);
                        } else if (mode == 0) {
                            for (int w = 0; w < kUmEpiWarps; ++w) {
                                const float2 pw = sh->part[w][m];
                                if (um_better_arg(pw.x, __float_as_int(pw.y), r.x, __float_as_int(r.y))) r = pw;
                            }
                        }
                        sh->run[m] = r;
                    }
                    asm volatile("bar.sync 1, %0;\n" ::"n"(kUmEpiWarps * 32) : "memory");
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh->acc_empty[buf]);
        }
        // one partial per row per CTA: tstats [S][k1][gridDim.x]
        if (fz.tstats && threadIdx.x < M && sh->col_mode[threadIdx.x] >= 0)
            reinterpret_cast<float2 *>(fz.tstats)[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = sh->run[threadIdx.x];
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kUmMmaWarp) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(kUmCols) : "memory");
    }
}

// ---------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

size_t g_umma_smem[kCacheDevices][4];  // dynamic shared memory each NPAD variant was configured for, per device

template <int NPAD>
cudaError_t launch_umma_variant(const CUtensorMap &map, int N, int nst, const uint8_t *img, const int *exps, int M,
                                float *Y, int ldy, unsigned int *status, int num_sms, cudaStream_t s,
                                const UmFuse &fz) {
    auto kern = q2_gemm_umma_kernel<NPAD>;
    const size_t smem = um_smem_bytes(NPAD);
    const int dv = cache_device();
    if (dv < 0 || g_umma_smem[dv][NPAD / 16 - 1] < smem) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dv >= 0) g_umma_smem[dv][NPAD / 16 - 1] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(umma_gemm_grid(N, num_sms));
    cfg.blockDim = dim3(kUmThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, map, N, nst, img, exps, M, Y, ldy, status, fz);
}

}  // namespace

bool umma_gemm_usable(int M, int K) { return M >= 1 && M <= 64 && K % 128 == 0; }

bool umma_gemm_preferred(int M, int N, int K, int sms) {
    if (!umma_gemm_usable(M, K)) return false;
    if (M > 16) return true;
    const long long rows_per_sm = (long long)N / (sms > 0 ? sms : 1);
    if (M >= 9) return rows_per_sm >= 108;
    if (M >= 5) return rows_per_sm >= 216;
    return false;
}

size_t umma_gemm_ws_bytes(int M, int K) {
    const int npad = cdiv(M, 16) * 16;
    const int nst = cdiv(K / kBlockK, kUmBlocks);
    return align_up((size_t)nst * um_bstage(npad), 256) + 256;
}

// The bounded wait's give-up path (q2_selftest_wait_timeout): one thread waits, through the
// same um_wait the GEMM's roles use, on an mbarrier that nothing arrives on.  It holds no
// copies and no tensor memory, so after the wait runs out the kernel simply returns.
__global__ void __launch_bounds__(32) q2_wait_selftest_kernel(unsigned int *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)um_wait(&bar, 0u, &abort_flag, status);
}

cudaError_t launch_wait_selftest(unsigned int *status, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(32);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, q2_wait_selftest_kernel, status);
}

cudaError_t launch_prep_umma(const uint16_t *A, int lda, int M, int K, void *ws_region, cudaStream_t s) {
    const int nb = K / kBlockK;
    const int nst = cdiv(nb, kUmBlocks);
    const int npad = cdiv(M, 16) * 16;
    uint8_t *img = static_cast<uint8_t *>(ws_region);
    int *exps = reinterpret_cast<int *>(img + align_up((size_t)nst * um_bstage(npad), 256));
    return launch_pdl(prep_umma_kernel, dim3(npad), dim3(32 * cdiv(nst * kUmBlocks, 32)), s, A, lda, M, nb, nst,
                      npad, img, exps);
}

cudaError_t launch_gemm_umma(const void *W, int N, int K, int M, const void *ws_region, float *Y, int ldy,
                             unsigned int *status, int num_sms, cudaStream_t s, const UmFuse &fz) {
    const EncodeTiledFn encode = encode_tiled();
    if (!encode) return cudaErrorNotSupported;
    const int nb = K / kBlockK;
    const int nst = cdiv(nb, kUmBlocks);
    const int npad = cdiv(M, 16) * 16;
    const uint8_t *img = static_cast<const uint8_t *>(ws_region);
    const int *exps = reinterpret_cast<const int *>(img + align_up((size_t)nst * um_bstage(npad), 256));
    // the weights as a 2-D byte tensor [N rows][row_bytes]; one box = 48 B x 128 rows
    CUtensorMap map;
    const size_t row_bytes = (size_t)nb * kBlockBytes;
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)kUmRawRow, (cuuint32_t)kUmRows};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(W), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    switch (npad) {
        case 16: return launch_umma_variant<16>(map, N, nst, img, exps, M, Y, ldy, status, num_sms, s, fz);
        case 32: return launch_umma_variant<32>(map, N, nst, img, exps, M, Y, ldy, status, num_sms, s, fz);
        case 48: return launch_umma_variant<48>(map, N, nst, img, exps, M, Y, ldy, status, num_sms, s, fz);
        default: return launch_umma_variant<64>(map, N, nst, img, exps, M, Y, ldy, status, num_sms, s, fz);
    }
}

}  // namespace q2v
