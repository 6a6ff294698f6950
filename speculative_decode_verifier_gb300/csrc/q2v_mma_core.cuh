// q2v_mma_core.cuh -- the small-M Q2B32 dequant-GEMM core (up to 8 activation rows
// per pass) on mma.sync tensor-core instructions.
//
// Work split: a CTA owns 16 weight rows (the MMA's M dimension) and one warp per K tile
// of 8 Q2B32 blocks (256 weights).  Thread (g = lane/4, t = lane%4) loads blocks 2t and
// 2t+1 of rows g and g+8 of its tile straight into registers (24 bytes per row), so a
// warp streams 16 rows x 96 contiguous bytes.  Operand mapping: a k16 MMA step takes, for
// thread t's logical columns (2t, 2t+1) and (2t+8, 2t+9), the code pairs (c_i, c_{i+8})
// and (c_{i+1}, c_{i+9}) of one 16-code word of thread t's own block, so the A fragments
// are decoded from the thread's own registers with no exchange.  The activation rows are
// the 8-wide B operand; a separate prep kernel writes them once per call, as f16 under an
// exact per-row power-of-two scale, in exactly this permuted order, so a thread's B
// fragments for a whole tile are 128 contiguous bytes.  The Q2B32 offset m enters as its
// own small contraction (m-values x per-block activation sums, split hi+lo in f16) on
// m16n8k8.  The warps' partial sums are reduced in shared memory in warp order.
#pragma once

#include "q2v_common.cuh"

namespace q2v {

constexpr int kRowsPerCta = 16;
constexpr int kTileBlocks = 8;    // Q2B32 blocks per warp tile
constexpr int kMaxTileWarps = 32; // K <= 32 tiles * 256 = 8192 per CTA pass

// Prepared activations in global memory (the B operand), for R rows and K columns:
//   act   [R][nbp][16] u32: pair slot p of block b holds f16x2 (a[32b + 16(p/8) + p%8],
//                           a[32b + 16(p/8) + p%8 + 8]) scaled by 2^-exps[row];
//   shi, slo [R][nbp/2] u32: f16x2 (S[b], S[b+1]) split into hi + lo, S[b] the sum of
//                           block b's scaled f16 activations;
//   exps  [R] int.
// nbp = blocks rounded up to whole tiles; padding blocks hold zeros.
struct PrepLayout {
    int nb, ntk, nbp;
    __host__ __device__ explicit PrepLayout(int K) {
        nb = K / kBlockK;
        ntk = cdiv(nb, kTileBlocks);
        nbp = ntk * kTileBlocks;
    }
    __host__ __device__ size_t act_words_per_row() const { return (size_t)nbp * 16; }
    __host__ __device__ size_t sum_words_per_row() const { return (size_t)nbp / 2; }
    __host__ __device__ size_t bytes(int R) const {
        return align_up((size_t)R * act_words_per_row() * 4, 256) +
               2 * align_up((size_t)R * sum_words_per_row() * 4, 256) + align_up((size_t)R * 4, 256);
    }
};

struct PrepPtrs {
    uint32_t *act;
    uint32_t *shi;
    uint32_t *slo;
    int *exps;
    __host__ __device__ static PrepPtrs carve(void *base, const PrepLayout &L, int R) {
        PrepPtrs p;
        char *c = static_cast<char *>(base);
        p.act = reinterpret_cast<uint32_t *>(c);
        c += align_up((size_t)R * L.act_words_per_row() * 4, 256);
        p.shi = reinterpret_cast<uint32_t *>(c);
        c += align_up((size_t)R * L.sum_words_per_row() * 4, 256);
        p.slo = reinterpret_cast<uint32_t *>(c);
        c += align_up((size_t)R * L.sum_words_per_row() * 4, 256);
        p.exps = reinterpret_cast<int *>(c);
        return p;
    }
};

struct TileRegs {
    uint32_t w[2][2][3];  // [row g | g+8][block 2t | 2t+1][code word 0, code word 1, d|m]
};

// Load blocks 2t, 2t+1 of tile `tile` for rows g and g+8.  Rows >= rows_valid and blocks
// >= nb read as zero (they then contribute nothing).  ALIGN8: row_bytes % 8 == 0.
template <bool ALIGN8>
__device__ __forceinline__ void load_tile(TileRegs &r, const uint8_t *__restrict__ W0, size_t row_bytes,
                                          int rows_valid, int nb, int tile, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const int b0 = tile * kTileBlocks + 2 * t;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int row = g + 8 * rr;
        const uint8_t *p = W0 + (size_t)row * row_bytes + (size_t)b0 * kBlockBytes;
        const bool vr = row < rows_valid;
        const bool v0 = vr && b0 < nb, v1 = vr && b0 + 1 < nb;
        if (ALIGN8) {
            uint2 x0 = make_uint2(0, 0), x1 = make_uint2(0, 0), x2 = make_uint2(0, 0);
            if (v1) {
                x0 = __ldg(reinterpret_cast<const uint2 *>(p));
                x1 = __ldg(reinterpret_cast<const uint2 *>(p + 8));
                x2 = __ldg(reinterpret_cast<const uint2 *>(p + 16));
            } else if (v0) {
                x0 = __ldg(reinterpret_cast<const uint2 *>(p));
                x1.x = __ldg(reinterpret_cast<const uint32_t *>(p + 8));
            }
            r.w[rr][0][0] = x0.x; r.w[rr][0][1] = x0.y; r.w[rr][0][2] = x1.x;
            r.w[rr][1][0] = x1.y; r.w[rr][1][1] = x2.x; r.w[rr][1][2] = x2.y;
        } else {
            const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                r.w[rr][0][j] = v0 ? __ldg(q + j) : 0u;
                r.w[rr][1][j] = v1 ? __ldg(q + 3 + j) : 0u;
            }
        }
    }
}

// B-operand registers of one tile for one thread: column g's 16 pair slots of blocks
// 2t and 2t+1 (32 words) and the hi/lo block-sum words of that block pair.
struct ActRegs {
    uint32_t a[32];
    uint32_t shi, slo;
};

// row < 0: a zero column (past the last activation row).
__device__ __forceinline__ void load_act(ActRegs &r, const PrepPtrs &P, const PrepLayout &L, int row,
                                         int tile, int lane) {
    const int t = lane & 3;
    if (row < 0) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r.a[j] = 0u;
        r.shi = r.slo = 0u;
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(
        P.act + (size_t)row * L.act_words_per_row() + (size_t)(tile * kTileBlocks + 2 * t) * 16);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 v = __ldg(src + j);
        r.a[4 * j] = v.x; r.a[4 * j + 1] = v.y; r.a[4 * j + 2] = v.z; r.a[4 * j + 3] = v.w;
    }
    const size_t si = (size_t)row * L.sum_words_per_row() + (size_t)tile * 4 + t;
    r.shi = __ldg(P.shi + si);
    r.slo = __ldg(P.slo + si);
}

// acc (fragment rows g, g+8; columns 2t, 2t+1 of the n8 tile) += this tile's products.
__device__ __forceinline__ void compute_tile(const TileRegs &r, const ActRegs &b, float (&acc)[4],
                                             bool &range_bad) {
#pragma unroll
    for (int bi = 0; bi < 2; ++bi) {
        uint32_t d2a, nda, d2b, ndb;
        scale_pair(r.w[0][bi][2], d2a, nda);
        scale_pair(r.w[1][bi][2], d2b, ndb);
        range_bad |= scale_out_of_range(r.w[0][bi][2]) | scale_out_of_range(r.w[1][bi][2]);
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            const uint32_t c0 = r.w[0][bi][w], c1 = r.w[1][bi][w];
#define Q2V_STEP(PP)                                                                          \
    {                                                                                         \
        const uint32_t a0 = dequant_pair<2 * (PP)>(c0, d2a, nda);                             \
        const uint32_t a2 = dequant_pair<2 * (PP) + 1>(c0, d2a, nda);                         \
        const uint32_t a1 = dequant_pair<2 * (PP)>(c1, d2b, ndb);                             \
        const uint32_t a3 = dequant_pair<2 * (PP) + 1>(c1, d2b, ndb);                         \
        mma_16816(acc, a0, a1, a2, a3, b.a[bi * 16 + 8 * w + 2 * (PP)],                      \
                  b.a[bi * 16 + 8 * w + 2 * (PP) + 1]);                                       \
    }
            Q2V_STEP(0) Q2V_STEP(1) Q2V_STEP(2) Q2V_STEP(3)
#undef Q2V_STEP
        }
    }
    // offsets: sum over the tile's blocks of m[row][b] * S[b][col], with S = hi + lo
    const uint32_t am0 = prmt(r.w[0][0][2], r.w[0][1][2], 0x7632u);
    const uint32_t am1 = prmt(r.w[1][0][2], r.w[1][1][2], 0x7632u);
    mma_1688(acc, am0, am1, b.shi);
    mma_1688(acc, am0, am1, b.slo);
}

// red[16][8] (this warp's slice) <- the fragment accumulators.
__device__ __forceinline__ void store_fragments(float *red, const float (&acc)[4], int lane) {
    const int g = lane >> 2, t = lane & 3;
    red[g * 8 + 2 * t] = acc[0];
    red[g * 8 + 2 * t + 1] = acc[1];
    red[(g + 8) * 8 + 2 * t] = acc[2];
    red[(g + 8) * 8 + 2 * t + 1] = acc[3];
}

// Per-row power-of-two exponent e so that max|a| * 2^-e lies in [2^9, 2^10): the scaled
// activations and their 32-element block sums then fit f16 with room to spare.
__device__ __forceinline__ int act_exponent(float maxabs) {
    if (!(maxabs > 0.0f) || !isfinite(maxabs)) return 0;
    return ilogbf(maxabs) - 9;
}

}  // namespace q2v
