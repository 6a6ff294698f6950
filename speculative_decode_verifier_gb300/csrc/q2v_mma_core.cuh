// q2v_mma_core.cuh -- the small-M Q2B32 dequant-GEMM core (up to 8 activation rows
// per pass) on mma.sync tensor-core instructions.
//
// Work split: a CTA owns 16 weight rows (the MMA's M dimension) and one warp per K tile
// of 8 Q2B32 blocks (256 weights).  Thread (g = lane/4, t = lane%4) loads blocks 2t and
// 2t+1 of rows g and g+8 of its tile straight into registers (24 bytes per row), so a
// warp streams 16 rows x 96 contiguous bytes.  Operand mapping: a k16 MMA step takes, for
// thread t's logical columns (2t, 2t+1) and (2t+8, 2t+9), the code pairs (c_i, c_{i+8})
// and (c_{i+1}, c_{i+9}) of one 16-code word of thread t's own block, so the A fragments
// are decoded from the thread's own registers with no exchange (see dequant_pos: one lop3
// and one fma per two weights).  The activation rows are
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
    if (ALIGN8 && rows_valid == kRowsPerCta && (tile + 1) * kTileBlocks <= nb) {
        // a whole tile: no predicates
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const uint2 *p = reinterpret_cast<const uint2 *>(W0 + (size_t)(g + 8 * rr) * row_bytes + (size_t)b0 * kBlockBytes);
            const uint2 x0 = __ldg(p), x1 = __ldg(p + 1), x2 = __ldg(p + 2);
            r.w[rr][0][0] = x0.x; r.w[rr][0][1] = x0.y; r.w[rr][0][2] = x1.x;
            r.w[rr][1][0] = x1.y; r.w[rr][1][1] = x2.x; r.w[rr][1][2] = x2.y;
        }
        return;
    }
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

// A whole tile from per-thread row pointers (blocks 2t, 2t+1 of rows g and g+8, 8-byte
// aligned rows): three 8-byte loads per row, no predicates.
__device__ __forceinline__ void load_tile_fast(TileRegs &r, const uint2 *__restrict__ pa, const uint2 *__restrict__ pb) {
    const uint2 a0 = __ldg(pa), a1 = __ldg(pa + 1), a2 = __ldg(pa + 2);
    const uint2 b0 = __ldg(pb), b1 = __ldg(pb + 1), b2 = __ldg(pb + 2);
    r.w[0][0][0] = a0.x; r.w[0][0][1] = a0.y; r.w[0][0][2] = a1.x;
    r.w[0][1][0] = a1.y; r.w[0][1][1] = a2.x; r.w[0][1][2] = a2.y;
    r.w[1][0][0] = b0.x; r.w[1][0][1] = b0.y; r.w[1][0][2] = b1.x;
    r.w[1][1][0] = b1.y; r.w[1][1][1] = b2.x; r.w[1][1][2] = b2.y;
}

// ---------------------------------------------------------------- asynchronous copies

__device__ __forceinline__ void cp_async8(void *smem_dst, const void *gmem_src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
// Bring the line holding `p` into L2 (no completion to wait for).
__device__ __forceinline__ void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p)); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
__device__ __forceinline__ void cp_async4(void *smem_dst, const void *gmem_src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(gmem_src) : "memory");
}

// A weight tile staged in shared memory as 16 rows x 96 bytes (the tile's 8 blocks of each
// row, copied with 16-byte asynchronous copies: lane l brings 48 bytes of row l/2).  Thread
// (g, t) then reads blocks 2t, 2t+1 of rows g and g+8: three 8-byte loads per row; rows are
// 24 words apart, so each load instruction touches every bank exactly twice.
constexpr int kTileRowWords = 24;
constexpr int kTileWords = kRowsPerCta * kTileRowWords;

__device__ __forceinline__ void issue_tile_cpasync(uint32_t *stage, const uint8_t *W0, size_t row_bytes, int tile,
                                                   int lane) {
    const int row = lane >> 1, half = lane & 1;
    const uint8_t *src = W0 + (size_t)row * row_bytes + (size_t)tile * (kTileBlocks * kBlockBytes) + half * 48;
    uint32_t *dst = stage + row * kTileRowWords + half * 12;
    cp_async16(dst, src);
    cp_async16(dst + 4, src + 16);
    cp_async16(dst + 8, src + 32);
}

__device__ __forceinline__ void read_tile_smem(TileRegs &r, const uint32_t *stage, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const uint2 *p = reinterpret_cast<const uint2 *>(stage + (g + 8 * rr) * kTileRowWords + 6 * t);
        const uint2 x0 = p[0], x1 = p[1], x2 = p[2];
        r.w[rr][0][0] = x0.x; r.w[rr][0][1] = x0.y; r.w[rr][0][2] = x1.x;
        r.w[rr][1][0] = x1.y; r.w[rr][1][1] = x2.x; r.w[rr][1][2] = x2.y;
    }
}

// ---------------------------------------------------------------- shared-memory B operand
//
// Staged activations for up to `ncols` columns.  An MMA column without a row in the current
// slice reads column 0: it only feeds its own output column, which is never stored (each
// output of an MMA is one row of A times one column of B).  Column c holds its blocks in
// pairs: block pair j = b/2 starts at word 36*j (32 words of data and 4 of skew).  Inside a
// pair the 8-byte B fragments of the two blocks are interleaved: fragment u = 4w + pp of block
// b%2 (k16 step w, slot pair pp) sits at word 4u + 2(b%2), so one 16-byte load brings the
// fragments of both blocks for one step.  A warp's 16-byte load has threads g = 0..7 on
// columns CS*g apart (CS == 16 mod 32) and t = 0..3 on block pairs 36 words (4 banks) apart:
// each quarter-warp covers the 32 banks once, so 4 wavefronts, the minimum for 512 bytes.
// Each thread's base address is fixed for a tile; every step's offset is a compile-time
// constant.  Block sums follow: shi/slo[c][SWW] words, SWW == 4 (mod 32), word j = f16x2
// (S[2j], S[2j+1]).
constexpr int kPairWords = 36;

struct SmemAct {
    int CS, SWW, ncols;
    __host__ __device__ SmemAct(const PrepLayout &L, int ncols_)
        : CS((int)align_up((size_t)L.nbp / 2 * kPairWords, 32) + 16),
          SWW((int)align_up((size_t)L.nbp / 2, 32) + 4),
          ncols(ncols_) {}
    __host__ __device__ size_t words() const { return (size_t)ncols * (CS + 2 * SWW); }
    __host__ __device__ size_t bytes() const { return words() * 4; }
    __device__ uint32_t *act(uint32_t *sm, int c) const { return sm + (size_t)c * CS; }
    __device__ uint32_t *shi(uint32_t *sm, int c) const { return sm + (size_t)ncols * CS + (size_t)c * SWW; }
    __device__ uint32_t *slo(uint32_t *sm, int c) const { return sm + (size_t)ncols * (CS + SWW) + (size_t)c * SWW; }
};

// Issue (and commit as one group) the asynchronous copies of the prepared rows rows[0..n)
// (n <= ncols) into shared memory.  The caller waits for the group and synchronises.
__device__ __forceinline__ void stage_act_issue(uint32_t *sm, const SmemAct &SA, const PrepPtrs &P,
                                                const PrepLayout &L, const int *rows, int n) {
    const int n16 = L.nbp * 4;  // 16-byte groups per row
    const FastDiv div16((uint32_t)n16);
    for (int j = threadIdx.x; j < n * n16; j += blockDim.x) {
        const int c = (int)div16.div((uint32_t)j), q = j - c * n16;
        const int b = q >> 2, grp = q & 3;
        const uint32_t *src = P.act + (size_t)rows[c] * L.act_words_per_row() + (size_t)q * 4;
        // fragments 2 grp and 2 grp + 1 of block b
        uint32_t *dst = SA.act(sm, c) + (b >> 1) * kPairWords + 8 * grp + 2 * (b & 1);
        cp_async8(dst, src);
        cp_async8(dst + 4, src + 2);
    }
    const int nw = L.nbp / 2;
    const FastDiv divw((uint32_t)nw);
    for (int j = threadIdx.x; j < n * nw; j += blockDim.x) {
        const int c = (int)divw.div((uint32_t)j), i = j - c * nw;
        cp_async4(SA.shi(sm, c) + i, P.shi + (size_t)rows[c] * L.sum_words_per_row() + i);
        cp_async4(SA.slo(sm, c) + i, P.slo + (size_t)rows[c] * L.sum_words_per_row() + i);
    }
    cp_async_commit();
}

// Copy the prepared rows rows[0..n) into shared memory (all copies in flight at once).
// Block-wide; ends synchronised.
__device__ __forceinline__ void stage_act(uint32_t *sm, const SmemAct &SA, const PrepPtrs &P, const PrepLayout &L,
                                          const int *rows, int n) {
    stage_act_issue(sm, SA, P, L, rows, n);
    cp_async_wait<0>();
    __syncthreads();
}

// acc[0] += block 2t and the offsets' hi part, acc[1] += block 2t+1 and the lo part: two
// independent MMA chains, issued alternately.  B fragments come from the staged operand,
// column c0 + g (column c0 when g has no row in the current slice of n columns; see SmemAct).
__device__ __forceinline__ void compute_tile_smem(const TileRegs &r, uint32_t *sm, const SmemAct &SA, int n,
                                                  int tile, int lane, float (&acc)[2][4], uint32_t &scale_max,
                                                  int c0 = 0) {
    const int g = lane >> 2, t = lane & 3;
    const int cg = (g < n ? g : 0) + c0;  // staged columns c0 .. c0 + n - 1 are this MMA's 8 columns
    const uint32_t *base = SA.act(sm, cg) + (tile * 4 + t) * kPairWords;  // block pair (2t, 2t+1)
    uint32_t d2[2][2], nd[2][2];  // [block 2t | 2t+1][row g | g+8]
#pragma unroll
    for (int bi = 0; bi < 2; ++bi) {
        scale_pair(r.w[0][bi][2], d2[bi][0], nd[bi][0]);
        scale_pair(r.w[1][bi][2], d2[bi][1], nd[bi][1]);
        scale_max = scale_mag_max(scale_max, r.w[0][bi][2]);
        scale_max = scale_mag_max(scale_max, r.w[1][bi][2]);
    }
#pragma unroll
    for (int w = 0; w < 2; ++w) {
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
            // the step's B fragments of both blocks of the pair
            const uint4 bb = *reinterpret_cast<const uint4 *>(base + 4 * (4 * w + pp));
#pragma unroll
            for (int bi = 0; bi < 2; ++bi) {
                const uint32_t c0 = r.w[0][bi][w], c1 = r.w[1][bi][w];
                const uint32_t va = pp < 2 ? c0 : (c0 >> 8), vb = pp < 2 ? c1 : (c1 >> 8);
                uint32_t a0, a1, a2, a3;
                if (pp & 1) {
                    a0 = dequant_pos<4>(va, d2[bi][0], nd[bi][0]);
                    a2 = dequant_pos<6>(va, d2[bi][0], nd[bi][0]);
                    a1 = dequant_pos<4>(vb, d2[bi][1], nd[bi][1]);
                    a3 = dequant_pos<6>(vb, d2[bi][1], nd[bi][1]);
                } else {
                    a0 = dequant_pos<0>(va, d2[bi][0], nd[bi][0]);
                    a2 = dequant_pos<2>(va, d2[bi][0], nd[bi][0]);
                    a1 = dequant_pos<0>(vb, d2[bi][1], nd[bi][1]);
                    a3 = dequant_pos<2>(vb, d2[bi][1], nd[bi][1]);
                }
                mma_16816(acc[bi], a0, a1, a2, a3, bi ? bb.z : bb.x, bi ? bb.w : bb.y);
            }
        }
    }
    const uint32_t am0 = prmt(r.w[0][0][2], r.w[0][1][2], 0x7632u);
    const uint32_t am1 = prmt(r.w[1][0][2], r.w[1][1][2], 0x7632u);
    mma_1688(acc[0], am0, am1, SA.shi(sm, cg)[tile * 4 + t]);
    mma_1688(acc[1], am0, am1, SA.slo(sm, cg)[tile * 4 + t]);
}

// red[16][8] (this warp's slice) <- the sum of the two fragment accumulator chains.
__device__ __forceinline__ void store_fragments(float *red, const float (&acc)[2][4], int lane) {
    const int g = lane >> 2, t = lane & 3;
    red[g * 8 + 2 * t] = acc[0][0] + acc[1][0];
    red[g * 8 + 2 * t + 1] = acc[0][1] + acc[1][1];
    red[(g + 8) * 8 + 2 * t] = acc[0][2] + acc[1][2];
    red[(g + 8) * 8 + 2 * t + 1] = acc[0][3] + acc[1][3];
}

// Per-row power-of-two exponent e so that max|a| * 2^-e lies in [2^9, 2^10): the scaled
// activations and their 32-element block sums then fit f16 with room to spare.
__device__ __forceinline__ int act_exponent(float maxabs) {
    if (!(maxabs > 0.0f) || !isfinite(maxabs)) return 0;
    return ilogbf(maxabs) - 9;
}

// Write prepared block b of one row from its 32 activations: 16 f16x2 pair slots (slot p
// holds elements k0 and k0+8, k0 = 16*(p/8) + p%8), element j scaled by 2^-e * 4^-(j%4)
// (the row scale and the code-position factor of dequant_pos, both exact), and the sum of
// the block's f16 activations under the row scale alone, split into hi + lo f16.  The
// padding blocks (v all zero) store zeros.
__device__ __forceinline__ void prep_store_block(const float (&v)[32], int e, uint32_t *act_row, __half *sh,
                                                 __half *sl, int b) {
    __half h[32];
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        h[j] = __float2half_rn(ldexpf(v[j], -e - 2 * (j & 3)));
        s += __half2float(__float2half_rn(ldexpf(v[j], -e)));
    }
    uint32_t w[16];
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        const int k0 = 16 * (p >> 3) + (p & 7);
        w[p] = pack_half2(h[k0], h[k0 + 8]);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(act_row + (size_t)b * 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    const __half hi = __float2half_rn(s);
    sh[b] = hi;
    sl[b] = __float2half_rn(s - __half2float(hi));
}

// Block-wide max of non-negative values (blockDim.x <= 1024); every thread gets the result.
__device__ __forceinline__ float block_max_nonneg(float v, float *scratch32) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) scratch32[warp] = v;
    __syncthreads();
    float m = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, scratch32[w]);
    return m;
}

// Prepare one activation row (the whole block takes part; thread b handles Q2B32 block b of
// 32 activations, K <= 8192 so at most 256 blocks): per-row exponent, permuted f16x2 pair
// slots, hi/lo block sums.  Prepared row r is source row srow (srow < 0: a zero row); source
// rows are bf16 with leading dimension ld (ld % 8 == 0, 16-byte base).
__device__ __forceinline__ void prep_row_bf16(const uint16_t *__restrict__ src, int ld, int srow, int r,
                                              const PrepPtrs &P, const PrepLayout &L, float *scratch32) {
    const int b = threadIdx.x;
    float v[32];
    float mx = 0.0f;
    if (b < L.nb && srow >= 0) {
        const uint4 *p = reinterpret_cast<const uint4 *>(src + (size_t)srow * ld + (size_t)b * kBlockK);
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
    const int e = act_exponent(block_max_nonneg(mx, scratch32));
    if (b == 0) P.exps[r] = e;
    if (b < L.nbp)
        prep_store_block(v, e, P.act + (size_t)r * L.act_words_per_row(),
                         reinterpret_cast<__half *>(P.shi + (size_t)r * L.sum_words_per_row()),
                         reinterpret_cast<__half *>(P.slo + (size_t)r * L.sum_words_per_row()), b);
}

// ---------------------------------------------------------------- streamed units
//
// The streaming kernels give each CTA a contiguous range of units [u0, u1) (16 weight rows of
// one matrix, ntk tiles each), and each warp streams its units' tiles through its own ring.
// Two ways to share the range among the CTA's nw warps:
//   strided (EVEN = false): warp w takes units u0 + w, u0 + w + nw, ...;
//   even (EVEN = true): the range is flattened to tiles f = (u - u0) * ntk + tile and cut into
//     nw contiguous warp ranges whose lengths differ by at most two tiles, so no warp has a
//     whole unit more to stream than another.  A unit cut between warps is finished by the warp that
//     began it: each later warp holding a piece of it leaves that piece's 16 x 8 partial sum in
//     shared memory (its first piece, one slot per warp), and after one barrier the first warp
//     adds them in warp order, so the result does not depend on timing.
// Cuts fall on multiples of 2 tiles when ntk allows it (192 bytes of every row).  A cut can
// split a 128-byte line between two warps, whose reads of it, far apart in time, would each
// bring it from DRAM; on single tiles that re-read 3% of the weights and was slower, on 4-tile
// steps none, but at the verifier's MoE shape (~688 tiles over 24 warps) 4-tile steps leave the
// busiest warp 32 tiles against 30: measured, gate+up took 54.9-55.4 us with 2-tile cuts,
// 55.7-56.2 with 4-tile and 56.2-56.3 with 1-tile cuts.
struct WarpTiles {
    int f0, f1;
};
__device__ __forceinline__ WarpTiles warp_tiles(int u0, int u1, int ntk, int nw, int w) {
    const int G = (ntk & 1) == 0 ? 2 : 1;
    const long long Tg = (long long)(u1 - u0) * (ntk / G);
    return {(int)(Tg * w / nw) * G, (int)(Tg * (w + 1) / nw) * G};
}

// A warp's first unit, first tile and tile count under either split.
template <bool EVEN>
__device__ __forceinline__ void warp_start(int u0, int u1, int ntk, int nw, int w, int &u, int &tile, int &n) {
    if (EVEN) {
        const WarpTiles r = warp_tiles(u0, u1, ntk, nw, w);
        u = u0 + r.f0 / ntk;
        tile = r.f0 - (u - u0) * ntk;
        n = r.f1 - r.f0;
    } else {
        u = u0 + w;
        tile = 0;
        n = u < u1 ? cdiv(u1 - u, nw) * ntk : 0;
    }
}

// Producer cursor over a warp's tiles: one cp.async group per call, empty once the warp's tiles
// are exhausted (the group count stays uniform).  unit_w(u) is the first weight row of unit u.
template <bool EVEN, class UnitW>
struct TileCursor {
    const uint8_t *W;
    int u, tile, left;
    __device__ __forceinline__ void begin(int u0, int u1, int ntk, int nw, int warp, const UnitW &unit_w) {
        warp_start<EVEN>(u0, u1, ntk, nw, warp, u, tile, left);
        W = left > 0 ? unit_w(u) : nullptr;
    }
    __device__ __forceinline__ void produce(uint32_t *stage, size_t row_bytes, int ntk, int nw, int lane,
                                            const UnitW &unit_w) {
        if (left > 0) {
            issue_tile_cpasync(stage, W, row_bytes, tile, lane);
            --left;
            if (++tile == ntk) {
                tile = 0;
                u += EVEN ? 1 : nw;
                if (left > 0) W = unit_w(u);
            }
        }
        cp_async_commit();
    }
};

// Consume a warp's tiles through its RING-stage ring (the caller has issued RING - 1 groups
// with `cur` and waited for the staged activations).  cols(u) gives unit u's MMA columns
// {n, c0} (columns c0 .. c0 + n - 1 of the staged activations); store(u, nc, v) writes the
// unit's result, nc = cols(u), v[q] the sum for rows g + 8 (q >> 1), column 2t + (q & 1).
// EVEN: part is nw x 128 floats of shared memory, and every thread of the CTA calls this (it
// holds one barrier); a unit cut at the range's start is recognised by its index, a cut at the
// end after the loop, so the loop carries no more state than the strided one.
template <int RING, bool EVEN, class UnitW, class Cols, class Store>
__device__ __forceinline__ void stream_warp_tiles(TileCursor<EVEN, UnitW> &cur, uint32_t *ring, uint32_t *sm_act,
                                                  const SmemAct &SA, float *part, int u0, int u1, int ntk,
                                                  size_t row_bytes, int nw, int warp, int lane, const UnitW &unit_w,
                                                  const Cols &cols, const Store &store, uint32_t &scale_max) {
    int cu, ctile, n;
    warp_start<EVEN>(u0, u1, ntk, nw, warp, cu, ctile, n);
    const int head_u = EVEN && ctile != 0 ? cu : -1;  // begun by an earlier warp
    int2 nc = n > 0 ? cols(cu) : make_int2(0, 0);
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    auto finish = [&](bool keep) {
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[q] = acc[0][q] + acc[1][q];
            acc[0][q] = 0.0f;
            acc[1][q] = 0.0f;
        }
        if (EVEN && cu == head_u)
            *reinterpret_cast<float4 *>(part + warp * 128 + lane * 4) = make_float4(v[0], v[1], v[2], v[3]);
        else if (!keep)
            store(cu, nc, v);
    };
    int pst = RING - 1, cst = 0;  // producer and consumer ring stages
    for (int it = 0; it < n; ++it) {
        cur.produce(ring + pst * kTileWords, row_bytes, ntk, nw, lane, unit_w);
        pst = pst == RING - 1 ? 0 : pst + 1;
        cp_async_wait<RING - 1>();  // this tile's group has landed
        __syncwarp();
        TileRegs tr;
        read_tile_smem(tr, ring + cst * kTileWords, lane);
        cst = cst == RING - 1 ? 0 : cst + 1;
        compute_tile_smem(tr, sm_act, SA, nc.x, ctile, lane, acc, scale_max, nc.y);
        if (++ctile == ntk) {
            finish(false);
            ctile = 0;
            cu += EVEN ? 1 : nw;
            if (it + 1 < n) nc = cols(cu);
        }
        __syncwarp();  // every lane has read this stage before a later copy refills it
    }
    cp_async_wait<0>();
    if (!EVEN) return;
    // the range ends inside unit cu: its piece is a later warp's part, or this warp began it
    const bool tail = ctile != 0 && cu != head_u;
    if (ctile != 0 && cu == head_u) finish(true);
    __syncthreads();  // every piece of a cut unit is in shared memory
    if (tail) {
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = acc[0][q] + acc[1][q];
        const int fend = (cu + 1 - u0) * ntk;  // first tile after the unit
        for (int w2 = warp + 1; w2 < nw; ++w2) {
            const WarpTiles r2 = warp_tiles(u0, u1, ntk, nw, w2);
            if (r2.f0 >= fend) break;
            if (r2.f1 > r2.f0) {
                const float4 p = *reinterpret_cast<const float4 *>(part + w2 * 128 + lane * 4);
                v[0] += p.x;
                v[1] += p.y;
                v[2] += p.z;
                v[3] += p.w;
            }
        }
        store(cu, nc, v);
    }
}

}  // namespace q2v
