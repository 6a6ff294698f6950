// q2v_moe.cu -- routed-expert FFN of the verify forward on sm_103a.
//
// The verifier "repeatedly executes attention, routed MoE, projections and the
// vocabulary head" over the K+1 rows ("Optimizing DeepSeek-V4-Flash on a single NVIDIA
// GB10/GX10 with DSpark speculative decoding", page 2, verifier-bottleneck reply); the
// engines fused the router, fused gate+up+SwiGLU for decode ("1x Spark tuned DSpark for
// DeepSeek-V4-Flash ...", reply on the decode arc) and deduplicated expert reads across
// rows ("ds4-on-spark", section "What the fork adds": MoE gate_up expert dedup).
//
// Steps (one stream, no host synchronisation):
//   1. route:    softmax over experts, top-k by logit (ties to the lower index), gate
//                weights, a deterministic counting sort of the (row, slot) pairs by expert
//                (pairs of one expert ordered by row), the list of active experts;
//   2. prep X:   the activation rows in the small-M GEMM's B-operand layout;
//   3. gate/up:  one grouped GEMM over (active expert, gate|up, 16-row tile) items; every
//                expert's weights are read once for all rows routed to it;
//   4. prep h:   h = silu(gate) * up, fused into the B-operand prep of the down GEMM;
//   5. down:     grouped GEMM over (active expert, 16-row tile) items;
//   6. combine:  Y[r] = sum over slots, in slot order, of g * out (deterministic).
#include <math.h>

#include "q2v_kernels.cuh"

namespace q2v {

constexpr int kRouteThreads = 1024;

__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(MoeArgs a, MoeWs w) {
    __shared__ int s_ids[64 * 16];
    __shared__ float s_g[64 * 16];
    __shared__ int s_cnt[257];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    const int E = a.E, K = a.topk, M = a.M;
    for (int e = tid; e <= E; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    for (int r = warp; r < M; r += nw) {
        const float *l = a.router + (size_t)r * E;
        float mx = -INFINITY;
        for (int e = lane; e < E; e += 32) mx = fmaxf(mx, l[e]);
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float z = 0.0f;
        for (int e = lane; e < E; e += 32) z += expf(l[e] - mx);
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        // top-k by logit: repeated arg-max, ties to the lower index
        unsigned taken = 0u;  // bit q: expert lane + 32q already selected
        float gsum = 0.0f;
        for (int t = 0; t < K; ++t) {
            float best = -INFINITY;
            int bi = 0x7fffffff;
            for (int e = lane, q = 0; e < E; e += 32, ++q) {
                const bool tk = (taken >> q) & 1u;
                const float v = l[e];
                if (!tk && (v > best || (v == best && e < bi) || bi == 0x7fffffff)) {
                    best = v;
                    bi = e;
                }
            }
            for (int o = 16; o > 0; o >>= 1) {
                const float ob = __shfl_xor_sync(0xffffffffu, best, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ob > best || (ob == best && oi < bi)) {
                    best = ob;
                    bi = oi;
                }
            }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            const float g = expf(best - mx) / z;
            gsum += g;
            if (lane == 0) {
                s_ids[r * K + t] = bi;
                s_g[r * K + t] = g;
            }
        }
        __syncwarp();
        if (lane == 0 && (a.flags & Q2_MOE_RENORMALIZE))
            for (int t = 0; t < K; ++t) s_g[r * K + t] /= gsum;
    }
    __syncthreads();
    const int P = M * K;
    for (int p = tid; p < P; p += blockDim.x) atomicAdd(&s_cnt[s_ids[p]], 1);
    __syncthreads();
    if (tid == 0) {
        int off = 0, na = 0;
        for (int e = 0; e < E; ++e) {
            w.offsets[e] = off;
            w.counts[e] = s_cnt[e];
            if (s_cnt[e] > 0) w.active[na++] = e;
            off += s_cnt[e];
        }
        w.offsets[E] = off;
        w.active[E] = na;
    }
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) {
        const int r = p / K, e = s_ids[p];
        int before = 0;  // rows < r routed to e (a row picks an expert at most once)
        for (int q = 0; q < r * K; ++q) before += (s_ids[q] == e);
        const int pos = w.offsets[e] + before;
        w.pair_row[pos] = r;
        w.pair_of[p] = pos;
        w.gate_w[p] = s_g[p];
        if (a.ids_out) a.ids_out[p] = e;
        if (a.w_out) a.w_out[p] = s_g[p];
    }
}

// h = silu(gate) * up for the grouped pairs, written straight into the down GEMM's
// B-operand layout (one CTA per pair; same scaling rules as prep_act_kernel).
__global__ void __launch_bounds__(256) moe_prep_h_kernel(const float *__restrict__ gu, int P, int F,
                                                         PrepPtrs Pp, PrepLayout L) {
    const int r = blockIdx.x;
    if (r >= P) return;
    const int tid = threadIdx.x;
    __shared__ float red[8];
    __shared__ int sexp;
    const float *G = gu + (size_t)r * F;
    const float *U = gu + (size_t)P * F + (size_t)r * F;
    auto h = [&](int k) -> float {
        const float z = G[k];
        return z / (1.0f + expf(-z)) * U[k];
    };
    float mx = 0.0f;
    for (int k = tid; k < F; k += blockDim.x) mx = fmaxf(mx, fabsf(h(k)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    if (tid == 0) {
        float m = 0.0f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
        sexp = act_exponent(m);
        Pp.exps[r] = sexp;
    }
    __syncthreads();
    const int e = sexp;
    uint32_t *act = Pp.act + (size_t)r * L.act_words_per_row();
    for (int j = tid; j < L.nbp * 16; j += blockDim.x) {
        const int b = j >> 4, p = j & 15;
        uint32_t v = 0;
        if (b < L.nb) {
            const int k0 = b * kBlockK + 16 * (p >> 3) + (p & 7);
            v = pack_half2(__float2half_rn(ldexpf(h(k0), -e)), __float2half_rn(ldexpf(h(k0 + 8), -e)));
        }
        act[j] = v;
    }
    __half *sh = reinterpret_cast<__half *>(Pp.shi + (size_t)r * L.sum_words_per_row());
    __half *sl = reinterpret_cast<__half *>(Pp.slo + (size_t)r * L.sum_words_per_row());
    for (int b = tid; b < L.nbp; b += blockDim.x) {
        float s = 0.0f;
        if (b < L.nb)
            for (int kk = 0; kk < kBlockK; ++kk) s += __half2float(__float2half_rn(ldexpf(h(b * kBlockK + kk), -e)));
        const __half hi = __float2half_rn(s);
        sh[b] = hi;
        sl[b] = __float2half_rn(s - __half2float(hi));
    }
}

// Grouped small-M GEMM over work items (active expert, matrix, 16-row tile).
//   GATEUP: matrices {Wg, Wu} [E][F][H/32], K = H, activation col c of expert e is the
//           prepared X row pair_row[offsets[e] + c]; output gu[matrix][pos][F].
//   DOWN:   matrix Wd [E][H][F/32], K = F, activation col c is prepared h row
//           offsets[e] + c; output out[pos][H].
// Each CTA takes a contiguous range of items (so consecutive items share an expert).
template <bool GATEUP, bool ALIGN8>
__global__ void __launch_bounds__(1024) moe_grouped_kernel(MoeArgs a, MoeWs w, float *__restrict__ outp) {
    __shared__ float red[kMaxTileWarps * kRowsPerCta * 8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const int K = GATEUP ? a.H : a.F;
    const int Nrows = GATEUP ? a.F : a.H;
    const PrepLayout L(K);
    const PrepPtrs &Pp = GATEUP ? w.prepX : w.prepH;
    const int tiles = cdiv(Nrows, kRowsPerCta);
    const int per_expert = (GATEUP ? 2 : 1) * tiles;
    const int n_active = w.active[a.E];
    const int total = n_active * per_expert;
    const int q = cdiv(total, gridDim.x);
    const int i0 = blockIdx.x * q, i1 = min(total, i0 + q);
    const size_t row_bytes = (size_t)L.nb * kBlockBytes;
    const size_t mat_bytes = (size_t)Nrows * row_bytes;
    const int P = a.M * a.topk;
    bool range_bad = false;
    for (int item = i0; item < i1; ++item) {
        const int ai = item / per_expert, rem = item - ai * per_expert;
        const int mat = GATEUP ? rem / tiles : 0;
        const int tile = GATEUP ? rem - mat * tiles : rem;
        const int e = w.active[ai];
        const int off = w.offsets[e], cnt = w.counts[e];
        const uint8_t *Wm = GATEUP ? (mat ? a.Wu : a.Wg) : a.Wd;
        const int n0 = tile * kRowsPerCta;
        const int rows_valid = min(kRowsPerCta, Nrows - n0);
        const uint8_t *W0 = Wm + (size_t)e * mat_bytes + (size_t)n0 * row_bytes;
        TileRegs wr;
        if (warp < L.ntk) load_tile<ALIGN8>(wr, W0, row_bytes, rows_valid, L.nb, warp, lane);
        float *dst = outp + (GATEUP ? (size_t)mat * P * Nrows : 0);
        for (int m0 = 0; m0 < cnt; m0 += 8) {
            const int mc = min(8, cnt - m0);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            if (warp < L.ntk) {
                const int col = lane >> 2;
                int prow = -1;
                if (col < mc) prow = GATEUP ? w.pair_row[off + m0 + col] : off + m0 + col;
                ActRegs ar;
                load_act(ar, Pp, L, prow, warp, lane);
                compute_tile(wr, ar, acc, range_bad);
            }
            store_fragments(red + warp * kRowsPerCta * 8, acc, lane);
            __syncthreads();
            for (int j = threadIdx.x; j < kRowsPerCta * mc; j += blockDim.x) {
                const int r = j % kRowsPerCta, m = j / kRowsPerCta;
                float s = 0.0f;
                for (int ww = 0; ww < nwarps; ++ww) s += red[ww * kRowsPerCta * 8 + r * 8 + m];
                const int pos = off + m0 + m;
                const int ex = GATEUP ? Pp.exps[w.pair_row[pos]] : Pp.exps[pos];
                if (r < rows_valid) dst[(size_t)pos * Nrows + n0 + r] = ldexpf(s, ex);
            }
            __syncthreads();
        }
    }
    if (range_bad) set_status(a.status, Q2_ERR_RANGE);
}

__global__ void moe_combine_kernel(MoeArgs a, MoeWs w) {
    const int H = a.H, K = a.topk;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)a.M * H;
         i += (size_t)gridDim.x * blockDim.x) {
        const int r = (int)(i / H), n = (int)(i - (size_t)r * H);
        float y = 0.0f;
        for (int t = 0; t < K; ++t) {
            const int p = r * K + t;
            y = fmaf(w.gate_w[p], w.out[(size_t)w.pair_of[p] * H + n], y);
        }
        a.Y[i] = y;
    }
}

cudaError_t launch_moe(const MoeArgs &a, const MoeWs &w, int num_sms, cudaStream_t s) {
    moe_route_kernel<<<1, kRouteThreads, 0, s>>>(a, w);
    const PrepLayout LX(a.H), LH(a.F);
    launch_prep(a.X, false, a.H, nullptr, a.M, a.H, w.prepX, LX, s);
    const int grid = 2 * num_sms;
    const int P = a.M * a.topk;
    if (LX.nb % 2 == 0)
        moe_grouped_kernel<true, true><<<grid, 32 * LX.ntk, 0, s>>>(a, w, w.h);
    else
        moe_grouped_kernel<true, false><<<grid, 32 * LX.ntk, 0, s>>>(a, w, w.h);
    moe_prep_h_kernel<<<P, 256, 0, s>>>(w.h, P, a.F, w.prepH, LH);
    if (LH.nb % 2 == 0)
        moe_grouped_kernel<false, true><<<grid, 32 * LH.ntk, 0, s>>>(a, w, w.out);
    else
        moe_grouped_kernel<false, false><<<grid, 32 * LH.ntk, 0, s>>>(a, w, w.out);
    moe_combine_kernel<<<min(cdiv(a.M * a.H, 256), 4 * num_sms), 256, 0, s>>>(a, w);
    return cudaGetLastError();
}

}  // namespace q2v
