// q2v_moe.cu -- routed-expert FFN of the verify forward on sm_103a.
//
// Each verify runs the routed-expert FFN (with attention, the projections and the vocabulary
// head) over the K+1 rows ("Optimizing DeepSeek-V4-Flash on a single NVIDIA
// GB10/GX10 with DSpark speculative decoding", page 2, verifier-bottleneck reply); the
// engines fused the router, fused gate+up+SwiGLU for decode ("1x Spark tuned DSpark for
// DeepSeek-V4-Flash ...", reply on the decode arc) and deduplicated expert reads across
// rows ("ds4-on-spark", section "What the fork adds").
//
// Steps (one stream, no host synchronisation):
//   1. route:    softmax over experts, top-k by logit (ties to the lower index), gate
//                weights, a deterministic counting sort of the (row, slot) pairs by expert
//                (pairs of one expert ordered by row), the list of active experts;
//   2. prep X:   the activation rows in the small-M GEMM's B-operand layout;
//   3. gate/up:  one grouped GEMM over units (active expert, gate|up, 16-row group, K split);
//                every active expert's weights are read once for all rows routed to it.  At
//                most 8 rows without a K split (the verifier shape): moe_gateup_stream_kernel,
//                one 24-warp CTA per SM with all X rows staged once and its tiles cut evenly
//                over the warps; otherwise moe_stream_kernel, whose CTAs stage the prepared rows
//                of each expert run and whose warps take units in turn; every warp streams its
//                weight tiles through its own cp.async ring;
//   4. prep h:   h = silu(sum of gate splits) * (sum of up splits), fused into the B-operand
//                prep of the down GEMM;
//   5. down:     the same over (active expert, 16-row group, K split) units:
//                moe_down_stream_kernel at the verifier shape (the h rows of the CTA's one or two
//                experts staged once), moe_stream_kernel otherwise;
//   6. combine:  Y[r] = sum over slots, in slot order, of g * (sum of the down splits).
// Every sum runs in a fixed order, so the result is deterministic.
#include <math.h>

#include "q2v_kernels.cuh"

namespace q2v {

constexpr int kRoutePrepThreads = 256;

// Routing of the M rows (one CTA): softmax over E, top-k by logit (ties to the lower index),
// counting sort of the (row, slot) pairs by expert.  E <= 256: a lane keeps its 8 logits in
// registers across the k arg-max rounds.
__device__ __forceinline__ void route_rows(const MoeArgs &a, const MoeWs &w, int *s_ids, float *s_g, int *s_cnt,
                                           int *s_off) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    const int E = a.E, K = a.topk, M = a.M;
    for (int e = tid; e <= E; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    for (int r = warp; r < M; r += nw) {
        const float *l = a.router + (size_t)r * E;
        float lv[8];
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = lane + 32 * q;
            lv[q] = e < E ? l[e] : -INFINITY;
            mx = fmaxf(mx, lv[q]);
        }
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float z = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (lane + 32 * q < E) z += expf(lv[q] - mx);
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        // top-k by logit: repeated arg-max, ties to the lower index
        unsigned taken = 0u;  // bit q: expert lane + 32q already selected
        float gsum = 0.0f;
        for (int t = 0; t < K; ++t) {
            float best = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int e = lane + 32 * q;
                const bool tk = (taken >> q) & 1u;
                if (e < E && !tk && (lv[q] > best || (lv[q] == best && e < bi) || bi == 0x7fffffff)) {
                    best = lv[q];
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
    if (warp == 0) {
        // expert offsets and the ascending list of active experts: lane l holds experts
        // 8l .. 8l+7 (E <= 256), one warp scan of the counts and of the active flags
        int c[8], sum = 0, nz = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = 8 * lane + q;
            c[q] = e < E ? s_cnt[e] : 0;
            sum += c[q];
            nz += c[q] > 0;
        }
        int isum = sum, inz = nz;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ts = __shfl_up_sync(0xffffffffu, isum, o), tz = __shfl_up_sync(0xffffffffu, inz, o);
            if (lane >= o) {
                isum += ts;
                inz += tz;
            }
        }
        int off = isum - sum, na = inz - nz;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = 8 * lane + q;
            if (e < E) {
                s_off[e] = off;
                w.offsets[e] = off;
                w.counts[e] = c[q];
                if (c[q] > 0) w.active[na++] = e;
            }
            off += c[q];
        }
        if (lane == 31) {
            s_off[E] = isum;
            w.offsets[E] = isum;
            w.active[E] = inz;
        }
    }
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) {
        const int r = p / K, e = s_ids[p];
        int before = 0;  // rows < r routed to e (a row picks an expert at most once)
        for (int q = 0; q < r * K; ++q) before += (s_ids[q] == e);
        const int pos = s_off[e] + before;
        w.pair_row[pos] = r;
        w.pair_of[p] = pos;
        w.slot_of[pos] = p;
        w.gate_w[p] = s_g[p];
        if (a.ids_out) a.ids_out[p] = e;
        if (a.w_out) a.w_out[p] = s_g[p];
    }
}

// CTAs 0..M-1 prepare the activation rows of X (the B operand of gate and up); CTA M routes.
// The two are independent, so one launch covers both.
__global__ void __launch_bounds__(kRoutePrepThreads) moe_route_prep_kernel(MoeArgs a, MoeWs w, PrepLayout LX) {
    __shared__ float scratch[32];
    __shared__ int s_ids[64 * 16];
    __shared__ float s_g[64 * 16];
    __shared__ int s_cnt[257];
    __shared__ int s_off[257];
    pdl_wait();
    pdl_trigger();
    if ((int)blockIdx.x < a.M) {
        prep_row_bf16(a.X, a.H, (int)blockIdx.x, (int)blockIdx.x, w.prepX, LX, scratch);
        return;
    }
    route_rows(a, w, s_ids, s_g, s_cnt, s_off);
}


// h for grouped pair r: silu(sum_ks G[ks][r]) * sum_ks U[ks][r] (fixed order), prepared as
// the down GEMM's B operand.  One CTA per pair, one thread per 32-element block of F.
__global__ void __launch_bounds__(256) moe_prep_h_kernel(const float *__restrict__ gu, int P, int F, int KS,
                                                         PrepPtrs Pp, PrepLayout L) {
    __shared__ float scratch[32];
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x, b = threadIdx.x;
    float v[32];
    float mx = 0.0f;
    if (b < L.nb) {
        float g[32], u[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) g[j] = u[j] = 0.0f;
        for (int ks = 0; ks < KS; ++ks) {
            const float4 *G = reinterpret_cast<const float4 *>(gu + ((size_t)(ks * 2 + 0) * P + r) * F + (size_t)b * 32);
            const float4 *U = reinterpret_cast<const float4 *>(gu + ((size_t)(ks * 2 + 1) * P + r) * F + (size_t)b * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 x = G[j], y = U[j];
                g[4 * j] += x.x; g[4 * j + 1] += x.y; g[4 * j + 2] += x.z; g[4 * j + 3] += x.w;
                u[4 * j] += y.x; u[4 * j + 1] += y.y; u[4 * j + 2] += y.z; u[4 * j + 3] += y.w;
            }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            v[j] = g[j] / (1.0f + expf(-g[j])) * u[j];
            mx = fmaxf(mx, fabsf(v[j]));
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.0f;
    }
    const int e = act_exponent(block_max_nonneg(mx, scratch));
    if (b == 0) Pp.exps[r] = e;
    if (b < L.nbp)
        prep_store_block(v, e, Pp.act + (size_t)r * L.act_words_per_row(),
                         reinterpret_cast<__half *>(Pp.shi + (size_t)r * L.sum_words_per_row()),
                         reinterpret_cast<__half *>(Pp.slo + (size_t)r * L.sum_words_per_row()), b);
}

// Grouped small-M GEMM over units u = (active expert, matrix, 16-row group, K split),
// enumerated expert-major.
//   GATEUP: matrices {Wg, Wu} [E][F][H/32], K = H; activation column c of expert e is the
//           prepared X row pair_row[offsets[e] + c]; output gu[ks][matrix][pos][F].
//   DOWN:   matrix Wd [E][H][F/32], K = F; activation column c is prepared h row
//           offsets[e] + c; output out[ks][slot_of[pos]][H] (by (row, slot), for the combine).
// Each CTA takes a contiguous range of units.  Within it, for each run of units of one
// expert (and each slice of 8 of its rows), the CTA stages those rows' prepared
// activations in shared memory once; its warps then take the run's units round-robin and
// stream their weight tiles with two tiles in flight ahead of the one being computed.
// Accumulators never leave the warp: each unit's 16 x 8 partial result is written straight
// to its K-split slot, so there are no cross-warp reductions.
struct UnitInfo {
    const uint8_t *W0;
    int rows_valid, n0, t0, t1, mat, ks, ai;
};

template <bool GATEUP>
struct UnitMap {
    FastDiv per_expert, groups, KS;
    int tps, ntk, Nrows;
    size_t row_bytes, mat_bytes;
    const uint8_t *Wg, *Wu, *Wd;
    const int *active;
    __device__ UnitInfo operator()(int u) const {
        UnitInfo ui;
        ui.ai = (int)per_expert.div((uint32_t)u);
        const uint32_t rem = (uint32_t)u - (uint32_t)ui.ai * per_expert.d;
        const uint32_t r1 = KS.div(rem);
        ui.ks = (int)(rem - r1 * KS.d);
        ui.mat = (int)groups.div(r1);
        const int grp = (int)(r1 - (uint32_t)ui.mat * groups.d);
        const int e = active[ui.ai];
        ui.n0 = grp * kRowsPerCta;
        ui.rows_valid = min(kRowsPerCta, Nrows - ui.n0);
        ui.t0 = ui.ks * tps;
        ui.t1 = min(ntk, ui.t0 + tps);
        const uint8_t *Wm = GATEUP ? (ui.mat ? Wu : Wg) : Wd;
        ui.W0 = Wm + (size_t)e * mat_bytes + (size_t)ui.n0 * row_bytes;
        return ui;
    }
};

constexpr int kRingStages = 4;  // weight tiles per warp in the shared-memory ring

template <bool GATEUP, bool ALIGN8>
__global__ void __launch_bounds__(256, 2) moe_stream_kernel(MoeArgs a, MoeWs w, int KS, int ncols,
                                                            float *__restrict__ outp) {
    extern __shared__ __align__(16) uint32_t sm_dyn[];
    __shared__ int s_active[257];
    __shared__ int s_off[256];
    __shared__ int s_cnt[256];
    __shared__ int s_prow[64 * 16];
    __shared__ int s_rows[8], s_exps[8], s_orow[8];
    // The gate/up GEMM needs the routing its predecessor writes.  The down GEMM's predecessor is
    // the h prep; the routing it needs was written two kernels earlier, by a grid that completed
    // before this one was launched, so the down GEMM reads it (from L2) before its programmatic
    // wait and has its first weight tiles requested by then.
    if (GATEUP) {
        pdl_wait();
        pdl_trigger();
    }
    const int P = a.M * a.topk;
    for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_active[i] = __ldcg(w.active + i);
    for (int i = threadIdx.x; i < a.E; i += blockDim.x) {
        s_off[i] = __ldcg(w.offsets + i);
        s_cnt[i] = __ldcg(w.counts + i);
    }
    if (GATEUP)
        for (int i = threadIdx.x; i < P; i += blockDim.x) s_prow[i] = w.pair_row[i];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const int K = GATEUP ? a.H : a.F;
    const PrepLayout L(K);
    const SmemAct SA(L, ncols);
    const PrepPtrs &Pp0 = GATEUP ? w.prepX : w.prepH;
    uint32_t *sm_act = sm_dyn;
    uint32_t *ring = sm_dyn + SA.words() + (size_t)warp * kRingStages * kTileWords;
    UnitMap<GATEUP> um;
    um.Nrows = GATEUP ? a.F : a.H;
    const int groups = cdiv(um.Nrows, kRowsPerCta);
    const int per_expert = (GATEUP ? 2 : 1) * groups * KS;
    um.groups = FastDiv((uint32_t)groups);
    um.KS = FastDiv((uint32_t)KS);
    um.per_expert = FastDiv((uint32_t)per_expert);
    um.ntk = L.ntk;
    um.tps = cdiv(L.ntk, KS);
    um.row_bytes = (size_t)L.nb * kBlockBytes;
    um.mat_bytes = (size_t)um.Nrows * um.row_bytes;
    um.Wg = a.Wg;
    um.Wu = a.Wu;
    um.Wd = a.Wd;
    um.active = s_active;
    const int total = s_active[a.E] * per_expert;
    const int q = cdiv(total, gridDim.x);
    const int i0 = blockIdx.x * q, i1 = min(total, i0 + q);
    const int g = lane >> 2, t = lane & 3;
    const int mats = GATEUP ? 2 : 1;
    // the ring path: whole 16-row groups, whole tiles, 16-byte aligned rows
    const bool ring_path = (um.Nrows % kRowsPerCta) == 0 && L.nb == L.ntk * kTileBlocks && (L.nb % 4) == 0;
    uint32_t scale_max = 0u;  // running max of |d|, |m| (f16x2)
    if (!GATEUP) {
        // this warp's first ring tiles into L2 (the lines each lane's copies will read)
        if (ring_path && i0 + warp < min(i1, (i0 / per_expert + 1) * per_expert)) {
            const UnitInfo ui = um(i0 + warp);
            for (int tt = ui.t0; tt < min(ui.t1, ui.t0 + kRingStages - 1); ++tt) {
                const uint8_t *p = ui.W0 + (size_t)(lane >> 1) * um.row_bytes + (size_t)tt * (kTileBlocks * kBlockBytes) +
                                   (lane & 1) * 48;
                prefetch_l2(p);
                prefetch_l2(p + 47);
            }
        }
        pdl_wait();
        pdl_trigger();
    }

    for (int seg0 = i0; seg0 < i1;) {
        // the run of units of one expert
        const int ai = seg0 / per_expert;
        const int seg1 = min(i1, (ai + 1) * per_expert);
        const int e = s_active[ai];
        const int off = s_off[e], cnt = s_cnt[e];
        for (int m0 = 0; m0 < cnt; m0 += 8) {
            const int mc = min(8, cnt - m0);
            __syncthreads();  // the previous run's warps are done with the staged operand
            if (threadIdx.x < 8) {
                const int c = threadIdx.x;
                const int r = c < mc ? (GATEUP ? s_prow[off + m0 + c] : off + m0 + c) : -1;
                s_rows[c] = r;
                s_exps[c] = r >= 0 ? Pp0.exps[r] : 0;
                // output row: the grouped position (gate/up, read by the h prep in that order)
                // or the (row, slot) index (down, read by the combine)
                s_orow[c] = c < mc ? (GATEUP ? off + m0 + c : w.slot_of[off + m0 + c]) : 0;
            }
            __syncthreads();
            stage_act_issue(sm_act, SA, Pp0, L, s_rows, mc);  // the oldest async group
            auto store_unit = [&](const UnitInfo &ui, float (&acc)[2][4]) {
                float *dst = outp + (size_t)(ui.ks * mats + ui.mat) * P * um.Nrows;
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const int c = 2 * t + (qq & 1), rr = g + 8 * (qq >> 1);
                    if (c < mc && rr < ui.rows_valid) {
                        dst[(size_t)s_orow[c] * um.Nrows + ui.n0 + rr] = ldexpf(acc[0][qq] + acc[1][qq], s_exps[c]);
                    }
                    acc[0][qq] = 0.0f;
                    acc[1][qq] = 0.0f;
                }
            };
            if (ring_path) {
                // this warp's tiles, in order: units seg0 + warp, + nwarps, ...; tiles t0..t1-1.
                // A producer cursor runs kRingStages-1 tiles ahead of the consumer.
                int pu = seg0 + warp, ptile = 0, pt1 = 0;
                const uint8_t *pW = nullptr;
                if (pu < seg1) {
                    const UnitInfo ui = um(pu);
                    ptile = ui.t0;
                    pt1 = ui.t1;
                    pW = ui.W0;
                }
                auto produce = [&](int stage) {
                    if (pu < seg1) {
                        issue_tile_cpasync(ring + stage * kTileWords, pW, um.row_bytes, ptile, lane);
                        if (++ptile >= pt1) {
                            pu += nwarps;
                            if (pu < seg1) {
                                const UnitInfo ui = um(pu);
                                ptile = ui.t0;
                                pt1 = ui.t1;
                                pW = ui.W0;
                            }
                        }
                    }
                    cp_async_commit();  // one group per slot, empty or not, keeps the count uniform
                };
#pragma unroll
                for (int sidx = 0; sidx < kRingStages - 1; ++sidx) produce(sidx);
                cp_async_wait<kRingStages - 1>();  // the activation group is done
                __syncthreads();
                int cu = seg0 + warp;
                UnitInfo cui;
                if (cu < seg1) cui = um(cu);
                int ctile = cui.t0;
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                for (int it = 0; cu < seg1; ++it) {
                    produce((it + kRingStages - 1) % kRingStages);
                    cp_async_wait<kRingStages - 1>();  // this tile's group has landed
                    __syncwarp();
                    TileRegs cur;
                    read_tile_smem(cur, ring + (it % kRingStages) * kTileWords, lane);
                    compute_tile_smem(cur, sm_act, SA, mc, ctile, lane, acc, scale_max);
                    if (++ctile >= cui.t1) {
                        store_unit(cui, acc);
                        cu += nwarps;
                        if (cu < seg1) {
                            cui = um(cu);
                            ctile = cui.t0;
                        }
                    }
                    __syncwarp();  // every lane has read this stage before a later copy refills it
                }
                cp_async_wait<0>();
            } else {
                cp_async_wait<0>();
                __syncthreads();
                for (int u = seg0 + warp; u < seg1; u += nwarps) {
                    const UnitInfo ui = um(u);
                    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    for (int tile = ui.t0; tile < ui.t1; ++tile) {
                        TileRegs b0;
                        load_tile<ALIGN8>(b0, ui.W0, um.row_bytes, ui.rows_valid, L.nb, tile, lane);
                        compute_tile_smem(b0, sm_act, SA, mc, tile, lane, acc, scale_max);
                    }
                    store_unit(ui, acc);
                }
            }
        }
        seg0 = seg1;
    }
    if (scale_mag_out_of_range(scale_max)) set_status(a.status, Q2_ERR_RANGE);
}

// Gate+up for M <= 8 activation rows and no K split: the streaming arrangement of the dense
// small-M GEMM (q2_gemm_stream_kernel) over the active experts' gate and up matrices.  One CTA of
// kGuWarps warps per SM; all M prepared X rows are staged in shared memory once per CTA (each
// expert's MMA columns are all of them, and only the rows routed to the expert are stored);
// the CTA's contiguous range of units (active expert, gate|up, 16-row group) is split evenly
// over its warps by tiles, each warp streaming its 16 x 256 tiles through its own cp.async ring.
// Compared with moe_stream_kernel there is no per-expert staging or barrier, and the smaller
// register footprint leaves room for three times the warps per scheduler.  Measured at the
// verifier shape (gate+up µs): even split, 24 warps, 3-tile rings: 55.4-55.6 (cuts on 2-tile
// steps; 56.1-56.4 on 4-tile steps); even, 28 warps (at the register limit, spilling): 64.3;
// even, 20 warps: 59.4; strided units, 28 x 3: 56.3 (24 x 3: 57.8, 28 x 4: 57.9, 32 x 3: 59.9,
// 16 x 5: 62.5); moe_stream_kernel 60.0.
constexpr int kGuWarps = 24;
constexpr int kGuRing = 3;
constexpr bool kGuEven = true;

__global__ void __launch_bounds__(kGuWarps * 32, 1) moe_gateup_stream_kernel(MoeArgs a, MoeWs w) {
    extern __shared__ __align__(16) uint32_t sm_dyn[];
    __shared__ int s_active[256];
    __shared__ int s_pos[256][8];  // grouped position of (active expert, X row), -1: not routed
    __shared__ int s_rows[8], s_exps[8];
    __shared__ int s_na;
    pdl_wait();
    pdl_trigger();
    const int M = a.M, F = a.F, P = a.M * a.topk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    if (threadIdx.x == 0) s_na = w.active[a.E];
    for (int i = threadIdx.x; i < a.E; i += blockDim.x) {
        s_active[i] = w.active[i];
#pragma unroll
        for (int c = 0; c < 8; ++c) s_pos[i][c] = -1;
    }
    if (threadIdx.x < 8) {
        s_rows[threadIdx.x] = threadIdx.x < M ? (int)threadIdx.x : 0;
        s_exps[threadIdx.x] = threadIdx.x < M ? w.prepX.exps[threadIdx.x] : 0;
    }
    __syncthreads();
    const int na = s_na;
    for (int ai = threadIdx.x; ai < na; ai += blockDim.x) {
        const int e = s_active[ai], off = w.offsets[e], cnt = w.counts[e];
        for (int c = 0; c < cnt; ++c) s_pos[ai][w.pair_row[off + c]] = off + c;
    }
    const PrepLayout L(a.H);
    const SmemAct SA(L, M);
    uint32_t *sm_act = sm_dyn;
    uint32_t *ring = sm_dyn + SA.words() + (size_t)warp * kGuRing * kTileWords;
    const size_t row_bytes = (size_t)L.nb * kBlockBytes;
    const size_t mat_bytes = (size_t)F * row_bytes;
    const int groups = F / kRowsPerCta, per_expert = 2 * groups;
    const int total = na * per_expert;
    const int q = cdiv(total, gridDim.x);
    const int u0 = blockIdx.x * q, u1 = min(total, u0 + q);
    auto unit_w = [&](int u) {
        const int ai = u / per_expert, r = u - ai * per_expert;
        const int mat = r / groups, grp = r - mat * groups;
        return (mat ? a.Wu : a.Wg) + (size_t)s_active[ai] * mat_bytes + (size_t)grp * kRowsPerCta * row_bytes;
    };
    TileCursor<kGuEven, decltype(unit_w)> pc;
    __syncthreads();  // s_pos complete
    pc.begin(u0, u1, L.ntk, kGuWarps, warp, unit_w);
#pragma unroll
    for (int sidx = 0; sidx < kGuRing - 1; ++sidx)
        pc.produce(ring + sidx * kTileWords, row_bytes, L.ntk, kGuWarps, lane, unit_w);
    stage_act_issue(sm_act, SA, w.prepX, L, s_rows, M);  // the newest group: wait for every group
    cp_async_wait<0>();
    __syncthreads();
    uint32_t scale_max = 0u;  // running max of |d|, |m| (f16x2)
    auto cols = [&](int) { return make_int2(M, 0); };
    // rows g, g+8 of the unit for X rows 2t, 2t+1, stored for the rows routed to the expert
    auto store = [&](int u, int2, const float *v) {
        const int ai = u / per_expert, r = u - ai * per_expert;
        const int mat = r / groups, grp = r - mat * groups;
        float *dst = w.h + (size_t)mat * P * F + (size_t)grp * kRowsPerCta;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            const int c = 2 * t + (qq & 1), rr = g + 8 * (qq >> 1);
            const int pos = c < M ? s_pos[ai][c] : -1;
            if (pos >= 0) dst[(size_t)pos * F + rr] = ldexpf(v[qq], s_exps[c]);
        }
    };
    float *part = reinterpret_cast<float *>(sm_dyn + SA.words() + (size_t)kGuWarps * kGuRing * kTileWords);
    stream_warp_tiles<kGuRing, kGuEven>(pc, ring, sm_act, SA, part, u0, u1, L.ntk, row_bytes, kGuWarps, warp, lane, unit_w,
                               cols, store, scale_max);
    if (scale_mag_out_of_range(scale_max)) set_status(a.status, Q2_ERR_RANGE);
}

// Down for M <= 8 and no K split, on the same streaming arrangement.  Units (active expert,
// 16-row group of H) are taken by the CTA's warps from its contiguous range; at these sizes a
// range meets at most kDnMaxExperts experts, so the CTA stages the h rows of all of their pairs
// (a window of consecutive grouped positions) once, and an expert's MMA columns are its pairs'
// columns in that window.  The routing comes from two kernels back (complete before this grid
// was launched), so the unit addresses are known and the first ring tiles are requested before
// the programmatic wait, which only the h rows need.
// Measured at the 5-row, 64-expert top-6 shape (whole verifier step, us): 20 warps -> 121.5,
// 24 -> 119.0, 28 -> 120.8; the grouped kernel it replaces -> 123.5.  Down kernel alone: strided
// units 34.5 us, the even split 38.8 (a 16-row unit here is only 8 tiles, so most units would be
// cut between warps).
constexpr int kDnWarps = 24;
constexpr bool kDnEven = false;
constexpr int kDnRing = 3;
constexpr int kDnMaxExperts = 2;

__global__ void __launch_bounds__(kDnWarps * 32, 1) moe_down_stream_kernel(MoeArgs a, MoeWs w, int win_max) {
    extern __shared__ __align__(16) uint32_t sm_dyn[];
    __shared__ int s_rows[64], s_exps[64], s_slot[64];
    // the CTA's experts (at most kDnMaxExperts): id, pair count, first column in the window
    __shared__ int s_e[kDnMaxExperts], s_cnt[kDnMaxExperts], s_col[kDnMaxExperts];
    __shared__ int s_ai0, s_pos0, s_win;
    const int H = a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const PrepLayout L(a.F);
    const size_t row_bytes = (size_t)L.nb * kBlockBytes;
    const size_t mat_bytes = (size_t)H * row_bytes;
    const int groups = H / kRowsPerCta;
    // the routing (written two kernels back), read from L2
    const int na = __ldcg(w.active + a.E);
    const int total = na * groups;
    const int q = cdiv(total, gridDim.x);
    const int u0 = blockIdx.x * q, u1 = min(total, u0 + q);
    if (threadIdx.x == 0) {
        int ai0 = 0, pos0 = 0, win = 0;
        if (u0 < u1) {
            ai0 = u0 / groups;
            const int ai1 = (u1 - 1) / groups;
            pos0 = __ldcg(w.offsets + __ldcg(w.active + ai0));
            for (int j = 0; j < kDnMaxExperts; ++j) {
                const int e = ai0 + j <= ai1 ? __ldcg(w.active + ai0 + j) : 0;
                s_e[j] = e;
                s_cnt[j] = ai0 + j <= ai1 ? __ldcg(w.counts + e) : 0;
                s_col[j] = __ldcg(w.offsets + e) - pos0;
                if (ai0 + j <= ai1) win = s_col[j] + s_cnt[j];
            }
            // a range over more experts than the window holds is refused below
            if (ai1 - ai0 >= kDnMaxExperts) win = win_max + 1;
        }
        s_ai0 = ai0;
        s_pos0 = pos0;
        s_win = win;
    }
    __syncthreads();
    const int ai0 = s_ai0;
    auto unit_w = [&](int u) {
        const int j = min(u / groups - ai0, kDnMaxExperts - 1);
        return a.Wd + (size_t)s_e[j] * mat_bytes + (size_t)(u % groups) * kRowsPerCta * row_bytes;
    };
    const SmemAct SA(L, win_max);
    uint32_t *sm_act = sm_dyn;
    uint32_t *ring = sm_dyn + SA.words() + (size_t)warp * kDnRing * kTileWords;
    const int pos0 = s_pos0, win = s_win;
    if (win > win_max) {
        // a range over more experts than the host sized the window for: refuse, no partial output
        if (threadIdx.x == 0) set_status(a.status, Q2_ERR_UNSUPPORTED);
        pdl_wait();
        pdl_trigger();
        return;
    }
    TileCursor<kDnEven, decltype(unit_w)> pc;
    pc.begin(u0, u1, L.ntk, kDnWarps, warp, unit_w);
#pragma unroll
    for (int sidx = 0; sidx < kDnRing - 1; ++sidx)
        pc.produce(ring + sidx * kTileWords, row_bytes, L.ntk, kDnWarps, lane, unit_w);
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x < win) {
        s_rows[threadIdx.x] = pos0 + threadIdx.x;
        s_exps[threadIdx.x] = w.prepH.exps[pos0 + threadIdx.x];
        s_slot[threadIdx.x] = __ldcg(w.slot_of + pos0 + threadIdx.x);
    }
    __syncthreads();
    stage_act_issue(sm_act, SA, w.prepH, L, s_rows, win);  // the newest group: wait for every group
    cp_async_wait<0>();
    __syncthreads();
    uint32_t scale_max = 0u;  // running max of |d|, |m| (f16x2)
    // an expert's MMA columns: its pairs' columns in the staged window
    auto cols = [&](int u) {
        const int j = min(u / groups - ai0, kDnMaxExperts - 1);
        return make_int2(s_cnt[j], s_col[j]);
    };
    // rows g, g+8 of the unit for the expert's pairs 2t, 2t+1, stored by (row, slot)
    auto store = [&](int u, int2 nc, const float *v) {
        float *dst = w.out + (size_t)(u % groups) * kRowsPerCta;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            const int c = 2 * t + (qq & 1), rr = g + 8 * (qq >> 1);
            if (c < nc.x) dst[(size_t)s_slot[nc.y + c] * H + rr] = ldexpf(v[qq], s_exps[nc.y + c]);
        }
    };
    float *part = reinterpret_cast<float *>(sm_dyn + SA.words() + (size_t)kDnWarps * kDnRing * kTileWords);  // even split only
    stream_warp_tiles<kDnRing, kDnEven>(pc, ring, sm_act, SA, part, u0, u1, L.ntk, row_bytes, kDnWarps, warp, lane,
                                        unit_w, cols, store, scale_max);
    if (scale_mag_out_of_range(scale_max)) set_status(a.status, Q2_ERR_RANGE);
}

__global__ void __launch_bounds__(256) moe_combine_kernel(MoeArgs a, MoeWs w, int KS) {
    pdl_wait();
    pdl_trigger();
    const int H = a.H, K = a.topk, P = a.M * a.topk;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)a.M * H;
         i += (size_t)gridDim.x * blockDim.x) {
        const int r = (int)(i / H), n = (int)(i - (size_t)r * H);
        // the down outputs are stored by (row, slot), so the gate weights and the outputs are
        // independent loads: one round trip
        float y = 0.0f;
        for (int t = 0; t < K; ++t) {
            float o = 0.0f;
            for (int ks = 0; ks < KS; ++ks) o += w.out[((size_t)ks * P + (size_t)r * K + t) * H + n];
            y = fmaf(w.gate_w[r * K + t], o, y);
        }
        a.Y[i] = y;
    }
}

namespace {
// per device: resident CTAs per SM of the four stream-kernel variants (0 = unknown) and the
// dynamic shared memory each was configured for
int g_stream_blocks[kCacheDevices][4];
size_t g_stream_smem[kCacheDevices][4];

template <bool GU, bool A8>
cudaError_t launch_stream_variant(int idx, const MoeArgs &a, const MoeWs &w, int KS, float *out, int num_sms,
                                  size_t smem, cudaStream_t s) {
    auto kern = moe_stream_kernel<GU, A8>;
    const int dv = cache_device();
    int blocks = dv >= 0 ? g_stream_blocks[dv][idx] : 0;
    if (dv < 0 || g_stream_smem[dv][idx] < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, 256, smem) != cudaSuccess || blocks <= 0)
            blocks = 1;
        if (dv >= 0) {
            g_stream_blocks[dv][idx] = blocks;
            g_stream_smem[dv][idx] = smem;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms * blocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, w, KS, min(8, a.M), out);
}

template <bool GU>
cudaError_t launch_stream(const MoeArgs &a, const MoeWs &w, int KS, float *out, int num_sms, const PrepLayout &L,
                          cudaStream_t s) {
    const size_t smem = SmemAct(L, min(8, a.M)).bytes() + (size_t)8 * kRingStages * kTileWords * 4;
    if (L.nb % 2 == 0) return launch_stream_variant<GU, true>(GU ? 0 : 2, a, w, KS, out, num_sms, smem, s);
    return launch_stream_variant<GU, false>(GU ? 1 : 3, a, w, KS, out, num_sms, smem, s);
}

size_t g_gu_smem[kCacheDevices];

cudaError_t launch_gateup_stream(const MoeArgs &a, const MoeWs &w, int num_sms, size_t smem, cudaStream_t s) {
    const int dv = cache_device();
    if (dv < 0 || g_gu_smem[dv] < smem) {
        const cudaError_t e =
            cudaFuncSetAttribute(moe_gateup_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dv >= 0) g_gu_smem[dv] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kGuWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_gateup_stream_kernel, a, w);
}

size_t g_dn_smem[kCacheDevices];

cudaError_t launch_down_stream(const MoeArgs &a, const MoeWs &w, int num_sms, int win_max, size_t smem,
                               cudaStream_t s) {
    const int dv = cache_device();
    if (dv < 0 || g_dn_smem[dv] < smem) {
        const cudaError_t e =
            cudaFuncSetAttribute(moe_down_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dv >= 0) g_dn_smem[dv] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kDnWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_down_stream_kernel, a, w, win_max);
}

// K splits so that the expected number of units is a few per resident warp.  Split ks takes
// tiles [ks * tps, min(ntk, (ks + 1) * tps)) with tps = cdiv(ntk, KS); the count is then
// reduced to cdiv(ntk, tps) so that no split is empty (the weight ring would otherwise fetch
// and multiply a tile past the end of the row for an empty split).
int choose_ks(int units_without_split, int ntk, int resident_warps) {
    int ks = 1;
    while (ks < kMaxKSplits && ks < ntk && (long long)units_without_split * ks < 2LL * resident_warps) ks *= 2;
    return cdiv(ntk, cdiv(ntk, ks));
}
}  // namespace

cudaError_t launch_moe(const MoeArgs &a, const MoeWs &w, int num_sms, cudaStream_t s) {
    const PrepLayout LX(a.H), LH(a.F);
    cudaError_t err = launch_pdl(moe_route_prep_kernel, dim3(a.M + 1), dim3(kRoutePrepThreads), s, a, w, LX);
    if (err != cudaSuccess) return err;
    const int P = a.M * a.topk;
    const int expect_active = min(a.E, P);
    const int resident_warps = num_sms * 24;
    const int ks_gu = choose_ks(expect_active * 2 * cdiv(a.F, kRowsPerCta), LX.ntk, resident_warps);
    const int ks_d = choose_ks(expect_active * cdiv(a.H, kRowsPerCta), LH.ntk, resident_warps);
    // the streaming gate+up when it applies: at most 8 X rows, no K split, whole 16-row groups and
    // whole K tiles, and the staged rows plus the rings fit in shared memory
    const size_t gu_smem = SmemAct(LX, min(8, a.M)).bytes() + (size_t)kGuWarps * (kGuRing * kTileWords + 128) * 4;
    const bool gu_stream = a.M <= 8 && ks_gu == 1 && a.F % kRowsPerCta == 0 && LX.nb == LX.ntk * kTileBlocks &&
                           LX.nb % 4 == 0 && gu_smem <= (size_t)220 * 1024;
    err = probed(kProbeMoeGateUp, s, [&] {
        return gu_stream ? launch_gateup_stream(a, w, num_sms, gu_smem, s)
                         : launch_stream<true>(a, w, ks_gu, w.h, num_sms, LX, s);
    });
    if (err != cudaSuccess) return err;
    err = launch_pdl(moe_prep_h_kernel, dim3(P), dim3(256), s, (const float *)w.h, P, a.F, ks_gu, w.prepH, LH);
    if (err != cudaSuccess) return err;
    // the streaming down GEMM when it applies: at most 8 X rows, no K split, whole groups and tiles,
    // every CTA's unit range within kDnMaxExperts experts (its staged window then holds at most
    // kDnMaxExperts x M pairs), and the window plus the rings fit in shared memory
    const int dn_units_max = expect_active * cdiv(a.H, kRowsPerCta);
    const int dn_q = cdiv(dn_units_max, num_sms);
    const int dn_win = min(P, kDnMaxExperts * a.M);
    const size_t dn_smem =
        SmemAct(LH, dn_win).bytes() + (size_t)kDnWarps * (kDnRing * kTileWords + (kDnEven ? 128 : 0)) * 4;
    const bool dn_stream = a.M <= 8 && ks_d == 1 && a.H % kRowsPerCta == 0 && LH.nb == LH.ntk * kTileBlocks &&
                           LH.nb % 4 == 0 && dn_q <= cdiv(a.H, kRowsPerCta) && dn_win <= 64 &&
                           dn_smem <= (size_t)220 * 1024;
    err = probed(kProbeMoeDown, s, [&] {
        return dn_stream ? launch_down_stream(a, w, num_sms, dn_win, dn_smem, s)
                         : launch_stream<false>(a, w, ks_d, w.out, num_sms, LH, s);
    });
    if (err != cudaSuccess) return err;
    return launch_pdl(moe_combine_kernel, dim3(max(1, min(cdiv(a.M * a.H, 256), 4 * num_sms))), dim3(256), s, a,
                      w, ks_d);
}

}  // namespace q2v
