// q2v_verify.cu -- the exact p/q rejection-sampling verify on sm_103a.
//
// What is computed ("Optimizing DeepSeek-V4-Flash on a single NVIDIA GB10/GX10 with
// DSpark speculative decoding", page 1, opening post: drafts from q, the target defines
// p, accept with probability min(1, p(x)/q(x)), replace a rejected draft from the
// positive residual; "1x Spark tuned DSpark for DeepSeek-V4-Flash ...", deep-dive, "On
// losslessness": the verify rows are the only token source, drawn with the request's own
// sampler), per session s:
//   p_i = softmax(target_i / T), q_i = softmax(draft_i / T);  accept x_i iff q_i(x_i) == 0
//   or u_acc < p_i(x_i) / q_i(x_i);  at the first rejection j draw from max(0, p_j - q_j)
//   (p_j if that is zero); if all k pass draw the extra token from p_k;  a draw returns the
//   smallest y whose cumulative mass exceeds u_fin times the total.
//
// Two tiers:
//   * small V (<= kWarpTierMaxV): one warp per session does everything in one kernel;
//   * large V: the vocabulary of each session is split into C chunks.  Kernel 1 streams
//     every row's chunk once and writes (max, sum exp) partials.  Kernel 2 combines the
//     partials, runs the accept scan, computes its chunk's residual (or bonus) mass from
//     one or two rows, and the last CTA of the session to finish (an atomic ticket; no
//     CTA ever waits on another) runs the inverse-CDF search inside the selected chunk.
// Row statistics and masses are combined across chunks in fp64; the accept ratio is
// evaluated in fp64.
#include <math.h>

#include "q2v_kernels.cuh"

namespace q2v {

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ const float *row_ptr(const PqArgs &a, int s, int r) {
    // rows 0..k: target rows; rows k+1..2k: draft rows 0..k-1
    if (r <= a.k) return a.target + ((size_t)s * (a.k + 1) + r) * a.V;
    return a.draft + ((size_t)s * a.k + (r - a.k - 1)) * a.V;
}

// Accept scan for session s, given row maxima and log2 of row sums (rows as above).
// Returns j in [0, k], or -1 if a draft token is out of range.
__device__ int accept_scan(const PqArgs &a, int s, const float *rowM, const double *rowL2Z) {
    for (int i = 0; i < a.k; ++i) {
        const int x = a.drafts[(size_t)s * a.k + i];
        if (x < 0 || x >= a.V) return -1;
    }
    for (int i = 0; i < a.k; ++i) {
        const int x = a.drafts[(size_t)s * a.k + i];
        const double tx = (double)row_ptr(a, s, i)[x], dx = (double)row_ptr(a, s, a.k + 1 + i)[x];
        const double lp = (tx - (double)rowM[i]) * a.beta64 - rowL2Z[i];
        const double lq = (dx - (double)rowM[a.k + 1 + i]) * a.beta64 - rowL2Z[a.k + 1 + i];
        const double q = exp2(lq);
        if (q == 0.0) continue;  // q(x) == 0 accepts
        const double ratio = exp2(lp) / q;
        if (!((double)a.u_acc[(size_t)s * a.k + i] < ratio)) return i;
    }
    return a.k;
}

// Weight of token y in the final draw.  mode 0: residual of row j; 1: p of row `rp`.
struct DrawRows {
    const float *t, *d;  // target row, draft row (d unused in mode 1)
    float mt, md;        // row maxima
    float lt, ld;        // log2 of row sums
    int mode;
};

__device__ __forceinline__ float draw_weight(const DrawRows &R, float beta, float xt, float xd) {
    const float p = ex2((xt - R.mt) * beta - R.lt);
    if (R.mode == 1) return p;
    const float q = ex2((xd - R.md) * beta - R.ld);
    return fmaxf(p - q, 0.0f);
}

__device__ __forceinline__ void write_tokens(const PqArgs &a, int s, int j, int y) {
    int32_t *out = a.tokens + (size_t)s * (a.k + 1);
    for (int i = 0; i <= a.k; ++i) out[i] = -1;
    if (j < 0) {
        a.n_acc[s] = -1;
        return;
    }
    for (int i = 0; i < j; ++i) out[i] = a.drafts[(size_t)s * a.k + i];
    out[j] = y;
    a.n_acc[s] = j;
}

// ===================================================================== small-V tier

constexpr int kWarpTierWarps = 8;

__global__ void __launch_bounds__(kWarpTierWarps * 32) pqv_warp_kernel(PqArgs a) {
    __shared__ float sM[kWarpTierWarps][kMaxRows];
    __shared__ double sL2Z[kWarpTierWarps][kMaxRows];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = 2 * a.k + 1;
    const float beta = a.beta;
    for (int s = blockIdx.x * kWarpTierWarps + warp; s < a.S; s += gridDim.x * kWarpTierWarps) {
        for (int r = 0; r < R; ++r) {
            const float *x = row_ptr(a, s, r);
            float m = -INFINITY, z = 0.0f;
            for (int y = lane; y < a.V; y += 32) {
                const float v = x[y];
                if (v > m) {
                    z = z * ex2((m - v) * beta) + 1.0f;
                    m = v;
                } else if (v > -INFINITY) {
                    z += ex2((v - m) * beta);
                }
            }
            const float M = warp_max_f(m);
            double zz = (m > -INFINITY) ? (double)z * (double)ex2((m - M) * beta) : 0.0;
            zz = warp_sum_d(zz);
            if (lane == 0) {
                sM[warp][r] = M;
                sL2Z[warp][r] = log2(zz);
            }
        }
        __syncwarp();
        int j = 0;
        if (lane == 0) j = accept_scan(a, s, sM[warp], sL2Z[warp]);
        j = __shfl_sync(0xffffffffu, j, 0);
        if (a.probs) {
            for (int r = 0; r < R; ++r) {
                const float *x = row_ptr(a, s, r);
                float *o = a.probs + ((size_t)s * R + r) * a.V;
                const float M = sM[warp][r], L2 = (float)sL2Z[warp][r];
                for (int y = lane; y < a.V; y += 32) o[y] = ex2((x[y] - M) * beta - L2);
            }
        }
        if (j < 0) {
            if (lane == 0) {
                set_status(a.status, Q2_ERR_BAD_TOKEN);
                write_tokens(a, s, -1, -1);
            }
            __syncwarp();
            continue;
        }
        DrawRows D;
        const int jr = j;  // target row of the draw
        D.t = row_ptr(a, s, jr);
        D.mt = sM[warp][jr];
        D.lt = (float)sL2Z[warp][jr];
        if (j < a.k) {
            D.d = row_ptr(a, s, a.k + 1 + j);
            D.md = sM[warp][a.k + 1 + j];
            D.ld = (float)sL2Z[warp][a.k + 1 + j];
            D.mode = 0;
        } else {
            D.d = D.t;
            D.md = D.mt;
            D.ld = D.lt;
            D.mode = 1;
        }
        // pass 1: total mass (chunks of 32 scanned exactly as in pass 2)
        double total = 0.0;
        for (int pass = 0; pass < 2; ++pass) {
            total = 0.0;
            for (int base = 0; base < a.V; base += 32) {
                const int y = base + lane;
                float w = 0.0f;
                if (y < a.V) w = draw_weight(D, beta, D.t[y], D.d[y]);
                float incl = w;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float n = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += n;
                }
                total += (double)__shfl_sync(0xffffffffu, incl, 31);
            }
            if (total > 0.0 || D.mode == 1) break;
            D.mode = 1;  // zero residual mass: draw from p_j
        }
        const double target = (double)a.u_fin[s] * total;
        double carry = 0.0;
        int y_sel = -1, last_pos = -1;
        for (int base = 0; base < a.V && y_sel < 0; base += 32) {
            const int y = base + lane;
            float w = 0.0f;
            if (y < a.V) w = draw_weight(D, beta, D.t[y], D.d[y]);
            float incl = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, w > 0.0f && carry + (double)incl > target);
            const unsigned pos = __ballot_sync(0xffffffffu, w > 0.0f);
            if (pos) last_pos = base + 31 - __clz(pos);
            if (hit) y_sel = base + __ffs(hit) - 1;
            carry += (double)__shfl_sync(0xffffffffu, incl, 31);
        }
        if (y_sel < 0) y_sel = last_pos;
        if (lane == 0) write_tokens(a, s, j, y_sel);
        __syncwarp();
    }
}

// ===================================================================== large-V tier

// Kernel 1: (max, sum 2^((x-max) beta)) of every row's chunk.  grid (C, S); warp w takes
// rows w, w + nwarps, ...
template <bool VEC>
__global__ void __launch_bounds__(512) pqv_stats_kernel(PqArgs a, PqSplit sp) {
    const int c = blockIdx.x, s = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const int R = 2 * a.k + 1;
    const int c0 = c * sp.L, c1 = min(a.V, c0 + sp.L);
    const float beta = a.beta;
    if (c == 0 && threadIdx.x == 0) sp.tickets[s] = 0u;
    for (int r = warp; r < R; r += nwarps) {
        const float *x = row_ptr(a, s, r);
        float m = -INFINITY, z = 0.0f;
        if (VEC) {
            const float4 *x4 = reinterpret_cast<const float4 *>(x + c0);
            const int n4 = (c1 - c0) >> 2;
            constexpr int U = 4;
            for (int base = 0; base < n4; base += 32 * U) {
                float4 v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = base + u * 32 + lane;
                    v[u] = i < n4 ? __ldcs(x4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                }
                float bm = m;
#pragma unroll
                for (int u = 0; u < U; ++u) bm = fmaxf(bm, fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)));
                if (bm > -INFINITY) {
                    float acc = (m > -INFINITY) ? z * ex2((m - bm) * beta) : 0.0f;
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        acc += ex2((v[u].x - bm) * beta) + ex2((v[u].y - bm) * beta);
                        acc += ex2((v[u].z - bm) * beta) + ex2((v[u].w - bm) * beta);
                    }
                    z = acc;
                    m = bm;
                }
            }
        } else {
            for (int y = c0 + lane; y < c1; y += 32) {
                const float v = x[y];
                if (v > m) {
                    z = z * ex2((m - v) * beta) + 1.0f;
                    m = v;
                } else if (v > -INFINITY) {
                    z += ex2((v - m) * beta);
                }
            }
        }
        const float M = warp_max_f(m);
        float zz = (m > -INFINITY) ? z * ex2((m - M) * beta) : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) zz += __shfl_xor_sync(0xffffffffu, zz, o);
        if (lane == 0) {
            float2 *st = reinterpret_cast<float2 *>(sp.stats) + ((size_t)s * R + r) * sp.C + c;
            *st = make_float2(M, zz);
        }
    }
}

__device__ __forceinline__ double block_sum_d(double v, double *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum_d(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    double t = 0.0;
    for (int w = 0; w < nw; ++w) t += scratch[w];
    return t;
}

// Kernel 2: combine, accept scan, chunk masses, last-arriver inverse-CDF search.
template <bool VEC>
__global__ void __launch_bounds__(256) pqv_verify_kernel(PqArgs a, PqSplit sp) {
    __shared__ float rowM[kMaxRows];
    __shared__ double rowL2Z[kMaxRows];
    __shared__ double scratch[32];
    __shared__ int s_j, s_last, s_y, s_lastpos;
    const int c = blockIdx.x, s = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
    const int R = 2 * a.k + 1;
    const float beta = a.beta;
    const int c0 = c * sp.L, c1 = min(a.V, c0 + sp.L);

    // 1. row statistics from the chunk partials (fp64 sums)
    for (int r = warp; r < R; r += nwarps) {
        const float2 *st = reinterpret_cast<const float2 *>(sp.stats) + ((size_t)s * R + r) * sp.C;
        float m = -INFINITY;
        for (int cc = lane; cc < sp.C; cc += 32) m = fmaxf(m, st[cc].x);
        m = warp_max_f(m);
        double z = 0.0;
        for (int cc = lane; cc < sp.C; cc += 32) {
            const float2 v = st[cc];
            if (v.x > -INFINITY) z += (double)v.y * exp2((double)(v.x - m) * a.beta64);
        }
        z = warp_sum_d(z);
        if (lane == 0) {
            rowM[r] = m;
            rowL2Z[r] = log2(z);
        }
    }
    __syncthreads();
    // 2. accept scan
    if (tid == 0) s_j = accept_scan(a, s, rowM, rowL2Z);
    __syncthreads();
    const int j = s_j;
    // optional probabilities of every row of this chunk
    if (a.probs) {
        for (int r = 0; r < R; ++r) {
            const float *x = row_ptr(a, s, r);
            float *o = a.probs + ((size_t)s * R + r) * a.V;
            const float M = rowM[r], L2 = (float)rowL2Z[r];
            for (int y = c0 + tid; y < c1; y += blockDim.x) o[y] = ex2((x[y] - M) * beta - L2);
        }
    }
    if (j < 0) {
        if (c == 0 && tid == 0) {
            set_status(a.status, Q2_ERR_BAD_TOKEN);
            write_tokens(a, s, -1, -1);
        }
        return;
    }
    DrawRows D;
    D.t = row_ptr(a, s, j);
    D.mt = rowM[j];
    D.lt = (float)rowL2Z[j];
    if (j < a.k) {
        D.d = row_ptr(a, s, a.k + 1 + j);
        D.md = rowM[a.k + 1 + j];
        D.ld = (float)rowL2Z[a.k + 1 + j];
        D.mode = 0;
    } else {
        D.d = D.t;
        D.md = D.mt;
        D.ld = D.lt;
        D.mode = 1;
    }
    // 3. this chunk's draw mass (and p_j mass for the zero-residual fallback)
    float wsum = 0.0f, psum = 0.0f;
    if (VEC) {
        const float4 *t4 = reinterpret_cast<const float4 *>(D.t + c0);
        const float4 *d4 = reinterpret_cast<const float4 *>(D.d + c0);
        const int n4 = (c1 - c0) >> 2;
        for (int i = tid; i < n4; i += blockDim.x) {
            const float4 xt = t4[i];
            const float4 xd = (D.mode == 0) ? d4[i] : xt;
            wsum += draw_weight(D, beta, xt.x, xd.x) + draw_weight(D, beta, xt.y, xd.y) +
                    draw_weight(D, beta, xt.z, xd.z) + draw_weight(D, beta, xt.w, xd.w);
            if (D.mode == 0)
                psum += ex2((xt.x - D.mt) * beta - D.lt) + ex2((xt.y - D.mt) * beta - D.lt) +
                        ex2((xt.z - D.mt) * beta - D.lt) + ex2((xt.w - D.mt) * beta - D.lt);
        }
    } else {
        for (int y = c0 + tid; y < c1; y += blockDim.x) {
            const float xt = D.t[y];
            const float xd = (D.mode == 0) ? D.d[y] : xt;
            wsum += draw_weight(D, beta, xt, xd);
            if (D.mode == 0) psum += ex2((xt - D.mt) * beta - D.lt);
        }
    }
    const double wtot = block_sum_d((double)wsum, scratch);
    const double ptot = block_sum_d((double)psum, scratch);
    if (tid == 0) {
        sp.mass[(size_t)s * sp.C + c] = wtot;
        sp.pmass[(size_t)s * sp.C + c] = ptot;
        __threadfence();
        const unsigned ticket = atomicAdd(sp.tickets + s, 1u);
        s_last = (ticket == (unsigned)(sp.C - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // 4. last CTA of the session: pick the chunk, then the token inside it
    __shared__ double s_prefix, s_target;
    __shared__ int s_chunk, s_mode;
    if (tid == 0) {
        const volatile double *mm = sp.mass + (size_t)s * sp.C;
        int mode = D.mode;
        double total = 0.0;
        for (int cc = 0; cc < sp.C; ++cc) total += mm[cc];
        if (mode == 0 && !(total > 0.0)) {  // zero residual mass: draw from p_j
            mode = 1;
            mm = sp.pmass + (size_t)s * sp.C;
            total = 0.0;
            for (int cc = 0; cc < sp.C; ++cc) total += mm[cc];
        }
        const double target = (double)a.u_fin[s] * total;
        double prefix = 0.0, last_prefix = 0.0;
        int chunk = -1, last_nz = -1;
        for (int cc = 0; cc < sp.C; ++cc) {
            const double mc = mm[cc];
            if (mc > 0.0) {
                last_nz = cc;
                last_prefix = prefix;
                if (prefix + mc > target) {
                    chunk = cc;
                    break;
                }
            }
            prefix += mc;
        }
        if (chunk < 0) {  // rounding put the target past the end: the last chunk with mass
            chunk = last_nz;
            prefix = last_prefix;
        }
        s_chunk = chunk;
        s_prefix = prefix;
        s_target = target;
        s_mode = mode;
        s_y = 0x7fffffff;
        s_lastpos = -1;
    }
    __syncthreads();
    D.mode = s_mode;
    const int cs = s_chunk;
    if (cs >= 0) {
        const double tgt = s_target;
        const int y0 = cs * sp.L, y1 = min(a.V, y0 + sp.L);
        double carry = s_prefix;
        for (int base = y0; base < y1; base += blockDim.x) {
            const int y = base + tid;
            float w = 0.0f;
            if (y < y1) w = draw_weight(D, beta, D.t[y], D.d[y]);
            // block inclusive scan of w in fp64 (thread order is token order)
            double incl = (double)w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            if (lane == 31) scratch[warp] = incl;
            __syncthreads();
            double woff = 0.0, tile_total = 0.0;
            for (int ww = 0; ww < nwarps; ++ww) {
                if (ww < warp) woff += scratch[ww];
                tile_total += scratch[ww];
            }
            if (w > 0.0f) {
                atomicMax(&s_lastpos, y);
                if (carry + woff + incl > tgt) atomicMin(&s_y, y);
            }
            __syncthreads();
            if (s_y != 0x7fffffff) break;
            carry += tile_total;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int y = s_y;
        if (y == 0x7fffffff) y = s_lastpos;
        write_tokens(a, s, j, y);
    }
}

cudaError_t launch_pq_verify(const PqArgs &a, const PqSplit &sp, bool warp_tier, int num_sms, cudaStream_t st) {
    if (warp_tier) {
        const int blocks = max(1, min(cdiv(a.S, kWarpTierWarps), num_sms * 8));
        pqv_warp_kernel<<<blocks, kWarpTierWarps * 32, 0, st>>>(a);
        return cudaGetLastError();
    }
    const bool vec = (a.V % 4) == 0 && (sp.L % 4) == 0;
    const int R = 2 * a.k + 1;
    const dim3 grid(sp.C, a.S);
    const int warps1 = min(R, 16);
    if (vec) {
        pqv_stats_kernel<true><<<grid, warps1 * 32, 0, st>>>(a, sp);
        pqv_verify_kernel<true><<<grid, 256, 0, st>>>(a, sp);
    } else {
        pqv_stats_kernel<false><<<grid, warps1 * 32, 0, st>>>(a, sp);
        pqv_verify_kernel<false><<<grid, 256, 0, st>>>(a, sp);
    }
    return cudaGetLastError();
}

}  // namespace q2v
