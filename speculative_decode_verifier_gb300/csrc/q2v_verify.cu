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
//   * small V (<= kWarpTierMaxV): one warp (V <= 512) or one CTA per session does everything
//     in one kernel;
//   * large V: the vocabulary of each session is split into C chunks.  Kernel 1 streams
//     every row's chunk once (leaving the rows in L2) and writes (max, sum exp) partials;
//     it also gathers both logits at each draft token.  Kernel 2 combines the partials,
//     runs the accept scan, computes its chunk's residual (or bonus) mass from one or two
//     rows, and the last CTA of the session to finish (an atomic ticket; no CTA ever waits
//     on another) runs the inverse-CDF search with all of its threads: a block-wide scan
//     over the session's segment masses, then one over the tokens of the chosen segment.
//
// Arithmetic is fp32 throughout (exponentials on the SFU via ex2.approx): reductions are
// trees, and the running cumulative sums of the draws are compensated (a hi + lo pair
// updated with an exact two-sum), so the CDF carries the accuracy of a much wider type
// at fp32 speed.  The accept ratio is formed in the log2 domain.
#include <math.h>

#include "q2v_kernels.cuh"

namespace q2v {

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Inclusive warp scan (lane order), fp32.
__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// A compensated running sum: hi + lo, each addition exact up to the final rounding of lo
// (Knuth's two-sum of hi and the addend).
struct CSum {
    float hi = 0.0f, lo = 0.0f;
    __device__ __forceinline__ void add(float b) {
        const float s = hi + b;
        const float bb = s - hi;
        const float err = (hi - (s - bb)) + (b - bb);
        hi = s;
        lo += err;
    }
    // carry + x compared with the target, without losing the low part
    __device__ __forceinline__ bool exceeds(float x, float target) const { return hi + (lo + x) > target; }
    __device__ __forceinline__ float value() const { return hi + lo; }
};

// a + b for two compensated sums: two-sum of the high parts, low parts added.
__device__ __forceinline__ CSum csum_plus(CSum a, const CSum &b) {
    a.add(b.hi);
    a.lo += b.lo;
    return a;
}

// Block-wide scan of compensated values in thread order (blockDim.x a multiple of 32, at most
// 1024): returns this thread's exclusive prefix and sets `total`.  `scratch` holds 64 floats;
// the call synchronises the block once and leaves scratch free again only after the next
// barrier.
__device__ __forceinline__ CSum block_excl_scan(const CSum &v, float *scratch, CSum &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    CSum inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        CSum n;
        n.hi = __shfl_up_sync(0xffffffffu, inc.hi, o);
        n.lo = __shfl_up_sync(0xffffffffu, inc.lo, o);
        if (lane >= o) inc = csum_plus(n, inc);
    }
    CSum ex;
    ex.hi = __shfl_up_sync(0xffffffffu, inc.hi, 1);
    ex.lo = __shfl_up_sync(0xffffffffu, inc.lo, 1);
    if (lane == 0) ex = CSum();
    if (lane == 31) {
        scratch[2 * warp] = inc.hi;
        scratch[2 * warp + 1] = inc.lo;
    }
    __syncthreads();
    CSum base, tot;
    for (int w = 0; w < nw; ++w) {
        CSum x;
        x.hi = scratch[2 * w];
        x.lo = scratch[2 * w + 1];
        if (w < warp) base = csum_plus(base, x);
        tot = csum_plus(tot, x);
    }
    total = tot;
    return csum_plus(base, ex);
}

__device__ __forceinline__ const float *row_ptr(const PqArgs &a, int s, int r) {
    // rows 0..k: target rows; rows k+1..2k: draft rows 0..k-1
    if (r <= a.k) return a.target + ((size_t)s * (a.k + 1) + r) * a.V;
    return a.draft + ((size_t)s * a.k + (r - a.k - 1)) * a.V;
}

// Accept scan for session s, given row maxima and log2 of row sums (rows as above).
// The ratio p/q is formed in the log2 domain: ratio = 2^(lp - lq) with
// lp = (t(x) - max_t) * beta - log2 Z_t (likewise lq), so neither probability underflows on
// its own; q(x) == 0 exactly (a -inf draft logit) accepts.  Returns j in [0, k], or -1 if
// a draft token is out of range.
__device__ int accept_scan(const PqArgs &a, int s, float beta, const float *rowM, const float *rowL2Z) {
    for (int i = 0; i < a.k; ++i) {
        const int x = a.drafts[(size_t)s * a.k + i];
        if (x < 0 || x >= a.V) return -1;
    }
    for (int i = 0; i < a.k; ++i) {
        const int x = a.drafts[(size_t)s * a.k + i];
        const float tx = row_ptr(a, s, i)[x], dx = row_ptr(a, s, a.k + 1 + i)[x];
        if (dx == -INFINITY) continue;  // q(x) == 0 accepts
        const float lp = (tx - rowM[i]) * beta - rowL2Z[i];
        const float lq = (dx - rowM[a.k + 1 + i]) * beta - rowL2Z[a.k + 1 + i];
        const float ratio = ex2(lp - lq);
        if (!(a.u_acc[(size_t)s * a.k + i] < ratio)) return i;
    }
    return a.k;
}

// How session s is verified: 1 = sampling with *beta = log2(e) / T, 0 = greedy (T = 0),
// -1 = a negative or non-finite temperature (the session is marked bad).
__device__ __forceinline__ int session_mode(const PqArgs &a, int s, float *beta) {
    if (!a.temps) {
        *beta = a.beta;
        return 1;
    }
    const float T = a.temps[s];
    *beta = 0.0f;
    if (T == 0.0f) return 0;
    if (!(T > 0.0f) || !(T < INFINITY)) return -1;
    *beta = (float)(1.4426950408889634 / (double)T);  // as the host computes it for pq_verify
    return 1;
}

// The greedy choice: the largest value, ties to the lower token index.  (m, i) pairs from
// lanes or chunks combine with better_arg.
__device__ __forceinline__ bool better_arg(float m2, int i2, float m1, int i1) {
    return m2 > m1 || (m2 == m1 && i2 < i1);
}
__device__ __forceinline__ void warp_argmax(float &m, int &i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
        if (better_arg(m2, i2, m, i)) {
            m = m2;
            i = i2;
        }
    }
}
// A lane's (max, first index of it) over y = y0 + lane, y0 + lane + 32, ... < y1.
__device__ __forceinline__ void lane_argmax(const float *x, int y0, int y1, int lane, float &m, int &i) {
    m = -INFINITY;
    i = 0x7FFFFFFF;
    for (int y = y0 + lane; y < y1; y += 32) {
        const float v = x[y];
        if (i == 0x7FFFFFFF || v > m) {
            m = v;
            i = y;
        }
    }
}

// The greedy verify's outcome from the target rows' argmaxes am[0..k]: j = the first draft
// that is not argmax p_i (k if none), the token after it argmax p_j.  -1: a bad draft token.
__device__ __forceinline__ int greedy_scan(const PqArgs &a, int s, const int *am) {
    for (int i = 0; i < a.k; ++i) {
        const int x = a.drafts[(size_t)s * a.k + i];
        if (x < 0 || x >= a.V) return -1;
    }
    for (int i = 0; i < a.k; ++i)
        if (a.drafts[(size_t)s * a.k + i] != am[i]) return i;
    return a.k;
}

// Weight of token y in the final draw.  mode 0: residual max(0, p_j - q_j); 1: p of row t.
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

__device__ __forceinline__ DrawRows draw_rows(const PqArgs &a, int s, int j, const float *rowM,
                                              const float *rowL2Z) {
    DrawRows D;
    D.t = row_ptr(a, s, j);
    D.mt = rowM[j];
    D.lt = rowL2Z[j];
    if (j < a.k) {
        D.d = row_ptr(a, s, a.k + 1 + j);
        D.md = rowM[a.k + 1 + j];
        D.ld = rowL2Z[a.k + 1 + j];
        D.mode = 0;
    } else {
        D.d = D.t;
        D.md = D.mt;
        D.ld = D.lt;
        D.mode = 1;
    }
    return D;
}

// ===================================================================== small-V tier
//
// V <= kWarpTierMaxV: a group of GW warps per session does everything in one kernel (one warp
// per session for V <= kSmallWarpMaxV, sixteen warps -- the whole CTA -- above).  The accept
// scan's inputs (draft tokens, uniforms, both logits at each draft) are requested first, so
// they arrive while the row statistics stream.  Every load is
// issued in batches before any of it is used: a row's statistics take one batch per 32 x 32
// floats (float4 loads) or 32 x 16 (scalar), the accept scan is lane-parallel (one lane per
// draft, a ballot finds the first rejection), and the draw gives each thread a contiguous run
// of at most 16 tokens whose logits it loads at once, then one compensated group-wide scan
// finds the run, and the run's owner the token.

constexpr int kSmallWarpMaxV = 512;   // one warp per session up to this V
constexpr int kSmallMaxRun = 16;      // tokens per lane in the draw, one warp per session
constexpr int kSegWarpRun = 8;       // a large-V draw segment of <= 32 x this many tokens is walked by one warp

// (max, log2 sum 2^((x - max) beta)) of one row of V logits, by one warp; loads in batches.
template <bool VEC>
__device__ __forceinline__ void warp_row_stats(const float *__restrict__ x, int V, float beta, int lane, float &M,
                                               float &L2Z) {
    float m = -INFINITY, z = 0.0f;
    constexpr int U = VEC ? 8 : 16;
    constexpr int W = VEC ? 4 : 1;  // floats per load
    for (int base = 0; base < V; base += 32 * U * W) {
        float v[U * W];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + (u * 32 + lane) * W;
            if (VEC) {
                const float4 q = i < V ? __ldg(reinterpret_cast<const float4 *>(x + i))
                                       : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                v[4 * u] = q.x; v[4 * u + 1] = q.y; v[4 * u + 2] = q.z; v[4 * u + 3] = q.w;
            } else {
                v[u] = i < V ? __ldg(x + i) : -INFINITY;
            }
        }
        float bm = m;
#pragma unroll
        for (int u = 0; u < U * W; ++u) bm = fmaxf(bm, v[u]);
        if (bm > -INFINITY) {
            float acc = (m > -INFINITY) ? z * ex2((m - bm) * beta) : 0.0f;
#pragma unroll
            for (int u = 0; u < U * W; ++u) acc += ex2((v[u] - bm) * beta);  // -inf entries add 0
            z = acc;
            m = bm;
        }
    }
    M = warp_max(m);
    const float zz = warp_sum((m > -INFINITY) ? z * ex2((m - M) * beta) : 0.0f);
    L2Z = log2f(zz);
}

// (max, first index of it) of one row by one warp; loads in batches of 16 per lane.
__device__ __forceinline__ int warp_row_argmax(const float *__restrict__ x, int V, int lane) {
    float m = -INFINITY;
    int i = 0x7FFFFFFF;
    for (int base = 0; base < V; base += 32 * 16) {
        float v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int y = base + u * 32 + lane;
            v[u] = y < V ? __ldg(x + y) : -INFINITY;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int y = base + u * 32 + lane;
            if (y < V && (i == 0x7FFFFFFF || v[u] > m)) {
                m = v[u];
                i = y;
            }
        }
    }
    warp_argmax(m, i);
    return i;
}

// Compensated exclusive scan over the threads of one warp (lane order); `total` gets the sum.
__device__ __forceinline__ CSum warp_excl_scan_c(const CSum &v, int lane, CSum &total) {
    CSum inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        CSum n;
        n.hi = __shfl_up_sync(0xffffffffu, inc.hi, o);
        n.lo = __shfl_up_sync(0xffffffffu, inc.lo, o);
        if (lane >= o) inc = csum_plus(n, inc);
    }
    CSum ex;
    ex.hi = __shfl_up_sync(0xffffffffu, inc.hi, 1);
    ex.lo = __shfl_up_sync(0xffffffffu, inc.lo, 1);
    if (lane == 0) ex = CSum();
    total.hi = __shfl_sync(0xffffffffu, inc.hi, 31);
    total.lo = __shfl_sync(0xffffffffu, inc.lo, 31);
    return ex;
}

constexpr int kSmallCtaWarps = 16;  // warps of the CTA-per-session variant

template <int GW>
struct SmallShared {
    float M[GW == 1 ? 8 : 1][kMaxRows];
    float L2Z[GW == 1 ? 8 : 1][kMaxRows];
    int arg[GW == 1 ? 8 : 1][kMaxRows];
    int j[GW == 1 ? 8 : 1];
    float scan[64];
    int first, lastpos;
};

template <int GW>
__device__ __forceinline__ void group_sync() {
    if (GW == 1) __syncwarp();
    else __syncthreads();
}

template <int GW, bool VEC>
__global__ void __launch_bounds__(GW == 1 ? 256 : 32 * GW) pqv_small_kernel(PqArgs a) {
    __shared__ SmallShared<GW> sh;
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gi = GW == 1 ? warp : 0;                      // this group's slot in shared memory
    const int gt = GW == 1 ? lane : (int)threadIdx.x;        // thread index inside the group
    const int gwarp = GW == 1 ? 0 : warp;                    // warp index inside the group
    const int gthreads = 32 * GW;
    const int s = GW == 1 ? (int)blockIdx.x * 8 + warp : (int)blockIdx.x;
    if (s >= a.S) return;  // whole groups only: no group barrier is skipped by part of a group
    const int R = 2 * a.k + 1;
    float beta;
    const int smode = session_mode(a, s, &beta);
    if (smode < 0) {
        if (gt == 0) {
            set_status(a.status, Q2_ERR_BAD_TEMPERATURE);
            write_tokens(a, s, -1, -1);
        }
        return;
    }
    if (smode == 0) {
        // greedy: the argmax of every row (the target rows decide; all rows for probs)
        for (int r = gwarp; r < R; r += GW) {
            const int i = warp_row_argmax(row_ptr(a, s, r), a.V, lane);
            if (lane == 0) sh.arg[gi][r] = i;
        }
        group_sync<GW>();
        if (a.probs)
            for (int r = 0; r < R; ++r) {
                float *o = a.probs + ((size_t)s * R + r) * a.V;
                const int am = sh.arg[gi][r];
                for (int y = gt; y < a.V; y += gthreads) o[y] = (y == am) ? 1.0f : 0.0f;
            }
        if (gt == 0) {
            const int j = greedy_scan(a, s, sh.arg[gi]);
            if (j < 0) set_status(a.status, Q2_ERR_BAD_TOKEN);
            write_tokens(a, s, j, j < 0 ? -1 : sh.arg[gi][j]);
        }
        return;
    }
    // 0. the accept scan's inputs, requested before the statistics (lane i: draft i)
    int xv = 0;
    float tx = 0.0f, dx = 0.0f, uv = 0.0f;
    if (gwarp == 0 && lane < a.k) {
        xv = a.drafts[(size_t)s * a.k + lane];
        uv = a.u_acc[(size_t)s * a.k + lane];
        if (xv >= 0 && xv < a.V) {
            tx = row_ptr(a, s, lane)[xv];
            dx = row_ptr(a, s, a.k + 1 + lane)[xv];
        }
    }
    // 1. every row's statistics (warps of the group take rows in turn)
    for (int r = gwarp; r < R; r += GW) {
        float M, L2;
        warp_row_stats<VEC>(row_ptr(a, s, r), a.V, beta, lane, M, L2);
        if (lane == 0) {
            sh.M[gi][r] = M;
            sh.L2Z[gi][r] = L2;
        }
    }
    group_sync<GW>();
    // 2. accept scan: lane i evaluates draft i, a ballot finds the first rejection
    if (gwarp == 0) {
        bool bad = false, rej = false;
        if (lane < a.k) {
            if (xv < 0 || xv >= a.V) {
                bad = true;
            } else if (dx != -INFINITY) {  // q(x) == 0 accepts
                const float lp = (tx - sh.M[gi][lane]) * beta - sh.L2Z[gi][lane];
                const float lq = (dx - sh.M[gi][a.k + 1 + lane]) * beta - sh.L2Z[gi][a.k + 1 + lane];
                rej = !(uv < ex2(lp - lq));
            }
        }
        const unsigned badm = __ballot_sync(0xffffffffu, bad), rejm = __ballot_sync(0xffffffffu, rej);
        if (lane == 0) sh.j[gi] = badm ? -1 : (rejm ? __ffs(rejm) - 1 : a.k);
    }
    group_sync<GW>();
    const int j = sh.j[gi];
    if (a.probs)
        for (int r = 0; r < R; ++r) {
            const float *x = row_ptr(a, s, r);
            float *o = a.probs + ((size_t)s * R + r) * a.V;
            const float M = sh.M[gi][r], L2 = sh.L2Z[gi][r];
            for (int y = gt; y < a.V; y += gthreads) o[y] = ex2((x[y] - M) * beta - L2);
        }
    if (j < 0) {
        if (gt == 0) {
            set_status(a.status, Q2_ERR_BAD_TOKEN);
            write_tokens(a, s, -1, -1);
        }
        return;
    }
    // 3. the draw: this thread's run of tokens, weights in registers
    DrawRows D = draw_rows(a, s, j, sh.M[gi], sh.L2Z[gi]);
    constexpr int MR = GW == 1 ? kSmallMaxRun : kWarpTierMaxV / (32 * GW);  // tokens per thread, at most
    const int run = cdiv(a.V, gthreads);  // <= MR
    const int y0 = min(a.V, gt * run), y1 = min(a.V, y0 + run);
    float xt[MR], xd[MR], w[MR];
#pragma unroll
    for (int u = 0; u < MR; ++u) {
        const int y = y0 + u;
        xt[u] = y < y1 ? D.t[y] : 0.0f;
        xd[u] = (y < y1 && D.mode == 0) ? D.d[y] : xt[u];
    }
    CSum own, excl, tot;
    int mode = D.mode;
    for (int pass = 0; pass < 2; ++pass) {  // pass 1 only when the residual has no mass
        D.mode = mode;
        own = CSum();
#pragma unroll
        for (int u = 0; u < MR; ++u) {
            w[u] = y0 + u < y1 ? draw_weight(D, beta, xt[u], xd[u]) : 0.0f;
            if (y0 + u < y1) own.add(w[u]);
        }
        if (GW == 1) {
            excl = warp_excl_scan_c(own, lane, tot);
        } else {
            group_sync<GW>();  // sh.scan is free again
            excl = block_excl_scan(own, sh.scan, tot);
        }
        if (mode == 1 || tot.hi > 0.0f) break;
        mode = 1;  // zero residual mass: draw from p_j
    }
    const float target = a.u_fin[s] * (tot.hi + tot.lo);
    const float own_m = own.hi + own.lo;
    const bool crosses = own_m > 0.0f && excl.exceeds(own_m, target);
    int first, lastpos;
    if (GW == 1) {
        const unsigned cm = __ballot_sync(0xffffffffu, crosses), pm = __ballot_sync(0xffffffffu, own_m > 0.0f);
        first = cm ? __ffs(cm) - 1 : gthreads;
        lastpos = pm ? 31 - __clz(pm) : -1;
    } else {
        if (gt == 0) {
            sh.first = gthreads;
            sh.lastpos = -1;
        }
        __syncthreads();
        if (own_m > 0.0f) atomicMax(&sh.lastpos, gt);
        if (crosses) atomicMin(&sh.first, gt);
        __syncthreads();
        first = sh.first;
        lastpos = sh.lastpos;
    }
    const int owner = first < gthreads ? first : lastpos;
    if (owner < 0) {
        if (gt == 0) write_tokens(a, s, j, -1);
        return;
    }
    if (gt == owner) {
        // the first token of this run whose cumulative mass passes the target (else its last
        // token with mass)
        CSum pre = excl;
        int found = -1, last_nz = -1;
#pragma unroll
        for (int u = 0; u < MR; ++u) {
            if (found < 0 && y0 + u < y1 && w[u] > 0.0f) {
                last_nz = y0 + u;
                if (first < gthreads && pre.exceeds(w[u], target)) found = y0 + u;
            }
            if (found < 0) pre.add(w[u]);
        }
        write_tokens(a, s, j, found >= 0 ? found : last_nz);
    }
}

// Level 1 of a large-V draw: the segment (one of the session's nseg segment masses) holding
// the crossing of u_fin * total.  The whole block stages the masses in shared memory (`sm`,
// nseg floats; the p_j masses in the zero-residual fallback); thread i sums the contiguous run
// of cdiv(nseg, threads) entries it owns, a compensated block scan gives each thread its prefix
// and every thread the total, and the first thread whose run crosses walks it (if rounding puts
// the target past the end, the last entry with mass is taken).  Returns, in every thread, the
// entry (-1: no mass at all), the compensated prefix before it, the target and the mode
// (0 residual, 1 p_j).  `scan` is block_excl_scan's scratch; s_first and s_lastpos are shared ints.
struct SegPick {
    int ent, mode;
    float pre_hi, pre_lo, target;
};

__device__ __forceinline__ SegPick pick_segment(const float *mass, const float *pmass, int nseg, int mode0, float u,
                                                float *sm, float *scan, int *s_first, int *s_lastpos,
                                                SegPick *shared_out) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int q = cdiv(nseg, nt);
    const int e0 = min(nseg, tid * q), e1 = min(nseg, e0 + q);
    CSum own, excl, tot;
    int mode = mode0;
    for (int pass = 0; pass < 2; ++pass) {  // pass 1 only when the residual has no mass
        const float *wsrc = pass == 0 ? mass : pmass;
        // up to 8 loads per thread in flight before any is stored
        for (int e = tid; e < nseg; e += 8 * nt) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = e + k * nt < nseg ? __ldcg(wsrc + e + k * nt) : 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (e + k * nt < nseg) sm[e + k * nt] = v[k];
        }
        __syncthreads();
        own = CSum();
        for (int e = e0; e < e1; ++e) own.add(sm[e]);
        excl = block_excl_scan(own, scan, tot);  // tot is the same in every thread
        if (mode == 1 || tot.hi > 0.0f) break;
        __syncthreads();  // sm and scan are refilled by the fallback pass
        mode = 1;         // zero residual mass: draw from p_j
    }
    const float target = u * (tot.hi + tot.lo);
    const float own_m = own.hi + own.lo;
    if (tid == 0) {
        *s_first = nt;
        *s_lastpos = -1;
    }
    __syncthreads();
    if (own_m > 0.0f) {
        atomicMax(s_lastpos, tid);
        if (excl.exceeds(own_m, target)) atomicMin(s_first, tid);
    }
    __syncthreads();
    const int first = *s_first;
    const int owner = first < nt ? first : *s_lastpos;
    if (owner < 0 && tid == 0) {
        shared_out->ent = -1;
        shared_out->mode = mode;
        shared_out->target = target;
    }
    if (tid == owner) {
        // the first entry of this run whose end passes the target (else its last entry with mass)
        CSum pre = excl, last_pre, found_pre;
        int found = -1, last_nz = -1;
        for (int e = e0; e < e1; ++e) {
            const float me = sm[e];
            if (me > 0.0f) {
                last_nz = e;
                last_pre = pre;
                if (first < nt && pre.exceeds(me, target)) {
                    found = e;
                    found_pre = pre;
                    break;
                }
            }
            pre.add(me);
        }
        const CSum pr = found >= 0 ? found_pre : last_pre;
        shared_out->ent = found >= 0 ? found : last_nz;
        shared_out->pre_hi = pr.hi;
        shared_out->pre_lo = pr.lo;
        shared_out->mode = mode;
        shared_out->target = target;
    }
    __syncthreads();
    return *shared_out;
}

// ===================================================================== large-V tier

// Kernel 1: (max, sum 2^((x-max) beta)) of every row's chunk.  grid (C, S); warp w takes
// rows w, w + nwarps, ...
template <bool VEC>
__global__ void __launch_bounds__(512) pqv_stats_kernel(PqArgs a, PqSplit sp) {
    pdl_wait();
    pdl_trigger();
    const int c = blockIdx.x, s = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const int R = 2 * a.k + 1;
    const int c0 = c * sp.L, c1 = min(a.V, c0 + sp.L);
    float beta;
    const int smode = session_mode(a, s, &beta);
    if (c == 0 && threadIdx.x == 0) sp.tickets[s] = 0u;
    if (smode < 0) return;
    if (smode == 0) {
        // greedy: (max, first index of it) of every row's chunk; the index travels as the
        // bits of the partial's second float
        for (int r = (sp.tstats ? a.k + 1 : 0) + warp; r < R; r += nwarps) {
            float m;
            int i;
            lane_argmax(row_ptr(a, s, r), c0, c1, lane, m, i);
            warp_argmax(m, i);
            if (lane == 0)
                reinterpret_cast<float2 *>(sp.stats)[((size_t)s * R + r) * sp.C + c] = make_float2(m, __int_as_float(i));
        }
        return;
    }
    // the accept scan's inputs, gathered here so kernel 2 reads them in its first round of
    // loads: the target and draft logits at each draft token (by a spare warp when the block
    // has one, else by warp 0 after its rows)
    const int gw = nwarps > R ? R : 0;
    const bool gather = c == 0 && warp == gw && lane < a.k;
    for (int r = (sp.tstats ? a.k + 1 : 0) + warp; r < R; r += nwarps) {
        const float *x = row_ptr(a, s, r);
        float m = -INFINITY, z = 0.0f;
        if (VEC) {
            const float4 *x4 = reinterpret_cast<const float4 *>(x + c0);
            const int n4 = (c1 - c0) >> 2;
            constexpr int U = 12;  // all of a lane's loads of a chunk row in one round at cfg3 sizes
            for (int base = 0; base < n4; base += 32 * U) {
                float4 v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = base + u * 32 + lane;
                    v[u] = i < n4 ? __ldg(x4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
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
        const float M = warp_max(m);
        const float zz = warp_sum((m > -INFINITY) ? z * ex2((m - M) * beta) : 0.0f);
        if (lane == 0) {
            float2 *st = reinterpret_cast<float2 *>(sp.stats) + ((size_t)s * R + r) * sp.C + c;
            *st = make_float2(M, zz);
        }
    }
    if (gather) {
        const int gx = a.drafts[(size_t)s * a.k + lane];
        float2 v = make_float2(0.0f, 0.0f);  // an out-of-range token is caught by kernel 2
        if (gx >= 0 && gx < a.V) v = make_float2(row_ptr(a, s, lane)[gx], row_ptr(a, s, a.k + 1 + lane)[gx]);
        sp.xin[(size_t)s * a.k + lane] = v;
    }
}

// The chunk partials of row r of session s and their count: the target rows' from the fused
// GEMM when it made them, else the statistics kernel's.
__device__ __forceinline__ const float2 *row_partials(const PqArgs &a, const PqSplit &sp, int s, int r, int &n) {
    if (sp.tstats && r <= a.k) {
        n = sp.Ct;
        return reinterpret_cast<const float2 *>(sp.tstats) + ((size_t)s * (a.k + 1) + r) * sp.Ct;
    }
    n = sp.C;
    return reinterpret_cast<const float2 *>(sp.stats) + ((size_t)s * (2 * a.k + 1) + r) * sp.C;
}

// Kernel 2: combine, accept scan, per-warp chunk masses, last-arriver inverse-CDF search.
//
// Each chunk of L tokens is cut into 8 contiguous warp segments; warp w of the CTA owns
// segment w and writes its draw mass (and its p_j mass, for the zero-residual fallback) to
// the workspace.  The last CTA of the session to finish picks the segment holding the
// crossing (a block-wide compensated scan over the session's C*8 masses) and then the token
// inside it (the same over the segment's tokens).  Every load of the first phase (partials,
// gathered draft logits) goes out in one round.
template <bool VEC>
__global__ void __launch_bounds__(256) pqv_verify_kernel(PqArgs a, PqSplit sp) {
    __shared__ float rowM[kMaxRows];
    __shared__ float rowL2Z[kMaxRows];
    __shared__ int s_j, s_last;
    extern __shared__ __align__(16) float pq_dyn[];  // the last CTA's copy of the segment masses
    pdl_wait();
    pdl_trigger();
    const int c = blockIdx.x, s = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int R = 2 * a.k + 1;
    float beta;
    const int smode = session_mode(a, s, &beta);
    const int c0 = c * sp.L, c1 = min(a.V, c0 + sp.L);
    const int Lw = sp.L / kSegsPerChunk;  // tokens per warp segment (a multiple of 16)
    if (smode < 0) {
        if (c == 0 && tid == 0) {
            set_status(a.status, Q2_ERR_BAD_TEMPERATURE);
            write_tokens(a, s, -1, -1);
        }
        return;
    }
    if (smode == 0) {
        // greedy: every row's argmax from the chunk partials (16 lanes per row; chunk order
        // and better_arg keep the lowest index among equal maxima), one-hot probabilities for
        // this chunk, and CTA 0 decides the tokens
        __shared__ int s_arg[kMaxRows];
        for (int r0 = 0; r0 < R; r0 += 16) {
            const int r = r0 + (tid >> 4), sub = tid & 15;
            float m = -INFINITY;
            int i = 0x7FFFFFFF;
            if (r < R) {
                int nc;
                const float2 *st = row_partials(a, sp, s, r, nc);
                for (int cc = sub; cc < nc; cc += 16) {
                    const float2 w = st[cc];
                    const int wi = __float_as_int(w.y);
                    if (better_arg(w.x, wi, m, i)) {
                        m = w.x;
                        i = wi;
                    }
                }
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
                const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
                if (better_arg(m2, i2, m, i)) {
                    m = m2;
                    i = i2;
                }
            }
            if (sub == 0 && r < R) s_arg[r] = i;
        }
        __syncthreads();
        if (a.probs)
            for (int r = 0; r < R; ++r) {
                float *o = a.probs + ((size_t)s * R + r) * a.V;
                const int am = s_arg[r];
                for (int y = c0 + tid; y < c1; y += blockDim.x) o[y] = (y == am) ? 1.0f : 0.0f;
            }
        if (c == 0 && tid == 0) {
            const int j = greedy_scan(a, s, s_arg);
            if (j < 0) set_status(a.status, Q2_ERR_BAD_TOKEN);
            write_tokens(a, s, j, j < 0 ? -1 : s_arg[j]);
        }
        return;
    }

    // 0. the accept scan's inputs (gathered by kernel 1): these loads go out in one round with
    //    the partials of step 1
    int xv = 0;
    float2 xl = make_float2(0.0f, 0.0f);
    float uv = 0.0f;
    if (warp == 0 && lane < a.k) {
        xv = a.drafts[(size_t)s * a.k + lane];
        xl = sp.xin[(size_t)s * a.k + lane];
        uv = a.u_acc[(size_t)s * a.k + lane];
    }

    // 1. row statistics from the chunk partials: 16 lanes per row, partials held in
    //    registers so the combine takes one round of loads
    for (int r0 = 0; r0 < R; r0 += 16) {
        const int r = r0 + (tid >> 4), sub = tid & 15;
        float2 v[8];
        float m = -INFINITY;
        int nc;
        const float2 *st = row_partials(a, sp, s, min(r, R - 1), nc);
        if (nc <= 16 * 8) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int cc = sub + 16 * u;
                v[u] = (r < R && cc < nc) ? st[cc] : make_float2(-INFINITY, 0.0f);
                m = fmaxf(m, v[u].x);
            }
        } else {
            for (int cc = sub; r < R && cc < nc; cc += 16) m = fmaxf(m, st[cc].x);
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float z = 0.0f;
        if (nc <= 16 * 8) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (v[u].x > -INFINITY) z += v[u].y * ex2((v[u].x - m) * beta);
        } else {
            for (int cc = sub; r < R && cc < nc; cc += 16) {
                const float2 w = st[cc];
                if (w.x > -INFINITY) z += w.y * ex2((w.x - m) * beta);
            }
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        if (sub == 0 && r < R) {
            rowM[r] = m;
            rowL2Z[r] = log2f(z);
        }
    }
    __syncthreads();
    // 2. accept scan: lane i evaluates draft i from the prefetched logits, a ballot finds
    //    the first rejection
    if (warp == 0) {
        bool bad = false, rej = false;
        if (lane < a.k) {
            if (xv < 0 || xv >= a.V) {
                bad = true;
            } else if (xl.y != -INFINITY) {  // q(x) == 0 accepts
                const float lp = (xl.x - rowM[lane]) * beta - rowL2Z[lane];
                const float lq = (xl.y - rowM[a.k + 1 + lane]) * beta - rowL2Z[a.k + 1 + lane];
                rej = !(uv < ex2(lp - lq));
            }
        }
        const unsigned badm = __ballot_sync(0xffffffffu, bad), rejm = __ballot_sync(0xffffffffu, rej);
        if (lane == 0) s_j = badm ? -1 : (rejm ? __ffs(rejm) - 1 : a.k);
    }
    __syncthreads();
    const int j = s_j;
    // optional probabilities of every row of this chunk
    if (a.probs) {
        for (int r = 0; r < R; ++r) {
            const float *x = row_ptr(a, s, r);
            float *o = a.probs + ((size_t)s * R + r) * a.V;
            const float M = rowM[r], L2 = rowL2Z[r];
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
    DrawRows D = draw_rows(a, s, j, rowM, rowL2Z);
    // 3. this warp's segment masses
    {
        const int y0 = c0 + warp * Lw, y1 = min(c1, y0 + Lw);
        float wsum = 0.0f, psum = 0.0f;
        if (VEC) {
            const float4 *t4 = reinterpret_cast<const float4 *>(D.t);
            const float4 *d4 = reinterpret_cast<const float4 *>(D.d);
            // four float4 of each row per lane in flight before any is used
            const int i1 = y1 >> 2;
            for (int i0 = (y0 >> 2) + lane; i0 < i1; i0 += 4 * 32) {
                float4 xt[4], xd[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + 32 * u;
                    xt[u] = i < i1 ? t4[i] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    xd[u] = (i < i1 && D.mode == 0) ? d4[i] : xt[u];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (i0 + 32 * u >= i1) break;
                    wsum += draw_weight(D, beta, xt[u].x, xd[u].x) + draw_weight(D, beta, xt[u].y, xd[u].y) +
                            draw_weight(D, beta, xt[u].z, xd[u].z) + draw_weight(D, beta, xt[u].w, xd[u].w);
                    if (D.mode == 0)
                        psum += ex2((xt[u].x - D.mt) * beta - D.lt) + ex2((xt[u].y - D.mt) * beta - D.lt) +
                                ex2((xt[u].z - D.mt) * beta - D.lt) + ex2((xt[u].w - D.mt) * beta - D.lt);
                }
            }
        } else {
            for (int y = y0 + lane; y < y1; y += 32) {
                const float xt = D.t[y];
                const float xd = (D.mode == 0) ? D.d[y] : xt;
                wsum += draw_weight(D, beta, xt, xd);
                if (D.mode == 0) psum += ex2((xt - D.mt) * beta - D.lt);
            }
        }
        wsum = warp_sum(wsum);
        psum = warp_sum(psum);
        if (lane == 0) {
            const size_t e = ((size_t)s * sp.C + c) * kSegsPerChunk + warp;
            sp.mass[e] = wsum;
            sp.pmass[e] = psum;
        }
    }
    __syncthreads();
    if (tid == 0) {
        // one acquire-release atomic: releases this CTA's masses (the barrier above ordered them
        // before it) and, for the last CTA, acquires the others' (read below with ld.cg)
        unsigned ticket;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;\n"
                     : "=r"(ticket)
                     : "l"(sp.tickets + s)
                     : "memory");
        s_last = ticket == (unsigned)(sp.C - 1);
    }
    __syncthreads();
    if (!s_last) return;

    // 4. last CTA: the segment holding the crossing of u_fin * total (pick_segment), then the
    //    token inside it, by a block-wide compensated scan: every thread sums a contiguous run
    //    of the segment's tokens, the scan gives its prefix, the first thread whose run
    //    crosses walks that run.  If rounding puts the target past the end, the last token
    //    with mass is taken.
    __shared__ float s_scan[64];
    __shared__ int s_first, s_lastpos, s_ent;
    __shared__ float s_pre[2];
    __shared__ SegPick s_pick;
    const int nseg = sp.C * kSegsPerChunk;
    const int nt = blockDim.x;
    const SegPick pk = pick_segment(sp.mass + (size_t)s * nseg, sp.pmass + (size_t)s * nseg, nseg, D.mode,
                                    a.u_fin[s], pq_dyn, s_scan, &s_first, &s_lastpos, &s_pick);
    D.mode = pk.mode;
    const float target = pk.target;
    const int owner1 = pk.ent;
    if (tid == 0) {
        s_ent = pk.ent;
        s_pre[0] = pk.pre_hi;
        s_pre[1] = pk.pre_lo;
    }
    __syncthreads();
    int y_sel = -1;
    if (owner1 >= 0) {
        // level 2: the tokens of the selected segment
        const int ent = s_ent;
        const int sc = ent / kSegsPerChunk, sw = ent - sc * kSegsPerChunk;
        const int ty0 = sc * sp.L + sw * Lw, ty1 = min(min(a.V, sc * sp.L + sp.L), ty0 + Lw);
        if (Lw <= 32 * kSegWarpRun) {
            // a segment of at most 32 x kSegWarpRun tokens: warp 0 alone, each lane a contiguous
            // run of the segment's weights in registers (loaded at once), one compensated warp
            // scan, a ballot for the first run that crosses (else the last run with mass) and
            // that lane's walk -- no block barrier
            if (warp == 0) {
                const int rl = cdiv(max(ty1 - ty0, 0), 32);
                const int y0 = min(ty1, ty0 + lane * rl), y1 = min(ty1, y0 + rl);
                CSum seg_pre;
                seg_pre.hi = s_pre[0];
                seg_pre.lo = s_pre[1];
                float wv[kSegWarpRun];
                CSum own, tot;
#pragma unroll
                for (int u = 0; u < kSegWarpRun; ++u) {
                    const int y = y0 + u;
                    wv[u] = y < y1 ? draw_weight(D, beta, D.t[y], D.d[y]) : 0.0f;
                    if (y < y1) own.add(wv[u]);
                }
                const CSum excl = csum_plus(seg_pre, warp_excl_scan_c(own, lane, tot));
                const float own_m = own.hi + own.lo;
                const unsigned cm = __ballot_sync(0xffffffffu, own_m > 0.0f && excl.exceeds(own_m, target));
                const unsigned pm = __ballot_sync(0xffffffffu, own_m > 0.0f);
                const int first = cm ? __ffs(cm) - 1 : 32;
                const int owner = first < 32 ? first : (pm ? 31 - __clz(pm) : -1);
                int pick = -1;
                if (lane == owner) {
                    // the first token of the run whose end passes the target, else its last token with mass
                    CSum pre = excl;
                    int found = -1, last_nz = -1;
                    bool done = false;
#pragma unroll
                    for (int u = 0; u < kSegWarpRun; ++u) {
                        const int y = y0 + u;
                        if (!done && y < y1) {
                            const float w = wv[u];
                            if (w > 0.0f) {
                                last_nz = y;
                                if (first < 32 && pre.exceeds(w, target)) {
                                    found = y;
                                    done = true;
                                }
                            }
                            if (!done) pre.add(w);
                        }
                    }
                    pick = found >= 0 ? found : last_nz;
                }
                const int y = owner >= 0 ? __shfl_sync(0xffffffffu, pick, owner) : -1;
                if (lane == 0) write_tokens(a, s, j, y);
            }
            return;
        }
        // larger segments: r tokens per thread, block-wide scan
        const int r = cdiv(max(ty1 - ty0, 0), nt);
        const int y0 = min(ty1, ty0 + tid * r), y1 = min(ty1, y0 + r);
        CSum seg_pre;
        seg_pre.hi = s_pre[0];
        seg_pre.lo = s_pre[1];
        // a thread's weights stay in registers for the walk when it has at most 4 tokens
        float wv[4];
        CSum own2, tot2;
        if (r <= 4) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int y = y0 + u;
                wv[u] = y < y1 ? draw_weight(D, beta, D.t[y], D.d[y]) : 0.0f;
                if (y < y1) own2.add(wv[u]);
            }
        } else {
            for (int y = y0; y < y1; ++y) own2.add(draw_weight(D, beta, D.t[y], D.d[y]));
        }
        __syncthreads();  // s_scan is reused
        const CSum excl2 = csum_plus(seg_pre, block_excl_scan(own2, s_scan, tot2));
        if (tid == 0) {
            s_first = nt;
            s_lastpos = -1;
        }
        __syncthreads();
        const float own2_m = own2.hi + own2.lo;
        if (own2_m > 0.0f) {
            atomicMax(&s_lastpos, tid);
            if (excl2.exceeds(own2_m, target)) atomicMin(&s_first, tid);
        }
        __syncthreads();
        const int owner2 = s_first < nt ? s_first : s_lastpos;
        if (tid == owner2) {
            CSum pre = excl2;
            int found = -1, last_nz = -1;
            for (int y = y0; y < y1; ++y) {
                const int u = y - y0;
                const float w = r > 4 ? draw_weight(D, beta, D.t[y], D.d[y])
                                      : (u == 0 ? wv[0] : u == 1 ? wv[1] : u == 2 ? wv[2] : wv[3]);
                if (w > 0.0f) {
                    last_nz = y;
                    if (s_first < nt && pre.exceeds(w, target)) {
                        found = y;
                        break;
                    }
                }
                pre.add(w);
            }
            s_ent = found >= 0 ? found : last_nz;
        }
        __syncthreads();
        y_sel = owner2 >= 0 ? s_ent : -1;
    }
    if (tid == 0) write_tokens(a, s, j, y_sel);
}

namespace {
// launch_pdl with dynamic shared memory
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_smem(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                            Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
}  // namespace

cudaError_t launch_pq_verify(const PqArgs &a, const PqSplit &sp, bool warp_tier, int num_sms, cudaStream_t st) {
    if (warp_tier) {
        const bool vec = (a.V % 4) == 0;
        if (a.V <= kSmallWarpMaxV) {  // one warp per session, 8 sessions per CTA
            const dim3 grid(cdiv(a.S, 8));
            return probed(kProbePqVerify, st, [&] {
                return vec ? launch_pdl(pqv_small_kernel<1, true>, grid, dim3(256), st, a)
                           : launch_pdl(pqv_small_kernel<1, false>, grid, dim3(256), st, a);
            });
        }
        const dim3 block(32 * kSmallCtaWarps);
        return probed(kProbePqVerify, st, [&] {  // one CTA per session
            return vec ? launch_pdl(pqv_small_kernel<kSmallCtaWarps, true>, dim3(a.S), block, st, a)
                       : launch_pdl(pqv_small_kernel<kSmallCtaWarps, false>, dim3(a.S), block, st, a);
        });
    }
    const bool vec = (a.V % 4) == 0 && (sp.L % 4) == 0;
    const int R = 2 * a.k + 1;
    const dim3 grid(sp.C, a.S);
    const int warps1 = min(R + 1, 16);  // a spare warp gathers the accept-scan inputs
    cudaError_t e = probed(kProbePqStats, st, [&] {
        return vec ? launch_pdl(pqv_stats_kernel<true>, grid, dim3(warps1 * 32), st, a, sp)
                   : launch_pdl(pqv_stats_kernel<false>, grid, dim3(warps1 * 32), st, a, sp);
    });
    if (e != cudaSuccess) return e;
    // dynamic shared memory: the last CTA's copy of the segment masses (at most
    // kMaxChunks * kSegsPerChunk floats)
    const size_t smem2 = (size_t)sp.C * kSegsPerChunk * sizeof(float);
    return probed(kProbePqVerify, st, [&] {
        return vec ? launch_pdl_smem(pqv_verify_kernel<true>, grid, dim3(256), smem2, st, a, sp)
                   : launch_pdl_smem(pqv_verify_kernel<false>, grid, dim3(256), smem2, st, a, sp);
    });
}

}  // namespace q2v
