// q2v_common.cuh -- shared device helpers of libq2v (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/q2v.h"

#define Q2V_VERSION 100

namespace q2v {

constexpr int kBlockK = 32;      // weights per Q2B32 block
constexpr int kBlockBytes = 12;  // bytes per Q2B32 block

// Status word at the start of every workspace.  Kernels record the first device error
// with atomicCAS (0 -> code); q2_get_device_status reads and clears it.
struct WsHeader {
    unsigned int status;
    unsigned int pad[63];
};
static_assert(sizeof(WsHeader) == Q2_WORKSPACE_HEADER_BYTES, "header size");

__device__ __forceinline__ void set_status(unsigned int *status, unsigned int code) {
    if (status) atomicCAS(status, 0u, code);
}

__host__ __device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------- programmatic dependent launch
//
// Every kernel of the library is launched with programmatic stream serialization, so it
// may start while the previous kernel in the stream is still running.  Each kernel calls
// pdl_wait() before touching anything a predecessor may write (it returns once every
// prerequisite grid has completed and its memory is visible) and then pdl_trigger() so its
// own successor can be scheduled early.  The only reads issued before pdl_wait() are of
// Q2B32 weights in GEMM kernels whose programmatic predecessor is the library's own prep
// kernel, which itself has already waited for everything before it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
__host__ __device__ __forceinline__ size_t align_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

// ---------------------------------------------------------------- tensor-core MMA (legacy path)

// D = A(16x16, f16, row) * B(16x8, f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A(16x8, f16, row) * B(8x8, f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t magic) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(r) : "r"(a), "r"(mask), "r"(magic));  // (a & b) | c
    return r;
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// Two Q2B32 codes -> their products with the block scale, as an f16x2, each exactly
// rounded once.
//
// A 32-bit code word holds 16 codes, code c at bits 2c.  Codes i and i+8 (i = 0..3) sit at
// the same bit offset 2i inside the low and the high 16-bit half; for i = 4..7 they do
// after one shift of the word by 8.  Or-ed into the f16 constant 1024 (0x6400), whose
// mantissa step is 1, the masked halves read exactly 1024 + q * 4^p with p = i mod 4.  Then
// fma(1024 + q*4^p, d, -1024 d) = q * 4^p * d, computed exactly and rounded once to f16
// (-1024 d is exact for |d| < 64, and 192 |d| stays below the f16 maximum).  The activation
// that meets this product in the MMA carries the matching factor 4^-p (applied, exactly, when
// the activations are prepared), so each product is q * d * a.  The offset m is applied
// separately, exactly.  Per two weights: one lop3 and one fma (plus one shift per 8 pairs).
template <int POS>
__device__ __forceinline__ uint32_t dequant_pos(uint32_t v, uint32_t d2, uint32_t nd1024) {
    uint32_t x, r;
    // (v & mask) | 1024.0h2 in one lop3 (mask as an immediate), then one f16x2 fma
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(x) : "r"(v), "n"(0x00030003u << POS), "r"(0x64006400u));
    asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(r) : "r"(x), "r"(d2), "r"(nd1024));
    return r;
}

// f16x2 {d, d} and {-1024 d, -1024 d} from a block's packed (d | m << 16) word: one byte
// permute and one f16x2 multiply (-1024 = 0xE400).
__device__ __forceinline__ void scale_pair(uint32_t dm, uint32_t &d2, uint32_t &nd1024) {
    d2 = prmt(dm, dm, 0x1010u);
    asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(nd1024) : "r"(d2), "r"(0xE400E400u));
}

// Division by a run-time constant d >= 1 for 0 <= u < 2^31 (round-up multiply-shift:
// s = ceil(log2 d), m = floor(2^32 (2^s - d) / d) + 1, u / d = (umulhi(u, m) + u) >> s).
struct FastDiv {
    uint32_t d, m, s;
    FastDiv() = default;
    __host__ __device__ explicit FastDiv(uint32_t d_) : d(d_) {
        s = 0;
        while ((1u << s) < d) ++s;
        m = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << s) - d)) / d + 1);
    }
    __device__ __forceinline__ uint32_t div(uint32_t u) const { return (__umulhi(u, m) + u) >> s; }
};

// Range of the scales.  dequant_pos is exact for |d| < 64 (-1024 d must be a finite f16).
// Kernels keep a running f16x2 maximum of |d|, |m| over the blocks they decode (two
// instructions per block; a NaN scale is skipped by the maximum and propagates to the
// outputs instead) and flag Q2_ERR_RANGE at the end if the |d| half reached 64 (0x5400),
// infinity included.
__device__ __forceinline__ uint32_t scale_mag_max(uint32_t acc, uint32_t dm) {
    uint32_t r;
    asm("max.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(dm & 0x7FFF7FFFu), "r"(acc));
    return r;
}
__device__ __forceinline__ bool scale_mag_out_of_range(uint32_t acc) { return (acc & 0xFFFFu) >= 0x5400u; }

}  // namespace q2v
