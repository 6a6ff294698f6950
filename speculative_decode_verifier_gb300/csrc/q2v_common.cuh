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

// Two Q2B32 codes -> their dequantised product q*d as an f16x2, exactly rounded once.
//
// Codes c_i (bits 2i..2i+1) and c_{i+8} (bits 2i+16..2i+17) of a 32-bit code word are
// moved to bits 8..9 of each 16-bit half and or-ed into the f16 constant 4.0 (0x4400):
// in [4, 8) the f16 spacing is 2^-8, so the halves read 4 + c exactly.  Then
// fma(4 + c, d, -4d) = c*d computed exactly and rounded once to f16 (-4d is exact for
// any |d| <= 16376).  The offset m is applied separately in fp32.
template <int I>
__device__ __forceinline__ uint32_t dequant_pair(uint32_t word, uint32_t d2, uint32_t nd4) {
    constexpr int sh = 8 - 2 * I;
    uint32_t v = sh >= 0 ? (word << (sh >= 0 ? sh : 0)) : (word >> (sh < 0 ? -sh : 0));
    uint32_t x = lop3_and_or(v, 0x03000300u, 0x44004400u);
    return hfma2_u32(x, d2, nd4);
}

// f16x2 {d, d} and {-4d, -4d} from a block's packed (d | m << 16) word.
__device__ __forceinline__ void scale_pair(uint32_t dm, uint32_t &d2, uint32_t &nd4) {
    uint32_t d = dm & 0xFFFFu;
    d2 = d | (d << 16);
    __half nd = __hmul(__ushort_as_half((unsigned short)d), __float2half_rn(-4.0f));
    uint32_t n = __half_as_ushort(nd);
    nd4 = n | (n << 16);
}

// |d| > 16376 makes -4d overflow: flag it.
__device__ __forceinline__ bool scale_out_of_range(uint32_t dm) {
    uint32_t mag = dm & 0x7FFFu;
    return mag > 0x73FFu && mag < 0x7C00u;  // 0x73FF = 16376; >= 0x7C00 is inf/nan (propagates)
}

}  // namespace q2v
