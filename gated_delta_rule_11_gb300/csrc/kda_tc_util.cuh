// Small device helpers shared by the tensor-core prefill kernels: bf16 /
// fp16 packing, MUFU approximations, tf32 rounding and the legacy warp-level
// products used for the 16x16 in-tile blocks.  Library-internal.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace kda {
namespace tcu {

__device__ __forceinline__ float bf16_at(const uint8_t *p) {
    return __bfloat162float(__ushort_as_bfloat16(*reinterpret_cast<const uint16_t *>(p)));
}
// One of the two bf16 values packed in a 32-bit word (ch 0 = low half).
__device__ __forceinline__ float bf16_half(uint32_t w, int ch) {
    return __uint_as_float(ch ? (w & 0xffff0000u) : (w << 16));
}
// One of the two fp16 values packed in a 32-bit word (ch 0 = low half).
__device__ __forceinline__ float f16_half(uint32_t w, int ch) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(ch ? (w >> 16) : (w & 0xffffu))));
}
__device__ __forceinline__ void st_h(uint8_t *p, float x) {
    *reinterpret_cast<uint16_t *>(p) = __half_as_ushort(__float2half_rn(x));
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}
constexpr float kLog2e = 1.4426950408889634f;
// Single-instruction MUFU approximations (rel. error ~2^-22 and 1 ulp).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float to_tf32(float x) {
    uint32_t u;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(u) : "f"(x));
    return __uint_as_float(u);
}
// x rounded to tf32 for a tf32 mma.sync operand, which reads only the upper
// 19 bits of each 32-bit element: adding half a tf32 ulp (bit 12) to the
// pattern rounds those bits to nearest, ties away from zero -- the value
// to_tf32 gives -- with one integer add; the low 13 bits are left as
// garbage, so the result is for mma operands only.
__device__ __forceinline__ float tf32_operand(float x) { return __uint_as_float(__float_as_uint(x) + 0x1000u); }
// D (16x8 fp32) += A (16x8 tf32, row) * B (8x8 tf32, col)
__device__ __forceinline__ void mma_1688_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D (16x8 fp32) += A (16x16 fp16, row) * B (16x8 fp16, col); a*, b* hold fp16 pairs
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace tcu
}  // namespace kda
