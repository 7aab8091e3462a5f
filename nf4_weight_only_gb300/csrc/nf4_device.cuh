// Device-side helpers shared by the NF4 kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace nf4 {

constexpr int kGroup = 64;  // weights per scale group (deep-fold README, format paragraph)

// The NormalFloat-4 table published with QLoRA (Dettmers et al., 2023, appendix), index 0..15.
// The published literals are the definition; each is an exact binary32 number.
__device__ __constant__ static const float kNF4[16] = {
    -1.0f,
    -0.6961928009986877f,
    -0.5250730514526367f,
    -0.39491748809814453f,
    -0.28444138169288635f,
    -0.18477343022823334f,
    -0.09105003625154495f,
    0.0f,
    0.07958029955625534f,
    0.16093020141124725f,
    0.24611230194568634f,
    0.33791524171829224f,
    0.44070982933044434f,
    0.5626170039176941f,
    0.7229568362236023f,
    1.0f,
};

// ---------------------------------------------------------------------------------------------
// Thin PTX wrappers
// ---------------------------------------------------------------------------------------------

// Byte permute: output byte i = byte sel_i of {b:a} (a = bytes 0-3, b = bytes 4-7); a selector
// nibble with bit 3 set replicates the sign bit of the addressed byte instead.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Per-bit select: bits of `b` where `mask` is 1, bits of `a` where it is 0.
__device__ __forceinline__ uint32_t select_bits(uint32_t a, uint32_t b, uint32_t mask) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xD8;" : "=r"(d) : "r"(a), "r"(b), "r"(mask));
    return d;
}

// acc + lo16(w) * lo16(x) and acc + hi16(w) * hi16(x) with bf16 operands: the product of two bf16
// numbers is exact in fp32, so each step rounds once (fp32 accumulate).
__device__ __forceinline__ void fma_bf16x2(float& acc_lo, float& acc_hi, uint32_t w, uint32_t x) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
        "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
        : "+f"(acc_lo), "+f"(acc_hi)
        : "r"(w), "r"(x));
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_ca_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_nc_u16(const uint16_t* p) {
    uint16_t v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

}  // namespace nf4
