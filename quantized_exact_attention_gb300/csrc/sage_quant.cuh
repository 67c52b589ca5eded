// sage_quant.cuh - the INT8 block-quantization arithmetic shared by the
// preparation kernels and the attention kernel's Q prologue, so that both
// produce the same codes and scales bit for bit (Experiment Log, "Phase 0
// Import And Verification": INT8 quantization of Q/K).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace sage {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 8 packed BF16 values -> FP32 (exact widening)
__device__ __forceinline__ void unpack8(const uint4& u, float (&x)[8]) {
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x);
    x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z);
    x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}

// |x| of 8 packed BF16 values, maximum folded into m (the sign bit is cleared
// on the packed words: BF16 -> FP32 widening is exact, so this equals the
// maximum of |x| over the widened values)
__device__ __forceinline__ float absmax8(const uint4& u, float m) {
    float x[8];
    unpack8(make_uint4(u.x & 0x7FFF7FFFu, u.y & 0x7FFF7FFFu, u.z & 0x7FFF7FFFu, u.w & 0x7FFF7FFFu), x);
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, x[e]);
    return m;
}

// Block scale and its inverse: scale = amax/127, inv = 127/amax (IEEE
// division); an all-zero block has scale 0 and codes 0.
__device__ __forceinline__ float int8_scale(float amax) { return amax > 0.f ? __fdiv_rn(amax, 127.0f) : 0.f; }
__device__ __forceinline__ float int8_inv(float amax) { return amax > 0.f ? __fdiv_rn(127.0f, amax) : 0.f; }

// code = clamp(rne(x * inv), -127, 127)
__device__ __forceinline__ int int8_code(float x, float inv) {
    int c = __float2int_rn(__fmul_rn(x, inv));
    return c > 127 ? 127 : (c < -127 ? -127 : c);
}

// An INT8 code as the bit pattern of the equal FP16 integer (exact).
__device__ __forceinline__ uint32_t half_code(int c) {
    return (uint32_t)__half_as_ushort(__int2half_rn(c));
}

// 8 codes -> 8 FP16 code images, packed like the source BF16 words.
__device__ __forceinline__ uint4 pack_half_codes(const int (&c)[8]) {
    uint4 hv;
    hv.x = half_code(c[0]) | (half_code(c[1]) << 16);
    hv.y = half_code(c[2]) | (half_code(c[3]) << 16);
    hv.z = half_code(c[4]) | (half_code(c[5]) << 16);
    hv.w = half_code(c[6]) | (half_code(c[7]) << 16);
    return hv;
}

}  // namespace sage
