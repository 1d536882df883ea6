// q8_0.cuh -- the Q8_0 block quantiser shared by the append kernel and the verify kernel's
// window slice, so that both write the same bytes.
//
// Source: "Engine perf(hip): MTP draft, shared expert, verify/sampler head", Summary item 4
// (a warp-per-block Q8_0 quantiser, bitwise equal to its CPU reference): the scale is
// max|x| / 127 of the 32-value block, stored as fp16; each code is x / scale (fp32 scale,
// IEEE division) rounded half away from zero and clamped to [-127, 127]; an all-zero block
// has scale 0 and codes 0.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace kvq8 {

// One 32-value block held by 8 consecutive lanes (lanes 8i .. 8i+7 of the warp), 4 values per
// lane in block order.  Every lane of the warp must call it (the max is a warp shuffle).
// Returns this lane's 4 codes packed little-endian; *scale_bits gets the block's fp16 scale.
__device__ __forceinline__ uint32_t q8_0_block(float4 v, uint16_t* scale_bits) {
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d32 = __fdiv_rn(amax, 127.0f);
    const float xs[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float r = 0.0f;
        if (d32 != 0.0f) r = fminf(fmaxf(roundf(__fdiv_rn(xs[e], d32)), -127.0f), 127.0f);
        packed |= (uint32_t)(uint8_t)(int8_t)(int)r << (8 * e);
    }
    *scale_bits = __half_as_ushort(__float2half_rn(d32));
    return packed;
}

}  // namespace kvq8

namespace kvq8 {

// The 4-bit V blocks of a K8V4 pool: the same 8-lane block layout, scale max|x| / 7 (fp32
// division, stored as fp16), codes round-half-away-from-zero of x / scale clamped to [-7, 7],
// stored as nibbles code + 8 with element 2m in the low nibble of byte m.  Returns this
// lane's 4 values as 2 bytes (little-endian in the low 16 bits).  The K8V4 pool is named,
// without its format, in "gfx12 WMMA kernel for the int8-KV QSA prompt attention" (Gating).
__device__ __forceinline__ uint32_t q4_block(float4 v, uint16_t* scale_bits) {
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d32 = __fdiv_rn(amax, 7.0f);
    const float xs[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float r = 0.0f;
        if (d32 != 0.0f) r = fminf(fmaxf(roundf(__fdiv_rn(xs[e], d32)), -7.0f), 7.0f);
        packed |= (uint32_t)((int)r + 8) << (4 * e);
    }
    *scale_bits = __half_as_ushort(__float2half_rn(d32));
    return packed;
}

}  // namespace kvq8
