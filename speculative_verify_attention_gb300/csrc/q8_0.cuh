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

// Codes of one lane's 4 values x / d, rounded half away from zero and clamped to [-qmax, qmax],
// equal to rounding the IEEE quotient fl(x / d).  The fast form rounds y = x * r, r =
// rcp.approx(d) (relative error about 2^-23), to the nearest integer: y differs from fl(x / d)
// by at most |x / d| (2^-23 + 2^-24 + 2^-24) < 2^-14 (|x / d| < 128 here), and rounding to an
// integer only changes at the half-integers, so when y is farther than 2^-12 from one the
// nearest integer of y is the code (and no tie arises).  A lane with a value that near a
// half-integer, or with a y that is not finite (d subnormal, flushed by the approximation),
// recomputes its codes with the IEEE division; the warp takes that branch only if some lane
// needs it.  d == 0 gives codes 0.  Every lane of the warp must call it.
// fl(a / b), the IEEE quotient, for a block maximum a >= 0 and b = QMAX (127 or 7), with r =
// RN(1 / b): q0 = a r, e = a - q0 b (exact through the FMA), q = q0 + e r rounded once.  This is
// the correction step for a divisor known in advance (Brisebarre, Muller and Raina, "Accelerating
// correctly rounded floating-point division when the divisor is known in advance", IEEE Trans.
// Computers 53(8), 2004); checked against the IEEE division on every non-negative finite fp32 a
// for both divisors, with no difference.  A non-finite maximum takes the division itself.
template <int QMAX>
__device__ __forceinline__ float scale_of(float amax) {
    constexpr float b = (float)QMAX;
    constexpr float r = 1.0f / (float)QMAX;
    if (!(amax < INFINITY)) return __fdiv_rn(amax, b);
    const float q0 = __fmul_rn(amax, r);
    const float e = __fmaf_rn(-q0, b, amax);
    return __fmaf_rn(e, r, q0);
}

template <int QMAX>
__device__ __forceinline__ void codes_of(const float (&x)[4], float d, int (&c)[4]) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    bool slow = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float y = x[e] * r;
        const float n = rintf(y);
        c[e] = (int)n;
        slow |= !(fabsf(y - n) <= 0.5f - 0x1p-12f);  // also true for a y that is not finite
    }
    if (d == 0.0f) {
        slow = false;
#pragma unroll
        for (int e = 0; e < 4; ++e) c[e] = 0;
    }
    if (__any_sync(0xffffffffu, slow) && slow) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            c[e] = (int)fminf(fmaxf(roundf(__fdiv_rn(x[e], d)), -(float)QMAX), (float)QMAX);
    }
}

// One 32-value block held by 8 consecutive lanes (lanes 8i .. 8i+7 of the warp), 4 values per
// lane in block order.  Every lane of the warp must call it (the max is a warp shuffle).
// Returns this lane's 4 codes packed little-endian; *scale_bits gets the block's fp16 scale.
__device__ __forceinline__ uint32_t q8_0_block(float4 v, uint16_t* scale_bits) {
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d32 = scale_of<127>(amax);
    const float xs[4] = {v.x, v.y, v.z, v.w};
    int c[4];
    codes_of<127>(xs, d32, c);
    // low bytes of the four codes, in order: two byte permutes pair them, a third joins the pairs
    uint32_t t01, t23, packed;
    asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(t01) : "r"(c[0]), "r"(c[1]));
    asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(t23) : "r"(c[2]), "r"(c[3]));
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(packed) : "r"(t01), "r"(t23));
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
    const float d32 = scale_of<7>(amax);
    const float xs[4] = {v.x, v.y, v.z, v.w};
    int c[4];
    codes_of<7>(xs, d32, c);
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) packed |= (uint32_t)(c[e] + 8) << (4 * e);
    *scale_bits = __half_as_ushort(__float2half_rn(d32));
    return packed;
}

}  // namespace kvq8
