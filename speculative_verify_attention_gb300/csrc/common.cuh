// common.cuh -- helpers shared by the kvq8attn kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kvq8attn.h"

namespace kvq8 {

constexpr int kQBlock = 32;          // values per Q8_0 block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<const __half2*>(&u); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The dynamic shared-memory opt-in of one kernel, set once per device (the attribute belongs to
// the kernel on the current device); one static object per kernel instantiation.
struct SmemOptIn {
    static constexpr int kMaxDev = 64;
    std::mutex mu;
    bool done[kMaxDev] = {};
    template <typename Kernel>
    int ensure(Kernel* kernel, int bytes) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return KVQ8_ERR_CUDA;
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
                return KVQ8_ERR_CUDA;
            done[dev] = true;
        }
        return KVQ8_OK;
    }
};

inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? KVQ8_OK : KVQ8_ERR_CUDA;
}

// Two int8 codes -> two fp16 values, exactly.  The input word x holds the codes already
// offset by +128 (sign bit flipped), so each is an unsigned byte u in [1, 255].  Placing u
// in the low mantissa byte of the fp16 pattern 0x64uu gives 1024 + u exactly; subtracting
// 1152 = 1024 + 128 leaves the signed code.  `sel` picks which two bytes of x are used.
template <unsigned kSel>
__device__ __forceinline__ uint32_t biased_bytes_to_half2(uint32_t x) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(0x64646464u), "n"(kSel));
    const __half2 h = *reinterpret_cast<const __half2*>(&r);
    const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480u));  // 1152.0
    const __half2 v = __hsub2(h, bias);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Nibble pairs -> fp16 pairs, exactly.  x holds two 16-bit halves (key a in the low half, key b
// in the high half), each 4 nibbles of 4 consecutive dims.  lo: nibbles 0 and 4 (dim 0 of both
// keys) placed in the fp16 pattern 0x640n is 1024 + n; subtracting 1032 gives n - 8.  hi:
// nibbles 1 and 5 masked in place are 16 n in the mantissa, 1024 + 16 n; times 1/16 minus 72
// gives n - 8.  (x >> 8 gives dims 2 and 3 the same way.)
__device__ __forceinline__ uint32_t nib_lo_to_half2(uint32_t x) {
    const uint32_t r = (x & 0x000F000Fu) | 0x64006400u;
    const __half2 v = __hsub2(u32_as_h2(r), __half2half2(__ushort_as_half((unsigned short)0x6408u)));  // 1032
    return h2_as_u32(v);
}
__device__ __forceinline__ uint32_t nib_hi_to_half2(uint32_t x) {
    const uint32_t r = (x & 0x00F000F0u) | 0x64006400u;
    const __half2 v = __hfma2(u32_as_h2(r), __half2half2(__ushort_as_half((unsigned short)0x2C00u)),   // 1/16
                              __half2half2(__ushort_as_half((unsigned short)0xD480u)));                // -72
    return h2_as_u32(v);
}

// Byte m of w (two 4-bit codes stored as nibble + 8, element 2k in the low nibble) -> the fp16
// pair (low - 8, high - 8), exactly: the byte placed in bytes 0 and 2 of a word and masked with
// 0x00F0000F gives, after OR with 0x64006400, the pair (1024 + lo, 1024 + 16 hi); one fma with
// (1, 1/16) and (-1032, -72) turns it into the two codes.
template <int M>
__device__ __forceinline__ uint32_t nib_byte_to_half2(uint32_t w) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(w), "r"(0u), "n"(0x4040u | (M * 0x0101u)));
    r = (r & 0x00F0000Fu) | 0x64006400u;
    const __half2 mul = __halves2half2(__ushort_as_half((unsigned short)0x3C00u), __ushort_as_half((unsigned short)0x2C00u));
    const __half2 add = __halves2half2(__ushort_as_half((unsigned short)0xE408u), __ushort_as_half((unsigned short)0xD480u));
    const __half2 v = __hfma2(*reinterpret_cast<const __half2*>(&r), mul, add);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Byte interleave of two words: result bytes = {a.b[i], b.b[i], a.b[j], b.b[j]}.
template <unsigned kSel>
__device__ __forceinline__ uint32_t prmt2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "n"(kSel));
    return r;
}

// D += A * B, m16n8k16, fp16 inputs, fp32 accumulate (register fragments).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B (C = 0), m16n8k16, fp16 inputs, fp32 result.
__device__ __forceinline__ void mma_f16_16816_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                 uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// 2^x with the hardware approximation (relative error about 2^-22); -inf gives 0.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}


__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy; bytes past src_bytes (0 or 16) are zero-filled.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
// 8-byte global -> shared copy (L1-allocating form); bytes past src_bytes are zero-filled.
__device__ __forceinline__ void cp_async_8(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ float half_bits_to_float(uint16_t b) { return __half2float(__ushort_as_half(b)); }

}  // namespace kvq8
