// selftest.cu -- kvq8_selftest_convert: the kernels' code -> fp16 conversions run on caller data,
// so a test can push every code value and every byte pair through them.
//
// Source: "gfx12 WMMA kernel for the int8-KV QSA prompt attention", How: the int8 -> fp16
// conversion of the codes is exact and was checked over all byte pairs; the same device
// functions that the verify and prompt kernels call (common.cuh) run here unchanged.
#include "common.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace kvq8 {
namespace {

constexpr int kSelfThreads = 256;

// kind 0 (QK / prompt dequantiser): in[i] holds 4 codes; out[2i], out[2i+1] = codes (0, 1), (2, 3).
// kind 1 (PV A fragments): in[2i], in[2i+1] are the words w0, w1 of two key rows; out[4i .. 4i+3] =
//        (w0.b0, w1.b0), (w0.b1, w1.b1), (w0.b2, w1.b2), (w0.b3, w1.b3) through the byte interleaves.
// kind 2 (4-bit PV fragments): in[i] = two 16-bit halves of nibbles; out[4i .. 4i+3] = nib_lo(x),
//        nib_hi(x), nib_lo(x >> 8), nib_hi(x >> 8).
// kind 3 (4-bit prompt dequantiser): in[i] = 4 bytes of nibble pairs; out[4i + m] = byte m's pair.
__global__ void __launch_bounds__(kSelfThreads) selftest_convert_kernel(int kind, const uint32_t* __restrict__ in,
                                                                        uint32_t* __restrict__ out, int n) {
    const int i = blockIdx.x * kSelfThreads + threadIdx.x;
    if (i >= n) return;
    if (kind == 0) {
        const uint32_t x = in[i] ^ 0x80808080u;
        out[2 * i] = biased_bytes_to_half2<0x4140>(x);
        out[2 * i + 1] = biased_bytes_to_half2<0x4342>(x);
    } else if (kind == 1) {
        const uint32_t w0 = in[2 * i] ^ 0x80808080u, w1 = in[2 * i + 1] ^ 0x80808080u;
        const uint32_t y01 = prmt2<0x5140>(w0, w1), y23 = prmt2<0x7362>(w0, w1);
        out[4 * i] = biased_bytes_to_half2<0x4140>(y01);
        out[4 * i + 1] = biased_bytes_to_half2<0x4342>(y01);
        out[4 * i + 2] = biased_bytes_to_half2<0x4140>(y23);
        out[4 * i + 3] = biased_bytes_to_half2<0x4342>(y23);
    } else if (kind == 2) {
        const uint32_t x = in[i];
        out[4 * i] = nib_lo_to_half2(x);
        out[4 * i + 1] = nib_hi_to_half2(x);
        out[4 * i + 2] = nib_lo_to_half2(x >> 8);
        out[4 * i + 3] = nib_hi_to_half2(x >> 8);
    } else {
        const uint32_t w = in[i];
        out[4 * i] = nib_byte_to_half2<0>(w);
        out[4 * i + 1] = nib_byte_to_half2<1>(w);
        out[4 * i + 2] = nib_byte_to_half2<2>(w);
        out[4 * i + 3] = nib_byte_to_half2<3>(w);
    }
}

// One thread waits on a barrier that nothing arrives on (phase 0 never completes), with the
// library's bounded wait; when the wait gives up it sets the device error flag, as the pipeline
// kernels do on a timeout, and the kernel returns.
__global__ void selftest_wait_kernel(unsigned int* err, uint32_t polls) {
    __shared__ __align__(8) uint64_t mbar;
    const uint32_t a = smem_u32(&mbar);
    if (threadIdx.x == 0) {
        tc::mbar_init(a, 1);
        tc::mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait(a, 0, polls)) atomicOr(err, 1u);
}

}  // namespace
}  // namespace kvq8

extern "C" int kvq8_selftest_convert(int kind, const uint32_t* in, uint32_t* out, int n, kvq8_stream_t stream) {
    if (kind < 0 || kind > 3 || n < 0 || (n > 0 && (!in || !out))) return KVQ8_ERR_INVALID_ARG;
    if (n == 0) return KVQ8_OK;
    if ((reinterpret_cast<uintptr_t>(in) & 3u) || (reinterpret_cast<uintptr_t>(out) & 3u)) return KVQ8_ERR_MISALIGNED;
    const int items = kind == 1 ? n / 2 : n;
    if (kind == 1 && (n & 1)) return KVQ8_ERR_INVALID_ARG;
    kvq8::selftest_convert_kernel<<<(items + kvq8::kSelfThreads - 1) / kvq8::kSelfThreads, kvq8::kSelfThreads, 0,
                                    (cudaStream_t)stream>>>(kind, in, out, items);
    return kvq8::launch_status();
}

extern "C" int kvq8_selftest_wait_timeout(int polls, kvq8_stream_t stream) {
    if (polls < 1 || polls > (1 << 20)) return KVQ8_ERR_INVALID_ARG;
    unsigned int* err = kvq8::device_error_flag();
    if (!err) return KVQ8_ERR_CUDA;
    kvq8::selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err, (uint32_t)polls);
    return kvq8::launch_status();
}
