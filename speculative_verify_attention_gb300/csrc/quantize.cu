// quantize.cu -- Q8_0 quantiser for KV-cache appends (kvq8_quantize).
//
// Source: "Engine perf(hip): MTP draft, shared expert, verify/sampler head", Summary item 4:
// a warp-per-block quantiser that reduces max|x| over the 32-value block with shuffles
// and writes the fp16 scale and 32 int8 codes, bitwise equal to its CPU reference.
//
// Here a warp covers four blocks: eight lanes per block, four values per lane (one
// 16-byte load), a 3-step shuffle max, then per value an IEEE fp32 division and round
// half away from zero (q8_0_block).  Bandwidth-bound: 4 bytes read, 1 + 1/16 bytes
// written per value.
// kvq8_append writes both planes (K and V) of a cache in one launch; kvk8v4_append does the
// same for a K8V4 pool (K as Q8_0, V as 4-bit blocks, q4_block).
#include "common.cuh"
#include "q8_0.cuh"

namespace kvq8 {
namespace {

// Plane 0 (x0 -> codes0/scales0) holds blocks [0, n_blocks); when x1 is given, plane 1
// (x1 -> codes1/scales1) holds blocks [n_blocks, 2 n_blocks) of the same launch.
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const float4* __restrict__ x0,
                                                            const float4* __restrict__ x1, int64_t n_blocks,
                                                            int n_kv_heads, int nb_per_head_row,
                                                            int8_t* __restrict__ codes0,
                                                            uint16_t* __restrict__ scales0,
                                                            int8_t* __restrict__ codes1,
                                                            uint16_t* __restrict__ scales1, int capacity,
                                                            int pos0) {
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t blk_all = gid >> 3;  // Q8_0 block handled by this lane's group of 8
    const bool second = blk_all >= n_blocks;
    const int64_t blk = second ? blk_all - n_blocks : blk_all;
    const float4* x = second ? x1 : x0;
    int8_t* codes = second ? codes1 : codes0;
    uint16_t* scales = second ? scales1 : scales0;
    const int sub = threadIdx.x & 7;
    const bool live = blk_all < (x1 ? 2 * n_blocks : n_blocks);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) v = __ldg(x + blk * 8 + sub);
    uint16_t scale_bits;
    const uint32_t packed = q8_0_block(v, &scale_bits);
    if (!live) return;

    // block index -> (token, kv head, block within the head row)
    const int64_t row_blocks = (int64_t)n_kv_heads * nb_per_head_row;
    const int64_t tok = blk / row_blocks;
    const int64_t rem = blk - tok * row_blocks;
    const int h = (int)(rem / nb_per_head_row);
    const int b = (int)(rem - (int64_t)h * nb_per_head_row);
    const int64_t row = (int64_t)h * capacity + pos0 + tok;
    int8_t* dst = codes + row * (int64_t)nb_per_head_row * kQBlock + b * kQBlock + sub * 4;
    *reinterpret_cast<uint32_t*>(dst) = packed;
    if (sub == 0) scales[row * nb_per_head_row + b] = scale_bits;
}

}  // namespace
}  // namespace kvq8

namespace kvq8 {
namespace {

int launch_quantize(const float* x0, const float* x1, int n_tok, int n_kv_heads, int head_dim, int8_t* codes0,
                    uint16_t* scales0, int8_t* codes1, uint16_t* scales1, int capacity, int pos0,
                    cudaStream_t stream) {
    const int nb = head_dim / kQBlock;
    const int64_t n_blocks = (int64_t)n_tok * n_kv_heads * nb;
    const int64_t threads = n_blocks * 8 * (x1 ? 2 : 1);
    const int64_t grid = (threads + 255) / 256;
    if (grid > 0x7fffffffLL) return KVQ8_ERR_UNSUPPORTED;
    quantize_q8_0_kernel<<<(unsigned)grid, 256, 0, stream>>>(reinterpret_cast<const float4*>(x0),
                                                           reinterpret_cast<const float4*>(x1), n_blocks,
                                                           n_kv_heads, nb, codes0, scales0, codes1, scales1,
                                                           capacity, pos0);
    return launch_status();
}

// K8V4 append: blocks [0, n_blocks) are K (Q8_0), [n_blocks, 2 n_blocks) V (4-bit), one
// 8-lane group per 32-value block as in the Q8_0 kernel.
__global__ void __launch_bounds__(256) append_k8v4_kernel(const float4* __restrict__ k, const float4* __restrict__ v,
                                                          int64_t n_blocks, int n_kv_heads, int nb_per_head_row,
                                                          int8_t* __restrict__ k_codes, uint16_t* __restrict__ k_scales,
                                                          uint8_t* __restrict__ v_codes,
                                                          uint16_t* __restrict__ v_scales, int capacity, int pos0) {
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t blk_all = gid >> 3;
    const bool is_v = blk_all >= n_blocks;
    const int64_t blk = is_v ? blk_all - n_blocks : blk_all;
    const int sub = threadIdx.x & 7;
    const bool live = blk_all < 2 * n_blocks;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) x = __ldg((is_v ? v : k) + blk * 8 + sub);
    // both quantisers run on every lane (their shuffles stay inside the lane's 8-lane group)
    // and each lane keeps its own plane's result
    uint16_t sq8, sq4;
    const uint32_t p8 = q8_0_block(x, &sq8);
    const uint32_t p4 = q4_block(x, &sq4);
    if (!live) return;
    const int64_t row_blocks = (int64_t)n_kv_heads * nb_per_head_row;
    const int64_t tok = blk / row_blocks;
    const int64_t rem = blk - tok * row_blocks;
    const int h = (int)(rem / nb_per_head_row);
    const int b = (int)(rem - (int64_t)h * nb_per_head_row);
    const int64_t row = (int64_t)h * capacity + pos0 + tok;
    if (!is_v) {
        *reinterpret_cast<uint32_t*>(k_codes + row * (int64_t)nb_per_head_row * kQBlock + b * kQBlock + sub * 4) = p8;
        if (sub == 0) k_scales[row * nb_per_head_row + b] = sq8;
    } else {
        *reinterpret_cast<uint16_t*>(v_codes + row * (int64_t)nb_per_head_row * (kQBlock / 2) + b * (kQBlock / 2) +
                                     sub * 2) = (uint16_t)p4;
        if (sub == 0) v_scales[row * nb_per_head_row + b] = sq4;
    }
}

}  // namespace
}  // namespace kvq8

extern "C" int kvk8v4_append(const float* k, const float* v, int n_tok, const kvk8v4_cache* kv, int pos0,
                             kvq8_stream_t stream) {
    using namespace kvq8;
    if (!kv || n_tok < 0 || pos0 < 0) return KVQ8_ERR_INVALID_ARG;
    if (kv->n_kv_heads <= 0 || kv->head_dim <= 0 || kv->capacity <= 0) return KVQ8_ERR_INVALID_ARG;
    if (kv->head_dim % kQBlock) return KVQ8_ERR_UNSUPPORTED;
    if ((int64_t)pos0 + n_tok > kv->capacity) return KVQ8_ERR_INVALID_ARG;
    if (n_tok == 0) return KVQ8_OK;
    if (!k || !v || !kv->k_codes || !kv->k_scales || !kv->v_codes || !kv->v_scales) return KVQ8_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(kv->k_codes) || !aligned16(kv->k_scales) ||
        !aligned16(kv->v_codes) || !aligned16(kv->v_scales))
        return KVQ8_ERR_MISALIGNED;
    const int nb = kv->head_dim / kQBlock;
    const int64_t n_blocks = (int64_t)n_tok * kv->n_kv_heads * nb;
    const int64_t grid = (n_blocks * 16 + 255) / 256;
    if (grid > 0x7fffffffLL) return KVQ8_ERR_UNSUPPORTED;
    append_k8v4_kernel<<<(unsigned)grid, 256, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const float4*>(k), reinterpret_cast<const float4*>(v), n_blocks, kv->n_kv_heads, nb,
        const_cast<int8_t*>(kv->k_codes), const_cast<uint16_t*>(kv->k_scales), const_cast<uint8_t*>(kv->v_codes),
        const_cast<uint16_t*>(kv->v_scales), kv->capacity, pos0);
    return launch_status();
}

extern "C" int kvq8_quantize(const float* x, int n_tok, int n_kv_heads, int head_dim, int8_t* codes,
                             uint16_t* scales, int capacity, int pos0, kvq8_stream_t stream) {
    using namespace kvq8;
    if (n_tok < 0 || n_kv_heads <= 0 || head_dim <= 0 || capacity <= 0 || pos0 < 0) return KVQ8_ERR_INVALID_ARG;
    if (head_dim % kQBlock) return KVQ8_ERR_UNSUPPORTED;
    if ((int64_t)pos0 + n_tok > capacity) return KVQ8_ERR_INVALID_ARG;
    if (n_tok == 0) return KVQ8_OK;
    if (!x || !codes || !scales) return KVQ8_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return KVQ8_ERR_MISALIGNED;
    return launch_quantize(x, nullptr, n_tok, n_kv_heads, head_dim, codes, scales, nullptr, nullptr, capacity, pos0,
                           (cudaStream_t)stream);
}

extern "C" int kvq8_append(const float* k, const float* v, int n_tok, const kvq8_cache* kv, int pos0,
                           kvq8_stream_t stream) {
    using namespace kvq8;
    if (!kv || n_tok < 0 || pos0 < 0) return KVQ8_ERR_INVALID_ARG;
    if (kv->n_kv_heads <= 0 || kv->head_dim <= 0 || kv->capacity <= 0) return KVQ8_ERR_INVALID_ARG;
    if (kv->head_dim % kQBlock) return KVQ8_ERR_UNSUPPORTED;
    if ((int64_t)pos0 + n_tok > kv->capacity) return KVQ8_ERR_INVALID_ARG;
    if (n_tok == 0) return KVQ8_OK;
    if (!k || !v || !kv->k_codes || !kv->k_scales || !kv->v_codes || !kv->v_scales) return KVQ8_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(kv->k_codes) || !aligned16(kv->k_scales) ||
        !aligned16(kv->v_codes) || !aligned16(kv->v_scales))
        return KVQ8_ERR_MISALIGNED;
    return launch_quantize(k, v, n_tok, kv->n_kv_heads, kv->head_dim, const_cast<int8_t*>(kv->k_codes),
                           const_cast<uint16_t*>(kv->k_scales), const_cast<int8_t*>(kv->v_codes),
                           const_cast<uint16_t*>(kv->v_scales), kv->capacity, pos0, (cudaStream_t)stream);
}

extern "C" const char* kvq8_status_str(int status) {
    switch (status) {
        case KVQ8_OK: return "ok";
        case KVQ8_ERR_INVALID_ARG: return "invalid argument";
        case KVQ8_ERR_UNSUPPORTED: return "unsupported shape";
        case KVQ8_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case KVQ8_ERR_WORKSPACE: return "workspace missing or too small";
        case KVQ8_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}
