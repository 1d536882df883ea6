// quantize.cu -- Q8_0 quantiser for KV-cache appends (kvq8_quantize).
//
// Source: "Engine perf(hip): MTP draft, shared expert, verify/sampler head", Summary item 4:
// a warp-per-block quantiser that reduces max|x| over the 32-value block with shuffles
// and writes the fp16 scale and 32 int8 codes, bitwise equal to its CPU reference.
//
// Here a warp covers four blocks of a token row: eight lanes per block, four values per lane
// (one 16-byte load), a 3-step shuffle max, then per value an IEEE fp32 division and round
// half away from zero (q8_0_block).  A thread keeps one column for four tokens, so the
// (head, block) position is worked out once per thread.  Bandwidth-bound: 4 bytes read,
// 1 + 1/16 bytes written per value.
// kvq8_append writes both planes (K and V) of a cache in one launch; kvk8v4_append does the
// same for a K8V4 pool (K as Q8_0, V as 4-bit blocks, q4_block).
#include "common.cuh"
#include "q8_0.cuh"

namespace kvq8 {
namespace {

// Grid (token groups, column chunks, planes): a block quantises columns
// [256 y, 256 y + 256) of kTokPerBlock consecutive token rows of one plane (plane z: x0 ->
// codes0/scales0, or x1 -> codes1/scales1).  A row holds n_kv_heads * head_dim values, read as
// float4 column j: head j / (head_dim/4), block (j mod head_dim/4) / 8 of that head.  A thread
// keeps one column for all its tokens, so the (head, block) split is done once per thread; its
// kTokPerBlock loads are issued before any is used.  Lanes past the row or past the last
// token quantise zeros (every lane takes part in the block's shuffle max) and store nothing.
constexpr int kQuantThreads = 256;
constexpr int kTokPerBlock = 4;

__global__ void __launch_bounds__(kQuantThreads) quantize_q8_0_kernel(const float4* __restrict__ x0,
                                                                      const float4* __restrict__ x1, int n_tok,
                                                                      int n_kv_heads, int head_dim,
                                                                      int8_t* __restrict__ codes0,
                                                                      uint16_t* __restrict__ scales0,
                                                                      int8_t* __restrict__ codes1,
                                                                      uint16_t* __restrict__ scales1, int capacity,
                                                                      int pos0) {
    const bool second = blockIdx.z != 0;
    const float4* x = second ? x1 : x0;
    int8_t* codes = second ? codes1 : codes0;
    uint16_t* scales = second ? scales1 : scales0;
    const int f4_head = head_dim / 4;
    const int row_f4 = n_kv_heads * f4_head;
    const int j = blockIdx.y * kQuantThreads + threadIdx.x;
    const bool col_ok = j < row_f4;
    const int h = j / f4_head, i = j - h * f4_head;  // head and float4 within the head row
    const int tok0 = blockIdx.x * kTokPerBlock;
    float4 v[kTokPerBlock];
#pragma unroll
    for (int t = 0; t < kTokPerBlock; ++t) {
        v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col_ok && tok0 + t < n_tok) v[t] = __ldg(x + (int64_t)(tok0 + t) * row_f4 + j);
    }
    const int nb = head_dim / kQBlock;
    const int64_t row0 = (int64_t)h * capacity + pos0 + tok0;  // cache row of the first token
#pragma unroll
    for (int t = 0; t < kTokPerBlock; ++t) {
        uint16_t scale_bits;
        const uint32_t packed = q8_0_block(v[t], &scale_bits);
        if (col_ok && tok0 + t < n_tok) {
            *reinterpret_cast<uint32_t*>(codes + (row0 + t) * head_dim + i * 4) = packed;
            if ((i & 7) == 0) scales[(row0 + t) * nb + (i >> 3)] = scale_bits;
        }
    }
}

}  // namespace
}  // namespace kvq8

namespace kvq8 {
namespace {

int launch_quantize(const float* x0, const float* x1, int n_tok, int n_kv_heads, int head_dim, int8_t* codes0,
                    uint16_t* scales0, int8_t* codes1, uint16_t* scales1, int capacity, int pos0,
                    cudaStream_t stream) {
    const int64_t row_f4 = (int64_t)n_kv_heads * head_dim / 4;
    const int64_t gy = (row_f4 + kQuantThreads - 1) / kQuantThreads;
    const int64_t gx = ((int64_t)n_tok + kTokPerBlock - 1) / kTokPerBlock;
    if (row_f4 > 0x7fffffffLL - kQuantThreads || gy > 65535) return KVQ8_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)gx, (unsigned)gy, x1 ? 2u : 1u);
    quantize_q8_0_kernel<<<grid, kQuantThreads, 0, stream>>>(reinterpret_cast<const float4*>(x0),
                                                             reinterpret_cast<const float4*>(x1), n_tok, n_kv_heads,
                                                             head_dim, codes0, scales0, codes1, scales1, capacity,
                                                             pos0);
    return launch_status();
}

// K8V4 append, the same grid: plane 0 quantises K to Q8_0, plane 1 V to 4-bit blocks.
__global__ void __launch_bounds__(kQuantThreads) append_k8v4_kernel(const float4* __restrict__ k,
                                                                    const float4* __restrict__ v, int n_tok,
                                                                    int n_kv_heads, int head_dim,
                                                                    int8_t* __restrict__ k_codes,
                                                                    uint16_t* __restrict__ k_scales,
                                                                    uint8_t* __restrict__ v_codes,
                                                                    uint16_t* __restrict__ v_scales, int capacity,
                                                                    int pos0) {
    const bool is_v = blockIdx.z != 0;
    const float4* x = is_v ? v : k;
    const int f4_head = head_dim / 4;
    const int row_f4 = n_kv_heads * f4_head;
    const int j = blockIdx.y * kQuantThreads + threadIdx.x;
    const bool col_ok = j < row_f4;
    const int h = j / f4_head, i = j - h * f4_head;
    const int tok0 = blockIdx.x * kTokPerBlock;
    float4 xv[kTokPerBlock];
#pragma unroll
    for (int t = 0; t < kTokPerBlock; ++t) {
        xv[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col_ok && tok0 + t < n_tok) xv[t] = __ldg(x + (int64_t)(tok0 + t) * row_f4 + j);
    }
    const int nb = head_dim / kQBlock;
    const int64_t row0 = (int64_t)h * capacity + pos0 + tok0;
#pragma unroll
    for (int t = 0; t < kTokPerBlock; ++t) {
        const bool st = col_ok && tok0 + t < n_tok;
        uint16_t sc;
        if (!is_v) {  // uniform per block: every lane of a warp runs the same quantiser
            const uint32_t p8 = q8_0_block(xv[t], &sc);
            if (st) {
                *reinterpret_cast<uint32_t*>(k_codes + (row0 + t) * head_dim + i * 4) = p8;
                if ((i & 7) == 0) k_scales[(row0 + t) * nb + (i >> 3)] = sc;
            }
        } else {
            const uint32_t p4 = q4_block(xv[t], &sc);
            if (st) {
                *reinterpret_cast<uint16_t*>(v_codes + (row0 + t) * (head_dim / 2) + i * 2) = (uint16_t)p4;
                if ((i & 7) == 0) v_scales[(row0 + t) * nb + (i >> 3)] = sc;
            }
        }
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
    const int64_t row_f4 = (int64_t)kv->n_kv_heads * kv->head_dim / 4;
    const int64_t gy = (row_f4 + kQuantThreads - 1) / kQuantThreads;
    const int64_t gx = ((int64_t)n_tok + kTokPerBlock - 1) / kTokPerBlock;
    if (row_f4 > 0x7fffffffLL - kQuantThreads || gy > 65535) return KVQ8_ERR_UNSUPPORTED;
    append_k8v4_kernel<<<dim3((unsigned)gx, (unsigned)gy, 2u), kQuantThreads, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const float4*>(k), reinterpret_cast<const float4*>(v), n_tok, kv->n_kv_heads, kv->head_dim,
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
