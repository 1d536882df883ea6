// head.cu -- verify-head acceptance (argmax_rows_top_prob): per row of [T][V] fp32 logits, the
// index of the maximum and the top probability softmax(row)[argmax].
//
// Source: "Engine perf(hip): MTP draft, shared expert, verify/sampler head", Summary item 1
// (multi-block argmax_rows and row_top_prob_split over T x 248,320 logits) and "Verification
// & Parity Evidence" (ties, NaN and -inf cases).  Readings where the pages give no rule: ties
// go to the smallest index; NaN ranks above every number (argmax = first NaN, probability
// NaN); +inf entries share the row's probability mass; a row of -inf only is the uniform
// limit (argmax 0, probability 1/V).
//
// One read of the logits computes both results.  Every thread reduces the logits it holds in
// registers to an accumulator -- the maximum m, the first index of m, s = sum exp(x - m) and
// the first NaN index -- and accumulators merge (s rescaled to the larger m), first across
// the warp, then across the block, then across the blocks of a row (second kernel, launched
// as a programmatic dependent).  HBM-bound: 4 bytes read per logit.
#include <climits>

#include "common.cuh"

namespace kvq8 {
namespace {

constexpr int kHeadThreads = 256;
constexpr int kMergeThreads = 128;

struct HeadAcc {
    float m;   // running maximum (-inf: nothing but -inf seen)
    float s;   // sum of exp(x - m) over the non-NaN elements
    int idx;   // first index holding m (INT_MAX: none)
    int nan;   // first NaN index (INT_MAX: none)
};

__device__ __forceinline__ HeadAcc acc_empty() { return HeadAcc{-INFINITY, 0.0f, INT_MAX, INT_MAX}; }

__device__ __forceinline__ HeadAcc acc_merge(const HeadAcc& a, const HeadAcc& b) {
    HeadAcc r;
    r.nan = min(a.nan, b.nan);
    if (a.m > b.m) {
        r.m = a.m;
        r.idx = a.idx;
        r.s = a.s + (b.m == -INFINITY ? 0.0f : b.s * __expf(b.m - a.m));
    } else if (b.m > a.m) {
        r.m = b.m;
        r.idx = b.idx;
        r.s = b.s + (a.m == -INFINITY ? 0.0f : a.s * __expf(a.m - b.m));
    } else {
        r.m = a.m;
        r.idx = min(a.idx, b.idx);
        r.s = a.s + b.s;
    }
    return r;
}

__device__ __forceinline__ HeadAcc acc_shfl_xor(const HeadAcc& a, int o) {
    HeadAcc b;
    b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
    b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
    b.idx = __shfl_xor_sync(0xffffffffu, a.idx, o);
    b.nan = __shfl_xor_sync(0xffffffffu, a.nan, o);
    return b;
}

// Accumulator of one thread's N register-resident logits, x[i] at index jx(i) (increasing in
// i): a pass for the maximum and its first index (predicated, no branches), a pass for
// s = sum 2^((x - m) log2 e), and a NaN scan only where the sum says there is one or the
// maximum is infinite (the rare cases).
template <int N, typename JF>
__device__ __forceinline__ HeadAcc acc_of(const float (&x)[N], JF jx) {
    float m = -INFINITY;
    int idx = INT_MAX;
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (x[i] > m) {
            m = x[i];
            idx = jx(i);
        }
    HeadAcc a{m, 0.0f, idx, INT_MAX};
    bool scan = true;
    if (m == INFINITY) {  // the +inf entries share the mass
#pragma unroll
        for (int i = 0; i < N; ++i) a.s += x[i] == INFINITY ? 1.0f : 0.0f;
    } else if (m != -INFINITY) {
        float sum = 0.0f;
#pragma unroll
        for (int i = 0; i < N; ++i) sum += ex2_approx((x[i] - m) * kLog2e);
        a.s = sum;
        scan = sum != sum;  // a NaN among the values makes the sum NaN
    }
    if (scan) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (x[i] != x[i]) a.nan = min(a.nan, jx(i));
    }
    return a;
}

template <int THREADS>
__device__ __forceinline__ HeadAcc block_merge(HeadAcc a, HeadAcc* s_acc) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = acc_merge(a, acc_shfl_xor(a, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) s_acc[warp] = a;
    __syncthreads();
    HeadAcc r = s_acc[0];
#pragma unroll
    for (int w = 1; w < THREADS / 32; ++w) r = acc_merge(r, s_acc[w]);
    return r;
}

// Block (b, row) reduces logits [b * chunk, min(V, (b + 1) * chunk)) of its row into one
// accumulator.  Each thread issues all of its loads before using any (kPer of them, 16-byte
// ones when VEC: V % 4 == 0 and the rows 16-byte aligned); lanes past the end load -inf,
// which changes no accumulator.
constexpr int kPer = 8;
constexpr int kChunkVec = 4 * kHeadThreads * kPer;    // logits per block, 16-byte loads
constexpr int kChunkScalar = kHeadThreads * kPer;     // logits per block, 4-byte loads

template <bool VEC>
__global__ void __launch_bounds__(kHeadThreads) head_partial_kernel(const float* __restrict__ logits, int vocab,
                                                                    HeadAcc* __restrict__ part) {
    __shared__ HeadAcc s_acc[kHeadThreads / 32];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int b = blockIdx.x, row = blockIdx.y;
    const float* x = logits + (int64_t)row * vocab;
    HeadAcc a = acc_empty();
    if (VEC) {
        const float4* x4 = reinterpret_cast<const float4*>(x);
        const int e4 = vocab >> 2;
        const int k0 = b * (kChunkVec / 4) + threadIdx.x;
        float v[4 * kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int k = k0 + u * kHeadThreads;
            const float4 f = k < e4 ? __ldg(x4 + k) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            v[4 * u] = f.x;
            v[4 * u + 1] = f.y;
            v[4 * u + 2] = f.z;
            v[4 * u + 3] = f.w;
        }
        a = acc_of(v, [&](int i) { return 4 * (k0 + (i >> 2) * kHeadThreads) + (i & 3); });
    } else {
        const int j0 = b * kChunkScalar + threadIdx.x;
        float v[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int j = j0 + u * kHeadThreads;
            v[u] = j < vocab ? __ldg(x + j) : -INFINITY;
        }
        a = acc_of(v, [&](int i) { return j0 + i * kHeadThreads; });
    }
    a = block_merge<kHeadThreads>(a, s_acc);
    if (threadIdx.x == 0) part[(int64_t)row * gridDim.x + b] = a;
}

__device__ __forceinline__ void head_write(const HeadAcc& a, int vocab, int row, int32_t* argmax, float* top_prob) {
    if (a.nan != INT_MAX) {
        argmax[row] = a.nan;
        top_prob[row] = __int_as_float(0x7fc00000);  // quiet NaN
    } else if (a.m == -INFINITY) {
        argmax[row] = 0;
        top_prob[row] = 1.0f / (float)vocab;
    } else {
        argmax[row] = a.idx;
        top_prob[row] = 1.0f / a.s;
    }
}

__global__ void __launch_bounds__(kMergeThreads) head_merge_kernel(const HeadAcc* __restrict__ part, int n_blocks,
                                                                   int vocab, int32_t* __restrict__ argmax,
                                                                   float* __restrict__ top_prob) {
    __shared__ HeadAcc s_acc[kMergeThreads / 32];
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the partial kernel's results are complete
    const int row = blockIdx.x;
    HeadAcc a = acc_empty();
    for (int b = threadIdx.x; b < n_blocks; b += kMergeThreads) a = acc_merge(a, part[(int64_t)row * n_blocks + b]);
    a = block_merge<kMergeThreads>(a, s_acc);
    if (threadIdx.x == 0) head_write(a, vocab, row, argmax, top_prob);
}

bool head_vec(const float* logits, int vocab) { return vocab % 4 == 0 && aligned16(logits); }

// Blocks per row: one per chunk of the row.
int head_blocks(int vocab, bool vec) {
    const int chunk = vec ? kChunkVec : kChunkScalar;
    return (vocab + chunk - 1) / chunk;
}

}  // namespace
}  // namespace kvq8

extern "C" size_t argmax_rows_top_prob_workspace_bytes(int n_rows, int vocab) {
    if (n_rows < 1 || vocab < 1) return 0;
    // sized for the 4-byte-load form, which has the most blocks per row
    return (size_t)n_rows * kvq8::head_blocks(vocab, false) * sizeof(kvq8::HeadAcc);
}

extern "C" int argmax_rows_top_prob(const float* logits, int n_rows, int vocab, int32_t* argmax, float* top_prob,
                                    void* workspace, size_t workspace_bytes, kvq8_stream_t stream) {
    using namespace kvq8;
    if (n_rows < 1 || n_rows > 65535 || vocab < 1) return KVQ8_ERR_INVALID_ARG;
    if (!logits || !argmax || !top_prob) return KVQ8_ERR_INVALID_ARG;
    const bool vec = head_vec(logits, vocab);
    const int B = head_blocks(vocab, vec);
    if (!workspace || workspace_bytes < (size_t)n_rows * B * sizeof(HeadAcc)) return KVQ8_ERR_WORKSPACE;
    if (!aligned16(workspace)) return KVQ8_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(argmax) |
         reinterpret_cast<uintptr_t>(top_prob)) & 3u)
        return KVQ8_ERR_MISALIGNED;
    cudaStream_t s = (cudaStream_t)stream;
    HeadAcc* part = static_cast<HeadAcc*>(workspace);
    dim3 grid(B, n_rows);
    if (vec)
        head_partial_kernel<true><<<grid, kHeadThreads, 0, s>>>(logits, vocab, part);
    else
        head_partial_kernel<false><<<grid, kHeadThreads, 0, s>>>(logits, vocab, part);
    if (launch_status() != KVQ8_OK) return KVQ8_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_rows);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, head_merge_kernel, static_cast<const HeadAcc*>(part), B, vocab,
                                             argmax, top_prob);
    return e == cudaSuccess ? KVQ8_OK : KVQ8_ERR_CUDA;
}
