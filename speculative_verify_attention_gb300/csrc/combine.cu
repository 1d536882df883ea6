// combine.cu -- log-sum-exp merge of split-context attention partials (attn_combine).
//
// Source: "perf(gfx1100): share Q8 KV scans across verifier rows", Summary: the
// split-context partials layout and its reducer.  Partial s of a row holds
// o_s = sum exp(s_n - m_s) v_n, m_s = max s_n (natural-log units) and l_s = sum exp(s_n - m_s);
// the merge is out = sum_s o_s e^(m_s - m*) / sum_s l_s e^(m_s - m*) with m* = max_s m_s.
//
// Launch shape: blocks of 256 threads = 32 column threads (one float4 of the row each) x 8
// split groups (one warp each); a row of HD floats takes ceil(HD/128) blocks.  Every load a
// block needs -- the (m, l) of all splits and each thread's first kPrefetch partial vectors --
// is issued before any of them is used, so a row costs about one memory round trip plus two
// block reductions.  The split groups' sums are added in shared memory at the end.
// With few splits and many rows (the prompt path) a flat kernel is used instead: one thread
// per four float4s of a row, looping over the splits.
#include "common.cuh"

namespace kvq8 {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kColThreads = 32;
constexpr int kSplitGroups = kCombineThreads / kColThreads;
constexpr int kPrefetch = 12;      // partial vectors per thread loaded up front
constexpr int kMaxSplits = 4096;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* s_red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float u = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmaxf(v, u) : v + u;
    }
    __syncthreads();  // s_red may still be read by a previous reduction
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    float r = s_red[0];
#pragma unroll
    for (int w = 1; w < kCombineThreads / 32; ++w) r = is_max ? fmaxf(r, s_red[w]) : r + s_red[w];
    return r;
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const float4* __restrict__ part_o,
                                                                  const float2* __restrict__ part_ml, int n_split,
                                                                  int rows, int hd4, float* __restrict__ out) {
    extern __shared__ float2 s_wl[];  // [n_split]: (m, l), then (weight, l)
    __shared__ float s_red[kCombineThreads / 32];
    __shared__ float4 s_acc[kSplitGroups - 1][kColThreads];
    const int row = blockIdx.x, tid = threadIdx.x;
    const int cl = tid % kColThreads, sg = tid / kColThreads;
    const int c = blockIdx.y * kColThreads + cl;
    const bool col_ok = c < hd4;
    const int64_t stride = (int64_t)rows * hd4;  // float4s between consecutive splits
    const float4* src = part_o + (int64_t)row * hd4 + c;
    // launched as a programmatic dependent of the split kernel: wait until its partials are complete
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the next call's split kernel may start its prologue now: every kernel before this one has
    // completed, and it writes no partials before its own wait for this grid
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    float4 o[kPrefetch];
#pragma unroll
    for (int k = 0; k < kPrefetch; ++k) {
        const int s = sg + k * kSplitGroups;
        o[k] = (col_ok && s < n_split) ? __ldg(src + s * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mx = -INFINITY;
    for (int s = tid; s < n_split; s += kCombineThreads) {
        const float2 ml = __ldg(part_ml + (int64_t)s * rows + row);
        s_wl[s] = ml;
        mx = fmaxf(mx, ml.x);
    }
    const float ms = block_reduce(mx, true, s_red);  // its barriers also publish s_wl
    float lsum = 0.0f;
    for (int s = tid; s < n_split; s += kCombineThreads) {
        const float2 ml = s_wl[s];
        const float w = (ms == -INFINITY || ml.x == -INFINITY) ? 0.0f : expf(ml.x - ms);
        s_wl[s].x = w;
        lsum += w * ml.y;
    }
    const float l = block_reduce(lsum, false, s_red);  // its barriers also publish the weights
    const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;

    // a partial with weight 0 (no keys: m = -inf) is skipped, never multiplied: its o slot
    // may hold anything
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kPrefetch; ++k) {
        const int s = sg + k * kSplitGroups;
        const float w = s < n_split ? s_wl[s].x : 0.0f;
        if (w == 0.0f) continue;
        acc.x = fmaf(w, o[k].x, acc.x);
        acc.y = fmaf(w, o[k].y, acc.y);
        acc.z = fmaf(w, o[k].z, acc.z);
        acc.w = fmaf(w, o[k].w, acc.w);
    }
    if (col_ok) {  // splits past the prefetched ones: four loads in flight per step
        for (int s0 = sg + kPrefetch * kSplitGroups; s0 < n_split; s0 += 4 * kSplitGroups) {
            float w[4];
            float4 v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int s = s0 + k * kSplitGroups;
                w[k] = s < n_split ? s_wl[s].x : 0.0f;
                v[k] = w[k] != 0.0f ? __ldg(src + s * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc.x = fmaf(w[k], v[k].x, acc.x);
                acc.y = fmaf(w[k], v[k].y, acc.y);
                acc.z = fmaf(w[k], v[k].z, acc.z);
                acc.w = fmaf(w[k], v[k].w, acc.w);
            }
        }
    }
    if (sg > 0) s_acc[sg - 1][cl] = acc;
    __syncthreads();
    if (sg == 0 && col_ok) {
#pragma unroll
        for (int k = 0; k < kSplitGroups - 1; ++k) {
            const float4 a = s_acc[k][cl];
            acc.x += a.x;
            acc.y += a.y;
            acc.z += a.z;
            acc.w += a.w;
        }
        reinterpret_cast<float4*>(out + (int64_t)row * (hd4 * 4))[c] =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
}

// Few splits, many rows (the prompt path): a thread takes kWideVec consecutive float4s of one
// row and loops over the splits itself, with every load of the row issued before use.
constexpr int kWideMaxSplits = 4;
constexpr int kWideThreads = 256;
constexpr int kWideVec = 4;

__global__ void __launch_bounds__(kWideThreads) combine_wide_kernel(const float4* __restrict__ part_o,
                                                                    const float2* __restrict__ part_ml,
                                                                    int n_split, int rows, int hd4,
                                                                    float* __restrict__ out) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int per_row = hd4 / kWideVec;
    const int64_t item = (int64_t)blockIdx.x * kWideThreads + threadIdx.x;
    if (item >= (int64_t)rows * per_row) return;
    const int row = (int)(item / per_row);
    const int64_t idx = (int64_t)row * hd4 + (int64_t)(item - (int64_t)row * per_row) * kWideVec;
    const int64_t stride = (int64_t)rows * hd4;
    float2 ml[kWideMaxSplits];
    float4 o[kWideMaxSplits][kWideVec];
    float ms = -INFINITY;
#pragma unroll
    for (int s = 0; s < kWideMaxSplits; ++s) {
        if (s < n_split) {
            ml[s] = __ldg(part_ml + (int64_t)s * rows + row);
#pragma unroll
            for (int v = 0; v < kWideVec; ++v) o[s][v] = __ldg(part_o + idx + s * stride + v);
            ms = fmaxf(ms, ml[s].x);
        }
    }
    float l = 0.0f;
    float4 acc[kWideVec];
#pragma unroll
    for (int v = 0; v < kWideVec; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < kWideMaxSplits; ++s) {
        if (s < n_split) {
            const float w = (ms == -INFINITY || ml[s].x == -INFINITY) ? 0.0f : expf(ml[s].x - ms);
            if (w == 0.0f) continue;  // an empty partial's o slot may hold anything
            l = fmaf(w, ml[s].y, l);
#pragma unroll
            for (int v = 0; v < kWideVec; ++v) {
                acc[v].x = fmaf(w, o[s][v].x, acc[v].x);
                acc[v].y = fmaf(w, o[s][v].y, acc[v].y);
                acc[v].z = fmaf(w, o[s][v].z, acc[v].z);
                acc[v].w = fmaf(w, o[s][v].w, acc[v].w);
            }
        }
    }
    const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
    float4* dst = reinterpret_cast<float4*>(out) + idx;
#pragma unroll
    for (int v = 0; v < kWideVec; ++v)
        dst[v] = make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv, acc[v].w * inv);
}

}  // namespace

int launch_combine(const float* part_o, const float* part_ml, int n_split, int rows, int head_dim, float* out,
                   cudaStream_t stream) {
    if (rows == 0) return KVQ8_OK;
    const int hd4 = head_dim / 4;
    // Programmatic dependent launch: the grid may be scheduled while the kernel before it in
    // the stream is still running; griddepcontrol.wait in the kernel orders the reads.
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    const int64_t threads = (int64_t)rows * (hd4 / kWideVec);
    if (n_split <= kWideMaxSplits && hd4 % kWideVec == 0 && threads >= (1 << 16)) {  // many rows
        cfg.gridDim = dim3((unsigned)((threads + kWideThreads - 1) / kWideThreads));
        cfg.blockDim = dim3(kWideThreads);
        cfg.dynamicSmemBytes = 0;
        e = cudaLaunchKernelEx(&cfg, combine_wide_kernel, reinterpret_cast<const float4*>(part_o),
                               reinterpret_cast<const float2*>(part_ml), n_split, rows, hd4, out);
    } else {
        cfg.gridDim = dim3(rows, (hd4 + kColThreads - 1) / kColThreads);
        cfg.blockDim = dim3(kCombineThreads);
        cfg.dynamicSmemBytes = (size_t)n_split * sizeof(float2);
        e = cudaLaunchKernelEx(&cfg, combine_kernel, reinterpret_cast<const float4*>(part_o),
                               reinterpret_cast<const float2*>(part_ml), n_split, rows, hd4, out);
    }
    return e == cudaSuccess ? KVQ8_OK : KVQ8_ERR_CUDA;
}

}  // namespace kvq8

extern "C" int attn_combine(const float* part_o, const float* part_ml, int n_split, int rows, int head_dim,
                            float* out, kvq8_stream_t stream) {
    using namespace kvq8;
    if (n_split < 1 || n_split > kMaxSplits || rows < 0 || head_dim <= 0) return KVQ8_ERR_INVALID_ARG;
    if (head_dim % 4 || head_dim > 1024) return KVQ8_ERR_UNSUPPORTED;
    if (rows == 0) return KVQ8_OK;
    if (!part_o || !part_ml || !out) return KVQ8_ERR_INVALID_ARG;
    if (!aligned16(part_o) || !aligned16(part_ml) || !aligned16(out)) return KVQ8_ERR_MISALIGNED;
    return launch_combine(part_o, part_ml, n_split, rows, head_dim, out, (cudaStream_t)stream);
}
