// combine.cu -- log-sum-exp merge of split-context attention partials (attn_combine).
//
// Source: "perf(gfx1100): share Q8 KV scans across verifier rows", Summary: the
// split-context partials layout and its reducer.  Partial s of a row holds
// o_s = sum exp(s_n - m_s) v_n, m_s = max s_n (natural-log units) and l_s = sum exp(s_n - m_s);
// the merge is out = sum_s o_s e^(m_s - m*) / sum_s l_s e^(m_s - m*) with m* = max_s m_s.
//
// One 256-thread block per row.  The block loads all (m_s, l_s) of its row in parallel,
// reduces m*, and keeps the weights w_s = e^(m_s - m*) in shared memory.  The o_s are then
// read by 64 column threads x 4 split groups, each thread with four independent loads in
// flight, and the four group sums are added in shared memory -- so a row costs a few
// memory round trips, not one per split.
#include "common.cuh"

namespace kvq8 {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kColThreads = 64;
constexpr int kSplitGroups = kCombineThreads / kColThreads;
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

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const float* __restrict__ part_o,
                                                                  const float2* __restrict__ part_ml, int n_split,
                                                                  int rows, int hd4, float* __restrict__ out) {
    __shared__ float s_w[kMaxSplits];
    __shared__ float s_red[kCombineThreads / 32];
    __shared__ float4 s_acc[kSplitGroups - 1][kColThreads];
    const int row = blockIdx.x, tid = threadIdx.x;

    float mx = -INFINITY;
    for (int s = tid; s < n_split; s += kCombineThreads) {
        const float m = __ldg(part_ml + (int64_t)s * rows + row).x;
        s_w[s] = m;
        mx = fmaxf(mx, m);
    }
    const float ms = block_reduce(mx, true, s_red);

    float lsum = 0.0f;
    for (int s = tid; s < n_split; s += kCombineThreads) {
        const float m = s_w[s];
        const float w = (ms == -INFINITY || m == -INFINITY) ? 0.0f : expf(m - ms);
        s_w[s] = w;
        if (w != 0.0f) lsum += w * __ldg(part_ml + (int64_t)s * rows + row).y;
    }
    const float l = block_reduce(lsum, false, s_red);  // its barriers also publish s_w
    const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;

    const int cl = tid % kColThreads, sg = tid / kColThreads;
    const int64_t stride = (int64_t)rows * hd4;
    for (int c0 = 0; c0 < hd4; c0 += kColThreads) {
        const int c = c0 + cl;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < hd4) {
            const float4* src = reinterpret_cast<const float4*>(part_o) + (int64_t)row * hd4 + c;
            int s = sg;
            for (; s + 3 * kSplitGroups < n_split; s += 4 * kSplitGroups) {
                float w[4];
                float4 o[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    w[k] = s_w[s + k * kSplitGroups];
                    o[k] = w[k] != 0.0f ? __ldg(src + (s + k * kSplitGroups) * stride)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    acc.x = fmaf(w[k], o[k].x, acc.x);
                    acc.y = fmaf(w[k], o[k].y, acc.y);
                    acc.z = fmaf(w[k], o[k].z, acc.z);
                    acc.w = fmaf(w[k], o[k].w, acc.w);
                }
            }
            for (; s < n_split; s += kSplitGroups) {
                const float w = s_w[s];
                if (w == 0.0f) continue;
                const float4 o = __ldg(src + s * stride);
                acc.x = fmaf(w, o.x, acc.x);
                acc.y = fmaf(w, o.y, acc.y);
                acc.z = fmaf(w, o.z, acc.z);
                acc.w = fmaf(w, o.w, acc.w);
            }
        }
        if (sg > 0) s_acc[sg - 1][cl] = acc;
        __syncthreads();
        if (sg == 0 && c < hd4) {
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
        __syncthreads();
    }
}

}  // namespace

int launch_combine(const float* part_o, const float* part_ml, int n_split, int rows, int head_dim, float* out,
                   cudaStream_t stream) {
    if (rows == 0) return KVQ8_OK;
    combine_kernel<<<rows, kCombineThreads, 0, stream>>>(part_o, reinterpret_cast<const float2*>(part_ml), n_split,
                                                         rows, head_dim / 4, out);
    return launch_status();
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
