// combine.cu -- log-sum-exp merge of split-context attention partials (attn_combine).
//
// Source: "perf(gfx1100): share Q8 KV scans across verifier rows", Summary: the
// split-context partials layout and its reducer.  Partial s of a row holds
// o_s = sum exp(s_n - m_s) v_n, m_s = max s_n (natural-log units) and l_s = sum exp(s_n - m_s);
// the merge is out = sum_s o_s e^(m_s - m*) / sum_s l_s e^(m_s - m*) with m* = max_s m_s.
#include "common.cuh"

namespace kvq8 {

// One thread block per row; thread c handles columns 4c..4c+3.  Every thread reads the
// n_split (m, l) pairs (a few KB, L1/L2 resident), then streams its float4 column slice.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ part_o,
                                                      const float2* __restrict__ part_ml, int n_split,
                                                      int rows, int hd4, float* __restrict__ out) {
    const int row = blockIdx.x;
    const int c = threadIdx.x;
    float ms = -INFINITY;
    for (int s = 0; s < n_split; ++s) ms = fmaxf(ms, __ldg(part_ml + (int64_t)s * rows + row).x);
    if (c >= hd4) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.0f;
    if (ms != -INFINITY) {
        for (int s = 0; s < n_split; ++s) {
            const float2 ml = __ldg(part_ml + (int64_t)s * rows + row);
            const float w = expf(ml.x - ms);  // 0 for an empty slice (m = -inf)
            if (w == 0.0f) continue;
            const float4 o = __ldg(reinterpret_cast<const float4*>(part_o + ((int64_t)s * rows + row) * (hd4 * 4)) + c);
            acc.x += w * o.x;
            acc.y += w * o.y;
            acc.z += w * o.z;
            acc.w += w * o.w;
            l += w * ml.y;
        }
        const float inv = 1.0f / l;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
    }
    reinterpret_cast<float4*>(out + (int64_t)row * (hd4 * 4))[c] = acc;
}

int launch_combine(const float* part_o, const float* part_ml, int n_split, int rows, int head_dim, float* out,
                   cudaStream_t stream) {
    if (rows == 0) return KVQ8_OK;
    const int hd4 = head_dim / 4;
    const int threads = ((hd4 + 31) / 32) * 32;
    combine_kernel<<<rows, threads, 0, stream>>>(part_o, reinterpret_cast<const float2*>(part_ml), n_split, rows,
                                                 hd4, out);
    return launch_status();
}

}  // namespace kvq8

extern "C" int attn_combine(const float* part_o, const float* part_ml, int n_split, int rows, int head_dim,
                            float* out, kvq8_stream_t stream) {
    using namespace kvq8;
    if (n_split < 1 || n_split > 4096 || rows < 0 || head_dim <= 0) return KVQ8_ERR_INVALID_ARG;
    if (head_dim % 4 || head_dim > 1024) return KVQ8_ERR_UNSUPPORTED;
    if (rows == 0) return KVQ8_OK;
    if (!part_o || !part_ml || !out) return KVQ8_ERR_INVALID_ARG;
    if (!aligned16(part_o) || !aligned16(part_ml) || !aligned16(out)) return KVQ8_ERR_MISALIGNED;
    return launch_combine(part_o, part_ml, n_split, rows, head_dim, out, (cudaStream_t)stream);
}
