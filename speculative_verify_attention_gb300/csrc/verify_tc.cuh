// verify_tc.cuh -- parameters and launch of the tcgen05 verify scan (verify_tc.cu), called by
// the entry points in verify.cu.
#pragma once

#include "tmap.cuh"
#include "verify_plan.cuh"

namespace kvq8 {

struct VerifyTcParams {
    const float* q;
    int8_t* k_codes;     // written only by the window slice of the append path
    uint16_t* k_scales;
    int8_t* v_codes;
    uint16_t* v_scales;
    float* part_o;       // [n_split][rows_total][HD]
    float2* part_ml;     // [n_split][rows_total]
    const float* k_new;  // append path: fp32 [n_rows][n_kv_heads][HD] window keys and values
    const float* v_new;
    unsigned int* err;   // the library's timeout flag (set by launch_verify_tc)
    const uint32_t* wmask;  // tree windows: bit j of wmask[i] = row i sees key q_pos0 + j; null = causal
    int n_rows, n_q_heads, group, group_magic, capacity, kv_len, q_pos0, keys_per_split, key_shift, n_ctx_splits,
        n_kv_heads, rows_per_chunk;
    float qscale;        // softmax_scale * log2(e)
    CUtensorMap tmap_k;  // code planes as bytes: dims (HD, kv_len, n_kv_heads), box 128 x 128 x 1
    CUtensorMap tmap_v;  // (encoded by launch_verify_tc)
};

// The tcgen05 verify scan of one call planned with make_plan(..., tc_blocks_per_sm, kTcMaxRows):
// one launch writing the slices' partials; `append` selects the window-slice variant, `v4` the
// 4-bit V plane of a K8V4 pool (v_codes then holds hd/2 bytes per key; causal, hd256 only).
int launch_verify_tc(VerifyTcParams& vp, const Plan& pl, int n_kv_heads, bool append, bool v4, cudaStream_t s);

}  // namespace kvq8
