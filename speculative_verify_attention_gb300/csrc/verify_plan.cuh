// verify_plan.cuh -- how a multi-row verify call is cut into thread blocks: row chunks of at
// most 8 * kMaxNT (row, q-head) pairs per KV head, times context slices of whole 16-key units.
// Shared by the Q8_0 and the fp16-pool verify kernels.
#pragma once

#include <algorithm>

#include "common.cuh"

namespace kvq8 {

constexpr int kKT = 128;        // keys per tile
constexpr int kSplitUnit = 16;  // context slices are whole multiples of this many keys
constexpr int kMaxNT = 4;       // n8 row tiles per chunk (<= 32 rows per thread block)

// resident thread blocks per SM of the Q8_0 verify kernel: two up to 24 rows per chunk
inline int q8_blocks_per_sm(int /*hd*/, int nt) { return nt <= 3 ? 2 : 1; }
// ... and of the tcgen05 verify kernel (all of tensor memory, about 196 KB of shared memory)
inline int tc_blocks_per_sm(int /*hd*/, int /*nt*/) { return 1; }
constexpr int kTcMaxRows = 24;  // rows per chunk of the tcgen05 verify kernel

struct Plan {
    int hd, nt, n_chunks, rows_per_chunk, n_split, keys_per_split, key_shift, n_ctx_splits;
    size_t ws_bytes;
};

// SM count of the current device, looked up once per device (concurrent first lookups store
// the same value).
inline int sm_count() {
    constexpr int kMaxDev = 64;
    static int cached[kMaxDev] = {};
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDev && cached[dev] > 0) return cached[dev];
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDev) cached[dev] = n;
    return n;
}

// window_keys > 0: the last window_keys keys get a slice of their own (the append-and-verify
// path), the context slices cover the keys before them.
// max_rows: rows (row x q-head pairs) per chunk at most, a multiple of 8 (32 for the all-mma.sync
// kernels, 24 for the tcgen05 one).  sms: SM count to plan for (0 = the current device's).
inline int make_plan(int n_rows, int n_q_heads, int head_dim, int kv_len, int n_kv_heads, int n_split_req, Plan* pl,
                     int window_keys = 0, int (*blocks_per_sm)(int hd, int nt) = q8_blocks_per_sm,
                     int max_rows = 8 * kMaxNT, int sms = 0) {
    if (n_rows < 1 || n_rows > 32 || n_q_heads < 1 || n_kv_heads < 1 || kv_len < 1) return KVQ8_ERR_INVALID_ARG;
    if (n_q_heads % n_kv_heads) return KVQ8_ERR_UNSUPPORTED;
    const int group = n_q_heads / n_kv_heads;
    if (group > 64) return KVQ8_ERR_UNSUPPORTED;
    if (head_dim != 128 && head_dim != 256) return KVQ8_ERR_UNSUPPORTED;
    if (n_split_req < 0 || n_split_req > 1024) return KVQ8_ERR_INVALID_ARG;
    const int R = n_rows * group;
    pl->hd = head_dim;
    pl->n_chunks = (R + max_rows - 1) / max_rows;
    pl->rows_per_chunk = (R + pl->n_chunks - 1) / pl->n_chunks;
    pl->nt = (pl->rows_per_chunk + 7) / 8;
    // slices are whole 16-key units, fine enough that the blocks of one wave get nearly equal
    // work; the automatic count fills every SM with as many thread blocks as fit at once
    // (blocks_per_sm of the kernel that will run)
    const int ctx_end = kv_len - window_keys;
    if (ctx_end < 0) return KVQ8_ERR_INVALID_ARG;
    const int n_units = (ctx_end + kSplitUnit - 1) / kSplitUnit;
    int ns = n_split_req;
    if (ns == 0) {
        if (sms <= 0) sms = sm_count();
        if (sms <= 0) sms = 152;
        const int per_sm = blocks_per_sm(head_dim, pl->nt);
        ns = std::max(1, (per_sm * sms) / (n_kv_heads * pl->n_chunks));
        // the window slice takes one of the blocks' places, so that the grid stays one wave
        if (window_keys > 0) ns = std::max(1, ns - 1);
    }
    ns = std::max(1, std::min(ns, n_units));
    // an automatic slice holds at least one whole 128-key tile; every slice is at least as
    // long as the window, whose slice spans keys_per_split keys from ctx_end
    const int min_units = std::max(n_split_req > 0 ? 1 : kKT / kSplitUnit,
                                   (window_keys + kSplitUnit - 1) / kSplitUnit);
    const int units_per_split = std::max(min_units, (n_units + ns - 1) / ns);
    pl->keys_per_split = units_per_split * kSplitUnit;
    pl->n_ctx_splits = (ctx_end + pl->keys_per_split - 1) / pl->keys_per_split;
    // with a window slice (window_keys <= keys_per_split) the context slices are aligned
    // to end at ctx_end, so the first one is the short one
    pl->key_shift = window_keys > 0 ? pl->n_ctx_splits * pl->keys_per_split - ctx_end : 0;
    pl->n_split = pl->n_ctx_splits + (window_keys > 0 ? 1 : 0);
    const size_t rows_total = (size_t)n_rows * n_q_heads;
    const size_t o_bytes = (size_t)pl->n_split * rows_total * head_dim * sizeof(float);
    pl->ws_bytes = ((o_bytes + 255) / 256) * 256 + (size_t)pl->n_split * rows_total * 2 * sizeof(float);
    return KVQ8_OK;
}


}  // namespace kvq8
