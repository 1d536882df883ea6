// verify.cu -- the verify entry points (attn_verify_q8 and its variants) and the all-mma.sync
// split-context scan used for K8V4 pools and short causal or tree-window scans.
//
// Source: "perf(gfx1100): share Q8 KV scans across verifier rows", Summary: one worker owns
// all the query rows of a verify window and shares each K/V scan across them; the context
// is split into slices whose partials are merged by a reducer.  "gfx12 WMMA kernel for the
// int8-KV QSA prompt attention", How: fp16 hi + lo split of q and p with fp32 accumulation,
// online softmax, V scale folded into p.
//
// Routing: causal and tree-shaped windows over a Q8_0 cache (attn_verify_q8,
// attn_verify_tree_q8, attn_verify_q8_partials, attn_verify_append_q8 and the host-buffer and
// no-allocation entries built on them) and causal windows over a K8V4 pool at hd256
// (attn_verify_k8v4) run the tcgen05 scan of verify_tc.cu, except short scans (fewer than two
// 128-key tiles per block, or hd128 chunks of <= 32 rows; see plan_causal) outside the append
// path, which run the kernel below; K8V4 pools at hd128 always run the kernel below.
//
// The kernel below (one thread block of 8 warps per (row chunk, context slice, KV head); the
// chunks and slices come from verify_plan.cuh):
//   * K/V codes and scales of a 128-key tile are staged in shared memory with 16-byte
//     cp.async copies into an XOR-swizzled layout (conflict-free fragment reads).  K of the
//     next tile streams in while the softmax and PV of this tile run, and V while QK runs,
//     so every K/V byte of the slice crosses HBM once for all T x group rows.
//   * QK runs transposed on the tensor cores (m16n8k16, fp32 accumulate): keys are the M
//     dimension (16 per fragment, 16 keys per warp) and query rows the N dimension (8 per
//     fragment), so a window of 4 rows x group 6 = 24 rows needs no padding.  int8 codes
//     become fp16 exactly in registers (byte permute + magic-bias subtract); q enters as
//     fp16 hi + lo, both accumulated into the same fragment; the K scale, which varies along
//     the contraction in 32-value blocks, is applied after each 32-deep step:
//     s += dK * (q.k)_b.
//   * Online softmax in base 2 (q pre-scaled by softmax_scale * log2 e) with a lazy
//     reference maximum per row: the exact cross-warp maxima and the O rescale run only on
//     tiles where some score passes its row's reference by more than 2^kLazy.
//   * PV runs transposed too (M = 16 output dims, N = 8 rows, K = 16 keys).  Each warp owns
//     a 32-dim output block (hd256) or half of one (hd128); its B fragments are
//     w = p * dV[n][block] * 2^E split into fp16 hi + lo, with E a per-warp power of two that
//     keeps w inside the fp16 normal range (the accumulator is rescaled when E changes).
//   * Each slice writes an unnormalised partial (o, m, l); attn_combine merges them.
// Instantiations: TREE (tree-shaped windows from per-row masks), V4 (K8V4 pools: 4-bit V
// codes expanded in registers).
// attn_verify_append_q8_host works from host buffers: pinned ones are read by a copy kernel
// and written in place by the merge, pageable ones go through copy-engine transfers.
#include <algorithm>

#include "common.cuh"
#include "verify_plan.cuh"
#include "verify_tc.cuh"

namespace kvq8 {

int launch_combine(const float* part_o, const float* part_ml, int n_split, int rows, int head_dim, float* out,
                   cudaStream_t stream);

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr float kLazy = 8.0f;  // log2 units: a row's reference maximum moves only when a score exceeds it by this
constexpr float kPShift = 4.0f;  // p is stored as p * 2^kPShift; with p <= 2^kLazy that stays <= 2^12

struct VerifyParams {
    const float* q;
    const int8_t* k_codes;
    const uint16_t* k_scales;
    const int8_t* v_codes;
    const uint16_t* v_scales;
    float* part_o;     // [n_split][rows_total][HD]
    float2* part_ml;   // [n_split][rows_total]
    int n_rows;        // T
    int n_q_heads;
    int group;
    int group_magic;     // ceil(2^20 / group): x / group == (x * group_magic) >> 20 for x * group < 2^20
    int capacity;
    int kv_len;
    int q_pos0;
    int keys_per_split;
    int n_kv_heads;
    int rows_per_chunk;  // real rows per chunk (<= 8 * NT)
    float qscale;        // softmax_scale * log2(e)
    const uint32_t* wmask;  // tree windows: bit j of wmask[i] = row i sees key q_pos0 + j; null = causal
};

template <int HD, int NT>
struct Smem {
    static constexpr int NB = HD / 32;      // scale blocks per token
    static constexpr int RP = 8 * NT;       // padded rows per chunk
    static constexpr int PS = RP + 4;       // P-tile entries per key pair (padding spreads banks)
    static constexpr int kK = 0;
    static constexpr int kKs = kK + kKT * HD;
    static constexpr int kV = kKs + kKT * NB * 2;
    static constexpr int kVs = kV + kKT * HD;
    static constexpr int kQ = kVs + kKT * NB * 2;
    static constexpr int kP = kQ + NB * NT * 1024;
    static constexpr int kDv = kP + (kKT / 2) * PS * 8;   // per warp: its block's V scales * 2^E as fp16
    static constexpr int kRed = kDv + kWarps * kKT * 2;   // [RP][kWarps] floats
    static constexpr int kWm = kRed + RP * kWarps * 4;    // [RP] window masks (tree windows)
    static constexpr int kBytes = kWm + RP * 4;
};

// Byte offset of code byte c of tile row n in the swizzled layout (16-byte chunks XOR row%8).
template <int HD>
__device__ __forceinline__ int swz(int n, int c) {
    return n * HD + ((((c >> 4) ^ (n & 7)) << 4) | (c & 15));
}

// A thread copies the chunks ci = tid + k * kThreads; since kThreads is a multiple of 8 rows'
// worth of chunks, its row advances by a fixed step and its swizzled column never changes,
// so every copy is a pointer increment.
template <int HD>
__device__ __forceinline__ void load_codes(uint8_t* smem, const int8_t* plane, int64_t head_row0, int tile_key0,
                                           int key_end) {
    constexpr int CPR = HD / 16;                 // 16-byte chunks per row
    constexpr int ROWS_PER_PASS = kThreads / CPR;
    static_assert(ROWS_PER_PASS % 8 == 0, "row step must keep the swizzle phase");
    const int n0 = threadIdx.x / CPR, c16 = threadIdx.x % CPR;
    const uint32_t dst0 = smem_u32(smem) + n0 * HD + ((c16 ^ (n0 & 7)) << 4);
    const int8_t* src0 = plane + (head_row0 + tile_key0 + n0) * HD + c16 * 16;
    if (key_end - tile_key0 >= kKT) {  // a whole tile: every copy is live, offsets are immediates
#pragma unroll
        for (int k = 0; k < kKT / ROWS_PER_PASS; ++k) cp_async_16(dst0 + k * ROWS_PER_PASS * HD, src0 + k * ROWS_PER_PASS * HD, 16);
        return;
    }
    const int valid = key_end - tile_key0 - n0;  // rows of this thread's column still inside the slice
#pragma unroll
    for (int k = 0; k < kKT / ROWS_PER_PASS; ++k) {
        const bool ok = k * ROWS_PER_PASS < valid;
        cp_async_16(dst0 + k * ROWS_PER_PASS * HD, ok ? src0 + (int64_t)k * ROWS_PER_PASS * HD : src0 - (int64_t)n0 * HD,
                    ok ? 16 : 0);
    }
}

// Scales of one tile: HD/16 bytes per token (16 at hd256, 8 at hd128), copied in
// per-token pieces so that no alignment beyond the token's own is assumed.
template <int HD>
__device__ __forceinline__ void load_scales(uint8_t* smem, const uint16_t* plane, int64_t head_row0, int tile_key0,
                                            int key_end) {
    constexpr int SB = HD / 16;
    const uint32_t base = smem_u32(smem);
    const uint16_t* src0 = plane + (head_row0 + tile_key0) * (HD / 32);
    static_assert(kThreads >= kKT, "one scale row per thread");
    if (key_end - tile_key0 >= kKT) {  // a whole tile
        if (threadIdx.x < kKT) {
            if constexpr (SB == 16)
                cp_async_16(base + threadIdx.x * SB, src0 + threadIdx.x * (HD / 32), 16);
            else
                cp_async_8(base + threadIdx.x * SB, src0 + threadIdx.x * (HD / 32), 8);
        }
        return;
    }
    for (int n = threadIdx.x; n < kKT; n += kThreads) {
        const bool ok = tile_key0 + n < key_end;
        const uint16_t* src = ok ? src0 + n * (HD / 32) : src0;
        if constexpr (SB == 16)
            cp_async_16(base + n * SB, src, ok ? 16 : 0);
        else
            cp_async_8(base + n * SB, src, ok ? 8 : 0);
    }
}

// Row index / group by a multiply: (x * ceil(2^20 / g)) >> 20 equals x / g whenever x g < 2^20,
// which holds for every row index here (x < 32 rows * 64 heads per group, g <= 64).
__device__ __forceinline__ int div_group(int x, const VerifyParams& p) {
    return (int)(((uint32_t)x * (uint32_t)p.group_magic) >> 20);
}

// frexp's exponent of a positive normal float (x = m 2^e, m in [0.5, 1)), and 2^n for a
// normal result (-126 <= n <= 127), from the exponent bits.  The V scales reaching them are
// fp16 values as fp32, so x is normal and n stays within [-60, 40].
__device__ __forceinline__ int frexp_exponent(float x) { return (int)((__float_as_uint(x) >> 23) & 0xFFu) - 126; }
__device__ __forceinline__ float exp2_int(int n) { return __uint_as_float((uint32_t)(n + 127) << 23); }

// 4-bit V codes of one tile (K8V4 pools): HD/2 bytes per key, 16-byte chunk c of row n stored
// at chunk c ^ ((n >> 1) & (CPR - 1)), so the four key rows a PV load touches (2t, t = 0..3)
// fall in four different chunks; rows at or past key_end are zero-filled.
template <int HD>
__device__ __forceinline__ void load_codes_v4(uint8_t* smem, const uint8_t* plane, int64_t head_row0, int tile_key0,
                                              int key_end) {
    constexpr int ROWB = HD / 2;
    constexpr int CPR = ROWB / 16;                 // 8 (hd256) or 4 (hd128) chunks per row
    constexpr int ROWS_PER_PASS = kThreads / CPR;  // 32 or 64
    static_assert(ROWS_PER_PASS % (2 * CPR) == 0, "row step must keep the swizzle phase");
    const int n0 = threadIdx.x / CPR, c16 = threadIdx.x % CPR;
    const uint32_t dst0 = smem_u32(smem) + n0 * ROWB + ((c16 ^ ((n0 >> 1) & (CPR - 1))) << 4);
    const uint8_t* src0 = plane + (head_row0 + tile_key0 + n0) * ROWB + c16 * 16;
    if (key_end - tile_key0 >= kKT) {
#pragma unroll
        for (int k = 0; k < kKT / ROWS_PER_PASS; ++k)
            cp_async_16(dst0 + k * ROWS_PER_PASS * ROWB, src0 + k * ROWS_PER_PASS * ROWB, 16);
        return;
    }
    const int valid = key_end - tile_key0 - n0;
#pragma unroll
    for (int k = 0; k < kKT / ROWS_PER_PASS; ++k) {
        const bool ok = k * ROWS_PER_PASS < valid;
        cp_async_16(dst0 + k * ROWS_PER_PASS * ROWB, ok ? src0 + (int64_t)k * ROWS_PER_PASS * ROWB : src0 - (int64_t)n0 * ROWB,
                    ok ? 16 : 0);
    }
}

// Work split inside a thread block (8 warps):
//   QK  : warp w owns keys 16w .. 16w+15 of the tile (one m16 fragment), all row tiles;
//   PV  : at hd256 warp w owns the 32-dim output block w (two m16 fragments); at hd128 warps
//         2b and 2b+1 share block b, one m16 fragment each.
// Row statistics live in the lanes that own the rows: lane (g, t) holds rows 8nt + 2t + c in
// both the S^T and the O^T fragments, so the softmax factors never leave the thread.
// TREE: the window's rows see the window keys their mask selects (p.wmask); otherwise the
// window is sequential (row i sees keys < q_pos0 + i + 1) and the mask code is compiled out.
template <int HD, int NT, bool TREE, bool V4 = false>
__global__ void __launch_bounds__(kThreads, (NT <= 3 ? 2 : 1)) verify_split_kernel(const VerifyParams p) {
    using L = Smem<HD, NT>;
    constexpr int NB = L::NB, RP = L::RP, PS = L::PS;
    constexpr int MTW = HD / 128;  // m16 fragments of V^T per warp in PV
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* sK = smem + L::kK;
    const uint16_t* sKs = reinterpret_cast<const uint16_t*>(smem + L::kKs);
    uint8_t* sV = smem + L::kV;
    const uint16_t* sVs = reinterpret_cast<const uint16_t*>(smem + L::kVs);
    __half* sQ = reinterpret_cast<__half*>(smem + L::kQ);
    // P tile: entry (key pair k, row r) = (hi, lo) fp16 pairs of (p[2k][r], p[2k+1][r]) * 2^kPShift
    uint2* sP = reinterpret_cast<uint2*>(smem + L::kP);
    float* sRed = reinterpret_cast<float*>(smem + L::kRed);
    uint32_t* sWm = reinterpret_cast<uint32_t*>(smem + L::kWm);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int chunk = blockIdx.x, split = blockIdx.y, kvh = blockIdx.z;
    const int R = p.n_rows * p.group;
    const int rows_total = p.n_rows * p.n_q_heads;
    const int row0 = chunk * p.rows_per_chunk;
    const int rows_here = min(p.rows_per_chunk, R - row0);
    // Slice s covers keys [s * keys_per_split, (s + 1) * keys_per_split) clipped to kv_len.
    const int key_begin = split * p.keys_per_split;
    const int key_end = min(key_begin + p.keys_per_split, p.kv_len);
    const int64_t head_row0 = (int64_t)kvh * p.capacity;
    const int pvb = HD == 256 ? warp : (warp >> 1);  // PV output block of this warp
    uint16_t* sDv = reinterpret_cast<uint16_t*>(smem + L::kDv) + warp * kKT;

    // The combine kernel may be launched now; it waits for this grid before reading.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // Stage q rows of this chunk as fp16 hi/lo in mma B-fragment order:
    // entry (block b, n-tile nt, hi|lo, lane g*4+t) holds row 8nt+g, dims 32b+8t .. +7.
    {
        constexpr int GPR = HD / 8;                       // 8-dim groups per row
        constexpr int PER = (RP * GPR + kThreads - 1) / kThreads;
        float4 v[PER][2];
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int idx = threadIdx.x + k * kThreads;
            const int r = idx / GPR, j8 = idx - r * GPR;
            v[k][0] = v[k][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (idx < RP * GPR && r < rows_here) {
                const int rr = row0 + r;
                const int i = div_group(rr, p), hh = rr - i * p.group;
                const float4* src =
                    reinterpret_cast<const float4*>(p.q + ((int64_t)i * p.n_q_heads + kvh * p.group + hh) * HD) + 2 * j8;
                v[k][0] = __ldg(src);
                v[k][1] = __ldg(src + 1);
            }
        }
        // The first K tile is requested after the q loads, so those are not queued behind
        // every block's first tile; K alone lands in about half the time of K + V.  The V
        // tile of each iteration is requested once its K has landed (top of the loop).
        if (key_begin < key_end) {
            load_codes<HD>(sK, p.k_codes, head_row0, key_begin, key_end);
            load_scales<HD>(smem + L::kKs, p.k_scales, head_row0, key_begin, key_end);
        }
        cp_async_commit();
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int idx = threadIdx.x + k * kThreads;
            if (idx >= RP * GPR) continue;
            const int r = idx / GPR, j8 = idx - r * GPR;
            const float x[8] = {v[k][0].x, v[k][0].y, v[k][0].z, v[k][0].w,
                                v[k][1].x, v[k][1].y, v[k][1].z, v[k][1].w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = x[2 * e] * p.qscale, b = x[2 * e + 1] * p.qscale;
                const __half2 h = __floats2half2_rn(a, b);
                const __half2 l = __floats2half2_rn(a - __low2float(h), b - __high2float(h));
                hi[e] = h2_as_u32(h);
                lo[e] = h2_as_u32(l);
            }
            const int b = j8 >> 2, tt = j8 & 3, nt = r >> 3, gg = r & 7;
            uint4* dst = reinterpret_cast<uint4*>(sQ + ((b * NT + nt) * 2) * 256 + (gg * 4 + tt) * 8);
            dst[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            dst[32] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    }

    // Visibility bound per owned row (row rr sees keys < vis_end; for a tree window, keys at
    // or past q_pos0 also need their mask bit) and its output row (-1 for padding rows).
    constexpr bool tree = TREE;
    int vis_end[NT][2], grow[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int r = 8 * nt + 2 * t + c;
            if (r < rows_here) {
                const int rr = row0 + r;
                const int i = div_group(rr, p), hh = rr - i * p.group;
                vis_end[nt][c] = min(min(tree ? p.q_pos0 + 32 : p.q_pos0 + i + 1, p.kv_len), key_end);
                grow[nt][c] = i * p.n_q_heads + kvh * p.group + hh;
            } else {
                vis_end[nt][c] = 0;
                grow[nt][c] = -1;
            }
        }

    if (TREE && threadIdx.x < RP) {  // the window mask of each row of the chunk (read in masked tiles)
        const int r = threadIdx.x;
        sWm[r] = r < rows_here ? __ldg(p.wmask + div_group(row0 + r, p)) : 0u;
    }  // published by the barrier at the top of the first tile

    // every real row of this chunk sees all keys below vis_min; padding rows hold q = 0 and
    // never reach the output, so tiles wholly below vis_min skip the mask
    const int vis_min = min(min(tree ? p.q_pos0 : p.q_pos0 + div_group(row0, p) + 1, p.kv_len), key_end);
    float m_ref[NT][2], l_w[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            m_ref[nt][c] = -INFINITY;
            l_w[nt][c] = 0.0f;
        }
    float O[MTW][NT][4];
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) O[mt][nt][c] = 0.0f;
    int E = INT32_MIN;  // unset

    // Per-lane shared-memory bases of the inner loops, fixed for the whole slice.
    // QK: row n0 = 16 warp + g reads bytes 32b + 8t .. +7, i.e. chunk 2b + t/2 of 16 bytes at
    // offset 8 (t & 1), stored at chunk (2b + t/2) ^ g = ((2b) ^ (g & 6)) + ((t/2) ^ (g & 1)).
    const int k_gh = g & 6;
    const uint8_t* const k_lane = sK + (warp * 16 + g) * HD + ((((t >> 1) ^ (g & 1))) << 4) + 8 * (t & 1);
    const uint4* const q_lane = reinterpret_cast<const uint4*>(sQ) + lane;
    // PV: rows 16 ks + 2t (+1, +8, +9) have swizzle phase 2t (2t + 1); the lane's 4 bytes sit at
    // dims 32 pvb + 4g, chunk 2 pvb + g/4, offset 4 (g & 3).
    const int v_cx = 2 * pvb + (g >> 2);
    const int v_off0 = (2 * t) * HD + ((v_cx ^ (2 * t)) << 4) + 4 * (g & 3);
    const int v_off1 = (2 * t + 1) * HD + ((v_cx ^ (2 * t + 1)) << 4) + 4 * (g & 3);
    // 4-bit V (K8V4): rows of HD/2 bytes; the lane's 4 dims are the 2 bytes at 2g of chunk pvb,
    // stored at chunk pvb ^ phase(row), phase(16 ks + 2t (+1)) = t and phase(16 ks + 2t + 8 (+9))
    // = (t + 4) mod (HD/32)
    constexpr int V4ROWB = HD / 2;
    const int v4_off0 = (2 * t) * V4ROWB + ((pvb ^ t) << 4) + 2 * g;
    const int v4_off8 = (2 * t + 8) * V4ROWB + ((pvb ^ ((t + 4) & (HD / 32 - 1))) << 4) + 2 * g;
    const uint2* const p_lane = sP + t * PS + g;

    for (int tile0 = key_begin; tile0 < key_end; tile0 += kKT) {
        const int nk = min(kKT, key_end - tile0);  // keys of this tile inside the slice
        cp_async_wait<0>();  // K of this tile landed (the only copy group in flight)
        __syncthreads();     // ... for every thread; and every warp is done with the previous sV
        if constexpr (V4)
            load_codes_v4<HD>(sV, reinterpret_cast<const uint8_t*>(p.v_codes), head_row0, tile0, key_end);
        else
            load_codes<HD>(sV, p.v_codes, head_row0, tile0, key_end);
        load_scales<HD>(smem + L::kVs, p.v_scales, head_row0, tile0, key_end);
        cp_async_commit();

        // ---------------- QK^T: S^T[key][row] for this warp's 16 keys ----------------
        float S[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) S[nt][c] = 0.0f;
        const int n0 = warp * 16 + g;
        if (warp * 16 < nk) {
#pragma unroll 2
            for (int b = 0; b < NB; ++b) {
                uint4 qh[NT], ql[NT];
                const uint4* qp = q_lane + b * NT * 64;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    qh[nt] = qp[nt * 64];
                    ql[nt] = qp[nt * 64 + 32];
                }
                // rows n0 and n0 + 8 share the swizzle phase g: chunk (2b + t/2) ^ g
                const uint8_t* kp = k_lane + (((2 * b) ^ k_gh) << 4);
                const uint2 k0 = *reinterpret_cast<const uint2*>(kp);
                const uint2 k1 = *reinterpret_cast<const uint2*>(kp + 8 * HD);
                const uint32_t x0 = k0.x ^ 0x80808080u, x1 = k1.x ^ 0x80808080u;
                const uint32_t y0 = k0.y ^ 0x80808080u, y1 = k1.y ^ 0x80808080u;
                const uint32_t a00 = biased_bytes_to_half2<0x4140>(x0), a01 = biased_bytes_to_half2<0x4140>(x1);
                const uint32_t a02 = biased_bytes_to_half2<0x4342>(x0), a03 = biased_bytes_to_half2<0x4342>(x1);
                const uint32_t a10 = biased_bytes_to_half2<0x4140>(y0), a11 = biased_bytes_to_half2<0x4140>(y1);
                const uint32_t a12 = biased_bytes_to_half2<0x4342>(y0), a13 = biased_bytes_to_half2<0x4342>(y1);
                float tmp[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_f16_16816_zc(tmp[nt], a00, a01, a02, a03, qh[nt].x, qh[nt].y);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_f16_16816(tmp[nt], a10, a11, a12, a13, qh[nt].z, qh[nt].w);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_f16_16816(tmp[nt], a00, a01, a02, a03, ql[nt].x, ql[nt].y);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_f16_16816(tmp[nt], a10, a11, a12, a13, ql[nt].z, ql[nt].w);
                const float dk0 = half_bits_to_float(sKs[n0 * NB + b]);
                const float dk1 = half_bits_to_float(sKs[(n0 + 8) * NB + b]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    S[nt][0] = fmaf(dk0, tmp[nt][0], S[nt][0]);
                    S[nt][1] = fmaf(dk0, tmp[nt][1], S[nt][1]);
                    S[nt][2] = fmaf(dk1, tmp[nt][2], S[nt][2]);
                    S[nt][3] = fmaf(dk1, tmp[nt][3], S[nt][3]);
                }
            }
        }

        // ---------------- mask; does any score pass its row's reference by more than kLazy? ----------------
        const bool tile_needs_mask = tile0 + kKT > vis_min;
        bool need = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int key = tile0 + n0 + 8 * h;
                    float& s = S[nt][2 * h + c];
                    if (tile_needs_mask) {
                        bool vis = key < vis_end[nt][c];
                        if (tree && vis && key >= p.q_pos0)
                            vis = (sWm[8 * nt + 2 * t + c] >> (key - p.q_pos0)) & 1u;
                        if (!vis) s = -INFINITY;
                    }
                    need |= s > m_ref[nt][c] + kLazy;
                }
        // barrier: every warp is done with sK, and the vote is known to all
        if (__syncthreads_or(need)) {
            // exact tile maxima: per warp over its 16 keys, then over the 8 warps
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float m = fmaxf(S[nt][c], S[nt][2 + c]);
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                    if (g == 0) sRed[(8 * nt + 2 * t + c) * kWarps + warp] = m;
                }
            __syncthreads();
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const float4* rp = reinterpret_cast<const float4*>(sRed + (8 * nt + 2 * t + c) * kWarps);
                    const float4 u = rp[0], w = rp[1];
                    const float mt_ = fmaxf(fmaxf(fmaxf(u.x, u.y), fmaxf(u.z, u.w)), fmaxf(fmaxf(w.x, w.y), fmaxf(w.z, w.w)));
                    const float m_old = m_ref[nt][c];
                    const float m_new = fmaxf(m_old, mt_);
                    const float a = (m_old == -INFINITY) ? 1.0f : ex2_approx(m_old - m_new);
                    m_ref[nt][c] = m_new;
                    l_w[nt][c] *= a;
#pragma unroll
                    for (int mt = 0; mt < MTW; ++mt) {
                        O[mt][nt][c] *= a;
                        O[mt][nt][2 + c] *= a;
                    }
                }
        }

        {  // stream the next tile's K while softmax and PV run
            const int next0 = tile0 + kKT;
            if (next0 < key_end) {
                load_codes<HD>(sK, p.k_codes, head_row0, next0, key_end);
                load_scales<HD>(smem + L::kKs, p.k_scales, head_row0, next0, key_end);
            }
            cp_async_commit();
        }

        // ---------------- softmax: p = 2^(s - m_ref), stored as p 2^kPShift ----------------
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const float mb = (m_ref[nt][c] == -INFINITY) ? 0.0f : m_ref[nt][c] - kPShift;
                float sum = 0.0f;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float& s = S[nt][2 * h + c];
                    s = ex2_approx(s - mb);
                    sum += s;
                }
                l_w[nt][c] += sum;
            }
        // P tile: a key and its pair partner sit in lanes 4 apart; each pair of lanes swaps one
        // value so that the even-g lane writes row 2t and the odd-g lane row 2t+1.
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float v0 = S[nt][2 * h], v1 = S[nt][2 * h + 1];
                const bool ev = (g & 1) == 0;
                const float recv = __shfl_xor_sync(0xffffffffu, ev ? v1 : v0, 4);
                const float pe = ev ? v0 : recv;  // even key
                const float po = ev ? recv : v1;  // odd key
                const __half2 ph = __floats2half2_rn(pe, po);
                const __half2 pl = __floats2half2_rn(pe - __low2float(ph), po - __high2float(ph));
                const int kl = n0 + 8 * h;
                sP[(kl >> 1) * PS + 8 * nt + 2 * t + (ev ? 0 : 1)] = make_uint2(h2_as_u32(ph), h2_as_u32(pl));
            }

        cp_async_wait<1>();  // V of this tile landed (next K may still be in flight)
        __syncthreads();

        // ---------------- PV: O^T[dim][row] += V^T * (p 2^kPShift) (dV 2^E) ----------------
        // Per output block, E keeps dV 2^E of the tile's largest scale in [2, 4), so that
        // w = (p 2^kPShift)(dV 2^E) < 2^14 stays in the fp16 range; w = hi + lo exactly up to
        // 2^-22: hi = fl(ph d), lo = fl((ph d - hi) + pl d), the first residual exact by FMA.
        // The warp's scaled block scales go to its own fp16 table, read as key pairs below.
        {
            float dv[kKT / 32];
            float dmax = 0.0f;
#pragma unroll
            for (int k = 0; k < kKT / 32; ++k) {
                dv[k] = half_bits_to_float(sVs[(lane + 32 * k) * NB + pvb]);
                dmax = fmaxf(dmax, dv[k]);
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
            if (dmax > 0.0f) {
                const int et = 2 - frexp_exponent(dmax);
                if (E == INT32_MIN) {
                    E = et;
                } else if (et < E) {
                    const float f = exp2_int(et - E);
#pragma unroll
                    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int c = 0; c < 4; ++c) O[mt][nt][c] *= f;
                    E = et;
                }
            }
            const float esc = (E == INT32_MIN) ? 0.0f : exp2_int(E);
#pragma unroll
            for (int k = 0; k < kKT / 32; ++k) sDv[lane + 32 * k] = __half_as_ushort(__float2half_rn(dv[k] * esc));
            __syncwarp();
        }
        auto pv_step = [&](const int ks) {
            const int kb = ks * 16;
            uint2 pp01[NT], pp89[NT];  // (hi, lo) pairs of keys (2t, 2t+1) and (2t+8, 2t+9), row g of n-tile
            const uint2* pp = p_lane + ks * 8 * PS;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                pp01[nt] = pp[8 * nt];
                pp89[nt] = pp[4 * PS + 8 * nt];
            }
            const __half2 d01 = u32_as_h2(*reinterpret_cast<const uint32_t*>(sDv + kb + 2 * t));
            const __half2 d89 = u32_as_h2(*reinterpret_cast<const uint32_t*>(sDv + kb + 2 * t + 8));
            uint32_t A[MTW][4];
            if constexpr (V4) {
                // keys (2t, 2t+1) and (2t+8, 2t+9) side by side: 4 nibbles of each key per half
                const uint8_t* vp = sV + ks * 16 * V4ROWB;
                const uint32_t x01 = (uint32_t)*reinterpret_cast<const uint16_t*>(vp + v4_off0) |
                                     ((uint32_t)*reinterpret_cast<const uint16_t*>(vp + v4_off0 + V4ROWB) << 16);
                const uint32_t x89 = (uint32_t)*reinterpret_cast<const uint16_t*>(vp + v4_off8) |
                                     ((uint32_t)*reinterpret_cast<const uint16_t*>(vp + v4_off8 + V4ROWB) << 16);
                if (HD == 256 || (warp & 1) == 0) {  // dims 4g, 4g+1
                    A[0][0] = nib_lo_to_half2(x01);
                    A[0][1] = nib_hi_to_half2(x01);
                    A[0][2] = nib_lo_to_half2(x89);
                    A[0][3] = nib_hi_to_half2(x89);
                }
                if (HD == 256 || (warp & 1) == 1) {  // dims 4g+2, 4g+3
                    A[MTW - 1][0] = nib_lo_to_half2(x01 >> 8);
                    A[MTW - 1][1] = nib_hi_to_half2(x01 >> 8);
                    A[MTW - 1][2] = nib_lo_to_half2(x89 >> 8);
                    A[MTW - 1][3] = nib_hi_to_half2(x89 >> 8);
                }
            } else {
                const uint8_t* vp = sV + ks * 16 * HD;
                const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vp + v_off0) ^ 0x80808080u;
                const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vp + v_off1) ^ 0x80808080u;
                const uint32_t w8 = *reinterpret_cast<const uint32_t*>(vp + v_off0 + 8 * HD) ^ 0x80808080u;
                const uint32_t w9 = *reinterpret_cast<const uint32_t*>(vp + v_off1 + 8 * HD) ^ 0x80808080u;
                if (HD == 256 || (warp & 1) == 0) {  // dims 4g, 4g+1 (and 4g+2, 4g+3 at hd256)
                    const uint32_t y01 = prmt2<0x5140>(w0, w1), y89 = prmt2<0x5140>(w8, w9);
                    A[0][0] = biased_bytes_to_half2<0x4140>(y01);
                    A[0][1] = biased_bytes_to_half2<0x4342>(y01);
                    A[0][2] = biased_bytes_to_half2<0x4140>(y89);
                    A[0][3] = biased_bytes_to_half2<0x4342>(y89);
                }
                if (HD == 256 || (warp & 1) == 1) {  // dims 4g+2, 4g+3
                    const uint32_t y01 = prmt2<0x7362>(w0, w1), y89 = prmt2<0x7362>(w8, w9);
                    A[MTW - 1][0] = biased_bytes_to_half2<0x4140>(y01);
                    A[MTW - 1][1] = biased_bytes_to_half2<0x4342>(y01);
                    A[MTW - 1][2] = biased_bytes_to_half2<0x4140>(y89);
                    A[MTW - 1][3] = biased_bytes_to_half2<0x4342>(y89);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const __half2 ph0 = u32_as_h2(pp01[nt].x), pl0 = u32_as_h2(pp01[nt].y);
                const __half2 ph1 = u32_as_h2(pp89[nt].x), pl1 = u32_as_h2(pp89[nt].y);
                const __half2 h0 = __hmul2(ph0, d01);
                const __half2 h1 = __hmul2(ph1, d89);
                const __half2 l0 = __hfma2(pl0, d01, __hfma2(ph0, d01, __hneg2(h0)));
                const __half2 l1 = __hfma2(pl1, d89, __hfma2(ph1, d89, __hneg2(h1)));
                const uint32_t bh0 = h2_as_u32(h0), bh1 = h2_as_u32(h1);
                const uint32_t bl0 = h2_as_u32(l0), bl1 = h2_as_u32(l1);
#pragma unroll
                for (int mt = 0; mt < MTW; ++mt) {
                    mma_f16_16816(O[mt][nt], A[mt][0], A[mt][1], A[mt][2], A[mt][3], bh0, bh1);
                    mma_f16_16816(O[mt][nt], A[mt][0], A[mt][1], A[mt][2], A[mt][3], bl0, bl1);
                }
            }
        };
        if constexpr (NT <= 3) {
            // 32-key steps (offsets fixed at compile time): key rows past nk hold p = 0 and
            // zero V codes and scales, so a ragged tile may round up
            const int n_u = (nk + 31) >> 5;
            for (int u4 = 0; u4 < n_u; ++u4) {
                pv_step(2 * u4);
                pv_step(2 * u4 + 1);
            }
        } else {
            const int n_ks = (nk + 15) >> 4;
#pragma unroll 2
            for (int ks = 0; ks < n_ks; ++ks) pv_step(ks);
        }
        __syncthreads();  // all warps done with sV, sP and the scale tables
    }
    cp_async_wait<0>();

    // ---------------- write the slice partial ----------------
    // row sums: over the lanes that share a row (g), then over the warps
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float l = l_w[nt][c];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            if (g == 0) sRed[(8 * nt + 2 * t + c) * kWarps + warp] = l;
        }
    __syncthreads();
    float* po = p.part_o + (int64_t)split * rows_total * HD;
    // O is (p 2^kPShift)(v 2^E) summed; lane owns dims 32b + 4g .. +3 (hd256) or the pair at
    // 32b + 4g + 2(w & 1) (hd128) of rows 8nt + 2t + c
    const float inv = (E == INT32_MIN) ? 1.0f : exp2_int(-E - (int)kPShift);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            if (grow[nt][c] < 0) continue;
            float* dst = po + (int64_t)grow[nt][c] * HD + 32 * pvb + 4 * g;
            if constexpr (HD == 256) {
                *reinterpret_cast<float4*>(dst) = make_float4(O[0][nt][c] * inv, O[0][nt][2 + c] * inv,
                                                              O[1][nt][c] * inv, O[1][nt][2 + c] * inv);
            } else {
                *reinterpret_cast<float2*>(dst + 2 * (warp & 1)) = make_float2(O[0][nt][c] * inv, O[0][nt][2 + c] * inv);
            }
        }
    if (warp == 0 && g == 0) {
        const float lscale = exp2_int(-(int)kPShift);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (grow[nt][c] < 0) continue;
                const float4* rp = reinterpret_cast<const float4*>(sRed + (8 * nt + 2 * t + c) * kWarps);
                const float4 u = rp[0], w = rp[1];
                const float l = ((u.x + u.y) + (u.z + u.w)) + ((w.x + w.y) + (w.z + w.w));
                const float m = m_ref[nt][c];
                p.part_ml[(int64_t)split * rows_total + grow[nt][c]] =
                    make_float2(m == -INFINITY ? -INFINITY : m * kLn2, l * lscale);
            }
    }
}

template <int HD, int NT, bool TREE, bool V4>
int launch_verify(const VerifyParams& vp, const Plan& pl, int n_kv_heads, cudaStream_t stream) {
    constexpr int bytes = Smem<HD, NT>::kBytes;
    static SmemOptIn opt;
    if (opt.ensure(verify_split_kernel<HD, NT, TREE, V4>, bytes) != KVQ8_OK) return KVQ8_ERR_CUDA;
    dim3 grid(pl.n_chunks, pl.n_split, n_kv_heads);
    verify_split_kernel<HD, NT, TREE, V4><<<grid, kThreads, bytes, stream>>>(vp);
    return launch_status();
}

template <int HD, bool TREE, bool V4 = false>
int dispatch_nt(const VerifyParams& vp, const Plan& pl, int n_kv_heads, cudaStream_t s) {
    switch (pl.nt) {
        case 1: return launch_verify<HD, 1, TREE, V4>(vp, pl, n_kv_heads, s);
        case 2: return launch_verify<HD, 2, TREE, V4>(vp, pl, n_kv_heads, s);
        case 3: return launch_verify<HD, 3, TREE, V4>(vp, pl, n_kv_heads, s);
        case 4: return launch_verify<HD, 4, TREE, V4>(vp, pl, n_kv_heads, s);
        default: return KVQ8_ERR_UNSUPPORTED;
    }
}

}  // namespace

// Plans of the two scan kernels: causal windows over a Q8_0 cache run the tcgen05 kernel
// (row chunks of <= 24 rows, one block per SM); short scans (plan_causal) and K8V4 pools at hd128
// the all-mma.sync one.
inline int plan_tc(int n_rows, int n_q_heads, int head_dim, int kv_len, int n_kv_heads, int n_split, Plan* pl,
                   int window_keys = 0) {
    return make_plan(n_rows, n_q_heads, head_dim, kv_len, n_kv_heads, n_split, pl, window_keys, tc_blocks_per_sm,
                     kTcMaxRows);
}
inline int plan_mma(int n_rows, int n_q_heads, int head_dim, int kv_len, int n_kv_heads, int n_split, Plan* pl) {
    return make_plan(n_rows, n_q_heads, head_dim, kv_len, n_kv_heads, n_split, pl);
}

// Plan of a causal window over a Q8_0 cache, and which kernel runs it.  The tcgen05 kernel has
// the longer pipeline fill: it runs a window when each of its blocks gets at least two 128-key
// tiles and the chunk is large enough to keep its roles busy (hd256, or more than 32 rows per
// KV head at hd128); otherwise the all-mma.sync kernel does (measured on GB300, 24q/4kv/hd256:
// ctx 4096 T = 4 9.9 vs 10.3 us; 32q/8kv/hd128 ctx 8192 T = 4 12.5 vs 13.2 us).  The append
// path always takes the tcgen05 kernel (its window slice lives there).  Every entry point that
// sizes or launches a causal scan goes through here, so counts and launches agree.
inline int plan_causal(int n_rows, int n_q_heads, int head_dim, int kv_len, int n_kv_heads, int n_split, Plan* pl,
                       bool* use_tc, int window_keys = 0) {
    const int rc = plan_tc(n_rows, n_q_heads, head_dim, kv_len, n_kv_heads, n_split, pl, window_keys);
    if (rc != KVQ8_OK) return rc;
    const int rows_per_kv_head = n_rows * (n_q_heads / n_kv_heads);
    const int tiles = (std::min(pl->keys_per_split, kv_len) + kKT - 1) / kKT;
    *use_tc = window_keys > 0 || (tiles >= 2 && (head_dim == 256 || rows_per_kv_head > 32));
    return *use_tc ? KVQ8_OK : plan_mma(n_rows, n_q_heads, head_dim, kv_len, n_kv_heads, n_split, pl);
}

}  // namespace kvq8

// The one workspace size that serves attn_verify_q8, attn_verify_tree_q8 and attn_verify_k8v4.
extern "C" size_t attn_verify_q8_workspace_bytes(int n_rows, int n_q_heads, int head_dim, int kv_len, int n_kv_heads,
                                                 int n_split) {
    kvq8::Plan a, b;
    if (kvq8::plan_tc(n_rows, n_q_heads, head_dim, kv_len, n_kv_heads, n_split, &a) != KVQ8_OK ||
        kvq8::plan_mma(n_rows, n_q_heads, head_dim, kv_len, n_kv_heads, n_split, &b) != KVQ8_OK)
        return 0;
    return std::max(a.ws_bytes, b.ws_bytes);
}

namespace kvq8 {
namespace {

// k_new / v_new (append-and-verify): the n_rows window tokens (kv_len must be q_pos0 + n_rows)
// get a slice of their own, whose blocks quantise them into their tiles and into the cache.
// part_o / part_ml (the partials entry point): the slices' partials go there, q_pos0 may be
// negative, and no combine runs; out and the workspace are unused.
int verify_impl(const float* q, int n_rows, int n_q_heads, const kvq8_cache* kv, int kv_len, int q_pos0,
                const uint32_t* wmask, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                int n_split, kvq8_stream_t stream, const float* k_new = nullptr, const float* v_new = nullptr,
                float* part_o = nullptr, float* part_ml = nullptr, bool v4 = false) {
    const bool append = k_new != nullptr;
    const bool partials = part_o != nullptr;
    if (!kv || !q || (!out && !partials) || (partials && !part_ml)) return KVQ8_ERR_INVALID_ARG;
    if (!kv->k_codes || !kv->k_scales || !kv->v_codes || !kv->v_scales) return KVQ8_ERR_INVALID_ARG;
    if (kv->n_kv_heads < 1 || kv->capacity < 1) return KVQ8_ERR_INVALID_ARG;
    if (partials ? q_pos0 < -(1 << 30) : q_pos0 < 0) return KVQ8_ERR_INVALID_ARG;
    if (kv_len > kv->capacity) return KVQ8_ERR_INVALID_ARG;
    if (!(softmax_scale == softmax_scale) || softmax_scale == INFINITY || softmax_scale == -INFINITY)
        return KVQ8_ERR_INVALID_ARG;
    if (append && (!v_new || kv_len != q_pos0 + n_rows)) return KVQ8_ERR_INVALID_ARG;
    // causal and tree windows over a Q8_0 cache and causal windows over a K8V4 pool at hd256: the
    // kernel plan_causal picks; K8V4 pools at hd128: the all-mma.sync kernel
    bool tc = false;
    Plan pl;
    const int rc = !v4 || kv->head_dim == 256
                       ? plan_causal(n_rows, n_q_heads, kv->head_dim, kv_len, kv->n_kv_heads, n_split, &pl, &tc,
                                     append ? n_rows : 0)
                       : plan_mma(n_rows, n_q_heads, kv->head_dim, kv_len, kv->n_kv_heads, n_split, &pl);
    if (rc != KVQ8_OK) return rc;
    if (!aligned16(q) || !aligned16(kv->k_codes) || !aligned16(kv->k_scales) || !aligned16(kv->v_codes) ||
        !aligned16(kv->v_scales))
        return KVQ8_ERR_MISALIGNED;
    if (append && (!aligned16(k_new) || !aligned16(v_new))) return KVQ8_ERR_MISALIGNED;
    if (partials) {
        if (!aligned16(part_o) || !aligned16(part_ml)) return KVQ8_ERR_MISALIGNED;
    } else {
        if (!aligned16(out)) return KVQ8_ERR_MISALIGNED;
        if (!workspace || workspace_bytes < pl.ws_bytes) return KVQ8_ERR_WORKSPACE;
        if (!aligned16(workspace)) return KVQ8_ERR_MISALIGNED;
    }

    VerifyParams vp;
    vp.q = q;
    vp.k_codes = kv->k_codes;
    vp.k_scales = kv->k_scales;
    vp.v_codes = kv->v_codes;
    vp.v_scales = kv->v_scales;
    const size_t rows_total = (size_t)n_rows * n_q_heads;
    const size_t o_bytes = (size_t)pl.n_split * rows_total * kv->head_dim * sizeof(float);
    vp.part_o = partials ? part_o : static_cast<float*>(workspace);
    vp.part_ml = partials ? reinterpret_cast<float2*>(part_ml)
                          : reinterpret_cast<float2*>(static_cast<char*>(workspace) + ((o_bytes + 255) / 256) * 256);
    vp.n_rows = n_rows;
    vp.n_q_heads = n_q_heads;
    vp.group = n_q_heads / kv->n_kv_heads;
    vp.group_magic = ((1 << 20) + vp.group - 1) / vp.group;  // exact: rows * group <= 32 * 64^2 < 2^20
    vp.capacity = kv->capacity;
    vp.kv_len = kv_len;
    vp.q_pos0 = q_pos0;
    vp.keys_per_split = pl.keys_per_split;
    vp.rows_per_chunk = pl.rows_per_chunk;
    vp.qscale = softmax_scale * kLog2e;
    vp.wmask = wmask;
    vp.n_kv_heads = kv->n_kv_heads;
    cudaStream_t s = (cudaStream_t)stream;
    int r1;
    if (tc) {
        VerifyTcParams tp;
        tp.q = q;
        tp.k_codes = const_cast<int8_t*>(kv->k_codes);
        tp.k_scales = const_cast<uint16_t*>(kv->k_scales);
        tp.v_codes = const_cast<int8_t*>(kv->v_codes);
        tp.v_scales = const_cast<uint16_t*>(kv->v_scales);
        tp.part_o = vp.part_o;
        tp.part_ml = vp.part_ml;
        tp.k_new = k_new;
        tp.v_new = v_new;
        tp.err = nullptr;
        tp.wmask = wmask;
        tp.n_rows = n_rows;
        tp.n_q_heads = n_q_heads;
        tp.group = vp.group;
        tp.group_magic = vp.group_magic;
        tp.capacity = kv->capacity;
        tp.kv_len = kv_len;
        tp.q_pos0 = q_pos0;
        tp.keys_per_split = pl.keys_per_split;
        tp.key_shift = pl.key_shift;
        tp.n_ctx_splits = pl.n_ctx_splits;
        tp.n_kv_heads = kv->n_kv_heads;
        tp.rows_per_chunk = pl.rows_per_chunk;
        tp.qscale = vp.qscale;
        r1 = launch_verify_tc(tp, pl, kv->n_kv_heads, append, v4, s);
    } else if (v4)  // K8V4 pools: causal windows, no append
        r1 = pl.hd == 128 ? dispatch_nt<128, false, true>(vp, pl, kv->n_kv_heads, s)
                          : dispatch_nt<256, false, true>(vp, pl, kv->n_kv_heads, s);
    else if (wmask)  // tree windows have no append variant
        r1 = pl.hd == 128 ? dispatch_nt<128, true>(vp, pl, kv->n_kv_heads, s)
                          : dispatch_nt<256, true>(vp, pl, kv->n_kv_heads, s);
    else if (!append)  // short causal scans (plan_causal)
        r1 = pl.hd == 128 ? dispatch_nt<128, false>(vp, pl, kv->n_kv_heads, s)
                          : dispatch_nt<256, false>(vp, pl, kv->n_kv_heads, s);
    else
        return KVQ8_ERR_UNSUPPORTED;
    if (r1 != KVQ8_OK || partials) return r1;
    return launch_combine(vp.part_o, reinterpret_cast<const float*>(vp.part_ml), pl.n_split, (int)rows_total,
                          kv->head_dim, out, s);
}

}  // namespace
}  // namespace kvq8

extern "C" int attn_verify_q8(const float* q, int n_rows, int n_q_heads, const kvq8_cache* kv, int kv_len,
                              int q_pos0, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                              int n_split, kvq8_stream_t stream) {
    return kvq8::verify_impl(q, n_rows, n_q_heads, kv, kv_len, q_pos0, nullptr, softmax_scale, out, workspace,
                             workspace_bytes, n_split, stream);
}

extern "C" int attn_verify_k8v4(const float* q, int n_rows, int n_q_heads, const kvk8v4_cache* kv, int kv_len,
                                int q_pos0, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                                int n_split, kvq8_stream_t stream) {
    if (!kv) return KVQ8_ERR_INVALID_ARG;
    // the Q8_0 view of the pool: the V plane pointer carries the nibbles
    const kvq8_cache view = {kv->k_codes, kv->k_scales, reinterpret_cast<const int8_t*>(kv->v_codes), kv->v_scales,
                             kv->n_kv_heads, kv->head_dim, kv->capacity};
    return kvq8::verify_impl(q, n_rows, n_q_heads, &view, kv_len, q_pos0, nullptr, softmax_scale, out, workspace,
                             workspace_bytes, n_split, stream, nullptr, nullptr, nullptr, nullptr, true);
}

extern "C" int attn_verify_q8_partials_count(int n_rows, int n_q_heads, int head_dim, int kv_len, int n_kv_heads,
                                             int n_split) {
    kvq8::Plan pl;
    bool tc = false;
    if (kvq8::plan_causal(n_rows, n_q_heads, head_dim, kv_len, n_kv_heads, n_split, &pl, &tc) != KVQ8_OK) return 0;
    return pl.n_split;
}

extern "C" int attn_verify_q8_partials(const float* q, int n_rows, int n_q_heads, const kvq8_cache* kv, int kv_len,
                                       int q_pos0, float softmax_scale, float* part_o, float* part_ml, int n_split,
                                       kvq8_stream_t stream) {
    if (!part_o || !part_ml) return KVQ8_ERR_INVALID_ARG;
    return kvq8::verify_impl(q, n_rows, n_q_heads, kv, kv_len, q_pos0, nullptr, softmax_scale, nullptr, nullptr, 0,
                             n_split, stream, nullptr, nullptr, part_o, part_ml);
}

extern "C" size_t attn_verify_append_q8_workspace_bytes(int n_rows, int n_q_heads, int head_dim, int q_pos0,
                                                        int n_kv_heads, int n_split) {
    kvq8::Plan pl;
    if (q_pos0 < 0 || kvq8::plan_tc(n_rows, n_q_heads, head_dim, q_pos0 + n_rows, n_kv_heads, n_split, &pl,
                                      n_rows) != KVQ8_OK)
        return 0;
    return pl.ws_bytes;
}

extern "C" int attn_verify_append_q8(const float* q, const float* k_new, const float* v_new, int n_rows,
                                     int n_q_heads, const kvq8_cache* kv, int q_pos0, float softmax_scale,
                                     float* out, void* workspace, size_t workspace_bytes, int n_split,
                                     kvq8_stream_t stream) {
    if (!k_new || !v_new || q_pos0 < 0) return KVQ8_ERR_INVALID_ARG;
    return kvq8::verify_impl(q, n_rows, n_q_heads, kv, q_pos0 + n_rows, q_pos0, nullptr, softmax_scale, out,
                             workspace, workspace_bytes, n_split, stream, k_new, v_new);
}

namespace {
// Scratch of the host-buffer entry: [q | k_new | v_new] fp32, out fp32, then the verify
// workspace, each part starting on a 256-byte boundary.
struct HostScratch {
    size_t in_bytes, out_off, ws_off, ws_bytes, total;
};
inline size_t round256(size_t x) { return (x + 255) / 256 * 256; }
bool host_scratch(int n_rows, int n_q_heads, int head_dim, int q_pos0, int n_kv_heads, int n_split, HostScratch* h) {
    kvq8::Plan pl;
    if (q_pos0 < 0 || kvq8::plan_tc(n_rows, n_q_heads, head_dim, q_pos0 + n_rows, n_kv_heads, n_split, &pl,
                                      n_rows) != KVQ8_OK)
        return false;
    const size_t q_bytes = (size_t)n_rows * n_q_heads * head_dim * sizeof(float);
    const size_t kv_bytes = (size_t)n_rows * n_kv_heads * head_dim * sizeof(float);
    h->in_bytes = q_bytes + 2 * kv_bytes;
    h->out_off = round256(h->in_bytes);
    h->ws_off = h->out_off + round256(q_bytes);
    h->ws_bytes = pl.ws_bytes;
    h->total = h->ws_off + pl.ws_bytes;
    return true;
}
}  // namespace

extern "C" size_t attn_verify_append_q8_host_scratch_bytes(int n_rows, int n_q_heads, int head_dim, int q_pos0,
                                                           int n_kv_heads, int n_split) {
    HostScratch h;
    return host_scratch(n_rows, n_q_heads, head_dim, q_pos0, n_kv_heads, n_split, &h) ? h.total : 0;
}

namespace {
// Device address of pinned host memory mapped into the device address space (null if `p` is
// not such memory: pageable memory goes through the copy engine instead).
const void* mapped_device_ptr(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// n16 16-byte words from mapped host memory to device memory: every word read once over the
// host link (lower latency than a copy-engine transfer for the few hundred KB of a window).
constexpr int kCopyThreads = 256, kCopyPer = 4;
__global__ void __launch_bounds__(kCopyThreads) host_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                                 int n16) {
    const int i0 = blockIdx.x * (kCopyThreads * kCopyPer) + threadIdx.x;
    uint4 v[kCopyPer];
#pragma unroll
    for (int k = 0; k < kCopyPer; ++k) {
        const int i = i0 + k * kCopyThreads;
        if (i < n16) v[k] = src[i];
    }
#pragma unroll
    for (int k = 0; k < kCopyPer; ++k) {
        const int i = i0 + k * kCopyThreads;
        if (i < n16) dst[i] = v[k];
    }
}
}  // namespace

extern "C" int attn_verify_append_q8_host(const float* h_in, int n_rows, int n_q_heads, const kvq8_cache* kv,
                                          int q_pos0, float softmax_scale, float* h_out, void* d_scratch,
                                          size_t scratch_bytes, int n_split, kvq8_stream_t stream) {
    if (!h_in || !h_out || !kv || q_pos0 < 0) return KVQ8_ERR_INVALID_ARG;
    HostScratch h;
    if (!host_scratch(n_rows, n_q_heads, kv->head_dim, q_pos0, kv->n_kv_heads, n_split, &h))
        return n_rows < 1 || n_rows > 32 || n_q_heads < 1 || kv->n_kv_heads < 1 ? KVQ8_ERR_INVALID_ARG
                                                                                  : KVQ8_ERR_UNSUPPORTED;
    if (!d_scratch || scratch_bytes < h.total) return KVQ8_ERR_WORKSPACE;
    if (!kvq8::aligned16(d_scratch)) return KVQ8_ERR_MISALIGNED;
    if (q_pos0 + n_rows > kv->capacity) return KVQ8_ERR_INVALID_ARG;
    // everything verify_impl checks past the shapes, before the input copy is queued
    if (!kv->k_codes || !kv->k_scales || !kv->v_codes || !kv->v_scales) return KVQ8_ERR_INVALID_ARG;
    if (!(softmax_scale == softmax_scale) || softmax_scale == INFINITY || softmax_scale == -INFINITY)
        return KVQ8_ERR_INVALID_ARG;
    if (!kvq8::aligned16(kv->k_codes) || !kvq8::aligned16(kv->k_scales) || !kvq8::aligned16(kv->v_codes) ||
        !kvq8::aligned16(kv->v_scales))
        return KVQ8_ERR_MISALIGNED;
    char* base = static_cast<char*>(d_scratch);
    const float* q = reinterpret_cast<const float*>(base);
    const float* k_new = q + (size_t)n_rows * n_q_heads * kv->head_dim;
    const float* v_new = k_new + (size_t)n_rows * kv->n_kv_heads * kv->head_dim;
    float* out = reinterpret_cast<float*>(base + h.out_off);
    cudaStream_t s = (cudaStream_t)stream;
    // Pinned (mapped) host buffers: the inputs come in through a copy kernel and the merge
    // writes the output into h_out itself; pageable ones go through the copy engine.
    const void* m_in = mapped_device_ptr(h_in);
    float* m_out = static_cast<float*>(const_cast<void*>(mapped_device_ptr(h_out)));
    if (m_in && kvq8::aligned16(m_in) && h.in_bytes % 16 == 0) {
        const int n16 = (int)(h.in_bytes / 16);
        host_copy_kernel<<<(n16 + kCopyThreads * kCopyPer - 1) / (kCopyThreads * kCopyPer), kCopyThreads, 0, s>>>(
            static_cast<const uint4*>(m_in), reinterpret_cast<uint4*>(base), n16);
        if (kvq8::launch_status() != KVQ8_OK) return KVQ8_ERR_CUDA;
    } else if (cudaMemcpyAsync(base, h_in, h.in_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        return KVQ8_ERR_CUDA;
    }
    const bool direct_out = m_out && kvq8::aligned16(m_out);
    const int rc = kvq8::verify_impl(q, n_rows, n_q_heads, kv, q_pos0 + n_rows, q_pos0, nullptr, softmax_scale,
                                     direct_out ? m_out : out, base + h.ws_off, h.ws_bytes, n_split, stream, k_new,
                                     v_new);
    if (rc != KVQ8_OK || direct_out) return rc;
    const size_t out_bytes = (size_t)n_rows * n_q_heads * kv->head_dim * sizeof(float);
    return cudaMemcpyAsync(h_out, out, out_bytes, cudaMemcpyDeviceToHost, s) == cudaSuccess ? KVQ8_OK
                                                                                              : KVQ8_ERR_CUDA;
}

extern "C" int attn_verify_tree_q8(const float* q, int n_rows, int n_q_heads, const kvq8_cache* kv, int kv_len,
                                   int q_pos0, const uint32_t* window_mask, float softmax_scale, float* out,
                                   void* workspace, size_t workspace_bytes, int n_split, kvq8_stream_t stream) {
    if (!window_mask) return KVQ8_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(window_mask) & 3u) != 0) return KVQ8_ERR_MISALIGNED;
    return kvq8::verify_impl(q, n_rows, n_q_heads, kv, kv_len, q_pos0, window_mask, softmax_scale, out, workspace,
                             workspace_bytes, n_split, stream);
}

// ---------------------------------------------------------------------------------------
// attn_verify_q8_noalloc: the same computation for callers that cannot allocate device
// memory.  The split partials live in one file-scope device array that every GPU loading
// this library holds until the process exits; the entry point looks up that array's device
// address once per device and never calls cudaMalloc / cudaFree.
// ---------------------------------------------------------------------------------------
#include <mutex>

static __device__ __align__(256) unsigned char g_verify_noalloc_scratch[KVQ8_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The first call on a device
// performs the lookup (cudaGetSymbolAddress) with that device current; later calls reuse it.
int noalloc_scratch(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ8_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_verify_noalloc_scratch) != cudaSuccess || !p) return KVQ8_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return KVQ8_OK;
}

}  // namespace

extern "C" int attn_verify_q8_noalloc(const float* q, int n_rows, int n_q_heads, const kvq8_cache* kv, int kv_len,
                                      int q_pos0, float softmax_scale, float* out, int n_split,
                                      kvq8_stream_t stream) {
    using namespace kvq8;
    if (!kv) return KVQ8_ERR_INVALID_ARG;
    Plan pl;
    bool tc = false;
    const int rc = plan_causal(n_rows, n_q_heads, kv->head_dim, kv_len, kv->n_kv_heads, n_split, &pl, &tc);
    if (rc != KVQ8_OK) return rc;
    // the partials of this plan must fit the array; nothing is launched otherwise
    if (pl.ws_bytes > (size_t)KVQ8_NOALLOC_SCRATCH_BYTES) return KVQ8_ERR_WORKSPACE;
    void* scratch = nullptr;
    const int rs = noalloc_scratch(&scratch);
    if (rs != KVQ8_OK) return rs;
    return attn_verify_q8(q, n_rows, n_q_heads, kv, kv_len, q_pos0, softmax_scale, out, scratch,
                          (size_t)KVQ8_NOALLOC_SCRATCH_BYTES, n_split, stream);
}
