// verify_f16.cu -- multi-row verify attention over an fp16 KV pool (attn_verify_f16) and the
// fp32 -> fp16 append into such a pool (kvf16_append).
//
// Source: the multi-row verifier of "perf(gfx1100): share Q8 KV scans across verifier rows"
// (Summary: one pass over each K/V tile shared by every row of the window, split-context
// partials and their reducer), applied to the fp16 pool that "gfx12 WMMA kernel for the
// int8-KV QSA prompt attention" (Gating and Limits) leaves on the older kernel.
//
// The work split is that of the Q8_0 kernel (verify.cu): one thread block per (row chunk,
// context slice, KV head), 8 warps, 128-key tiles, q as fp16 hi + lo B fragments, lazy
// row maxima, P as fp16 hi + lo through shared memory, log-sum-exp partials merged by the
// combine kernel.  What the fp16 pool changes:
//   * K and V tiles are fp16 (twice the bytes of Q8_0): no dequantisation, no block scales;
//   * QK reads each K row's 8-dim group as one 16-byte load straight into the A fragment;
//   * PV reads the V^T A fragments with ldmatrix.trans from the row-major V tile, and the P
//     fragments are the B operand as they are (no per-block V scale to fold in);
//   * tiles are 16-byte-chunk swizzled with phase phi(row) = ((row & 1) << 2) | ((row >> 1) & 3)
//     (a permutation of 0..7 in which rows 2k and 2k+1 differ in bit 2), which keeps both the
//     QK quarter-warp loads and the ldmatrix row sets free of bank conflicts.
// Shared memory holds one K and one V tile (64 KB each at hd256), so hd256 runs one block per
// SM and hd128 two (up to 24 rows per chunk).
#include "common.cuh"
#include "verify_plan.cuh"

namespace kvq8 {

int launch_combine(const float* part_o, const float* part_ml, int n_split, int rows, int head_dim, float* out,
                   cudaStream_t stream);

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr float kLazy = 8.0f;    // log2 units: a row's reference maximum moves only when a score exceeds it by this
constexpr float kPShift = 4.0f;  // p is stored as p * 2^kPShift; with p <= 2^kLazy that stays <= 2^12

struct F16Params {
    const float* q;
    const uint16_t* k;  // fp16 bits [n_kv_heads][capacity][HD]
    const uint16_t* v;
    float* part_o;      // [n_split][rows_total][HD]
    float2* part_ml;    // [n_split][rows_total]
    int n_rows, n_q_heads, group, group_magic, capacity, kv_len, q_pos0, keys_per_split, rows_per_chunk;
    float qscale;       // softmax_scale * log2(e)
};

template <int HD, int NT>
struct SmemF16 {
    static constexpr int NB = HD / 32;       // 32-dim blocks
    static constexpr int RP = 8 * NT;        // padded rows per chunk
    static constexpr int PS = RP + 4;        // P-tile entries per key pair
    static constexpr int ROWB = HD * 2;      // bytes per key row of a tile
    static constexpr int kK = 0;
    static constexpr int kV = kK + kKT * ROWB;
    static constexpr int kQ = kV + kKT * ROWB;
    static constexpr int kP = kQ + NB * NT * 1024;
    static constexpr int kRed = kP + (kKT / 2) * PS * 8;
    static constexpr int kBytes = kRed + RP * kWarps * 4;
};

template <int HD, int NT>
constexpr int f16_min_blocks() {
    return (HD == 128 && NT <= 3) ? 2 : 1;
}
inline int f16_blocks_per_sm(int hd, int nt) { return (hd == 128 && nt <= 3) ? 2 : 1; }

__device__ __forceinline__ int phi(int row) { return ((row & 1) << 2) | ((row >> 1) & 3); }

__device__ __forceinline__ int div_group(int x, const F16Params& p) {
    return (int)(((uint32_t)x * (uint32_t)p.group_magic) >> 20);
}

// Rows [tile_key0, tile_key0 + kKT) of one fp16 plane into a swizzled tile; rows at or past
// key_end are zero-filled.  A thread copies the 16-byte chunks tid + k * kThreads: its row
// advances by a multiple of 8, so its swizzled chunk never changes.
template <int HD>
__device__ __forceinline__ void load_tile(uint8_t* smem, const uint16_t* plane, int64_t head_row0, int tile_key0,
                                          int key_end) {
    constexpr int ROWB = HD * 2;
    constexpr int CPR = ROWB / 16;                // chunks per row
    constexpr int ROWS_PER_PASS = kThreads / CPR;  // 8 (hd256) or 16 (hd128)
    static_assert(ROWS_PER_PASS % 8 == 0, "row step must keep the swizzle phase");
    const int n0 = threadIdx.x / CPR, c16 = threadIdx.x % CPR;
    const uint32_t dst0 = smem_u32(smem) + n0 * ROWB + ((c16 ^ phi(n0)) << 4);
    const uint16_t* src0 = plane + (head_row0 + tile_key0 + n0) * HD + c16 * 8;
    if (key_end - tile_key0 >= kKT) {  // a whole tile: every copy is live, offsets are immediates
#pragma unroll
        for (int k = 0; k < kKT / ROWS_PER_PASS; ++k) cp_async_16(dst0 + k * ROWS_PER_PASS * ROWB, src0 + k * ROWS_PER_PASS * HD, 16);
        return;
    }
    const int valid = key_end - tile_key0 - n0;
#pragma unroll
    for (int k = 0; k < kKT / ROWS_PER_PASS; ++k) {
        const bool ok = k * ROWS_PER_PASS < valid;
        cp_async_16(dst0 + k * ROWS_PER_PASS * ROWB, ok ? src0 + (int64_t)k * ROWS_PER_PASS * HD : src0 - (int64_t)n0 * HD,
                    ok ? 16 : 0);
    }
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ float exp2_int(int n) { return __uint_as_float((uint32_t)(n + 127) << 23); }

// Work split (8 warps):
//   QK : warp w owns keys 16w .. 16w+15 of the tile, all row tiles (as in the Q8_0 kernel);
//   PV : at hd256 warp w owns dims 32w .. 32w+31 (two m16 fragments), at hd128 dims
//        16w .. 16w+15 (one); each V^T fragment is one ldmatrix.x4.trans.
template <int HD, int NT>
__global__ void __launch_bounds__(kThreads, f16_min_blocks<HD, NT>()) verify_f16_kernel(const F16Params p) {
    using L = SmemF16<HD, NT>;
    constexpr int NB = L::NB, RP = L::RP, PS = L::PS, ROWB = L::ROWB;
    constexpr int MTW = HD / 128;  // m16 fragments of V^T per warp in PV
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* sK = smem + L::kK;
    uint8_t* sV = smem + L::kV;
    __half* sQ = reinterpret_cast<__half*>(smem + L::kQ);
    uint2* sP = reinterpret_cast<uint2*>(smem + L::kP);
    float* sRed = reinterpret_cast<float*>(smem + L::kRed);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int chunk = blockIdx.x, split = blockIdx.y, kvh = blockIdx.z;
    const int R = p.n_rows * p.group;
    const int rows_total = p.n_rows * p.n_q_heads;
    const int row0 = chunk * p.rows_per_chunk;
    const int rows_here = min(p.rows_per_chunk, R - row0);
    const int key_begin = split * p.keys_per_split;
    const int key_end = min(key_begin + p.keys_per_split, p.kv_len);
    const int64_t head_row0 = (int64_t)kvh * p.capacity;

    // The combine kernel may be launched now; it waits for this grid before reading.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // q rows of this chunk as fp16 hi/lo in mma B-fragment order (the Q8_0 kernel's layout):
    // entry (block b, n-tile nt, hi|lo, lane g*4+t) holds row 8nt+g, dims 32b+8t .. +7.
    {
        constexpr int GPR = HD / 8;
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
        if (key_begin < key_end) load_tile<HD>(sK, p.k, head_row0, key_begin, key_end);
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

    // visibility bound and output row of each owned row (-1 for padding rows)
    int vis_end[NT][2], grow[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int r = 8 * nt + 2 * t + c;
            if (r < rows_here) {
                const int rr = row0 + r;
                const int i = div_group(rr, p), hh = rr - i * p.group;
                vis_end[nt][c] = min(min(p.q_pos0 + i + 1, p.kv_len), key_end);
                grow[nt][c] = i * p.n_q_heads + kvh * p.group + hh;
            } else {
                vis_end[nt][c] = 0;
                grow[nt][c] = -1;
            }
        }
    const int vis_min = min(min(p.q_pos0 + div_group(row0, p) + 1, p.kv_len), key_end);
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

    // Per-lane shared-memory bases, fixed for the slice.
    // QK: row n0 = 16 warp + g (phase phi(g)) reads dims 32b + 8t .. +7 = chunk 4b + t, stored at
    // chunk (4b + t) ^ phi(g) = 4 (b ^ (phi(g) >> 2)) + (t ^ (phi(g) & 3)).
    const int k_ph = phi(g);
    const int k_hi = k_ph >> 2;
    const uint8_t* const k_lane = sK + (warp * 16 + g) * ROWB + ((t ^ (k_ph & 3)) << 4);
    const uint4* const q_lane = reinterpret_cast<const uint4*>(sQ) + lane;
    // PV: the four 8x8 matrices of a V^T fragment (dims d0 .. d0+15, keys 16 ks .. +15) are
    // rows of keys: matrix mi = lane / 8 covers keys 8 (mi >> 1) + r (r = lane & 7, phase
    // phi(r)) and the 8-dim chunk d0/8 + (mi & 1).
    uint32_t v_lane[MTW];
    {
        const int mi = lane >> 3, r = lane & 7;
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt) {
            const int d0 = HD == 256 ? 32 * warp + 16 * mt : 16 * warp;
            const int c16 = (d0 >> 3) + (mi & 1);
            v_lane[mt] = smem_u32(sV) + (8 * (mi >> 1) + r) * ROWB + ((c16 ^ phi(r)) << 4);
        }
    }
    const uint2* const p_lane = sP + t * PS + g;

#pragma unroll 1
    for (int tile0 = key_begin; tile0 < key_end; tile0 += kKT) {
        const int nk = min(kKT, key_end - tile0);
        cp_async_wait<0>();  // K of this tile landed
        __syncthreads();     // ... for every thread; every warp is done with the previous V
        load_tile<HD>(sV, p.v, head_row0, tile0, key_end);
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
                const uint8_t* kp = k_lane + ((b ^ k_hi) << 6);
                const uint4 k0 = *reinterpret_cast<const uint4*>(kp);             // row n0, dims 8t .. +7 of block b
                const uint4 k1 = *reinterpret_cast<const uint4*>(kp + 8 * ROWB);  // row n0 + 8
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_f16_16816(S[nt], k0.x, k1.x, k0.y, k1.y, qh[nt].x, qh[nt].y);
                    mma_f16_16816(S[nt], k0.z, k1.z, k0.w, k1.w, qh[nt].z, qh[nt].w);
                    mma_f16_16816(S[nt], k0.x, k1.x, k0.y, k1.y, ql[nt].x, ql[nt].y);
                    mma_f16_16816(S[nt], k0.z, k1.z, k0.w, k1.w, ql[nt].z, ql[nt].w);
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
                    if (tile_needs_mask && !(key < vis_end[nt][c])) s = -INFINITY;
                    need |= s > m_ref[nt][c] + kLazy;
                }
        if (__syncthreads_or(need)) {
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

        // every warp is done with K (the vote was a barrier): stream the next tile's K
        {
            const int next0 = tile0 + kKT;
            if (next0 < key_end) load_tile<HD>(sK, p.k, head_row0, next0, key_end);
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
        // P tile entry (key pair k, row r) = (hi, lo) of (p[2k][r], p[2k+1][r]); the partner key of
        // a pair sits 4 lanes away, so lane pairs swap one value.
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float v0 = S[nt][2 * h], v1 = S[nt][2 * h + 1];
                const bool ev = (g & 1) == 0;
                const float recv = __shfl_xor_sync(0xffffffffu, ev ? v1 : v0, 4);
                const float pe = ev ? v0 : recv;
                const float po = ev ? recv : v1;
                const __half2 ph = __floats2half2_rn(pe, po);
                const __half2 pl = __floats2half2_rn(pe - __low2float(ph), po - __high2float(ph));
                const int kl = n0 + 8 * h;
                sP[(kl >> 1) * PS + 8 * nt + 2 * t + (ev ? 0 : 1)] = make_uint2(h2_as_u32(ph), h2_as_u32(pl));
            }

        cp_async_wait<1>();  // V of this tile landed (the next K may still be in flight)
        __syncthreads();

        // ---------------- PV: O^T[dim][row] += V^T * (p 2^kPShift) ----------------
        const int n_ks = (nk + 15) >> 4;
#pragma unroll 2
        for (int ks = 0; ks < n_ks; ++ks) {
            uint2 pp01[NT], pp89[NT];  // (hi, lo) pairs of keys (2t, 2t+1) and (2t+8, 2t+9), row g of n-tile
            const uint2* pp = p_lane + ks * 8 * PS;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                pp01[nt] = pp[8 * nt];
                pp89[nt] = pp[4 * PS + 8 * nt];
            }
            uint32_t A[MTW][4];
#pragma unroll
            for (int mt = 0; mt < MTW; ++mt) ldmatrix_x4_trans(v_lane[mt] + ks * 16 * ROWB, A[mt]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int mt = 0; mt < MTW; ++mt) {
                    mma_f16_16816(O[mt][nt], A[mt][0], A[mt][1], A[mt][2], A[mt][3], pp01[nt].x, pp89[nt].x);
                    mma_f16_16816(O[mt][nt], A[mt][0], A[mt][1], A[mt][2], A[mt][3], pp01[nt].y, pp89[nt].y);
                }
        }
    }
    cp_async_wait<0>();
    __syncthreads();  // every warp is done with sP before sRed is reused

    // ---------------- write the slice partial ----------------
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
    const float inv = exp2_int(-(int)kPShift);
    // O^T fragment: lane holds dims d0 + g (c0, c1) and d0 + g + 8 (c2, c3) of rows 8nt + 2t + c
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            if (grow[nt][c] < 0) continue;
            float* dst = po + (int64_t)grow[nt][c] * HD;
#pragma unroll
            for (int mt = 0; mt < MTW; ++mt) {
                const int d0 = HD == 256 ? 32 * warp + 16 * mt : 16 * warp;
                dst[d0 + g] = O[mt][nt][c] * inv;
                dst[d0 + g + 8] = O[mt][nt][2 + c] * inv;
            }
        }
    if (warp == 0 && g == 0) {
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
                    make_float2(m == -INFINITY ? -INFINITY : m * kLn2, l * inv);
            }
    }
}

template <int HD, int NT>
int launch_f16(const F16Params& fp, const Plan& pl, int n_kv_heads, cudaStream_t stream) {
    constexpr int bytes = SmemF16<HD, NT>::kBytes;
    static SmemOptIn opt;
    if (opt.ensure(verify_f16_kernel<HD, NT>, bytes) != KVQ8_OK) return KVQ8_ERR_CUDA;
    dim3 grid(pl.n_chunks, pl.n_split, n_kv_heads);
    verify_f16_kernel<HD, NT><<<grid, kThreads, bytes, stream>>>(fp);
    return launch_status();
}

template <int HD>
int dispatch_f16(const F16Params& fp, const Plan& pl, int n_kv_heads, cudaStream_t s) {
    switch (pl.nt) {
        case 1: return launch_f16<HD, 1>(fp, pl, n_kv_heads, s);
        case 2: return launch_f16<HD, 2>(fp, pl, n_kv_heads, s);
        case 3: return launch_f16<HD, 3>(fp, pl, n_kv_heads, s);
        case 4: return launch_f16<HD, 4>(fp, pl, n_kv_heads, s);
        default: return KVQ8_ERR_UNSUPPORTED;
    }
}

// fp32 -> fp16 (round to nearest even) of K and V tokens into both planes of a pool: one
// thread per 4 values of one plane.
__global__ void __launch_bounds__(256) f16_append_kernel(const float4* __restrict__ k, const float4* __restrict__ v,
                                                         int64_t n_vec, int n_kv_heads, int hd4, uint16_t* kp,
                                                         uint16_t* vp, int capacity, int pos0) {
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= 2 * n_vec) return;
    const bool second = gid >= n_vec;
    const int64_t i = second ? gid - n_vec : gid;
    const float4 x = __ldg((second ? v : k) + i);
    const int64_t row_vecs = (int64_t)n_kv_heads * hd4;
    const int64_t tok = i / row_vecs;
    const int64_t rem = i - tok * row_vecs;
    const int h = (int)(rem / hd4), j4 = (int)(rem - (int64_t)h * hd4);
    uint16_t* dst = (second ? vp : kp) + (((int64_t)h * capacity + pos0 + tok) * hd4 + j4) * 4;
    const __half2 a = __floats2half2_rn(x.x, x.y), b = __floats2half2_rn(x.z, x.w);
    *reinterpret_cast<uint2*>(dst) = make_uint2(h2_as_u32(a), h2_as_u32(b));
}

}  // namespace
}  // namespace kvq8

extern "C" size_t attn_verify_f16_workspace_bytes(int n_rows, int n_q_heads, int head_dim, int kv_len,
                                                  int n_kv_heads, int n_split) {
    kvq8::Plan pl;
    if (kvq8::make_plan(n_rows, n_q_heads, head_dim, kv_len, n_kv_heads, n_split, &pl, 0,
                        kvq8::f16_blocks_per_sm) != KVQ8_OK)
        return 0;
    return pl.ws_bytes;
}

extern "C" int attn_verify_f16(const float* q, int n_rows, int n_q_heads, const kvf16_cache* kv, int kv_len,
                               int q_pos0, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                               int n_split, kvq8_stream_t stream) {
    using namespace kvq8;
    if (!kv || !q || !out || !kv->k || !kv->v) return KVQ8_ERR_INVALID_ARG;
    if (kv->n_kv_heads < 1 || kv->capacity < 1 || q_pos0 < 0 || kv_len > kv->capacity) return KVQ8_ERR_INVALID_ARG;
    if (!(softmax_scale == softmax_scale) || softmax_scale == INFINITY || softmax_scale == -INFINITY)
        return KVQ8_ERR_INVALID_ARG;
    Plan pl;
    const int rc = make_plan(n_rows, n_q_heads, kv->head_dim, kv_len, kv->n_kv_heads, n_split, &pl, 0,
                             f16_blocks_per_sm);
    if (rc != KVQ8_OK) return rc;
    if (!aligned16(q) || !aligned16(out) || !aligned16(kv->k) || !aligned16(kv->v)) return KVQ8_ERR_MISALIGNED;
    if (!workspace || workspace_bytes < pl.ws_bytes) return KVQ8_ERR_WORKSPACE;
    if (!aligned16(workspace)) return KVQ8_ERR_MISALIGNED;
    F16Params fp;
    fp.q = q;
    fp.k = kv->k;
    fp.v = kv->v;
    const size_t rows_total = (size_t)n_rows * n_q_heads;
    const size_t o_bytes = (size_t)pl.n_split * rows_total * kv->head_dim * sizeof(float);
    fp.part_o = static_cast<float*>(workspace);
    fp.part_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) + ((o_bytes + 255) / 256) * 256);
    fp.n_rows = n_rows;
    fp.n_q_heads = n_q_heads;
    fp.group = n_q_heads / kv->n_kv_heads;
    fp.group_magic = ((1 << 20) + fp.group - 1) / fp.group;  // exact: rows * group <= 32 * 64^2 < 2^20
    fp.capacity = kv->capacity;
    fp.kv_len = kv_len;
    fp.q_pos0 = q_pos0;
    fp.keys_per_split = pl.keys_per_split;
    fp.rows_per_chunk = pl.rows_per_chunk;
    fp.qscale = softmax_scale * kLog2e;
    cudaStream_t s = (cudaStream_t)stream;
    const int r1 = pl.hd == 128 ? dispatch_f16<128>(fp, pl, kv->n_kv_heads, s)
                                : dispatch_f16<256>(fp, pl, kv->n_kv_heads, s);
    if (r1 != KVQ8_OK) return r1;
    return launch_combine(fp.part_o, reinterpret_cast<const float*>(fp.part_ml), pl.n_split, (int)rows_total,
                          kv->head_dim, out, s);
}

extern "C" int kvf16_append(const float* k, const float* v, int n_tok, const kvf16_cache* kv, int pos0,
                            kvq8_stream_t stream) {
    using namespace kvq8;
    if (!kv || n_tok < 0 || pos0 < 0) return KVQ8_ERR_INVALID_ARG;
    if (kv->n_kv_heads <= 0 || kv->head_dim <= 0 || kv->capacity <= 0) return KVQ8_ERR_INVALID_ARG;
    if (kv->head_dim % 4) return KVQ8_ERR_UNSUPPORTED;
    if ((int64_t)pos0 + n_tok > kv->capacity) return KVQ8_ERR_INVALID_ARG;
    if (n_tok == 0) return KVQ8_OK;
    if (!k || !v || !kv->k || !kv->v) return KVQ8_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(kv->k) || !aligned16(kv->v)) return KVQ8_ERR_MISALIGNED;
    const int hd4 = kv->head_dim / 4;
    const int64_t n_vec = (int64_t)n_tok * kv->n_kv_heads * hd4;
    const int64_t grid = (2 * n_vec + 255) / 256;
    if (grid > 0x7fffffffLL) return KVQ8_ERR_UNSUPPORTED;
    f16_append_kernel<<<(unsigned)grid, 256, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const float4*>(k), reinterpret_cast<const float4*>(v), n_vec, kv->n_kv_heads, hd4,
        const_cast<uint16_t*>(kv->k), const_cast<uint16_t*>(kv->v), kv->capacity, pos0);
    return launch_status();
}
