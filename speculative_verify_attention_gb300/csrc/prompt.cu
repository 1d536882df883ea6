// prompt.cu -- prompt-chunk attention over a Q8_0 GQA cache on the tcgen05 tensor cores
// (attn_prompt_q8).
//
// Source: "gfx12 WMMA kernel for the int8-KV QSA prompt attention", How: int8-KV prompt
// attention on the tensor cores with fp32 accumulation, online softmax, the V scale folded
// into the operands, and the heads that share one KV head stacked as the rows of the
// tile; Measurements: a 32K-token int8 context with a 2,048-query chunk.
//
// GB300 design: one CTA per (128-row tile of (query, head) pairs, KV head); rows r = i*g + hh
// of one KV head, so the 12 heads of a query and ~11 consecutive queries share every K/V
// tile.  Sixteen warps, each with one role:
//   warp 0      producer: 1-D bulk async copies of the int8 codes and fp16 scales of a
//               64-key tile into a 2-stage staging ring (mbarrier transaction counts);
//   warp 1      MMA issuer (one thread) and tensor-memory owner;
//   warps 2-5   softmax, one thread per row (each warp reads its 32-lane quarter of TMEM);
//   warps 6-15  dequantisers: int8 -> fp16 exactly (byte permute + magic-bias subtract), then
//               times the block scale (one fp16 rounding), written to double-buffered
//               128-byte-swizzled K^ and V^ tiles in shared memory.
// With an fp16 pool (or the fp16 copy of the two-pass route) there is nothing to dequantise:
// warp 0 loads the K tiles and warp 6 the V tiles straight into K^ / V^ by tensor copies, and
// warps 7-15 idle.
// Tensor memory (512 columns): Q as fp16 pairs (128), O fp32 (256), two S buffers (64 each)
// whose first 32 columns take P as fp16 pairs after the softmax has read S.
//   S = Q K^T : tcgen05.mma kind::f16, A = Q from TMEM, B = K^ (K-major), M=128 N=64 K=256
//   O += P V^ : A = P from TMEM, B = V^ (MN-major), M=128 N=256 K=64
// The softmax keeps a per-row reference maximum and rescales the O row in TMEM only when a
// new maximum exceeds it by more than 2^8, so p stays <= 256 in fp16.  Tiles past the
// causal bound of the last row are never loaded; only the diagonal tile is masked.
// Barriers that many threads signal take one arrival per warp (after __syncwarp), not one
// per thread.  Every mbarrier wait is bounded: on timeout the kernel records an error flag (read with
// kvq8_device_error) and returns after releasing its tensor memory.
#include <mutex>

#include "common.cuh"
#include "tc.cuh"
#include "tmap.cuh"

__device__ unsigned int g_kvq8_device_error = 0;

namespace kvq8 {

int launch_combine(const float* part_o, const float* part_ml, int n_split, int rows, int head_dim, float* out,
                   cudaStream_t stream);

namespace {

constexpr int BM = 128;
// keys per tile: 64 at hd256, 128 at hd128 (where a 64-key tile leaves the tensor core idle
// behind the per-row softmax)
__host__ __device__ constexpr int bn_for(int hd) { return hd == 128 ? 128 : 64; }
constexpr int kSoftWarp0 = 2, kDeqWarp0 = 6, kDeqThreads = 320;
constexpr int kThreads = (kDeqWarp0 + kDeqThreads / 32) * 32;   // 512: 128 registers per thread fill the SM
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMaxSegments = 8;

// tensor memory columns: Q (hd/2 columns of fp16 pairs) at 0, O (hd fp32 columns) at 128, then
// two S buffers of BN columns (384 + 2 x 64 at hd256, 256 + 2 x 128 at hd128)
constexpr uint32_t TM_Q = 0, TM_O = 128, TM_NCOLS = 512;

// A K^ buffer is free again when its QK has completed (B_S_FULL) and a V^ buffer when its PV has
// (B_PV_DONE): those commits already mark the events, and every commit costs the one issuing
// thread (two extra commits per tile measured 4-5 % slower at hd256).
enum { B_ST_FULL = 0, B_ST_EMPTY = 2, B_K_FULL = 4, B_V_FULL = 6, B_S_FULL = 8, B_P_FULL = 10, B_PV_DONE = 12,
       B_Q_READY = 14, B_COUNT = 15 };

// Shared memory layout for head dim HD (bytes, 1024-aligned tiles):
//   K^, V^ : 2 buffers each of [HD/64 atoms][64 keys][128 B], 128B-swizzled fp16 (K-major for
//            K^, read as MN-major for V^)
//   staging: 2 stages of K codes | V codes | K scales | V scales for one tile; at hd128 each
//            scale area has 16 spare bytes so that a tile's scales sit at the same offset mod 16
//            as in global memory
template <int HD>
struct PL {
    static constexpr int BN = bn_for(HD);
    static constexpr uint32_t TM_S0 = HD == 128 ? 256 : 384;
    static_assert(TM_S0 + 2 * BN <= TM_NCOLS && TM_O + HD <= TM_S0, "tensor memory map");
    static constexpr int HAT_BYTES = (HD / 64) * BN * 128;
    static constexpr int SM_KHAT = 0;
    static constexpr int SM_VHAT = 2 * HAT_BYTES;
    static constexpr int SM_STAGE = 4 * HAT_BYTES;
    static constexpr int SC_PAD = HD == 128 ? 16 : 0;
    static constexpr int ST_KC = 0, ST_VC = BN * HD, ST_KS = 2 * BN * HD, ST_VS = ST_KS + BN * HD / 16 + SC_PAD;
    static constexpr int STAGE_BYTES = (2 * BN * HD + 2 * (BN * HD / 16 + SC_PAD) + 1023) / 1024 * 1024;
    static constexpr int SM_BAR = SM_STAGE + 2 * STAGE_BYTES;
    static constexpr int SM_TMEM_SLOT = SM_BAR + B_COUNT * 8;
    static constexpr int SM_SEG = SM_TMEM_SLOT + 16;  // this CTA's work segments (written by thread 0)
    static constexpr int SMEM_BYTES = SM_SEG + 8 * 5 * 4 + 16;
    static constexpr int kChunks = BN * HD / 16;      // 16-code chunks of one plane of a tile
    static constexpr uint32_t IDESC_QK = tc::idesc_f16_f32(BM, BN, false);
    static constexpr uint32_t IDESC_PV = tc::idesc_f16_f32(BM, HD, true);
    static_assert(STAGE_BYTES % 1024 == 0 && HAT_BYTES % 1024 == 0, "tiles stay 1024-byte aligned");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct PromptParams {
    const uint16_t* q;
    const int8_t* kc;
    const uint16_t* ks;
    const int8_t* vc;
    const uint16_t* vs;
    float* part_o;     // [n_parts][n_q * n_q_heads][HD]
    float2* part_ml;   // [n_parts][n_q * n_q_heads]
    int n_q, n_q_heads, group, capacity, kv_len, q_pos0, rows, n_mtiles, n_items, n_parts;
    long long units;   // total tiles over all (KV head, row tile) items
    float scale_log2;
    // fp16 pools: 3-D tensor maps (dims, keys < kv_len, KV heads) of the K and V planes with a
    // 64-dim x 64-key box and the 128-byte swizzle of the K^/V^ tiles
    CUtensorMap tmap_k, tmap_v;
};

// Pool formats of the prompt kernel.
enum { kPoolQ8 = 0, kPoolK8V4 = 1, kPoolF16 = 2 };

// Geometry of one work item: rows [r0, r0 + rows_here) of KV head kvh see keys < key_hi;
// every row sees at least the keys < key_lo.
struct Item {
    int kvh, r0, rows_here, key_lo, key_hi, n_tiles;
};

__host__ __device__ inline Item item_geometry(int it, int n_mtiles, int rows, int group, int kv_len, int q_pos0,
                                              int bn) {
    Item g;
    g.kvh = it / n_mtiles;
    const int m = it - g.kvh * n_mtiles;
    g.r0 = m * BM;
    g.rows_here = rows - g.r0 < BM ? rows - g.r0 : BM;
    const long long hi = (long long)q_pos0 + (g.r0 + g.rows_here - 1) / group + 1;
    const long long lo = (long long)q_pos0 + g.r0 / group + 1;
    g.key_hi = (int)(hi < kv_len ? hi : kv_len);
    g.key_lo = (int)(lo < kv_len ? lo : kv_len);
    g.n_tiles = (g.key_hi + bn - 1) / bn;
    return g;
}

// Stream-K split: CTA c of G owns the units [floor(c U / G), floor((c+1) U / G)).
__host__ __device__ inline long long unit_begin(long long c, long long U, long long G) { return c * U / G; }
// First CTA whose range contains unit u.
__host__ __device__ inline long long cta_of_unit(long long u, long long U, long long G) { return ((u + 1) * G - 1) / U; }

struct Segment {
    int item, t0, t1, part, last;  // tiles [t0, t1) of item; part index; last = owns the item's final tile
};

template <int BN>
__device__ int cta_segments(const PromptParams& p, int c, int G, Segment* seg) {
    const long long u0 = unit_begin(c, p.units, G), u1 = unit_begin(c + 1, p.units, G);
    int n = 0;
    long long s = 0;
    for (int it = 0; it < p.n_items && s < u1 && n < kMaxSegments; ++it) {
        const Item g = item_geometry(it, p.n_mtiles, p.rows, p.group, p.kv_len, p.q_pos0, BN);
        const long long e = s + g.n_tiles;
        if (e > u0) {
            const long long a = s > u0 ? s : u0, b = e < u1 ? e : u1;
            seg[n].item = it;
            seg[n].t0 = (int)(a - s);
            seg[n].t1 = (int)(b - s);
            seg[n].part = (int)(c - cta_of_unit(s, p.units, G));
            seg[n].last = (b == e) ? 1 : 0;
            ++n;
        }
        s = e;
    }
    return n;
}

__device__ __forceinline__ void flag_timeout() { atomicOr(&g_kvq8_device_error, 1u); }

// (a, b) * s + c, one packed fp32 FMA: each half rounded exactly as fmaf would.
__device__ __forceinline__ float2 fma2_sc(float a, float b, float s, float c) {
    float2 r;
    asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %4};\n mov.b64 z, {%5, %5};\n"
        " fma.rn.f32x2 z, x, y, z;\n mov.b64 {%0, %1}, z;\n}\n"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a), "f"(b), "f"(s), "f"(c));
    return r;
}
// (s0, s1) += (a, b), one packed fp32 add: each half rounded as a plain add.
__device__ __forceinline__ void add2(float& s0, float& s1, float a, float b) {
    asm("{\n .reg .b64 x, z;\n mov.b64 x, {%2, %3};\n mov.b64 z, {%0, %1};\n"
        " add.rn.f32x2 z, z, x;\n mov.b64 {%0, %1}, z;\n}\n"
        : "+f"(s0), "+f"(s1)
        : "f"(a), "f"(b));
}

// The order in which the dequantisers take a tile's 16-dim chunks (one chunk: 16 codes of one
// key, written as two 16-byte swizzled pieces):
//   c = ((m * 2 + sw) * NAP + ap) * 8 + kp * 4 + jj  ->  key 2m + kp, atom 2 ap + (sw ^ kp), chunk jj
// (NAP = HD / 128 atom pairs).  A quarter warp (8 consecutive chunks) thus holds the 4 chunks of
// one 64-dim atom of key 2m and the 4 chunks of the neighbouring atom of key 2m + 1: its swizzled
// stores cover the 32 banks once (key 2m lands on even chunk slots, key 2m + 1 on odd ones), and
// so do its 16-byte code loads (the two keys' 64-byte runs sit 128 bytes apart modulo the bank
// line).  A half warp holds key 2m's atoms {sw, sw + 2} and key 2m + 1's other two, so the 8-byte
// loads of 4-bit codes (two pieces of 32 bytes per key) fill distinct banks as well.
template <int HD>
__device__ __forceinline__ void chunk_of(int c, int& n, int& j16) {
    constexpr int NAP = HD / 128;
    const int jj = c & 3, kp = (c >> 2) & 1, ap = (c >> 3) % NAP;
    const int rest = (c >> 3) / NAP, sw = rest & 1, m = rest >> 1;
    n = 2 * m + kp;
    j16 = 4 * (2 * ap + (sw ^ kp)) + jj;
}

// Convert one plane tile (codes + scales in staging) into the swizzled fp16 tile:
// element (key n, dim j) -> atom j/64, row n, 16-byte chunk ((j%64)/8) ^ (n%8).
// kDeqThreads threads share the tile's kChunks chunks of 16 codes (HD/16 chunks per key), in
// the chunk_of order.
template <int HD>
__device__ __forceinline__ void dequant_tile(const uint8_t* codes, const uint16_t* scales, uint8_t* hat, int nk,
                                             int d) {
    constexpr int kChunks = PL<HD>::kChunks;
#pragma unroll
    for (int k = 0; k < (kChunks + kDeqThreads - 1) / kDeqThreads; ++k) {
        const int c = d + kDeqThreads * k;
        if (c >= kChunks) break;
        int n, j16;
        chunk_of<HD>(c, n, j16);
        uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
        if (n < nk) {
            const uint4 raw = *reinterpret_cast<const uint4*>(codes + n * HD + j16 * 16);
            const __half2 sc = __half2half2(__ushort_as_half(scales[n * (HD / 32) + (j16 >> 1)]));
            const uint32_t w[4] = {raw.x ^ 0x80808080u, raw.y ^ 0x80808080u, raw.z ^ 0x80808080u,
                                   raw.w ^ 0x80808080u};
            uint32_t h[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint32_t lo = biased_bytes_to_half2<0x4140>(w[e]);
                uint32_t hi = biased_bytes_to_half2<0x4342>(w[e]);
                const __half2 a = __hmul2(*reinterpret_cast<const __half2*>(&lo), sc);
                const __half2 b = __hmul2(*reinterpret_cast<const __half2*>(&hi), sc);
                h[2 * e] = *reinterpret_cast<const uint32_t*>(&a);
                h[2 * e + 1] = *reinterpret_cast<const uint32_t*>(&b);
            }
            o0 = make_uint4(h[0], h[1], h[2], h[3]);
            o1 = make_uint4(h[4], h[5], h[6], h[7]);
        }
        const int base = (j16 >> 2) * (PL<HD>::BN * 128) + (n >> 3) * 1024 + (n & 7) * 128;
        const int c0 = 2 * (j16 & 3);
        *reinterpret_cast<uint4*>(hat + base + ((c0 ^ (n & 7)) << 4)) = o0;
        *reinterpret_cast<uint4*>(hat + base + (((c0 + 1) ^ (n & 7)) << 4)) = o1;
    }
}

// The 4-bit V tile of a K8V4 pool (HD/2 bytes per key, element 2m in the low nibble of byte
// m, value (nibble - 8) * scale) into the same swizzled fp16 tile: each byte becomes its two
// codes exactly (nib_byte_to_half2), and one multiply by the scale rounds once, as for Q8_0.
// Chunks in the chunk_of order.
template <int HD>
__device__ __forceinline__ void dequant_tile_v4(const uint8_t* codes, const uint16_t* scales, uint8_t* hat, int nk,
                                                int d) {
    constexpr int kChunks = PL<HD>::kChunks;  // 16-dim items per tile
#pragma unroll
    for (int k = 0; k < (kChunks + kDeqThreads - 1) / kDeqThreads; ++k) {
        const int c = d + kDeqThreads * k;
        if (c >= kChunks) break;
        int n, j16;
        chunk_of<HD>(c, n, j16);
        uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
        if (n < nk) {
            const uint2 raw = *reinterpret_cast<const uint2*>(codes + n * (HD / 2) + j16 * 8);
            const __half2 sc = __half2half2(__ushort_as_half(scales[n * (HD / 32) + (j16 >> 1)]));
            const uint32_t e[8] = {nib_byte_to_half2<0>(raw.x), nib_byte_to_half2<1>(raw.x), nib_byte_to_half2<2>(raw.x),
                                   nib_byte_to_half2<3>(raw.x), nib_byte_to_half2<0>(raw.y), nib_byte_to_half2<1>(raw.y),
                                   nib_byte_to_half2<2>(raw.y), nib_byte_to_half2<3>(raw.y)};
            uint32_t h[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) h[m] = h2_as_u32(__hmul2(u32_as_h2(e[m]), sc));
            o0 = make_uint4(h[0], h[1], h[2], h[3]);
            o1 = make_uint4(h[4], h[5], h[6], h[7]);
        }
        const int base = (j16 >> 2) * (PL<HD>::BN * 128) + (n >> 3) * 1024 + (n & 7) * 128;
        const int c0 = 2 * (j16 & 3);
        *reinterpret_cast<uint4*>(hat + base + ((c0 ^ (n & 7)) << 4)) = o0;
        *reinterpret_cast<uint4*>(hat + base + (((c0 + 1) ^ (n & 7)) << 4)) = o1;
    }
}

// The dequantising pass of the two-pass route: keys < n_keys of the pool's K and V planes
// ([n_kv_heads][capacity] rows of codes and scales) as fp16 planes [n_kv_heads][n_keys][hd] in
// the workspace.  Each value is code x scale rounded once to fp16, exactly as the
// dequantisers of the one-pass kernel compute it, so both routes feed the tensor cores the
// same operands.  One thread per 8 consecutive values: 8 code bytes (4 for a 4-bit V plane) and
// their scale in, 16 bytes out, so that each warp instruction loads 256 (128) and stores 512
// contiguous bytes (one thread per 32-value block, with its four 16-byte stores 64 bytes apart
// across the warp, half-filled every sector and measured 1-2 % slower on the prompt call).
// blockIdx.y = plane * n_kv_heads + KV head (plane 0 = K, 1 = V); blocks stride along x.
struct DequantParams {
    const int8_t* kc;
    const uint16_t* ks;
    const int8_t* vc;
    const uint16_t* vs;
    uint16_t* k16;
    uint16_t* v16;
    int hd, n_keys, capacity, n_kv_heads;
};

template <bool V4>
__global__ void __launch_bounds__(256) dequant_planes_kernel(const DequantParams p) {
    const int plane = blockIdx.y / p.n_kv_heads, h = blockIdx.y - plane * p.n_kv_heads;
    const bool vplane = plane == 1;
    const int g_shift = p.hd == 256 ? 5 : 4;  // 8-value groups per key: 32 or 16
    const int8_t* codes = vplane ? p.vc : p.kc;
    const uint16_t* scales = (vplane ? p.vs : p.ks) + (size_t)h * p.capacity * (p.hd / 32);
    uint16_t* dst_plane = (vplane ? p.v16 : p.k16) + (size_t)h * p.n_keys * p.hd;
    const int n_groups = p.n_keys << g_shift;
    for (int b = blockIdx.x * 256 + threadIdx.x; b < n_groups; b += gridDim.x * 256) {
        const int n = b >> g_shift, g8 = b & ((1 << g_shift) - 1);
        const __half2 sc = __half2half2(__ushort_as_half(scales[(size_t)n * (p.hd / 32) + (g8 >> 2)]));
        uint32_t o[4];
        if (V4 && vplane) {
            const uint32_t w =
                *reinterpret_cast<const uint32_t*>(codes + ((size_t)h * p.capacity + n) * (p.hd / 2) + 4 * g8);
            o[0] = h2_as_u32(__hmul2(u32_as_h2(nib_byte_to_half2<0>(w)), sc));
            o[1] = h2_as_u32(__hmul2(u32_as_h2(nib_byte_to_half2<1>(w)), sc));
            o[2] = h2_as_u32(__hmul2(u32_as_h2(nib_byte_to_half2<2>(w)), sc));
            o[3] = h2_as_u32(__hmul2(u32_as_h2(nib_byte_to_half2<3>(w)), sc));
        } else {
            const uint2 r = *reinterpret_cast<const uint2*>(codes + ((size_t)h * p.capacity + n) * p.hd + 8 * g8);
            const uint32_t x0 = r.x ^ 0x80808080u, x1 = r.y ^ 0x80808080u;
            o[0] = h2_as_u32(__hmul2(u32_as_h2(biased_bytes_to_half2<0x4140>(x0)), sc));
            o[1] = h2_as_u32(__hmul2(u32_as_h2(biased_bytes_to_half2<0x4342>(x0)), sc));
            o[2] = h2_as_u32(__hmul2(u32_as_h2(biased_bytes_to_half2<0x4140>(x1)), sc));
            o[3] = h2_as_u32(__hmul2(u32_as_h2(biased_bytes_to_half2<0x4342>(x1)), sc));
        }
        *reinterpret_cast<uint4*>(dst_plane + (size_t)n * p.hd + 8 * g8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// One box of a 3-D tensor map into shared memory, completion counted on `mbar` in bytes.
// x (the dim coordinate) is a multiple of 64 fp16 = 128 bytes, as a tiled copy requires.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar)
        : "memory");
}

// POOL: kPoolQ8, kPoolK8V4 (4-bit V codes) or kPoolF16 (the producer loads the fp16 tiles
// straight into K^ and V^ with tensor copies; no staging and no dequantisation).
template <int HD, int POOL = kPoolQ8>
__global__ void __launch_bounds__(kThreads, 1) prompt_attn_kernel(const __grid_constant__ PromptParams p) {
    constexpr bool V4 = POOL == kPoolK8V4, F16 = POOL == kPoolF16;
    using L = PL<HD>;
    constexpr int SM_KHAT = L::SM_KHAT, SM_VHAT = L::SM_VHAT, HAT_BYTES = L::HAT_BYTES, SM_STAGE = L::SM_STAGE;
    constexpr int STAGE_BYTES = L::STAGE_BYTES, SM_BAR = L::SM_BAR, SM_TMEM_SLOT = L::SM_TMEM_SLOT, SM_SEG = L::SM_SEG;
    constexpr int ST_KC = L::ST_KC, ST_VC = L::ST_VC, ST_KS = L::ST_KS, ST_VS = L::ST_VS;
    constexpr uint32_t IDESC_QK = L::IDESC_QK, IDESC_PV = L::IDESC_PV;
    constexpr int BN = L::BN;
    constexpr uint32_t TM_S0 = L::TM_S0;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar = sbase + SM_BAR;
    auto B = [&](int id) { return bar + 8u * (uint32_t)id; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM_TMEM_SLOT);

    Segment* seg = reinterpret_cast<Segment*>(smem + SM_SEG);
    int* n_seg_slot = reinterpret_cast<int*>(smem + SM_SEG + kMaxSegments * (int)sizeof(Segment));

    if (threadIdx.x == 0) {
        *n_seg_slot = cta_segments<BN>(p, blockIdx.x, gridDim.x, seg);
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(B(B_ST_FULL + s), 1);
            tc::mbar_init(B(B_ST_EMPTY + s), kDeqThreads / 32);  // one arrival per warp
            tc::mbar_init(B(B_K_FULL + s), F16 ? 1 : kDeqThreads / 32);  // F16: the producer's expect_tx
            tc::mbar_init(B(B_V_FULL + s), F16 ? 1 : kDeqThreads / 32);
            tc::mbar_init(B(B_S_FULL + s), 1);
            tc::mbar_init(B(B_P_FULL + s), 4);
            tc::mbar_init(B(B_PV_DONE + s), 1);
        }
        tc::mbar_init(B(B_Q_READY), 4);
        tc::mbar_init_fence();
    }
    if (warp == 1) tc::tmem_alloc(smem_u32(tmem_slot), TM_NCOLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int n_seg = *n_seg_slot;

    if ((warp == 0 || warp == kDeqWarp0) && F16) {
        // ---------------------------------------------------------------- producers (fp16 pool)
        // K copies from warp 0, V copies from the first (idle) dequantiser warp: a K slot frees
        // when its QK completes, a V slot only when its PV does, and one thread issuing both
        // held each K copy behind the previous tile's V slot (1-2 % at hd256)
        const bool vprod = warp == kDeqWarp0;
        if (lane == 0) {
            constexpr uint32_t plane_bytes = (uint32_t)(HD / 64) * BN * 128;  // full boxes, past-the-end keys zero-filled
            int j = 0;
            bool ok = true;
            for (int si = 0; ok && si < n_seg; ++si) {
                const Item g = item_geometry(seg[si].item, p.n_mtiles, p.rows, p.group, p.kv_len, p.q_pos0, BN);
                for (int t = seg[si].t0; t < seg[si].t1; ++t, ++j) {
                    const int b = j & 1, use = j >> 1;
                    const int key0 = t * BN;
                    // slot b frees when QK (K) or PV (V) of tile j - 2 completes; that commit cannot
                    // have moved on a further phase, since tile j's MMAs need this very copy
                    const int e_bar = vprod ? B_PV_DONE : B_S_FULL, f_bar = vprod ? B_V_FULL : B_K_FULL;
                    if (j >= 2 && !tc::mbar_wait(B(e_bar + b), (use - 1) & 1, kWaitLimit)) { ok = false; break; }
                    tc::mbar_arrive_expect_tx(B(f_bar + b), plane_bytes);
                    const uint32_t dst = sbase + (vprod ? SM_VHAT : SM_KHAT) + b * HAT_BYTES;
                    const CUtensorMap* map = vprod ? &p.tmap_v : &p.tmap_k;
                    for (int a = 0; a < HD / 64; ++a)
                        tma_load_3d(dst + a * (BN * 128), map, 64 * a, key0, g.kvh, B(f_bar + b));
                }
            }
            if (!ok) flag_timeout();
            // never leave the block while a copy into its shared memory is in flight
            const int f_bar = vprod ? B_V_FULL : B_K_FULL;
            for (int i = max(0, j - 2); i < j; ++i)
                if (!tc::mbar_wait(B(f_bar + (i & 1)), (i >> 1) & 1, kWaitLimit)) flag_timeout();
        }
    } else if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            int j = 0;
            bool ok = true;
            for (int si = 0; ok && si < n_seg; ++si) {
                const Item g = item_geometry(seg[si].item, p.n_mtiles, p.rows, p.group, p.kv_len, p.q_pos0, BN);
                for (int t = seg[si].t0; t < seg[si].t1; ++t, ++j) {
                    const int s = j & 1, use = j >> 1;
                    if (j >= 2 && !tc::mbar_wait(B(B_ST_EMPTY + s), (use - 1) & 1, kWaitLimit)) { ok = false; break; }
                    const int key0 = t * BN;
                    const int nk = min(BN, g.key_hi - key0);
                    const int64_t row0 = (int64_t)g.kvh * p.capacity + key0;
                    const uint32_t st = sbase + SM_STAGE + s * STAGE_BYTES;
                    constexpr int v_row = V4 ? HD / 2 : HD;  // V code bytes per key
                    if constexpr (HD == 256) {  // code rows and a key's 16 bytes of scales: 16-byte multiples
                        tc::mbar_arrive_expect_tx(B(B_ST_FULL + s), (uint32_t)(nk * (HD + v_row + 2 * (HD / 16))));
                        tc::bulk_g2s(st + ST_KC, p.kc + row0 * HD, nk * HD, B(B_ST_FULL + s));
                        tc::bulk_g2s(st + ST_VC, p.vc + row0 * v_row, nk * v_row, B(B_ST_FULL + s));
                        tc::bulk_g2s(st + ST_KS, p.ks + row0 * (HD / 32), nk * (HD / 16), B(B_ST_FULL + s));
                        tc::bulk_g2s(st + ST_VS, p.vs + row0 * (HD / 32), nk * (HD / 16), B(B_ST_FULL + s));
                    } else {
                        // a key's scales are 8 bytes: the tile's scales start 0 or 8 bytes past a
                        // 16-byte boundary (off) and land at the same offset in the stage.  The
                        // 16-byte aligned interior goes by bulk copy, an 8-byte head or tail by a
                        // plain load; the arrival comes after the plain stores (release).
                        const int off = (int)(row0 & 1) * 8, end = off + nk * 8;
                        const int a = off == 0 ? 0 : 16, bnd = end & ~15;
                        const int inner = bnd > a ? bnd - a : 0;
                        tc::mbar_expect_tx(B(B_ST_FULL + s), (uint32_t)(nk * (HD + v_row) + 2 * inner));
                        tc::bulk_g2s(st + ST_KC, p.kc + row0 * HD, nk * HD, B(B_ST_FULL + s));
                        tc::bulk_g2s(st + ST_VC, p.vc + row0 * v_row, nk * v_row, B(B_ST_FULL + s));
                        const uint8_t* gk = reinterpret_cast<const uint8_t*>(p.ks + row0 * (HD / 32)) - off;
                        const uint8_t* gv = reinterpret_cast<const uint8_t*>(p.vs + row0 * (HD / 32)) - off;
                        if (inner > 0) {
                            tc::bulk_g2s(st + ST_KS + a, gk + a, inner, B(B_ST_FULL + s));
                            tc::bulk_g2s(st + ST_VS + a, gv + a, inner, B(B_ST_FULL + s));
                        }
                        uint8_t* sst = smem + SM_STAGE + s * STAGE_BYTES;
                        if (off == 8) {
                            *reinterpret_cast<uint2*>(sst + ST_KS + 8) = __ldg(reinterpret_cast<const uint2*>(gk + 8));
                            *reinterpret_cast<uint2*>(sst + ST_VS + 8) = __ldg(reinterpret_cast<const uint2*>(gv + 8));
                        }
                        if ((end & 15) == 8) {
                            *reinterpret_cast<uint2*>(sst + ST_KS + end - 8) =
                                __ldg(reinterpret_cast<const uint2*>(gk + end - 8));
                            *reinterpret_cast<uint2*>(sst + ST_VS + end - 8) =
                                __ldg(reinterpret_cast<const uint2*>(gv + end - 8));
                        }
                        tc::mbar_arrive(B(B_ST_FULL + s));
                    }
                }
            }
            if (!ok) flag_timeout();
            // never leave the block while a copy into its shared memory is in flight
            for (int i = max(0, j - 2); i < j; ++i)
                if (!tc::mbar_wait(B(B_ST_FULL + (i & 1)), (i >> 1) & 1, kWaitLimit)) flag_timeout();
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            int j = 0, pv_issued = 0;
            // One thread issues every MMA, and its issue rate sets the tile period, so the shared-
            // memory descriptors are built once: a descriptor's address field is (address >> 4)
            // in 14 bits, and every operand lies below 228 KB on a 16-byte boundary, so the
            // descriptor of base + off is the base descriptor + (off >> 4), a constant per MMA
            // (building each from its address measured 4-5 % slower on the 32K x 2048 chunks).
            const uint64_t kdesc0 = tc::smem_desc_sw128(sbase + SM_KHAT, 16, 1024);
            const uint64_t vdesc0 = tc::smem_desc_sw128(sbase + SM_VHAT, BN * 128, 1024);
            auto issue_pv = [&](int jj, bool first) -> bool {
                const int bb = jj & 1, u = jj >> 1;
                if (!tc::mbar_wait(B(B_P_FULL + bb), u & 1, kWaitLimit)) return false;
                if (!tc::mbar_wait(B(B_V_FULL + bb), u & 1, kWaitLimit)) return false;
                tc::fence_after_sync();
                const uint64_t vdesc = vdesc0 + (uint64_t)((bb * HAT_BYTES) >> 4);
                const uint32_t pcol = tmem + TM_S0 + bb * BN;
#pragma unroll
                for (int ks = 0; ks < BN / 16; ++ks)
                    tc::mma_ts(tmem + TM_O, pcol + ks * 8, vdesc + (uint64_t)((ks * 2048) >> 4),
                               IDESC_PV, (!first || ks > 0) ? 1u : 0u);
                tc::mma_commit(B(B_PV_DONE + bb));
                pv_issued = jj + 1;
                return true;
            };
            for (int si = 0; ok && si < n_seg; ++si) {
                if (!tc::mbar_wait(B(B_Q_READY), si & 1, kWaitLimit)) { ok = false; break; }
                tc::fence_after_sync();
                const int jfirst = j;
                for (int t = seg[si].t0; t < seg[si].t1; ++t, ++j) {
                    const int b = j & 1, use = j >> 1;
                    // S(j) overwrites the columns from which PV(j-2) reads P(j-2); both MMAs come
                    // from this thread and tcgen05 MMAs run in issue order, so QK(j) is issued
                    // without waiting for PV(j-2) to complete (waiting cost 5-7 % on the 32K x 2048
                    // chunks: the tensor pipe drained once per tile)
                    if (!tc::mbar_wait(B(B_K_FULL + b), use & 1, kWaitLimit)) { ok = false; break; }
                    tc::fence_after_sync();
                    const uint64_t kdesc = kdesc0 + (uint64_t)((b * HAT_BYTES) >> 4);
#pragma unroll
                    for (int ks = 0; ks < HD / 16; ++ks)
                        tc::mma_ts(tmem + TM_S0 + b * BN, tmem + TM_Q + ks * 8,
                                   kdesc + (uint64_t)((((ks >> 2) * (BN * 128)) + (ks & 3) * 32) >> 4),
                                   IDESC_QK, ks > 0 ? 1u : 0u);
                    tc::mma_commit(B(B_S_FULL + b));
                    if (j > jfirst && !issue_pv(j - 1, j - 1 == jfirst)) { ok = false; break; }
                }
                if (ok && j > jfirst && !issue_pv(j - 1, j - 1 == jfirst)) ok = false;
            }
            if (!ok) flag_timeout();
            // tensor memory is released only after the last committed MMA has completed
            if (pv_issued > 0 &&
                !tc::mbar_wait(B(B_PV_DONE + ((pv_issued - 1) & 1)), ((pv_issued - 1) >> 1) & 1, kWaitLimit))
                flag_timeout();
        }
        __syncwarp();
    } else if (warp >= kSoftWarp0 && warp < kDeqWarp0) {
        // ---------------------------------------------------------------- softmax (one row per thread)
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const float cs = p.scale_log2;
        const int rows_out = p.n_q * p.n_q_heads;
        bool ok = true;
        int j = 0;
        for (int si = 0; ok && si < n_seg; ++si) {
            const Item g = item_geometry(seg[si].item, p.n_mtiles, p.rows, p.group, p.kv_len, p.q_pos0, BN);
            const bool valid = r < g.rows_here;
            const int rr = g.r0 + r;
            const int iq = valid ? rr / p.group : 0;
            const int qh = g.kvh * p.group + (valid ? rr - iq * p.group : 0);
            const int vis_end = valid ? min(p.kv_len, p.q_pos0 + iq + 1) : 0;
            // Q row -> TMEM (fp16 pairs, A operand of S = Q K^T); the previous segment's
            // epilogue has already waited for every MMA that read the old Q.
            {
                const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)iq * p.n_q_heads + qh) * HD);
#pragma unroll 1
                for (int c = 0; c < HD / 64; ++c) {   // 64 fp16 dims = 32 TMEM columns per store
                    uint32_t w[32];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (valid) v = __ldg(src + c * 8 + k);
                        w[4 * k] = v.x;
                        w[4 * k + 1] = v.y;
                        w[4 * k + 2] = v.z;
                        w[4 * k + 3] = v.w;
                    }
                    tc::tmem_st32(tmem + lane_base + TM_Q + 32 * c, w);
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(B(B_Q_READY));
            }
            float m_ref = -INFINITY, l = 0.0f;
            for (int t = seg[si].t0; t < seg[si].t1; ++t, ++j) {
                const int b = j & 1, use = j >> 1;
                const bool ready = tc::mbar_wait(B(B_S_FULL + b), use & 1, kWaitLimit);
                if (!__all_sync(0xffffffffu, ready)) { ok = false; break; }
                tc::fence_after_sync();
                if constexpr (BN == 64) {  // one 64-key tile per S buffer, held in registers throughout
                    uint32_t s0[32], s1[32];
                    const uint32_t scol = tmem + lane_base + TM_S0 + b * BN;
                    tc::tmem_ld32(scol, s0);
                    tc::tmem_ld32(scol + 32, s1);
                    tc::tmem_wait_ld();
                    float x[64];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        x[c] = __uint_as_float(s0[c]);
                        x[32 + c] = __uint_as_float(s1[c]);
                    }
                    const int key0 = t * BN;
                    if (key0 + BN > g.key_lo) {  // the causal diagonal (or rows past kv_len) crosses this tile
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            if (key0 + c >= vis_end) x[c] = -INFINITY;
                    }
                    float mq[4] = {x[0], x[1], x[2], x[3]};  // four chains
#pragma unroll
                    for (int c = 4; c < 64; ++c) mq[c & 3] = fmaxf(mq[c & 3], x[c]);
                    const float mt = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
                    const float m_new = fmaxf(m_ref, mt * cs);
                    const bool need = m_new > m_ref + kRescaleThreshold || (m_ref == -INFINITY && m_new != -INFINITY);
                    if (__any_sync(0xffffffffu, need)) {
                        float alpha = 1.0f;
                        if (need) {
                            alpha = (m_ref == -INFINITY) ? 0.0f : ex2_approx(m_ref - m_new);
                            m_ref = m_new;
                            l *= alpha;
                        }
                        if (t > seg[si].t0) {  // rescale the O row once every earlier PV has landed
                            const int pj = j - 1;
                            const bool done = tc::mbar_wait(B(B_PV_DONE + (pj & 1)), (pj >> 1) & 1, kWaitLimit);
                            if (!__all_sync(0xffffffffu, done)) { ok = false; break; }
                            tc::fence_after_sync();
#pragma unroll 1
                            for (int c = 0; c < HD / 32; ++c) {
                                uint32_t o[32];
                                tc::tmem_ld32(tmem + lane_base + TM_O + 32 * c, o);
                                tc::tmem_wait_ld();
#pragma unroll
                                for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                                tc::tmem_st32(tmem + lane_base + TM_O + 32 * c, o);
                            }
                        }
                    }
                    uint32_t pk[32];
                    float sq[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // four chains
                    const bool live = m_ref != -INFINITY;
                    const float neg = live ? -m_ref : 0.0f;
                    // Packed fp32x2 FMA and sums (fewer issue slots) for the K8V4 and fp16 pools;
                    // the Q8_0 pool at this tile size measured 1 % slower with them (0.828 vs 0.818
                    // ms on the 32K x 2048 chunk; K8V4 0.850 vs 0.881 ms) and keeps the scalar form.
                    if constexpr (POOL != kPoolQ8) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {  // a key pair per packed FMA, two packed sum chains
                            const float2 e = fma2_sc(x[2 * c], x[2 * c + 1], cs, neg);
                            const float a = live ? ex2_approx(e.x) : 0.0f;
                            const float bq = live ? ex2_approx(e.y) : 0.0f;
                            add2(sq[2 * (c & 1)], sq[2 * (c & 1) + 1], a, bq);
                            const __half2 h = __floats2half2_rn(a, bq);
                            pk[c] = *reinterpret_cast<const uint32_t*>(&h);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const float a = live ? ex2_approx(fmaf(x[2 * c], cs, neg)) : 0.0f;
                            const float bq = live ? ex2_approx(fmaf(x[2 * c + 1], cs, neg)) : 0.0f;
                            sq[c & 3] += a + bq;
                            const __half2 h = __floats2half2_rn(a, bq);
                            pk[c] = *reinterpret_cast<const uint32_t*>(&h);
                        }
                    }
                    l += (sq[0] + sq[1]) + (sq[2] + sq[3]);
                    tc::tmem_st32(scol, pk);  // P overwrites the first 32 columns of this S buffer
                } else {  // 128-key tiles: the S row in two 64-column halves, read twice
                    const uint32_t scol = tmem + lane_base + TM_S0 + b * BN;
                    const int key0 = t * BN;
                    const bool diag = key0 + BN > g.key_lo;  // the causal diagonal (or rows past kv_len) crosses this tile
                    // S row of this thread, 64 columns at a time (the tile's BN/64 halves), masked
                    auto load_half = [&](int h, float (&x)[64]) {
                        uint32_t s0[32], s1[32];
                        tc::tmem_ld32(scol + 64 * h, s0);
                        tc::tmem_ld32(scol + 64 * h + 32, s1);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            x[c] = __uint_as_float(s0[c]);
                            x[32 + c] = __uint_as_float(s1[c]);
                        }
                        if (diag) {
#pragma unroll
                            for (int c = 0; c < 64; ++c)
                                if (key0 + 64 * h + c >= vis_end) x[c] = -INFINITY;
                        }
                    };
                    float x[64];
                    float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four chains
#pragma unroll 1
                    for (int h = 0; h < BN / 64; ++h) {
                        load_half(h, x);
#pragma unroll
                        for (int c = 0; c < 64; ++c) mq[c & 3] = fmaxf(mq[c & 3], x[c]);
                    }
                    const float mt = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
                    const float m_new = fmaxf(m_ref, mt * cs);
                    const bool need = m_new > m_ref + kRescaleThreshold || (m_ref == -INFINITY && m_new != -INFINITY);
                    if (__any_sync(0xffffffffu, need)) {
                        float alpha = 1.0f;
                        if (need) {
                            alpha = (m_ref == -INFINITY) ? 0.0f : ex2_approx(m_ref - m_new);
                            m_ref = m_new;
                            l *= alpha;
                        }
                        if (t > seg[si].t0) {  // rescale the O row once every earlier PV has landed
                            const int pj = j - 1;
                            const bool done = tc::mbar_wait(B(B_PV_DONE + (pj & 1)), (pj >> 1) & 1, kWaitLimit);
                            if (!__all_sync(0xffffffffu, done)) { ok = false; break; }
                            tc::fence_after_sync();
#pragma unroll 1
                            for (int c = 0; c < HD / 32; ++c) {
                                uint32_t o[32];
                                tc::tmem_ld32(tmem + lane_base + TM_O + 32 * c, o);
                                tc::tmem_wait_ld();
#pragma unroll
                                for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                                tc::tmem_st32(tmem + lane_base + TM_O + 32 * c, o);
                            }
                        }
                    }
                    const bool live = m_ref != -INFINITY;
                    const float neg = live ? -m_ref : 0.0f;
                    // P of keys 64h .. 64h+63 goes to columns 32h .. 32h+31 of this S buffer: those
                    // hold S of keys 32h .. 32h+63, already read (half 0 by now, half 1 below)
#pragma unroll 1
                    for (int h = 0; h < BN / 64; ++h) {
                        if (BN > 64) load_half(h, x);  // at BN = 64 the half is still in registers
                        uint32_t pk[32];
                        float sq[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // four chains
                        // packed fp32x2 FMA and sums: this issue-bound path measured 8.5 % faster
                        // with them (Q8_0 hd128 1.157 vs 1.263 ms on the 32K x 2048 chunk)
#pragma unroll
                        for (int c = 0; c < 32; ++c) {  // a key pair per packed FMA, two packed sum chains
                            const float2 e = fma2_sc(x[2 * c], x[2 * c + 1], cs, neg);
                            const float a = live ? ex2_approx(e.x) : 0.0f;
                            const float bq = live ? ex2_approx(e.y) : 0.0f;
                            add2(sq[2 * (c & 1)], sq[2 * (c & 1) + 1], a, bq);
                            const __half2 hh = __floats2half2_rn(a, bq);
                            pk[c] = *reinterpret_cast<const uint32_t*>(&hh);
                        }
                        l += (sq[0] + sq[1]) + (sq[2] + sq[3]);
                        tc::tmem_st32(scol + 32 * h, pk);
                    }
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(B(B_P_FULL + b));
            }
            if (!ok) break;
            // epilogue: the unnormalised partial (o, m, l) of this segment
            const int pj = j - 1;
            const bool done = tc::mbar_wait(B(B_PV_DONE + (pj & 1)), (pj >> 1) & 1, kWaitLimit);
            if (!__all_sync(0xffffffffu, done)) { ok = false; break; }
            tc::fence_after_sync();
            const int64_t orow = (int64_t)iq * p.n_q_heads + qh;
            float4* dst = reinterpret_cast<float4*>(p.part_o + ((int64_t)seg[si].part * rows_out + orow) * HD);
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t o[32];
                tc::tmem_ld32(tmem + lane_base + TM_O + 32 * c, o);
                tc::tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[c * 8 + k] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                                     __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
                }
            }
            if (valid) {
                p.part_ml[(int64_t)seg[si].part * rows_out + orow] =
                    make_float2(m_ref == -INFINITY ? -INFINITY : m_ref * kLn2, l);
                if (seg[si].last)  // the slots of parts this item does not have hold an empty partial
                    for (int q2 = seg[si].part + 1; q2 < p.n_parts; ++q2)
                        p.part_ml[(int64_t)q2 * rows_out + orow] = make_float2(-INFINITY, 0.0f);
            }
        }
        if (!ok) flag_timeout();
    } else if (!F16) {
        // ---------------------------------------------------------------- dequantisers
        const int d = threadIdx.x - kDeqWarp0 * 32;
        int j = 0;
        bool ok = true;
        for (int si = 0; ok && si < n_seg; ++si) {
            const Item g = item_geometry(seg[si].item, p.n_mtiles, p.rows, p.group, p.kv_len, p.q_pos0, BN);
            for (int t = seg[si].t0; t < seg[si].t1; ++t, ++j) {
                const int s = j & 1, use = j >> 1;
                // waits are decided per warp, so that a warp arrives (lane 0) only as a whole
                if (!__all_sync(0xffffffffu, tc::mbar_wait(B(B_ST_FULL + s), use & 1, kWaitLimit))) { ok = false; break; }
                const int nk = min(BN, g.key_hi - t * BN);
                const uint8_t* st = smem + SM_STAGE + s * STAGE_BYTES;
                // at hd128 the scales sit at the tile's 0- or 8-byte offset from a 16-byte boundary
                const int soff = HD == 256 ? 0 : (int)(((int64_t)g.kvh * p.capacity + t * BN) & 1) * 8;
                const uint16_t* k_sc = reinterpret_cast<const uint16_t*>(st + ST_KS + soff);
                const uint16_t* v_sc = reinterpret_cast<const uint16_t*>(st + ST_VS + soff);
                if (j >= 2 && !__all_sync(0xffffffffu, tc::mbar_wait(B(B_S_FULL + s), (use - 1) & 1, kWaitLimit))) {
                    ok = false;
                    break;
                }
                dequant_tile<HD>(st + ST_KC, k_sc, smem + SM_KHAT + s * HAT_BYTES, nk, d);
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(B(B_K_FULL + s));
                if (j >= 2 && !__all_sync(0xffffffffu, tc::mbar_wait(B(B_PV_DONE + s), (use - 1) & 1, kWaitLimit))) {
                    ok = false;
                    break;
                }
                if constexpr (V4)
                    dequant_tile_v4<HD>(st + ST_VC, v_sc, smem + SM_VHAT + s * HAT_BYTES, nk, d);
                else
                    dequant_tile<HD>(st + ST_VC, v_sc, smem + SM_VHAT + s * HAT_BYTES, nk, d);
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(B(B_V_FULL + s));
                    tc::mbar_arrive(B(B_ST_EMPTY + s));
                }
            }
        }
        if (!ok) flag_timeout();
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, TM_NCOLS);
}

struct PromptPlan {
    int n_mtiles, n_items, n_parts, grid;
    long long units;
    // two-pass route: the fp16 copy of keys < copy_keys of both planes at byte copy_off of the
    // workspace (copy_keys = 0: the one-pass kernel dequantises in shared memory)
    int copy_keys;
    size_t part_bytes, copy_off, ws_bytes;  // partials alone; the copy's offset; the whole workspace
};

// Row tiles per KV head from which a Q8_0 or K8V4 chunk takes the two-pass route.  The one-pass
// kernel dequantises every K/V tile once per row tile that sees it; the two-pass route pays one
// pass over the planes (6.1 bytes of traffic per value) and then runs without staging.  Measured
// on GB300 over a 32K context: at hd256 (12q/1kv) the routes tie at 17 row tiles and the
// two-pass route is 3 % faster at 24, 7 % at 48; at hd128 (32q/8kv) it is 2 % slower at 16 row
// tiles and 15 % faster at 64.
constexpr int kTwoPassMinMtiles = 24;

int prompt_plan(int n_q, int n_q_heads, int head_dim, int kv_len, int q_pos0, int n_kv_heads, PromptPlan* pl) {
    if (n_q < 1 || n_q_heads < 1 || n_kv_heads < 1 || kv_len < 1 || q_pos0 < 0) return KVQ8_ERR_INVALID_ARG;
    if ((head_dim != 128 && head_dim != 256) || n_q_heads % n_kv_heads) return KVQ8_ERR_UNSUPPORTED;
    const int group = n_q_heads / n_kv_heads;
    const long long rows = (long long)n_q * group;
    if (rows > 0x7fffffffLL || (long long)n_q * n_q_heads > 0x7fffffffLL) return KVQ8_ERR_UNSUPPORTED;
    pl->n_mtiles = (int)((rows + BM - 1) / BM);
    const long long items = (long long)pl->n_mtiles * n_kv_heads;
    if (items > (1 << 24)) return KVQ8_ERR_UNSUPPORTED;
    pl->n_items = (int)items;
    long long U = 0;
    for (int it = 0; it < pl->n_items; ++it)
        U += item_geometry(it, pl->n_mtiles, (int)rows, group, kv_len, q_pos0, bn_for(head_dim)).n_tiles;
    pl->units = U;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms <= 0)
        sms = 152;
    pl->grid = (int)(U < sms ? U : sms);
    // parts per item: CTAs its units span; segments per CTA: items its units touch
    int parts = 1;
    long long s = 0;
    int max_seg = 0, cur_cta = -1, cur_seg = 0;
    for (int it = 0; it < pl->n_items; ++it) {
        const int nt = item_geometry(it, pl->n_mtiles, (int)rows, group, kv_len, q_pos0, bn_for(head_dim)).n_tiles;
        const long long c0 = cta_of_unit(s, U, pl->grid), c1 = cta_of_unit(s + nt - 1, U, pl->grid);
        parts = (int)(c1 - c0 + 1) > parts ? (int)(c1 - c0 + 1) : parts;
        for (long long c = c0; c <= c1; ++c) {
            if (c != cur_cta) { cur_cta = (int)c; cur_seg = 0; }
            ++cur_seg;
            max_seg = cur_seg > max_seg ? cur_seg : max_seg;
        }
        s += nt;
    }
    if (max_seg > kMaxSegments) return KVQ8_ERR_UNSUPPORTED;
    pl->n_parts = parts;
    const size_t rows_out = (size_t)n_q * n_q_heads;
    const size_t o_bytes = (size_t)parts * rows_out * head_dim * sizeof(float);
    const size_t part_bytes = ((o_bytes + 255) / 256) * 256 + (size_t)parts * rows_out * 2 * sizeof(float);
    pl->part_bytes = part_bytes;
    // the highest key any row sees is q_pos0 + n_q - 1 (or the context's end)
    const long long last = (long long)q_pos0 + n_q;
    pl->copy_keys = pl->n_mtiles >= kTwoPassMinMtiles ? (int)(last < kv_len ? last : kv_len) : 0;
    pl->copy_off = ((part_bytes + 255) / 256) * 256;
    pl->ws_bytes = pl->copy_keys ? pl->copy_off + 2 * (size_t)n_kv_heads * pl->copy_keys * head_dim * sizeof(uint16_t)
                                 : part_bytes;
    return KVQ8_OK;
}

int launch_dequant_planes(const DequantParams& dp, bool v4, cudaStream_t s) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms <= 0)
        sms = 152;
    const int planes = 2 * dp.n_kv_heads;
    const long long blocks = (long long)dp.n_keys * (dp.hd / 8);   // 8-value groups per plane
    if (planes > 65535 || blocks > 0x7fffffffLL) return KVQ8_ERR_UNSUPPORTED;
    // about eight 256-thread blocks per SM over all planes and heads, each looping over its share
    // of the 8-value groups
    long long gx = (blocks + 255) / 256, cap = (8LL * sms + planes - 1) / planes;
    gx = gx < cap ? gx : cap;
    const dim3 grid((unsigned)(gx > 0 ? gx : 1), (unsigned)planes);
    if (v4)
        dequant_planes_kernel<true><<<grid, 256, 0, s>>>(dp);
    else
        dequant_planes_kernel<false><<<grid, 256, 0, s>>>(dp);
    return launch_status();
}

template <int HD, int POOL>
int launch_prompt(const PromptParams& pp, int grid, cudaStream_t s) {
    static SmemOptIn opt;
    if (opt.ensure(prompt_attn_kernel<HD, POOL>, PL<HD>::SMEM_BYTES) != KVQ8_OK) return KVQ8_ERR_CUDA;
    prompt_attn_kernel<HD, POOL><<<grid, kThreads, PL<HD>::SMEM_BYTES, s>>>(pp);
    return launch_status();
}

// Tensor map of one fp16 plane [n_kv_heads][capacity][hd]: dims (hd, kv_len, n_kv_heads), so
// keys at or past kv_len read as zeros; box 64 dims x 64 keys x 1 head, 128-byte swizzle.
bool encode_f16_plane(CUtensorMap* map, const uint16_t* plane, int hd, int kv_len, int n_kv_heads, int capacity) {
    const int BN = bn_for(hd);
    const EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)kv_len, (cuuint64_t)n_kv_heads};
    const cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)capacity * hd * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)BN, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t*>(plane), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace kvq8

extern "C" size_t attn_prompt_q8_workspace_bytes(int n_q, int n_q_heads, int head_dim, int kv_len, int q_pos0,
                                                 int n_kv_heads) {
    kvq8::PromptPlan pl;
    if (kvq8::prompt_plan(n_q, n_q_heads, head_dim, kv_len, q_pos0, n_kv_heads, &pl) != KVQ8_OK) return 0;
    return pl.ws_bytes;
}

extern "C" size_t attn_prompt_f16_workspace_bytes(int n_q, int n_q_heads, int head_dim, int kv_len, int q_pos0,
                                                  int n_kv_heads) {
    kvq8::PromptPlan pl;
    if (kvq8::prompt_plan(n_q, n_q_heads, head_dim, kv_len, q_pos0, n_kv_heads, &pl) != KVQ8_OK) return 0;
    return pl.part_bytes;
}

namespace kvq8 {
namespace {

// kv: the pool's planes seen as a kvq8_cache (for an fp16 pool k_codes / v_codes carry the fp16
// planes and there are no scales).
int prompt_impl(const uint16_t* q, int n_q, int n_q_heads, const kvq8_cache* kv, int kv_len, int q_pos0,
                float softmax_scale, float* out, void* workspace, size_t workspace_bytes, kvq8_stream_t stream,
                int pool) {
    if (!kv || !q || !out) return KVQ8_ERR_INVALID_ARG;
    if (!kv->k_codes || !kv->v_codes) return KVQ8_ERR_INVALID_ARG;
    if (pool != kPoolF16 && (!kv->k_scales || !kv->v_scales)) return KVQ8_ERR_INVALID_ARG;
    if (kv->n_kv_heads < 1 || kv_len > kv->capacity) return KVQ8_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.0f) || softmax_scale == INFINITY) return KVQ8_ERR_INVALID_ARG;
    PromptPlan pl;
    const int rc = prompt_plan(n_q, n_q_heads, kv->head_dim, kv_len, q_pos0, kv->n_kv_heads, &pl);
    if (rc != KVQ8_OK) return rc;
    if (!aligned16(q) || !aligned16(out) || !aligned16(kv->k_codes) || !aligned16(kv->v_codes) ||
        (pool != kPoolF16 && (!aligned16(kv->k_scales) || !aligned16(kv->v_scales))))
        return KVQ8_ERR_MISALIGNED;
    // an fp16 pool needs the partials only; the fp16 copy is for the dequantising pools
    if (!workspace || workspace_bytes < (pool == kPoolF16 ? pl.part_bytes : pl.ws_bytes)) return KVQ8_ERR_WORKSPACE;
    if (!aligned16(workspace)) return KVQ8_ERR_MISALIGNED;
    const int HD = kv->head_dim;
    const size_t rows_out = (size_t)n_q * n_q_heads;
    const size_t o_bytes = (size_t)pl.n_parts * rows_out * HD * sizeof(float);
    PromptParams pp;
    pp.q = q;
    pp.kc = kv->k_codes;
    pp.ks = kv->k_scales;
    pp.vc = kv->v_codes;
    pp.vs = kv->v_scales;
    pp.part_o = static_cast<float*>(workspace);
    pp.part_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) + ((o_bytes + 255) / 256) * 256);
    pp.n_q = n_q;
    pp.n_q_heads = n_q_heads;
    pp.group = n_q_heads / kv->n_kv_heads;
    pp.capacity = kv->capacity;
    pp.kv_len = kv_len;
    pp.q_pos0 = q_pos0;
    pp.rows = n_q * pp.group;
    pp.n_mtiles = pl.n_mtiles;
    pp.n_items = pl.n_items;
    pp.n_parts = pl.n_parts;
    pp.units = pl.units;
    pp.scale_log2 = softmax_scale * kLog2e;
    cudaStream_t s = (cudaStream_t)stream;
    // two-pass route (long chunks over Q8_0 / K8V4 pools): dequantise the planes once into the
    // workspace, then run the tensor-copy kernel of fp16 pools over that copy
    const bool two_pass = pool != kPoolF16 && pl.copy_keys > 0;
    if (two_pass) {
        uint16_t* k16 = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + pl.copy_off);
        uint16_t* v16 = k16 + (size_t)kv->n_kv_heads * pl.copy_keys * HD;
        // the maps need only the addresses: encode them before launching anything
        if (!encode_f16_plane(&pp.tmap_k, k16, HD, pl.copy_keys, kv->n_kv_heads, pl.copy_keys) ||
            !encode_f16_plane(&pp.tmap_v, v16, HD, pl.copy_keys, kv->n_kv_heads, pl.copy_keys))
            return KVQ8_ERR_CUDA;
        const DequantParams dp = {kv->k_codes, kv->k_scales, kv->v_codes, kv->v_scales, k16, v16,
                                  HD, pl.copy_keys, kv->capacity, kv->n_kv_heads};
        const int r0 = launch_dequant_planes(dp, pool == kPoolK8V4, s);
        if (r0 != KVQ8_OK) return r0;
    } else if (pool == kPoolF16) {
        const uint16_t* kp = reinterpret_cast<const uint16_t*>(kv->k_codes);
        const uint16_t* vp = reinterpret_cast<const uint16_t*>(kv->v_codes);
        if (!encode_f16_plane(&pp.tmap_k, kp, HD, kv_len, kv->n_kv_heads, kv->capacity) ||
            !encode_f16_plane(&pp.tmap_v, vp, HD, kv_len, kv->n_kv_heads, kv->capacity))
            return KVQ8_ERR_CUDA;
    }
    int r1;
    if (pool == kPoolF16 || two_pass)
        r1 = HD == 128 ? launch_prompt<128, kPoolF16>(pp, pl.grid, s) : launch_prompt<256, kPoolF16>(pp, pl.grid, s);
    else if (pool == kPoolK8V4)
        r1 = HD == 128 ? launch_prompt<128, kPoolK8V4>(pp, pl.grid, s) : launch_prompt<256, kPoolK8V4>(pp, pl.grid, s);
    else
        r1 = HD == 128 ? launch_prompt<128, kPoolQ8>(pp, pl.grid, s) : launch_prompt<256, kPoolQ8>(pp, pl.grid, s);
    if (r1 != KVQ8_OK) return r1;
    return launch_combine(pp.part_o, reinterpret_cast<const float*>(pp.part_ml), pl.n_parts, (int)rows_out, HD, out, s);
}

}  // namespace
}  // namespace kvq8

extern "C" int attn_prompt_q8(const uint16_t* q, int n_q, int n_q_heads, const kvq8_cache* kv, int kv_len, int q_pos0,
                              float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                              kvq8_stream_t stream) {
    return kvq8::prompt_impl(q, n_q, n_q_heads, kv, kv_len, q_pos0, softmax_scale, out, workspace, workspace_bytes,
                             stream, kvq8::kPoolQ8);
}

extern "C" int attn_prompt_k8v4(const uint16_t* q, int n_q, int n_q_heads, const kvk8v4_cache* kv, int kv_len,
                                int q_pos0, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                                kvq8_stream_t stream) {
    if (!kv) return KVQ8_ERR_INVALID_ARG;
    // the Q8_0 view of the pool: the V plane pointer carries the nibbles
    const kvq8_cache view = {kv->k_codes, kv->k_scales, reinterpret_cast<const int8_t*>(kv->v_codes), kv->v_scales,
                             kv->n_kv_heads, kv->head_dim, kv->capacity};
    return kvq8::prompt_impl(q, n_q, n_q_heads, &view, kv_len, q_pos0, softmax_scale, out, workspace, workspace_bytes,
                             stream, kvq8::kPoolK8V4);
}

extern "C" int attn_prompt_f16(const uint16_t* q, int n_q, int n_q_heads, const kvf16_cache* kv, int kv_len, int q_pos0,
                               float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                               kvq8_stream_t stream) {
    if (!kv) return KVQ8_ERR_INVALID_ARG;
    // the fp16 planes ride in the code pointers of a scale-less view
    const kvq8_cache view = {reinterpret_cast<const int8_t*>(kv->k), nullptr, reinterpret_cast<const int8_t*>(kv->v),
                             nullptr, kv->n_kv_heads, kv->head_dim, kv->capacity};
    return kvq8::prompt_impl(q, n_q, n_q_heads, &view, kv_len, q_pos0, softmax_scale, out, workspace, workspace_bytes,
                             stream, kvq8::kPoolF16);
}

namespace kvq8 {
// The flag's device address per device, looked up with that device current (concurrent first
// lookups store the same value).
unsigned int* device_error_flag() {
    constexpr int kMaxDev = 64;
    static unsigned int* cached[kMaxDev] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    if (!cached[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_kvq8_device_error) != cudaSuccess) return nullptr;
        cached[dev] = static_cast<unsigned int*>(ptr);
    }
    return cached[dev];
}
}  // namespace kvq8

extern "C" int kvq8_device_error(int reset) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_kvq8_device_error, sizeof v) != cudaSuccess) return -1;
    if (reset && v) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_kvq8_device_error, &z, sizeof z) != cudaSuccess) return -1;
    }
    return (int)v;
}
