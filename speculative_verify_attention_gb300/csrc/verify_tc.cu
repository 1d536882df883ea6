// verify_tc.cu -- the split-context verify scan over a Q8_0 cache with QK on the tcgen05 tensor
// cores (the causal windows of attn_verify_q8, attn_verify_q8_partials and
// attn_verify_append_q8, the tree windows of attn_verify_tree_q8, and the causal windows of
// attn_verify_k8v4 at hd256, whose V plane holds 4-bit codes expanded in the PV warps).
//
// Source: "perf(gfx1100): share Q8 KV scans across verifier rows", Summary: one worker owns all
// query rows of a verify window and shares each K/V scan across them; context slices write
// partials that a reducer merges.  "gfx12 WMMA kernel for the int8-KV QSA prompt attention",
// How: fp16 hi + lo split of q and p with fp32 accumulation, online softmax, the V scale
// folded into p.
//
// GB300 design.  One thread block (one per SM) per (row chunk of <= 24 (row, q-head) pairs,
// context slice, KV head); 19 warps with fixed roles, coupled by mbarriers:
//   warp 16      K producer: 128-key tiles of int8 codes by tensor copies (128-byte swizzle, keys
//                past kv_len read as zeros) into a 2-stage ring, the fp16 block scales by 16/8-byte
//                async copies that arrive on the same barrier.  Tile 0 goes out first and alone;
//   warp 17      V producer: the same for V, starting once K tile 0 has landed; a V slot is
//                refilled when the PV warps release that tile's P buffer;
//   warp 18      tensor-memory owner and MMA issuer (one thread);
//   warps 0-7    "fold" warps, one key per thread (TMEM lane quadrant warp % 4, half warp / 4):
//                convert the K codes of tile t to fp16 (exact) straight into tensor memory,
//                then take the QK accumulators of tile t-1 out of tensor memory and fold the
//                K scales in, mask, keep the lazy row maxima and write p as fp16 hi + lo
//                (published once V of that tile has landed, so the PV warps wait once a tile);
//   warps 8-15   PV warps: O^T += V^T (p dV) on mma.sync, each warp one 32-dim output block
//                (hd256) or half of one (hd128), as in the all-mma.sync kernel.
// The kernel is launched as a programmatic dependent: its prologue and K tile 0 overlap the
// kernel before it in the stream; q, the window's cache writes and the partials wait for it.
// QK on tcgen05, transposed (keys are M = 128): A = the tile's K codes as fp16 in tensor memory
// (lane = key, column c = dims 2c, 2c + 1), B = the chunk's q rows as fp16 hi and lo stacked
// along N (N = 2 RP, K-major, 128-byte swizzle), one accumulator D_b [128 keys x N] per 32-dim
// scale block b, so the K scale -- which varies along the contraction -- is applied exactly by
// the fold warps: s = sum_b dK_b (D_b[hi] + D_b[lo]).  Products are exact (int8 codes x fp16
// halves) and accumulate in fp32, as on the mma.sync path.  The QK MMAs of tile t run while the
// fold warps finish tile t-1 and the PV warps run tile t-2.
// Every mbarrier wait is bounded; on a timeout the kernel records the library's error flag and
// runs to its end without further waits (named barriers of the fold warps stay matched), frees
// its tensor memory and returns.
#include "common.cuh"
#include "q8_0.cuh"
#include "tc.cuh"
#include "verify_tc.cuh"

namespace kvq8 {

namespace {

// Warp roles (19 warps; at most 5 per SM sub-partition, so 96 registers per thread):
constexpr int kFoldWarp0 = 0;    // warps 0-7: K conversion, fold and softmax, one key per thread
                                 // (TMEM lane quadrant warp % 4, dims and row half warp / 4)
constexpr int kPvWarp0 = 8;      // warps 8-15: PV warps
constexpr int kKProdWarp = 16;   // K producer
constexpr int kVProdWarp = 17;   // V producer
constexpr int kMmaWarp = 18;     // tensor-memory owner and MMA issuer
constexpr int kTcWarps = 19;
constexpr int kVKeys = 128;      // keys per V ring slot
constexpr int kVSlots = 2;       // V ring slots
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kWorkThreads = kTcThreads - 64;  // every warp but the two producers
constexpr uint32_t kTcWait = 1u << 24;   // polls per mbarrier wait
constexpr uint32_t kProdSleepNs = 200, kMmaSleepNs = 32;  // sleeps between polls
constexpr float kLazyTc = 8.0f;          // log2 units: a row's reference maximum moves only past this
constexpr float kPShiftTc = 4.0f;        // p is stored as p 2^4 (<= 2^12)

template <int HD, int RP, bool V4 = false>
struct TcLayout {
    static constexpr int NB = HD / 32;          // scale blocks per key
    static constexpr int RPH = RP / 2;          // rows per fold-warp half
    static constexpr int N = 2 * RP;            // B rows: q hi and lo of RP rows
    static constexpr int PS = RP + 4;           // P-tile entries per key pair (padding spreads banks)
    static constexpr int NBOX = HD / 128;       // 128-byte tensor-copy boxes per key row
    static constexpr int BOX = kKT * 128;
    static constexpr int CODES = NBOX * BOX;
    static constexpr int SCALES = kKT * NB * 2;
    static constexpr int STAGE = (CODES + SCALES + 1023) / 1024 * 1024;
    static constexpr int QATOM = N * 128;       // one 64-dim atom of the q tile
    static constexpr int Q = 0;
    static constexpr int KST = Q + (HD / 64) * QATOM;   // 2 K stages
    // V: a ring of kVSlots units of kVKeys keys (a whole tile or a fraction of one)
    static constexpr int HKEYS = kVKeys;
    static constexpr int HBOX = HKEYS * 128;
    // V codes per key: HD bytes, or HD/2 bytes of 4-bit codes (K8V4 pools, hd256 only: one box)
    static constexpr int NBOXV = V4 ? 1 : NBOX;
    static constexpr int HCODES = NBOXV * HBOX;
    static constexpr int HSTAGE = (HCODES + HKEYS * NB * 2 + 1023) / 1024 * 1024;
    static constexpr int VST = KST + 2 * STAGE;
    static constexpr int P = VST + kVSlots * HSTAGE;
    static constexpr int PBUF = (kKT / 2) * PS * 8;
    static constexpr int PH = P + 2 * PBUF;     // per P buffer: rescale flag, 3 pad words, a[RP]
    static constexpr int PHB = 16 + RP * 4;
    static constexpr int DV = PH + 2 * PHB;     // per PV warp: its block's V scales x 2^E, fp16
    static constexpr int RED = DV + 8 * kKT * 2;
    static constexpr int LRED = RED + 4 * RP * 4;
    static constexpr int VIS = LRED + 4 * RP * 4;
    static constexpr int WM = VIS + RP * 4;    // tree windows: each row's window mask
    static constexpr int BARS = (WM + RP * 4 + 7) / 8 * 8;
    // (VE: unused; a V slot is released with its tile's P buffer, PE)
    enum { KF = 0, KE = 2, VF = 4, VE = VF + kVSlots, PF = VE + kVSlots, PE = PF + 2, GO = PE + 2, QKD = GO + 1,
           VGO = QKD + 1, NBARS = VGO + 1 };
    static constexpr int KH = GO;               // K^ of the tile written (the fold warps)
    static constexpr int SLOT = BARS + NBARS * 8;
    static constexpr int BYTES = SLOT + 16;
    static constexpr uint32_t TM_KH = 0, TM_D = HD / 2;
    static constexpr uint32_t TM_USED = TM_D + NB * N;
    static constexpr uint32_t TM_COLS = TM_USED <= 128 ? 128 : TM_USED <= 256 ? 256 : 512;
    static constexpr uint32_t IDESC = tc::idesc_f16_f32(128, N, false);
    static_assert(RP % 8 == 0 && RP <= 24, "rows per chunk");
    static_assert(!V4 || HD == 256, "4-bit V tiles of one 128-byte box per key");
    static_assert(TM_USED <= 512, "tensor memory");
    static_assert(QATOM % 1024 == 0 && STAGE % 1024 == 0 && HSTAGE % 1024 == 0, "swizzled tiles stay 1024-byte aligned");
    static_assert(BYTES <= 227 * 1024, "shared memory");
};

// A bounded wait for the roles that wait long (the producers for a stage to be released, the
// MMA issuer for the next K^): between polls the warp sleeps, so that its polling takes fewer
// issue slots from the fold and PV warps that share its sub-partition.  The producers have
// slack and sleep longer; the MMA issuer's wake-up is on the tile's critical path.
template <uint32_t kSleepNs>
__device__ __forceinline__ bool mbar_wait_idle(uint32_t mbar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (tc::mbar_try_wait(mbar, parity)) return true;
        __nanosleep(kSleepNs);
    }
    return false;
}

__device__ __forceinline__ void flag_timeout(unsigned int* err) {
    if (err) atomicOr(err, 1u);
}

// Row index / group by a multiply (exact for every row index here; see make_plan's bounds).
__device__ __forceinline__ int div_group_tc(int x, int magic) { return (int)(((uint32_t)x * (uint32_t)magic) >> 20); }

__device__ __forceinline__ int frexp_exp(float x) { return (int)((__float_as_uint(x) >> 23) & 0xFFu) - 126; }
__device__ __forceinline__ float pow2i(int n) { return __uint_as_float((uint32_t)(n + 127) << 23); }

// One box of a 3-D byte tensor map into shared memory, completion counted on `mbar` in bytes.
// x is 0 or 128 (bytes), as a tiled copy of a byte tensor requires (a multiple of 16).
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar)
        : "memory");
}

// Arrive on `mbar` once every cp.async this thread has issued so far has landed (the arrival is
// one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint32_t mbar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(mbar) : "memory");
}

// Barrier `id` over `n` threads, returning the OR of `pred` over them.
__device__ __forceinline__ bool bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void bar_named(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// (s0, s1) += (a, a) * (b0, b1): one packed fp32 FMA, each half rounded as fmaf would.
__device__ __forceinline__ void fma2(float& s0, float& s1, float a, float b0, float b1) {
    asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %2};\n mov.b64 y, {%3, %4};\n mov.b64 z, {%0, %1};\n"
        " fma.rn.f32x2 z, x, y, z;\n mov.b64 {%0, %1}, z;\n}\n"
        : "+f"(s0), "+f"(s1)
        : "f"(a), "f"(b0), "f"(b1));
}

// (s0, s1) -= (a, b) and (s0, s1) += (a, b): one packed fp32 instruction, each half rounded as
// the scalar operation would.
__device__ __forceinline__ void sub2(float& s0, float& s1, float a, float b) {
    asm("{\n .reg .b64 x, z;\n mov.b64 x, {%2, %3};\n mov.b64 z, {%0, %1};\n sub.rn.f32x2 z, z, x;\n"
        " mov.b64 {%0, %1}, z;\n}\n"
        : "+f"(s0), "+f"(s1)
        : "f"(a), "f"(b));
}
__device__ __forceinline__ void add2(float& s0, float& s1, float a, float b) {
    asm("{\n .reg .b64 x, z;\n mov.b64 x, {%2, %3};\n mov.b64 z, {%0, %1};\n add.rn.f32x2 z, z, x;\n"
        " mov.b64 {%0, %1}, z;\n}\n"
        : "+f"(s0), "+f"(s1)
        : "f"(a), "f"(b));
}

// RP columns of one accumulator block (this warp's rows: RP/2 hi then RP/2 lo columns).
template <int RP>
__device__ __forceinline__ void ld_rows(uint32_t taddr, uint32_t (&d)[RP]) {
    if constexpr (RP == 24) {
        tc::tmem_ld16(taddr, d);
        tc::tmem_ld8(taddr + 16, d + 16);
    } else if constexpr (RP == 16) {
        tc::tmem_ld16(taddr, d);
    } else {
        tc::tmem_ld8(taddr, d);
    }
}

template <int HD, int RP, bool APPEND, bool TREE, bool V4>
__global__ void __launch_bounds__(kTcThreads, 1) verify_tc_kernel(const __grid_constant__ VerifyTcParams p) {
    using L = TcLayout<HD, RP, V4>;
    constexpr int NB = L::NB, RPH = L::RPH, N = L::N, PS = L::PS, NT = RP / 8, MTW = HD / 128;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) { return sb + (uint32_t)L::BARS + 8u * (uint32_t)i; };
    const int chunk = blockIdx.x, split = blockIdx.y, kvh = blockIdx.z;
    const int R = p.n_rows * p.group;
    const int rows_total = p.n_rows * p.n_q_heads;
    const int row0 = chunk * p.rows_per_chunk;
    const int rows_here = min(p.rows_per_chunk, R - row0);
    // slice s covers keys [s kps - key_shift, (s + 1) kps - key_shift) clipped to [0, kv_len); on
    // the append path slice n_ctx_splits holds the window keys alone (see make_plan)
    const int key_base = split * p.keys_per_split - p.key_shift;
    const int key_begin = split == 0 ? 0 : key_base;
    const int key_end = min(key_base + p.keys_per_split, p.kv_len);
    const int n_tiles = key_end > key_begin ? (key_end - key_begin + kKT - 1) / kKT : 0;
    const int64_t head_row0 = (int64_t)kvh * p.capacity;
    const bool window = APPEND && split >= p.n_ctx_splits;
    const bool producer = warp == kKProdWarp || warp == kVProdWarp;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::SLOT);
    int* sVis = reinterpret_cast<int*>(smem + L::VIS);
    uint32_t* sWm = reinterpret_cast<uint32_t*>(smem + L::WM);
    constexpr bool tree = TREE;  // rows see the window keys their masks select (p.wmask)

    // The merge kernel may be launched now; it waits for this grid before reading.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(bar(L::KF + s), 33);  // the tensor-copy arrival + 32 scale-copy arrivals
            tc::mbar_init(bar(L::KE + s), 8);   // the fold warps
            tc::mbar_init(bar(L::PF + s), 8);   // the fold warps
            tc::mbar_init(bar(L::PE + s), 8);   // the PV warps
        }
        for (int s = 0; s < kVSlots; ++s) {
            tc::mbar_init(bar(L::VF + s), 33);
        }
        tc::mbar_init(bar(L::KH), 8);   // K^ of the tile written (and the previous accumulators read)
        tc::mbar_init(bar(L::QKD), 1);
        tc::mbar_init(bar(L::VGO), 1);  // K tile 0 has landed: the other stages may go out
        tc::mbar_init_fence();
    }
    if (warp == kMmaWarp) tc::tmem_alloc(smem_u32(tmem_slot), L::TM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- producers (all 32 lanes): K tile t into stage t & 1, or V unit h (keys
    // key_begin + kVKeys h ..) into slot h % kVSlots; codes by tensor copies, scales by async copies
    auto load_stage = [&](bool vplane, int t) {
        const int nkeys = vplane ? L::HKEYS : kKT;
        const int key0 = key_begin + t * nkeys;
        const uint32_t st = sb + (uint32_t)(vplane ? L::VST + (t % kVSlots) * L::HSTAGE : L::KST + (t & 1) * L::STAGE);
        const uint32_t full = bar(vplane ? L::VF + t % kVSlots : L::KF + (t & 1));
        const int codes = vplane ? L::HCODES : L::CODES;
        if (lane == 0) {
            tc::mbar_arrive_expect_tx(full, (uint32_t)codes);
#pragma unroll
            for (int bx = 0; bx < (vplane ? L::NBOXV : L::NBOX); ++bx)
                tma_box(st + (uint32_t)(bx * (vplane ? L::HBOX : L::BOX)), vplane ? &p.tmap_v : &p.tmap_k, 128 * bx,
                        key0, kvh, full);
        }
        const uint16_t* plane = vplane ? p.v_scales : p.k_scales;
        for (int n = lane; n < nkeys; n += 32) {
            const int key = key0 + n;
            const bool live = key < p.kv_len;
            const uint16_t* src = plane + (head_row0 + (live ? key : 0)) * NB;
            const uint32_t dst = st + (uint32_t)(codes + n * NB * 2);
            if constexpr (NB * 2 == 16)
                cp_async_16(dst, src, live ? 16 : 0);
            else
                cp_async_8(dst, src, live ? 8 : 0);
        }
        cp_async_arrive(full);
    };
    const int n_halves = (kKT / kVKeys) * n_tiles;  // V units
    // K tile 0 goes out first and alone, before the q rows are staged, so that it reaches every
    // block ahead of the other stages' bytes (all blocks start at once); the other first stages
    // follow once it has landed.  The window slice of the append path first writes its tokens
    // into the cache, below.
    if (warp == kKProdWarp && !window && n_tiles > 0) load_stage(false, 0);
    // Launched as a programmatic dependent: the kernel before this one in the stream may still be
    // running (the previous call's merge kernel).  Reading K tile 0 before this wait is safe: no
    // kernel of the library that lets a dependent start early writes the cache.  Everything else
    // (q, the window tokens' cache writes, the partials) comes after it.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (!producer) {
        const int wtid = threadIdx.x - (warp > kVProdWarp ? 64 : 0);  // 0 .. kWorkThreads - 1
        // ---- q rows of the chunk -> B operand: fp16 hi and lo, row order [hi h0 | lo h0 | hi h1 |
        // lo h1] (h = fold half), 64-dim atoms of N rows x 128 bytes, 128-byte swizzle
        constexpr int GPR = HD / 8;
        for (int idx = wtid; idx < RP * GPR; idx += kWorkThreads) {
            const int r = idx / GPR, j8 = idx - r * GPR;
            float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (r < rows_here) {
                const int rr = row0 + r;
                const int i = div_group_tc(rr, p.group_magic), hh = rr - i * p.group;
                const float4* src =
                    reinterpret_cast<const float4*>(p.q + ((int64_t)i * p.n_q_heads + kvh * p.group + hh) * HD) + 2 * j8;
                const float4 a = __ldg(src), b = __ldg(src + 1);
                x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
            }
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = x[2 * e] * p.qscale, b = x[2 * e + 1] * p.qscale;
                const __half2 hv = __floats2half2_rn(a, b);
                const __half2 lv = __floats2half2_rn(a - __low2float(hv), b - __high2float(hv));
                hi[e] = h2_as_u32(hv);
                lo[e] = h2_as_u32(lv);
            }
            const int nh = (r / RPH) * RP + (r % RPH), nl = nh + RPH;
            const int d0 = 8 * j8, c = (d0 & 63) >> 3;
            uint8_t* atom = smem + L::Q + (d0 >> 6) * L::QATOM;
            *reinterpret_cast<uint4*>(atom + nh * 128 + ((c ^ (nh & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(atom + nl * 128 + ((c ^ (nl & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        // visibility bound of each row of the chunk (padding rows: 0); a tree window's row sees
        // every key below q_pos0 and the window keys q_pos0 + j its mask selects (bit j)
        if (wtid < RP) {
            const int r = wtid;
            int v = 0;
            uint32_t wm = 0u;
            if (r < rows_here) {
                const int i = div_group_tc(row0 + r, p.group_magic);
                v = min(min(tree ? p.q_pos0 + 32 : p.q_pos0 + i + 1, p.kv_len), key_end);
                if (tree) wm = __ldg(p.wmask + i);
            }
            sVis[r] = v;
            sWm[r] = wm;
        }
        if (APPEND && window) {
            // the window tokens' keys and values -> Q8_0 in the cache (bit-exact with the append
            // kernel: the same block quantiser), then read back by the tensor copies like any
            // tile.  Every row chunk's window block stores the same bytes.
            const int nk = key_end - key_begin, nblk = nk * NB;
            const int t8 = wtid >> 3, sub = wtid & 7;
            for (int base = 0; base < 2 * nblk; base += kWorkThreads / 8) {  // same trip count in every warp
                const int blk = base + t8;
                const bool live = blk < 2 * nblk;
                const bool vplane = blk >= nblk;
                const int bb = vplane ? blk - nblk : blk;
                const int j = bb / NB, b = bb - j * NB;
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (live)
                    x = __ldg(reinterpret_cast<const float4*>((vplane ? p.v_new : p.k_new) +
                                                              ((int64_t)j * p.n_kv_heads + kvh) * HD + 32 * b) + sub);
                uint16_t scale_bits;
                const uint32_t packed = q8_0_block(x, &scale_bits);
                if (!live) continue;
                const int64_t row = head_row0 + key_begin + j;
                int8_t* codes = vplane ? p.v_codes : p.k_codes;
                uint16_t* scales = vplane ? p.v_scales : p.k_scales;
                *reinterpret_cast<uint32_t*>(codes + row * HD + 32 * b + 4 * sub) = packed;
                if (sub == 0) scales[row * NB + b] = scale_bits;
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");  // the stores above before the tensor copies
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the q tile before the tensor cores read it
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (producer) {
        // ---------------------------------------------------------------- K / V producers
        // Each refills the stage of tile t with tile t + 2 once its consumers release tile t.
        const bool vplane = warp == kVProdWarp;
        const int slots = vplane ? kVSlots : 2;        // ring depth
        const int total = vplane ? n_halves : n_tiles;  // loads of this plane
        const int issued0 = min(total, slots);
        int issued = issued0;
        bool ok = true;
        if (!vplane) {
            if (window && n_tiles > 0) load_stage(false, 0);
            // this warp alone refills slot 0, so the slot cannot run a phase ahead of this wait
            if (n_tiles > 0) ok = __all_sync(0xffffffffu, mbar_wait_idle<kProdSleepNs>(bar(L::KF), 0, kTcWait));
            for (int t = 1; t < issued0; ++t) load_stage(false, t);
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar(L::VGO));
        } else {
            ok = __all_sync(0xffffffffu, mbar_wait_idle<kProdSleepNs>(bar(L::VGO), 0, kTcWait));
            for (int t = 0; t < issued0; ++t) load_stage(true, t);
        }
        if (!ok && lane == 0) flag_timeout(p.err);
        ok = true;
        // a V slot (one tile) is free when the PV warps release that tile's P buffer
        static_assert(kVKeys == kKT && kVSlots == 2, "one V slot per tile, paired with the P buffers");
        const uint32_t empty0 = bar(vplane ? L::PE : L::KE);
        for (int t = 0; t + slots < total; ++t) {  // load t + slots into the slot load t leaves
            ok = __all_sync(0xffffffffu, mbar_wait_idle<kProdSleepNs>(empty0 + 8u * (uint32_t)(t % slots), (t / slots) & 1, kTcWait));
            if (!ok) break;
            load_stage(vplane, t + slots);
            issued = t + slots + 1;
        }
        if (!ok && lane == 0) flag_timeout(p.err);
        // never leave the block while a copy into its shared memory is in flight
        const uint32_t full0 = bar(vplane ? L::VF : L::KF);
        for (int i = max(0, issued - slots); i < issued; ++i)
            if (!tc::mbar_wait(full0 + 8u * (uint32_t)(i % slots), (i / slots) & 1, kTcWait) && lane == 0)
                flag_timeout(p.err);
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- QK MMA issuer
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            for (int t = 0; t < n_tiles; ++t) {
                if (!mbar_wait_idle<kMmaSleepNs>(bar(L::KH), t & 1, kTcWait)) { ok = false; break; }
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < HD / 16; ++ks)
                    tc::mma_ts(tmem + L::TM_D + (uint32_t)((ks >> 1) * N), tmem + L::TM_KH + (uint32_t)(ks * 8),
                               tc::smem_desc_sw128(sb + (uint32_t)(L::Q + (ks >> 2) * L::QATOM + (ks & 3) * 32), 16,
                                                   1024),
                               L::IDESC, (uint32_t)(ks & 1));
                tc::mma_commit(bar(L::QKD));
                issued = t + 1;
            }
            if (!ok) flag_timeout(p.err);
            // tensor memory is released only after the last committed MMA has completed
            if (issued > 0 && !tc::mbar_wait(bar(L::QKD), (issued - 1) & 1, kTcWait)) flag_timeout(p.err);
        }
        __syncwarp();
    } else if (warp < kPvWarp0) {
        // ---------------------------------------------------------------- fold warps
        // Iteration t: the K codes of tile t -> fp16 (exact) -> the A operand in tensor memory
        // (this warp's half of the dims), after the QK accumulators of tile t - 1 have been
        // read and their K scales folded in; then tile t - 1's mask, lazy row maxima and p.
        const int fw = warp - kFoldWarp0;
        const int qd = fw & 3, h = fw >> 2;
        const int key_lane = 32 * qd + lane;
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        const int vis_min =
            min(min(tree ? p.q_pos0 : p.q_pos0 + div_group_tc(row0, p.group_magic) + 1, p.kv_len), key_end);
        float m_ref[RPH], l_acc[RPH], s[RPH];
#pragma unroll
        for (int rr = 0; rr < RPH; ++rr) {
            m_ref[rr] = -INFINITY;
            l_acc[rr] = 0.0f;
            s[rr] = 0.0f;
        }
        uint32_t dk_prev[NB / 2], dk_cur[NB / 2];
#pragma unroll
        for (int i = 0; i < NB / 2; ++i) dk_prev[i] = dk_cur[i] = 0u;
        bool ok = true;
        for (int t = 0; t <= n_tiles; ++t) {
            if (t >= 1) {
                // ---- S of tile t-1: the K scales folded into the per-block accumulators
                if (ok) ok = tc::mbar_wait(bar(L::QKD), (t - 1) & 1, kTcWait);
                ok = __all_sync(0xffffffffu, ok);
                tc::fence_after_sync();
#pragma unroll
                for (int rr = 0; rr < RPH; ++rr) s[rr] = 0.0f;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    uint32_t d[RP];
                    ld_rows<RP>(tmem + lane_base + L::TM_D + (uint32_t)(b * N + h * RP), d);
                    tc::tmem_wait_ld();
                    const uint32_t w = dk_prev[b >> 1];
                    const float dk = __half2float(__ushort_as_half((unsigned short)((b & 1) ? (w >> 16) : (w & 0xFFFFu))));
#pragma unroll
                    for (int rr = 0; rr < RPH; rr += 2) {
                        fma2(s[rr], s[rr + 1], dk, __uint_as_float(d[rr]), __uint_as_float(d[rr + 1]));
                        fma2(s[rr], s[rr + 1], dk, __uint_as_float(d[RPH + rr]), __uint_as_float(d[RPH + rr + 1]));
                    }
                }
            }
            if (t < n_tiles) {
                // ---- K codes of tile t -> fp16 -> tensor memory (K^ is free: its MMAs completed)
                const int st = t & 1;
                if (ok) ok = tc::mbar_wait(bar(L::KF + st), (t >> 1) & 1, kTcWait);
                ok = __all_sync(0xffffffffu, ok);
                const uint8_t* kst = smem + L::KST + st * L::STAGE;
                if constexpr (NB == 8) {
                    const uint4 v = *reinterpret_cast<const uint4*>(kst + L::CODES + key_lane * 16);
                    dk_cur[0] = v.x; dk_cur[1] = v.y; dk_cur[2] = v.z; dk_cur[3] = v.w;
                } else {
                    const uint2 v = *reinterpret_cast<const uint2*>(kst + L::CODES + key_lane * 8);
                    dk_cur[0] = v.x; dk_cur[1] = v.y;
                }
#pragma unroll
                for (int pass = 0; pass < HD / 64; ++pass) {  // 32 dims = 16 columns per store
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int gc = h * (HD / 32) + pass * 2 + j;  // 16-byte chunk of the key's row
                        const int bx = gc >> 3, cib = gc & 7;
                        const uint4 x = *reinterpret_cast<const uint4*>(kst + bx * L::BOX + key_lane * 128 +
                                                                       ((cib ^ (key_lane & 7)) << 4));
                        const uint32_t xs[4] = {x.x ^ 0x80808080u, x.y ^ 0x80808080u, x.z ^ 0x80808080u,
                                                x.w ^ 0x80808080u};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            w[8 * j + 2 * e] = biased_bytes_to_half2<0x4140>(xs[e]);
                            w[8 * j + 2 * e + 1] = biased_bytes_to_half2<0x4342>(xs[e]);
                        }
                    }
                    tc::tmem_st16(tmem + lane_base + L::TM_KH + (uint32_t)(h * (HD / 4) + pass * 16), w);
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(L::KE + st));
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(L::KH));
            }
            if (t >= 1) {
                // ---- tile t-1: mask, lazy row maxima, p = 2^(s - ref) as fp16 hi + lo
                const int tile0 = key_begin + (t - 1) * kKT;
                const int key = tile0 + key_lane;
                if (tile0 + kKT > vis_min) {
#pragma unroll
                    for (int rr = 0; rr < RPH; ++rr)
                        if (key >= sVis[h * RPH + rr] ||
                            (tree && key >= p.q_pos0 && !((sWm[h * RPH + rr] >> (key - p.q_pos0)) & 1u)))
                            s[rr] = -INFINITY;
                }
                bool need = false;
#pragma unroll
                for (int rr = 0; rr < RPH; ++rr) need |= s[rr] > m_ref[rr] + kLazyTc;
                need = bar_or(1, 256, need);
                float afac[RPH];
#pragma unroll
                for (int rr = 0; rr < RPH; ++rr) afac[rr] = 1.0f;
                if (need) {
                    float* red = reinterpret_cast<float*>(smem + L::RED);
#pragma unroll
                    for (int rr = 0; rr < RPH; ++rr) {
                        float m = s[rr];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                        if (lane == 0) red[qd * RP + h * RPH + rr] = m;
                    }
                    bar_named(1, 256);
#pragma unroll
                    for (int rr = 0; rr < RPH; ++rr) {
                        const int r = h * RPH + rr;
                        const float tmax = fmaxf(fmaxf(red[r], red[RP + r]), fmaxf(red[2 * RP + r], red[3 * RP + r]));
                        const float m_old = m_ref[rr];
                        const float m_new = fmaxf(m_old, tmax);
                        const float a = m_old == -INFINITY ? 1.0f : ex2_approx(m_old - m_new);
                        m_ref[rr] = m_new;
                        l_acc[rr] *= a;
                        afac[rr] = a;
                    }
                }
#pragma unroll
                for (int rr = 0; rr < RPH; rr += 2) {  // row pairs: packed subtract and sum
                    const float mb0 = m_ref[rr] == -INFINITY ? 0.0f : m_ref[rr] - kPShiftTc;
                    const float mb1 = m_ref[rr + 1] == -INFINITY ? 0.0f : m_ref[rr + 1] - kPShiftTc;
                    sub2(s[rr], s[rr + 1], mb0, mb1);
                    s[rr] = ex2_approx(s[rr]);
                    s[rr + 1] = ex2_approx(s[rr + 1]);
                    add2(l_acc[rr], l_acc[rr + 1], s[rr], s[rr + 1]);
                }
                // P(t-1) into buffer (t-1) & 1 once the PV warps are done with tile t-3
                const int pb = (t - 1) & 1, pu = (t - 1) >> 1;
                if (pu >= 1 && ok) ok = tc::mbar_wait(bar(L::PE + pb), (pu - 1) & 1, kTcWait);
                ok = __all_sync(0xffffffffu, ok);
                uint2* sP = reinterpret_cast<uint2*>(smem + L::P + pb * L::PBUF);
                // a key and its pair partner sit in adjacent lanes: the even lane writes the first
                // half of this warp's rows, the odd lane the second half
                const bool ev = (lane & 1) == 0;
                const int kp = key_lane >> 1;
#pragma unroll
                for (int k = 0; k < RPH / 2; ++k) {
                    const float send = ev ? s[RPH / 2 + k] : s[k];
                    const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
                    const float pe = ev ? s[k] : recv;
                    const float po = ev ? recv : s[RPH / 2 + k];
                    const __half2 ph = __floats2half2_rn(pe, po);
                    float re = pe, ro = po;  // the residuals p - hi, one packed subtract
                    sub2(re, ro, __low2float(ph), __high2float(ph));
                    const __half2 pl = __floats2half2_rn(re, ro);
                    const int row = h * RPH + (ev ? k : RPH / 2 + k);
                    sP[kp * PS + row] = make_uint2(h2_as_u32(ph), h2_as_u32(pl));
                }
                float* hdr = reinterpret_cast<float*>(smem + L::PH + pb * L::PHB);
                if (qd == 0 && lane < RPH) {
                    float av = 1.0f;
#pragma unroll
                    for (int rr = 0; rr < RPH; ++rr)
                        if (lane == rr) av = afac[rr];
                    hdr[4 + h * RPH + lane] = av;
                }
                if (fw == 0 && lane == 0) *reinterpret_cast<int*>(hdr) = need ? 1 : 0;
                // fold warp 0 publishes P(t-1) only once V(t-1) has landed, so that the PV warps
                // wait on one barrier per tile; the V slot cannot run a phase ahead of this wait
                // (it is refilled only after the PV warps have released tile t-1).  Lane 0, the
                // one that arrives, waits itself.
                if (fw == 0 && lane == 0 && ok)
                    ok = tc::mbar_wait(bar(L::VF + (t - 1) % kVSlots), ((t - 1) / kVSlots) & 1, kTcWait);
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(L::PF + pb));
            }
#pragma unroll
            for (int i = 0; i < NB / 2; ++i) dk_prev[i] = dk_cur[i];
        }
        if (!ok && lane == 0) flag_timeout(p.err);
        // ---- row sums over the tile's keys (lanes, then lane quadrants) and the (m, l) partial
        float* lred = reinterpret_cast<float*>(smem + L::LRED);
#pragma unroll
        for (int rr = 0; rr < RPH; ++rr) {
            float v = l_acc[rr];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) lred[qd * RP + h * RPH + rr] = v;
        }
        bar_named(1, 256);
        if (qd == 0 && lane < RPH) {
            const int r = h * RPH + lane;
            float m = -INFINITY;
#pragma unroll
            for (int rr = 0; rr < RPH; ++rr)
                if (lane == rr) m = m_ref[rr];
            if (r < rows_here) {
                const float l = (lred[r] + lred[RP + r]) + (lred[2 * RP + r] + lred[3 * RP + r]);
                const int rr = row0 + r;
                const int i = div_group_tc(rr, p.group_magic), hh = rr - i * p.group;
                const int grow = i * p.n_q_heads + kvh * p.group + hh;
                p.part_ml[(int64_t)split * rows_total + grow] =
                    make_float2(m == -INFINITY ? -INFINITY : m * kLn2, l * pow2i(-(int)kPShiftTc));
            }
        }
    } else {
        // ---------------------------------------------------------------- PV warps
        const int pw = warp - kPvWarp0;
        const int g = lane >> 2, tq = lane & 3;
        const int pvb = HD == 256 ? pw : (pw >> 1);  // output block of this warp
        uint16_t* sDv = reinterpret_cast<uint16_t*>(smem + L::DV) + pw * kKT;
        float O[MTW][NT][4];
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c) O[mt][nt][c] = 0.0f;
        int E = INT32_MIN;  // unset
        // the lane's 4 code bytes of rows 2tq (+1): dims 32 pvb + 4g, box (32 pvb) / 128, 16-byte
        // chunk 2 (pvb % 4) + g / 4 stored at chunk ^ (row % 8); rows + 8 share the phase
        const int hb = (32 * pvb) >> 7;
        const int cq = 2 * (pvb & 3) + (g >> 2);
        const int v_off0 = hb * L::HBOX + (2 * tq) * 128 + ((cq ^ (2 * tq)) << 4) + 4 * (g & 3);
        const int v_off1 = hb * L::HBOX + (2 * tq + 1) * 128 + ((cq ^ (2 * tq + 1)) << 4) + 4 * (g & 3);
        // 4-bit V (hd256): the lane's dims 32 pvb + 4g .. +3 are the 2 bytes at 2g of chunk pvb
        // (4 nibbles, element 2m in the low nibble of byte m), stored at chunk pvb ^ (row % 8)
        const int v4_off0 = (2 * tq) * 128 + ((pvb ^ (2 * tq)) << 4) + 2 * g;
        const int v4_off1 = (2 * tq + 1) * 128 + ((pvb ^ (2 * tq + 1)) << 4) + 2 * g;
        bool ok = true;
        for (int t = 0; t < n_tiles && ok; ++t) {
            const int b = t & 1, u = t >> 1;
            if (!__all_sync(0xffffffffu, tc::mbar_wait(bar(L::PF + b), u & 1, kTcWait))) { ok = false; break; }
            const float* hdr = reinterpret_cast<const float*>(smem + L::PH + b * L::PHB);
            if (*reinterpret_cast<const int*>(hdr)) {  // the row maxima moved: rescale O first
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const float a = hdr[4 + 8 * nt + 2 * tq + c];
#pragma unroll
                        for (int mt = 0; mt < MTW; ++mt) {
                            O[mt][nt][c] *= a;
                            O[mt][nt][2 + c] *= a;
                        }
                    }
            }
            const int tile0 = key_begin + t * kKT;
            const int nk = min(kKT, key_end - tile0);
            const uint2* p_tile = reinterpret_cast<const uint2*>(smem + L::P + b * L::PBUF) + tq * PS + g;
            for (int hh = 0; hh < kKT / kVKeys; ++hh) {
                const int hv = (kKT / kVKeys) * t + hh;  // V unit
                const int slot = hv % kVSlots;
                // the tile's V codes have landed: fold warp 0 saw VF before it published P
                const uint8_t* vst = smem + L::VST + slot * L::HSTAGE;
                const uint16_t* sVs = reinterpret_cast<const uint16_t*>(vst + L::HCODES);
                const int nkh = min(max(nk - L::HKEYS * hh, 0), L::HKEYS);  // the slice's keys in this half
                // Per output block, E keeps dV 2^E of the largest scale seen in [2, 4), so that
                // w = (p 2^4)(dV 2^E) < 2^14 stays in the fp16 range; w = hi + lo exactly up to
                // 2^-22: hi = fl(ph d), lo = fl((ph d - hi) + pl d), the first residual exact by FMA.
                // Only the slice's own keys count: the half's rows past key_end hold other keys
                // (or, on the append path, window rows being written), which p masks anyway.
                {
                    float dv[L::HKEYS / 32];
                    float dmax = 0.0f;
#pragma unroll
                    for (int k = 0; k < L::HKEYS / 32; ++k) {
                        dv[k] = lane + 32 * k < nkh ? half_bits_to_float(sVs[(lane + 32 * k) * NB + pvb]) : 0.0f;
                        dmax = fmaxf(dmax, dv[k]);
                    }
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
                    if (dmax > 0.0f) {
                        const int et = 2 - frexp_exp(dmax);
                        if (E == INT32_MIN) {
                            E = et;
                        } else if (et < E) {
                            const float f = pow2i(et - E);
#pragma unroll
                            for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                    for (int c = 0; c < 4; ++c) O[mt][nt][c] *= f;
                            E = et;
                        }
                    }
                    const float esc = (E == INT32_MIN) ? 0.0f : pow2i(E);
#pragma unroll
                    for (int k = 0; k < L::HKEYS / 32; ++k)
                        sDv[lane + 32 * k] = __half_as_ushort(__float2half_rn(dv[k] * esc));
                    __syncwarp();
                }
                const uint2* p_lane = p_tile + hh * (L::HKEYS / 16) * 8 * PS;
                auto pv_step = [&](const int ks) {  // 16 keys of this half
                    const int kb = ks * 16;
                    uint2 pp01[NT], pp89[NT];  // (hi, lo) pairs of keys (2tq, 2tq+1) and (2tq+8, 2tq+9), row g of n-tile
                    const uint2* pp = p_lane + ks * 8 * PS;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        pp01[nt] = pp[8 * nt];
                        pp89[nt] = pp[4 * PS + 8 * nt];
                    }
                    const __half2 d01 = u32_as_h2(*reinterpret_cast<const uint32_t*>(sDv + kb + 2 * tq));
                    const __half2 d89 = u32_as_h2(*reinterpret_cast<const uint32_t*>(sDv + kb + 2 * tq + 8));
                    uint32_t A[MTW][4];
                    const uint8_t* vp = vst + ks * 16 * 128;
                    if constexpr (V4) {
                        // keys (2tq, 2tq+1) and (2tq+8, 2tq+9) side by side, 4 nibbles of each per
                        // half: dims 4g, 4g+1 (mt 0) and 4g+2, 4g+3 (mt 1), exactly as fp16
                        const uint32_t x01 = (uint32_t)*reinterpret_cast<const uint16_t*>(vp + v4_off0) |
                                             ((uint32_t)*reinterpret_cast<const uint16_t*>(vp + v4_off1) << 16);
                        const uint32_t x89 = (uint32_t)*reinterpret_cast<const uint16_t*>(vp + v4_off0 + 8 * 128) |
                                             ((uint32_t)*reinterpret_cast<const uint16_t*>(vp + v4_off1 + 8 * 128) << 16);
                        A[0][0] = nib_lo_to_half2(x01);
                        A[0][1] = nib_hi_to_half2(x01);
                        A[0][2] = nib_lo_to_half2(x89);
                        A[0][3] = nib_hi_to_half2(x89);
                        A[MTW - 1][0] = nib_lo_to_half2(x01 >> 8);
                        A[MTW - 1][1] = nib_hi_to_half2(x01 >> 8);
                        A[MTW - 1][2] = nib_lo_to_half2(x89 >> 8);
                        A[MTW - 1][3] = nib_hi_to_half2(x89 >> 8);
                    } else {
                        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vp + v_off0) ^ 0x80808080u;
                        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vp + v_off1) ^ 0x80808080u;
                        const uint32_t w8 = *reinterpret_cast<const uint32_t*>(vp + v_off0 + 8 * 128) ^ 0x80808080u;
                        const uint32_t w9 = *reinterpret_cast<const uint32_t*>(vp + v_off1 + 8 * 128) ^ 0x80808080u;
                        if (HD == 256 || (pw & 1) == 0) {  // dims 4g, 4g+1 (and 4g+2, 4g+3 at hd256)
                            const uint32_t y01 = prmt2<0x5140>(w0, w1), y89 = prmt2<0x5140>(w8, w9);
                            A[0][0] = biased_bytes_to_half2<0x4140>(y01);
                            A[0][1] = biased_bytes_to_half2<0x4342>(y01);
                            A[0][2] = biased_bytes_to_half2<0x4140>(y89);
                            A[0][3] = biased_bytes_to_half2<0x4342>(y89);
                        }
                        if (HD == 256 || (pw & 1) == 1) {  // dims 4g+2, 4g+3
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
                // 32-key steps: key rows past nkh hold p = 0 (masked) and finite codes and scales
                // (zeros past kv_len), so a ragged half may round up
                const int n_u = (nkh + 31) >> 5;
#pragma unroll 2
                for (int u4 = 0; u4 < n_u; ++u4) {
                    pv_step(2 * u4);
                    pv_step(2 * u4 + 1);
                }
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar(L::PE + b));  // P buffer and V slot of tile t free
        }
        if (!ok && lane == 0) flag_timeout(p.err);
        // ---- the slice partial: O is (p 2^4)(v 2^E) summed; lane owns dims 32 pvb + 4g .. +3
        // (hd256) or the pair at 32 pvb + 4g + 2 (pw & 1) (hd128) of rows 8nt + 2tq + c
        float* po = p.part_o + (int64_t)split * rows_total * HD;
        const float inv = (E == INT32_MIN) ? 1.0f : pow2i(-E - (int)kPShiftTc);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int r = 8 * nt + 2 * tq + c;
                if (r >= rows_here) continue;
                const int rr = row0 + r;
                const int i = div_group_tc(rr, p.group_magic), hh = rr - i * p.group;
                const int grow = i * p.n_q_heads + kvh * p.group + hh;
                float* dst = po + (int64_t)grow * HD + 32 * pvb + 4 * g;
                if constexpr (HD == 256) {
                    *reinterpret_cast<float4*>(dst) = make_float4(O[0][nt][c] * inv, O[0][nt][2 + c] * inv,
                                                                  O[1][nt][c] * inv, O[1][nt][2 + c] * inv);
                } else {
                    *reinterpret_cast<float2*>(dst + 2 * (pw & 1)) =
                        make_float2(O[0][nt][c] * inv, O[0][nt][2 + c] * inv);
                }
            }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == kMmaWarp) tc::tmem_dealloc(tmem, L::TM_COLS);
}

// Tensor map of one code plane [n_kv_heads][capacity][row_bytes] (bytes; row_bytes = hd, or hd/2
// for 4-bit codes): dims (row_bytes, kv_len, n_kv_heads), so keys at or past kv_len read as zeros;
// box 128 bytes x box_keys keys x 1 head, 128-byte swizzle.
bool encode_code_plane(CUtensorMap* map, const int8_t* plane, int row_bytes, int kv_len, int n_kv_heads, int capacity,
                       int box_keys) {
    const EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)row_bytes, (cuuint64_t)kv_len, (cuuint64_t)n_kv_heads};
    const cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)capacity * row_bytes};
    const cuuint32_t box[3] = {128, (cuuint32_t)box_keys, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<int8_t*>(plane), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HD, int RP, bool APPEND, bool TREE, bool V4>
int launch_tc(const VerifyTcParams& vp, dim3 grid, cudaStream_t s) {
    using L = TcLayout<HD, RP, V4>;
    static SmemOptIn opt;
    if (opt.ensure(verify_tc_kernel<HD, RP, APPEND, TREE, V4>, L::BYTES) != KVQ8_OK) return KVQ8_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = L::BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, verify_tc_kernel<HD, RP, APPEND, TREE, V4>, vp) == cudaSuccess ? KVQ8_OK
                                                                                                 : KVQ8_ERR_CUDA;
}

template <int HD, bool APPEND, bool TREE, bool V4 = false>
int dispatch_rp(const VerifyTcParams& vp, int rp, dim3 grid, cudaStream_t s) {
    switch (rp) {
        case 8: return launch_tc<HD, 8, APPEND, TREE, V4>(vp, grid, s);
        case 16: return launch_tc<HD, 16, APPEND, TREE, V4>(vp, grid, s);
        case 24: return launch_tc<HD, 24, APPEND, TREE, V4>(vp, grid, s);
        default: return KVQ8_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_verify_tc(VerifyTcParams& vp, const Plan& pl, int n_kv_heads, bool append, bool v4, cudaStream_t s) {
    // 4-bit V (K8V4 pools): causal windows at hd256 only, the V plane rows hd/2 bytes long
    if (v4 && (append || vp.wmask || pl.hd != 256)) return KVQ8_ERR_UNSUPPORTED;
    if (!encode_code_plane(&vp.tmap_k, vp.k_codes, pl.hd, vp.kv_len, n_kv_heads, vp.capacity, kKT) ||
        !encode_code_plane(&vp.tmap_v, vp.v_codes, v4 ? pl.hd / 2 : pl.hd, vp.kv_len, n_kv_heads, vp.capacity,
                           kVKeys))
        return KVQ8_ERR_CUDA;
    vp.err = device_error_flag();
    if (!vp.err) return KVQ8_ERR_CUDA;
    const int rp = 8 * pl.nt;
    const dim3 grid(pl.n_chunks, pl.n_split, n_kv_heads);
    // tree windows have no append variant (the append path is causal)
    if (append && vp.wmask) return KVQ8_ERR_UNSUPPORTED;
    if (v4) return dispatch_rp<256, false, false, true>(vp, rp, grid, s);
    if (pl.hd == 128)
        return append ? dispatch_rp<128, true, false>(vp, rp, grid, s)
                      : (vp.wmask ? dispatch_rp<128, false, true>(vp, rp, grid, s)
                                  : dispatch_rp<128, false, false>(vp, rp, grid, s));
    return append ? dispatch_rp<256, true, false>(vp, rp, grid, s)
                  : (vp.wmask ? dispatch_rp<256, false, true>(vp, rp, grid, s)
                              : dispatch_rp<256, false, false>(vp, rp, grid, s));
}

}  // namespace kvq8
