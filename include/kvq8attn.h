/*
 * kvq8attn.h -- C ABI of the Q8_0 GQA verify / prompt attention library (GB300, sm_103a).
 *
 * The operation: multi-row causal attention of fp32 (verify) or fp16 (prompt) query rows
 * over a grouped-query KV cache stored in the Q8_0 format -- int8 codes plus one fp16
 * scale per 32-value block.  Sources (titles and sections of the pages):
 *   - "perf(gfx1100): share Q8 KV scans across verifier rows", Summary: one wave owns
 *     four or eight Q8 attention query rows and shares each K/V scan across them; the
 *     partials layout and reducer stay as they are; the route is limited to Q8 KV,
 *     head_dim 128 or 256 and sequential (non-tree) windows of 4-32 rows.
 *   - "gfx12 WMMA kernel for the int8-KV QSA prompt attention", How: int8-KV prompt
 *     attention with online softmax and the V scale folded into p; the heads that
 *     share one KV head fill the rows of the tensor-core tile.
 *   - "Engine perf(hip): MTP draft, shared expert, verify/sampler head", Summary
 *     item 4: the warp-per-block Q8_0 quantiser, bitwise equal to its CPU reference.
 *
 * Layout of the cache (all device memory, owned by the caller):
 *   codes  int8   [n_kv_heads][capacity][head_dim]        one row of head_dim codes per token
 *   scales uint16 [n_kv_heads][capacity][head_dim / 32]   fp16 bit patterns, one per 32-code block
 * The dequantised value of element j of token n is codes[h][n][j] * fp16(scales[h][n][j/32]).
 *
 * Conventions shared by every entry point:
 *   - Query head h reads KV head h / (n_q_heads / n_kv_heads).
 *   - Query row i of a call sees keys n with n <= q_pos0 + i and n < kv_len.  A verify
 *     window of T rows after ctx cached tokens uses q_pos0 = ctx, kv_len = ctx + T; a
 *     prompt chunk of n_q rows ending the context uses q_pos0 = kv_len - n_q.
 *   - All pointers are device pointers (cudaMalloc / torch), 16-byte aligned, caller-owned.
 *     The library never allocates, frees or synchronises and keeps no state between
 *     calls; work is enqueued on `stream` (NULL = the legacy default stream).
 *   - Every call validates its arguments on the host first and, on any error, returns a
 *     nonzero status and launches nothing ("fail closed": there is no fallback route).
 *     A CUDA launch error is returned as KVQ8_ERR_CUDA.
 */
#ifndef KVQ8ATTN_H
#define KVQ8ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* kvq8_stream_t;

enum kvq8_status {
    KVQ8_OK = 0,
    KVQ8_ERR_INVALID_ARG = 1,   /* null pointer, negative or inconsistent size          */
    KVQ8_ERR_UNSUPPORTED = 2,   /* head_dim, group or row count outside what is built   */
    KVQ8_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned                     */
    KVQ8_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required           */
    KVQ8_ERR_CUDA = 5           /* a CUDA call or kernel launch failed                  */
};

/* The caller's cache planes.  head_dim is 128 or 256; capacity >= kv_len of any call. */
typedef struct {
    const int8_t* k_codes;
    const uint16_t* k_scales;
    const int8_t* v_codes;
    const uint16_t* v_scales;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t capacity;
} kvq8_cache;

/* A K8V4 KV pool: K as Q8_0 planes (as kvq8_cache), V as 4-bit blocks: v_codes holds
 * [n_kv_heads][capacity][head_dim / 2] bytes, element 2m in the low nibble of byte m stored
 * as code + 8 (code in [-7, 7]), v_scales one fp16 scale per 32 values as for Q8_0.
 * The pages run such a pool without stating its V format; the reading is the Q8_0 rule with
 * 7 in place of 127 ("gfx12 WMMA kernel for the int8-KV QSA prompt attention", Gating). */
typedef struct {
    const int8_t* k_codes;
    const uint16_t* k_scales;
    const uint8_t* v_codes;
    const uint16_t* v_scales;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t capacity;
} kvk8v4_cache;

/* An fp16 KV pool: K and V as IEEE binary16 bits, [n_kv_heads][capacity][head_dim] each,
 * device memory owned by the caller.  The pool format the pages keep on their older kernel
 * ("gfx12 WMMA kernel for the int8-KV QSA prompt attention", Gating and Limits). */
typedef struct {
    const uint16_t* k;
    const uint16_t* v;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t capacity;
} kvf16_cache;

/*
 * kvq8_quantize -- append n_tok tokens of K (or V) values to one plane pair.
 *   x      : fp32 [n_tok][n_kv_heads][head_dim]
 *   codes  : int8 plane [n_kv_heads][capacity][head_dim]; tokens land at [pos0, pos0 + n_tok)
 *   scales : uint16 plane [n_kv_heads][capacity][head_dim / 32]
 * Per 32-value block: amax = max |x|; d32 = amax / 127 (IEEE fp32 division); the stored
 * scale is fp16(d32) rounded to nearest even; code = clamp(round-half-away-from-zero(x / d32),
 * -127, 127) with an IEEE fp32 division; a block with d32 == 0 stores scale 0 and zero codes.
 * Results are bit-exact with that definition.  Inputs must be finite; for amax > 65504 * 127
 * the stored scale is +inf.  head_dim must be a multiple of 32.
 * Source: "Engine perf(hip): ...", Summary item 4 (warp-per-block Q8_0 quantiser).
 */
int kvq8_quantize(const float* x, int n_tok, int n_kv_heads, int head_dim,
                  int8_t* codes, uint16_t* scales, int capacity, int pos0, kvq8_stream_t stream);

/*
 * kvq8_append -- append n_tok tokens of K and V to both planes of a cache in one launch.
 *   k, v : fp32 [n_tok][kv->n_kv_heads][kv->head_dim], device memory; tokens land at
 *          positions [pos0, pos0 + n_tok) of every KV head.
 * Each plane is quantised exactly as kvq8_quantize would (bit-exact with it); the cache's
 * plane pointers are written through although the struct declares them const.
 * Errors: INVALID_ARG for null pointers, negative n_tok or pos0, or pos0 + n_tok > capacity;
 * UNSUPPORTED when head_dim is not a multiple of 32; MISALIGNED unless every pointer is
 * 16-byte aligned.
 * Source: "Engine perf(hip): ...", Summary item 4 (warp-per-block Q8_0 quantiser).
 */
int kvq8_append(const float* k, const float* v, int n_tok, const kvq8_cache* kv, int pos0,
                kvq8_stream_t stream);

/* Bytes of workspace attn_verify_q8 needs for this shape (n_split 0 = the automatic choice). */
size_t attn_verify_q8_workspace_bytes(int n_rows, int n_q_heads, int head_dim, int kv_len,
                                      int n_kv_heads, int n_split);

/*
 * attn_verify_q8 -- speculative-decode verify attention over a Q8_0 cache.
 *   q        : fp32 [n_rows][n_q_heads][head_dim], 1 <= n_rows <= 32
 *   kv       : the cache (head_dim 128 or 256; n_q_heads / n_kv_heads integral, <= 64)
 *   kv_len   : tokens of the cache to attend over; q_pos0: position of row 0 (see above)
 *   out      : fp32 [n_rows][n_q_heads][head_dim], normalised attention output
 *   workspace: device scratch of at least attn_verify_q8_workspace_bytes(...) bytes,
 *              caller-owned; holds the split-context partials between the two kernels
 *   n_split  : context slices per KV head (0 = automatic; otherwise 1..1024)
 * One thread block per (KV head, context slice) reads each K/V block of its slice from
 * HBM once for all n_rows x group query rows; the per-slice (o, m, l) partials are then
 * merged by log-sum-exp.  fp32 result; q and p enter the tensor cores as fp16 hi + lo
 * pairs, so the result stays within 1e-4 of the fp64 oracle (max |err| / max |out|).
 * Source: "perf(gfx1100): share Q8 KV scans across verifier rows", Summary.
 */
int attn_verify_q8(const float* q, int n_rows, int n_q_heads, const kvq8_cache* kv, int kv_len,
                   int q_pos0, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                   int n_split, kvq8_stream_t stream);

/* Partials attn_verify_q8_partials writes for this shape (its resolved n_split; 0 = invalid). */
int attn_verify_q8_partials_count(int n_rows, int n_q_heads, int head_dim, int kv_len, int n_kv_heads,
                                  int n_split);

/*
 * attn_verify_q8_partials -- the split-context scan of attn_verify_q8 without the merge: the
 * per-slice partials of the window rows over cache positions [0, kv_len).
 *   q_pos0   : position of row 0 in this cache's coordinates; row i sees positions <= q_pos0 + i.
 *              It may be negative (down to -2^30): a rank holding a later context slice in a
 *              cache of its own passes q_pos0 - (its slice's first key), and rows that see
 *              none of its keys get empty partials.
 *   part_o   : fp32 [n][n_rows * n_q_heads][head_dim], n = attn_verify_q8_partials_count(...)
 *   part_ml  : fp32 [n][n_rows * n_q_heads][2]
 *   The layout attn_combine takes: per slice and row, o = sum exp(s_n - m) v_n (unnormalised),
 *   m = max s_n in natural-log units (-inf when the row sees no key of the slice, o = 0 and
 *   l = 0 then) and l = sum exp(s_n - m).
 * Concatenating the partials of several calls (other ranks' slices of one context, in any
 * order) and passing them to attn_combine gives the attention over the union of the
 * slices.  Other arguments and errors as for attn_verify_q8; no workspace is used.
 * Source: "perf(gfx1100): share Q8 KV scans across verifier rows", Summary: the partials
 * layout and the reducer are kept; here they are the exchange of a context-sharded verify.
 */
int attn_verify_q8_partials(const float* q, int n_rows, int n_q_heads, const kvq8_cache* kv, int kv_len,
                            int q_pos0, float softmax_scale, float* part_o, float* part_ml, int n_split,
                            kvq8_stream_t stream);

/* Bytes of workspace attn_verify_append_q8 needs (kv_len = q_pos0 + n_rows; n_split as there). */
size_t attn_verify_append_q8_workspace_bytes(int n_rows, int n_q_heads, int head_dim, int q_pos0,
                                             int n_kv_heads, int n_split);

/*
 * attn_verify_append_q8 -- kvq8_append of the window's K and V, then attn_verify_q8 over
 * kv_len = q_pos0 + n_rows, as one call.
 *   k_new, v_new : fp32 [n_rows][kv->n_kv_heads][kv->head_dim], device, 16-byte aligned:
 *                  the window tokens' keys and values, quantised into positions
 *                  [q_pos0, q_pos0 + n_rows) of the cache (bit-exact with kvq8_append).
 *   n_split      : context slices over the keys below q_pos0 (0 = automatic); the window
 *                  keys get one more slice of their own.
 * Two launches, as attn_verify_q8: the verify grid gets one more slice per KV head holding
 * the window keys alone, and that slice's blocks quantise k_new / v_new themselves (into
 * their tiles and into the cache) while every other block scans the old keys.  The cache
 * bytes equal kvq8_append's; the result equals kvq8_append followed by attn_verify_q8 up to
 * rounding order (the slices differ).
 * Errors: as for kvq8_append and attn_verify_q8; INVALID_ARG also when k_new or v_new is
 * null or q_pos0 + n_rows > capacity.
 * No counterpart on the pages: the verify rows of "perf(gfx1100): share Q8 KV scans across
 * verifier rows" (Summary) attend to the window's own keys, so those keys must be in the
 * cache first; this entry point fuses that write (the quantiser of "Engine perf(hip): ...",
 * Summary item 4) with the scan so the two overlap.
 */
int attn_verify_append_q8(const float* q, const float* k_new, const float* v_new, int n_rows,
                          int n_q_heads, const kvq8_cache* kv, int q_pos0, float softmax_scale,
                          float* out, void* workspace, size_t workspace_bytes, int n_split,
                          kvq8_stream_t stream);

/* Device scratch attn_verify_append_q8_host needs (inputs, output and the verify workspace). */
size_t attn_verify_append_q8_host_scratch_bytes(int n_rows, int n_q_heads, int head_dim, int q_pos0,
                                                int n_kv_heads, int n_split);

/*
 * attn_verify_append_q8_host -- attn_verify_append_q8 from and to HOST buffers: the one entry
 * point that touches host memory.
 *   h_in   : host fp32, q [n_rows][n_q_heads][head_dim] followed by k_new and v_new
 *            [n_rows][n_kv_heads][head_dim] each (pinned memory keeps the copy asynchronous)
 *   h_out  : host fp32 [n_rows][n_q_heads][head_dim]
 *   d_scratch : device, 16-byte aligned, attn_verify_append_q8_host_scratch_bytes(...) bytes
 * Pinned host buffers (mapped into the device address space, as every pinned allocation is
 * on unified-addressing systems): a copy kernel reads h_in once over the host link into the
 * scratch, the two kernels of attn_verify_append_q8 run, and the merge writes h_out in place.
 * Pageable buffers: a host-to-device copy-engine transfer, the two kernels, a device-to-host
 * transfer.  All queued on `stream`; h_out is valid once the stream has reached the end (the
 * call itself does not synchronise).  Errors as for attn_verify_append_q8, WORKSPACE for a
 * short scratch; nothing is queued on error.
 */
int attn_verify_append_q8_host(const float* h_in, int n_rows, int n_q_heads, const kvq8_cache* kv,
                               int q_pos0, float softmax_scale, float* h_out, void* d_scratch,
                               size_t scratch_bytes, int n_split, kvq8_stream_t stream);

/*
 * kvk8v4_append -- append n_tok tokens of K (to Q8_0) and V (to 4-bit blocks) into a K8V4
 * pool at positions [pos0, pos0 + n_tok), one launch.  k, v: fp32 [n_tok][n_kv_heads][head_dim]
 * on the device.  The K bytes equal kvq8_append's.  Errors as for kvq8_append.
 */
int kvk8v4_append(const float* k, const float* v, int n_tok, const kvk8v4_cache* kv, int pos0,
                  kvq8_stream_t stream);

/*
 * attn_verify_k8v4 -- attn_verify_q8 over a K8V4 pool: the same window semantics, shapes,
 * workspace (attn_verify_q8_workspace_bytes), precision bound and errors; the V codes are
 * expanded from their nibbles in registers.
 */
int attn_verify_k8v4(const float* q, int n_rows, int n_q_heads, const kvk8v4_cache* kv, int kv_len,
                     int q_pos0, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                     int n_split, kvq8_stream_t stream);

/*
 * attn_prompt_k8v4 -- attn_prompt_q8 over a K8V4 pool (the same shapes, routes, workspace
 * from attn_prompt_q8_workspace_bytes, precision bound and errors); the dequantisers expand
 * the 4-bit V blocks (value (nibble - 8) * scale, rounded once to fp16) into the V tiles or,
 * on the two-pass route, into the fp16 copy.
 */
int attn_prompt_k8v4(const uint16_t* q, int n_q, int n_q_heads, const kvk8v4_cache* kv, int kv_len,
                     int q_pos0, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                     kvq8_stream_t stream);

/*
 * Bytes of workspace attn_prompt_f16 needs for this shape: the partials only (an fp16 pool has
 * no copy to make).  Never more than attn_prompt_q8_workspace_bytes for the same shape.
 */
size_t attn_prompt_f16_workspace_bytes(int n_q, int n_q_heads, int head_dim, int kv_len, int q_pos0,
                                       int n_kv_heads);

/*
 * attn_prompt_f16 -- attn_prompt_q8 over an fp16 pool (the same shapes, precision bound and
 * errors; workspace from attn_prompt_f16_workspace_bytes).  The K and V tiles are loaded
 * straight into the tensor-core operand layout by tensor copies over (head_dim, kv_len,
 * n_kv_heads), so keys at or past kv_len read as zeros; the caller's pool needs no padding.
 */
int attn_prompt_f16(const uint16_t* q, int n_q, int n_q_heads, const kvf16_cache* kv, int kv_len,
                    int q_pos0, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                    kvq8_stream_t stream);

/*
 * kvf16_append -- round n_tok tokens of K and V (fp32 [n_tok][n_kv_heads][head_dim], device)
 * to fp16 (nearest even) into both planes of an fp16 pool at positions [pos0, pos0 + n_tok).
 * Errors: INVALID_ARG for null pointers, negative sizes or pos0 + n_tok > capacity;
 * UNSUPPORTED when head_dim is not a multiple of 4; MISALIGNED unless every pointer is
 * 16-byte aligned.  The pool's plane pointers are written through.
 */
int kvf16_append(const float* k, const float* v, int n_tok, const kvf16_cache* kv, int pos0,
                 kvq8_stream_t stream);

/* Bytes of workspace attn_verify_f16 needs for this shape (n_split 0 = the automatic choice). */
size_t attn_verify_f16_workspace_bytes(int n_rows, int n_q_heads, int head_dim, int kv_len,
                                       int n_kv_heads, int n_split);

/*
 * attn_verify_f16 -- attn_verify_q8 over an fp16 KV pool: the same window semantics, shapes
 * (head_dim 128 or 256, 1 <= n_rows <= 32), split-context partials, merge, precision bound
 * (q and p as fp16 hi + lo, fp32 accumulation; within 1e-4 of the fp64 oracle) and errors.
 * The K and V values enter the tensor cores as they are stored; there are no block scales.
 * Source: "perf(gfx1100): share Q8 KV scans across verifier rows", Summary, for the
 * multi-row scan; the fp16 pool of "gfx12 WMMA kernel for the int8-KV QSA prompt
 * attention", Gating and Limits.
 */
int attn_verify_f16(const float* q, int n_rows, int n_q_heads, const kvf16_cache* kv, int kv_len,
                    int q_pos0, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                    int n_split, kvq8_stream_t stream);

/*
 * attn_verify_tree_q8 -- attn_verify_q8 for a tree-shaped verify window.
 *   window_mask : device uint32 [n_rows], 4-byte aligned: row i sees every key n < q_pos0
 *                 and the window key q_pos0 + j (j < 32, q_pos0 + j < kv_len) exactly when
 *                 bit j of window_mask[i] is set.  The sequential window of attn_verify_q8
 *                 is window_mask[i] = 2^(i+1) - 1; a tree of drafted tokens sets the bits
 *                 of a row's ancestors and of itself.  A row that sees no key gets zeros.
 * Everything else (shapes, workspace from attn_verify_q8_workspace_bytes, n_split,
 * precision, errors) is as for attn_verify_q8; a null window_mask is INVALID_ARG and a
 * misaligned one MISALIGNED.
 * The pages admit only sequential windows on the multi-row route and send trees to the
 * fallback ("perf(gfx1100): share Q8 KV scans across verifier rows", Summary: route
 * conditions); here a tree costs the same K/V scan as a chain.
 */
int attn_verify_tree_q8(const float* q, int n_rows, int n_q_heads, const kvq8_cache* kv, int kv_len,
                        int q_pos0, const uint32_t* window_mask, float softmax_scale, float* out,
                        void* workspace, size_t workspace_bytes, int n_split, kvq8_stream_t stream);

/*
 * argmax_rows_top_prob -- verify-head acceptance: per row of fp32 logits [n_rows][vocab]
 * (device, 4-byte aligned), argmax[i] (int32) = the first index of the row's maximum and
 * top_prob[i] (fp32) = softmax(row)[argmax[i]] = 1 / sum_j exp(x_j - max).
 * Special values: a row holding NaN gives the index of its first NaN and probability NaN;
 * +inf entries share the probability mass equally (argmax = the first +inf); a row of -inf
 * only gives index 0 and probability 1 / vocab; otherwise -inf entries carry probability 0.
 * argmax is exact; top_prob is within 1e-5 (relative) of its fp64 value.
 * workspace: device scratch of argmax_rows_top_prob_workspace_bytes(n_rows, vocab) bytes,
 * 16-byte aligned.  1 <= n_rows <= 65535, vocab >= 1.  Errors: INVALID_ARG, WORKSPACE,
 * MISALIGNED.  Two kernel launches; asynchronous on `stream`.
 * Source: "Engine perf(hip): MTP draft, shared expert, verify/sampler head", Summary item 1
 * and "Verification & Parity Evidence" (argmax_rows, row_top_prob over T x 248,320 logits).
 */
size_t argmax_rows_top_prob_workspace_bytes(int n_rows, int vocab);
int argmax_rows_top_prob(const float* logits, int n_rows, int vocab, int32_t* argmax, float* top_prob,
                         void* workspace, size_t workspace_bytes, kvq8_stream_t stream);

/*
 * attn_combine -- merge split-context partials (log-sum-exp reducer).
 *   part_o  : fp32 [n_split][rows][head_dim]  unnormalised o_s = sum_n exp(s_n - m_s) v_n
 *   part_ml : fp32 [n_split][rows][2]         (m_s, l_s): m_s = max s_n over the slice in natural-log
 *             units (-inf for an empty slice), l_s = sum_n exp(s_n - m_s)
 *   out     : fp32 [rows][head_dim] = sum_s o_s e^(m_s - m*) / sum_s l_s e^(m_s - m*), m* = max_s m_s;
 *             a row whose every slice is empty is written as zeros
 * head_dim is a multiple of 4, <= 1024; 1 <= n_split <= 4096.
 * Source: "perf(gfx1100): share Q8 KV scans across verifier rows", Summary (partials + reducer).
 */
int attn_combine(const float* part_o, const float* part_ml, int n_split, int rows, int head_dim,
                 float* out, kvq8_stream_t stream);

/*
 * Bytes of workspace attn_prompt_q8 (and attn_prompt_k8v4 / attn_prompt_f16) needs for this
 * shape (on the current device): the partials, plus, for chunks of 24 or more 128-row tiles
 * per KV head, room for the fp16 copy of both planes (2 * n_kv_heads * min(kv_len, q_pos0 +
 * n_q) * head_dim * 2 bytes) that the two-pass route writes.  fp16 pools never use that room
 * (attn_prompt_f16_workspace_bytes gives their smaller size).
 */
size_t attn_prompt_q8_workspace_bytes(int n_q, int n_q_heads, int head_dim, int kv_len, int q_pos0,
                                      int n_kv_heads);

/*
 * attn_prompt_q8 -- prompt-chunk attention: many query rows over a long Q8_0 context.
 *   q        : fp16 bits [n_q][n_q_heads][head_dim], head_dim 128 or 256
 *   kv       : the cache (the same head_dim, any n_kv_heads dividing n_q_heads)
 *   out      : fp32 [n_q][n_q_heads][head_dim]
 *   workspace: device scratch of at least attn_prompt_q8_workspace_bytes(...) bytes,
 *              caller-owned; holds the per-slice partials merged by the last kernel and,
 *              on the two-pass route, the fp16 copy of the planes
 *   softmax_scale must be > 0.
 * Row i sees keys n <= q_pos0 + i, n < kv_len.  K and V are dequantised to fp16 (code *
 * scale, one rounding) and contracted on the tcgen05 tensor cores with fp32 accumulation in
 * tensor memory; p enters the PV product as fp16.  Short chunks (fewer than 24 row tiles per
 * KV head) dequantise each tile on chip, once per row tile that sees it.  Longer chunks take
 * the two-pass route: one pass writes the fp16 planes of keys < min(kv_len, q_pos0 + n_q)
 * into the workspace, and the kernel of attn_prompt_f16 runs over that copy; the operands, and
 * so the results, are the same on both routes.  The work -- key tiles
 * (64 keys at head_dim 256, 128 at 128) of 128-row tiles of (query, head) pairs of every
 * KV head -- is cut into one equal
 * contiguous share per SM (a persistent grid); each share writes partials that the
 * log-sum-exp combine merges into `out`.  Tiles past a row tile's causal bound are
 * skipped.  Within 2e-3 of the fp64 oracle (max |err| / max |out|) for values inside the
 * fp16 range.  Every internal wait is bounded; a timeout sets the flag that
 * kvq8_device_error reports (the output is then undefined).
 * Source: "gfx12 WMMA kernel for the int8-KV QSA prompt attention", How and Measurements.
 */
int attn_prompt_q8(const uint16_t* q, int n_q, int n_q_heads, const kvq8_cache* kv, int kv_len,
                   int q_pos0, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                   kvq8_stream_t stream);

/*
 * attn_verify_q8_noalloc -- attn_verify_q8 for callers that cannot allocate device memory.
 *
 * No counterpart on the pages: this is a library convenience.  Some callers cannot call
 * cudaMalloc at the point where they run attention: a runtime that hands all device memory
 * out of its own fixed arena and forbids other allocations, code running inside a custom
 * allocator's callback (where allocating again would re-enter the allocator), or a plug-in
 * that is not allowed to touch the process allocator at all.  This entry point takes the same
 * arguments as attn_verify_q8 minus the workspace: the split-context partials live in one
 * static device array of KVQ8_NOALLOC_SCRATCH_BYTES bytes built into the library, which
 * every GPU that loads the library holds until the process exits.
 *   - It never calls cudaMalloc, cudaFree or any allocating library routine.
 *   - The first call on each device looks up the array's device address (with that device
 *     current); make that first call before any stream capture.
 *   - All calls share the one array: calls that overlap on the GPU (different streams, or
 *     several host threads) race on it and must be serialised by the caller.
 *   - With n_split = 0 the automatic plan is used: each KV head and row chunk (up to 24
 *     row x q-head pairs) gets at most SM count / (KV heads x chunks) context slices, so the
 *     partials take at most about SM count x 24 x (head_dim + 2) x 4 bytes (3.8 MB at
 *     head_dim 256 on 152 SMs).  When there are more KV heads x chunks than SMs every chunk
 *     gets one slice, n_rows * n_q_heads * (head_dim + 2) * 4 bytes in all.  A plan, automatic
 *     or from an explicit n_split, whose partials exceed the array returns KVQ8_ERR_WORKSPACE
 *     and launches nothing.
 */
#define KVQ8_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
int attn_verify_q8_noalloc(const float* q, int n_rows, int n_q_heads, const kvq8_cache* kv, int kv_len,
                           int q_pos0, float softmax_scale, float* out, int n_split, kvq8_stream_t stream);

/*
 * kvq8_selftest_convert -- a self-test hook: runs the code -> fp16 conversions that the verify
 * and prompt kernels use, unchanged, on caller data, so that a test can check them exhaustively.
 *   kind 0: in[i] = 4 int8 codes; out[2i], out[2i+1] = fp16 pairs of codes (0, 1) and (2, 3)
 *           (the K operand of the verify scans, the prompt dequantisers).  out: 2n words.
 *   kind 1: in[2i], in[2i+1] = words w0, w1 of 4 codes each (two key rows); out[4i + m] = the fp16
 *           pair (w0 byte m, w1 byte m) through the byte interleave of the PV operands.  n even;
 *           out: 2n words.
 *   kind 2: in[i] = two 16-bit halves of 4 nibbles each (stored code + 8); out[4i .. 4i+3] = the
 *           pairs of nibbles (0, 4), (1, 5), (2, 6), (3, 7), one from each half (the 4-bit PV
 *           operands).  out: 4n words.
 *   kind 3: in[i] = 4 bytes of nibble pairs; out[4i + m] = the pair (low, high) of byte m as
 *           codes (the 4-bit prompt dequantiser).  out: 4n words.
 * Each fp16 value must equal the code exactly.  in, out: device, 4-byte aligned.  Errors:
 * INVALID_ARG (kind, n, null pointers), MISALIGNED.  One launch on `stream`.
 * Source: "gfx12 WMMA kernel for the int8-KV QSA prompt attention", How: the exact int8 -> fp16
 * conversion, checked over all byte pairs.
 */
int kvq8_selftest_convert(int kind, const uint32_t* in, uint32_t* out, int n, kvq8_stream_t stream);

/*
 * kvq8_selftest_wait_timeout -- a self-test hook for the kernels' failure path: one launch whose
 * thread waits on an mbarrier that nothing arrives on, with the bounded wait every pipeline
 * kernel of the library uses, limited to `polls` polls.  The wait gives up, the kernel sets the
 * library's device error flag (read with kvq8_device_error) and returns; the context stays
 * usable.  polls: 1 .. 1 << 20.  Errors: INVALID_ARG (polls out of range), CUDA (no device
 * flag).  One launch on `stream`.
 */
int kvq8_selftest_wait_timeout(int polls, kvq8_stream_t stream);

/*
 * kvq8_device_error -- read (and with reset != 0, clear) the library's device error flag.
 * Nonzero means a kernel gave up on an internal wait after its bounded poll count and
 * returned early.  Returns the flag, or -1 if it could not be read.  Unlike every other
 * entry point this one synchronises: it copies the flag from the current device.
 */
int kvq8_device_error(int reset);

/* Human-readable name of a status code (static string). */
const char* kvq8_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* KVQ8ATTN_H */
