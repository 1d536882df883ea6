"""kvk8v4_append / attn_verify_k8v4 on the GPU against the fp64 oracle's K8V4 pool: the
append bit for bit (K as Q8_0, V as 4-bit nibbles + fp16 scales), attention within 1e-4."""
import numpy as np
import pytest

import oracle
from speculative_verify_attention_gb300 import workloads

from ._util import VERIFY_TOL, rel_err

pytestmark = pytest.mark.gpu


def _pools(inp, capacity=None, pos0=0, junk=True):
    """The same fp32 K/V appended to a library K8V4 pool and an oracle one; positions outside
    the written range hold the same junk (finite scales) in both."""
    import torch

    from speculative_verify_attention_gb300 import KVCacheK8V4
    L, hkv, hd = inp.k.shape
    cap = capacity or (pos0 + L)
    gpu = KVCacheK8V4(hkv, hd, cap, device="cuda")
    orc = oracle.CacheK8V4(hkv, hd, cap)
    if junk and cap > pos0 + L:
        rng = np.random.default_rng(2468)
        kc = rng.integers(-128, 128, (hkv, cap, hd), dtype=np.int8)
        vc = rng.integers(0, 256, (hkv, cap, hd // 2), dtype=np.uint8)
        sc = rng.integers(0, 1 << 16, (hkv, cap, hd // 32), dtype=np.uint16)
        sc[(sc & 0x7C00) == 0x7C00] = 0x7BFF
        orc.k_codes[:], orc.v_q4[:], orc.k_scales[:], orc.v_scales[:] = kc, vc, sc, sc
        gpu.k_codes.copy_(torch.from_numpy(kc))
        gpu.v_codes.copy_(torch.from_numpy(vc))
        gpu.k_scales.copy_(torch.from_numpy(sc.view(np.float16)))
        gpu.v_scales.copy_(torch.from_numpy(sc.view(np.float16)))
    gpu.append(torch.from_numpy(inp.k).cuda(), torch.from_numpy(inp.v).cuda(), pos0)
    orc.append(inp.k, inp.v, pos0)
    torch.cuda.synchronize()
    return gpu, orc


def _run(gpu, q, kv_len, q_pos0, scale, n_split=0):
    import torch

    from speculative_verify_attention_gb300 import attn_verify_k8v4
    out = attn_verify_k8v4(torch.from_numpy(np.ascontiguousarray(q, np.float32)).cuda(), gpu, kv_len, q_pos0, scale,
                           n_split=n_split)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_append_matches_oracle_bitwise(lib):
    inp = workloads.random_small(1300, 8, 2, 256, 45, 4)
    gpu, orc = _pools(inp, capacity=60, pos0=9)
    assert np.array_equal(gpu.k_codes.cpu().numpy(), orc.k_codes)
    assert np.array_equal(gpu.k_scales.cpu().numpy().view(np.uint16), orc.k_scales)
    assert np.array_equal(gpu.v_codes.cpu().numpy(), orc.v_q4)
    assert np.array_equal(gpu.v_scales.cpu().numpy().view(np.uint16), orc.v_scales)


def test_append_k_plane_equals_q8_append(lib):
    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8
    inp = workloads.random_small(1301, 8, 2, 128, 33, 4)
    gpu, _ = _pools(inp, junk=False)
    q8 = KVCacheQ8(2, 128, 33, device="cuda")
    q8.append(torch.from_numpy(inp.k).cuda(), torch.from_numpy(inp.v).cuda(), 0)
    torch.cuda.synchronize()
    assert torch.equal(gpu.k_codes, q8.k_codes) and torch.equal(gpu.k_scales, q8.k_scales)


@pytest.mark.parametrize("T,n_split", [(4, 0), (8, 0), (16, 0), (32, 0), (4, 3), (8, 1)])
def test_27b_shape(lib, T, n_split):
    w = workloads.verify_workload(f"k8v4-24q4kv-hd256-ctx1000-T{T}", 24, 4, 256, 1000, T, k_outliers=4,
                                  seed=1310 + T)
    inp = workloads.make_inputs(w)
    gpu, orc = _pools(inp, capacity=w.kv_len + 30)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, n_split)
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    assert rel_err(got, ref) <= VERIFY_TOL


@pytest.mark.parametrize("hq,hkv,L,T,pos0,n_split", [
    (6, 1, 3001, 1, 3000, 3),      # one 8-row chunk of 6 rows, ragged last tile
    (6, 1, 2500, 3, 2497, 4),      # 18 rows: one 24-row chunk
    (16, 1, 3333, 2, 3331, 2),     # group 16: 32 rows in two 16-row chunks
    (8, 8, 2000, 4, 1996, 2),      # MHA, eight KV heads
    (24, 4, 2600, 32, 2568, 2),    # T = 32: eight 24-row chunks per KV head
    (4, 1, 1500, 6, 1600, 2),      # rows past kv_len see kv_len keys
    (4, 1, 3000, 4, 2000, 3),      # kv_len beyond the window
    (24, 4, 2055, 8, 2047, 5),     # slices end mid-tile
])
def test_hd256_on_the_tcgen05_scan(lib, hq, hkv, L, T, pos0, n_split):
    """hd256 K8V4 windows whose blocks get several 128-key tiles run the tcgen05 scan with the
    4-bit V plane; junk codes and scales past kv_len stay unseen."""
    inp = workloads.random_small(1500 + hq + L + T, hq, hkv, 256, L, T, k_gain=1.5)
    gpu, orc = _pools(inp, capacity=L + 40)
    got = _run(gpu, inp.q, L, pos0, 0.0625, n_split)
    ref = oracle.attention(orc, inp.q, L, pos0, 0.0625)
    assert np.all(np.isfinite(got))
    assert rel_err(got, ref) <= VERIFY_TOL


def test_hd256_routes_agree(lib):
    """One window through the all-mma.sync kernel (the automatic plan of a short scan) and the
    tcgen05 scan (two slices): both within the tolerance of the oracle and of each other."""
    inp = workloads.random_small(1520, 24, 4, 256, 1024, 4)
    gpu, orc = _pools(inp, capacity=1100)
    a = _run(gpu, inp.q, 1024, 1020, 0.0625, 0)
    b = _run(gpu, inp.q, 1024, 1020, 0.0625, 2)
    ref = oracle.attention(orc, inp.q, 1024, 1020, 0.0625)
    assert rel_err(a, ref) <= VERIFY_TOL and rel_err(b, ref) <= VERIFY_TOL
    assert rel_err(a, b) <= VERIFY_TOL


@pytest.mark.parametrize("T", [4, 8, 12, 32])
def test_hd128_shape(lib, T):
    w = workloads.verify_workload(f"k8v4-32q8kv-hd128-ctx700-T{T}", 32, 8, 128, 700, T, seed=1350 + T)
    inp = workloads.make_inputs(w)
    gpu, orc = _pools(inp, capacity=w.kv_len + 9)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    assert rel_err(got, ref) <= VERIFY_TOL


@pytest.mark.parametrize("kv_len,q_pos0,T,hd", [(5, 1, 4, 128), (128, 120, 8, 256), (129, 125, 4, 128),
                                                (300, 0, 6, 256), (1, 0, 1, 256)])
def test_edges(lib, kv_len, q_pos0, T, hd):
    inp = workloads.random_small(1370 + kv_len + hd, 6, 2, hd, kv_len, T)
    gpu, orc = _pools(inp, capacity=kv_len + 16)
    got = _run(gpu, inp.q, kv_len, q_pos0, 0.09)
    ref = oracle.attention(orc, inp.q, kv_len, q_pos0, 0.09)
    assert rel_err(got, ref) <= VERIFY_TOL


@pytest.mark.parametrize("ctx,T", [(20676, 4), (32768, 8)])
def test_full_size_sampled(lib, ctx, T):
    w = workloads.long_verify(ctx, T)
    inp = workloads.make_inputs(w)
    gpu, orc = _pools(inp, junk=False)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    rng = np.random.default_rng(4)
    sel = [(i, int(rng.integers(w.n_q_heads))) for i in range(w.n_q)]
    sel += [(int(rng.integers(w.n_q)), h) for h in range(w.n_q_heads)]
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, sel=sel)
    assert rel_err(np.stack([got[i, h] for i, h in sel]), ref) <= VERIFY_TOL
    assert np.all(np.isfinite(got))


def test_k8v4_rejects_bad_arguments(lib):
    import ctypes

    import torch

    from speculative_verify_attention_gb300 import KVCacheK8V4
    from speculative_verify_attention_gb300.binding import (KVQ8_ERR_INVALID_ARG, KVQ8_ERR_MISALIGNED,
                                                             KVQ8_ERR_WORKSPACE, load_library)
    lib_ = load_library()
    cache = KVCacheK8V4(2, 128, 64, device="cuda")
    q = torch.zeros((4, 8, 128), device="cuda")
    out = torch.empty_like(q)
    nb = lib_.attn_verify_q8_workspace_bytes(4, 8, 128, 64, 2, 0)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")

    def call(qp=q.data_ptr(), kv_len=64, wsb=nb):
        return lib_.attn_verify_k8v4(qp, 4, 8, ctypes.byref(cache.struct()), kv_len, 60, 0.1, out.data_ptr(),
                                     ws.data_ptr(), wsb, 0, None)

    assert call() == 0
    assert call(qp=None) == KVQ8_ERR_INVALID_ARG
    assert call(kv_len=65) == KVQ8_ERR_INVALID_ARG
    assert call(qp=q.data_ptr() + 4) == KVQ8_ERR_MISALIGNED
    assert call(wsb=nb - 1) == KVQ8_ERR_WORKSPACE
    k = torch.zeros((3, 2, 128), device="cuda")
    assert lib_.kvk8v4_append(k.data_ptr(), k.data_ptr(), 3, ctypes.byref(cache.struct()), 62, None) == KVQ8_ERR_INVALID_ARG
    torch.cuda.synchronize()


def _prompt(gpu, q16, kv_len, q_pos0, scale):
    import torch

    from speculative_verify_attention_gb300 import attn_prompt_k8v4
    q = torch.from_numpy(np.ascontiguousarray(q16)).cuda()
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    attn_prompt_k8v4(q, gpu, kv_len, q_pos0, scale, out=out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("hq,hkv,hd,L,nq,pos0,capacity", [
    (12, 1, 256, 64, 11, 53, None),
    (12, 1, 256, 200, 50, 150, 203),
    (24, 2, 256, 512, 64, 448, None),
    (32, 8, 128, 333, 40, 290, 335),
    (16, 4, 128, 300, 60, 280, 301),
    (12, 1, 256, 900, 342, 558, 933),   # 33 row tiles per KV head: the two-pass route
    (32, 8, 128, 1100, 1030, 70, 1103),
])
def test_prompt_k8v4_small_shapes(lib, hq, hkv, hd, L, nq, pos0, capacity):
    from ._util import PROMPT_TOL
    inp = workloads.random_small(1400 + hq + L, hq, hkv, hd, L, nq, q_dtype="f16")
    gpu, orc = _pools(inp, capacity=capacity)
    scale = 1.0 / float(np.sqrt(hd))
    got = _prompt(gpu, inp.q, L, pos0, scale)
    ref = oracle.attention(orc, inp.q, L, pos0, scale)
    assert np.all(np.isfinite(got))
    assert rel_err(got, ref) <= PROMPT_TOL


@pytest.mark.parametrize("hq,hkv,L,nq,pos0,hd", [
    (12, 1, 900, 342, 558, 256),
    (32, 8, 1100, 1030, 70, 128),
])
def test_prompt_k8v4_two_pass_equals_the_f16_pool_of_the_dequantised_values(lib, hq, hkv, L, nq, pos0, hd):
    """On the two-pass route the operands are fp16(code x scale) for K and fp16((nibble - 8) x
    scale) for V, each rounded once: attn_prompt_f16 over a pool holding exactly those values
    (computed here with numpy; element 2m of a V row is the low nibble of byte m) gives the same
    output bit for bit."""
    import torch

    from speculative_verify_attention_gb300 import KVCacheF16, attn_prompt_f16, attn_prompt_k8v4
    inp = workloads.random_small(1700 + hq + L, hq, hkv, hd, L, nq, q_dtype="f16")
    gpu, _ = _pools(inp, junk=False)
    f16 = KVCacheF16(hkv, hd, gpu.capacity)
    kc = gpu.k_codes.cpu().numpy()[:, :L].astype(np.float16)
    ks = np.repeat(gpu.k_scales.cpu().numpy()[:, :L], 32, axis=2)
    f16.k[:, :L].copy_(torch.from_numpy(kc * ks))
    vb = gpu.v_codes.cpu().numpy()[:, :L]
    vq = np.stack([(vb & 15).astype(np.int16) - 8, (vb >> 4).astype(np.int16) - 8], axis=-1)
    vs = np.repeat(gpu.v_scales.cpu().numpy()[:, :L], 32, axis=2)
    f16.v[:, :L].copy_(torch.from_numpy(vq.reshape(hkv, L, hd).astype(np.float16) * vs))
    q = torch.from_numpy(np.ascontiguousarray(inp.q)).cuda()
    scale = 1.0 / float(np.sqrt(hd))
    a = attn_prompt_k8v4(q, gpu, L, pos0, scale)
    b = attn_prompt_f16(q, f16, L, pos0, scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_prompt_k8v4_full_workload_sampled(lib):
    from ._util import PROMPT_TOL
    from speculative_verify_attention_gb300 import kvq8_device_error
    w = workloads.PROMPT
    inp = workloads.make_inputs(w)
    gpu, orc = _pools(inp, junk=False)
    got = _prompt(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    rng = np.random.default_rng(8)
    sel = [(int(i), int(rng.integers(w.n_q_heads))) for i in rng.integers(0, w.n_q, 30)]
    sel += [(0, h) for h in range(w.n_q_heads)] + [(w.n_q - 1, h) for h in range(w.n_q_heads)]
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, sel=sel)
    assert np.all(np.isfinite(got))
    assert rel_err(np.stack([got[i, h] for i, h in sel]), ref) <= PROMPT_TOL
    assert kvq8_device_error(reset=True) == 0


def test_q4_quotients_near_half_integers_bit_exact(lib):
    """4-bit V blocks with values a few ulps around (k + 1/2) d: the append kernel's codes
    equal the oracle's IEEE-division codes."""
    import torch

    from speculative_verify_attention_gb300 import KVCacheK8V4, kvk8v4_append
    rng = np.random.default_rng(31)
    n_blk = 2048
    amax = (rng.uniform(0.5, 2.0, n_blk) * np.exp2(rng.integers(-16, 16, n_blk))).astype(np.float32)
    d = (amax / np.float32(7.0)).astype(np.float32)
    kk = rng.integers(-7, 7, (n_blk, 31)).astype(np.float32)
    base = ((kk + np.float32(0.5)) * d[:, None]).astype(np.float32)
    steps = rng.integers(-4, 5, (n_blk, 31)).astype(np.int32)
    vals = (base.view(np.int32) + np.where(base >= 0, steps, -steps)).view(np.float32)
    vals = np.clip(vals, -amax[:, None], amax[:, None])
    v = np.concatenate([amax[:, None], vals], axis=1).reshape(n_blk // 8, 1, 256)
    n_tok = v.shape[0]
    cache = KVCacheK8V4(1, 256, n_tok, device="cuda")
    kvk8v4_append(torch.from_numpy(v).cuda(), torch.from_numpy(v).cuda(), cache, 0)
    torch.cuda.synchronize()
    q4, d4 = oracle.quantize_q4(v)
    got_codes = cache.v_codes.cpu().numpy()[0]
    got_scales = cache.v_scales.cpu().numpy().view(np.uint16)[0]
    assert np.array_equal(got_scales, d4[:, 0, :])
    assert np.array_equal(got_codes, q4[:, 0, :])
