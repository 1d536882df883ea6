"""attn_prompt_q8 (tcgen05) against the fp64 oracle: max|gpu - oracle| / max|oracle| <= 2e-3."""
import numpy as np
import pytest

import oracle
from speculative_verify_attention_gb300 import workloads

from ._util import PROMPT_TOL, build_caches, rel_err, report_err

pytestmark = pytest.mark.gpu


def _run(gpu_cache, q16, kv_len, q_pos0, scale):
    import torch

    from speculative_verify_attention_gb300 import attn_prompt_q8
    q = torch.from_numpy(np.ascontiguousarray(q16)).cuda()
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    attn_prompt_q8(q, gpu_cache, kv_len, q_pos0, scale, out=out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _check(hq, hkv, L, nq, pos0, seed, capacity=None, sel_every=None, hd=256):
    inp = workloads.random_small(seed, hq, hkv, hd, L, nq, q_dtype="f16")
    gpu, orc = build_caches(inp, capacity=capacity)
    scale = 1.0 / float(np.sqrt(hd))
    got = _run(gpu, inp.q, L, pos0, scale)
    if sel_every is None:
        ref = oracle.attention(orc, inp.q, L, pos0, scale)
        err = rel_err(got, ref)
    else:
        rng = np.random.default_rng(seed)
        sel = [(i, int(rng.integers(hq))) for i in range(0, nq, sel_every)]
        sel += [(nq - 1, h) for h in range(hq)]
        ref = oracle.attention(orc, inp.q, L, pos0, scale, sel=sel)
        err = rel_err(np.stack([got[i, h] for i, h in sel]), ref)
    assert np.all(np.isfinite(got)), "non-finite output"
    assert err <= PROMPT_TOL, f"rel err {err:.3e}"
    return err


@pytest.mark.parametrize("hq,hkv,L,nq,pos0", [
    (12, 1, 64, 11, 53),       # one tile, 132 rows over two CTAs
    (12, 1, 200, 50, 150),     # ragged last tile
    (12, 1, 1, 1, 0),          # a single key
    (4, 1, 333, 40, 290),      # group 4, rows crossing tiles
    (2, 2, 130, 130, 0),       # MHA, pure causal from position 0
    (24, 2, 512, 64, 448),     # two KV heads
    (12, 1, 300, 60, 280),     # rows past kv_len see kv_len keys
])
def test_small_shapes(lib, hq, hkv, L, nq, pos0):
    _check(hq, hkv, L, nq, pos0, seed=hq * 100 + L)


@pytest.mark.parametrize("hq,hkv,L,nq,pos0,capacity", [
    (12, 1, 64, 11, 53, None),      # one tile
    (12, 1, 200, 50, 150, 203),     # ragged last tile (odd key count), odd capacity
    (4, 1, 1, 1, 0, 7),             # a single key, odd capacity
    (32, 8, 333, 40, 290, 335),     # the 32q/8kv hd128 shape, rows crossing tiles, odd capacity
    (8, 8, 130, 130, 0, None),      # MHA from position 0
    (16, 4, 300, 60, 280, 301),     # rows past kv_len
])
def test_hd128_shapes(lib, hq, hkv, L, nq, pos0, capacity):
    """hd128: a key's scales are 8 bytes, so odd capacities and odd key counts put tiles on
    8-byte boundaries (the dequantisers read those scales from global memory)."""
    _check(hq, hkv, L, nq, pos0, seed=hq * 100 + L + 7, capacity=capacity, hd=128)


def test_hd128_medium_chunk(lib):
    _check(32, 8, 2048, 256, 1792, seed=79, sel_every=5, hd=128)


def test_capacity_larger_than_kv_len(lib):
    _check(12, 1, 700, 100, 600, seed=77, capacity=2048)


def test_medium_chunk(lib):
    _check(12, 1, 4096, 512, 3584, seed=78, sel_every=3)


def test_full_prompt_workload_sampled(lib):
    import torch

    w = workloads.PROMPT
    inp = workloads.make_inputs(w)
    gpu, orc = build_caches(inp, garbage_tail=False)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    rng = np.random.default_rng(5)
    sel = [(int(i), int(rng.integers(w.n_q_heads))) for i in rng.integers(0, w.n_q, 40)]
    sel += [(0, h) for h in range(w.n_q_heads)] + [(w.n_q - 1, h) for h in range(w.n_q_heads)]
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, sel=sel)
    err = report_err(w.name, np.stack([got[i, h] for i, h in sel]), ref)
    assert np.all(np.isfinite(got))
    assert err <= PROMPT_TOL, f"rel err {err:.3e}"
    from speculative_verify_attention_gb300 import kvq8_device_error
    assert kvq8_device_error(reset=True) == 0
    del torch


def test_prompt_rejects_bad_arguments(lib):
    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8, KVQ8Error, attn_prompt_q8
    q = torch.zeros((4, 12, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(KVQ8Error) as e:       # head_dim 64 has no prompt kernel
        attn_prompt_q8(torch.zeros((4, 4, 64), dtype=torch.float16, device="cuda"), KVCacheQ8(1, 64, 64), 64, 60,
                       0.1)
    assert e.value.status == 2
    with pytest.raises(KVQ8Error) as e:       # kv_len beyond capacity
        attn_prompt_q8(q, KVCacheQ8(1, 256, 64), 65, 61, 0.1)
    assert e.value.status == 1
    with pytest.raises(KVQ8Error) as e:       # 12 q heads over 5 kv heads
        attn_prompt_q8(q, KVCacheQ8(5, 256, 64), 64, 60, 0.1)
    assert e.value.status == 2


def test_full_hd128_prompt_workload_sampled(lib):
    w = workloads.PROMPT_HD128
    inp = workloads.make_inputs(w)
    gpu, orc = build_caches(inp, garbage_tail=False)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    rng = np.random.default_rng(6)
    sel = [(int(i), int(rng.integers(w.n_q_heads))) for i in rng.integers(0, w.n_q, 40)]
    sel += [(0, h) for h in range(w.n_q_heads)] + [(w.n_q - 1, h) for h in range(w.n_q_heads)]
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, sel=sel)
    err = report_err(w.name, np.stack([got[i, h] for i, h in sel]), ref)
    assert np.all(np.isfinite(got))
    assert err <= PROMPT_TOL, f"rel err {err:.3e}"
    from speculative_verify_attention_gb300 import kvq8_device_error
    assert kvq8_device_error(reset=True) == 0


def test_prompt_rows_sharded_as_virtual_ranks(lib):
    """prompt_rows_sharded over 3 row ranges of a 512-row chunk: the concatenated rows match the
    oracle (sampled) and the unsharded call."""
    import torch

    from speculative_verify_attention_gb300 import attn_prompt_q8, multigpu
    hq, hkv, L, nq = 12, 1, 2048, 512
    inp = workloads.random_small(90, hq, hkv, 256, L, nq, q_dtype="f16")
    gpu, orc = build_caches(inp)
    scale = 1.0 / 16.0
    q = torch.from_numpy(np.ascontiguousarray(inp.q)).cuda()
    parts = [multigpu.prompt_rows_sharded(q, gpu, L, L - nq, scale, *multigpu.prompt_row_range(nq, 3, r))
             for r in range(3)]
    full = attn_prompt_q8(q, gpu, L, L - nq, scale)
    torch.cuda.synchronize()
    got = torch.cat(parts, dim=0).cpu().numpy()
    assert rel_err(got, full.cpu().numpy()) <= PROMPT_TOL
    rng = np.random.default_rng(91)
    sel = [(int(i), int(rng.integers(hq))) for i in rng.integers(0, nq, 40)] + [(nq - 1, h) for h in range(hq)]
    ref = oracle.attention(orc, inp.q, L, L - nq, scale, sel=sel)
    assert rel_err(np.stack([got[i, h] for i, h in sel]), ref) <= PROMPT_TOL


@pytest.mark.parametrize("hq,hkv,L,nq,pos0,capacity,hd", [
    (12, 1, 900, 342, 558, 933, 256),   # 33 row tiles per KV head (the last one 8 rows), odd capacity
    (12, 1, 1100, 342, 500, 1200, 256), # the copy stops at q_pos0 + n_q = 842, short of kv_len
    (12, 1, 500, 360, 300, None, 256),  # rows past kv_len see all 500 keys
    (24, 2, 900, 360, 540, None, 256),  # two KV heads, each its own plane in the copy
    (32, 8, 1100, 1030, 70, 1103, 128), # hd128, 33 row tiles per KV head, odd capacity
])
def test_two_pass_route(lib, hq, hkv, L, nq, pos0, capacity, hd):
    """Chunks of 24 or more 128-row tiles per KV head take the two-pass route (the planes
    dequantised into the workspace, then the tensor-copy kernel over that fp16 copy)."""
    _check(hq, hkv, L, nq, pos0, seed=hq * 100 + L + 11, capacity=capacity, hd=hd,
           sel_every=None if hd == 256 else 3)


@pytest.mark.parametrize("hq,hkv,L,nq,pos0,hd", [
    (12, 1, 900, 342, 558, 256),
    (32, 8, 1100, 1030, 70, 128),
])
def test_two_pass_equals_the_f16_pool_of_the_dequantised_values(lib, hq, hkv, L, nq, pos0, hd):
    """The two-pass route's operands are fp16(code x scale), rounded once: attn_prompt_f16 over
    a pool holding exactly those values (computed here with numpy from the cache's codes and
    scales) gives the same output bit for bit."""
    import torch

    from speculative_verify_attention_gb300 import KVCacheF16, attn_prompt_f16, attn_prompt_q8
    inp = workloads.random_small(hq * 10 + L, hq, hkv, hd, L, nq, q_dtype="f16")
    gpu, _ = build_caches(inp)
    f16 = KVCacheF16(hkv, hd, gpu.capacity)
    for codes, scales, dst in ((gpu.k_codes, gpu.k_scales, f16.k), (gpu.v_codes, gpu.v_scales, f16.v)):
        c = codes.cpu().numpy()[:, :L].astype(np.float16)
        s = np.repeat(scales.cpu().numpy()[:, :L], 32, axis=2)
        dst[:, :L].copy_(torch.from_numpy(c * s))   # numpy rounds the exact product once to fp16
    q = torch.from_numpy(np.ascontiguousarray(inp.q)).cuda()
    scale = 1.0 / float(np.sqrt(hd))
    a = attn_prompt_q8(q, gpu, L, pos0, scale)
    b = attn_prompt_f16(q, f16, L, pos0, scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
