"""attn_verify_f16 / kvf16_append on the GPU against the fp64 oracle's fp16 pool:
the append bit for bit, attention within 1e-4 (max|gpu - oracle| / max|oracle|)."""
import numpy as np
import pytest

import oracle
from speculative_verify_attention_gb300 import workloads

from ._util import VERIFY_TOL, rel_err

pytestmark = pytest.mark.gpu


def _pools(inp, capacity=None, pos0=0, junk=True):
    """The same fp32 K/V appended to a library fp16 pool and an oracle fp16 pool; positions
    outside the written range hold the same junk (finite) fp16 values in both."""
    import torch

    from speculative_verify_attention_gb300 import KVCacheF16
    L, hkv, hd = inp.k.shape
    cap = capacity or (pos0 + L)
    gpu = KVCacheF16(hkv, hd, cap, device="cuda")
    orc = oracle.CacheF16(hkv, hd, cap)
    if junk and cap > pos0 + L:
        rng = np.random.default_rng(4321)
        j = (rng.standard_normal((hkv, cap, hd)) * 30).astype(np.float16)
        for a in (orc.k, orc.v):
            a[:] = j.view(np.uint16)
        for t in (gpu.k, gpu.v):
            t.copy_(torch.from_numpy(j))
    gpu.append(torch.from_numpy(inp.k).cuda(), torch.from_numpy(inp.v).cuda(), pos0)
    orc.append(inp.k, inp.v, pos0)
    torch.cuda.synchronize()
    return gpu, orc


def _run(gpu, q, kv_len, q_pos0, scale, n_split=0):
    import torch

    from speculative_verify_attention_gb300 import attn_verify_f16
    out = attn_verify_f16(torch.from_numpy(np.ascontiguousarray(q, np.float32)).cuda(), gpu, kv_len, q_pos0, scale,
                          n_split=n_split)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_append_matches_oracle_bitwise(lib):
    inp = workloads.random_small(1200, 8, 2, 128, 77, 4)
    gpu, orc = _pools(inp, capacity=90, pos0=5)
    assert np.array_equal(gpu.k.cpu().numpy().view(np.uint16), orc.k)
    assert np.array_equal(gpu.v.cpu().numpy().view(np.uint16), orc.v)


@pytest.mark.parametrize("T,n_split", [(4, 0), (8, 0), (16, 0), (32, 0), (4, 3), (8, 1)])
def test_27b_shape(lib, T, n_split):
    w = workloads.verify_workload(f"f16-24q4kv-hd256-ctx1000-T{T}", 24, 4, 256, 1000, T, k_outliers=4, seed=1210 + T)
    inp = workloads.make_inputs(w)
    gpu, orc = _pools(inp, capacity=w.kv_len + 30)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, n_split)
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    assert rel_err(got, ref) <= VERIFY_TOL


@pytest.mark.parametrize("T", [4, 8, 12, 32])
def test_hd128_shape(lib, T):
    w = workloads.verify_workload(f"f16-32q8kv-hd128-ctx700-T{T}", 32, 8, 128, 700, T, seed=1250 + T)
    inp = workloads.make_inputs(w)
    gpu, orc = _pools(inp, capacity=w.kv_len + 9)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    assert rel_err(got, ref) <= VERIFY_TOL


@pytest.mark.parametrize("kv_len,q_pos0,T", [(5, 1, 4), (128, 120, 8), (129, 125, 4), (300, 0, 6), (1, 0, 1)])
def test_edges(lib, kv_len, q_pos0, T):
    """Contexts shorter than a tile, ending on and past a tile edge, q_pos0 = 0 and a single row."""
    inp = workloads.random_small(1270 + kv_len, 6, 2, 128, kv_len, T)
    gpu, orc = _pools(inp, capacity=kv_len + 16)
    got = _run(gpu, inp.q, kv_len, q_pos0, 0.09)
    ref = oracle.attention(orc, inp.q, kv_len, q_pos0, 0.09)
    assert rel_err(got, ref) <= VERIFY_TOL


def test_full_size_sampled(lib):
    """The ctx 20,676 T = 8 long-context cell, sampled (row, head) outputs against the oracle."""
    w = workloads.long_verify(20676, 8)
    inp = workloads.make_inputs(w)
    gpu, orc = _pools(inp, junk=False)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    rng = np.random.default_rng(3)
    sel = [(i, int(rng.integers(w.n_q_heads))) for i in range(w.n_q)]
    sel += [(int(rng.integers(w.n_q)), h) for h in range(w.n_q_heads)]
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, sel=sel)
    assert rel_err(np.stack([got[i, h] for i, h in sel]), ref) <= VERIFY_TOL
    assert np.all(np.isfinite(got))


def test_f16_rejects_bad_arguments(lib):
    import ctypes

    import torch

    from speculative_verify_attention_gb300 import KVCacheF16
    from speculative_verify_attention_gb300.binding import (KVQ8_ERR_INVALID_ARG, KVQ8_ERR_MISALIGNED,
                                                             KVQ8_ERR_UNSUPPORTED, KVQ8_ERR_WORKSPACE, load_library)
    lib_ = load_library()
    cache = KVCacheF16(2, 128, 64, device="cuda")
    q = torch.zeros((4, 8, 128), device="cuda")
    out = torch.empty_like(q)
    nb = lib_.attn_verify_f16_workspace_bytes(4, 8, 128, 64, 2, 0)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")

    def call(qp=q.data_ptr(), kv_len=64, pos=60, wsb=nb, hq=8):
        return lib_.attn_verify_f16(qp, 4, hq, ctypes.byref(cache.struct()), kv_len, pos, 0.1, out.data_ptr(),
                                    ws.data_ptr(), wsb, 0, None)

    assert call() == 0
    assert call(qp=None) == KVQ8_ERR_INVALID_ARG
    assert call(kv_len=65) == KVQ8_ERR_INVALID_ARG
    assert call(pos=-1) == KVQ8_ERR_INVALID_ARG
    assert call(hq=7) == KVQ8_ERR_UNSUPPORTED
    assert call(qp=q.data_ptr() + 4) == KVQ8_ERR_MISALIGNED
    assert call(wsb=nb - 1) == KVQ8_ERR_WORKSPACE
    k = torch.zeros((3, 2, 128), device="cuda")
    assert lib_.kvf16_append(k.data_ptr(), k.data_ptr(), 3, ctypes.byref(cache.struct()), 62, None) == KVQ8_ERR_INVALID_ARG
    assert lib_.kvf16_append(k.data_ptr() + 4, k.data_ptr(), 3, ctypes.byref(cache.struct()), 0, None) == KVQ8_ERR_MISALIGNED
    torch.cuda.synchronize()


def _prompt_f16(gpu, q16, kv_len, q_pos0, scale):
    import torch

    from speculative_verify_attention_gb300 import attn_prompt_f16
    q = torch.from_numpy(np.ascontiguousarray(q16)).cuda()
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    attn_prompt_f16(q, gpu, kv_len, q_pos0, scale, out=out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("hq,hkv,hd,L,nq,pos0,capacity", [
    (12, 1, 256, 64, 11, 53, None),
    (12, 1, 256, 200, 50, 150, 203),     # ragged last tile
    (24, 2, 256, 512, 64, 448, None),
    (32, 8, 128, 333, 40, 290, 335),
    (16, 4, 128, 300, 60, 280, 301),     # rows past kv_len
    (12, 1, 256, 1, 1, 0, 9),            # a single key
])
def test_prompt_f16_small_shapes(lib, hq, hkv, hd, L, nq, pos0, capacity):
    """Positions past kv_len hold NaN: the tensor copies are bounded by kv_len, so those keys
    arrive as zeros and never reach the output."""
    import torch

    from ._util import PROMPT_TOL
    inp = workloads.random_small(1500 + hq + L, hq, hkv, hd, L, nq, q_dtype="f16")
    gpu, orc = _pools(inp, capacity=capacity, junk=False)
    if capacity and capacity > L:
        gpu.k[:, L:] = float("nan")
        gpu.v[:, L:] = float("nan")
        torch.cuda.synchronize()
    scale = 1.0 / float(np.sqrt(hd))
    got = _prompt_f16(gpu, inp.q, L, pos0, scale)
    ref = oracle.attention(orc, inp.q, L, pos0, scale)
    assert np.all(np.isfinite(got))
    assert rel_err(got, ref) <= PROMPT_TOL


def test_prompt_f16_full_workload_sampled(lib):
    from speculative_verify_attention_gb300 import kvq8_device_error

    from ._util import PROMPT_TOL
    w = workloads.PROMPT
    inp = workloads.make_inputs(w)
    gpu, orc = _pools(inp, junk=False)
    got = _prompt_f16(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    rng = np.random.default_rng(9)
    sel = [(int(i), int(rng.integers(w.n_q_heads))) for i in rng.integers(0, w.n_q, 30)]
    sel += [(0, h) for h in range(w.n_q_heads)] + [(w.n_q - 1, h) for h in range(w.n_q_heads)]
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, sel=sel)
    assert np.all(np.isfinite(got))
    assert rel_err(np.stack([got[i, h] for i, h in sel]), ref) <= PROMPT_TOL
    assert kvq8_device_error(reset=True) == 0
