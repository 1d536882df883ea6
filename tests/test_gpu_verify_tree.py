"""attn_verify_tree_q8 on the GPU against the fp64 oracle's tree-window attention:
max|gpu - oracle| / max|oracle| <= 1e-4."""
import numpy as np
import pytest

import oracle
from speculative_verify_attention_gb300 import workloads

from ._util import VERIFY_TOL, build_caches, rel_err

pytestmark = pytest.mark.gpu


def _tree_masks(parents):
    masks = []
    for i in range(len(parents)):
        m, a = 0, i
        while a >= 0:
            m |= 1 << a
            a = parents[a]
        masks.append(m)
    return np.array(masks, dtype=np.uint32)


def _binary_tree(T):
    return _tree_masks([-1] + [(i - 1) // 2 for i in range(1, T)])


def _run(gpu_cache, q, kv_len, q_pos0, scale, mask, n_split=0):
    import torch

    from speculative_verify_attention_gb300 import attn_verify_tree_q8
    m = torch.from_numpy(np.ascontiguousarray(mask, np.uint32).view(np.int32)).cuda()
    out = attn_verify_tree_q8(torch.from_numpy(np.ascontiguousarray(q, np.float32)).cuda(), gpu_cache, kv_len,
                              q_pos0, m, scale, n_split=n_split)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("T,n_split", [(8, 0), (8, 5), (16, 0), (32, 3)])
def test_binary_tree_27b_shape(lib, T, n_split):
    w = workloads.verify_workload(f"tree-24q4kv-hd256-ctx1000-T{T}", 24, 4, 256, 1000, T, k_outliers=4, seed=900 + T)
    inp = workloads.make_inputs(w)
    gpu, orc = build_caches(inp)
    mask = _binary_tree(T)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, mask, n_split)
    ref = oracle.attention_tree(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, mask)
    assert rel_err(got, ref) <= VERIFY_TOL


def test_random_masks_hd128_and_context_free_rows(lib):
    inp = workloads.random_small(902, 8, 2, 128, 300, 12)
    gpu, orc = build_caches(inp, capacity=320)
    rng = np.random.default_rng(3)
    mask = rng.integers(0, 1 << 32, 12, dtype=np.uint64).astype(np.uint32)
    mask[0] = 0
    for q_pos0 in (288, 0):                      # q_pos0 = 0: rows see only their masked window keys
        got = _run(gpu, inp.q, 300, q_pos0, 0.08, mask)
        ref = oracle.attention_tree(orc, inp.q, 300, q_pos0, 0.08, mask)
        assert rel_err(got, ref) <= VERIFY_TOL
        if q_pos0 == 0:
            assert not got[0].any()              # row 0 sees nothing


def test_chain_mask_matches_causal_call(lib):
    """A chain mask is the sequential window: the tree kernel and the causal call (a different
    kernel, with its own rounding order) agree far inside the oracle tolerance."""
    import torch

    from speculative_verify_attention_gb300 import attn_verify_q8
    w = workloads.verify_27b(8)
    inp = workloads.make_inputs(w)
    gpu, orc = build_caches(inp, garbage_tail=False)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, oracle.chain_mask(8))
    ref = attn_verify_q8(torch.from_numpy(inp.q).cuda(), gpu, w.kv_len, w.q_pos0, w.softmax_scale)
    torch.cuda.synchronize()
    assert rel_err(got, ref.cpu().numpy()) <= 1e-5
    assert rel_err(got, oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)) <= VERIFY_TOL


def test_tree_rejects_bad_arguments(lib):
    import ctypes

    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8, load_library
    c = KVCacheQ8(1, 128, 64)
    q = torch.zeros((4, 4, 128), device="cuda")
    out = torch.empty_like(q)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    lib_ = load_library()
    st = lib_.attn_verify_tree_q8(ctypes.c_void_p(q.data_ptr()), 4, 4, ctypes.byref(c.struct()), 40, 36, None,
                                  ctypes.c_float(0.1), ctypes.c_void_p(out.data_ptr()),
                                  ctypes.c_void_p(ws.data_ptr()), ws.numel(), 0, None)
    assert st == 1                                # null window mask


@pytest.mark.parametrize("T", [8, 32])
def test_binary_tree_full_context_sampled(lib, T):
    """A binary-tree window at the long-context shape (24q/4kv/hd256, ctx 20676; the tcgen05 scan
    with the automatic plan): every row and every q head sampled against the oracle."""
    w = workloads.long_verify(20676, T)
    inp = workloads.make_inputs(w)
    gpu, orc = build_caches(inp, garbage_tail=False)
    mask = _binary_tree(T)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, mask)
    rng = np.random.default_rng(40 + T)
    sel = [(i, int(rng.integers(w.n_q_heads))) for i in range(w.n_q)]
    sel += [(int(rng.integers(w.n_q)), h) for h in range(w.n_q_heads)]
    ref = oracle.attention_tree(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, mask, sel=sel)
    assert np.all(np.isfinite(got))
    assert rel_err(np.stack([got[i, h] for i, h in sel]), ref) <= VERIFY_TOL
