"""attn_verify_q8_partials on the GPU: the per-rank kernel of a context-sharded verify.

Virtual ranks on one GPU: the context is cut into slices, each slice sits in a cache of its
own (positions relative to its first key, so q_pos0 goes negative for later slices), the
partials of every slice are concatenated and merged by attn_combine; the result must match
the fp64 oracle's attention over the whole context within 1e-4."""
import numpy as np
import pytest

import oracle
from speculative_verify_attention_gb300 import multigpu, workloads

from ._util import VERIFY_TOL, build_caches, rel_err

pytestmark = pytest.mark.gpu


def _slice_inputs(inp, b, e):
    return workloads.Inputs(k=inp.k[b:e], v=inp.v[b:e], q=inp.q)


def _sharded(inp, kv_len, q_pos0, scale, world, n_split=0, align=128):
    import torch

    from speculative_verify_attention_gb300 import attn_combine, attn_verify_q8_partials
    q = torch.from_numpy(np.ascontiguousarray(inp.q, np.float32)).cuda()
    pos, pml = [], []
    for b, e in multigpu.context_slices(kv_len, world, align):
        if e <= b:
            continue
        gpu, _ = build_caches(_slice_inputs(inp, b, e), capacity=e - b + 16)
        o, ml = attn_verify_q8_partials(q, gpu, e - b, q_pos0 - b, scale, n_split=n_split)
        pos.append(o)
        pml.append(ml)
    out = attn_combine(torch.cat(pos), torch.cat(pml))
    torch.cuda.synchronize()
    return out.cpu().numpy().reshape(inp.q.shape)


@pytest.mark.parametrize("world,n_split", [(1, 0), (2, 0), (3, 0), (4, 2), (5, 1)])
def test_27b_shape_virtual_ranks(lib, world, n_split):
    w = workloads.verify_workload("partials-24q4kv-hd256-ctx1500-T8", 24, 4, 256, 1500, 8, k_outliers=4, seed=990)
    inp = workloads.make_inputs(w)
    got = _sharded(inp, w.kv_len, w.q_pos0, w.softmax_scale, world, n_split)
    _, orc = build_caches(inp)
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    assert rel_err(got, ref) <= VERIFY_TOL


def test_hd128_window_straddles_ranks(lib):
    """Slices of 64 keys, the window (positions 250 .. 261) across the last two: rows 0-5 see
    none of the last slice's keys and get empty partials from it."""
    inp = workloads.random_small(991, 8, 2, 128, 262, 12)
    got = _sharded(inp, 262, 250, 0.088, 5, align=64)
    _, orc = build_caches(inp)
    ref = oracle.attention(orc, inp.q, 262, 250, 0.088)
    assert rel_err(got, ref) <= VERIFY_TOL


def test_rows_before_the_cache_get_empty_partials(lib):
    import torch

    from speculative_verify_attention_gb300 import attn_verify_q8_partials, attn_verify_q8_partials_count
    inp = workloads.random_small(992, 6, 2, 128, 200, 4)
    gpu, _ = build_caches(inp, capacity=208)
    n = attn_verify_q8_partials_count(4, 6, 128, 200, 2, 4)
    assert n == 4                                  # 4 slices of 64 keys (whole 16-key units)
    assert attn_verify_q8_partials_count(4, 6, 128, 200, 2, 3) == 3   # 3 asked: 80-key slices
    o, ml = attn_verify_q8_partials(torch.from_numpy(inp.q).cuda(), gpu, 200, -4, 0.1, n_split=4)
    torch.cuda.synchronize()
    assert o.shape == (4, 24, 128) and ml.shape == (4, 24, 2)
    assert torch.all(ml[..., 0] == -float("inf")) and torch.all(ml[..., 1] == 0)
    assert torch.all(o == 0)


def test_partials_match_the_merged_entry_point(lib):
    """Merging the partials of one call gives attn_verify_q8's output bit for bit (the same
    slices and the same merge)."""
    import torch

    from speculative_verify_attention_gb300 import attn_combine, attn_verify_q8, attn_verify_q8_partials
    w = workloads.verify_27b(4)
    inp = workloads.make_inputs(w)
    gpu, _ = build_caches(inp, garbage_tail=False)
    q = torch.from_numpy(inp.q).cuda()
    o, ml = attn_verify_q8_partials(q, gpu, w.kv_len, w.q_pos0, w.softmax_scale)
    merged = attn_combine(o, ml)
    ref = attn_verify_q8(q, gpu, w.kv_len, w.q_pos0, w.softmax_scale)
    torch.cuda.synchronize()
    assert torch.equal(merged.reshape(ref.shape), ref)


def test_verify_context_sharded_single_rank(lib):
    """The host function of the sharded path, one rank (no process group): equals the oracle."""
    import torch

    inp = workloads.random_small(993, 24, 4, 256, 900, 4)
    gpu, orc = build_caches(inp)
    out = multigpu.verify_context_sharded(torch.from_numpy(inp.q).cuda(), gpu, 900, 896, 0.0625)
    torch.cuda.synchronize()
    ref = oracle.attention(orc, inp.q, 900, 896, 0.0625)
    assert rel_err(out.cpu().numpy(), ref) <= VERIFY_TOL


def test_partials_reject_bad_arguments(lib):
    import ctypes

    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8
    from speculative_verify_attention_gb300.binding import KVQ8_ERR_INVALID_ARG, KVQ8_ERR_MISALIGNED, load_library
    lib_ = load_library()
    cache = KVCacheQ8(2, 128, 64, device="cuda")
    q = torch.zeros((4, 8, 128), device="cuda")
    po = torch.empty((4, 32, 128), device="cuda")
    pm = torch.empty((4, 32, 2), device="cuda")

    def call(o=po.data_ptr(), m=pm.data_ptr(), pos=10, kv_len=64):
        return lib_.attn_verify_q8_partials(q.data_ptr(), 4, 8, ctypes.byref(cache.struct()), kv_len, pos, 0.1, o, m,
                                            4, None)

    assert call() == 0
    assert call(o=None) == KVQ8_ERR_INVALID_ARG
    assert call(m=None) == KVQ8_ERR_INVALID_ARG
    assert call(kv_len=65) == KVQ8_ERR_INVALID_ARG
    assert call(pos=-(1 << 30) - 1) == KVQ8_ERR_INVALID_ARG
    assert call(o=po.data_ptr() + 4) == KVQ8_ERR_MISALIGNED
    assert lib_.attn_verify_q8_partials_count(4, 8, 128, 0, 2, 0) == 0
    torch.cuda.synchronize()


def test_kv_head_sharding_as_virtual_ranks(lib):
    """verify_kv_head_sharded over 1-3 head ranges, each with a cache of its own heads: the
    concatenated outputs match the oracle (no exchange is involved)."""
    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8, multigpu
    w = workloads.verify_27b(4)
    inp = workloads.make_inputs(w)
    g = w.group
    orc = oracle.Cache(w.n_kv_heads, w.head_dim, w.kv_len)
    orc.append(inp.k, inp.v, 0)
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    q = torch.from_numpy(inp.q).cuda()
    for world in (1, 2, 3):
        outs = []
        for r in range(world):
            h0, h1 = multigpu.kv_head_range(w.n_kv_heads, world, r)
            c = KVCacheQ8(h1 - h0, w.head_dim, w.kv_len, device="cuda")
            c.append(torch.from_numpy(np.ascontiguousarray(inp.k[:, h0:h1])).cuda(),
                     torch.from_numpy(np.ascontiguousarray(inp.v[:, h0:h1])).cuda(), 0)
            outs.append(multigpu.verify_kv_head_sharded(q, c, w.kv_len, w.q_pos0, w.softmax_scale, h0, h1, g))
        torch.cuda.synchronize()
        got = torch.cat(outs, dim=1).cpu().numpy()
        assert got.shape == ref.shape
        assert rel_err(got, ref) <= VERIFY_TOL
