"""The tcgen05 verify scan on edge shapes, against the fp64 oracle (max|gpu - oracle| /
max|oracle| <= 1e-4).  Causal and tree-shaped windows over a Q8_0 cache run the tcgen05 kernel
when each block gets at least two 128-key tiles and (hd256, or more than 32 rows per KV head);
the explicit split counts below give every block several tiles at moderate context lengths, so
each case runs that kernel: row chunks of 8, 16 and 24 rows (T = 1 .. 32, group 1 .. 16), ragged
last tiles, rows past kv_len, kv_len beyond the window, junk bytes past kv_len in the cache, and
tree windows from random ancestor masks."""
import numpy as np
import pytest

import oracle
from speculative_verify_attention_gb300 import workloads

from ._util import VERIFY_TOL, build_caches, rel_err

pytestmark = pytest.mark.gpu


def _run(gpu_cache, q, kv_len, q_pos0, scale, n_split):
    import torch

    from speculative_verify_attention_gb300 import attn_verify_q8
    out = attn_verify_q8(torch.from_numpy(np.ascontiguousarray(q, np.float32)).cuda(), gpu_cache, kv_len, q_pos0,
                         scale, n_split=n_split)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("hq,hkv,hd,L,T,pos0,n_split", [
    (6, 1, 256, 3001, 1, 3000, 3),     # T = 1: one 8-row chunk of 6 rows, ragged last tile
    (6, 1, 256, 2500, 3, 2497, 4),     # 18 rows: one 24-row chunk
    (12, 2, 256, 4000, 2, 3998, 3),    # 12 rows per KV head: a 16-row chunk
    (16, 1, 256, 3333, 2, 3331, 2),    # group 16: 32 rows in two 16-row chunks
    (8, 8, 256, 2000, 4, 1996, 2),     # MHA (group 1), eight KV heads, 4 rows each
    (24, 4, 256, 2600, 32, 2568, 2),   # T = 32: 192 rows per KV head in eight 24-row chunks
    (32, 8, 128, 3000, 16, 2984, 3),   # hd128 with 64 rows per KV head
    (4, 1, 256, 1500, 6, 1600, 2),     # rows past kv_len see kv_len keys
    (4, 1, 256, 3000, 4, 2000, 3),     # kv_len beyond the window: row i sees keys <= q_pos0 + i
    (24, 4, 256, 2055, 8, 2047, 5),    # 2055 keys: slices end mid-tile, chunks of 24 rows x 2
])
def test_edge_shapes_on_the_tcgen05_scan(lib, hq, hkv, hd, L, T, pos0, n_split):
    inp = workloads.random_small(hq * 1000 + L + T, hq, hkv, hd, L, T, k_gain=1.5)
    gpu, orc = build_caches(inp, capacity=L + 40)
    scale = 1.0 / np.sqrt(hd)
    got = _run(gpu, inp.q, L, pos0, scale, n_split)
    ref = oracle.attention(orc, inp.q, L, pos0, scale)
    assert np.all(np.isfinite(got))
    assert rel_err(got, ref) <= VERIFY_TOL


def test_both_kernels_agree_on_one_window(lib):
    """The same window through both routes -- the automatic plan (a short scan: the all-mma.sync
    kernel) and an explicit two-slice plan (the tcgen05 kernel) -- agrees with the oracle and
    with each other within the tolerance."""
    inp = workloads.random_small(777, 24, 4, 256, 1024, 4)
    gpu, orc = build_caches(inp)
    scale = 1.0 / 16.0
    a = _run(gpu, inp.q, 1024, 1020, scale, 0)
    b = _run(gpu, inp.q, 1024, 1020, scale, 2)
    ref = oracle.attention(orc, inp.q, 1024, 1020, scale)
    assert rel_err(a, ref) <= VERIFY_TOL
    assert rel_err(b, ref) <= VERIFY_TOL
    assert rel_err(a, b) <= VERIFY_TOL


def _run_tree(gpu_cache, q, kv_len, q_pos0, scale, mask, n_split):
    import torch

    from speculative_verify_attention_gb300 import attn_verify_tree_q8
    m = torch.from_numpy(np.ascontiguousarray(mask, np.uint32).view(np.int32)).cuda()
    out = attn_verify_tree_q8(torch.from_numpy(np.ascontiguousarray(q, np.float32)).cuda(), gpu_cache, kv_len,
                              q_pos0, m, scale, n_split=n_split)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("hq,hkv,hd,L,T,pos0,n_split,seed", [
    (24, 4, 256, 3000, 8, 2992, 3, 1),     # binary-tree-sized window, two 24-row chunks
    (24, 4, 256, 2500, 16, 2484, 2, 2),    # T = 16: four chunks
    (12, 1, 256, 2000, 3, 1990, 2, 3),     # window keys past kv_len (q_pos0 + j >= kv_len) are unseen
    (32, 8, 128, 3000, 16, 2984, 3, 4),    # hd128 with 64 rows per KV head
    (8, 2, 256, 1200, 12, 0, 2, 5),        # q_pos0 = 0: rows see only the window keys their masks pick
])
def test_tree_windows_on_the_tcgen05_scan(lib, hq, hkv, hd, L, T, pos0, n_split, seed):
    """Random ancestor masks (a row with no bit set sees only the keys before the window; bits
    past T or past kv_len select nothing) against the oracle's tree attention."""
    inp = workloads.random_small(4000 + seed, hq, hkv, hd, L, T)
    gpu, orc = build_caches(inp, capacity=L + 40)
    rng = np.random.default_rng(seed)
    mask = rng.integers(0, 1 << 32, T, dtype=np.uint64).astype(np.uint32)
    mask[0] = 0
    scale = 1.0 / np.sqrt(hd)
    got = _run_tree(gpu, inp.q, L, pos0, scale, mask, n_split)
    ref = oracle.attention_tree(orc, inp.q, L, pos0, scale, mask)
    assert np.all(np.isfinite(got))
    assert rel_err(got, ref) <= VERIFY_TOL


def test_chain_mask_tree_call_matches_the_causal_call_on_the_tcgen05_scan(lib):
    """A chain mask (row i sees window keys 0..i) is the causal window: both calls agree."""
    inp = workloads.random_small(4100, 24, 4, 256, 3000, 8)
    gpu, orc = build_caches(inp)
    mask = np.array([(1 << (i + 1)) - 1 for i in range(8)], dtype=np.uint32)
    a = _run_tree(gpu, inp.q, 3000, 2992, 1.0 / 16.0, mask, 3)
    b = _run(gpu, inp.q, 3000, 2992, 1.0 / 16.0, 3)
    ref = oracle.attention(orc, inp.q, 3000, 2992, 1.0 / 16.0)
    assert rel_err(a, ref) <= VERIFY_TOL
    assert rel_err(a, b) <= VERIFY_TOL
