"""The N > 1 host path on CPU: two gloo ranks.

* max_over_ranks / barrier behave as the benchmark's timing reduction needs.
* Context-slice sharding: each rank computes the partials of its key range (with the fp64
  oracle standing in for the per-rank kernel), combine_sharded pads them to a common count,
  all-gathers them, and the log-sum-exp merge equals unsharded attention."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from speculative_verify_attention_gb300 import multigpu


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist

    import oracle
    from speculative_verify_attention_gb300 import workloads

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # timing reduction
        m = multigpu.max_over_ranks(float(rank + 1))
        multigpu.barrier()
        # context-slice sharding of one verify problem: rank r's partials of its key range
        # (the oracle standing in for the per-rank kernel; rank 0 cuts its range in two, so
        # the counts differ and combine_sharded pads), then the exchange and the merge
        inp = workloads.random_small(77, 6, 2, 128, 700, 4)
        c = oracle.Cache(2, 128, 700)
        c.append(inp.k, inp.v, 0)
        b, e = multigpu.context_slices(700, world, align=128)[rank]
        cuts = [b, (b + e) // 2, e] if rank == 0 else [b, e]
        parts = [oracle.attention_partial(c, inp.q, 700, 696, 0.09, x, y) for x, y in zip(cuts[:-1], cuts[1:])]
        part_o = torch.from_numpy(np.stack([p[0].reshape(-1, 128) for p in parts]))
        part_ml = torch.from_numpy(np.stack([np.stack([p[1].reshape(-1), p[2].reshape(-1)], axis=-1)
                                             for p in parts]))
        shapes = []

        def merge(go, gml):
            shapes.append(tuple(go.shape))
            return oracle.combine(go.numpy(), gml[..., 0].numpy(), gml[..., 1].numpy())

        out = multigpu.combine_sharded(part_o, part_ml, merge)
        ref = oracle.attention(c, inp.q, 700, 696, 0.09).reshape(-1, 128)
        results[rank] = (m, float(np.max(np.abs(out - ref))), shapes[0])
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_merge_context_slices():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=240)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        for r in range(world):
            m, err, shape = results[r]
            assert m == 2.0
            assert err < 1e-12
            assert shape == (4, 24, 128)   # 2 ranks x 2 partials (rank 1 padded with an empty one)


def _head_worker(rank, world, port, results):
    import torch.distributed as dist

    import oracle
    from speculative_verify_attention_gb300 import workloads

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # KV-head sharding of one verify problem with 3 KV heads over 2 ranks (2 + 1 heads):
        # each rank attends with its own heads' cache (the oracle standing in for the kernel),
        # nothing is exchanged until the outputs are gathered for the comparison
        group, hkv, hd, L, T = 2, 3, 128, 300, 4
        inp = workloads.random_small(81, hkv * group, hkv, hd, L, T)
        h0, h1 = multigpu.kv_head_range(hkv, world, rank)
        c = oracle.Cache(h1 - h0, hd, L)
        c.append(np.ascontiguousarray(inp.k[:, h0:h1]), np.ascontiguousarray(inp.v[:, h0:h1]), 0)
        out_local = oracle.attention(c, np.ascontiguousarray(inp.q[:, h0 * group:h1 * group]), L, L - T, 0.09)
        full = multigpu.gather_head_outputs(torch.from_numpy(out_local), hkv, group)
        cf = oracle.Cache(hkv, hd, L)
        cf.append(inp.k, inp.v, 0)
        ref = oracle.attention(cf, inp.q, L, L - T, 0.09)
        results[rank] = (h1 - h0, tuple(full.shape), float(np.max(np.abs(full.numpy() - ref))))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_kv_heads_without_exchange():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_head_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=240)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        assert results[0][0] == 2 and results[1][0] == 1
        for r in range(world):
            assert results[r][1] == (4, 6, 128)
            assert results[r][2] == 0.0   # per-head attention is independent: bit-identical


def test_prompt_row_ranges_match_the_unsharded_rows():
    """Prompt rows cut across 3 ranks: each range, placed at q_pos0 + r0, gives the same rows as
    the unsharded chunk (the oracle standing in for the per-rank kernel)."""
    import oracle
    from speculative_verify_attention_gb300 import workloads
    hq, hkv, hd, L, nq = 4, 1, 128, 260, 37
    inp = workloads.random_small(83, hq, hkv, hd, L, nq, q_dtype="f16")
    c = oracle.Cache(hkv, hd, L)
    c.append(inp.k, inp.v, 0)
    ref = oracle.attention(c, inp.q, L, L - nq, 0.09)
    parts = []
    for r in range(3):
        r0, r1 = multigpu.prompt_row_range(nq, 3, r)
        parts.append(oracle.attention(c, np.ascontiguousarray(inp.q[r0:r1]), L, L - nq + r0, 0.09))
    assert np.array_equal(np.concatenate(parts, axis=0), ref)


def test_kv_head_ranges_partition_the_heads():
    for n, world in ((4, 2), (3, 2), (8, 8), (2, 4), (5, 3), (0, 2)):
        rs = [multigpu.kv_head_range(n, world, r) for r in range(world)]
        assert rs[0][0] == 0 and rs[-1][1] == n
        for (a0, a1), (b0, _) in zip(rs[:-1], rs[1:]):
            assert a1 == b0 and a0 <= a1
        assert max(h1 - h0 for h0, h1 in rs) - min(h1 - h0 for h0, h1 in rs) <= 1
    with pytest.raises(ValueError):
        multigpu.kv_head_range(4, 2, 2)


def test_context_slices_cover_the_context_in_whole_tiles():
    for kv_len, world in ((700, 2), (4100, 8), (100, 4), (0, 3), (129, 2)):
        sl = multigpu.context_slices(kv_len, world)
        assert len(sl) == world and sl[0][0] == 0 and sl[-1][1] == kv_len
        for (b0, e0), (b1, _) in zip(sl[:-1], sl[1:]):
            assert e0 == b1 and b0 <= e0
            assert b0 % 128 == 0 or b0 == kv_len
    with pytest.raises(ValueError):
        multigpu.context_slices(10, 0)


def test_single_process_helpers_are_identities():
    assert multigpu.max_over_ranks(3.5) == 3.5
    o, m = torch.zeros(1, 2, 4), torch.zeros(1, 2, 2)
    assert multigpu.allgather_partials(o, m)[0] is o
