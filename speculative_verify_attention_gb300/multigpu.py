"""Host-side helpers for running the attention path on several GPUs of one node.

Two ways to use N GPUs, both built from the single-GPU entry points:

* replicas -- every rank runs its own independent verify / prompt problems (different
  sequences); no data crosses ranks, only the benchmark's timing reduction does.
* KV heads -- each rank owns a contiguous range of KV heads (and the q heads of their
  groups) in a cache of its own and computes their outputs with no exchange at all; only a
  caller that wants every head on every rank gathers the outputs afterwards.
* prompt rows -- a prompt chunk's query rows are cut into N contiguous ranges; a rank runs
  the prompt kernel on its rows (their positions shift with the range) against the whole
  context, with no exchange.
* context slices -- one long context is cut into N contiguous key ranges, each rank
  computes the unnormalised partials (o, m, l) of its range, the partials are all-gathered,
  and the log-sum-exp merge (attn_combine) produces the output.  This is the one real
  exchange step the path has ("perf(gfx1100): share Q8 KV scans across verifier rows",
  Summary: split-context partials and their reducer).

Everything here is plain torch.distributed (NCCL between GPUs, gloo on CPU); the tests run
the context-slice exchange with two gloo ranks, and the per-rank kernel
(attn_verify_q8_partials) as virtual ranks on one GPU.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def env_world() -> tuple[int, int, int]:
    """(world_size, rank, local_rank) from the torchrun environment (1, 0, 0 without it)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def barrier() -> None:
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a scalar over all ranks (the value itself when not distributed)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def kv_head_range(n_kv_heads: int, world: int, rank: int) -> tuple[int, int]:
    """KV heads [h0, h1) of `rank`: contiguous ranges as equal as possible (the first
    n_kv_heads % world ranks hold one more; ranks past n_kv_heads hold none)."""
    if n_kv_heads < 0 or world < 1 or not 0 <= rank < world:
        raise ValueError("bad head-range arguments")
    base, extra = divmod(n_kv_heads, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def verify_kv_head_sharded(q: torch.Tensor, cache, kv_len: int, q_pos0: int, softmax_scale: float,
                           h0: int, h1: int, group: int, n_split: int = 0) -> torch.Tensor:
    """Verify attention for KV heads [h0, h1): `cache` holds exactly those heads, `q` is the
    full window [T][Hq][hd] (q head h belongs to KV head h // group).  Returns this rank's
    output [T][(h1 - h0) * group][hd]; nothing crosses ranks."""
    from .binding import attn_verify_q8
    q_local = q[:, h0 * group:h1 * group].contiguous()
    return attn_verify_q8(q_local, cache, kv_len, q_pos0, softmax_scale, n_split=n_split)


def gather_head_outputs(out_local: torch.Tensor, n_kv_heads: int, group: int) -> torch.Tensor:
    """Every rank's [T][heads_r * group][hd] output gathered into [T][n_kv_heads * group][hd] in
    head order (ranks with fewer heads are padded for the all_gather, then trimmed)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return out_local
    w = dist.get_world_size()
    ranges = [kv_head_range(n_kv_heads, w, r) for r in range(w)]
    width = max(h1 - h0 for h0, h1 in ranges) * group
    T, n_loc, hd = out_local.shape
    padded = torch.zeros((T, width, hd), dtype=out_local.dtype, device=out_local.device)
    padded[:, :n_loc] = out_local
    parts = [torch.empty_like(padded) for _ in range(w)]
    dist.all_gather(parts, padded)
    return torch.cat([parts[r][:, :(h1 - h0) * group] for r, (h0, h1) in enumerate(ranges)], dim=1)


def prompt_row_range(n_q: int, world: int, rank: int) -> tuple[int, int]:
    """Query rows [r0, r1) of `rank` for a prompt chunk: contiguous and as equal as possible."""
    return kv_head_range(n_q, world, rank)


def prompt_rows_sharded(q: torch.Tensor, cache, kv_len: int, q_pos0: int, softmax_scale: float, r0: int,
                        r1: int) -> torch.Tensor:
    """Prompt attention for rows [r0, r1) of the chunk q [n_q][Hq][hd] (row i at position
    q_pos0 + i): the rank's rows sit at q_pos0 + r0 onwards and see keys up to their own
    positions, so the result equals rows r0..r1-1 of the unsharded call."""
    from .binding import attn_prompt_q8
    return attn_prompt_q8(q[r0:r1].contiguous(), cache, kv_len, q_pos0 + r0, softmax_scale)


def context_slices(kv_len: int, world: int, align: int = 128) -> list[tuple[int, int]]:
    """Cut keys [0, kv_len) into `world` contiguous ranges of whole `align`-key tiles
    (the last ranges may be empty when there are fewer tiles than ranks)."""
    if kv_len < 0 or world < 1 or align < 1:
        raise ValueError("bad slice arguments")
    tiles = (kv_len + align - 1) // align
    per = (tiles + world - 1) // world
    out = []
    for r in range(world):
        b = min(kv_len, r * per * align)
        e = min(kv_len, (r + 1) * per * align)
        out.append((b, e))
    return out


def allgather_partials(part_o: torch.Tensor, part_ml: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """Gather every rank's partials: part_o [n][rows][hd], part_ml [n][rows][2] ->
    ([world * n][rows][hd], [world * n][rows][2]) in rank order, ready for attn_combine."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return part_o, part_ml
    w = dist.get_world_size()
    os_ = [torch.empty_like(part_o) for _ in range(w)]
    ms_ = [torch.empty_like(part_ml) for _ in range(w)]
    dist.all_gather(os_, part_o.contiguous())
    dist.all_gather(ms_, part_ml.contiguous())
    return torch.cat(os_, dim=0), torch.cat(ms_, dim=0)


def empty_partials(n: int, rows: int, head_dim: int, device=None) -> tuple[torch.Tensor, torch.Tensor]:
    """n partials that hold no key (o = 0, m = -inf, l = 0): the merge skips them."""
    po = torch.zeros((n, rows, head_dim), dtype=torch.float32, device=device)
    pml = torch.zeros((n, rows, 2), dtype=torch.float32, device=device)
    pml[..., 0] = -float("inf")
    return po, pml


def combine_sharded(part_o: torch.Tensor, part_ml: torch.Tensor, combine) -> torch.Tensor:
    """The exchange step of a context-sharded verify: pad this rank's partials to the largest
    count over the ranks with empty ones (all_gather wants equal shapes), gather them all and
    merge with `combine(part_o, part_ml) -> out [rows][hd]` (attn_combine on GPUs)."""
    n = part_o.shape[0]
    dist_on = dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1
    if dist_on:
        t = torch.tensor([n], dtype=torch.int64, device=part_o.device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        n_max = int(t.item())
        if n_max > n:
            eo, eml = empty_partials(n_max - n, part_o.shape[1], part_o.shape[2], part_o.device)
            part_o = torch.cat([part_o, eo], dim=0)
            part_ml = torch.cat([part_ml, eml], dim=0)
    go, gml = allgather_partials(part_o, part_ml)
    return combine(go, gml)


def verify_context_sharded(q: torch.Tensor, cache, kv_len: int, q_pos0: int, softmax_scale: float,
                           n_split: int = 0) -> torch.Tensor:
    """Verify attention with the context cut across ranks.  `cache` holds this rank's keys
    (positions [0, kv_len) of it are global keys [first, first + kv_len)) and `q_pos0` is the
    window's first position minus `first` (negative for a rank whose keys all come after it).
    Every rank gets the full output fp32 [T][Hq][hd]."""
    from .binding import attn_combine, attn_verify_q8_partials
    T, n_q_heads, head_dim = q.shape
    if kv_len > 0:
        po, pml = attn_verify_q8_partials(q, cache, kv_len, q_pos0, softmax_scale, n_split)
    else:
        po, pml = empty_partials(1, T * n_q_heads, head_dim, q.device)
    out = combine_sharded(po, pml, attn_combine)
    return out.reshape(T, n_q_heads, head_dim)
