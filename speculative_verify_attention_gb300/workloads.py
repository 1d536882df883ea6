"""Seeded synthetic workloads for Q8_0 GQA verify and prompt attention.

This module holds random draws only -- shapes, seeds and value distributions -- and
none of the method's arithmetic (no quantisation, no attention).  Both the CUDA path
and the CPU oracle take their inputs from here, so they see identical fp32 values.

Workload shapes follow the pages' measurements:
  * "perf(gfx1100): share Q8 KV scans across verifier rows", "Kernel evidence":
    24 Q heads / 4 KV heads / head_dim 256 at contexts 2,048 - 32,768, and an hd128
    screen at context 8,192; sequential verify windows of 4-32 rows.
  * "gfx12 WMMA kernel for the int8-KV QSA prompt attention", "How" and
    "Measurements": 12 heads sharing one KV head, head_dim 256 (four 64-dim groups),
    an int8 context of 32K with a 2,048-query chunk.
The pages measured on real model KV and a long-code prompt; seeded N(0, 1) tensors of
the same shapes stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "verify" or "prompt"
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ctx: int                  # cached tokens before the query window
    n_q: int                  # query rows (T for verify, chunk length for prompt)
    k_outliers: int = 0       # channels per KV head whose K values are scaled by outlier_gain
    outlier_gain: float = 8.0
    q_dtype: str = "f32"      # "f32" (verify) or "f16" (prompt)
    seed: int = 0

    @property
    def kv_len(self) -> int:
        return self.ctx + self.n_q

    @property
    def q_pos0(self) -> int:
        return self.ctx

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def softmax_scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim))

    def kv_bytes(self) -> int:
        """Bytes of the Q8_0 K and V planes read for kv_len tokens (codes + fp16 scales)."""
        per_tok = 2 * (self.head_dim + 2 * (self.head_dim // 32))
        return self.n_kv_heads * self.kv_len * per_tok

    def causal_flops(self) -> int:
        """Algorithmic flops: 2 contractions x 2 flops x head_dim per visible (row, head, key)."""
        vis = sum(self.ctx + i + 1 for i in range(self.n_q))
        return 4 * self.head_dim * self.n_q_heads * vis


def verify_workload(name, n_q_heads, n_kv_heads, head_dim, ctx, T, k_outliers=0, seed=0) -> Workload:
    return Workload(name, "verify", n_q_heads, n_kv_heads, head_dim, ctx, T, k_outliers, 8.0, "f32", seed)


def prompt_workload(name, n_q_heads, n_kv_heads, head_dim, kv_len, n_q, seed=0) -> Workload:
    return Workload(name, "prompt", n_q_heads, n_kv_heads, head_dim, kv_len - n_q, n_q, 0, 8.0, "f16", seed)


# The five workload families (seed = family index * 1000 + variant).
TINY = verify_workload("tiny-verify-4q1kv-hd128-ctx512-T4", 4, 1, 128, 512, 4, seed=0)


def verify_27b(T: int) -> Workload:
    return verify_workload(f"verify-24q4kv-hd256-ctx4096-T{T}-outliers", 24, 4, 256, 4096, T,
                           k_outliers=4, seed=1000 + T)


def long_verify(ctx: int, T: int) -> Workload:
    return verify_workload(f"verify-24q4kv-hd256-ctx{ctx}-T{T}", 24, 4, 256, ctx, T, seed=2000 + T)


def hd128_verify(T: int) -> Workload:
    return verify_workload(f"verify-32q8kv-hd128-ctx8192-T{T}", 32, 8, 128, 8192, T, seed=3000 + T)


PROMPT = prompt_workload("prompt-12q1kv-hd256-kv32768-nq2048", 12, 1, 256, 32768, 2048, seed=4000)
# the second prompt shape: the hd128 head layout of the 32q/8kv family, same chunk and context
PROMPT_HD128 = prompt_workload("prompt-32q8kv-hd128-kv32768-nq2048", 32, 8, 128, 32768, 2048, seed=4001)

VERIFY_27B_T = (4, 8)
LONG_CTX = (2048, 20676, 32768)
LONG_T = (4, 8, 16, 32)
HD128_T = (4, 8, 16, 32)


def all_workloads() -> list[Workload]:
    out = [TINY] + [verify_27b(t) for t in VERIFY_27B_T]
    out += [long_verify(c, t) for c in LONG_CTX for t in LONG_T]
    out += [hd128_verify(t) for t in HD128_T]
    out.append(PROMPT)
    return out


@dataclass
class Inputs:
    """fp32 K/V values to be quantised into the cache, and the query rows."""
    k: np.ndarray             # [kv_len][n_kv_heads][head_dim] float32
    v: np.ndarray             # [kv_len][n_kv_heads][head_dim] float32
    q: np.ndarray             # [n_q][n_q_heads][head_dim] float32 or float16
    outlier_channels: np.ndarray = field(default_factory=lambda: np.zeros((0, 0), np.int64))


def make_inputs(w: Workload, kv_len: int | None = None) -> Inputs:
    """Draw the seeded inputs of a workload (optionally for a shorter kv_len, same seed).

    K and V are N(0, 1) fp32; with k_outliers > 0, that many channels per KV head (drawn
    without replacement from [0, head_dim) by the same generator) have their K values
    multiplied by outlier_gain.  q is N(0, 1) in the workload's q dtype."""
    L = w.kv_len if kv_len is None else kv_len
    rng = np.random.default_rng(w.seed)
    k = rng.standard_normal((L, w.n_kv_heads, w.head_dim), dtype=np.float32)
    v = rng.standard_normal((L, w.n_kv_heads, w.head_dim), dtype=np.float32)
    ch = np.zeros((w.n_kv_heads, w.k_outliers), dtype=np.int64)
    for h in range(w.n_kv_heads):
        if w.k_outliers:
            ch[h] = rng.choice(w.head_dim, size=w.k_outliers, replace=False)
            k[:, h, ch[h]] *= np.float32(w.outlier_gain)
    q = rng.standard_normal((w.n_q, w.n_q_heads, w.head_dim), dtype=np.float32)
    if w.q_dtype == "f16":
        q = q.astype(np.float16)
    return Inputs(k=k, v=v, q=q, outlier_channels=ch)


def random_small(seed: int, n_q_heads: int, n_kv_heads: int, head_dim: int, kv_len: int, n_q: int,
                 q_dtype: str = "f32", k_gain: float = 1.0) -> Inputs:
    """Small seeded case for edge-case tests (N(0,1) values, K scaled by k_gain)."""
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((kv_len, n_kv_heads, head_dim), dtype=np.float32) * np.float32(k_gain)
    v = rng.standard_normal((kv_len, n_kv_heads, head_dim), dtype=np.float32)
    q = rng.standard_normal((n_q, n_q_heads, head_dim), dtype=np.float32)
    if q_dtype == "f16":
        q = q.astype(np.float16)
    return Inputs(k=k, v=v, q=q)
