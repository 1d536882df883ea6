"""Pins of the oracle's fp16 KV pool (the pool format the pages leave on their old kernel:
"gfx12 WMMA kernel for the int8-KV QSA prompt attention", Gating and Limits), checked
against things other than the oracle's own code:

* the append's fp32 -> fp16 rounding equals numpy's float16 conversion (round to nearest even)
  bit for bit, over ties, subnormals, overflow and signed zeros;
* attention over an fp16 pool equals a textbook numpy softmax attention (matmul, mask, exp)
  computed from numpy's own float16 -> float64 conversion;
* on values both formats hold exactly (Q8_0 codes times power-of-two scales), the fp16-pool
  attention equals the Q8_0 attention.
"""
import numpy as np
import pytest

import oracle


def test_append_rounds_like_numpy_float16():
    rng = np.random.default_rng(1)
    special = np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 6.1e-5, 5.96e-8,
                        2.98e-8, 2.99e-8, 1e-9, 1 + 2 ** -11, 1 + 3 * 2 ** -11, 2049.0, 2051.0, np.inf, -np.inf],
                       dtype=np.float32)
    vals = np.concatenate([special, rng.standard_normal(4000).astype(np.float32) * 10,
                           rng.standard_normal(1000).astype(np.float32) * 1e-5])
    n = vals.size // 64 * 64
    x = vals[:n].reshape(-1, 2, 32)
    c = oracle.CacheF16(2, 32, x.shape[0] + 3)
    c.append(x, -x, 3)
    with np.errstate(over="ignore"):        # 1e6 rounds to inf on both sides
        want_k = x.astype(np.float16).view(np.uint16)
        want_v = (-x).astype(np.float16).view(np.uint16)
    assert np.array_equal(c.k[:, 3:].transpose(1, 0, 2), want_k)
    assert np.array_equal(c.v[:, 3:].transpose(1, 0, 2), want_v)


def _textbook(q, k, v, kv_len, q_pos0, scale, group):
    """softmax(q k^T * scale, causal) v per (row, head), from float64 copies of the fp16 values."""
    n_q, hq, hd = q.shape
    out = np.zeros((n_q, hq, hd))
    for i in range(n_q):
        vis = min(q_pos0 + i + 1, kv_len)
        for h in range(hq):
            kh, vh = k[h // group, :vis], v[h // group, :vis]
            s = (kh @ q[i, h]) * scale
            if vis == 0:
                continue
            p = np.exp(s - s.max())
            out[i, h] = (p / p.sum()) @ vh
    return out


@pytest.mark.parametrize("hkv,g,hd,kv_len,n_q,q_pos0", [(1, 4, 64, 37, 3, 34), (2, 3, 128, 90, 5, 85),
                                                        (2, 2, 32, 20, 4, 0), (1, 1, 32, 10, 2, 3)])
def test_attention_matches_textbook(hkv, g, hd, kv_len, n_q, q_pos0):
    rng = np.random.default_rng(hd + kv_len)
    k = rng.standard_normal((kv_len, hkv, hd)).astype(np.float32)
    v = rng.standard_normal((kv_len, hkv, hd)).astype(np.float32)
    q = rng.standard_normal((n_q, hkv * g, hd))
    c = oracle.CacheF16(hkv, hd, kv_len + 2)
    c.append(k, v, 0)
    k64 = c.k.view(np.float16).astype(np.float64)
    v64 = c.v.view(np.float16).astype(np.float64)
    ref = _textbook(q, k64, v64, kv_len, q_pos0, 0.11, g)
    got = oracle.attention(c, q, kv_len, q_pos0, 0.11)
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_equals_q8_attention_on_exactly_representable_values():
    rng = np.random.default_rng(5)
    hkv, hd, cap = 2, 64, 50
    codes_k = rng.integers(-127, 128, (hkv, cap, hd), dtype=np.int8)
    codes_v = rng.integers(-127, 128, (hkv, cap, hd), dtype=np.int8)
    e_k = rng.integers(-12, 3, (hkv, cap, hd // 32))
    e_v = rng.integers(-12, 3, (hkv, cap, hd // 32))
    sk = np.ldexp(1.0, e_k).astype(np.float16)
    sv = np.ldexp(1.0, e_v).astype(np.float16)
    q8 = oracle.Cache.from_planes(codes_k, sk.view(np.uint16), codes_v, sv.view(np.uint16))
    kval = codes_k.astype(np.float64) * np.repeat(sk.astype(np.float64), 32, axis=-1)
    vval = codes_v.astype(np.float64) * np.repeat(sv.astype(np.float64), 32, axis=-1)
    assert np.array_equal(kval.astype(np.float16).astype(np.float64), kval)   # exact in fp16
    f16 = oracle.CacheF16.from_planes(kval.astype(np.float16).view(np.uint16),
                                      vval.astype(np.float16).view(np.uint16))
    q = rng.standard_normal((6, 6, hd))
    a = oracle.attention(q8, q, 48, 42, 0.07)
    b = oracle.attention(f16, q, 48, 42, 0.07)
    assert np.array_equal(a, b)
    pa = oracle.attention_partial(q8, q, 48, 42, 0.07, 10, 30)
    pb = oracle.attention_partial(f16, q, 48, 42, 0.07, 10, 30)
    for x, y in zip(pa, pb):
        assert np.array_equal(x, y)
