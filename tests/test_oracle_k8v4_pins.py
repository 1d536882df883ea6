"""Pins of the oracle's K8V4 pool (Q8_0 K, 4-bit V; the 4-bit format is a reading, stated in
tests/golden/q4_v_hand_cases.txt), checked against things other than the oracle's own code:

* hand-derived blocks (zero, exact integers, halfway ties, power-of-two scales), including the
  nibble packing order;
* the round-trip bound: every value is within half a step (plus the fp16 rounding of the
  scale) of its input, and the largest magnitude of a block maps to +-7;
* attention over a K8V4 pool equals a textbook numpy attention over values decoded here from
  the nibbles, and equals the Q8_0 attention when the Q8_0 V codes are the same small codes.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "q4_v_hand_cases.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            elif key == "x":
                cur["x"] = [float(v) for v in vals]
            elif key == "scale":
                cur["scale"] = int(vals[0], 16)
            elif key == "q":
                cur["q"] = [int(v) for v in vals]
            elif key == "bytes":
                cur["bytes"] = [int(v, 16) for v in vals]
    return cases


def _decode(packed):
    """Nibbles -> codes, element 2m low, 2m+1 high (independent of the oracle's packing code)."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 15).astype(np.int32) - 8
    hi = (p >> 4).astype(np.int32) - 8
    return np.stack([lo, hi], axis=-1).reshape(p.shape[:-1] + (p.shape[-1] * 2,))


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_cases(case):
    x = np.zeros(32, np.float32)
    x[: len(case["x"])] = case["x"]
    packed, d = oracle.quantize_q4(x)
    want = np.zeros(32, np.int32)
    want[: len(case["q"])] = case["q"]
    assert int(d[0]) == case["scale"]
    assert np.array_equal(_decode(packed), want)
    if "bytes" in case:
        assert list(packed[: len(case["bytes"])]) == case["bytes"]


def test_round_trip_bound_and_extremes():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((500, 32)) * rng.uniform(1e-3, 50, (500, 1))).astype(np.float32)
    packed, d = oracle.quantize_q4(x)
    q = _decode(packed)
    d16 = d.view(np.float16).astype(np.float64)[:, None]
    d32 = np.abs(x).max(axis=1, keepdims=True).astype(np.float64) / 7
    err = np.abs(q * d16 - x)
    assert np.all(err <= d32 / 2 + 7 * np.abs(d16 - d32) + 1e-6 * d32)
    amax_pos = np.abs(x).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(500), amax_pos]) == 7)
    assert np.all(np.sign(q[np.arange(500), amax_pos]) == np.sign(x[np.arange(500), amax_pos]))
    assert q.min() >= -7 and q.max() <= 7


def _textbook(q, kval, vval, kv_len, q_pos0, scale, group):
    n_q, hq, hd = q.shape
    out = np.zeros((n_q, hq, hd))
    for i in range(n_q):
        vis = min(q_pos0 + i + 1, kv_len)
        for h in range(hq):
            s = (kval[h // group, :vis] @ q[i, h]) * scale
            p = np.exp(s - s.max())
            out[i, h] = (p / p.sum()) @ vval[h // group, :vis]
    return out


@pytest.mark.parametrize("hkv,g,hd,kv_len,n_q,q_pos0", [(1, 6, 256, 45, 4, 41), (2, 4, 128, 70, 6, 64)])
def test_attention_matches_textbook(hkv, g, hd, kv_len, n_q, q_pos0):
    rng = np.random.default_rng(hd + kv_len)
    k = rng.standard_normal((kv_len, hkv, hd)).astype(np.float32)
    v = rng.standard_normal((kv_len, hkv, hd)).astype(np.float32)
    q = rng.standard_normal((n_q, hkv * g, hd))
    c = oracle.CacheK8V4(hkv, hd, kv_len)
    c.append(k, v, 0)
    ks = np.repeat(c.k_scales.view(np.float16).astype(np.float64), 32, axis=-1)
    vs = np.repeat(c.v_scales.view(np.float16).astype(np.float64), 32, axis=-1)
    kval = c.k_codes.astype(np.float64) * ks
    vval = _decode(c.v_q4).astype(np.float64) * vs
    ref = _textbook(q, kval, vval, kv_len, q_pos0, 0.07, g)
    got = oracle.attention(c, q, kv_len, q_pos0, 0.07)
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_equals_q8_attention_on_small_codes():
    rng = np.random.default_rng(17)
    hkv, hd, cap = 2, 64, 40
    kc = rng.integers(-127, 128, (hkv, cap, hd), dtype=np.int8)
    ks = rng.uniform(0.01, 0.05, (hkv, cap, hd // 32)).astype(np.float16).view(np.uint16)
    vq = rng.integers(-7, 8, (hkv, cap, hd))
    vs = rng.uniform(0.01, 0.2, (hkv, cap, hd // 32)).astype(np.float16).view(np.uint16)
    packed = ((vq[..., 0::2] + 8) | ((vq[..., 1::2] + 8) << 4)).astype(np.uint8)
    a = oracle.CacheK8V4.from_planes(kc, ks, packed, vs)
    b = oracle.Cache.from_planes(kc, ks, vq.astype(np.int8), vs)
    q = rng.standard_normal((5, 8, hd))
    assert np.array_equal(oracle.attention(a, q, 38, 33, 0.09), oracle.attention(b, q, 38, 33, 0.09))


@pytest.mark.parametrize("hkv,hd,cap,pos0,n_tok", [(2, 64, 23, 7, 5), (3, 128, 40, 31, 9)])
def test_append_places_each_token_at_its_row(hkv, hd, cap, pos0, n_tok):
    """The 4-bit append at pos0 > 0 with several KV heads: the nibbles of token t of head h
    decode (here, not with the oracle's code) to values within the round-trip bound of that
    token's own inputs, so a wrong row stride, head/token order or pos0 offset in the append
    fails; every row outside [pos0, pos0 + n_tok) keeps its zero-code filler and zero scale."""
    rng = np.random.default_rng(hkv * 100 + pos0)
    k = rng.standard_normal((n_tok, hkv, hd)).astype(np.float32)
    v = (rng.standard_normal((n_tok, hkv, hd)) * rng.uniform(0.1, 10.0, (n_tok, hkv, 1))).astype(np.float32)
    c = oracle.CacheK8V4(hkv, hd, cap)
    c.append(k, v, pos0)
    q = _decode(c.v_q4).astype(np.float64)                                    # [hkv][cap][hd]
    d16 = np.repeat(c.v_scales.view(np.float16).astype(np.float64), 32, axis=-1)
    for h in range(hkv):
        for t in range(n_tok):
            x = v[t, h].astype(np.float64)
            d32 = np.repeat(np.abs(x).reshape(-1, 32).max(axis=1) / 7, 32)
            row = pos0 + t
            err = np.abs(q[h, row] * d16[h, row] - x)
            assert np.all(err <= d32 / 2 + 7 * np.abs(d16[h, row] - d32) + 1e-6 * d32), (h, t)
            # each block's largest magnitude lands on +-7 with the input's sign
            blk = np.abs(x).reshape(-1, 32).argmax(axis=1) + 32 * np.arange(hd // 32)
            assert np.all(q[h, row, blk] == 7 * np.sign(x[blk]))
    untouched = np.ones(cap, bool)
    untouched[pos0:pos0 + n_tok] = False
    assert np.all(c.v_q4[:, untouched] == 0x88)
    assert np.all(c.v_scales[:, untouched] == 0)
    # the K plane of the same append lands at the same rows (Q8_0 round-trip bound)
    kq = c.k_codes.astype(np.float64)
    ks = np.repeat(c.k_scales.view(np.float16).astype(np.float64), 32, axis=-1)
    for h in range(hkv):
        for t in range(n_tok):
            x = k[t, h].astype(np.float64)
            d32 = np.repeat(np.abs(x).reshape(-1, 32).max(axis=1) / 127, 32)
            err = np.abs(kq[h, pos0 + t] * ks[h, pos0 + t] - x)
            assert np.all(err <= d32 / 2 + 127 * np.abs(ks[h, pos0 + t] - d32) + 1e-6 * d32), (h, t)
    assert np.all(c.k_codes[:, untouched] == 0) and np.all(c.k_scales[:, untouched] == 0)
