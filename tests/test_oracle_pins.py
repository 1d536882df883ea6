"""Pins of the CPU oracle against facts that do not come from the oracle itself:
hand-derived values, closed forms, invariants, brute force with library routines.

Each test is chosen so that a plausible slip in the oracle (a dropped scale, a wrong
sign or index, a transposed operand, an off-by-one causal bound, the wrong tie rule,
the wrong GQA head map) fails at least one of them."""
import os

import numpy as np
import pytest
import scipy.special

import oracle
from speculative_verify_attention_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- fp16

def test_f16_to_f64_exhaustive_matches_numpy():
    bits = np.arange(1 << 16, dtype=np.uint16)
    got = oracle.f16_bits_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f32_to_f16_matches_numpy_rne():
    # strided sweep over all fp32 bit patterns
    u = np.arange(0, 1 << 32, 9973, dtype=np.uint64).astype(np.uint32)
    # every fp16 rounding midpoint (and its two fp32 neighbours) below the overflow bound
    h = np.arange(0, 0x7bff, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)   # exact: midpoints need at most 12 bits
    mu = mid.view(np.uint32)
    extra = np.concatenate([mu, mu + 1, mu - 1, mu | 0x80000000])
    x = np.concatenate([u, extra]).view(np.float32)
    got = oracle.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x3FF) != 0)


# --------------------------------------------------------------------------- Q8_0

def _read_hand_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "q8_0_hand_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest}
                cases.append(cur)
            elif key == "x":
                cur["x"] = [float(t) for t in rest.split()]
            elif key == "scale":
                cur["scale"] = int(rest, 16)
            elif key == "q":
                cur["q"] = [int(t) for t in rest.split()]
    return cases


@pytest.mark.parametrize("case", _read_hand_cases(), ids=lambda c: c["name"])
def test_quantize_hand_cases(case):
    x = np.zeros(32, np.float32)
    x[: len(case["x"])] = case["x"]
    exp_q = np.zeros(32, np.int8)
    exp_q[: len(case["q"])] = case["q"]
    q, d = oracle.quantize_q8_0(x)
    assert int(d[0]) == case["scale"]
    assert np.array_equal(q, exp_q)


def test_quantize_invariants_random():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((4096, 32)).astype(np.float32) * rng.uniform(1e-3, 1e3, (4096, 1)).astype(np.float32)
    q, d = oracle.quantize_q8_0(x)
    qn, dn = oracle.quantize_q8_0(-x)
    # odd symmetry, same scale
    assert np.array_equal(qn, -q) and np.array_equal(dn, d)
    # the largest |x| of every non-zero block maps to +-127
    assert np.all(np.abs(q).max(axis=1) == 127)
    # reconstruction bound |x - q d| <= d32/2 + 127 |d32 - d| (plus fp32 rounding slack)
    d32 = (np.abs(x).max(axis=1) / np.float32(127)).astype(np.float64)
    dd = d.astype(np.uint16).view(np.float16).astype(np.float64)[:, 0]
    err = np.abs(x.astype(np.float64) - q.astype(np.float64) * dd[:, None])
    bound = d32 / 2 * (1 + 1e-6) + 127 * np.abs(d32 - dd)
    assert np.all(err <= bound[:, None])


def test_quantize_matches_independent_numpy_formulation():
    """Same rule, written with numpy vector operations instead of a per-block C loop."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((262144, 32)).astype(np.float32)
    x *= np.exp2(rng.integers(-20, 12, (262144, 1))).astype(np.float32)
    x[3, 5] = 0.0
    q, d = oracle.quantize_q8_0(x)
    amax = np.abs(x).max(axis=1, keepdims=True)
    d32 = (amax / np.float32(127)).astype(np.float32)            # IEEE fp32 division
    t = (x / d32).astype(np.float32).astype(np.float64)          # IEEE fp32 division
    r = np.clip(np.trunc(t + np.copysign(0.5, t)), -127, 127)    # half away from zero, exact in fp64
    assert np.array_equal(q, r.astype(np.int8))
    assert np.array_equal(d[:, 0], d32[:, 0].astype(np.float16).view(np.uint16))


def test_quantize_tiny_and_huge_blocks():
    # amax so small that amax/127 underflows to 0 in fp32: stored d = 0, codes 0
    x = np.zeros(32, np.float32)
    x[0] = np.float32(1e-45)
    q, d = oracle.quantize_q8_0(x)
    assert int(d[0]) == 0 and not q.any()
    # d32 below the fp16 subnormal range rounds to scale 0 while codes stay +-127
    x[0] = np.float32(1e-10)
    q, d = oracle.quantize_q8_0(x)
    assert int(d[0]) == 0 and q[0] == 127
    # d32 above the fp16 range stores +inf
    x[0] = np.float32(1e7)
    q, d = oracle.quantize_q8_0(x)
    assert int(d[0]) == 0x7C00 and q[0] == 127


def test_kv_append_places_blocks():
    rng = np.random.default_rng(3)
    c = oracle.Cache(n_kv_heads=2, head_dim=64, capacity=10)
    k = rng.standard_normal((3, 2, 64)).astype(np.float32)
    v = rng.standard_normal((3, 2, 64)).astype(np.float32)
    c.append(k, v, pos0=5)
    for t in range(3):
        for h in range(2):
            qk, dk = oracle.quantize_q8_0(k[t, h])
            assert np.array_equal(c.k_codes[h, 5 + t], qk) and np.array_equal(c.k_scales[h, 5 + t], dk)
            qv, dv = oracle.quantize_q8_0(v[t, h])
            assert np.array_equal(c.v_codes[h, 5 + t], qv) and np.array_equal(c.v_scales[h, 5 + t], dv)
    assert not c.k_codes[:, :5].any() and not c.k_codes[:, 8:].any()
    with pytest.raises(ValueError):
        c.append(k, v, pos0=8)


# --------------------------------------------------------------------------- attention

def _dense_reference(cache, q, kv_len, q_pos0, scale):
    """Brute force: dequantise with numpy's fp16, dense masked softmax with scipy."""
    n_q, hq, hd = q.shape
    g = hq // cache.n_kv_heads
    kd = cache.k_codes.astype(np.float64) * np.repeat(cache.k_scales.view(np.float16).astype(np.float64), 32, axis=-1)
    vd = cache.v_codes.astype(np.float64) * np.repeat(cache.v_scales.view(np.float16).astype(np.float64), 32, axis=-1)
    out = np.zeros((n_q, hq, hd))
    n = np.arange(kv_len)
    for h in range(hq):
        kh, vh = kd[h // g, :kv_len], vd[h // g, :kv_len]
        s = scale * (q[:, h, :].astype(np.float64) @ kh.T)             # [n_q][kv_len]
        mask = n[None, :] <= (q_pos0 + np.arange(n_q))[:, None]
        s = np.where(mask, s, -np.inf)
        out[:, h, :] = scipy.special.softmax(s, axis=1) @ vh
    return out


def _cache_from(inp, capacity=None):
    L, hkv, hd = inp.k.shape
    c = oracle.Cache(hkv, hd, capacity or L)
    c.append(inp.k, inp.v, 0)
    return c


@pytest.mark.parametrize("hq,hkv,hd,L,nq,pos0", [(1, 1, 32, 9, 1, 8), (4, 2, 64, 40, 5, 35), (6, 2, 32, 33, 4, 20),
                                                 (3, 3, 64, 17, 3, 0), (4, 1, 32, 12, 4, 10)])
def test_attention_matches_dense_bruteforce(hq, hkv, hd, L, nq, pos0):
    inp = workloads.random_small(hq * 100 + L, hq, hkv, hd, L, nq, k_gain=2.0)
    c = _cache_from(inp)
    scale = 0.37
    got = oracle.attention(c, inp.q, L, pos0, scale)
    ref = _dense_reference(c, inp.q, L, pos0, scale)
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_single_visible_key_returns_its_value_exactly():
    inp = workloads.random_small(5, 2, 1, 64, 6, 1)
    c = _cache_from(inp)
    out = oracle.attention(c, inp.q, kv_len=6, q_pos0=0, scale=0.125)
    v0 = c.v_codes[0, 0].astype(np.float64) * np.repeat(c.v_scales[0, 0].view(np.float16).astype(np.float64), 32)
    assert np.array_equal(out[0, 0], v0) and np.array_equal(out[0, 1], v0)


def test_two_keys_closed_form():
    c = oracle.Cache(1, 32, 2)
    one = 0x3C00  # fp16 1.0
    c.k_codes[0, 0, 0] = 1
    c.k_codes[0, 1, 1] = 1
    c.k_scales[0, :, :] = one
    c.v_codes[0, 0, 0] = 10
    c.v_codes[0, 1, 1] = 20
    c.v_scales[0, :, :] = 0x3800  # fp16 0.5
    a, b = 0.7, -1.9
    q = np.zeros((1, 1, 32))
    q[0, 0, 0], q[0, 0, 1] = a, b
    scale = 1.5
    out = oracle.attention(c, q, kv_len=2, q_pos0=1, scale=scale)[0, 0]
    p0 = 1.0 / (1.0 + np.exp(scale * (b - a)))
    assert abs(out[0] - 5.0 * p0) < 1e-15 and abs(out[1] - 10.0 * (1 - p0)) < 1e-14
    assert not out[2:].any()


def test_zero_query_gives_mean_of_visible_values():
    inp = workloads.random_small(9, 3, 1, 64, 20, 3)
    c = _cache_from(inp)
    q = np.zeros((3, 3, 64))
    out = oracle.attention(c, q, kv_len=20, q_pos0=10, scale=0.3)
    vd = c.v_codes[0].astype(np.float64) * np.repeat(c.v_scales[0].view(np.float16).astype(np.float64), 32, -1)
    for i in range(3):
        ref = vd[: 10 + i + 1].mean(axis=0)
        assert np.max(np.abs(out[i] - ref[None, :])) < 1e-13


def test_uniform_keys_give_mean_of_visible_values():
    inp = workloads.random_small(10, 2, 1, 32, 15, 2)
    c = _cache_from(inp)
    c.k_codes[0, :] = c.k_codes[0, 0]
    c.k_scales[0, :] = c.k_scales[0, 0]
    out = oracle.attention(c, inp.q, kv_len=15, q_pos0=12, scale=0.5)
    vd = c.v_codes[0].astype(np.float64) * np.repeat(c.v_scales[0].view(np.float16).astype(np.float64), 32, -1)
    for i in range(2):
        assert np.max(np.abs(out[i] - vd[: 13 + i].mean(axis=0)[None, :])) < 1e-13


def test_unit_values_sum_to_one():
    inp = workloads.random_small(12, 4, 2, 64, 30, 4, k_gain=3.0)
    c = _cache_from(inp)
    c.v_codes[:] = 1
    c.v_scales[:] = 0x3C00
    out = oracle.attention(c, inp.q, kv_len=30, q_pos0=26, scale=0.2)
    assert np.max(np.abs(out - 1.0)) < 1e-14


def test_permuting_visible_keys_and_perturbing_hidden_keys():
    inp = workloads.random_small(13, 2, 1, 64, 24, 1)
    c = _cache_from(inp)
    base = oracle.attention(c, inp.q, kv_len=24, q_pos0=15, scale=0.25)
    perm = np.random.default_rng(1).permutation(16)
    c2 = oracle.Cache.from_planes(c.k_codes.copy(), c.k_scales.copy(), c.v_codes.copy(), c.v_scales.copy())
    for plane in (c2.k_codes, c2.k_scales, c2.v_codes, c2.v_scales):
        plane[0, :16] = plane[0, perm]
    assert np.max(np.abs(oracle.attention(c2, inp.q, 24, 15, 0.25) - base)) < 1e-13
    c3 = oracle.Cache.from_planes(c.k_codes.copy(), c.k_scales.copy(), c.v_codes.copy(), c.v_scales.copy())
    c3.k_codes[0, 16:] = 99
    c3.v_codes[0, 16:] = -99
    assert np.array_equal(oracle.attention(c3, inp.q, 24, 15, 0.25), base)
    c3.k_codes[0, 15] = 99   # the last visible key does matter
    assert not np.array_equal(oracle.attention(c3, inp.q, 24, 15, 0.25), base)


def test_gqa_equals_mha_with_repeated_kv_heads():
    hq, hkv, hd, L = 6, 2, 64, 21
    inp = workloads.random_small(14, hq, hkv, hd, L, 3)
    c = _cache_from(inp)
    g = hq // hkv
    rep = lambda a: np.repeat(a, g, axis=0)   # kv head h//g for q head h
    mha = oracle.Cache.from_planes(rep(c.k_codes), rep(c.k_scales), rep(c.v_codes), rep(c.v_scales))
    a = oracle.attention(c, inp.q, L, 18, 0.3)
    b = oracle.attention(mha, inp.q, L, 18, 0.3)
    assert np.array_equal(a, b)


def test_selected_pairs_match_full_output():
    inp = workloads.random_small(15, 4, 2, 32, 40, 6)
    c = _cache_from(inp)
    full = oracle.attention(c, inp.q, 40, 34, 0.4)
    sel = [(5, 3), (0, 0), (2, 1)]
    part = oracle.attention(c, inp.q, 40, 34, 0.4, sel=sel)
    for t, (i, h) in enumerate(sel):
        assert np.array_equal(part[t], full[i, h])


def test_split_and_combine_equals_unsplit():
    inp = workloads.random_small(16, 6, 2, 64, 50, 4)
    c = _cache_from(inp)
    full = oracle.attention(c, inp.q, 50, 46, 0.35)
    for bounds in ([0, 50], [0, 13, 50], [0, 1, 2, 48, 50], [0, 25, 47, 49, 50], [0, 0, 30, 50, 50]):
        parts = [oracle.attention_partial(c, inp.q, 50, 46, 0.35, a, b) for a, b in zip(bounds[:-1], bounds[1:])]
        po = np.stack([p[0].reshape(-1, 64) for p in parts])
        pm = np.stack([p[1].reshape(-1) for p in parts])
        pl = np.stack([p[2].reshape(-1) for p in parts])
        out = oracle.combine(po, pm, pl).reshape(full.shape)
        assert np.max(np.abs(out - full)) < 1e-13


def test_empty_partial_and_combine_hand_case():
    inp = workloads.random_small(17, 1, 1, 32, 8, 1)
    c = _cache_from(inp)
    o, m, l = oracle.attention_partial(c, inp.q, 8, 3, 1.0, 5, 8)   # keys 5..7 are all beyond row 0's bound 3
    assert m[0, 0] == -np.inf and l[0, 0] == 0 and not o.any()
    # two partials with known (o, m, l): out = (o1 e^{m1-M} + o2 e^{m2-M}) / (l1 e^{m1-M} + l2 e^{m2-M})
    po = np.array([[[2.0, 4.0]], [[3.0, -1.0]], [[7.0, 7.0]]])
    pm = np.array([[1.0], [np.log(2.0) + 1.0], [-np.inf]])
    pl = np.array([[1.0], [3.0], [0.0]])
    out = oracle.combine(po, pm, pl)
    assert np.allclose(out, [[(2.0 * 0.5 + 3.0) / (0.5 + 3.0), (4.0 * 0.5 - 1.0) / (0.5 + 3.0)]], rtol=0, atol=1e-15)


# --------------------------------------------------------------------------- tree-shaped windows

def _dense_tree_reference(cache, q, kv_len, q_pos0, scale, mask):
    """Brute force with an explicit boolean mask: key n is visible to row i when n < q_pos0,
    or when n = q_pos0 + j < kv_len and bit j of mask[i] is set; a row that sees nothing is 0."""
    n_q, hq, hd = q.shape
    g = hq // cache.n_kv_heads
    kd = cache.k_codes.astype(np.float64) * np.repeat(cache.k_scales.view(np.float16).astype(np.float64), 32, axis=-1)
    vd = cache.v_codes.astype(np.float64) * np.repeat(cache.v_scales.view(np.float16).astype(np.float64), 32, axis=-1)
    vis = np.zeros((n_q, kv_len), dtype=bool)
    for i in range(n_q):
        vis[i, : min(q_pos0, kv_len)] = True
        for j in range(32):
            if (int(mask[i]) >> j) & 1 and q_pos0 + j < kv_len:
                vis[i, q_pos0 + j] = True
    out = np.zeros((n_q, hq, hd))
    for h in range(hq):
        kh, vh = kd[h // g, :kv_len], vd[h // g, :kv_len]
        s = np.where(vis, scale * (q[:, h, :].astype(np.float64) @ kh.T), -np.inf)
        live = vis.any(axis=1)
        out[live, h, :] = scipy.special.softmax(s[live], axis=1) @ vh
    return out


def _tree_masks(parents):
    """Ancestor-or-self masks of a tree given each node's parent (-1 for a root)."""
    masks = []
    for i in range(len(parents)):
        m, a = 0, i
        while a >= 0:
            m |= 1 << a
            a = parents[a]
        masks.append(m)
    return np.array(masks, dtype=np.uint32)


def test_tree_chain_mask_equals_causal_attention():
    inp = workloads.random_small(401, 4, 2, 64, 40, 6)
    c = _cache_from(inp)
    got = oracle.attention_tree(c, inp.q, 40, 34, 0.3, oracle.chain_mask(6))
    assert np.max(np.abs(got - oracle.attention(c, inp.q, 40, 34, 0.3))) <= 1e-15


@pytest.mark.parametrize("parents,pos0,L", [([-1, 0, 0, 1, 1, 2, 5], 20, 27),     # a draft tree
                                            ([-1, -1, 0, 1, 2, 3], 9, 15),        # two branches
                                            ([-1, 0, 1, 2], 0, 4)])               # no context
def test_tree_matches_dense_bruteforce(parents, pos0, L):
    T = len(parents)
    inp = workloads.random_small(500 + T + pos0, 6, 2, 32, L, T, k_gain=2.0)
    c = _cache_from(inp)
    mask = _tree_masks(parents)
    got = oracle.attention_tree(c, inp.q, L, pos0, 0.41, mask)
    ref = _dense_tree_reference(c, inp.q, L, pos0, 0.41, mask)
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_tree_arbitrary_masks_and_bits_past_kv_len():
    inp = workloads.random_small(601, 3, 1, 64, 30, 8)
    c = _cache_from(inp)
    rng = np.random.default_rng(5)
    mask = rng.integers(0, 1 << 32, 8, dtype=np.uint64).astype(np.uint32)
    mask[0] = 0                                     # sees the context only
    got = oracle.attention_tree(c, inp.q, 30, 24, 0.2, mask)
    ref = _dense_tree_reference(c, inp.q, 30, 24, 0.2, mask)
    assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
    clipped = mask & np.uint32((1 << 6) - 1)        # keys 24..29 exist, bits 6.. point past kv_len
    assert np.array_equal(oracle.attention_tree(c, inp.q, 30, 24, 0.2, clipped), got)
    zero = oracle.attention_tree(c, inp.q[:1], 30, 0, 0.2, np.zeros(1, np.uint32))
    assert not zero.any()                           # nothing visible: zeros


def test_tree_permuting_window_tokens_with_their_bits():
    """Reordering the window tokens in the cache, and the mask bits with them, changes nothing."""
    parents = [-1, 0, 0, 1, 2]
    T, pos0, L = 5, 11, 16
    inp = workloads.random_small(701, 4, 1, 64, L, T)
    c = _cache_from(inp)
    mask = _tree_masks(parents)
    base = oracle.attention_tree(c, inp.q, L, pos0, 0.3, mask)
    perm = np.array([3, 0, 4, 1, 2])                # slot s of the new window holds old token perm[s]
    c2 = oracle.Cache.from_planes(c.k_codes.copy(), c.k_scales.copy(), c.v_codes.copy(), c.v_scales.copy())
    for plane in (c2.k_codes, c2.k_scales, c2.v_codes, c2.v_scales):
        plane[0, pos0:pos0 + T] = plane[0, pos0 + perm]
    inv = np.argsort(perm)
    mask2 = np.array([sum(1 << int(inv[j]) for j in range(T) if (int(m) >> j) & 1) for m in mask], np.uint32)
    assert np.max(np.abs(oracle.attention_tree(c2, inp.q, L, pos0, 0.3, mask2) - base)) < 1e-13
