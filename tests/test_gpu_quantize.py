"""kvq8_quantize on the GPU: bit-exact against the oracle's Q8_0 quantiser."""
import numpy as np
import pytest

import oracle
from speculative_verify_attention_gb300 import workloads

from ._util import build_caches, planes_equal
from .test_oracle_pins import _read_hand_cases

pytestmark = pytest.mark.gpu


def _gpu_quant(x):
    import torch

    from speculative_verify_attention_gb300 import kvq8_quantize
    n_tok, h, hd = x.shape
    codes = torch.zeros((h, n_tok, hd), dtype=torch.int8, device="cuda")
    scales = torch.zeros((h, n_tok, hd // 32), dtype=torch.float16, device="cuda")
    kvq8_quantize(torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda(), codes, scales, 0)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)


def test_hand_cases_bit_exact(lib):
    cases = _read_hand_cases()
    x = np.zeros((len(cases), 1, 32), np.float32)
    for i, c in enumerate(cases):
        x[i, 0, : len(c["x"])] = c["x"]
    codes, scales = _gpu_quant(x)
    for i, c in enumerate(cases):
        exp_q = np.zeros(32, np.int8)
        exp_q[: len(c["q"])] = c["q"]
        assert int(scales[0, i, 0]) == c["scale"], c["name"]
        assert np.array_equal(codes[0, i], exp_q), c["name"]


def test_random_wide_range_bit_exact(lib):
    rng = np.random.default_rng(21)
    x = rng.standard_normal((4096, 2, 256)).astype(np.float32)
    x *= np.exp2(rng.integers(-30, 14, (4096, 2, 8)).repeat(32, axis=2)).astype(np.float32)
    x[5, 1, :32] = 0.0
    x[6, 0, :32] = -0.0
    x[7, 0, 0] = np.float32(1e-45)
    x[8, 1, 3] = np.float32(1e7)
    codes, scales = _gpu_quant(x)
    q, d = oracle.quantize_q8_0(x)          # [n_tok][h][hd], [n_tok][h][nb]
    assert np.array_equal(codes, q.transpose(1, 0, 2))
    assert np.array_equal(scales, d.transpose(1, 0, 2))


def test_exact_ties_bit_exact(lib):
    # d = 1 blocks (amax 127) whose other values are k + 0.5: every quotient is an exact tie
    rng = np.random.default_rng(22)
    x = (rng.integers(-127, 127, (512, 1, 128)) + 0.5).astype(np.float32)
    x[:, :, ::32] = 127.0
    codes, scales = _gpu_quant(x)
    q, d = oracle.quantize_q8_0(x)
    assert np.array_equal(codes, q.transpose(1, 0, 2)) and np.array_equal(scales, d.transpose(1, 0, 2))


def test_append_at_offset_and_capacity(lib):
    import torch

    inp = workloads.random_small(23, 4, 2, 128, 37, 1)
    gpu, orc = build_caches(inp, capacity=64, pos0=11)
    assert planes_equal(gpu, orc)
    # n_tok = 0 is a no-op
    from speculative_verify_attention_gb300 import kvq8_quantize
    before = gpu.k_codes.clone()
    kvq8_quantize(torch.zeros((0, 2, 128), device="cuda"), gpu.k_codes, gpu.k_scales, 5)
    torch.cuda.synchronize()
    assert torch.equal(before, gpu.k_codes)


def test_full_long_context_planes_bit_exact(lib):
    w = workloads.long_verify(32768, 32)
    inp = workloads.make_inputs(w)
    gpu, orc = build_caches(inp, garbage_tail=False)
    assert planes_equal(gpu, orc)


def test_outlier_workload_planes_bit_exact(lib):
    w = workloads.verify_27b(8)
    inp = workloads.make_inputs(w)
    assert inp.outlier_channels.shape == (4, 4)
    gpu, orc = build_caches(inp, garbage_tail=False)
    assert planes_equal(gpu, orc)


def test_quantize_rejects_bad_arguments(lib):
    import torch

    from speculative_verify_attention_gb300 import KVQ8Error, kvq8_quantize
    codes = torch.zeros((1, 8, 64), dtype=torch.int8, device="cuda")
    scales = torch.zeros((1, 8, 2), dtype=torch.float16, device="cuda")
    with pytest.raises(KVQ8Error) as e:   # does not fit the capacity
        kvq8_quantize(torch.zeros((4, 1, 64), device="cuda"), codes, scales, 6)
    assert e.value.status == 1
    with pytest.raises(KVQ8Error) as e:   # head_dim not a multiple of 32
        kvq8_quantize(torch.zeros((1, 1, 48), device="cuda"), torch.zeros((1, 8, 48), dtype=torch.int8,
                      device="cuda"), scales, 0)
    assert e.value.status == 2
    buf = torch.zeros(4 * 64 + 1, device="cuda")
    with pytest.raises(KVQ8Error) as e:   # misaligned input pointer
        kvq8_quantize(buf[1:].view(4, 1, 64), codes, scales, 0)
    assert e.value.status == 3


def test_append_both_planes_bit_exact_against_two_quantize_calls(lib):
    """kvq8_append (one launch, K and V) writes the same bits as the oracle's quantiser and as
    two kvq8_quantize calls, at an offset, and leaves the other positions untouched."""
    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8, kvq8_append, kvq8_quantize
    inp = workloads.random_small(91, 8, 2, 256, 37, 4)
    k = torch.from_numpy(inp.k).cuda()
    v = torch.from_numpy(inp.v).cuda()
    a = KVCacheQ8(2, 256, 64, device="cuda")
    b = KVCacheQ8(2, 256, 64, device="cuda")
    kvq8_append(k, v, a, 20)
    kvq8_quantize(k, b.k_codes, b.k_scales, 20)
    kvq8_quantize(v, b.v_codes, b.v_scales, 20)
    torch.cuda.synchronize()
    for name in ("k_codes", "k_scales", "v_codes", "v_scales"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    orc = oracle.Cache(2, 256, 64)
    orc.append(inp.k, inp.v, 20)
    assert planes_equal(a, orc)
    assert not a.k_codes[:, :20].any() and not a.v_codes[:, 57:].any()


def test_append_rejects_bad_arguments(lib):
    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8, KVQ8Error, kvq8_append
    c = KVCacheQ8(1, 128, 16, device="cuda")
    k = torch.zeros((4, 1, 128), device="cuda")
    with pytest.raises(KVQ8Error) as e:       # past capacity
        kvq8_append(k, k, c, 13)
    assert e.value.status == 1
    with pytest.raises(ValueError):           # shape does not match the cache
        kvq8_append(torch.zeros((4, 2, 128), device="cuda"), k, c, 0)


def test_quotients_near_half_integers_bit_exact(lib):
    """Values one to four ulps either side of (k + 1/2) d for many block scales d: the
    quotients x / d sit right at the rounding boundaries, where a quotient computed as x times
    an approximate reciprocal could round the other way than the IEEE division does."""
    rng = np.random.default_rng(23)
    n_blk = 4096
    amax = (rng.uniform(0.5, 2.0, n_blk) * np.exp2(rng.integers(-20, 20, n_blk))).astype(np.float32)
    d = (amax / np.float32(127.0)).astype(np.float32)            # the IEEE fp32 scale the quantiser uses
    k = rng.integers(-127, 127, (n_blk, 31)).astype(np.float32)
    base = ((k + np.float32(0.5)) * d[:, None]).astype(np.float32)
    steps = rng.integers(-4, 5, (n_blk, 31)).astype(np.int32)
    vals = base.view(np.int32) + np.where(base >= 0, steps, -steps)
    vals = vals.view(np.float32)
    vals = np.clip(vals, -amax[:, None], amax[:, None])          # keep amax the block maximum
    x = np.concatenate([amax[:, None], vals], axis=1).reshape(n_blk // 8, 1, 256)
    codes, scales = _gpu_quant(x)
    q, dd = oracle.quantize_q8_0(x)
    assert np.array_equal(codes, q.transpose(1, 0, 2)) and np.array_equal(scales, dd.transpose(1, 0, 2))


def test_subnormal_scales_bit_exact(lib):
    """Blocks whose scale max|x| / 127 is an fp32 subnormal (the reciprocal approximation flushes
    it, so every code comes from the IEEE division), next to blocks with normal scales."""
    rng = np.random.default_rng(24)
    x = rng.standard_normal((64, 1, 256)).astype(np.float32)
    tiny = np.array([1e-36, 3e-37, 1e-38, 1e-39, 1e-41, 1.4e-45], np.float32)
    for i, t in enumerate(tiny):
        x[i, 0, :32] = (rng.uniform(-1.0, 1.0, 32) * t).astype(np.float32)
        x[i, 0, 7] = t
    codes, scales = _gpu_quant(x)
    q, d = oracle.quantize_q8_0(x)
    assert np.array_equal(codes, q.transpose(1, 0, 2)) and np.array_equal(scales, d.transpose(1, 0, 2))


def test_block_maxima_over_every_exponent_bit_exact(lib):
    """Block maxima at every fp32 exponent (subnormal to near the fp16-scale limit) with edge and
    random mantissas, the other values at (k + 1/2) d one ulp either side: the scale
    fl(max / 127) and every code match the IEEE-division oracle."""
    rng = np.random.default_rng(25)
    exps = np.arange(-149, 20)
    mants = np.concatenate([[1.0, 1.0 + 2.0 ** -23, 2.0 - 2.0 ** -23], rng.uniform(1.0, 2.0, 13)])
    amax = np.array([np.ldexp(m, e) for e in exps for m in mants], dtype=np.float64).astype(np.float32)
    amax = amax[amax > 0]
    n_blk = amax.size - amax.size % 8
    amax = amax[:n_blk]
    d = (amax / np.float32(127.0)).astype(np.float32)
    k = rng.integers(-127, 127, (n_blk, 31)).astype(np.float32)
    base = ((k + np.float32(0.5)) * d[:, None]).astype(np.float32)
    steps = rng.choice(np.array([-1, 1], np.int32), (n_blk, 31))
    vals = (base.view(np.int32) + np.where(base >= 0, steps, -steps)).view(np.float32)
    vals = np.clip(np.nan_to_num(vals), -amax[:, None], amax[:, None])
    x = np.concatenate([amax[:, None], vals], axis=1).reshape(n_blk // 8, 1, 256)
    codes, scales = _gpu_quant(x)
    q, dd = oracle.quantize_q8_0(x)
    assert np.array_equal(codes, q.transpose(1, 0, 2)) and np.array_equal(scales, dd.transpose(1, 0, 2))
