"""The kernels' code -> fp16 conversions, exhaustively, bit for bit against numpy's float16 of the
code ("gfx12 WMMA kernel for the int8-KV QSA prompt attention", How: the int8 -> fp16 conversion
is exact and was checked over all 65,536 byte pairs).  kvq8_selftest_convert runs the very device
functions the verify and prompt kernels call."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _run(kind, words):
    import torch

    from speculative_verify_attention_gb300 import kvq8_selftest_convert
    w = torch.from_numpy(np.ascontiguousarray(words, np.uint32).view(np.int32)).cuda()
    out = kvq8_selftest_convert(kind, w)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint32)


def _f16_bits(values):
    return np.asarray(values, np.float16).view(np.uint16).astype(np.uint32)


def _pair(lo, hi):
    return _f16_bits(lo) | (_f16_bits(hi) << 16)


def test_int8_pairs_every_byte_pair_both_selectors(lib):
    """QK operand / prompt dequantiser: every (b0, b1) and (b2, b3) byte pair of a word."""
    i = np.arange(1 << 16, dtype=np.uint32)
    words = i | (i << 16)                                # both halves of the word take pair i
    out = _run(0, words).reshape(-1, 2)
    b0 = (i & 0xFF).astype(np.uint8).view(np.int8)
    b1 = (i >> 8).astype(np.uint8).view(np.int8)
    want = _pair(b0, b1)
    assert np.array_equal(out[:, 0], want)               # selector of bytes 0, 1
    assert np.array_equal(out[:, 1], want)               # selector of bytes 2, 3
    # every code value -128 .. 127 appears, including -128 (which the quantiser never writes)
    assert set(np.unique(b0)) == set(range(-128, 128))


def test_int8_interleaved_pairs_every_byte_pair(lib):
    """PV operand: codes of two key rows interleaved byte by byte, for all 65,536 (a, b) pairs at
    every byte position."""
    a = np.repeat(np.arange(256, dtype=np.uint32), 256)
    b = np.tile(np.arange(256, dtype=np.uint32), 256)
    w0 = a * 0x01010101
    w1 = b * 0x01010101
    words = np.stack([w0, w1], axis=1).reshape(-1)
    out = _run(1, words).reshape(-1, 4)
    want = _pair(a.astype(np.uint8).view(np.int8), b.astype(np.uint8).view(np.int8))
    for m in range(4):
        assert np.array_equal(out[:, m], want), m
    # distinct bytes per position: the interleave takes byte m of each word, in order
    rng = np.random.default_rng(5)
    w = rng.integers(0, 1 << 32, 2 * 4096, dtype=np.uint64).astype(np.uint32)
    out = _run(1, w).reshape(-1, 4)
    w0, w1 = w[0::2], w[1::2]
    for m in range(4):
        x = ((w0 >> (8 * m)) & 0xFF).astype(np.uint8).view(np.int8)
        y = ((w1 >> (8 * m)) & 0xFF).astype(np.uint8).view(np.int8)
        assert np.array_equal(out[:, m], _pair(x, y)), m


def test_nibble_pairs_of_the_4bit_verify_operand(lib):
    """4-bit PV operand: every 16-bit half (4 nibbles) in both halves of the word."""
    v = np.arange(1 << 16, dtype=np.uint32)
    rev = v[::-1].copy()
    words = v | (rev << 16)
    out = _run(2, words).reshape(-1, 4)
    nib = lambda x, k: ((x >> (4 * k)) & 15).astype(np.int32) - 8   # noqa: E731
    for m, (k_lo, k_hi) in enumerate([(0, 0), (1, 1), (2, 2), (3, 3)]):
        assert np.array_equal(out[:, m], _pair(nib(v, k_lo), nib(rev, k_hi))), m


def test_nibble_bytes_of_the_4bit_prompt_dequantiser(lib):
    """4-bit prompt dequantiser: every byte value at every byte position of a word."""
    b = np.arange(256, dtype=np.uint32)
    rng = np.random.default_rng(9)
    others = rng.integers(0, 256, (256, 4)).astype(np.uint32)
    words = []
    for m in range(4):
        w = others.copy()
        w[:, m] = b
        words.append(w[:, 0] | (w[:, 1] << 8) | (w[:, 2] << 16) | (w[:, 3] << 24))
    words = np.concatenate(words)
    out = _run(3, words).reshape(-1, 4)
    for m in range(4):
        byte = (words >> (8 * m)) & 0xFF
        assert np.array_equal(out[:, m], _pair((byte & 15).astype(np.int32) - 8, (byte >> 4).astype(np.int32) - 8)), m


def test_rejects_bad_arguments(lib):
    import torch

    from speculative_verify_attention_gb300 import KVQ8Error, kvq8_selftest_convert
    with pytest.raises(KVQ8Error):
        kvq8_selftest_convert(4, torch.zeros(4, dtype=torch.int32, device="cuda"))
    with pytest.raises(KVQ8Error):
        kvq8_selftest_convert(1, torch.zeros(3, dtype=torch.int32, device="cuda"))
