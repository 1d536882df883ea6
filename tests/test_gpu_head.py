"""argmax_rows_top_prob on the GPU against the oracle: argmax exact, top probability within
1e-5 (relative), on the 248,320-token vocabulary and on the special values."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

V = 248320
TOP_TOL = 1e-5


def _run(x):
    import torch

    from speculative_verify_attention_gb300 import argmax_rows_top_prob
    idx, top = argmax_rows_top_prob(torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda())
    torch.cuda.synchronize()
    return idx.cpu().numpy(), top.cpu().numpy()


def _check(x):
    idx, top = _run(x)
    ridx, rtop = oracle.argmax_rows_top_prob(x)
    assert np.array_equal(idx, ridx)
    nan = np.isnan(rtop)
    assert np.array_equal(np.isnan(top), nan)
    assert np.all(np.abs(top[~nan] - rtop[~nan]) <= TOP_TOL * rtop[~nan])


@pytest.mark.parametrize("T", [1, 4, 8, 32])
def test_random_logits_full_vocab(lib, T):
    rng = np.random.default_rng(1000 + T)
    _check((rng.standard_normal((T, V)) * 3.0).astype(np.float32))


def test_ties_across_blocks_and_special_values(lib):
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((8, V)) * 2.0).astype(np.float32)
    x[0, [5, 200000, 248319]] = 50.0              # a tie spread over far-apart blocks
    x[1, 240000] = np.nan                         # a late NaN
    x[1, 240001] = np.nan
    x[2, :] = -np.inf                             # nothing but -inf
    x[3, ::2] = -np.inf                           # half -inf
    x[4, [10, 99999]] = np.inf                    # two +inf share the mass
    x[5, :] = 1.25                                # uniform row
    x[6, 0] = np.float32(3.0e38)                  # a huge finite maximum
    x[7, 123456] = 30.0                           # one dominant logit
    _check(x)


@pytest.mark.parametrize("vocab", [1, 3, 1001, 65537])
def test_vocab_not_a_multiple_of_four(lib, vocab):
    rng = np.random.default_rng(vocab)
    x = (rng.standard_normal((3, vocab)) * 4.0).astype(np.float32)
    if vocab > 3:
        x[1, vocab - 1] = x[1].max() + 2.0        # the maximum in the scalar tail
    _check(x)


@pytest.mark.parametrize("vocab", [4, 8, 12, 4096])
def test_small_vocab_multiple_of_four(lib, vocab):
    rng = np.random.default_rng(vocab + 5)
    x = (rng.standard_normal((5, vocab)) * 4.0).astype(np.float32)
    x[2, :] = x[2, 0]                             # uniform: the first index wins the tie
    _check(x)


def test_ties_and_nan_on_block_boundaries(lib):
    """A block reduces 8192 logits (16-byte loads): ties straddling a block boundary go to the
    smaller index, and a NaN in a late block still wins."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((3, V)) * 2.0).astype(np.float32)
    x[0, [8191, 8192]] = 40.0
    x[1, [29 * 8192 - 1, 29 * 8192]] = 40.0
    x[2, 30 * 8192 + 5] = np.nan
    _check(x)


@pytest.mark.parametrize("n_rows", [64, 65, 130])
def test_many_rows(lib, n_rows):
    rng = np.random.default_rng(n_rows)
    x = (rng.standard_normal((n_rows, 20000)) * 3.0).astype(np.float32)
    x[n_rows - 1, 19999] = 99.0
    _check(x)


def test_rejects_bad_arguments(lib):
    import torch

    from speculative_verify_attention_gb300 import KVQ8Error, argmax_rows_top_prob
    x = torch.zeros((2, 64), device="cuda")
    with pytest.raises(KVQ8Error) as e:
        argmax_rows_top_prob(x, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 4                    # workspace too small
