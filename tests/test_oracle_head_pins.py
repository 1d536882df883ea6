"""Pins of the verify-head oracle (argmax and top probability per row) against hand cases,
closed forms and an independent library formulation."""
import numpy as np
import scipy.special

import oracle


def test_hand_cases():
    ninf, inf, nan = -np.inf, np.inf, np.nan
    rows = np.array([[1.0, 3.0, 3.0, 2.0],          # tie: first maximum
                     [0.0, nan, 5.0, nan],          # NaN ranks highest, first NaN
                     [ninf, ninf, ninf, ninf],      # all -inf: uniform limit
                     [ninf, 2.0, ninf, 2.0],        # -inf entries carry nothing
                     [1.0, inf, 0.0, inf],          # two +inf share the mass
                     [7.0, 7.0, 7.0, 7.0]], dtype=np.float32)
    idx, top = oracle.argmax_rows_top_prob(rows)
    assert idx.tolist() == [1, 1, 0, 1, 1, 0]
    e = np.exp
    assert abs(top[0] - 1.0 / (e(-2.0) + 1 + 1 + e(-1.0))) < 1e-15
    assert np.isnan(top[1])
    assert top[2] == 0.25 and top[3] == 0.5 and top[4] == 0.5 and top[5] == 0.25


def test_closed_forms():
    V = 248320
    x = np.zeros((2, V), np.float32)
    x[1, 12345] = 40.0                               # one dominant logit
    idx, top = oracle.argmax_rows_top_prob(x)
    assert idx.tolist() == [0, 12345]
    assert abs(top[0] - 1.0 / V) < 1e-18            # uniform row
    assert abs(top[1] - 1.0 / (1.0 + (V - 1) * np.exp(-40.0))) < 1e-15


def test_matches_library_softmax_and_argmax():
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((6, 5000)) * 3.0).astype(np.float32)
    x[2, 100] = x[2, 4000] = x[2].max() + 1.0       # a planted tie
    idx, top = oracle.argmax_rows_top_prob(x)
    ref_idx = np.argmax(x, axis=1)
    p = scipy.special.softmax(x.astype(np.float64), axis=1)
    assert np.array_equal(idx, ref_idx)
    assert np.max(np.abs(top - p[np.arange(6), ref_idx])) < 1e-15
    assert idx[2] == 100
