"""Verify-head acceptance oracle: per row of a [T][V] logits matrix, the argmax and the top
probability softmax(row)[argmax].

TEST INFRASTRUCTURE ONLY (same status as the rest of this package): the product path never
imports it.  Plain numpy, fp64 for the probability.

Source: "Engine perf(hip): MTP draft, shared expert, verify/sampler head", Summary item 1 and
"Verification & Parity Evidence" (argmax_rows and row_top_prob over T x 248,320 logits, checked
on ties, NaN and -inf).  The pages name the cases but not the rules; the readings here:
  * argmax: the first index of the row's maximum (ties go to the smallest index);
  * top probability: softmax(row)[argmax] = 1 / sum_j exp(x_j - max);
  * NaN ranks above every number: a row holding NaN has argmax = its first NaN and top
    probability NaN;
  * +inf: the row's probability mass is shared equally by its +inf entries (the limit of
    softmax), argmax = the first +inf;
  * a row of -inf only is the limit of equal logits: argmax 0, top probability 1 / V;
  * otherwise -inf entries carry probability 0.
"""
from __future__ import annotations

import numpy as np


def argmax_rows_top_prob(logits) -> tuple[np.ndarray, np.ndarray]:
    """logits [T][V] (float32 values, compared exactly) -> (argmax int32 [T], top_prob float64 [T])."""
    x = np.asarray(logits)
    if x.ndim != 2 or x.shape[1] < 1:
        raise ValueError("logits must be [T][V] with V >= 1")
    T, V = x.shape
    idx = np.zeros(T, dtype=np.int32)
    top = np.zeros(T, dtype=np.float64)
    for i in range(T):
        row = x[i].astype(np.float64)
        nan = np.flatnonzero(np.isnan(row))
        if nan.size:
            idx[i], top[i] = nan[0], np.nan
            continue
        m = row.max()
        if m == -np.inf:
            idx[i], top[i] = 0, 1.0 / V
            continue
        idx[i] = int(np.flatnonzero(row == m)[0])
        if m == np.inf:
            top[i] = 1.0 / np.count_nonzero(row == np.inf)
            continue
        top[i] = 1.0 / np.sum(np.exp(row - m))
    return idx, top
