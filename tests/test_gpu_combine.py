"""attn_combine on the GPU: merges oracle partials like the oracle's own reducer."""
import numpy as np
import pytest

import oracle
from speculative_verify_attention_gb300 import workloads

from ._util import VERIFY_TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bounds", [[0, 300], [0, 1, 2, 299, 300], [0, 100, 100, 250, 300], [0, 7, 280, 300]])
def test_combine_matches_oracle(lib, bounds):
    import torch

    from speculative_verify_attention_gb300 import attn_combine
    inp = workloads.random_small(51, 6, 2, 128, 300, 5)
    c = oracle.Cache(2, 128, 300)
    c.append(inp.k, inp.v, 0)
    parts = [oracle.attention_partial(c, inp.q, 300, 290, 0.09, a, b) for a, b in zip(bounds[:-1], bounds[1:])]
    po = np.stack([p[0].reshape(-1, 128) for p in parts])
    pm = np.stack([p[1].reshape(-1) for p in parts])
    pl = np.stack([p[2].reshape(-1) for p in parts])
    ref = oracle.combine(po, pm, pl)
    ml = np.stack([pm, pl], axis=-1).astype(np.float32)
    out = attn_combine(torch.from_numpy(po.astype(np.float32)).cuda(), torch.from_numpy(ml).cuda())
    torch.cuda.synchronize()
    assert rel_err(out.cpu().numpy(), ref) <= VERIFY_TOL


def test_combine_all_empty_rows_are_zero(lib):
    import torch

    from speculative_verify_attention_gb300 import attn_combine
    po = torch.randn((3, 4, 64), device="cuda")
    ml = torch.zeros((3, 4, 2), device="cuda")
    ml[:, :, 0] = -float("inf")
    ml[1, 2] = torch.tensor([0.5, 2.0])
    out = attn_combine(po, ml)
    torch.cuda.synchronize()
    exp = torch.zeros((4, 64), device="cuda")
    exp[2] = po[1, 2] / 2.0
    assert torch.allclose(out, exp, rtol=1e-6, atol=0)


@pytest.mark.parametrize("n_split", [1, 2, 3, 4, 5])
def test_combine_many_rows_matches_oracle(lib, n_split):
    """Prompt-sized merges (thousands of rows, a few partials) take the flat one-thread-per-
    four-float4s kernel up to 4 partials and the row-per-block kernel beyond; both must agree
    with the oracle's reducer, including partials with no keys (m = -inf, l = 0) whose o slots
    hold NaN."""
    import torch

    from speculative_verify_attention_gb300 import attn_combine
    rows, hd = 5000, 256
    rng = np.random.default_rng(700 + n_split)
    po = rng.standard_normal((n_split, rows, hd)).astype(np.float32)
    pm = rng.normal(0.0, 3.0, (n_split, rows)).astype(np.float32)
    pl = rng.uniform(0.5, 50.0, (n_split, rows)).astype(np.float32)
    empty = rng.random((n_split, rows)) < 0.1
    empty[:, :3] = True                         # rows 0-2: no partial has keys
    pm[empty] = -np.inf
    pl[empty] = 0.0
    po[empty] = 0.0
    ref = oracle.combine(po.astype(np.float64), pm.astype(np.float64), pl.astype(np.float64))
    po[empty] = np.nan                          # an empty partial's o slot is never read
    ml = np.stack([pm, pl], axis=-1)
    out = attn_combine(torch.from_numpy(po).cuda(), torch.from_numpy(ml).cuda())
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.all(got[:3] == 0.0)
    assert rel_err(got, ref) <= VERIFY_TOL
