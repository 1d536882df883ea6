"""attn_verify_q8_noalloc: the verify entry point for callers that cannot allocate device
memory (a runtime that owns every byte through its own arena, an allocator callback, a
plug-in barred from the allocator).  It keeps the split partials in a static device array
inside the library instead of a caller workspace.  These tests call it through the C ABI
twice in a row -- the second call reuses the array the first one left dirty -- and compare
each result with the regular entry point's and with the fp64 oracle, within the verify
tolerance.  This file is named so that pytest collects it last."""
import numpy as np
import pytest

import oracle
from speculative_verify_attention_gb300 import workloads

from ._util import VERIFY_TOL, build_caches, rel_err

pytestmark = pytest.mark.gpu


def _pair(w, n_split=0):
    """(noalloc result, attn_verify_q8 result, inputs, oracle cache) for workload w."""
    import torch

    from speculative_verify_attention_gb300 import attn_verify_q8, attn_verify_q8_noalloc
    inp = workloads.make_inputs(w)
    gpu, orc = build_caches(inp, garbage_tail=False)
    q = torch.from_numpy(inp.q).cuda()
    ref = attn_verify_q8(q, gpu, w.kv_len, w.q_pos0, w.softmax_scale, n_split=n_split)
    out = torch.full_like(q, float("nan"))
    attn_verify_q8_noalloc(q, gpu, w.kv_len, w.q_pos0, w.softmax_scale, out=out, n_split=n_split)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ref.cpu().numpy(), inp, orc


def _oracle_sampled(w, inp, orc, got, seed=0):
    """max |got - oracle| / max |oracle| over (row, head) pairs covering every row and head."""
    rng = np.random.default_rng(seed)
    sel = [(i, int(rng.integers(w.n_q_heads))) for i in range(w.n_q)]
    sel += [(int(rng.integers(w.n_q)), h) for h in range(w.n_q_heads)]
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, sel=sel)
    return rel_err(np.stack([got[i, h] for i, h in sel]), ref)


def test_two_calls_in_a_row_match_the_workspace_entry_point_and_the_oracle(lib):
    # first call: long context (many slices); second call: a smaller shape on the dirty array
    for w in (workloads.long_verify(20676, 8), workloads.verify_27b(4)):
        got, ref, inp, orc = _pair(w)
        assert np.all(np.isfinite(got))
        assert rel_err(got, ref) <= VERIFY_TOL, w.name
        assert _oracle_sampled(w, inp, orc, got) <= VERIFY_TOL, w.name


def test_largest_verify_shape_fits_the_array(lib):
    # T = 32 at a 32K context: the automatic plan's partials fit the array without shrinking
    w = workloads.long_verify(32768, 32)
    got, ref, inp, orc = _pair(w)
    assert rel_err(got, ref) <= VERIFY_TOL
    assert _oracle_sampled(w, inp, orc, got, seed=1) <= VERIFY_TOL


def test_explicit_small_split_count_matches_the_oracle(lib):
    # an explicit split count shorter than a tile per slice (n_split 7 over 300 keys)
    w = workloads.verify_workload("noalloc-explicit-split", 12, 2, 256, 300, 5, seed=777)
    got, ref, inp, orc = _pair(w, n_split=7)
    assert rel_err(got, ref) <= VERIFY_TOL
    full = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    assert rel_err(got, full) <= VERIFY_TOL


def test_shapes_beyond_the_array_are_rejected(lib):
    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8, KVQ8Error, attn_verify_q8_noalloc
    from speculative_verify_attention_gb300.binding import NOALLOC_SCRATCH_BYTES
    # 32 rows x 256 q heads x (256 + 2) fp32 > 8 MiB even with a single slice
    assert 32 * 256 * 258 * 4 > NOALLOC_SCRATCH_BYTES
    c = KVCacheQ8(16, 256, 64)
    q = torch.zeros((32, 256, 256), device="cuda")
    with pytest.raises(KVQ8Error) as e:
        attn_verify_q8_noalloc(q, c, 40, 8, 0.0625)
    assert e.value.status == 4
    # an explicit split count whose partials do not fit is refused too
    with pytest.raises(KVQ8Error) as e:
        attn_verify_q8_noalloc(torch.zeros((32, 24, 256), device="cuda"), KVCacheQ8(4, 256, 40000), 32800, 32768,
                               0.0625, n_split=1000)
    assert e.value.status == 4
