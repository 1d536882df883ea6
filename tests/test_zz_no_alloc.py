"""attn_verify_q8_noalloc: the verify entry point for callers that cannot allocate device
memory (a runtime that owns every byte through its own arena, an allocator callback, a
plug-in barred from the allocator).  It keeps the split partials in a static device array
inside the library instead of a caller workspace.  These tests call it through the C ABI
twice in a row -- the second call reuses the array the first one left dirty -- and compare
each result with the regular entry point's, within the verify tolerance.  This file is named
so that pytest collects it last."""
import numpy as np
import pytest

from speculative_verify_attention_gb300 import workloads

from ._util import VERIFY_TOL, build_caches, rel_err

pytestmark = pytest.mark.gpu


def _pair(w):
    import torch

    from speculative_verify_attention_gb300 import attn_verify_q8, attn_verify_q8_noalloc
    inp = workloads.make_inputs(w)
    gpu, _ = build_caches(inp, garbage_tail=False)
    q = torch.from_numpy(inp.q).cuda()
    ref = attn_verify_q8(q, gpu, w.kv_len, w.q_pos0, w.softmax_scale)
    out = torch.full_like(q, float("nan"))
    attn_verify_q8_noalloc(q, gpu, w.kv_len, w.q_pos0, w.softmax_scale, out=out)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ref.cpu().numpy()


def test_two_calls_in_a_row_match_the_workspace_entry_point(lib):
    # first call: long context (many slices); second call: a smaller shape on the dirty array
    for w in (workloads.long_verify(20676, 8), workloads.verify_27b(4)):
        got, ref = _pair(w)
        assert np.all(np.isfinite(got))
        assert rel_err(got, ref) <= VERIFY_TOL, w.name


def test_automatic_split_count_shrinks_to_fit(lib):
    # T = 32 at 32K context needs more partials than the array holds with the default split
    w = workloads.long_verify(32768, 32)
    got, ref = _pair(w)
    assert rel_err(got, ref) <= VERIFY_TOL


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
