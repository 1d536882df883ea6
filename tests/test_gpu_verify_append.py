"""attn_verify_append_q8 on the GPU: the window's K/V land in the cache bit-exactly as
kvq8_append writes them, and the attention over q_pos0 + T keys matches the fp64 oracle
(max|gpu - oracle| / max|oracle| <= 1e-4)."""
import numpy as np
import pytest

import oracle
from speculative_verify_attention_gb300 import workloads

from ._util import VERIFY_TOL, build_caches, planes_equal, rel_err

pytestmark = pytest.mark.gpu


def _context_only(inp: workloads.Inputs, q_pos0: int) -> workloads.Inputs:
    return workloads.Inputs(k=inp.k[:q_pos0], v=inp.v[:q_pos0], q=inp.q)


def _append_verify(inp, q_pos0, scale, capacity, n_split=0):
    """Library cache holding the context only (junk past it), then one fused call; the oracle
    cache gets every key by its own quantiser."""
    import torch

    from speculative_verify_attention_gb300 import attn_verify_append_q8
    T = inp.q.shape[0]
    gpu, _ = build_caches(_context_only(inp, q_pos0), capacity=capacity)
    orc = oracle.Cache(inp.k.shape[1], inp.k.shape[2], capacity)
    orc.append(inp.k[: q_pos0 + T], inp.v[: q_pos0 + T], 0)
    kn = torch.from_numpy(np.ascontiguousarray(inp.k[q_pos0: q_pos0 + T])).cuda()
    vn = torch.from_numpy(np.ascontiguousarray(inp.v[q_pos0: q_pos0 + T])).cuda()
    out = attn_verify_append_q8(torch.from_numpy(np.ascontiguousarray(inp.q, np.float32)).cuda(), kn, vn, gpu,
                                q_pos0, scale, n_split=n_split)
    torch.cuda.synchronize()
    return gpu, orc, out.cpu().numpy()


def _written_equal(gpu, orc, end):
    """Cache planes equal on positions [0, end) of every head (junk beyond is not compared)."""
    ok = True
    for name in ("k_codes", "v_codes"):
        ok &= np.array_equal(getattr(gpu, name).cpu().numpy()[:, :end], getattr(orc, name)[:, :end])
    for name in ("k_scales", "v_scales"):
        ok &= np.array_equal(getattr(gpu, name).cpu().numpy().view(np.uint16)[:, :end],
                             getattr(orc, name)[:, :end])
    return bool(ok)


@pytest.mark.parametrize("T,n_split", [(4, 0), (8, 0), (16, 0), (32, 0), (4, 5), (8, 1), (32, 100)])
def test_27b_shape_matches_oracle(lib, T, n_split):
    w = workloads.verify_workload(f"append-24q4kv-hd256-ctx1000-T{T}", 24, 4, 256, 1000, T, k_outliers=4,
                                  seed=950 + T)
    inp = workloads.make_inputs(w)
    gpu, orc, got = _append_verify(inp, w.q_pos0, w.softmax_scale, w.kv_len + 40, n_split)
    assert _written_equal(gpu, orc, w.kv_len)
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    assert rel_err(got, ref) <= VERIFY_TOL


@pytest.mark.parametrize("q_pos0", [0, 1, 63, 64, 127, 128, 129, 511])
def test_hd128_window_slice_boundaries(lib, q_pos0):
    """Context ends on and off 64-key and 128-key boundaries; q_pos0 = 0 leaves the window
    slice alone."""
    T = 12
    inp = workloads.random_small(960 + q_pos0, 8, 2, 128, q_pos0 + T, T)
    gpu, orc, got = _append_verify(inp, q_pos0, 0.088, q_pos0 + T + 7)
    assert _written_equal(gpu, orc, q_pos0 + T)
    ref = oracle.attention(orc, inp.q, q_pos0 + T, q_pos0, 0.088)
    assert rel_err(got, ref) <= VERIFY_TOL


def test_matches_append_then_verify(lib):
    """Same cache bytes as kvq8_append, and the same attention as kvq8_append followed by
    attn_verify_q8 up to the rounding order of a different slicing."""
    import torch

    from speculative_verify_attention_gb300 import attn_verify_q8
    w = workloads.verify_27b(8)
    inp = workloads.make_inputs(w)
    gpu, orc, got = _append_verify(inp, w.q_pos0, w.softmax_scale, w.kv_len)
    assert planes_equal(gpu, orc)
    ref_gpu, _ = build_caches(inp, garbage_tail=False)
    assert planes_equal(ref_gpu, orc)
    two_step = attn_verify_q8(torch.from_numpy(inp.q).cuda(), ref_gpu, w.kv_len, w.q_pos0, w.softmax_scale)
    torch.cuda.synchronize()
    two_step = two_step.cpu().numpy()
    assert rel_err(got, two_step) <= VERIFY_TOL
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    assert rel_err(got, ref) <= VERIFY_TOL


def test_repeated_calls_in_one_stream(lib):
    """Back-to-back windows on one stream: each call's append is ordered after the previous
    call's combine and its scan sees every earlier window."""
    import torch

    from speculative_verify_attention_gb300 import attn_verify_append_q8
    T, ctx, steps = 4, 700, 5
    inp = workloads.random_small(977, 24, 4, 256, ctx + T * steps, T * steps)
    gpu, _ = build_caches(_context_only(inp, ctx), capacity=ctx + T * steps)
    orc = oracle.Cache(4, 256, ctx + T * steps)
    orc.append(inp.k, inp.v, 0)
    outs = []
    for s in range(steps):
        p0 = ctx + s * T
        q = torch.from_numpy(np.ascontiguousarray(inp.q[s * T:(s + 1) * T])).cuda()
        kn = torch.from_numpy(np.ascontiguousarray(inp.k[p0:p0 + T])).cuda()
        vn = torch.from_numpy(np.ascontiguousarray(inp.v[p0:p0 + T])).cuda()
        outs.append(attn_verify_append_q8(q, kn, vn, gpu, p0, 0.0625))
    torch.cuda.synchronize()
    assert planes_equal(gpu, orc)
    for s in range(steps):
        p0 = ctx + s * T
        ref = oracle.attention(orc, inp.q[s * T:(s + 1) * T], p0 + T, p0, 0.0625)
        assert rel_err(outs[s].cpu().numpy(), ref) <= VERIFY_TOL


def test_append_verify_rejects_bad_arguments(lib):
    import ctypes

    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8, attn_verify_append_q8_workspace_bytes
    from speculative_verify_attention_gb300.binding import (KVQ8_ERR_INVALID_ARG, KVQ8_ERR_MISALIGNED,
                                                             KVQ8_ERR_WORKSPACE, load_library)
    lib_ = load_library()
    cache = KVCacheQ8(2, 128, 64, device="cuda")
    q = torch.zeros((4, 8, 128), device="cuda")
    kn = torch.zeros((4, 2, 128), device="cuda")
    out = torch.empty_like(q)
    nb = attn_verify_append_q8_workspace_bytes(4, 8, 128, 40, 2)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")

    def call(qp=q.data_ptr(), k=kn.data_ptr(), v=kn.data_ptr(), pos=40, wsb=nb, o=out.data_ptr()):
        return lib_.attn_verify_append_q8(qp, k, v, 4, 8, ctypes.byref(cache.struct()), pos, 0.1, o,
                                          ws.data_ptr(), wsb, 0, None)

    assert call() == 0
    assert call(k=None) == KVQ8_ERR_INVALID_ARG
    assert call(v=None) == KVQ8_ERR_INVALID_ARG
    assert call(pos=61) == KVQ8_ERR_INVALID_ARG          # 61 + 4 > capacity 64
    assert call(pos=-1) == KVQ8_ERR_INVALID_ARG
    assert call(k=kn.data_ptr() + 4) == KVQ8_ERR_MISALIGNED
    assert call(wsb=nb - 1) == KVQ8_ERR_WORKSPACE
    torch.cuda.synchronize()


@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffer_entry_matches_device_entry(lib, pinned):
    """attn_verify_append_q8_host gives the device entry's output bit for bit and the same
    cache bytes: with pinned buffers (inputs through a copy kernel, the output written in
    place by the merge) and with pageable ones (copy-engine transfers)."""
    import torch

    from speculative_verify_attention_gb300 import (attn_verify_append_q8, attn_verify_append_q8_host,
                                                    attn_verify_append_q8_host_scratch_bytes)
    w = workloads.verify_27b(4)
    inp = workloads.make_inputs(w)
    T, ctx = w.n_q, w.q_pos0
    g1, _ = build_caches(_context_only(inp, ctx), capacity=w.kv_len)
    g2, _ = build_caches(_context_only(inp, ctx), capacity=w.kv_len)
    kn, vn = inp.k[ctx:ctx + T], inp.v[ctx:ctx + T]
    h_in = torch.from_numpy(np.concatenate([inp.q.ravel(), kn.ravel(), vn.ravel()]).astype(np.float32))
    h_out = torch.full((inp.q.size,), float("nan"), dtype=torch.float32)
    if pinned:
        h_in, h_out = h_in.pin_memory(), h_out.pin_memory()
    scratch = torch.empty(attn_verify_append_q8_host_scratch_bytes(T, 24, 256, ctx, 4), dtype=torch.uint8,
                          device="cuda")
    attn_verify_append_q8_host(h_in, T, 24, g1, ctx, w.softmax_scale, h_out, scratch)
    ref = attn_verify_append_q8(torch.from_numpy(inp.q).cuda(), torch.from_numpy(np.ascontiguousarray(kn)).cuda(),
                                torch.from_numpy(np.ascontiguousarray(vn)).cuda(), g2, ctx, w.softmax_scale)
    torch.cuda.synchronize()
    assert torch.equal(h_out.reshape(ref.shape), ref.cpu())
    for a, b in ((g1.k_codes, g2.k_codes), (g1.v_codes, g2.v_codes), (g1.k_scales, g2.k_scales),
                 (g1.v_scales, g2.v_scales)):
        assert torch.equal(a, b)
    from speculative_verify_attention_gb300.binding import KVQ8Error
    with pytest.raises(KVQ8Error):
        attn_verify_append_q8_host(h_in, T, 24, g1, ctx, w.softmax_scale, h_out, scratch[:-16])


def test_prepared_host_call_repeats_the_call(lib):
    """PreparedAppendVerifyHost: the same output as the one-off host call, over repeated use."""
    import torch

    from speculative_verify_attention_gb300 import (PreparedAppendVerifyHost, attn_verify_append_q8_host,
                                                    attn_verify_append_q8_host_scratch_bytes)
    inp = workloads.random_small(981, 8, 2, 128, 300, 6)
    ctx, T = 294, 6
    g1, _ = build_caches(_context_only(inp, ctx), capacity=300)
    g2, _ = build_caches(_context_only(inp, ctx), capacity=300)
    h_in = torch.from_numpy(np.concatenate([inp.q.ravel(), inp.k[ctx:].ravel(), inp.v[ctx:].ravel()])
                            .astype(np.float32)).pin_memory()
    o1 = torch.empty(inp.q.size, dtype=torch.float32).pin_memory()
    o2 = torch.empty(inp.q.size, dtype=torch.float32).pin_memory()
    nb = attn_verify_append_q8_host_scratch_bytes(T, 8, 128, ctx, 2)
    s1 = torch.empty(nb, dtype=torch.uint8, device="cuda")
    s2 = torch.empty(nb, dtype=torch.uint8, device="cuda")
    call = PreparedAppendVerifyHost(h_in, T, 8, g1, ctx, 0.088, o1, s1)
    for _ in range(3):
        call()
    attn_verify_append_q8_host(h_in, T, 8, g2, ctx, 0.088, o2, s2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
