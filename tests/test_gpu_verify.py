"""attn_verify_q8 on the GPU against the fp64 oracle: max|gpu - oracle| / max|oracle| <= 1e-4."""
import numpy as np
import pytest

import oracle
from speculative_verify_attention_gb300 import workloads

from ._util import VERIFY_TOL, build_caches, planes_equal, rel_err, report_err

pytestmark = pytest.mark.gpu


def _run(gpu_cache, q, kv_len, q_pos0, scale, n_split=0):
    import torch

    from speculative_verify_attention_gb300 import attn_verify_q8
    out = attn_verify_q8(torch.from_numpy(np.ascontiguousarray(q, np.float32)).cuda(), gpu_cache, kv_len, q_pos0,
                         scale, n_split=n_split)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _check_full(w: workloads.Workload, n_split=0):
    inp = workloads.make_inputs(w)
    gpu, orc = build_caches(inp)
    assert planes_equal(gpu, orc)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, n_split)
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    err = report_err(w.name, got, ref)
    assert err <= VERIFY_TOL, f"{w.name}: rel err {err:.3e}"
    return err


def _check_sampled(w: workloads.Workload, n_pairs=24, seed=0):
    """Full-size workload: compare sampled (row, head) outputs, every row and head covered."""
    inp = workloads.make_inputs(w)
    gpu, orc = build_caches(inp, garbage_tail=False)
    got = _run(gpu, inp.q, w.kv_len, w.q_pos0, w.softmax_scale)
    rng = np.random.default_rng(seed)
    sel = [(i, int(rng.integers(w.n_q_heads))) for i in range(w.n_q)]
    sel += [(int(rng.integers(w.n_q)), h) for h in range(w.n_q_heads)]
    sel = sel[: max(n_pairs, w.n_q)]
    ref = oracle.attention(orc, inp.q, w.kv_len, w.q_pos0, w.softmax_scale, sel=sel)
    g = np.stack([got[i, h] for i, h in sel])
    err = report_err(w.name, g, ref)
    assert err <= VERIFY_TOL, f"{w.name}: rel err {err:.3e}"
    assert np.all(np.isfinite(got))
    return err


def test_tiny_workload(lib):
    _check_full(workloads.TINY)


@pytest.mark.parametrize("T", workloads.VERIFY_27B_T)
def test_27b_outlier_workload(lib, T):
    _check_full(workloads.verify_27b(T))


@pytest.mark.parametrize("T", workloads.HD128_T)
def test_hd128_workload(lib, T):
    w = workloads.hd128_verify(T)
    if T <= 8:
        _check_full(w)
    else:
        _check_sampled(w)


@pytest.mark.parametrize("ctx", workloads.LONG_CTX)
@pytest.mark.parametrize("T", workloads.LONG_T)
def test_long_context_workload(lib, ctx, T):
    from speculative_verify_attention_gb300 import kvq8_device_error
    kvq8_device_error(reset=True)
    _check_sampled(workloads.long_verify(ctx, T))
    assert kvq8_device_error(reset=True) == 0, "a kernel gave up on an internal wait"


@pytest.mark.parametrize("hq,hkv,hd,L,T,pos0", [
    (4, 1, 128, 1, 1, 0),        # a single key
    (6, 2, 256, 129, 3, 126),    # one key past a tile boundary
    (6, 6, 128, 300, 5, 295),    # group 1 (MHA), ragged tail
    (16, 1, 256, 777, 2, 775),   # group 16: 32 rows, one chunk
    (24, 2, 128, 515, 7, 508),   # 84 rows in three chunks
    (8, 2, 256, 1000, 32, 968),  # T = 32
    (4, 1, 128, 200, 4, 150),    # kv_len beyond the window: rows see q_pos0 + i only
    (4, 1, 256, 90, 6, 88),      # rows past kv_len see kv_len keys
])
def test_edge_shapes(lib, hq, hkv, hd, L, T, pos0):
    inp = workloads.random_small(hq * 1000 + L, hq, hkv, hd, L, T, k_gain=1.5)
    gpu, orc = build_caches(inp, capacity=((L + 200) // 8) * 8 + 8)
    got = _run(gpu, inp.q, L, pos0, 1.0 / np.sqrt(hd))
    ref = oracle.attention(orc, inp.q, L, pos0, 1.0 / np.sqrt(hd))
    assert rel_err(got, ref) <= VERIFY_TOL


@pytest.mark.parametrize("n_split", [1, 2, 7, 40])
def test_forced_split_counts(lib, n_split):
    inp = workloads.random_small(31, 12, 2, 256, 5000, 4)
    gpu, orc = build_caches(inp)
    got = _run(gpu, inp.q, 5000, 4996, 0.0625, n_split=n_split)
    ref = oracle.attention(orc, inp.q, 5000, 4996, 0.0625)
    assert rel_err(got, ref) <= VERIFY_TOL


def test_large_value_scales_stay_finite(lib):
    """V values up to ~1e3 (scale ~8): the power-of-two shift keeps p*dV inside fp16."""
    rng = np.random.default_rng(41)
    inp = workloads.random_small(41, 6, 1, 256, 700, 4)
    inp.v *= np.float32(1000.0)
    inp.v[rng.integers(0, 700, 50)] *= np.float32(1e-4)
    gpu, orc = build_caches(inp)
    got = _run(gpu, inp.q, 700, 696, 0.0625)
    ref = oracle.attention(orc, inp.q, 700, 696, 0.0625)
    assert rel_err(got, ref) <= VERIFY_TOL


def test_deterministic_and_graph_capture(lib):
    import torch

    from speculative_verify_attention_gb300 import attn_verify_q8, attn_verify_q8_workspace_bytes
    w = workloads.verify_27b(4)
    inp = workloads.make_inputs(w)
    gpu, _ = build_caches(inp, garbage_tail=False)
    q = torch.from_numpy(inp.q).cuda()
    ws = torch.empty(attn_verify_q8_workspace_bytes(w.n_q, w.n_q_heads, w.head_dim, w.kv_len, w.n_kv_heads),
                     dtype=torch.uint8, device="cuda")
    out1 = attn_verify_q8(q, gpu, w.kv_len, w.q_pos0, w.softmax_scale, workspace=ws).clone()
    out2 = attn_verify_q8(q, gpu, w.kv_len, w.q_pos0, w.softmax_scale, workspace=ws).clone()
    assert torch.equal(out1, out2)
    out3 = torch.zeros_like(out1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        attn_verify_q8(q, gpu, w.kv_len, w.q_pos0, w.softmax_scale, out=out3, workspace=ws)  # warm (attributes)
    torch.cuda.current_stream().wait_stream(s)
    out3.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        attn_verify_q8(q, gpu, w.kv_len, w.q_pos0, w.softmax_scale, out=out3, workspace=ws)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out1, out3)


def test_verify_rejects_bad_arguments(lib):
    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8, KVQ8Error, attn_verify_q8
    c = KVCacheQ8(1, 128, 64)
    q = torch.zeros((4, 4, 128), device="cuda")
    for kwargs, status in [(dict(kv_len=65), 1), (dict(kv_len=0), 1)]:
        with pytest.raises(KVQ8Error) as e:
            attn_verify_q8(q, c, q_pos0=0, softmax_scale=0.1, **kwargs)
        assert e.value.status == status
    with pytest.raises(KVQ8Error) as e:       # 33 rows
        attn_verify_q8(torch.zeros((33, 4, 128), device="cuda"), c, 40, 0, 0.1)
    assert e.value.status == 1
    with pytest.raises(KVQ8Error) as e:       # head_dim 64 is not built
        attn_verify_q8(torch.zeros((4, 4, 64), device="cuda"), KVCacheQ8(1, 64, 64), 40, 0, 0.1)
    assert e.value.status == 2
    with pytest.raises(KVQ8Error) as e:       # 5 q heads over 2 kv heads
        attn_verify_q8(torch.zeros((4, 5, 128), device="cuda"), KVCacheQ8(2, 128, 64), 40, 0, 0.1)
    assert e.value.status == 2
    with pytest.raises(KVQ8Error) as e:       # workspace too small
        attn_verify_q8(q, c, 40, 0, 0.1, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 4


def test_second_device_after_the_first(lib):
    """The kernels' shared-memory opt-in is per device: a process that drives a second GPU runs
    the verify and prompt kernels there after running them on the first."""
    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8, attn_prompt_q8, attn_verify_q8
    if torch.cuda.device_count() < 2:
        pytest.skip("one GPU visible")
    w = workloads.TINY
    inp = workloads.make_inputs(w)
    pw = workloads.prompt_workload("two-device-prompt", 12, 1, 256, 512, 128, seed=4011)
    pin = workloads.make_inputs(pw)
    outs = []
    for dev in (0, 1):
        with torch.cuda.device(dev):
            c = KVCacheQ8(w.n_kv_heads, w.head_dim, w.kv_len, device=f"cuda:{dev}")
            c.append(torch.from_numpy(inp.k).to(f"cuda:{dev}"), torch.from_numpy(inp.v).to(f"cuda:{dev}"), 0)
            o = attn_verify_q8(torch.from_numpy(inp.q).to(f"cuda:{dev}"), c, w.kv_len, w.q_pos0, w.softmax_scale)
            pc = KVCacheQ8(1, 256, pw.kv_len, device=f"cuda:{dev}")
            pc.append(torch.from_numpy(pin.k).to(f"cuda:{dev}"), torch.from_numpy(pin.v).to(f"cuda:{dev}"), 0)
            po = attn_prompt_q8(torch.from_numpy(pin.q).to(f"cuda:{dev}"), pc, pw.kv_len, pw.q_pos0, pw.softmax_scale)
            torch.cuda.synchronize(dev)
            outs.append((o.cpu().numpy(), po.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])
