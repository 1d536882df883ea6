"""Shared helpers for the GPU parity tests: build both caches (library and oracle) from the
same seeded fp32 values, and the error metric max|gpu - oracle| / max|oracle|."""
from __future__ import annotations

import numpy as np

import oracle
from speculative_verify_attention_gb300 import workloads

VERIFY_TOL = 1e-4    # fp32 verify path
PROMPT_TOL = 2e-3    # fp16 tensor-core prompt path


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


def report_err(name: str, got, ref) -> float:
    """rel_err, printed with the output scale it is relative to (max |oracle|) and the largest
    absolute difference, so that a run with -s records the error each workload reaches."""
    err = rel_err(got, ref)
    scale = float(np.max(np.abs(np.asarray(ref, dtype=np.float64))))
    print(f"\nACHIEVED {name}: max|gpu - oracle| / max|oracle| = {err:.3e}, max|oracle| = {scale:.4g}, "
          f"max|gpu - oracle| = {err * scale:.3e}")
    return err


def build_caches(inp: workloads.Inputs, capacity: int | None = None, pos0: int = 0, garbage_tail: bool = True):
    """Quantise inp.k / inp.v at positions pos0.. into a library cache (on the GPU) and an
    oracle cache (on the CPU).  Positions outside the written range hold junk bytes in both,
    so a kernel that reads past kv_len is caught."""
    import torch

    from speculative_verify_attention_gb300 import KVCacheQ8

    L, hkv, hd = inp.k.shape
    cap = capacity or (pos0 + L)
    gpu = KVCacheQ8(hkv, hd, cap, device="cuda")
    orc = oracle.Cache(hkv, hd, cap)
    if garbage_tail and cap > pos0 + L:
        rng = np.random.default_rng(12345)
        junk_c = rng.integers(-128, 128, (hkv, cap, hd), dtype=np.int8)
        junk_s = rng.integers(0, 1 << 16, (hkv, cap, hd // 32), dtype=np.uint16)
        junk_s[(junk_s & 0x7C00) == 0x7C00] = 0x7BFF   # keep the junk finite
        for a in (orc.k_codes, orc.v_codes):
            a[:] = junk_c
        for a in (orc.k_scales, orc.v_scales):
            a[:] = junk_s
        for t in (gpu.k_codes, gpu.v_codes):
            t.copy_(torch.from_numpy(junk_c))
        for t in (gpu.k_scales, gpu.v_scales):
            t.copy_(torch.from_numpy(junk_s.view(np.float16)))
    gpu.append(torch.from_numpy(inp.k).cuda(), torch.from_numpy(inp.v).cuda(), pos0)
    orc.append(inp.k, inp.v, pos0)
    torch.cuda.synchronize()
    return gpu, orc


def planes_equal(gpu, orc) -> bool:
    ok = True
    for name in ("k_codes", "v_codes"):
        ok &= np.array_equal(getattr(gpu, name).cpu().numpy(), getattr(orc, name))
    for name in ("k_scales", "v_scales"):
        ok &= np.array_equal(getattr(gpu, name).cpu().numpy().view(np.uint16), getattr(orc, name))
    return bool(ok)
