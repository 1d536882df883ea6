"""The C-ABI library builds for sm_103a, loads, and exports every entry point that
include/kvq8attn.h declares (no kernel is launched: this runs without a GPU)."""
import ctypes
import os
import re

from speculative_verify_attention_gb300 import EXPORTED, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kvq8attn.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+([a-z][a-z0-9_]*)\s*\(", text, re.M)))


def test_header_declares_the_binding_names():
    assert sorted(EXPORTED) == _declared()


def test_library_exports_every_declared_symbol():
    path = build.build()
    lib = ctypes.CDLL(path)
    for name in _declared():
        assert hasattr(lib, name), name
    lib.kvq8_status_str.restype = ctypes.c_char_p
    assert lib.kvq8_status_str(0) == b"ok"
    assert lib.kvq8_status_str(4) == b"workspace missing or too small"


def test_automatic_plans_fill_one_wave_of_a_152_sm_part():
    """The automatic split count keeps the verify grid (slices x row chunks x KV heads) within one
    block per SM, the append path's window slice included; derived from the workspace size
    (n_split x rows x (head_dim + 2) x 4 bytes), with no GPU present (the planner assumes 152
    SMs then)."""
    lib = ctypes.CDLL(build.build())
    for fn in (lib.attn_verify_append_q8_workspace_bytes, lib.attn_verify_q8_workspace_bytes):
        fn.restype = ctypes.c_size_t
    hq, hkv, hd = 24, 4, 256
    for ctx in (512, 4096, 20676, 32768):
        for T in (1, 2, 4, 8, 16, 24, 32):
            rows = T * hq
            chunks = -(-T * (hq // hkv) // 24)
            ws = lib.attn_verify_append_q8_workspace_bytes(T, hq, hd, ctx, hkv, 0)
            assert ws % (rows * (hd + 2) * 4) == 0
            n_split = ws // (rows * (hd + 2) * 4)
            assert 2 <= n_split and n_split * chunks * hkv <= 152, (ctx, T, n_split)
            if ctx >= 20676:   # long enough for every slice to hold whole 128-key tiles and fill the SMs
                assert (n_split + 1) * chunks * hkv > 152 - chunks * hkv, (ctx, T, n_split)


def _partials_bytes_match(ws, rows_out, hd):
    """ws is the partials layout (o aligned to 256 bytes, then (m, l)) for some part count."""
    for parts in range(1, 257):
        o = parts * rows_out * hd * 4
        if ws == -(-o // 256) * 256 + parts * rows_out * 8:
            return True
    return False


def test_prompt_workspace_adds_the_fp16_copy_from_24_row_tiles():
    """attn_prompt_q8_workspace_bytes: the partials alone below 24 128-row tiles per KV head;
    from 24 on, the partials rounded up to 256 bytes plus the fp16 copy of both planes, keys
    < min(kv_len, q_pos0 + n_q) (computed without a GPU: the planner assumes 152 SMs)."""
    lib = ctypes.CDLL(build.build())
    fn = lib.attn_prompt_q8_workspace_bytes
    fn.restype = ctypes.c_size_t
    for hq, hkv, hd, kv_len, nq, pos0 in ((12, 1, 256, 32768, 245, 32523),   # 23 row tiles
                                          (12, 1, 256, 32768, 246, 32522),   # 24 (2952 rows)
                                          (12, 1, 256, 4096, 342, 1000),     # 33; copy stops at 1342
                                          (32, 8, 128, 32768, 2048, 30720),  # 64
                                          (32, 8, 128, 8192, 768, 7424),     # 24 (3072 rows)
                                          (32, 8, 128, 8192, 736, 7456)):    # 23
        ws = fn(nq, hq, hd, kv_len, pos0, hkv)
        rows_out = nq * hq
        mtiles = -(-nq * (hq // hkv) // 128)
        if mtiles < 24:
            assert _partials_bytes_match(ws, rows_out, hd), (hq, nq)
            continue
        copy = 2 * hkv * min(kv_len, pos0 + nq) * hd * 2
        part = ws - copy
        assert part % 256 == 0 and part > 0, (hq, nq)
        assert any(_partials_bytes_match(part - pad, rows_out, hd) for pad in range(0, 256, 8)), (hq, nq)


def test_prompt_f16_workspace_is_the_partials_alone():
    """attn_prompt_f16_workspace_bytes: an fp16 pool makes no copy, so its workspace is the
    partials part of attn_prompt_q8_workspace_bytes: equal to it below 24 row tiles per KV head,
    that part rounded to 256 bytes (the copy's offset) plus the copy from 24 on."""
    lib = ctypes.CDLL(build.build())
    for fn in (lib.attn_prompt_q8_workspace_bytes, lib.attn_prompt_f16_workspace_bytes):
        fn.restype = ctypes.c_size_t
    for hq, hkv, hd, kv_len, nq, pos0 in ((12, 1, 256, 32768, 245, 32523), (12, 1, 256, 32768, 2048, 30720),
                                          (32, 8, 128, 32768, 2048, 30720), (32, 8, 128, 8192, 736, 7456)):
        q8 = lib.attn_prompt_q8_workspace_bytes(nq, hq, hd, kv_len, pos0, hkv)
        f16 = lib.attn_prompt_f16_workspace_bytes(nq, hq, hd, kv_len, pos0, hkv)
        mtiles = -(-nq * (hq // hkv) // 128)
        if mtiles < 24:
            assert f16 == q8, (hq, nq)
        else:
            copy = 2 * hkv * min(kv_len, pos0 + nq) * hd * 2
            assert q8 == -(-f16 // 256) * 256 + copy, (hq, nq)
            assert _partials_bytes_match(f16, nq * hq, hd), (hq, nq)
