"""CPU oracle for Q8_0 GQA attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it; see ``oracle.c`` for the definitions it follows and the
readings taken where the pages are silent.

The C source is compiled with gcc into ``liboracle.so`` next to it on first use
(or by ``build()``).  All arithmetic happens in that C file; this module only
marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

QBLOCK = 32


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain C11, -O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cache(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("k_scales", ctypes.c_void_p),
                ("v_codes", ctypes.c_void_p), ("v_scales", ctypes.c_void_p),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("capacity", ctypes.c_int),
                ("format", ctypes.c_int), ("k_f16", ctypes.c_void_p), ("v_f16", ctypes.c_void_p),
                ("v_q4", ctypes.c_void_p)]


_Q8_0, _F16, _K8V4 = 0, 1, 2


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_f16_bits_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_bits_to_f64.restype = f64
            lib.oracle_f32_to_f16_bits.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_f16_bits.restype = ctypes.c_uint16
            lib.oracle_f16_bits_to_f64_array.argtypes = [vp, i64, vp]
            lib.oracle_f16_bits_to_f64_array.restype = None
            lib.oracle_f32_to_f16_bits_array.argtypes = [vp, i64, vp]
            lib.oracle_f32_to_f16_bits_array.restype = None
            lib.oracle_quantize_q8_0.argtypes = [vp, i64, vp, vp]
            lib.oracle_quantize_q8_0.restype = None
            lib.oracle_kv_append_q8_0.argtypes = [vp, i32, i32, i32, vp, vp, i32, i32]
            lib.oracle_kv_append_q8_0.restype = i32
            lib.oracle_kv_append_f16.argtypes = [vp, i32, i32, i32, vp, i32, i32]
            lib.oracle_kv_append_f16.restype = i32
            lib.oracle_quantize_q4.argtypes = [vp, i64, vp, vp]
            lib.oracle_quantize_q4.restype = None
            lib.oracle_kv_append_q4.argtypes = [vp, i32, i32, i32, vp, vp, i32, i32]
            lib.oracle_kv_append_q4.restype = i32
            lib.oracle_attention_partial.argtypes = [ctypes.POINTER(_Cache), vp, i32, i32, i32, i32, f64,
                                                     i64, i64, vp, vp, i64, vp, vp, vp]
            lib.oracle_attention_partial.restype = i32
            lib.oracle_attention.argtypes = [ctypes.POINTER(_Cache), vp, i32, i32, i32, i32, f64,
                                             vp, vp, i64, vp]
            lib.oracle_attention.restype = i32
            lib.oracle_attention_tree.argtypes = [ctypes.POINTER(_Cache), vp, i32, i32, i32, i32, vp, f64,
                                                  vp, vp, i64, vp]
            lib.oracle_attention_tree.restype = i32
            lib.oracle_combine.argtypes = [vp, vp, vp, i32, i64, i32, vp]
            lib.oracle_combine.restype = i32
            lib.oracle_set_threads.argtypes = [i32]
            lib.oracle_set_threads.restype = None
            lib.oracle_get_threads.argtypes = []
            lib.oracle_get_threads.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def f16_bits_to_f64(bits) -> np.ndarray:
    """Element-wise fp16 bits -> float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_f16_bits_to_f64_array(_ptr(b), b.size, _ptr(out))
    return out


def f32_to_f16_bits(x) -> np.ndarray:
    """Element-wise fp32 -> fp16 bits, round to nearest even."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_f32_to_f16_bits_array(_ptr(a), a.size, _ptr(out))
    return out


def quantize_q8_0(x) -> tuple[np.ndarray, np.ndarray]:
    """Quantise fp32 values [..., n*32] block by block -> (codes int8 same shape, scales uint16 [..., n])."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    if a.shape[-1] % QBLOCK:
        raise ValueError("last dimension must be a multiple of 32")
    nb = a.size // QBLOCK
    q = np.empty(a.shape, dtype=np.int8)
    d = np.empty(a.shape[:-1] + (a.shape[-1] // QBLOCK,), dtype=np.uint16)
    _load().oracle_quantize_q8_0(_ptr(a), nb, _ptr(q), _ptr(d))
    return q, d


class Cache:
    """Q8_0 KV planes held as numpy arrays, laid out like the library's planes:
    codes [n_kv_heads][capacity][head_dim] int8 and scales [n_kv_heads][capacity][head_dim/32]
    as fp16 bits (uint16)."""

    def __init__(self, n_kv_heads: int, head_dim: int, capacity: int):
        self.n_kv_heads, self.head_dim, self.capacity = n_kv_heads, head_dim, capacity
        nb = head_dim // QBLOCK
        self.k_codes = np.zeros((n_kv_heads, capacity, head_dim), dtype=np.int8)
        self.v_codes = np.zeros((n_kv_heads, capacity, head_dim), dtype=np.int8)
        self.k_scales = np.zeros((n_kv_heads, capacity, nb), dtype=np.uint16)
        self.v_scales = np.zeros((n_kv_heads, capacity, nb), dtype=np.uint16)

    @classmethod
    def from_planes(cls, k_codes, k_scales, v_codes, v_scales):
        h, cap, hd = k_codes.shape
        c = cls.__new__(cls)
        c.n_kv_heads, c.head_dim, c.capacity = h, hd, cap
        c.k_codes = np.ascontiguousarray(k_codes, dtype=np.int8)
        c.v_codes = np.ascontiguousarray(v_codes, dtype=np.int8)
        c.k_scales = np.ascontiguousarray(k_scales, dtype=np.uint16)
        c.v_scales = np.ascontiguousarray(v_scales, dtype=np.uint16)
        return c

    def _struct(self) -> _Cache:
        return _Cache(self.k_codes.ctypes.data, self.k_scales.ctypes.data, self.v_codes.ctypes.data,
                      self.v_scales.ctypes.data, self.n_kv_heads, self.head_dim, self.capacity, _Q8_0, None, None,
                      None)

    def append(self, k, v, pos0: int) -> None:
        """Quantise and write K and V values [n_tok][n_kv_heads][head_dim] at positions pos0.."""
        lib = _load()
        for x, codes, scales in ((k, self.k_codes, self.k_scales), (v, self.v_codes, self.v_scales)):
            a = np.ascontiguousarray(x, dtype=np.float32)
            if a.ndim != 3 or a.shape[1:] != (self.n_kv_heads, self.head_dim):
                raise ValueError(f"bad K/V shape {a.shape}")
            rc = lib.oracle_kv_append_q8_0(_ptr(a), a.shape[0], self.n_kv_heads, self.head_dim,
                                           _ptr(codes), _ptr(scales), self.capacity, int(pos0))
            if rc:
                raise ValueError("oracle_kv_append_q8_0 rejected its arguments")


def quantize_q4(x) -> tuple[np.ndarray, np.ndarray]:
    """4-bit V blocks of fp32 values [..., n*32] -> (nibbles uint8 [..., n*16], scales uint16 [..., n])."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    if a.shape[-1] % QBLOCK:
        raise ValueError("last dimension must be a multiple of 32")
    nb = a.size // QBLOCK
    q = np.empty(a.shape[:-1] + (a.shape[-1] // 2,), dtype=np.uint8)
    d = np.empty(a.shape[:-1] + (a.shape[-1] // QBLOCK,), dtype=np.uint16)
    _load().oracle_quantize_q4(_ptr(a), nb, _ptr(q), _ptr(d))
    return q, d


class CacheK8V4:
    """K8V4 pool held as numpy arrays: K as Q8_0 planes (k_codes int8 [Hkv][cap][hd], k_scales
    uint16 [Hkv][cap][hd/32]) and V as 4-bit planes (v_q4 uint8 [Hkv][cap][hd/2] nibbles,
    v_scales uint16 [Hkv][cap][hd/32]).  Every attention function here takes it."""

    def __init__(self, n_kv_heads: int, head_dim: int, capacity: int):
        self.n_kv_heads, self.head_dim, self.capacity = n_kv_heads, head_dim, capacity
        nb = head_dim // QBLOCK
        self.k_codes = np.zeros((n_kv_heads, capacity, head_dim), dtype=np.int8)
        self.k_scales = np.zeros((n_kv_heads, capacity, nb), dtype=np.uint16)
        self.v_q4 = np.full((n_kv_heads, capacity, head_dim // 2), 0x88, dtype=np.uint8)
        self.v_scales = np.zeros((n_kv_heads, capacity, nb), dtype=np.uint16)

    @classmethod
    def from_planes(cls, k_codes, k_scales, v_q4, v_scales):
        h, cap, hd = k_codes.shape
        c = cls.__new__(cls)
        c.n_kv_heads, c.head_dim, c.capacity = h, hd, cap
        c.k_codes = np.ascontiguousarray(k_codes, dtype=np.int8)
        c.k_scales = np.ascontiguousarray(k_scales, dtype=np.uint16)
        c.v_q4 = np.ascontiguousarray(v_q4, dtype=np.uint8)
        c.v_scales = np.ascontiguousarray(v_scales, dtype=np.uint16)
        return c

    def _struct(self) -> _Cache:
        return _Cache(self.k_codes.ctypes.data, self.k_scales.ctypes.data, None, self.v_scales.ctypes.data,
                      self.n_kv_heads, self.head_dim, self.capacity, _K8V4, None, None, self.v_q4.ctypes.data)

    def append(self, k, v, pos0: int) -> None:
        """Quantise K (Q8_0) and V (4-bit) values [n_tok][n_kv_heads][head_dim] at positions pos0.."""
        lib = _load()
        a_k = np.ascontiguousarray(k, dtype=np.float32)
        a_v = np.ascontiguousarray(v, dtype=np.float32)
        for a in (a_k, a_v):
            if a.ndim != 3 or a.shape[1:] != (self.n_kv_heads, self.head_dim):
                raise ValueError(f"bad K/V shape {a.shape}")
        rc = lib.oracle_kv_append_q8_0(_ptr(a_k), a_k.shape[0], self.n_kv_heads, self.head_dim,
                                       _ptr(self.k_codes), _ptr(self.k_scales), self.capacity, int(pos0))
        rc |= lib.oracle_kv_append_q4(_ptr(a_v), a_v.shape[0], self.n_kv_heads, self.head_dim,
                                      _ptr(self.v_q4), _ptr(self.v_scales), self.capacity, int(pos0))
        if rc:
            raise ValueError("oracle K8V4 append rejected its arguments")


class CacheF16:
    """fp16 KV pool held as numpy arrays of fp16 bits (uint16), laid out like the library's
    fp16 pool: k, v [n_kv_heads][capacity][head_dim].  Every attention function here takes
    it in place of a Q8_0 Cache."""

    def __init__(self, n_kv_heads: int, head_dim: int, capacity: int):
        self.n_kv_heads, self.head_dim, self.capacity = n_kv_heads, head_dim, capacity
        self.k = np.zeros((n_kv_heads, capacity, head_dim), dtype=np.uint16)
        self.v = np.zeros((n_kv_heads, capacity, head_dim), dtype=np.uint16)

    @classmethod
    def from_planes(cls, k_bits, v_bits):
        h, cap, hd = k_bits.shape
        c = cls.__new__(cls)
        c.n_kv_heads, c.head_dim, c.capacity = h, hd, cap
        c.k = np.ascontiguousarray(k_bits, dtype=np.uint16)
        c.v = np.ascontiguousarray(v_bits, dtype=np.uint16)
        return c

    def _struct(self) -> _Cache:
        return _Cache(None, None, None, None, self.n_kv_heads, self.head_dim, self.capacity, _F16,
                      self.k.ctypes.data, self.v.ctypes.data, None)

    def append(self, k, v, pos0: int) -> None:
        """Round K and V values [n_tok][n_kv_heads][head_dim] (fp32) to fp16 at positions pos0.."""
        lib = _load()
        for x, plane in ((k, self.k), (v, self.v)):
            a = np.ascontiguousarray(x, dtype=np.float32)
            if a.ndim != 3 or a.shape[1:] != (self.n_kv_heads, self.head_dim):
                raise ValueError(f"bad K/V shape {a.shape}")
            rc = lib.oracle_kv_append_f16(_ptr(a), a.shape[0], self.n_kv_heads, self.head_dim, _ptr(plane),
                                          self.capacity, int(pos0))
            if rc:
                raise ValueError("oracle_kv_append_f16 rejected its arguments")


def _sel(sel, n_q, n_q_heads):
    if sel is None:
        return None, None, n_q * n_q_heads
    rows = np.ascontiguousarray([p[0] for p in sel], dtype=np.int32)
    heads = np.ascontiguousarray([p[1] for p in sel], dtype=np.int32)
    return rows, heads, len(rows)


def attention(cache: Cache, q, kv_len: int, q_pos0: int, scale: float, sel=None) -> np.ndarray:
    """fp64 attention. q: [n_q][n_q_heads][head_dim] (any float dtype, converted exactly to fp64).
    Returns [n_q][n_q_heads][head_dim] when sel is None, else [len(sel)][head_dim] for the
    listed (row, q_head) pairs."""
    qa = np.ascontiguousarray(q, dtype=np.float64)
    n_q, n_q_heads, hd = qa.shape
    if hd != cache.head_dim:
        raise ValueError("head_dim mismatch")
    rows, heads, n_sel = _sel(sel, n_q, n_q_heads)
    out = np.empty((n_sel, hd), dtype=np.float64)
    st = cache._struct()
    rc = _load().oracle_attention(ctypes.byref(st), _ptr(qa), n_q, n_q_heads, int(kv_len), int(q_pos0),
                                  float(scale), None if rows is None else _ptr(rows),
                                  None if heads is None else _ptr(heads), n_sel, _ptr(out))
    if rc:
        raise ValueError("oracle_attention rejected its arguments")
    return out.reshape(n_q, n_q_heads, hd) if sel is None else out


def chain_mask(n_rows: int) -> np.ndarray:
    """Window mask of the sequential window: row i sees window keys 0..i."""
    return np.array([(1 << (i + 1)) - 1 for i in range(n_rows)], dtype=np.uint32)


def attention_tree(cache: Cache, q, kv_len: int, q_pos0: int, scale: float, mask, sel=None) -> np.ndarray:
    """fp64 attention of a tree-shaped window: row i sees every key n < q_pos0 and the window
    key q_pos0 + j when bit j of mask[i] (uint32) is set.  Shapes as in attention()."""
    qa = np.ascontiguousarray(q, dtype=np.float64)
    n_q, n_q_heads, hd = qa.shape
    if hd != cache.head_dim:
        raise ValueError("head_dim mismatch")
    mk = np.ascontiguousarray(mask, dtype=np.uint32)
    if mk.shape != (n_q,):
        raise ValueError("mask must hold one uint32 per row")
    rows, heads, n_sel = _sel(sel, n_q, n_q_heads)
    out = np.empty((n_sel, hd), dtype=np.float64)
    st = cache._struct()
    rc = _load().oracle_attention_tree(ctypes.byref(st), _ptr(qa), n_q, n_q_heads, int(kv_len), int(q_pos0),
                                       _ptr(mk), float(scale), None if rows is None else _ptr(rows),
                                       None if heads is None else _ptr(heads), n_sel, _ptr(out))
    if rc:
        raise ValueError("oracle_attention_tree rejected its arguments")
    return out.reshape(n_q, n_q_heads, hd) if sel is None else out


def attention_partial(cache: Cache, q, kv_len: int, q_pos0: int, scale: float, key_begin: int, key_end: int):
    """Unnormalised partial over keys [key_begin, key_end): returns (o [n_q][Hq][hd], m [n_q][Hq], l [n_q][Hq])."""
    qa = np.ascontiguousarray(q, dtype=np.float64)
    n_q, n_q_heads, hd = qa.shape
    o = np.empty((n_q * n_q_heads, hd), dtype=np.float64)
    m = np.empty(n_q * n_q_heads, dtype=np.float64)
    l = np.empty(n_q * n_q_heads, dtype=np.float64)
    st = cache._struct()
    rc = _load().oracle_attention_partial(ctypes.byref(st), _ptr(qa), n_q, n_q_heads, int(kv_len), int(q_pos0),
                                          float(scale), int(key_begin), int(key_end), None, None,
                                          n_q * n_q_heads, _ptr(o), _ptr(m), _ptr(l))
    if rc:
        raise ValueError("oracle_attention_partial rejected its arguments")
    return o.reshape(n_q, n_q_heads, hd), m.reshape(n_q, n_q_heads), l.reshape(n_q, n_q_heads)


def combine(part_o, part_m, part_l) -> np.ndarray:
    """Merge partials part_o [n_split][rows][hd], part_m / part_l [n_split][rows] -> [rows][hd]."""
    o = np.ascontiguousarray(part_o, dtype=np.float64)
    m = np.ascontiguousarray(part_m, dtype=np.float64)
    l = np.ascontiguousarray(part_l, dtype=np.float64)
    n_split, rows, hd = o.shape
    out = np.empty((rows, hd), dtype=np.float64)
    rc = _load().oracle_combine(_ptr(o), _ptr(m), _ptr(l), n_split, rows, hd, _ptr(out))
    if rc:
        raise ValueError("oracle_combine rejected its arguments")
    return out


from .head import argmax_rows_top_prob  # noqa: E402  (verify-head acceptance oracle)
