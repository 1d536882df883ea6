"""ctypes binding of libkvq8attn.so -- argument marshalling only.

Every entry point mirrors the C ABI in include/kvq8attn.h under the same name.  Tensors
are torch CUDA tensors; their data pointers and the current CUDA stream are passed
through unchanged, and every step of the computation runs in the library's kernels.
There is no fallback: a missing library raises, and a nonzero status raises
KVQ8Error with the library's own message.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

KVQ8_OK = 0
KVQ8_ERR_INVALID_ARG = 1
KVQ8_ERR_UNSUPPORTED = 2
KVQ8_ERR_MISALIGNED = 3
KVQ8_ERR_WORKSPACE = 4
KVQ8_ERR_CUDA = 5

# Entry points declared in include/kvq8attn.h.
EXPORTED = ("kvq8_quantize", "kvq8_append", "attn_verify_q8_workspace_bytes", "attn_verify_q8", "attn_verify_tree_q8",
            "attn_verify_append_q8_workspace_bytes", "attn_verify_append_q8", "attn_verify_q8_partials_count",
            "attn_verify_q8_partials", "attn_verify_append_q8_host_scratch_bytes", "attn_verify_append_q8_host",
            "kvf16_append", "attn_verify_f16_workspace_bytes", "attn_verify_f16", "kvk8v4_append", "attn_verify_k8v4",
            "attn_prompt_k8v4", "attn_prompt_f16_workspace_bytes", "attn_prompt_f16", "attn_combine",
            "attn_prompt_q8_workspace_bytes", "attn_prompt_q8", "attn_verify_q8_noalloc", "kvq8_device_error", "kvq8_status_str",
            "argmax_rows_top_prob_workspace_bytes", "argmax_rows_top_prob", "kvq8_selftest_convert",
            "kvq8_selftest_wait_timeout")
NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024


class KVQ8Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed with status {status}: {kvq8_status_str(status)}")


class kvf16_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("capacity", ctypes.c_int32)]


class kvk8v4_cache(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("k_scales", ctypes.c_void_p),
                ("v_codes", ctypes.c_void_p), ("v_scales", ctypes.c_void_p),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("capacity", ctypes.c_int32)]


class kvq8_cache(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("k_scales", ctypes.c_void_p),
                ("v_codes", ctypes.c_void_p), ("v_scales", ctypes.c_void_p),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("capacity", ctypes.c_int32)]


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load the in-tree library (built by ``build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        cp = ctypes.POINTER(kvq8_cache)
        lib.kvq8_quantize.argtypes = [vp, i32, i32, i32, vp, vp, i32, i32, vp]
        lib.kvq8_quantize.restype = i32
        lib.kvq8_append.argtypes = [vp, vp, i32, cp, i32, vp]
        lib.kvq8_append.restype = i32
        lib.attn_verify_q8_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.attn_verify_q8_workspace_bytes.restype = sz
        lib.attn_verify_q8.argtypes = [vp, i32, i32, cp, i32, i32, f32, vp, vp, sz, i32, vp]
        lib.attn_verify_q8.restype = i32
        lib.attn_verify_tree_q8.argtypes = [vp, i32, i32, cp, i32, i32, vp, f32, vp, vp, sz, i32, vp]
        lib.attn_verify_tree_q8.restype = i32
        lib.attn_verify_q8_partials_count.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.attn_verify_q8_partials_count.restype = i32
        lib.attn_verify_q8_partials.argtypes = [vp, i32, i32, cp, i32, i32, f32, vp, vp, i32, vp]
        lib.attn_verify_q8_partials.restype = i32
        lib.attn_verify_append_q8_host_scratch_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.attn_verify_append_q8_host_scratch_bytes.restype = sz
        lib.attn_verify_append_q8_host.argtypes = [vp, i32, i32, cp, i32, f32, vp, vp, sz, i32, vp]
        lib.attn_verify_append_q8_host.restype = i32
        c44 = ctypes.POINTER(kvk8v4_cache)
        lib.kvk8v4_append.argtypes = [vp, vp, i32, c44, i32, vp]
        lib.kvk8v4_append.restype = i32
        lib.attn_verify_k8v4.argtypes = [vp, i32, i32, c44, i32, i32, f32, vp, vp, sz, i32, vp]
        lib.attn_verify_k8v4.restype = i32
        lib.attn_prompt_k8v4.argtypes = [vp, i32, i32, c44, i32, i32, f32, vp, vp, sz, vp]
        lib.attn_prompt_k8v4.restype = i32
        cf = ctypes.POINTER(kvf16_cache)
        lib.kvf16_append.argtypes = [vp, vp, i32, cf, i32, vp]
        lib.kvf16_append.restype = i32
        lib.attn_verify_f16_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.attn_verify_f16_workspace_bytes.restype = sz
        lib.attn_verify_f16.argtypes = [vp, i32, i32, cf, i32, i32, f32, vp, vp, sz, i32, vp]
        lib.attn_verify_f16.restype = i32
        lib.attn_prompt_f16.argtypes = [vp, i32, i32, cf, i32, i32, f32, vp, vp, sz, vp]
        lib.attn_prompt_f16.restype = i32
        lib.attn_verify_append_q8_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.attn_verify_append_q8_workspace_bytes.restype = sz
        lib.attn_verify_append_q8.argtypes = [vp, vp, vp, i32, i32, cp, i32, f32, vp, vp, sz, i32, vp]
        lib.attn_verify_append_q8.restype = i32
        lib.argmax_rows_top_prob_workspace_bytes.argtypes = [i32, i32]
        lib.argmax_rows_top_prob_workspace_bytes.restype = sz
        lib.argmax_rows_top_prob.argtypes = [vp, i32, i32, vp, vp, vp, sz, vp]
        lib.argmax_rows_top_prob.restype = i32
        lib.kvq8_selftest_convert.argtypes = [i32, vp, vp, i32, vp]
        lib.kvq8_selftest_convert.restype = i32
        lib.kvq8_selftest_wait_timeout.argtypes = [i32, vp]
        lib.kvq8_selftest_wait_timeout.restype = i32
        lib.attn_combine.argtypes = [vp, vp, i32, i32, i32, vp, vp]
        lib.attn_combine.restype = i32
        lib.attn_prompt_q8_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.attn_prompt_q8_workspace_bytes.restype = sz
        lib.attn_prompt_f16_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.attn_prompt_f16_workspace_bytes.restype = sz
        lib.attn_prompt_q8.argtypes = [vp, i32, i32, cp, i32, i32, f32, vp, vp, sz, vp]
        lib.attn_prompt_q8.restype = i32
        lib.attn_verify_q8_noalloc.argtypes = [vp, i32, i32, cp, i32, i32, f32, vp, i32, vp]
        lib.attn_verify_q8_noalloc.restype = i32
        lib.kvq8_device_error.argtypes = [i32]
        lib.kvq8_device_error.restype = i32
        lib.kvq8_status_str.argtypes = [i32]
        lib.kvq8_status_str.restype = ctypes.c_char_p
        _lib = lib
        return lib


def kvq8_status_str(status: int) -> str:
    return load_library().kvq8_status_str(int(status)).decode()


def kvq8_device_error(reset: bool = False) -> int:
    """The library's device error flag (nonzero: a kernel timed out on an internal wait).
    Synchronises the current device."""
    return int(load_library().kvq8_device_error(1 if reset else 0))


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _check(fn: str, status: int) -> None:
    if status != KVQ8_OK:
        raise KVQ8Error(fn, status)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype) -> None:
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor (got {t.dtype}, {t.device})")


class KVCacheQ8:
    """Caller-owned Q8_0 K/V planes on one device (the layout of include/kvq8attn.h):
    codes int8 [n_kv_heads][capacity][head_dim], scales fp16 [n_kv_heads][capacity][head_dim/32]."""

    def __init__(self, n_kv_heads: int, head_dim: int, capacity: int, device="cuda"):
        self.n_kv_heads, self.head_dim, self.capacity = n_kv_heads, head_dim, capacity
        nb = head_dim // 32
        self.k_codes = torch.zeros((n_kv_heads, capacity, head_dim), dtype=torch.int8, device=device)
        self.v_codes = torch.zeros((n_kv_heads, capacity, head_dim), dtype=torch.int8, device=device)
        self.k_scales = torch.zeros((n_kv_heads, capacity, nb), dtype=torch.float16, device=device)
        self.v_scales = torch.zeros((n_kv_heads, capacity, nb), dtype=torch.float16, device=device)

    @classmethod
    def from_planes(cls, k_codes, k_scales, v_codes, v_scales):
        c = cls.__new__(cls)
        c.n_kv_heads, c.capacity, c.head_dim = k_codes.shape
        c.k_codes, c.k_scales, c.v_codes, c.v_scales = k_codes, k_scales, v_codes, v_scales
        return c

    def struct(self) -> kvq8_cache:
        return kvq8_cache(self.k_codes.data_ptr(), self.k_scales.data_ptr(), self.v_codes.data_ptr(),
                          self.v_scales.data_ptr(), self.n_kv_heads, self.head_dim, self.capacity)

    def append(self, k: torch.Tensor, v: torch.Tensor, pos0: int, stream=None) -> None:
        """Quantise K and V values [n_tok][n_kv_heads][head_dim] (fp32) into positions pos0..
        (one kvq8_append launch for both planes)."""
        kvq8_append(k, v, self, pos0, stream)


class KVCacheK8V4:
    """Caller-owned K8V4 pool on one device (kvk8v4_cache of include/kvq8attn.h): K as Q8_0
    planes, V as 4-bit nibbles v_codes uint8 [n_kv_heads][capacity][head_dim/2] with fp16
    scales v_scales [n_kv_heads][capacity][head_dim/32]."""

    def __init__(self, n_kv_heads: int, head_dim: int, capacity: int, device="cuda"):
        self.n_kv_heads, self.head_dim, self.capacity = n_kv_heads, head_dim, capacity
        nb = head_dim // 32
        self.k_codes = torch.zeros((n_kv_heads, capacity, head_dim), dtype=torch.int8, device=device)
        self.k_scales = torch.zeros((n_kv_heads, capacity, nb), dtype=torch.float16, device=device)
        self.v_codes = torch.full((n_kv_heads, capacity, head_dim // 2), 0x88, dtype=torch.uint8, device=device)
        self.v_scales = torch.zeros((n_kv_heads, capacity, nb), dtype=torch.float16, device=device)

    def struct(self) -> kvk8v4_cache:
        return kvk8v4_cache(self.k_codes.data_ptr(), self.k_scales.data_ptr(), self.v_codes.data_ptr(),
                            self.v_scales.data_ptr(), self.n_kv_heads, self.head_dim, self.capacity)

    def append(self, k: torch.Tensor, v: torch.Tensor, pos0: int, stream=None) -> None:
        """Quantise K (Q8_0) and V (4-bit) values [n_tok][n_kv_heads][head_dim] (fp32) at pos0.."""
        kvk8v4_append(k, v, self, pos0, stream)


def kvk8v4_append(k: torch.Tensor, v: torch.Tensor, cache: KVCacheK8V4, pos0: int, stream=None) -> None:
    _need(k, "k", torch.float32)
    _need(v, "v", torch.float32)
    if k.shape != v.shape or k.dim() != 3 or k.shape[1:] != (cache.n_kv_heads, cache.head_dim):
        raise ValueError(f"k and v must both be [n_tok][{cache.n_kv_heads}][{cache.head_dim}]")
    st = load_library().kvk8v4_append(_ptr(k), _ptr(v), k.shape[0], ctypes.byref(cache.struct()), int(pos0),
                                      _stream(stream))
    _check("kvk8v4_append", st)


def attn_verify_k8v4(q: torch.Tensor, cache: KVCacheK8V4, kv_len: int, q_pos0: int, softmax_scale: float,
                     out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, n_split: int = 0,
                     stream=None) -> torch.Tensor:
    """Verify attention of fp32 q [T][Hq][hd] over a K8V4 pool; returns fp32 [T][Hq][hd]."""
    _need(q, "q", torch.float32)
    n_rows, n_q_heads, head_dim = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float32)
    if workspace is None:
        nbytes = attn_verify_q8_workspace_bytes(n_rows, n_q_heads, head_dim, kv_len, cache.n_kv_heads, n_split)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = load_library().attn_verify_k8v4(_ptr(q), n_rows, n_q_heads, ctypes.byref(cache.struct()), int(kv_len),
                                         int(q_pos0), float(softmax_scale), _ptr(out), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), int(n_split), _stream(stream))
    _check("attn_verify_k8v4", st)
    return out


def attn_prompt_k8v4(q: torch.Tensor, cache: KVCacheK8V4, kv_len: int, q_pos0: int, softmax_scale: float,
                     out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """Prompt-chunk attention of fp16 q [n_q][Hq][hd] over a K8V4 pool; returns fp32 [n_q][Hq][hd]."""
    _need(q, "q", torch.float16)
    n_q, n_q_heads, head_dim = q.shape
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    if workspace is None:
        nbytes = attn_prompt_q8_workspace_bytes(n_q, n_q_heads, head_dim, kv_len, q_pos0, cache.n_kv_heads)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = load_library().attn_prompt_k8v4(_ptr(q), n_q, n_q_heads, ctypes.byref(cache.struct()), int(kv_len),
                                         int(q_pos0), float(softmax_scale), _ptr(out), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream))
    _check("attn_prompt_k8v4", st)
    return out


class KVCacheF16:
    """Caller-owned fp16 KV pool on one device (kvf16_cache of include/kvq8attn.h):
    k, v fp16 [n_kv_heads][capacity][head_dim]."""

    def __init__(self, n_kv_heads: int, head_dim: int, capacity: int, device="cuda"):
        self.n_kv_heads, self.head_dim, self.capacity = n_kv_heads, head_dim, capacity
        self.k = torch.zeros((n_kv_heads, capacity, head_dim), dtype=torch.float16, device=device)
        self.v = torch.zeros((n_kv_heads, capacity, head_dim), dtype=torch.float16, device=device)

    def struct(self) -> kvf16_cache:
        return kvf16_cache(self.k.data_ptr(), self.v.data_ptr(), self.n_kv_heads, self.head_dim, self.capacity)

    def append(self, k: torch.Tensor, v: torch.Tensor, pos0: int, stream=None) -> None:
        """Round K and V values [n_tok][n_kv_heads][head_dim] (fp32) to fp16 at positions pos0.."""
        kvf16_append(k, v, self, pos0, stream)


def kvf16_append(k: torch.Tensor, v: torch.Tensor, cache: KVCacheF16, pos0: int, stream=None) -> None:
    _need(k, "k", torch.float32)
    _need(v, "v", torch.float32)
    if k.shape != v.shape or k.dim() != 3 or k.shape[1:] != (cache.n_kv_heads, cache.head_dim):
        raise ValueError(f"k and v must both be [n_tok][{cache.n_kv_heads}][{cache.head_dim}]")
    st = load_library().kvf16_append(_ptr(k), _ptr(v), k.shape[0], ctypes.byref(cache.struct()), int(pos0),
                                     _stream(stream))
    _check("kvf16_append", st)


def attn_verify_f16_workspace_bytes(n_rows: int, n_q_heads: int, head_dim: int, kv_len: int, n_kv_heads: int,
                                    n_split: int = 0) -> int:
    return int(load_library().attn_verify_f16_workspace_bytes(n_rows, n_q_heads, head_dim, kv_len, n_kv_heads,
                                                              n_split))


def attn_verify_f16(q: torch.Tensor, cache: KVCacheF16, kv_len: int, q_pos0: int, softmax_scale: float,
                    out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, n_split: int = 0,
                    stream=None) -> torch.Tensor:
    """Verify attention of fp32 q [T][Hq][hd] over an fp16 pool; returns fp32 [T][Hq][hd]."""
    _need(q, "q", torch.float32)
    n_rows, n_q_heads, head_dim = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float32)
    if workspace is None:
        nbytes = attn_verify_f16_workspace_bytes(n_rows, n_q_heads, head_dim, kv_len, cache.n_kv_heads, n_split)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = load_library().attn_verify_f16(_ptr(q), n_rows, n_q_heads, ctypes.byref(cache.struct()), int(kv_len),
                                        int(q_pos0), float(softmax_scale), _ptr(out), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), int(n_split), _stream(stream))
    _check("attn_verify_f16", st)
    return out


def attn_prompt_f16(q: torch.Tensor, cache: KVCacheF16, kv_len: int, q_pos0: int, softmax_scale: float,
                    out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """Prompt-chunk attention of fp16 q [n_q][Hq][hd] over an fp16 pool; returns fp32 [n_q][Hq][hd]."""
    _need(q, "q", torch.float16)
    n_q, n_q_heads, head_dim = q.shape
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    if workspace is None:
        nbytes = attn_prompt_f16_workspace_bytes(n_q, n_q_heads, head_dim, kv_len, q_pos0, cache.n_kv_heads)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = load_library().attn_prompt_f16(_ptr(q), n_q, n_q_heads, ctypes.byref(cache.struct()), int(kv_len),
                                        int(q_pos0), float(softmax_scale), _ptr(out), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream))
    _check("attn_prompt_f16", st)
    return out


def kvq8_quantize(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, pos0: int, stream=None) -> None:
    _need(x, "x", torch.float32)
    _need(codes, "codes", torch.int8)
    _need(scales, "scales", torch.float16)
    n_tok, n_kv_heads, head_dim = x.shape
    capacity = codes.shape[1]
    st = load_library().kvq8_quantize(_ptr(x), n_tok, n_kv_heads, head_dim, _ptr(codes), _ptr(scales),
                                      capacity, int(pos0), _stream(stream))
    _check("kvq8_quantize", st)


def kvq8_append(k: torch.Tensor, v: torch.Tensor, cache: "KVCacheQ8", pos0: int, stream=None) -> None:
    """Quantise K and V values [n_tok][n_kv_heads][head_dim] (fp32) into both planes of
    `cache` at positions pos0.. in one launch."""
    _need(k, "k", torch.float32)
    _need(v, "v", torch.float32)
    if k.shape != v.shape or k.dim() != 3 or k.shape[1:] != (cache.n_kv_heads, cache.head_dim):
        raise ValueError(f"k and v must both be [n_tok][{cache.n_kv_heads}][{cache.head_dim}]")
    st = load_library().kvq8_append(_ptr(k), _ptr(v), k.shape[0], ctypes.byref(cache.struct()), int(pos0),
                                    _stream(stream))
    _check("kvq8_append", st)


def attn_verify_q8_workspace_bytes(n_rows: int, n_q_heads: int, head_dim: int, kv_len: int, n_kv_heads: int,
                                   n_split: int = 0) -> int:
    return int(load_library().attn_verify_q8_workspace_bytes(n_rows, n_q_heads, head_dim, kv_len, n_kv_heads,
                                                             n_split))


def attn_verify_q8(q: torch.Tensor, cache: KVCacheQ8, kv_len: int, q_pos0: int, softmax_scale: float,
                   out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, n_split: int = 0,
                   stream=None) -> torch.Tensor:
    """Verify attention of fp32 q [T][Hq][hd] over the cache; returns fp32 [T][Hq][hd]."""
    _need(q, "q", torch.float32)
    n_rows, n_q_heads, head_dim = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float32)
    if workspace is None:
        nbytes = attn_verify_q8_workspace_bytes(n_rows, n_q_heads, head_dim, kv_len, cache.n_kv_heads, n_split)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = load_library().attn_verify_q8(_ptr(q), n_rows, n_q_heads, ctypes.byref(cache.struct()), int(kv_len),
                                       int(q_pos0), float(softmax_scale), _ptr(out), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), int(n_split), _stream(stream))
    _check("attn_verify_q8", st)
    return out


def attn_verify_tree_q8(q: torch.Tensor, cache: KVCacheQ8, kv_len: int, q_pos0: int, window_mask: torch.Tensor,
                        softmax_scale: float, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        n_split: int = 0, stream=None) -> torch.Tensor:
    """Verify attention of a tree-shaped window: fp32 q [T][Hq][hd]; window_mask int32 [T] on
    the device, bit j of row i's word = row i sees key q_pos0 + j (keys before q_pos0 are
    always visible).  Returns fp32 [T][Hq][hd]."""
    _need(q, "q", torch.float32)
    _need(window_mask, "window_mask", torch.int32)
    n_rows, n_q_heads, head_dim = q.shape
    if window_mask.shape != (n_rows,):
        raise ValueError(f"window_mask must hold one word per row ({n_rows})")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float32)
    if workspace is None:
        nbytes = attn_verify_q8_workspace_bytes(n_rows, n_q_heads, head_dim, kv_len, cache.n_kv_heads, n_split)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = load_library().attn_verify_tree_q8(_ptr(q), n_rows, n_q_heads, ctypes.byref(cache.struct()), int(kv_len),
                                            int(q_pos0), _ptr(window_mask), float(softmax_scale), _ptr(out),
                                            _ptr(workspace), workspace.numel() * workspace.element_size(),
                                            int(n_split), _stream(stream))
    _check("attn_verify_tree_q8", st)
    return out


def attn_verify_q8_partials_count(n_rows: int, n_q_heads: int, head_dim: int, kv_len: int, n_kv_heads: int,
                                  n_split: int = 0) -> int:
    return int(load_library().attn_verify_q8_partials_count(n_rows, n_q_heads, head_dim, kv_len, n_kv_heads,
                                                            n_split))


def attn_verify_q8_partials(q: torch.Tensor, cache: KVCacheQ8, kv_len: int, q_pos0: int, softmax_scale: float,
                            n_split: int = 0, part_o: torch.Tensor | None = None,
                            part_ml: torch.Tensor | None = None, stream=None):
    """Per-slice partials of verify attention of fp32 q [T][Hq][hd] over cache positions
    [0, kv_len), row i seeing positions <= q_pos0 + i (q_pos0 may be negative).  Returns
    (part_o fp32 [n][T*Hq][hd], part_ml fp32 [n][T*Hq][2]) in attn_combine's layout."""
    _need(q, "q", torch.float32)
    n_rows, n_q_heads, head_dim = q.shape
    n = attn_verify_q8_partials_count(n_rows, n_q_heads, head_dim, kv_len, cache.n_kv_heads, n_split)
    if n <= 0:
        raise KVQ8Error("attn_verify_q8_partials_count", KVQ8_ERR_INVALID_ARG)
    rows = n_rows * n_q_heads
    if part_o is None:
        part_o = torch.empty((n, rows, head_dim), dtype=torch.float32, device=q.device)
    if part_ml is None:
        part_ml = torch.empty((n, rows, 2), dtype=torch.float32, device=q.device)
    _need(part_o, "part_o", torch.float32)
    _need(part_ml, "part_ml", torch.float32)
    if part_o.shape != (n, rows, head_dim) or part_ml.shape != (n, rows, 2):
        raise ValueError(f"part_o / part_ml must be [{n}][{rows}][{head_dim}] / [{n}][{rows}][2]")
    st = load_library().attn_verify_q8_partials(_ptr(q), n_rows, n_q_heads, ctypes.byref(cache.struct()), int(kv_len),
                                                int(q_pos0), float(softmax_scale), _ptr(part_o), _ptr(part_ml),
                                                int(n_split), _stream(stream))
    _check("attn_verify_q8_partials", st)
    return part_o, part_ml


def attn_verify_append_q8_workspace_bytes(n_rows: int, n_q_heads: int, head_dim: int, q_pos0: int,
                                          n_kv_heads: int, n_split: int = 0) -> int:
    return int(load_library().attn_verify_append_q8_workspace_bytes(n_rows, n_q_heads, head_dim, q_pos0,
                                                                    n_kv_heads, n_split))


def attn_verify_append_q8(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, cache: KVCacheQ8, q_pos0: int,
                          softmax_scale: float, out: torch.Tensor | None = None,
                          workspace: torch.Tensor | None = None, n_split: int = 0, stream=None) -> torch.Tensor:
    """Append the window's fp32 keys and values [T][Hkv][hd] to the cache at q_pos0.. and run
    verify attention of fp32 q [T][Hq][hd] over q_pos0 + T keys, in one call; returns fp32
    [T][Hq][hd]."""
    _need(q, "q", torch.float32)
    _need(k_new, "k_new", torch.float32)
    _need(v_new, "v_new", torch.float32)
    n_rows, n_q_heads, head_dim = q.shape
    if k_new.shape != v_new.shape or k_new.shape != (n_rows, cache.n_kv_heads, cache.head_dim):
        raise ValueError(f"k_new and v_new must both be [{n_rows}][{cache.n_kv_heads}][{cache.head_dim}]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float32)
    if workspace is None:
        nbytes = attn_verify_append_q8_workspace_bytes(n_rows, n_q_heads, head_dim, q_pos0, cache.n_kv_heads,
                                                       n_split)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = load_library().attn_verify_append_q8(_ptr(q), _ptr(k_new), _ptr(v_new), n_rows, n_q_heads,
                                              ctypes.byref(cache.struct()), int(q_pos0), float(softmax_scale),
                                              _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                              int(n_split), _stream(stream))
    _check("attn_verify_append_q8", st)
    return out


def attn_verify_append_q8_host_scratch_bytes(n_rows: int, n_q_heads: int, head_dim: int, q_pos0: int,
                                             n_kv_heads: int, n_split: int = 0) -> int:
    return int(load_library().attn_verify_append_q8_host_scratch_bytes(n_rows, n_q_heads, head_dim, q_pos0,
                                                                       n_kv_heads, n_split))


def attn_verify_append_q8_host(h_in: torch.Tensor, n_rows: int, n_q_heads: int, cache: KVCacheQ8, q_pos0: int,
                               softmax_scale: float, h_out: torch.Tensor, scratch: torch.Tensor, n_split: int = 0,
                               stream=None) -> None:
    """attn_verify_append_q8 from and to host tensors: h_in (CPU fp32) holds q [T][Hq][hd] then
    k_new and v_new [T][Hkv][hd]; h_out (CPU fp32 [T][Hq][hd]) is written once the stream gets
    there.  Pinned tensors are read by a copy kernel and written in place by the merge;
    pageable ones go through copy-engine transfers.  scratch: device bytes from the
    scratch-size query."""
    for t, name in ((h_in, "h_in"), (h_out, "h_out")):
        if t.device.type != "cpu" or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU float32 tensor")
    hd, hkv = cache.head_dim, cache.n_kv_heads
    if h_in.numel() != n_rows * (n_q_heads + 2 * hkv) * hd or h_out.numel() != n_rows * n_q_heads * hd:
        raise ValueError("h_in / h_out sizes do not match the shape")
    if scratch.device.type != "cuda" or not scratch.is_contiguous():
        raise ValueError("scratch must be a contiguous device tensor")
    st = load_library().attn_verify_append_q8_host(h_in.data_ptr(), n_rows, n_q_heads, ctypes.byref(cache.struct()),
                                                   int(q_pos0), float(softmax_scale), h_out.data_ptr(),
                                                   _ptr(scratch), scratch.numel() * scratch.element_size(),
                                                   int(n_split), _stream(stream))
    _check("attn_verify_append_q8_host", st)


class PreparedAppendVerifyHost:
    """attn_verify_append_q8_host with its arguments marshalled once, for a loop that repeats
    one call (same buffers, cache and window position): calling it is one C-ABI call.  The
    tensors must stay alive and in place while the object is used."""

    def __init__(self, h_in: torch.Tensor, n_rows: int, n_q_heads: int, cache: KVCacheQ8, q_pos0: int,
                 softmax_scale: float, h_out: torch.Tensor, scratch: torch.Tensor, n_split: int = 0, stream=None):
        for t, name in ((h_in, "h_in"), (h_out, "h_out")):
            if t.device.type != "cpu" or t.dtype != torch.float32 or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CPU float32 tensor")
        hd, hkv = cache.head_dim, cache.n_kv_heads
        if h_in.numel() != n_rows * (n_q_heads + 2 * hkv) * hd or h_out.numel() != n_rows * n_q_heads * hd:
            raise ValueError("h_in / h_out sizes do not match the shape")
        if scratch.device.type != "cuda" or not scratch.is_contiguous():
            raise ValueError("scratch must be a contiguous device tensor")
        self._keep = (h_in, h_out, scratch, cache)
        self._struct = cache.struct()
        self._fn = load_library().attn_verify_append_q8_host
        self._args = (ctypes.c_void_p(h_in.data_ptr()), ctypes.c_int(n_rows), ctypes.c_int(n_q_heads),
                      ctypes.byref(self._struct), ctypes.c_int(int(q_pos0)), ctypes.c_float(float(softmax_scale)),
                      ctypes.c_void_p(h_out.data_ptr()), _ptr(scratch),
                      ctypes.c_size_t(scratch.numel() * scratch.element_size()), ctypes.c_int(int(n_split)),
                      _stream(stream))

    def __call__(self) -> None:
        st = self._fn(*self._args)
        if st != KVQ8_OK:
            raise KVQ8Error("attn_verify_append_q8_host", st)


def argmax_rows_top_prob(logits: torch.Tensor, workspace: torch.Tensor | None = None, argmax=None, top_prob=None,
                         stream=None):
    """Verify-head acceptance over fp32 logits [T][V] on the device: returns (argmax int32 [T],
    top_prob fp32 [T]) -- the first index of each row's maximum and softmax(row) there."""
    _need(logits, "logits", torch.float32)
    if logits.dim() != 2:
        raise ValueError("logits must be [T][V]")
    n_rows, vocab = logits.shape
    if argmax is None:
        argmax = torch.empty(n_rows, dtype=torch.int32, device=logits.device)
    if top_prob is None:
        top_prob = torch.empty(n_rows, dtype=torch.float32, device=logits.device)
    _need(argmax, "argmax", torch.int32)
    _need(top_prob, "top_prob", torch.float32)
    lib = load_library()
    if workspace is None:
        workspace = torch.empty(max(int(lib.argmax_rows_top_prob_workspace_bytes(n_rows, vocab)), 16),
                                dtype=torch.uint8, device=logits.device)
    st = lib.argmax_rows_top_prob(_ptr(logits), n_rows, vocab, _ptr(argmax), _ptr(top_prob), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    _check("argmax_rows_top_prob", st)
    return argmax, top_prob


def kvq8_selftest_convert(kind: int, words: torch.Tensor, stream=None) -> torch.Tensor:
    """Run the kernels' code -> fp16 conversion `kind` (0-3, see the header) over int32 words on the
    device; returns the fp16 pairs as int32 words (2 per input word for kinds 0 and 1, 4 for 2 and 3)."""
    _need(words, "words", torch.int32)
    n = words.numel()
    out = torch.empty(n * (2 if kind in (0, 1) else 4), dtype=torch.int32, device=words.device)
    st = load_library().kvq8_selftest_convert(int(kind), _ptr(words), _ptr(out), n, _stream(stream))
    _check("kvq8_selftest_convert", st)
    return out


def kvq8_selftest_wait_timeout(polls: int = 4096, stream=None) -> None:
    """One launch whose bounded wait on a barrier that nothing arrives on gives up after `polls`
    polls and sets the device error flag (read it with kvq8_device_error)."""
    st = load_library().kvq8_selftest_wait_timeout(int(polls), _stream(stream))
    _check("kvq8_selftest_wait_timeout", st)


def attn_combine(part_o: torch.Tensor, part_ml: torch.Tensor, out: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """Merge partials part_o [n_split][rows][hd], part_ml [n_split][rows][2] -> out [rows][hd] (fp32)."""
    _need(part_o, "part_o", torch.float32)
    _need(part_ml, "part_ml", torch.float32)
    n_split, rows, head_dim = part_o.shape
    if out is None:
        out = torch.empty((rows, head_dim), dtype=torch.float32, device=part_o.device)
    _need(out, "out", torch.float32)
    st = load_library().attn_combine(_ptr(part_o), _ptr(part_ml), n_split, rows, head_dim, _ptr(out),
                                     _stream(stream))
    _check("attn_combine", st)
    return out


def attn_prompt_q8_workspace_bytes(n_q: int, n_q_heads: int, head_dim: int, kv_len: int, q_pos0: int,
                                   n_kv_heads: int) -> int:
    return int(load_library().attn_prompt_q8_workspace_bytes(n_q, n_q_heads, head_dim, kv_len, q_pos0, n_kv_heads))


def attn_prompt_f16_workspace_bytes(n_q: int, n_q_heads: int, head_dim: int, kv_len: int, q_pos0: int,
                                    n_kv_heads: int) -> int:
    return int(load_library().attn_prompt_f16_workspace_bytes(n_q, n_q_heads, head_dim, kv_len, q_pos0, n_kv_heads))


def attn_prompt_q8(q: torch.Tensor, cache: KVCacheQ8, kv_len: int, q_pos0: int, softmax_scale: float,
                   out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """Prompt-chunk attention of fp16 q [n_q][Hq][hd] over the cache; returns fp32 [n_q][Hq][hd]."""
    _need(q, "q", torch.float16)
    n_q, n_q_heads, head_dim = q.shape
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32)
    if workspace is None:
        nbytes = attn_prompt_q8_workspace_bytes(n_q, n_q_heads, head_dim, kv_len, q_pos0, cache.n_kv_heads)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = load_library().attn_prompt_q8(_ptr(q), n_q, n_q_heads, ctypes.byref(cache.struct()), int(kv_len),
                                       int(q_pos0), float(softmax_scale), _ptr(out), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream))
    _check("attn_prompt_q8", st)
    return out


def attn_verify_q8_noalloc(q: torch.Tensor, cache: KVCacheQ8, kv_len: int, q_pos0: int, softmax_scale: float,
                           out: torch.Tensor | None = None, n_split: int = 0, stream=None) -> torch.Tensor:
    """attn_verify_q8 without a workspace, for callers that cannot allocate device memory at
    call time: the library keeps the split partials in its own static device array.  The
    first call on a device must come before any stream capture; calls that overlap on the
    GPU share that array and must be serialised by the caller.  `out` must be given by such
    callers (it is only allocated here when omitted, as a convenience)."""
    _need(q, "q", torch.float32)
    n_rows, n_q_heads, _ = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float32)
    st = load_library().attn_verify_q8_noalloc(_ptr(q), n_rows, n_q_heads, ctypes.byref(cache.struct()),
                                               int(kv_len), int(q_pos0), float(softmax_scale), _ptr(out),
                                               int(n_split), _stream(stream))
    _check("attn_verify_q8_noalloc", st)
    return out
