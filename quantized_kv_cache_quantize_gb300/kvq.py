"""Thin Python binding of libkvq (ctypes).  Argument marshalling only: every
step of the computation runs in the library's CUDA kernels; torch is used for
device memory and streams.  There is no CPU fallback: if libkvq.so is missing
the first call raises."""
from __future__ import annotations

import contextlib
import ctypes
import functools
import math
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVQ_LIBRARY selects another build of the same C ABI, e.g. the checked
# build (libkvq_checked.so, index checks in every kernel)
LIB_PATH = os.environ.get("KVQ_LIBRARY") or os.path.join(_HERE, "libkvq.so")

KVQ_OK = 0
KVQ_ERR_INVALID_ARG = 1
KVQ_ERR_UNSUPPORTED = 2
KVQ_ERR_CAPACITY = 3
KVQ_ERR_CUDA = 4
KVQ_ERR_TIMEOUT = 5
KVQ_ERR_ALIGNMENT = 6
KVQ_ERR_TOO_LARGE = 7
KVQ_ERR_RANGE = 8
KVQ_ERR_BOUNDS = 9
NOALLOC_SCRATCH_BYTES = 32 << 20

KEYS_PER_TOKEN = 0
KEYS_PER_CHANNEL = 1
KEY_BLOCK = 128

CORR_NONE = 0
CORR_TAYLOR = 1
CORR_EXACT = 2
FLAG_PRECISE_QUERY = 1
FLAG_NO_KV_SPLIT = 2
FLAG_ONE_CTA = 4
FLAG_STAGED_WORDS = 8


class KVQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class CacheStruct(ctypes.Structure):
    """Mirror of ``kvq_cache`` in include/kvq.h."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("bits", ctypes.c_int32), ("group", ctypes.c_int32),
        ("chunk_tokens", ctypes.c_int32), ("n_chunks", ctypes.c_int32),
        ("len", ctypes.c_int32), ("head_slot", ctypes.c_int32),
        ("sign_bits", ctypes.c_uint32 * 4),
        ("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
        ("k_sz", ctypes.c_void_p), ("v_sz", ctypes.c_void_p),
        ("key_mode", ctypes.c_int32),
    ]


_P = ctypes.c_void_p
_SIGNATURES = {
    "kvq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kvq_abi_version": (ctypes.c_int32, []),
    "kvq_cache_bytes": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_size_t),
                                       ctypes.POINTER(ctypes.c_size_t)]),
    "kvq_cache_meta_bytes": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_size_t),
                                            ctypes.POINTER(ctypes.c_size_t)]),
    "kvq_quantize_append": (ctypes.c_int, [_P, _P, _P, ctypes.c_int32, _P]),
    "kvq_workspace_bytes": (ctypes.c_size_t, [_P, ctypes.c_int32, ctypes.c_int32]),
    "kvq_attention_corrected": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.c_float, ctypes.c_int32, ctypes.c_int32, _P,
                                               ctypes.c_size_t, _P, _P, _P, _P]),
    "kvq_attention_mass": (ctypes.c_int, [_P, _P, _P, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_float, ctypes.c_int32, ctypes.c_int32, _P,
                                          ctypes.c_size_t, _P, _P, _P]),
    "kvq_rotate": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P, _P]),
    "kvq_last_device_status": (ctypes.c_int, [_P]),
    "kvq_debug_bounds_site": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32), _P]),
    "kvq_debug_bounds_build": (ctypes.c_int32, []),
    "kvq_profile_kernel_launches": (ctypes.c_int64, []),
    "kvq_set_wait_limit_ns": (ctypes.c_int, [ctypes.c_uint64]),
    "kvq_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint64, _P]),
    "kvq_attention_corrected_noalloc": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int32,
                                                       ctypes.c_int32, ctypes.c_float,
                                                       ctypes.c_int32, ctypes.c_int32, _P, _P, _P,
                                                       _P]),
    "kvq_profile_begin": (ctypes.c_int, []),
    "kvq_profile_end": (ctypes.c_int, [_P, _P]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libkvq.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkvq.so not built ({LIB_PATH}); run __graft_entry__.build()")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib = h
    return _lib


def _nvtx(name: str):
    """Mark each call of the decorated entry point as an NVTX range (for
    Nsight timelines and ncu --nvtx filters); host-side only."""
    def deco(fn):
        @functools.wraps(fn)
        def wrapped(*args, **kwargs):
            if not torch.cuda.is_available():
                return fn(*args, **kwargs)
            torch.cuda.nvtx.range_push(name)
            try:
                return fn(*args, **kwargs)
            finally:
                torch.cuda.nvtx.range_pop()
        return wrapped
    return deco


def status_string(status: int) -> str:
    return lib().kvq_status_string(status).decode()


def _check(status: int, what: str):
    if status != KVQ_OK:
        raise KVQError(status, what)


def _stream(stream, device=None) -> ctypes.c_void_p:
    """The stream handle for a call on ``device``: torch's current stream of
    that device when none is given; a torch stream of another device is
    refused (its kernels would run on the wrong GPU)."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif device is not None and getattr(stream, "device", device) != device:
        raise ValueError(f"stream belongs to {stream.device}, the call's tensors to {device}")
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _on_device(device):
    """Make ``device`` the current CUDA device for the duration of a call.
    The library launches on the current device and looks its status word and
    scratch up there, so a call whose tensors live on another GPU than the
    current one must switch first.  No-op for host tensors (shape checks)."""
    if device is None or device.type != "cuda":
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def sign_bits(signs) -> list[int]:
    """Bit c of word c // 32 set where sigma_c = -1."""
    s = np.asarray(signs).reshape(-1)
    words = [0, 0, 0, 0]
    for c, v in enumerate(s):
        if v < 0:
            words[c >> 5] |= 1 << (c & 31)
    return words


def _bf16_dev(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    return t


def _check_bhnd(cache: "KVCache", t: torch.Tensor, name: str) -> int:
    """The library reads [batch, heads, n, head_dim] rows of the cache's
    geometry from a plain device pointer and cannot see the buffer's size, so
    the tensor's shape is checked here, before its pointer is passed on.
    Returns n."""
    want = (cache.batch, cache.heads, cache.head_dim)
    if t.dim() != 4 or (t.shape[0], t.shape[1], t.shape[3]) != want:
        raise ValueError(f"{name} must have shape [{want[0]}, {want[1]}, n, {want[2]}] "
                         f"(the cache's batch, heads and head_dim), got {list(t.shape)}")
    return int(t.shape[2])


def _check_device(cache: "KVCache", *tensors):
    dev = cache.k_codes.device
    for name, t in tensors:
        if t is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the cache on {dev}")


def _check_out(q: torch.Tensor, out: torch.Tensor):
    if tuple(out.shape) != tuple(q.shape):
        raise ValueError(f"out must have the shape of q {list(q.shape)}, got {list(out.shape)}")
    _bf16_dev(out, "out")


def _check_qkv(cache: "KVCache", q, k_cur, v_cur) -> tuple:
    """Shapes, then dtype and device, of the attention inputs; returns
    (n_q, n_r)."""
    n_q = _check_bhnd(cache, q, "q")
    n_r = _check_bhnd(cache, k_cur, "k_cur")
    if v_cur is not None and tuple(v_cur.shape) != tuple(k_cur.shape):
        raise ValueError(f"v_cur must have the shape of k_cur {list(k_cur.shape)}, "
                         f"got {list(v_cur.shape)}")
    _bf16_dev(q, "q")
    _bf16_dev(k_cur, "k_cur")
    if v_cur is not None:
        _bf16_dev(v_cur, "v_cur")
    _check_device(cache, ("q", q), ("k_cur", k_cur), ("v_cur", v_cur))
    return n_q, n_r


def _workspace_arg(workspace: torch.Tensor, device) -> tuple:
    if not workspace.is_contiguous() or workspace.device != device:
        raise ValueError(f"workspace must be a contiguous tensor on {device}")
    return _ptr(workspace), workspace.numel() * workspace.element_size()


class KVCache:
    """A quantized sliding-window KV cache in device memory (torch-allocated)
    and its ``kvq_cache`` descriptor."""

    def __init__(self, batch: int, heads: int, head_dim: int, bits: int, group: int,
                 chunk_tokens: int, n_chunks: int, signs, device="cuda",
                 key_mode: int = KEYS_PER_TOKEN):
        c = CacheStruct()
        c.batch, c.heads, c.head_dim = batch, heads, head_dim
        c.bits, c.group = bits, group
        c.chunk_tokens, c.n_chunks = chunk_tokens, n_chunks
        c.len, c.head_slot = 0, 0
        c.key_mode = key_mode
        for i, w in enumerate(sign_bits(signs)):
            c.sign_bits[i] = w
        codes_b, sz_b = ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib().kvq_cache_bytes(ctypes.byref(c), ctypes.byref(codes_b), ctypes.byref(sz_b)),
               "kvq_cache_bytes")
        k_b, v_b = ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib().kvq_cache_meta_bytes(ctypes.byref(c), ctypes.byref(k_b), ctypes.byref(v_b)),
               "kvq_cache_meta_bytes")
        self.signs = np.asarray(signs, dtype=np.float32)
        self.k_codes = torch.zeros(codes_b.value, dtype=torch.uint8, device=device)
        self.v_codes = torch.zeros(codes_b.value, dtype=torch.uint8, device=device)
        self.k_sz = torch.zeros(k_b.value // 2, dtype=torch.int16, device=device)
        self.v_sz = torch.zeros(v_b.value // 2, dtype=torch.int16, device=device)
        c.k_codes, c.v_codes = self.k_codes.data_ptr(), self.v_codes.data_ptr()
        c.k_sz, c.v_sz = self.k_sz.data_ptr(), self.v_sz.data_ptr()
        self.struct = c

    # geometry
    batch = property(lambda self: self.struct.batch)
    heads = property(lambda self: self.struct.heads)
    head_dim = property(lambda self: self.struct.head_dim)
    bits = property(lambda self: self.struct.bits)
    group = property(lambda self: self.struct.group)
    chunk_tokens = property(lambda self: self.struct.chunk_tokens)
    n_chunks = property(lambda self: self.struct.n_chunks)
    capacity = property(lambda self: self.struct.chunk_tokens * self.struct.n_chunks)
    len = property(lambda self: self.struct.len)
    head_slot = property(lambda self: self.struct.head_slot)

    def codes_view(self, which: str) -> torch.Tensor:
        t = self.k_codes if which == "k" else self.v_codes
        return t.view(self.batch, self.heads, self.capacity, self.head_dim * self.bits // 8)

    key_mode = property(lambda self: self.struct.key_mode)

    def sz_view(self, which: str) -> torch.Tensor:
        """(step, zero) as int16 BF16 bits: [B, H, capacity, d / group, 2], or
        for per-channel keys [B, H, n_chunks, blocks per chunk, d, 2]."""
        if which == "k" and self.key_mode == KEYS_PER_CHANNEL:
            bpc = (self.chunk_tokens + KEY_BLOCK - 1) // KEY_BLOCK
            return self.k_sz.view(self.batch, self.heads, self.n_chunks, bpc, self.head_dim, 2)
        t = self.k_sz if which == "k" else self.v_sz
        return t.view(self.batch, self.heads, self.capacity, self.head_dim // self.group, 2)

    def workspace_bytes(self, n_q: int, n_r: int) -> int:
        return int(lib().kvq_workspace_bytes(ctypes.byref(self.struct), n_q, n_r))


@_nvtx("kvq_quantize_append")
def quantize_append(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
    """kvq_quantize_append: k_new/v_new [B, H, n_new, d] bf16 on the device."""
    n_new = _check_bhnd(cache, k_new, "k_new")
    if tuple(k_new.shape) != tuple(v_new.shape):
        raise ValueError("k_new and v_new shapes differ")
    _bf16_dev(k_new, "k_new")
    _bf16_dev(v_new, "v_new")
    _check_device(cache, ("k_new", k_new), ("v_new", v_new))
    dev = cache.k_codes.device
    with _on_device(dev):
        _check(lib().kvq_quantize_append(ctypes.byref(cache.struct), _ptr(k_new), _ptr(v_new),
                                         n_new, _stream(stream, dev)), "kvq_quantize_append")


@_nvtx("kvq_attention_corrected")
def attention_corrected(cache: KVCache, q, k_cur, v_cur, scale: float | None = None,
                        corr: int = CORR_TAYLOR, out=None, with_mass: bool = False,
                        workspace=None, stream=None, flags: int = 0):
    """kvq_attention_corrected.  q [B, H, n_q, d], k_cur/v_cur [B, H, n_r, d]
    bf16 on the device.  Returns out (and (p_s, p_r) when with_mass)."""
    n_q, n_r = _check_qkv(cache, q, k_cur, v_cur)
    d = cache.head_dim
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if out is None:
        out = torch.empty_like(q)
    _check_out(q, out)
    _check_device(cache, ("out", out))
    ps = pr = None
    if with_mass:
        ps = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
        pr = torch.empty_like(ps)
    with _on_device(q.device):
        # the workspace size depends on the device's SM count
        ws_bytes = cache.workspace_bytes(n_q, n_r)
        if workspace is None:
            workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
        ws_ptr, ws_size = _workspace_arg(workspace, q.device)
        _check(lib().kvq_attention_corrected(
            ctypes.byref(cache.struct), _ptr(q), _ptr(k_cur), _ptr(v_cur), n_q, n_r,
            ctypes.c_float(scale), corr, flags, ws_ptr, ws_size, _ptr(out),
            _ptr(ps), _ptr(pr), _stream(stream, q.device)), "kvq_attention_corrected")
    return (out, ps, pr) if with_mass else out


@_nvtx("kvq_attention_corrected_noalloc")
def attention_corrected_noalloc(cache: KVCache, q, k_cur, v_cur, scale: float | None = None,
                                corr: int = CORR_TAYLOR, out=None, with_mass: bool = False,
                                stream=None, flags: int = 0):
    """kvq_attention_corrected_noalloc: like attention_corrected, with the
    library's built-in scratch buffer instead of a workspace (for callers
    that cannot allocate device memory when they call).  Outputs are still
    the caller's (allocated here by torch when not given)."""
    n_q, n_r = _check_qkv(cache, q, k_cur, v_cur)
    scale = 1.0 / math.sqrt(cache.head_dim) if scale is None else scale
    if out is None:
        out = torch.empty_like(q)
    _check_out(q, out)
    _check_device(cache, ("out", out))
    ps = pr = None
    if with_mass:
        ps = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
        pr = torch.empty_like(ps)
    with _on_device(q.device):
        _check(lib().kvq_attention_corrected_noalloc(
            ctypes.byref(cache.struct), _ptr(q), _ptr(k_cur), _ptr(v_cur), n_q, n_r,
            ctypes.c_float(scale), corr, flags, _ptr(out), _ptr(ps), _ptr(pr),
            _stream(stream, q.device)), "kvq_attention_corrected_noalloc")
    return (out, ps, pr) if with_mass else out


@_nvtx("kvq_attention_mass")
def attention_mass(cache: KVCache, q, k_cur, scale: float | None = None,
                   corr: int = CORR_TAYLOR, workspace=None, stream=None, flags: int = 0):
    """kvq_attention_mass: returns (p_s, p_r), each [B, H, n_q] fp32."""
    n_q, n_r = _check_qkv(cache, q, k_cur, None)
    scale = 1.0 / math.sqrt(cache.head_dim) if scale is None else scale
    ps = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    pr = torch.empty_like(ps)
    with _on_device(q.device):
        ws_bytes = cache.workspace_bytes(n_q, n_r)
        if workspace is None:
            workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
        ws_ptr, ws_size = _workspace_arg(workspace, q.device)
        _check(lib().kvq_attention_mass(
            ctypes.byref(cache.struct), _ptr(q), _ptr(k_cur), n_q, n_r, ctypes.c_float(scale),
            corr, flags, ws_ptr, ws_size, _ptr(ps), _ptr(pr), _stream(stream, q.device)),
            "kvq_attention_mass")
    return ps, pr


@_nvtx("kvq_rotate")
def rotate(x: torch.Tensor, signs, out_dtype=torch.float32, stream=None) -> torch.Tensor:
    """kvq_rotate: x [..., d] bf16 -> H x in fp32 (the values the quantizer
    sees) or fp16 (the attention kernel's tensor-core operands)."""
    _bf16_dev(x, "x")
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    out = torch.empty(x.shape, dtype=out_dtype, device=x.device)
    sb = (ctypes.c_uint32 * 4)(*sign_bits(signs))
    if out_dtype not in (torch.float32, torch.float16):
        raise ValueError("out_dtype must be float32 or float16")
    f32 = out if out_dtype == torch.float32 else None
    f16 = out if out_dtype == torch.float16 else None
    with _on_device(x.device):
        _check(lib().kvq_rotate(_ptr(x), rows, d, sb, _ptr(f32), _ptr(f16),
                                _stream(stream, x.device)), "kvq_rotate")
    return out


def last_device_status(stream=None, device=None) -> int:
    """kvq_last_device_status on ``device`` (default: the current device)."""
    dev = None if device is None else torch.device(device)
    with _on_device(dev):
        return int(lib().kvq_last_device_status(_stream(stream, dev)))


def debug_bounds_site(stream=None, device=None) -> int:
    """kvq_debug_bounds_site: the source line of the first failed index
    check of the checked build since the last call (0: none)."""
    dev = None if device is None else torch.device(device)
    line = ctypes.c_int32(0)
    with _on_device(dev):
        _check(lib().kvq_debug_bounds_site(ctypes.byref(line), _stream(stream, dev)),
               "kvq_debug_bounds_site")
    return int(line.value)


def debug_bounds_build() -> bool:
    """True when the loaded library is the checked build."""
    return bool(lib().kvq_debug_bounds_build())


def set_wait_limit_ns(limit_ns: int):
    _check(lib().kvq_set_wait_limit_ns(int(limit_ns)), "kvq_set_wait_limit_ns")


def selftest_wait_timeout(limit_ns: int, stream=None):
    _check(lib().kvq_selftest_wait_timeout(int(limit_ns), _stream(stream)),
           "kvq_selftest_wait_timeout")


def profile_begin():
    """Start recording CUDA events around every libkvq kernel launch."""
    _check(lib().kvq_profile_begin(), "kvq_profile_begin")


def profile_kernel_launches() -> int:
    """Kernels launched by the library since profile_begin (while recording)."""
    return int(lib().kvq_profile_kernel_launches())


def profile_end() -> dict:
    """Stop recording; per kernel kind, summed device ms and launch count."""
    ms = (ctypes.c_double * 3)()
    n = (ctypes.c_int32 * 3)()
    _check(lib().kvq_profile_end(ms, n), "kvq_profile_end")
    kinds = ("quantize_append", "rotate", "attention")
    return {k: {"ms_total": float(ms[i]), "launches": int(n[i])} for i, k in enumerate(kinds)}
