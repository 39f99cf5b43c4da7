"""Thin ctypes binding of the C ABI declared in include/h2o.h.

Functions keep the ABI's names and only marshal arguments: torch tensors
become device pointers, the current torch stream becomes the cudaStream_t,
and non-zero status codes become H2OError with the library's message.  Every
computation runs in the CUDA library; if it is missing this module raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import _build

H2O_F16, H2O_F32 = 0, 1
H2O_DECODE_WARP_PER_PAIR = -1  # h2o_cache_set_decode_shape: one warp per pair
STATUS = {0: "H2O_OK", -1: "H2O_EINVAL", -2: "H2O_ENOMEM", -3: "H2O_ECUDA", -4: "H2O_ESTATE", -5: "H2O_EDEVICE"}
HEADER_INTS = 16
MAGIC = 0x48324F31

_lib = None
_lock = threading.Lock()

# every function declared in include/h2o.h: name -> (restype, argtypes)
_c_int, _c_void_p, _c_float, _c_size_t = ctypes.c_int, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "h2o_cache_create": (_c_int, [_c_int] * 6 + [ctypes.POINTER(_c_void_p)]),
    "h2o_cache_destroy": (None, [_c_void_p]),
    "h2o_prefill": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int, _c_float, _c_void_p, _c_void_p]),
    "h2o_prefill_ex": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int, _c_float, _c_void_p,
                                _c_void_p, _c_void_p, _c_void_p]),
    "h2o_prefill_ragged": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_int, _c_void_p, _c_float,
                                    _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "h2o_decode_step": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_float, _c_void_p, _c_void_p,
                                 _c_void_p]),
    "h2o_cache_reset": (_c_int, [_c_void_p, _c_void_p]),
    "h2o_cache_state_bytes": (_c_size_t, [_c_void_p]),
    "h2o_cache_export_state": (_c_int, [_c_void_p, _c_void_p, _c_size_t, _c_void_p]),
    "h2o_cache_import_state": (_c_int, [_c_void_p, _c_void_p, _c_size_t, _c_void_p]),
    "h2o_cache_check": (_c_int, [_c_void_p, _c_void_p]),
    "h2o_cache_set_decode_shape": (_c_int, [_c_void_p, _c_int, _c_int]),
    "h2o_cache_info": (_c_int, [_c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    "h2o_prefill_colsum_static": (_c_int, [_c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                           _c_void_p, _c_void_p]),
    "h2o_prefill_colsum_static_check": (_c_int, [_c_void_p]),
    "h2o_cache_set_position_rolling": (_c_int, [_c_void_p, _c_float]),
    "h2o_cache_set_rolling_digits": (_c_int, [_c_void_p, _c_int, _c_int]),
    "h2o_cache_rolling_digits": (_c_int, [_c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    "h2o_cache_set_static_pattern": (_c_int, [_c_void_p, _c_int, _c_int, _c_int]),
    "h2o_selftest_wait_timeout": (_c_int, [ctypes.c_uint, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_ulonglong)]),
    "h2o_debug_fail_alloc": (_c_int, [_c_int]),
    "h2o_last_error": (ctypes.c_char_p, []),
}


class H2OError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load the CUDA library (building it first if allowed and needed)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and _build.is_stale():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"H2O CUDA library not built: {path} (run __graft_entry__.build())")
            cdll = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(cdll, name)
                fn.restype = res
                fn.argtypes = args
            _lib = cdll
    return _lib


def _check(code: int):
    if code != 0:
        raise H2OError(code, lib().h2o_last_error().decode())


def _stream(stream):
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t, dtype=None, shape=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


class Cache:
    """Handle of an h2o_cache (freed by h2o_cache_destroy or on collection)."""

    def __init__(self, handle: int, batch, heads, head_dim, heavy, recent, kv_dtype):
        self.handle = handle
        self.batch, self.heads, self.head_dim = batch, heads, head_dim
        self.heavy, self.recent, self.kv_dtype = heavy, recent, kv_dtype

    @property
    def slots(self):
        return self.heavy + self.recent

    @property
    def pairs(self):
        return self.batch * self.heads

    def torch_dtype(self):
        import torch

        return torch.float16 if self.kv_dtype == H2O_F16 else torch.float32

    def np_dtype(self):
        return np.float16 if self.kv_dtype == H2O_F16 else np.float32

    def __del__(self):
        try:
            if self.handle and _lib is not None:
                _lib.h2o_cache_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


# ------------------------------------------------------------------ ABI functions
def h2o_cache_create(batch, heads, head_dim, heavy_budget, recent_budget, kv_dtype) -> Cache:
    out = ctypes.c_void_p()
    _check(lib().h2o_cache_create(batch, heads, head_dim, heavy_budget, recent_budget, kv_dtype, ctypes.byref(out)))
    return Cache(out.value, batch, heads, head_dim, heavy_budget, recent_budget, kv_dtype)


def h2o_cache_destroy(cache: Cache):
    if cache is not None and cache.handle:
        lib().h2o_cache_destroy(cache.handle)
        cache.handle = None


def h2o_prefill_ex(cache: Cache, q, k, v, scale, out=None, colsum=None, lse=None, stream=None):
    import torch

    B, H, D = cache.batch, cache.heads, cache.head_dim
    L = q.shape[2]
    dt = cache.torch_dtype()
    shp = (B, H, L, D)
    _check(lib().h2o_prefill_ex(
        cache.handle, _ptr(q, dt, shp, "q"), _ptr(k, dt, shp, "k"), _ptr(v, dt, shp, "v"), L, float(scale),
        _ptr(out, torch.float32, shp, "out"), _ptr(colsum, torch.float32, (B, H, L), "colsum"),
        _ptr(lse, torch.float32, (B, H, L), "lse"), _stream(stream)))


def h2o_prefill_ragged(cache: Cache, q, k, v, lengths, scale, out=None, colsum=None, lse=None, stream=None):
    """q, k, v: [B, H, max_len, D]; lengths: int32 CUDA tensor [B] of prompt lengths."""
    import torch

    B, H, D = cache.batch, cache.heads, cache.head_dim
    L = q.shape[2]
    dt = cache.torch_dtype()
    shp = (B, H, L, D)
    _check(lib().h2o_prefill_ragged(
        cache.handle, _ptr(q, dt, shp, "q"), _ptr(k, dt, shp, "k"), _ptr(v, dt, shp, "v"), L,
        _ptr(lengths, torch.int32, (B,), "lengths"), float(scale), _ptr(out, torch.float32, shp, "out"),
        _ptr(colsum, torch.float32, (B, H, L), "colsum"), _ptr(lse, torch.float32, (B, H, L), "lse"),
        _stream(stream)))


def h2o_prefill(cache: Cache, q, k, v, scale, out=None, stream=None):
    import torch

    B, H, D = cache.batch, cache.heads, cache.head_dim
    L = q.shape[2]
    dt = cache.torch_dtype()
    shp = (B, H, L, D)
    _check(lib().h2o_prefill(cache.handle, _ptr(q, dt, shp, "q"), _ptr(k, dt, shp, "k"), _ptr(v, dt, shp, "v"),
                             L, float(scale), _ptr(out, torch.float32, shp, "out"), _stream(stream)))


def h2o_decode_step(cache: Cache, q, k_new, v_new, scale, out, evicted=None, stream=None):
    import torch

    shp = (cache.batch, cache.heads, cache.head_dim)
    dt = cache.torch_dtype()
    _check(lib().h2o_decode_step(
        cache.handle, _ptr(q, dt, shp, "q"), _ptr(k_new, dt, shp, "k_new"), _ptr(v_new, dt, shp, "v_new"),
        float(scale), _ptr(out, torch.float32, shp, "out"),
        _ptr(evicted, torch.int32, shp[:2], "evicted"), _stream(stream)))


def h2o_cache_reset(cache: Cache, stream=None):
    _check(lib().h2o_cache_reset(cache.handle, _stream(stream)))


def h2o_cache_state_bytes(cache: Cache) -> int:
    return int(lib().h2o_cache_state_bytes(cache.handle))


def h2o_cache_export_state(cache: Cache, stream=None) -> np.ndarray:
    n = h2o_cache_state_bytes(cache)
    buf = np.empty(n, dtype=np.uint8)
    _check(lib().h2o_cache_export_state(cache.handle, buf.ctypes.data, n, _stream(stream)))
    return buf


def h2o_cache_import_state(cache: Cache, buf: np.ndarray, stream=None):
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    _check(lib().h2o_cache_import_state(cache.handle, buf.ctypes.data, buf.size, _stream(stream)))


def h2o_cache_check(cache: Cache, stream=None):
    _check(lib().h2o_cache_check(cache.handle, _stream(stream)))


def h2o_cache_set_decode_shape(cache: Cache, splits: int = 0, stages: int = 0):
    _check(lib().h2o_cache_set_decode_shape(cache.handle, splits, stages))


def h2o_cache_set_position_rolling(cache: Cache, rope_base: float):
    """Rotary embedding at positions inside the cache (0 turns it off)."""
    _check(lib().h2o_cache_set_position_rolling(cache.handle, float(rope_base)))


def h2o_cache_set_rolling_digits(cache: Cache, low_bits: int = 0, hi_bits: int = 0):
    """Digit widths of position rolling's rank decomposition (0, 0: automatic)."""
    _check(lib().h2o_cache_set_rolling_digits(cache.handle, int(low_bits), int(hi_bits)))


def h2o_cache_rolling_digits(cache: Cache) -> list[int]:
    """[low_bits, hi_bits, levels, table entries] of position rolling (zeros when off)."""
    d = (ctypes.c_int32 * 4)()
    _check(lib().h2o_cache_rolling_digits(cache.handle, d))
    return list(d)


def h2o_cache_set_static_pattern(cache: Cache, offset: int, stride: int, count: int):
    """Protect positions offset, offset + stride, ... (count of them, count <= heavy)."""
    _check(lib().h2o_cache_set_static_pattern(cache.handle, int(offset), int(stride), int(count)))


def h2o_cache_info(cache: Cache) -> list[int]:
    info = (ctypes.c_int32 * 10)()
    _check(lib().h2o_cache_info(cache.handle, info))
    return list(info)


def h2o_selftest_wait_timeout(polls: int) -> tuple[list[int], int]:
    """Run the bounded-wait self-test; returns ([CTA-scope gave up, cluster-scope
    gave up], elapsed device nanoseconds)."""
    gave_up = (ctypes.c_int * 2)()
    ns = ctypes.c_ulonglong(0)
    _check(lib().h2o_selftest_wait_timeout(int(polls), gave_up, ctypes.byref(ns)))
    return list(gave_up), int(ns.value)


def h2o_prefill_colsum_static(q, k, scale, colsum, kv_dtype=None, stream=None):
    """Column sums of a prompt with no device allocation (fixed library
    scratch; see include/h2o.h for the size limit and the no-overlap rule)."""
    import torch

    B, H, L, D = q.shape
    dt = q.dtype
    code = H2O_F16 if dt == torch.float16 else H2O_F32
    if kv_dtype is not None and kv_dtype != code:
        raise ValueError("kv_dtype does not match the tensors")
    _check(lib().h2o_prefill_colsum_static(
        _ptr(q, dt, (B, H, L, D), "q"), _ptr(k, dt, (B, H, L, D), "k"), B, H, D, L, code, float(scale),
        _ptr(colsum, torch.float32, (B, H, L), "colsum"), _stream(stream)))


def h2o_prefill_colsum_static_check(stream=None):
    """Raise H2OError if the last h2o_prefill_colsum_static call's kernels
    latched a device error (synchronises the stream)."""
    _check(lib().h2o_prefill_colsum_static_check(_stream(stream)))


def h2o_debug_fail_alloc(after: int):
    """Make the library's device allocation number after+1 from now fail (-1: off)."""
    _check(lib().h2o_debug_fail_alloc(int(after)))


def h2o_last_error() -> str:
    return lib().h2o_last_error().decode()


# ------------------------------------------------------------------ state image
def state_layout(batch, heads, head_dim, heavy, recent, kv_dtype):
    """Byte offsets of the export/import image (see include/h2o.h)."""
    P, C, R, D = batch * heads, heavy + recent, recent, head_dim
    e = 2 if kv_dtype == H2O_F16 else 4
    parts = [("K", P * C * D * e), ("V", P * C * D * e), ("score", P * C * 4), ("pos", P * C * 4),
             ("ring", P * R * 4), ("ctr", P * 16)]
    off, out = HEADER_INTS * 4, {}
    for name, n in parts:
        out[name] = (off, n)
        off += n
    out["total"] = off
    return out


def unpack_state(cache: Cache, buf: np.ndarray) -> dict:
    """Split an exported image into numpy arrays (views into `buf`)."""
    lay = state_layout(cache.batch, cache.heads, cache.head_dim, cache.heavy, cache.recent, cache.kv_dtype)
    P, C, R, D = cache.pairs, cache.slots, cache.recent, cache.head_dim

    def view(name, dtype, shape):
        off, n = lay[name]
        return buf[off:off + n].view(dtype).reshape(shape)

    ctr = view("ctr", np.int32, (P, 4))
    return {"K": view("K", cache.np_dtype(), (P, C, D)), "V": view("V", cache.np_dtype(), (P, C, D)),
            "score": view("score", np.float32, (P, C)), "pos": view("pos", np.int32, (P, C)),
            "ring": view("ring", np.int32, (P, R)), "p": ctr[:, 0], "count": ctr[:, 1], "head": ctr[:, 2]}


def pack_state(cache: Cache, K, V, score, pos, ring, p, count, head) -> np.ndarray:
    """Build an import image from per-pair arrays (host-side marshalling)."""
    lay = state_layout(cache.batch, cache.heads, cache.head_dim, cache.heavy, cache.recent, cache.kv_dtype)
    buf = np.zeros(lay["total"], dtype=np.uint8)
    hdr = buf[:HEADER_INTS * 4].view(np.int32)
    hdr[:8] = [MAGIC, 1, cache.batch, cache.heads, cache.head_dim, cache.heavy, cache.recent, cache.kv_dtype]
    st = unpack_state(cache, buf)
    st["K"][...] = K
    st["V"][...] = V
    st["score"][...] = score
    st["pos"][...] = pos
    st["ring"][...] = ring
    ctr = buf[lay["ctr"][0]:].view(np.int32).reshape(cache.pairs, 4)
    ctr[:, 0], ctr[:, 1], ctr[:, 2] = p, count, head
    return buf
