"""fp64 CPU oracle for decode attention over a static KV cache.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package. It shares no code with the
CUDA library and the library never imports it.

The arithmetic lives in ``oracle.c`` (plain C, double precision); this module
only loads it and marshals numpy arrays of raw 16-bit storage. Inputs are the
bit patterns of fp16 or bf16 values (``numpy.uint16``), so the oracle decodes
the very values the GPU reads.
"""
from __future__ import annotations

import ctypes
import pathlib

import numpy as np

from . import build as _build

F16 = 0
BF16 = 1
DTYPE_CODES = {"f16": F16, "fp16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16}

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)
_f32p = ctypes.POINTER(ctypes.c_float)


def dtype_code(dtype) -> int:
    """Map 'f16'/'bf16' (or a torch dtype's name) to the oracle's code."""
    name = str(dtype).replace("torch.", "")
    if name not in DTYPE_CODES:
        raise ValueError(f"unsupported dtype {dtype!r}")
    return DTYPE_CODES[name]


class Oracle:
    """A loaded oracle library. ``Oracle()`` loads the default build; a path
    loads another build of the same source (the tests use this)."""

    def __init__(self, lib_path: str | pathlib.Path | None = None):
        if lib_path is None:
            lib_path = _build.ensure_built()
        self.path = pathlib.Path(lib_path)
        lib = ctypes.CDLL(str(self.path))
        lib.oracle_decode_attn.argtypes = [_u16p, _u16p, _u16p, _i32p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_double, _f64p, ctypes.c_int]
        lib.oracle_decode_attn.restype = ctypes.c_int
        lib.oracle_kvcache_append.argtypes = [_u16p, _u16p, _u16p, _u16p, _i32p, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_kvcache_append.restype = ctypes.c_int
        lib.oracle_decode_bits.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int, _f64p]
        lib.oracle_decode_bits.restype = ctypes.c_int
        lib.oracle_encode_f32.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int, _u16p]
        lib.oracle_encode_f32.restype = ctypes.c_int
        lib.oracle_rope.argtypes = [_u16p, _f32p, _f32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, _u16p]
        lib.oracle_rope.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        self._lib = lib

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _u16(a) -> np.ndarray:
        a = np.ascontiguousarray(a)
        if a.dtype != np.uint16:
            raise TypeError(f"expected raw 16-bit storage (numpy.uint16), got {a.dtype}")
        return a

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())

    def decode_bits(self, bits, dtype) -> np.ndarray:
        bits = self._u16(bits)
        out = np.empty(bits.shape, dtype=np.float64)
        rc = self._lib.oracle_decode_bits(bits.ctypes.data_as(_u16p), bits.size, dtype_code(dtype),
                                          out.ctypes.data_as(_f64p))
        if rc != 0:
            raise ValueError(f"oracle_decode_bits returned {rc}")
        return out

    def encode_f32(self, values, dtype) -> np.ndarray:
        """fp32 values -> raw 16-bit storage, round to nearest even."""
        v = np.ascontiguousarray(values, dtype=np.float32)
        out = np.empty(v.shape, dtype=np.uint16)
        rc = self._lib.oracle_encode_f32(v.ctypes.data_as(_f32p), v.size, dtype_code(dtype),
                                         out.ctypes.data_as(_u16p))
        if rc != 0:
            raise ValueError(f"oracle_encode_f32 returned {rc}")
        return out

    def rope(self, x, cos_table, sin_table, position_ids, dtype) -> tuple[np.ndarray, int]:
        """Rotary embedding of x [B, heads, D] (raw 16-bit) with the table rows
        [rows, D] (fp32) at position_ids[b]; returns (rotated raw 16-bit, count
        of out-of-range positions, whose rows are left zero)."""
        x = self._u16(x)
        c = np.ascontiguousarray(cos_table, dtype=np.float32)
        sn = np.ascontiguousarray(sin_table, dtype=np.float32)
        pos = np.ascontiguousarray(position_ids, dtype=np.int32)
        B, heads, D = x.shape
        if c.shape != sn.shape or c.ndim != 2 or c.shape[1] != D or pos.shape != (B,):
            raise ValueError("inconsistent shapes")
        out = np.zeros_like(x)
        rc = self._lib.oracle_rope(x.ctypes.data_as(_u16p), c.ctypes.data_as(_f32p), sn.ctypes.data_as(_f32p),
                                   pos.ctypes.data_as(_i32p), B, heads, D, c.shape[0], dtype_code(dtype),
                                   out.ctypes.data_as(_u16p))
        if rc < 0:
            raise ValueError(f"oracle_rope returned {rc}")
        return out, int(rc)

    def decode_attn(self, q, k_cache, v_cache, kv_len, n_head: int, n_kv_head: int, dtype,
                    scale: float | None = None, threads: int = 1) -> np.ndarray:
        """out[B, n_head, D] (float64) for q [B, n_head, D] and caches
        [B, n_kv_head, capacity, D], all raw 16-bit; kv_len int32 [B]."""
        q, k_cache, v_cache = self._u16(q), self._u16(k_cache), self._u16(v_cache)
        kv_len = np.ascontiguousarray(kv_len, dtype=np.int32)
        B, H, D = q.shape
        Bk, Hkv, cap, Dk = k_cache.shape
        if (Bk, Dk) != (B, D) or v_cache.shape != k_cache.shape or H != n_head or Hkv != n_kv_head:
            raise ValueError("inconsistent shapes")
        if kv_len.shape != (B,):
            raise ValueError("kv_len must have shape [B]")
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        out = np.empty((B, H, D), dtype=np.float64)
        rc = self._lib.oracle_decode_attn(q.ctypes.data_as(_u16p), k_cache.ctypes.data_as(_u16p),
                                          v_cache.ctypes.data_as(_u16p), kv_len.ctypes.data_as(_i32p),
                                          B, n_head, n_kv_head, D, cap, dtype_code(dtype),
                                          float(scale), out.ctypes.data_as(_f64p), int(threads))
        if rc != 0:
            raise ValueError(f"oracle_decode_attn returned {rc}")
        return out

    def kvcache_append(self, k_cache, v_cache, k_new, v_new, position_ids) -> int:
        """Write k_new/v_new [B, n_kv_head, D] into row position_ids[b] of the
        caches, in place. Returns how many positions were out of range."""
        for a in (k_cache, v_cache):
            if not (isinstance(a, np.ndarray) and a.dtype == np.uint16 and a.flags.c_contiguous):
                raise TypeError("caches must be C-contiguous numpy.uint16 arrays (updated in place)")
        k_new, v_new = self._u16(k_new), self._u16(v_new)
        pos = np.ascontiguousarray(position_ids, dtype=np.int32)
        B, Hkv, cap, D = k_cache.shape
        if v_cache.shape != k_cache.shape or k_new.shape != (B, Hkv, D) or v_new.shape != k_new.shape:
            raise ValueError("inconsistent shapes")
        rc = self._lib.oracle_kvcache_append(k_cache.ctypes.data_as(_u16p), v_cache.ctypes.data_as(_u16p),
                                             k_new.ctypes.data_as(_u16p), v_new.ctypes.data_as(_u16p),
                                             pos.ctypes.data_as(_i32p), B, Hkv, D, cap)
        if rc < 0:
            raise ValueError(f"oracle_kvcache_append returned {rc}")
        return int(rc)


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT


def decode_attn(*args, **kwargs) -> np.ndarray:
    return default().decode_attn(*args, **kwargs)


def kvcache_append(*args, **kwargs) -> int:
    return default().kvcache_append(*args, **kwargs)
