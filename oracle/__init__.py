"""Paged-KV-cache attention oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow, single-threaded float64 CPU restatement of the paged attention
path (``pa_oracle.c``) plus a ctypes shim.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package.  The library (``paged_kv_cache_99_gb300``) never imports it and shares
no code with it; the only thing both sides use is the seeded input generator
module, which holds none of the method's arithmetic.

Every function cites the passage it restates:

* [P1] "Basics of LLM Inference and vLLM Internals: KV Cache, PagedAttention,
  and Scheduler" -- s.2 (KV cache, sizing formula, GQA, FP8), s.4 (blocks of 16,
  block table, shared prefix), s.6 (chunked prefill).
* [P2] drpranayjha.com, Red Hat AI Inference Server part -- "How PagedAttention
  pages the KV cache" and the sizing snippet under it.
* [P3] "The Memory Trick Behind Fast LLM Serving" -- "PagedAttention changes
  the shape of the problem", "Batching does not merge the conversations".

Pins: see ``tests/test_oracle_*.py`` -- sizing values printed on the pages,
block counts of the worked examples, an FP8 encoder checked by brute force over
every code, equality with a dense library attention, invariance under
relabelling of physical blocks, alias identity, closed forms.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

from .sizing import kv_bytes_per_token, num_logical_blocks, last_block_fill  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, f"libpa_oracle_{platform.machine()}.so")

BF16, FP16, FP8_E4M3 = 0, 1, 2
_ERRORS = {1: "invalid argument", 2: "index out of range", 3: "out of memory"}

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f32, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        lib.or_e4m3_encode.argtypes = [f32]
        lib.or_e4m3_encode.restype = ctypes.c_uint8
        lib.or_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.or_e4m3_to_double.restype = f64
        lib.or_e4m3_encode_array.argtypes = [P, P, i64]
        lib.or_e4m3_encode_array.restype = None
        lib.or_quantize_array.argtypes = [P, i32, f32, P, i64]
        lib.or_quantize_array.restype = None
        lib.or_decode_array.argtypes = [P, i32, P, i64]
        lib.or_decode_array.restype = None
        lib.or_reshape_and_cache.argtypes = [P, P, i32, P, P, i32, P, i32, i32, i32, i32, i32, f32, f32]
        lib.or_reshape_and_cache.restype = i32
        lib.or_decode.argtypes = [P, P, i32, P, P, i32, f64, f64, P, i32, P, i32, i32, i32, i32, i32, i32, f64]
        lib.or_decode.restype = i32
        lib.or_mixed.argtypes = [P, P, i32, P, P, P, i32, f64, f64, P, i32, P, i32, i32, i32, i32, i32, i32, f64]
        lib.or_mixed.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: {_ERRORS.get(rc, rc)}")


def _bits(a: np.ndarray, dtype_code: int) -> np.ndarray:
    """Raw storage bits: uint16 for 16-bit types, uint8 for FP8."""
    a = np.asarray(a)
    want = np.uint8 if dtype_code == FP8_E4M3 else np.uint16
    if a.dtype != want:
        raise TypeError(f"expected raw {want.__name__} storage bits, got {a.dtype}")
    return np.ascontiguousarray(a)


# -- element formats ---------------------------------------------------------

def e4m3_encode(x) -> np.ndarray:
    """float32 values -> E4M3 codes (RNE, ties to even mantissa, satfinite)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().or_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def quantize(bits, src_dtype: int, scale: float) -> np.ndarray:
    """The slot-write FP8 rule: e4m3(fl32(x) / scale) for 16-bit source bits."""
    bits = _bits(bits, src_dtype)
    out = np.empty(bits.shape, np.uint8)
    _load().or_quantize_array(_ptr(bits), src_dtype, float(scale), _ptr(out), bits.size)
    return out


def decode_bits(bits, dtype_code: int) -> np.ndarray:
    """Raw bf16 / fp16 / e4m3 bits -> float64 values."""
    bits = _bits(bits, dtype_code)
    out = np.empty(bits.shape, np.float64)
    _load().or_decode_array(_ptr(bits), dtype_code, _ptr(out), bits.size)
    return out


# -- the path -----------------------------------------------------------------

def reshape_and_cache(k_bits, v_bits, src_dtype, k_cache, v_cache, cache_dtype, slot_mapping,
                      k_scale: float = 1.0, v_scale: float = 1.0):
    """Slot write [P1 s.4; P3 "PagedAttention changes the shape of the problem"].

    k_bits, v_bits: [T, H_kv, d] raw 16-bit bits.  k_cache, v_cache:
    [num_blocks, H_kv, block_size, d] raw bits; returns updated copies.
    """
    k_bits = _bits(k_bits, src_dtype)
    v_bits = _bits(v_bits, src_dtype)
    kc = _bits(k_cache, cache_dtype).copy()
    vc = _bits(v_cache, cache_dtype).copy()
    slots = _c(slot_mapping, np.int64)
    T, H, d = k_bits.shape
    nb, H2, bs, d2 = kc.shape
    if (H2, d2) != (H, d) or vc.shape != kc.shape or v_bits.shape != k_bits.shape or slots.shape != (T,):
        raise ValueError("shape mismatch")
    rc = _load().or_reshape_and_cache(_ptr(k_bits), _ptr(v_bits), src_dtype, _ptr(kc), _ptr(vc),
                                      cache_dtype, _ptr(slots), T, H, d, bs, nb,
                                      float(k_scale), float(v_scale))
    _check(rc, "reshape_and_cache")
    return kc, vc


def decode(q_bits, q_dtype, k_cache, v_cache, cache_dtype, block_tables, seq_lens, scale,
           k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """Decode attention over the paged cache [P1 s.2, s.4]; float64 [B, H_q, d]."""
    q_bits = _bits(q_bits, q_dtype)
    kc = _bits(k_cache, cache_dtype)
    vc = _bits(v_cache, cache_dtype)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    B, Hq, d = q_bits.shape
    nb, Hkv, bs, d2 = kc.shape
    if d2 != d or vc.shape != kc.shape or bt.ndim != 2 or bt.shape[0] != B or sl.shape != (B,):
        raise ValueError("shape mismatch")
    out = np.zeros((B, Hq, d), np.float64)
    rc = _load().or_decode(_ptr(out), _ptr(q_bits), q_dtype, _ptr(kc), _ptr(vc), cache_dtype,
                           float(k_scale), float(v_scale), _ptr(bt), bt.shape[1], _ptr(sl), B,
                           Hq, Hkv, d, bs, nb, float(scale))
    _check(rc, "decode")
    return out


def mixed(q_bits, q_dtype, query_start_loc, k_cache, v_cache, cache_dtype, block_tables, seq_lens,
          scale, k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """Mixed decode rows + causal prefill chunks [P1 s.6; P3 "Batching does not
    merge the conversations"]; float64 [total_q, H_q, d]."""
    q_bits = _bits(q_bits, q_dtype)
    kc = _bits(k_cache, cache_dtype)
    vc = _bits(v_cache, cache_dtype)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    total_q, Hq, d = q_bits.shape
    nb, Hkv, bs, d2 = kc.shape
    B = sl.shape[0]
    if d2 != d or vc.shape != kc.shape or bt.shape[0] != B or qsl.shape != (B + 1,) or qsl[-1] != total_q:
        raise ValueError("shape mismatch")
    out = np.zeros((total_q, Hq, d), np.float64)
    rc = _load().or_mixed(_ptr(out), _ptr(q_bits), q_dtype, _ptr(qsl), _ptr(kc), _ptr(vc),
                          cache_dtype, float(k_scale), float(v_scale), _ptr(bt), bt.shape[1],
                          _ptr(sl), B, Hq, Hkv, d, bs, nb, float(scale))
    _check(rc, "mixed")
    return out
