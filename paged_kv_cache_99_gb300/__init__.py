"""Paged-KV-cache attention on one GB300 (sm_103a): a thin ctypes binding of libpa.so.

Every function here only marshals torch tensors into the C ABI declared in
``include/pa.h`` (pointers, sizes, dtypes, the current CUDA stream) and raises
``PagedAttentionError`` on a non-zero status; all the work runs in the
library's CUDA kernels.  There is no CPU fallback: if libpa.so is missing the
import of the binding fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build_ext

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_TIMEOUT, PA_ERR_OUT_OF_RANGE, \
    PA_ERR_WORKSPACE = range(7)
PA_BF16, PA_FP16, PA_FP8_E4M3, PA_FP8_E4M3_PER_HEAD = 0, 1, 2, 3

_DTYPE = {torch.bfloat16: PA_BF16, torch.float16: PA_FP16, torch.uint8: PA_FP8_E4M3,
          torch.float8_e4m3fn: PA_FP8_E4M3}


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {_lib().pa_status_string(status).decode()} (status {status})"
        if status == PA_ERR_CUDA:
            msg += f": {_lib().pa_last_error().decode()}"
        super().__init__(msg)


_LIB = None


def library_path() -> str:
    return build_ext.LIB_PATH


def _lib():
    global _LIB
    if _LIB is not None:
        return _LIB
    path = build_ext.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"libpa.so is not built ({path}); run __graft_entry__.build() "
                          "or python -m paged_kv_cache_99_gb300.build_ext")
    lib = ctypes.CDLL(path)
    P, I, Z, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    lib.pa_status_string.argtypes = [I]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_version.argtypes = []
    lib.pa_version.restype = I
    lib.pa_kernel_launches.argtypes = []
    lib.pa_kernel_launches.restype = ctypes.c_ulonglong
    lib.pa_last_error.argtypes = []
    lib.pa_last_error.restype = ctypes.c_char_p
    lib.pa_reshape_and_cache.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, P, P, P]
    lib.pa_reshape_and_cache.restype = I
    lib.pa_workspace_size.argtypes = [I, I, I, I]
    lib.pa_workspace_size.restype = Z
    lib.pa_workspace_size_shared_prefix.argtypes = [I, I, I, I]
    lib.pa_workspace_size_shared_prefix.restype = Z
    lib.pa_default_workers.argtypes = []
    lib.pa_default_workers.restype = I
    lib.pa_decode.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, I, P, P, P, Z, P]
    lib.pa_decode.restype = I
    lib.pa_decode_ex.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, I, P, P, P, Z, I, P]
    lib.pa_decode_append.argtypes = [P, P, P, P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, I, P, P, P, Z, P]
    lib.pa_decode_append.restype = I
    lib.pa_decode_append_ex.argtypes = [P, P, P, P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, I, P, P, P, Z, I, P]
    lib.pa_decode_append_ex.restype = I
    lib.pa_decode_ex.restype = I
    lib.pa_decode_shared_prefix.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I, F, I, I, P, P, P, Z, P]
    lib.pa_decode_shared_prefix.restype = I
    lib.pa_mixed.argtypes = [P, P, P, P, P, P, I, P, I, I, I, I, I, I, I, I, F, I, I, P, P, P, Z, P]
    lib.pa_mixed.restype = I
    lib.pa_decode_noalloc.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, I, P, P, P]
    lib.pa_decode_noalloc.restype = I
    lib.pa_read_device_status.argtypes = [P, P]
    lib.pa_read_device_status.restype = I
    lib.pa_selftest_wait_timeout.argtypes = [P, Z, ctypes.c_uint, P]
    lib.pa_selftest_wait_timeout.restype = I
    lib.pa_copy_blocks.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P]
    lib.pa_copy_blocks.restype = I
    lib.pa_pool_create.argtypes = [I, I]
    lib.pa_pool_create.restype = P
    lib.pa_pool_destroy.argtypes = [P]
    lib.pa_pool_destroy.restype = None
    for name in ("pa_pool_num_free", "pa_pool_num_cached"):
        getattr(lib, name).argtypes = [P]
        getattr(lib, name).restype = I
    lib.pa_pool_ref_count.argtypes = [P, I]
    lib.pa_pool_ref_count.restype = I
    lib.pa_pool_allocate.argtypes = [P, I, P]
    lib.pa_pool_allocate.restype = I
    lib.pa_pool_share.argtypes = [P, P, I]
    lib.pa_pool_share.restype = I
    lib.pa_pool_free.argtypes = [P, P, I]
    lib.pa_pool_free.restype = I
    lib.pa_pool_allocate_prompt.argtypes = [P, P, I, ctypes.c_uint64, P, ctypes.POINTER(I)]
    lib.pa_pool_allocate_prompt.restype = I
    lib.pa_pool_copy_on_write.argtypes = [P, P, I, P, P, ctypes.POINTER(I)]
    lib.pa_pool_copy_on_write.restype = I
    _LIB = lib
    return lib


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _need(t: torch.Tensor, name: str, dtypes=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")


def _cache_code(cache, k_scale, num_kv_heads: int) -> int:
    """pa_dtype of a cache: an e4m3 cache with one scale per KV head is PA_FP8_E4M3_PER_HEAD."""
    code = _DTYPE[cache.dtype]
    if code == PA_FP8_E4M3 and k_scale is not None and k_scale.numel() > 1:
        if k_scale.numel() != num_kv_heads:
            raise ValueError("FP8 scales must hold one value or one per KV head")
        return PA_FP8_E4M3_PER_HEAD
    return code


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedAttentionError(status, what)


def pa_version() -> int:
    return _lib().pa_version()


def pa_status_string(status: int) -> str:
    return _lib().pa_status_string(status).decode()


def pa_kernel_launches() -> int:
    """Kernels the library has enqueued in this process (launches into a captured
    stream count at capture)."""
    return int(_lib().pa_kernel_launches())


def pa_default_workers() -> int:
    return _lib().pa_default_workers()


def pa_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int = 128) -> int:
    return int(_lib().pa_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim))


def pa_workspace_size_shared_prefix(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int = 128) -> int:
    return int(_lib().pa_workspace_size_shared_prefix(num_seqs, num_q_heads, num_kv_heads, head_dim))


def new_workspace(num_seqs: int, num_q_heads: int, num_kv_heads: int, device=None,
                  shared_prefix: bool = False) -> torch.Tensor:
    """Workspace of pa_workspace_size bytes (zeroed, so the status word starts clear);
    with shared_prefix, pa_workspace_size_shared_prefix bytes (every prefix split)."""
    size = pa_workspace_size_shared_prefix if shared_prefix else pa_workspace_size
    n = size(num_seqs, num_q_heads, num_kv_heads)
    if n == 0:
        raise ValueError("invalid workspace arguments")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def pa_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, k_scale=None, v_scale=None, stream=None):
    """Slot write: k, v [T, H_kv, 128] -> caches [num_blocks, H_kv, bs, 128] (bs = 8, 16, 32) at slot_mapping[T] (int64)."""
    for t, n in ((k, "k"), (v, "v")):
        _need(t, n, (torch.bfloat16, torch.float16))
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, tuple(_DTYPE))
    _need(slot_mapping, "slot_mapping", (torch.int64,))
    T, H, d = k.shape
    nb, H2, bs, d2 = k_cache.shape
    if v.shape != k.shape or v_cache.shape != k_cache.shape or H2 != H or d2 != d or slot_mapping.shape != (T,):
        raise ValueError("shape mismatch")
    st = _lib().pa_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), T, H, d,
                                     bs, nb, _DTYPE[k.dtype], _cache_code(k_cache, k_scale, k_cache.shape[1]), _ptr(k_scale),
                                     _ptr(v_scale), _stream(stream))
    _check(st, "pa_reshape_and_cache")


def pa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, scale, workspace, k_scale=None, v_scale=None,
              num_workers: int = 0, stream=None):
    """Decode attention: q, out [B, H_q, 128]; block_tables int32 [B, max_blocks]; seq_lens int32 [B]."""
    _need(q, "q", (torch.bfloat16, torch.float16))
    _need(out, "out", (q.dtype,))
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, tuple(_DTYPE))
    _need(block_tables, "block_tables", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    _need(workspace, "workspace", (torch.uint8,))
    B, Hq, d = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    if out.shape != q.shape or block_tables.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("shape mismatch")
    st = _lib().pa_decode_ex(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                             block_tables.shape[1], _ptr(seq_lens), B, Hq, Hkv, d, bs, nb, float(scale),
                             _DTYPE[q.dtype], _cache_code(k_cache, k_scale, k_cache.shape[1]), _ptr(k_scale), _ptr(v_scale),
                             _ptr(workspace), workspace.numel(), int(num_workers), _stream(stream))
    _check(st, "pa_decode")


def pa_decode_append(out, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, seq_lens, scale, workspace,
                     k_scale=None, v_scale=None, num_workers: int = 0, stream=None):
    """pa_reshape_and_cache of one new token per sequence (k_new, v_new [B, H_kv, 128] at
    slot_mapping[B], int64, the slot of position seq_lens[s] - 1) fused with pa_decode;
    num_workers > 0 goes through pa_decode_append_ex with that worker count."""
    _need(q, "q", (torch.bfloat16, torch.float16))
    _need(out, "out", (q.dtype,))
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, n, (q.dtype,))
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, tuple(_DTYPE))
    _need(slot_mapping, "slot_mapping", (torch.int64,))
    _need(block_tables, "block_tables", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    _need(workspace, "workspace", (torch.uint8,))
    B, Hq, d = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    if (out.shape != q.shape or block_tables.shape[0] != B or seq_lens.shape != (B,) or
            k_new.shape != (B, Hkv, d) or v_new.shape != k_new.shape or slot_mapping.shape != (B,)):
        raise ValueError("shape mismatch")
    args = (_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
            _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B, Hq, Hkv, d, bs, nb, float(scale),
            _DTYPE[q.dtype], _cache_code(k_cache, k_scale, k_cache.shape[1]), _ptr(k_scale), _ptr(v_scale),
            _ptr(workspace), workspace.numel())
    if num_workers:
        st = _lib().pa_decode_append_ex(*args, int(num_workers), _stream(stream))
    else:
        st = _lib().pa_decode_append(*args, _stream(stream))
    _check(st, "pa_decode_append")


def pa_decode_shared_prefix(out, q, k_cache, v_cache, block_tables, seq_lens, prefix_blocks, scale, workspace,
                            k_scale=None, v_scale=None, stream=None):
    """pa_decode for tables that share their first prefix_blocks entries (cascade: the shared
    prefix as one dense tensor-core contraction, the private suffixes through the decode kernel)."""
    _need(q, "q", (torch.bfloat16, torch.float16))
    _need(out, "out", (q.dtype,))
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, tuple(_DTYPE))
    _need(block_tables, "block_tables", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    _need(workspace, "workspace", (torch.uint8,))
    B, Hq, d = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    if out.shape != q.shape or block_tables.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("shape mismatch")
    st = _lib().pa_decode_shared_prefix(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                        block_tables.shape[1], _ptr(seq_lens), B, int(prefix_blocks), Hq, Hkv, d,
                                        bs, nb, float(scale), _DTYPE[q.dtype], _cache_code(k_cache, k_scale, k_cache.shape[1]),
                                        _ptr(k_scale), _ptr(v_scale), _ptr(workspace), workspace.numel(),
                                        _stream(stream))
    _check(st, "pa_decode_shared_prefix")


def pa_mixed(out, q, query_start_loc, k_cache, v_cache, block_tables, seq_lens, max_q_len, scale, workspace,
             k_scale=None, v_scale=None, stream=None):
    """Mixed decode rows + causal prefill chunks: q, out [total_q, H_q, 128]; query_start_loc int32 [B+1]."""
    _need(q, "q", (torch.bfloat16, torch.float16))
    _need(out, "out", (q.dtype,))
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, tuple(_DTYPE))
    _need(query_start_loc, "query_start_loc", (torch.int32,))
    _need(block_tables, "block_tables", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    _need(workspace, "workspace", (torch.uint8,))
    total_q, Hq, d = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    B = seq_lens.shape[0]
    if out.shape != q.shape or block_tables.shape[0] != B or query_start_loc.shape != (B + 1,):
        raise ValueError("shape mismatch")
    st = _lib().pa_mixed(_ptr(out), _ptr(q), _ptr(query_start_loc), _ptr(k_cache), _ptr(v_cache),
                         _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B, total_q, int(max_q_len), Hq,
                         Hkv, d, bs, nb, float(scale), _DTYPE[q.dtype], _cache_code(k_cache, k_scale, k_cache.shape[1]), _ptr(k_scale),
                         _ptr(v_scale), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "pa_mixed")


def pa_decode_noalloc(out, q, k_cache, v_cache, block_tables, seq_lens, scale, k_scale=None, v_scale=None,
                      stream=None):
    """pa_decode for callers that cannot allocate: no workspace argument; the library's
    static device scratch is used instead (see include/pa.h for its limit and rules)."""
    _need(q, "q", (torch.bfloat16, torch.float16))
    _need(out, "out", (q.dtype,))
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, tuple(_DTYPE))
    _need(block_tables, "block_tables", (torch.int32,))
    _need(seq_lens, "seq_lens", (torch.int32,))
    B, Hq, d = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    if out.shape != q.shape or block_tables.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("shape mismatch")
    st = _lib().pa_decode_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                  block_tables.shape[1], _ptr(seq_lens), B, Hq, Hkv, d, bs, nb, float(scale),
                                  _DTYPE[q.dtype], _cache_code(k_cache, k_scale, k_cache.shape[1]), _ptr(k_scale), _ptr(v_scale),
                                  _stream(stream))
    _check(st, "pa_decode_noalloc")


def pa_read_device_status(workspace, stream=None) -> int:
    """Device status word of a workspace (synchronises the stream, clears the word)."""
    _need(workspace, "workspace", (torch.uint8,))
    return int(_lib().pa_read_device_status(_ptr(workspace), _stream(stream)))


def pa_selftest_wait_timeout(workspace, timeout_us: int, stream=None) -> None:
    _need(workspace, "workspace", (torch.uint8,))
    _check(_lib().pa_selftest_wait_timeout(_ptr(workspace), workspace.numel(), int(timeout_us), _stream(stream)),
           "pa_selftest_wait_timeout")


def pa_copy_blocks(k_cache, v_cache, src, dst, workspace=None, stream=None):
    """Copy-on-write block copies: block dst[i] <- src[i] (int32 device tensors) in both caches."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, tuple(_DTYPE))
    _need(src, "src", (torch.int32,))
    _need(dst, "dst", (torch.int32,))
    if src.shape != dst.shape or src.dim() != 1:
        raise ValueError("src and dst must be 1-D and of equal length")
    nb, Hkv, bs, d = k_cache.shape
    st = _lib().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src), _ptr(dst), int(src.numel()), Hkv, d, bs,
                               nb, _DTYPE[k_cache.dtype], _ptr(workspace), _stream(stream))
    _check(st, "pa_copy_blocks")


class BlockPool:
    """Host block pool (pa_pool_*): free queue with a null block 0, reference counts,
    prefix caching over chained block hashes, copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        self._lib = _lib()
        self._p = self._lib.pa_pool_create(int(num_blocks), int(block_size))
        if not self._p:
            raise ValueError("pa_pool_create failed")
        self.block_size = int(block_size)

    def __del__(self):
        if getattr(self, "_p", None):
            self._lib.pa_pool_destroy(self._p)
            self._p = None

    @staticmethod
    def _ids(blocks):
        import numpy as np
        a = np.ascontiguousarray(np.asarray(blocks, dtype=np.int32))
        return a, a.ctypes.data

    @property
    def num_free(self) -> int:
        return self._lib.pa_pool_num_free(self._p)

    @property
    def num_cached(self) -> int:
        return self._lib.pa_pool_num_cached(self._p)

    def ref_count(self, block: int) -> int:
        return self._lib.pa_pool_ref_count(self._p, int(block))

    def allocate(self, n: int) -> list:
        import numpy as np
        out = np.zeros(max(int(n), 1), dtype=np.int32)
        _check(self._lib.pa_pool_allocate(self._p, int(n), out.ctypes.data), "pa_pool_allocate")
        return out[:int(n)].tolist()

    def share(self, blocks) -> None:
        a, ptr = self._ids(blocks)
        _check(self._lib.pa_pool_share(self._p, ptr, a.size), "pa_pool_share")

    def free(self, blocks) -> None:
        a, ptr = self._ids(blocks)
        _check(self._lib.pa_pool_free(self._p, ptr, a.size), "pa_pool_free")

    def allocate_prompt(self, tokens, extra_key: int = 0):
        """-> (blocks, hit_tokens) for a prompt of len(tokens) tokens."""
        import numpy as np
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n = -(-t.size // self.block_size)
        out = np.zeros(max(n, 1), dtype=np.int32)
        hit = ctypes.c_int(0)
        _check(self._lib.pa_pool_allocate_prompt(self._p, t.ctypes.data, t.size, ctypes.c_uint64(extra_key),
                                                 out.ctypes.data, ctypes.byref(hit)), "pa_pool_allocate_prompt")
        return out[:n].tolist(), hit.value

    def copy_on_write(self, blocks):
        """-> (new_blocks, src, dst): shared blocks replaced by private ones, and the copies to make."""
        import numpy as np
        a = np.ascontiguousarray(np.asarray(blocks, dtype=np.int32)).copy()
        src = np.zeros(max(a.size, 1), dtype=np.int32)
        dst = np.zeros(max(a.size, 1), dtype=np.int32)
        c = ctypes.c_int(0)
        _check(self._lib.pa_pool_copy_on_write(self._p, a.ctypes.data, a.size, src.ctypes.data, dst.ctypes.data,
                                               ctypes.byref(c)), "pa_pool_copy_on_write")
        return a.tolist(), src[:c.value].tolist(), dst[:c.value].tolist()
