"""Dense (unpaged) attention built from library routines, used to pin the oracle.

The gather here is the test's own: contiguous K/V per sequence by numpy fancy
indexing of the block tables.  Attention is torch's float64
scaled_dot_product_attention with the KV heads repeated for the GQA groups.
"""
import numpy as np
import torch

import oracle
from paged_kv_cache_99_gb300 import workloads as W

CODE = {"bf16": oracle.BF16, "fp16": oracle.FP16, "fp8": oracle.FP8_E4M3}


def raw(t: torch.Tensor) -> np.ndarray:
    """Storage bits of a CPU/GPU tensor as a numpy array (uint16 or uint8)."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.uint8:
        return t.numpy()
    raise TypeError(t.dtype)


def values(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.uint8:
        return t.view(torch.float8_e4m3fn).double().numpy()
    return t.double().numpy()


def dense_kv(k_cache_vals, v_cache_vals, table_row, n, block_size=16):
    """[n, H_kv, d] contiguous K and V of one sequence."""
    t = np.arange(n)
    phys = np.asarray(table_row)[t // block_size]
    off = t % block_size
    return k_cache_vals[phys, :, off, :], v_cache_vals[phys, :, off, :]


def sdpa(q, K, V, scale, mask=None):
    """q [m, Hq, d], K/V [n, Hkv, d] float64 -> [m, Hq, d]."""
    Hq, Hkv = q.shape[1], K.shape[1]
    G = Hq // Hkv
    qt = torch.from_numpy(np.ascontiguousarray(q)).permute(1, 0, 2)          # Hq, m, d
    Kt = torch.from_numpy(np.ascontiguousarray(K)).permute(1, 0, 2).repeat_interleave(G, 0)
    Vt = torch.from_numpy(np.ascontiguousarray(V)).permute(1, 0, 2).repeat_interleave(G, 0)
    m = None if mask is None else torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, attn_mask=m, scale=scale)
    return o.permute(1, 0, 2).numpy()


def workload_values(w: W.Workload, layer=0):
    kc, vc = values(w.k_cache[layer]), values(w.v_cache[layer])
    if w.cache_dtype == "fp8":
        kc = kc * float(w.k_scale[layer])
        vc = vc * float(w.v_scale[layer])
    return kc, vc


def oracle_decode(w: W.Workload, layer=0, k_cache=None, v_cache=None, tables=None, seq_lens=None, q=None):
    kc = raw(w.k_cache[layer]) if k_cache is None else k_cache
    vc = raw(w.v_cache[layer]) if v_cache is None else v_cache
    return oracle.decode(raw(w.q[layer]) if q is None else q, CODE[w.q_dtype], kc, vc, CODE[w.cache_dtype],
                         (w.block_tables.cpu().numpy() if tables is None else tables),
                         (w.seq_lens.cpu().numpy() if seq_lens is None else seq_lens), w.scale,
                         float(w.k_scale[layer]) if w.k_scale is not None else 1.0,
                         float(w.v_scale[layer]) if w.v_scale is not None else 1.0)
