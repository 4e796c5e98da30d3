"""The allocation-free decode entry point, through the C ABI.

pa_decode_noalloc serves callers that cannot allocate device memory (a host
framework that hands over only inputs and outputs, or a path where cudaMalloc
would synchronise the device): it uses the library's static device scratch
instead of a caller workspace.  Its outputs must agree with pa_decode's on the
same inputs, on two calls in a row (the scratch keeps the previous call's
contents), and a batch too large for the scratch must be refused.  This file
sorts last so that, in a run that stops at the first failure, every other test
has already run; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_99_gb300 as pa
from paged_kv_cache_99_gb300 import build_ext
from paged_kv_cache_99_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2   # the attention tolerance used by every parity test


@pytest.fixture(scope="module", autouse=True)
def _library():
    build_ext.build()


def _with_workspace(w, layer=0):
    ks = w.k_scale[layer:layer + 1] if w.k_scale is not None else None
    vs = w.v_scale[layer:layer + 1] if w.v_scale is not None else None
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(w.q[layer])
    pa.pa_decode(out, w.q[layer], w.k_cache[layer], w.v_cache[layer], w.block_tables, w.seq_lens, w.scale, ws,
                 ks, vs)
    return out


def _no_alloc(w, layer=0):
    ks = w.k_scale[layer:layer + 1] if w.k_scale is not None else None
    vs = w.v_scale[layer:layer + 1] if w.v_scale is not None else None
    out = torch.empty_like(w.q[layer])
    pa.pa_decode_noalloc(out, w.q[layer], w.k_cache[layer], w.v_cache[layer], w.block_tables, w.seq_lens,
                         w.scale, ks, vs)
    return out


def _close(a, b, what):
    x, y = a.double().cpu().numpy(), b.double().cpu().numpy()
    assert np.all(np.isfinite(x)), what
    assert np.all(np.abs(x - y) <= ATOL + RTOL * np.abs(y)), f"{what}: max diff {np.abs(x - y).max():.3e}"


@pytest.mark.parametrize("cache,qd", [("bf16", "bf16"), ("fp8", "bf16")])
def test_no_alloc_matches_workspace_entry_point_twice(cache, qd):
    w = W.build_workload(name="noalloc", seed=61, device="cuda", num_layers=2,
                         seq_lens=[1, 15, 16, 17, 300, 2048, 4000, 0, 777], q_lens=[1] * 9,
                         num_q_heads=12, num_kv_heads=2, q_dtype=qd, cache_dtype=cache, write_new=False)
    ref0 = _with_workspace(w, 0)
    ref1 = _with_workspace(w, 1)
    first = _no_alloc(w, 0)
    second = _no_alloc(w, 1)   # same scratch, left holding the first call's partials
    torch.cuda.synchronize()
    _close(first, ref0, "first call")
    _close(second, ref1, "second call")


def test_no_alloc_refuses_a_batch_beyond_its_scratch():
    B, Hkv = 4096, 8            # 32768 units: far beyond the 16 MiB scratch
    q = torch.zeros(B, Hkv, 128, dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros(1, Hkv, 16, 128, dtype=torch.bfloat16, device="cuda")
    tables = torch.zeros(B, 1, dtype=torch.int32, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.pa_decode_noalloc(out, q, cache, cache, tables, lens, 0.088)
    assert e.value.status == pa.PA_ERR_WORKSPACE
    assert "static scratch" in pa._lib().pa_last_error().decode()
