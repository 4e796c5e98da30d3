"""The allocation-free decode entry point, through the C ABI.

pa_decode_noalloc serves callers that cannot allocate device memory (a host
framework that hands over only inputs and outputs, or a path where cudaMalloc
would synchronise the device): it uses the library's static device scratch
instead of a caller workspace.  Its outputs must agree with pa_decode's and
with the oracle on the same inputs, on two calls in a row (the scratch keeps
the previous call's contents, including the counter from which warps claim
pieces of work on long rows), and a batch must be accepted up to the limit the
header states and refused one sequence beyond it.  This file sorts last so
that, in a run that stops at the first failure, every other test has already
run; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_99_gb300 as pa
from paged_kv_cache_99_gb300 import build_ext
from paged_kv_cache_99_gb300 import workloads as W
from tests._gpu import compare, oracle_step

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2   # the attention tolerance used by every parity test
SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module", autouse=True)
def _library():
    build_ext.build()


def _scales(w, layer):
    return (w.k_scale[layer:layer + 1] if w.k_scale is not None else None,
            w.v_scale[layer:layer + 1] if w.v_scale is not None else None)


def _with_workspace(w, layer=0):
    ks, vs = _scales(w, layer)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(w.q[layer])
    pa.pa_decode(out, w.q[layer], w.k_cache[layer], w.v_cache[layer], w.block_tables, w.seq_lens, w.scale, ws,
                 ks, vs)
    return out


def _no_alloc(w, layer=0):
    ks, vs = _scales(w, layer)
    out = torch.empty_like(w.q[layer])
    pa.pa_decode_noalloc(out, w.q[layer], w.k_cache[layer], w.v_cache[layer], w.block_tables, w.seq_lens,
                         w.scale, ks, vs)
    return out


def _close(a, b, what):
    x, y = a.double().cpu().numpy(), b.double().cpu().numpy()
    assert np.all(np.isfinite(x)), what
    assert np.all(np.abs(x - y) <= ATOL + RTOL * np.abs(y)), f"{what}: max diff {np.abs(x - y).max():.3e}"


def _scratch_needed(S, Hq, Hkv, workers):
    """Bytes of scratch a call needs, by the formula the header states."""
    r = lambda x: -(-x // 256) * 256
    n = S * Hkv * -(-(Hq // Hkv) // 8) + 2 * workers
    return 256 + r(4 * (S + 1)) + r(512 * S * Hq) + r(8 * S * Hq) + r(64 * n) + 4096 * n


@pytest.mark.parametrize("cache,qd", [("bf16", "bf16"), ("fp8", "bf16")])
def test_no_alloc_matches_workspace_entry_point_and_oracle_twice(cache, qd):
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
    for layer, out in ((0, first), (1, second)):
        rows, ref = oracle_step(w, layer)
        compare(out, rows, ref, f"no-alloc {cache} layer {layer}")


def test_no_alloc_claimed_pieces_twice_after_a_workspace_call():
    # units of 4 query heads and long rows (>= 48 16-key units per warp at the
    # default worker count): the last share of the work goes to pieces claimed from
    # the counter at the head of the static scratch, which each call resets
    workers = pa.pa_default_workers()
    lens = [61000, 59000, 60500, 58000, 62000, 57000, 60000, 63000]
    blocks = sum(-(-n // 16) for n in lens) * 2
    assert blocks // workers >= 48, "rows too short for claimed pieces on this GPU"
    w = W.build_workload(name="noalloc-pieces", seed=62, device="cuda", num_layers=2, seq_lens=lens,
                         q_lens=[1] * len(lens), num_q_heads=8, num_kv_heads=2, q_dtype="bf16",
                         cache_dtype="bf16", write_new=False)
    assert _scratch_needed(w.num_seqs, 8, 2, workers) <= SCRATCH_BYTES
    ref0 = _with_workspace(w, 0)
    ref1 = _with_workspace(w, 1)
    first = _no_alloc(w, 0)
    second = _no_alloc(w, 1)
    torch.cuda.synchronize()
    _close(first, ref0, "first call")
    _close(second, ref1, "second call")
    pick = [0, 3, len(lens) - 1]          # the last sequence's tail is in claimed pieces
    for layer, out in ((0, first), (1, second)):
        rows, ref = oracle_step(w, layer, pick)
        compare(out, rows, ref, f"no-alloc pieces layer {layer}")


def _batch(S, Hq, Hkv, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    lens = torch.randint(1, 40, (S,), generator=g, dtype=torch.int32)
    return W.build_workload(name="noalloc-limit", seed=seed, device="cuda", num_layers=1, seq_lens=lens.tolist(),
                            q_lens=[1] * S, num_q_heads=Hq, num_kv_heads=Hkv, write_new=False)


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (32, 8)])
def test_no_alloc_limit_is_the_stated_one(Hq, Hkv):
    workers = pa.pa_default_workers()
    S = 1
    while _scratch_needed(S + 1, Hq, Hkv, workers) <= SCRATCH_BYTES:
        S += 1
    # the largest batch the stated formula allows runs and agrees with pa_decode
    w = _batch(S, Hq, Hkv, 63)
    ref = _with_workspace(w)
    out = _no_alloc(w)
    torch.cuda.synchronize()
    _close(out, ref, f"{S} sequences (the limit)")
    # one sequence more is refused before anything runs
    w2 = _batch(S + 1, Hq, Hkv, 64)
    out2 = torch.zeros_like(w2.q[0])
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.pa_decode_noalloc(out2, w2.q[0], w2.k_cache[0], w2.v_cache[0], w2.block_tables, w2.seq_lens, w2.scale)
    assert e.value.status == pa.PA_ERR_WORKSPACE
    assert "static scratch" in pa._lib().pa_last_error().decode()
    assert torch.count_nonzero(out2) == 0


def test_no_alloc_refuses_a_batch_far_beyond_its_scratch():
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
