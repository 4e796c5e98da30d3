"""The ends of the supported range: an empty batch, and the largest batch the
library takes (8192 sequences) in decode, fused-append and mixed form.  The large
cases are checked against the oracle on a sample of sequences (the first, the
last, the longest, the chunks and a few drawn at random)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_99_gb300 as pa
from paged_kv_cache_99_gb300 import workloads as W
from tests._gpu import compare, gpu_step, oracle_step

pytestmark = pytest.mark.gpu
DEV = "cuda"
MAX_SEQS = 8192


def test_empty_batch_launches_nothing():
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    q = torch.empty(0, 8, 128, dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(q)
    tables = torch.empty(0, 4, dtype=torch.int32, device=DEV)
    lens = torch.empty(0, dtype=torch.int32, device=DEV)
    ws = pa.new_workspace(0, 8, 2)
    pa.pa_decode(out, q, kc, vc, tables, lens, 0.088, ws)
    qsl = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_mixed(out, q, qsl, kc, vc, tables, lens, 0, 0.088, ws)
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(ws) == pa.PA_OK


def _sample(w, extra=()):
    lens = w.seq_lens.cpu().numpy()
    rng = np.random.default_rng(7)
    pick = {0, w.num_seqs - 1, int(lens.argmax()), int(lens.argmin()), *extra}
    pick.update(int(x) for x in rng.choice(w.num_seqs, 8, replace=False))
    return sorted(pick)


def _max_batch(seed, cache, q_lens=None):
    g = np.random.default_rng(seed)
    lens = [int(x) for x in g.integers(1, 49, MAX_SEQS)]
    q_lens = q_lens or [1] * MAX_SEQS
    lens = [max(n, q) for n, q in zip(lens, q_lens)]
    return W.build_workload(name="max-batch", seed=seed, device=DEV, num_layers=1, seq_lens=lens, q_lens=q_lens,
                            num_q_heads=8, num_kv_heads=2, q_dtype="bf16", cache_dtype=cache)


@pytest.mark.parametrize("cache", ["bf16", "fp8"])
def test_decode_max_batch(cache):
    w = _max_batch(11, cache)
    out, _, _ = gpu_step(w)
    rows, ref = oracle_step(w, 0, _sample(w))
    compare(out, rows, ref, f"{MAX_SEQS} sequences, {cache}")


def test_append_max_batch():
    w = _max_batch(12, "bf16")
    kc, vc = w.k_cache[0].clone(), w.v_cache[0].clone()
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(w.q[0])
    pa.pa_decode_append(out, w.q[0], w.k_new[0], w.v_new[0], w.slot_mapping, kc, vc, w.block_tables, w.seq_lens,
                        w.scale, ws)
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(ws) == pa.PA_OK
    rows, ref = oracle_step(w, 0, _sample(w))
    compare(out, rows, ref, f"fused append, {MAX_SEQS} sequences")


def test_mixed_max_batch():
    q_lens = [1] * MAX_SEQS
    chunks = {5: 33, 4000: 100, 8190: 7}
    for s, ql in chunks.items():
        q_lens[s] = ql
    w = _max_batch(13, "bf16", q_lens)
    out, _, _ = gpu_step(w)
    rows, ref = oracle_step(w, 0, _sample(w, chunks))
    compare(out, rows, ref, f"mixed, {MAX_SEQS} sequences")
