"""FP8 caches with one scale per KV head (PA_FP8_E4M3_PER_HEAD): heads of
different magnitude, so that a kernel applying another head's scale fails.  The
oracle runs once per KV head with that head's scales (a head's outputs depend
on its own elements only)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_99_gb300 as pa
from paged_kv_cache_99_gb300 import workloads as W
from tests._dense import CODE, raw
from tests._gpu import compare, gpu_step, oracle_step

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed, lens, G, Hkv=4, q_lens=None, prefix=0, write_new=True, qd="bf16"):
    return W.build_workload(name="fp8-head", seed=seed, device=DEV, num_layers=1, seq_lens=lens,
                            q_lens=q_lens or [1] * len(lens), num_q_heads=G * Hkv, num_kv_heads=Hkv,
                            q_dtype=qd, cache_dtype="fp8", fp8_scale="head", shared_prefix_blocks=prefix,
                            write_new=write_new)


@pytest.mark.parametrize("qd", ["bf16", "fp16"])
def test_per_head_slot_write_bit_exact(qd):
    w = _case(90, [5, 16, 17, 40, 300], 2, qd=qd)
    assert w.k_scale.shape == (1, 4)
    kc, vc = w.k_cache[0].clone(), w.v_cache[0].clone()
    ks, vs = w.k_scale[0:1], w.v_scale[0:1]
    pa.pa_reshape_and_cache(w.k_new[0], w.v_new[0], kc, vc, w.slot_mapping, ks, vs)
    torch.cuda.synchronize()
    for h in range(w.num_kv_heads):
        ek, ev = oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), CODE[qd], raw(w.k_cache[0]),
                                          raw(w.v_cache[0]), CODE["fp8"], w.slot_mapping.cpu().numpy(),
                                          float(ks[0, h]), float(vs[0, h]))
        assert np.array_equal(raw(kc)[:, h], ek[:, h]) and np.array_equal(raw(vc)[:, h], ev[:, h]), f"head {h}"


@pytest.mark.parametrize("G", [1, 4, 8])
def test_per_head_decode(G):
    w = _case(91 + G, [30, 100, 513, 1, 1200, 77], G)
    out, _, _ = gpu_step(w)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"per-head fp8 decode G={G}")


def test_per_head_mixed():
    w = _case(95, [30, 100, 64, 1, 700], 8, q_lens=[1, 20, 64, 1, 300])
    out, _, _ = gpu_step(w)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, "per-head fp8 mixed")


def test_per_head_cascade():
    w = _case(96, [5 * 16 + x for x in (0, 9, 16, 200)], 4, prefix=5, write_new=False)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(w.q[0])
    pa.pa_decode_shared_prefix(out, w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables, w.seq_lens, 5, w.scale, ws,
                               w.k_scale[0:1], w.v_scale[0:1])
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(ws) == pa.PA_OK
    rows, ref = oracle_step(w)
    compare(out, rows, ref, "per-head fp8 cascade")


def test_per_head_scale_count_checked():
    w = _case(97, [40, 50], 2)
    out = torch.empty_like(w.q[0])
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    with pytest.raises(ValueError):
        pa.pa_decode(out, w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables, w.seq_lens, w.scale, ws,
                     w.k_scale[0, :3], w.v_scale[0, :3])
