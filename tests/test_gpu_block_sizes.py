"""Blocks of 8 and 32 tokens ("Basics of LLM Inference and vLLM Internals", s.4
and s.11 question 3: the block size trades the last block's waste against the
kernels' contiguous runs; 16 is the default).  The kernels walk the cache in
16-key units, so a 32-token block is read as two units and an 8-token block as
half of one; every path is checked against the oracle, which takes the block
size from the cache shape, with lengths that end anywhere in a block."""
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

# lengths that end on either side of 8-, 16- and 32-token boundaries
LENS = [1, 7, 8, 9, 15, 16, 17, 24, 31, 32, 33, 100, 513, 1200]


def _case(seed, lens, G, bs, cache="bf16", Hkv=2, q_lens=None, prefix=0, write_new=True, qd="bf16",
          fp8_scale="tensor"):
    return W.build_workload(name=f"bs{bs}", seed=seed, device=DEV, num_layers=1, seq_lens=lens,
                            q_lens=q_lens or [1] * len(lens), num_q_heads=G * Hkv, num_kv_heads=Hkv,
                            q_dtype=qd, cache_dtype=cache, block_size=bs, shared_prefix_blocks=prefix,
                            write_new=write_new, fp8_scale=fp8_scale)


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("cache,qd", [("bf16", "bf16"), ("fp16", "fp16"), ("fp8", "bf16"), ("fp8", "fp16")])
def test_slot_write_bit_exact(bs, cache, qd):
    w = _case(300 + bs, LENS, 2, bs, cache=cache, qd=qd)
    assert w.k_cache[0].shape[2] == bs
    kc, vc = w.k_cache[0].clone(), w.v_cache[0].clone()
    ks = w.k_scale[0:1] if w.k_scale is not None else None
    vs = w.v_scale[0:1] if w.v_scale is not None else None
    pa.pa_reshape_and_cache(w.k_new[0], w.v_new[0], kc, vc, w.slot_mapping, ks, vs)
    torch.cuda.synchronize()
    ek, ev = oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), CODE[qd], raw(w.k_cache[0]),
                                      raw(w.v_cache[0]), CODE[cache], w.slot_mapping.cpu().numpy(),
                                      float(ks) if ks is not None else 1.0, float(vs) if vs is not None else 1.0)
    assert np.array_equal(raw(kc), ek) and np.array_equal(raw(vc), ev)


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("cache", ["bf16", "fp8"])
@pytest.mark.parametrize("G", [1, 4, 8, 12])
def test_decode(bs, cache, G):
    w = _case(310 + bs + G, LENS, G, bs, cache=cache)
    out, _, _ = gpu_step(w)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"decode bs={bs} {cache} G={G}")


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("workers", [1, 7, 40, 333])
def test_decode_worker_splits(bs, workers):
    # ranges that start and end inside sequences, and inside the two halves of a
    # 32-token block
    w = _case(330 + workers, [45, 200, 17, 640, 9, 333], 4, bs, cache="fp16", qd="fp16")
    out, _, _ = gpu_step(w, num_workers=workers)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"decode bs={bs} workers={workers}")


@pytest.mark.parametrize("bs", [8, 32])
def test_decode_fp8_per_head(bs):
    w = _case(340 + bs, LENS, 4, bs, cache="fp8", Hkv=4, fp8_scale="head")
    out, _, _ = gpu_step(w)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"per-head fp8 decode bs={bs}")


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("cache,G", [("bf16", 4), ("bf16", 8), ("fp8", 8), ("fp16", 1)])
def test_mixed(bs, cache, G):
    # chunks that start mid-block, span several 128-key steps and end ragged
    lens = [30, 100, 64, 1, 700, 9, 385]
    q_lens = [1, 20, 64, 1, 300, 9, 1]
    qd = "fp16" if cache == "fp16" else "bf16"
    w = _case(350 + bs + G, lens, G, bs, cache=cache, q_lens=q_lens, qd=qd)
    out, _, _ = gpu_step(w)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"mixed bs={bs} {cache} G={G}")


@pytest.mark.parametrize("bs,prefix", [(8, 4), (8, 7), (8, 1), (32, 2), (32, 3)])
@pytest.mark.parametrize("cache", ["bf16", "fp8"])
def test_shared_prefix(bs, prefix, cache):
    # an odd number of 8-token blocks: the split falls at the last 16-key boundary
    # inside the prefix, the rest is read with each sequence's own blocks
    lens = [prefix * bs + x for x in (0, 1, 9, 16, 40, 300)]
    w = _case(360 + bs + prefix, lens, 4, bs, cache=cache, prefix=prefix, write_new=False)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(w.q[0])
    ks = w.k_scale[0:1] if w.k_scale is not None else None
    vs = w.v_scale[0:1] if w.v_scale is not None else None
    pa.pa_decode_shared_prefix(out, w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables, w.seq_lens, prefix,
                               w.scale, ws, ks, vs)
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(ws) == pa.PA_OK
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"shared prefix bs={bs} prefix={prefix} {cache}")


@pytest.mark.parametrize("bs", [8, 32])
def test_shared_prefix_violation_recorded(bs):
    # sequence 1's table differs from sequence 0's inside the shared part
    w = _case(370 + bs, [64 + 5, 64 + 20, 64 + 3], 4, bs, prefix=64 // bs, write_new=False)
    tables = w.block_tables.clone()
    tables[1, 0] = tables[2, 0] = int(tables[0, 1])
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(w.q[0])
    pa.pa_decode_shared_prefix(out, w.q[0], w.k_cache[0], w.v_cache[0], tables, w.seq_lens, 64 // bs, w.scale, ws)
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(ws) == pa.PA_ERR_OUT_OF_RANGE


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("cache", ["bf16", "fp8"])
def test_copy_blocks_bit_exact(bs, cache):
    g = torch.Generator().manual_seed(bs)
    nb, hkv = 200, 4
    if cache == "fp8":
        k = torch.randint(0, 256, (nb, hkv, bs, 128), generator=g, dtype=torch.uint8)
        v = torch.randint(0, 256, (nb, hkv, bs, 128), generator=g, dtype=torch.uint8)
    else:
        k = torch.randn(nb, hkv, bs, 128, generator=g).to(torch.bfloat16)
        v = torch.randn(nb, hkv, bs, 128, generator=g).to(torch.bfloat16)
    k, v = k.to(DEV), v.to(DEV)
    perm = torch.randperm(nb, generator=g)
    src, dst = perm[:60].int(), perm[60:120].int()
    want_k, want_v = raw(k).copy(), raw(v).copy()
    want_k[dst.numpy()] = want_k[src.numpy()]
    want_v[dst.numpy()] = want_v[src.numpy()]
    pa.pa_copy_blocks(k, v, src.to(DEV), dst.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(raw(k), want_k) and np.array_equal(raw(v), want_v)


@pytest.mark.parametrize("bs", [4, 64, 12])
def test_other_block_sizes_rejected(bs):
    w = _case(380, [40, 50], 2, 16)
    q = w.q[0]
    kc = torch.zeros(8, 2, bs, 128, dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    out = torch.empty_like(q)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.pa_decode(out, q, kc, vc, w.block_tables, w.seq_lens, w.scale, ws)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    with pytest.raises(pa.PagedAttentionError):
        pa.pa_reshape_and_cache(w.k_new[0], w.v_new[0], kc, vc, w.slot_mapping)


def test_same_tokens_same_result_across_block_sizes():
    # the same keys and values stored in blocks of 8, 16 and 32: the attention
    # output does not depend on the block size (only the summation order can)
    lens = [5, 77, 300, 1]
    outs = []
    base = _case(390, lens, 4, 16, write_new=False)
    for bs in (8, 16, 32):
        w = _case(390, lens, 4, bs, write_new=False)
        # copy base's token rows into this layout
        kc, vc = torch.zeros_like(w.k_cache[0]), torch.zeros_like(w.v_cache[0])
        bt, bbt = w.block_tables.cpu(), base.block_tables.cpu()
        for s, n in enumerate(lens):
            for t in range(n):
                src = int(bbt[s, t // 16]), t % 16
                dst = int(bt[s, t // bs]), t % bs
                kc[dst[0], :, dst[1]] = base.k_cache[0][src[0], :, src[1]]
                vc[dst[0], :, dst[1]] = base.v_cache[0][src[0], :, src[1]]
        out = torch.empty_like(base.q[0])
        ws = pa.new_workspace(len(lens), base.num_q_heads, base.num_kv_heads)
        pa.pa_decode(out, base.q[0], kc, vc, w.block_tables, w.seq_lens, base.scale, ws)
        torch.cuda.synchronize()
        assert pa.pa_read_device_status(ws) == pa.PA_OK
        outs.append(out.float().cpu())
    assert torch.allclose(outs[0], outs[1], atol=2e-3, rtol=2e-3)
    assert torch.allclose(outs[2], outs[1], atol=2e-3, rtol=2e-3)
