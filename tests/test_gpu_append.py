"""pa_decode_append: the slot write of each sequence's new token fused into the
decode.  It must leave the cache bit for bit as pa_reshape_and_cache does, give
exactly the outputs of pa_reshape_and_cache followed by pa_decode, and match the
oracle's write-then-decode."""
import numpy as np
import pytest
import torch

import paged_kv_cache_99_gb300 as pa
from paged_kv_cache_99_gb300 import workloads as W
from tests._dense import raw
from tests._gpu import compare, oracle_step

pytestmark = pytest.mark.gpu
DEV = "cuda"
LENS = [1, 7, 8, 9, 15, 16, 17, 31, 32, 33, 100, 513, 1200, 4000]


def _case(seed, G, cache="bf16", qd="bf16", bs=16, Hkv=2, fp8_scale="tensor", lens=LENS, write_new=True):
    return W.build_workload(name="append", seed=seed, device=DEV, num_layers=1, seq_lens=lens,
                            q_lens=[1] * len(lens), num_q_heads=G * Hkv, num_kv_heads=Hkv, q_dtype=qd,
                            cache_dtype=cache, block_size=bs, fp8_scale=fp8_scale, write_new=write_new)


def _scales(w):
    return (w.k_scale[0:1] if w.k_scale is not None else None,
            w.v_scale[0:1] if w.v_scale is not None else None)


def _separate(w):
    kc, vc = w.k_cache[0].clone(), w.v_cache[0].clone()
    ks, vs = _scales(w)
    pa.pa_reshape_and_cache(w.k_new[0], w.v_new[0], kc, vc, w.slot_mapping, ks, vs)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(w.q[0])
    pa.pa_decode(out, w.q[0], kc, vc, w.block_tables, w.seq_lens, w.scale, ws, ks, vs)
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(ws) == pa.PA_OK
    return out, kc, vc


def _fused(w, slots=None, lens=None):
    kc, vc = w.k_cache[0].clone(), w.v_cache[0].clone()
    ks, vs = _scales(w)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(w.q[0])
    pa.pa_decode_append(out, w.q[0], w.k_new[0], w.v_new[0], w.slot_mapping if slots is None else slots, kc, vc,
                        w.block_tables, w.seq_lens if lens is None else lens, w.scale, ws, ks, vs)
    torch.cuda.synchronize()
    return out, kc, vc, pa.pa_read_device_status(ws)


@pytest.mark.parametrize("cache,qd,fp8_scale", [("bf16", "bf16", "tensor"), ("fp16", "fp16", "tensor"),
                                                ("fp8", "bf16", "tensor"), ("fp8", "fp16", "head")])
@pytest.mark.parametrize("G", [1, 4, 8, 12])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_append_equals_write_then_decode(cache, qd, fp8_scale, G, bs):
    w = _case(500 + G + bs, G, cache=cache, qd=qd, bs=bs, Hkv=4 if fp8_scale == "head" else 2, fp8_scale=fp8_scale)
    out, kc, vc, st = _fused(w)
    assert st == pa.PA_OK, pa.pa_status_string(st)
    ref_out, ref_k, ref_v = _separate(w)
    assert np.array_equal(raw(kc), raw(ref_k)) and np.array_equal(raw(vc), raw(ref_v))
    assert torch.equal(out, ref_out)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"append {cache} G={G} bs={bs}")


def test_append_qwen_layer_sampled():
    w = W.make("qwen2.5-1.5b", DEV, num_layers=1)
    out, kc, vc, st = _fused(w)
    assert st == pa.PA_OK
    ref_out, ref_k, ref_v = _separate(w)
    # compared as bits: the unused slots hold NaN poison
    assert torch.equal(kc.view(torch.int16), ref_k.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), ref_v.view(torch.int16))
    assert torch.equal(out, ref_out)
    lens = w.seq_lens.cpu().numpy()
    pick = sorted({0, int(lens.argmax()), int(lens.argmin()), w.num_seqs - 1})
    rows, ref = oracle_step(w, 0, pick)
    compare(out, rows, ref, "qwen layer, sampled rows")


def test_append_padding_slot_writes_nothing():
    # sequence 2 is padding (slot -1): nothing is written, its poisoned slot is read
    # as it is, exactly as with the separate slot write
    w = _case(520, 4)
    slots = w.slot_mapping.clone()
    slots[2] = -1
    out, kc, vc, st = _fused(w, slots=slots)
    assert st == pa.PA_OK
    ref_k, ref_v = w.k_cache[0].clone(), w.v_cache[0].clone()
    pa.pa_reshape_and_cache(w.k_new[0], w.v_new[0], ref_k, ref_v, slots)
    ref_out = torch.empty_like(out)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    pa.pa_decode(ref_out, w.q[0], ref_k, ref_v, w.block_tables, w.seq_lens, w.scale, ws)
    torch.cuda.synchronize()
    assert torch.equal(kc.view(torch.int16), ref_k.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), ref_v.view(torch.int16))
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))   # bit for bit, NaN rows included


def test_append_wrong_slot_is_recorded_and_not_written():
    w = _case(521, 4)
    slots = w.slot_mapping.clone()
    slots[5] = slots[5] - 1               # a slot of sequence 5, but not position n - 1
    before_k = w.k_cache[0].clone()
    _, kc, _, st = _fused(w, slots=slots)
    assert st == pa.PA_ERR_OUT_OF_RANGE
    b, off = int(slots[5]) // w.block_size, int(slots[5]) % w.block_size
    assert torch.equal(kc[b, :, off].view(torch.int16), before_k[b, :, off].view(torch.int16))


def test_append_empty_sequence_with_a_slot_is_recorded():
    w = _case(522, 4, lens=[1, 40, 17])
    lens_t = torch.tensor([0, 40, 17], dtype=torch.int32, device=DEV)
    out, _, _, st = _fused(w, lens=lens_t)
    assert st == pa.PA_ERR_OUT_OF_RANGE
    assert torch.count_nonzero(out[0]) == 0
