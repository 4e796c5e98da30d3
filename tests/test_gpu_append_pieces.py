"""The fused decode step (pa_decode_append) on the path where the last ~10% of
the work is handed out at run time in pieces.

That path runs when the warps' ranges are long (at least 48 16-key units per
warp), the cache is 16-bit and a KV head serves at most 4 query heads: the
40-layer GQA decode at 8k contexts is exactly that case.  The new token of a
sequence sits in the sequence's last 16 keys, so with several sequences it
lands both in static ranges (earlier sequences) and in claimed pieces (the
last sequences of the flattened order); the tests check where it lands, then
compare the outputs with the oracle's write-then-decode and the written cache
bytes with the oracle's slot write ("Basics of LLM Inference and vLLM
Internals", s.4: a token's slot comes from its block-table entry)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_99_gb300 as pa
from paged_kv_cache_99_gb300 import workloads as W
from tests._dense import CODE, raw
from tests._gpu import compare, oracle_step

pytestmark = pytest.mark.gpu
DEV = "cuda"

# split of the flattened order, as the library describes it: kDynShare256 / 256 of
# the units in pieces of max(8, range / 8) once a static range holds >= 48 units
DYN_SHARE_256, MIN_PIECE, MIN_PIECE_RANGE = 26, 8, 48


def _split(T, workers):
    per = T // max(workers, 1)
    dyn = 0 if per < MIN_PIECE_RANGE else T * DYN_SHARE_256 // 256
    P = min(workers, dyn // max(MIN_PIECE, per // 8))
    if P <= 0:
        return T, 0
    S = -(-dyn // P)
    return T - dyn, -(-dyn // S)


def _new_token_places(w, workers):
    """(static, pieces): how many (sequence, KV head) units hold their new token in a
    static range and how many in a claimed piece."""
    lens = w.seq_lens.cpu().tolist()
    G = w.num_q_heads // w.num_kv_heads
    UH = w.num_kv_heads * (-(-G // 8))
    blocks = [-(-n // 16) for n in lens]
    T = sum(b * UH for b in blocks)
    Ts, P = _split(T, workers)
    static = pieces = 0
    f = 0
    for b in blocks:
        for _ in range(UH):
            last = f + b - 1
            if last < Ts:
                static += 1
            else:
                pieces += 1
            f += b
    return static, pieces, P


def _scales(w):
    return (w.k_scale[0:1] if w.k_scale is not None else None,
            w.v_scale[0:1] if w.v_scale is not None else None)


def _fused(w, workers=0):
    kc, vc = w.k_cache[0].clone(), w.v_cache[0].clone()
    ks, vs = _scales(w)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(w.q[0])
    pa.pa_decode_append(out, w.q[0], w.k_new[0], w.v_new[0], w.slot_mapping, kc, vc, w.block_tables, w.seq_lens,
                        w.scale, ws, ks, vs, num_workers=workers)
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(ws) == pa.PA_OK
    return out, kc, vc


def _separate(w, workers=0):
    kc, vc = w.k_cache[0].clone(), w.v_cache[0].clone()
    ks, vs = _scales(w)
    pa.pa_reshape_and_cache(w.k_new[0], w.v_new[0], kc, vc, w.slot_mapping, ks, vs)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(w.q[0])
    pa.pa_decode(out, w.q[0], kc, vc, w.block_tables, w.seq_lens, w.scale, ws, ks, vs, num_workers=workers)
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(ws) == pa.PA_OK
    return out, kc, vc


def _written_blocks_match_oracle(w, kc, vc):
    """The blocks holding the new tokens, as the GPU left them, against the oracle's
    slot write into the same blocks as they were before the step."""
    slots = w.slot_mapping.cpu().numpy()
    blocks = sorted({int(s) // w.block_size for s in slots if s >= 0})
    idx = torch.tensor(blocks, dtype=torch.int64, device=DEV)
    remap = {b: i for i, b in enumerate(blocks)}
    sub_slots = np.array([remap[int(s) // w.block_size] * w.block_size + int(s) % w.block_size for s in slots],
                         np.int64)
    ks, vs = (float(w.k_scale[0]), float(w.v_scale[0])) if w.k_scale is not None else (1.0, 1.0)
    ref_k, ref_v = oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), CODE[w.q_dtype],
                                            raw(w.k_cache[0].index_select(0, idx)),
                                            raw(w.v_cache[0].index_select(0, idx)), CODE[w.cache_dtype],
                                            sub_slots, ks, vs)
    assert np.array_equal(raw(kc.index_select(0, idx)), ref_k)
    assert np.array_equal(raw(vc.index_select(0, idx)), ref_v)


@pytest.mark.parametrize("workers", [6, 8, 13])
@pytest.mark.parametrize("cache", ["bf16", "fp16"])
def test_append_claimed_pieces_small(workers, cache):
    lens = [100, 1000, 3000, 2500, 777, 1, 16, 1201]
    w = W.build_workload(name="append-pieces", seed=700 + workers, device=DEV, num_layers=1, seq_lens=lens,
                         q_lens=[1] * len(lens), num_q_heads=8, num_kv_heads=2, q_dtype=cache, cache_dtype=cache)
    static, pieces, P = _new_token_places(w, workers)
    assert P > 0 and static > 0 and pieces > 0, (static, pieces, P)   # both places are exercised
    out, kc, vc = _fused(w, workers)
    ref_out, ref_k, ref_v = _separate(w, workers)
    # the same split with and without the fused write: bit-identical results
    assert torch.equal(kc.view(torch.int16), ref_k.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), ref_v.view(torch.int16))
    assert torch.equal(out, ref_out)
    _written_blocks_match_oracle(w, kc, vc)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"append pieces {cache} W={workers}")


def test_append_claimed_pieces_repeated_calls_one_workspace():
    # the piece counter carries over from call to call in one workspace
    lens = [2000, 3100, 64, 2900]
    w = W.build_workload(name="append-pieces-rep", seed=731, device=DEV, num_layers=1, seq_lens=lens,
                         q_lens=[1] * len(lens), num_q_heads=4, num_kv_heads=1, q_dtype="bf16", cache_dtype="bf16")
    _, pieces, P = _new_token_places(w, 6)
    assert P > 0 and pieces > 0
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    rows, ref = oracle_step(w)
    first = None
    for _ in range(4):
        kc, vc = w.k_cache[0].clone(), w.v_cache[0].clone()
        out = torch.empty_like(w.q[0])
        pa.pa_decode_append(out, w.q[0], w.k_new[0], w.v_new[0], w.slot_mapping, kc, vc, w.block_tables,
                            w.seq_lens, w.scale, ws, num_workers=6)
        torch.cuda.synchronize()
        assert pa.pa_read_device_status(ws) == pa.PA_OK
        compare(out, rows, ref, "repeated call")
        if first is None:
            first = out.clone()
        assert torch.equal(out, first)


def test_append_gqa40_8k_layer_default_workers():
    # one layer of the 40-layer GQA decode, in the launch configuration the
    # benchmark times (default worker count): claimed pieces are on
    w = W.make("gqa40-8k", DEV, num_layers=1)
    try:
        static, pieces, P = _new_token_places(w, pa.pa_default_workers())
        assert P > 0 and pieces > 0 and static > 0, (static, pieces, P)
        out, kc, vc = _fused(w)
        ref_out, ref_k, ref_v = _separate(w)
        assert torch.equal(kc.view(torch.int16), ref_k.view(torch.int16))
        assert torch.equal(vc.view(torch.int16), ref_v.view(torch.int16))
        assert torch.equal(out, ref_out)
        del ref_k, ref_v
        _written_blocks_match_oracle(w, kc, vc)
        # sampled sequences: the first, the last (new tokens in pieces) and two more
        g = np.random.default_rng(5)
        pick = sorted({0, w.num_seqs - 1, w.num_seqs - 2} | set(g.choice(w.num_seqs, 2, replace=False).tolist()))
        rows, ref = oracle_step(w, 0, pick)
        err, rms = compare(out, rows, ref, "gqa40-8k layer, fused step")
        print(f"gqa40-8k fused layer: max err {err:.2e}, rms {rms:.2e}, rows {list(rows)}")
    finally:
        del w
        torch.cuda.empty_cache()
