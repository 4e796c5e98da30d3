"""Parity of the shared-prefix (cascade) decode: the shared blocks as one dense
tensor-core contraction, the private suffixes through the decode kernel, merged
by the combine.  The result must be the oracle's decode of every row over its
whole sequence; the precondition (identical leading table entries, sequences at
least as long as the prefix) is checked on the device."""
import numpy as np
import pytest
import torch

import paged_kv_cache_99_gb300 as pa
from paged_kv_cache_99_gb300 import workloads as W
from tests._gpu import compare, oracle_step

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed, prefix, suffixes, G, Hkv=2, cache="bf16", qd="bf16"):
    lens = [prefix * W.BLOCK_SIZE + x for x in suffixes]
    return W.build_workload(name="cascade", seed=seed, device=DEV, num_layers=1, seq_lens=lens,
                            q_lens=[1] * len(lens), num_q_heads=G * Hkv, num_kv_heads=Hkv, q_dtype=qd,
                            cache_dtype=cache, shared_prefix_blocks=prefix, write_new=False)


def _scales(w):
    return (w.k_scale[0:1] if w.k_scale is not None else None,
            w.v_scale[0:1] if w.v_scale is not None else None)


def _cascade(w, prefix, ws=None, tables=None, lens=None):
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads) if ws is None else ws
    out = torch.empty_like(w.q[0])
    ks, vs = _scales(w)
    pa.pa_decode_shared_prefix(out, w.q[0], w.k_cache[0], w.v_cache[0],
                               w.block_tables if tables is None else tables,
                               w.seq_lens if lens is None else lens, prefix, w.scale, ws, ks, vs)
    torch.cuda.synchronize()
    return out, pa.pa_read_device_status(ws)


# suffix lengths: none, one token, a partial block, exactly one block, one more, longer
SUFFIXES = [0, 1, 15, 16, 17, 200, 531]


@pytest.mark.parametrize("cache,qd", [("bf16", "bf16"), ("fp16", "fp16"), ("fp8", "bf16")])
@pytest.mark.parametrize("G", [1, 4, 6, 8, 12])
@pytest.mark.parametrize("prefix", [3, 8])
def test_cascade_matches_oracle(cache, qd, G, prefix):
    w = _case(60 + G + prefix, prefix, SUFFIXES, G, cache=cache, qd=qd)
    out, st = _cascade(w, prefix)
    assert st == pa.PA_OK, pa.pa_status_string(st)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"cascade {cache} G={G} prefix={prefix}")


@pytest.mark.parametrize("prefix", [37, 40])
def test_cascade_many_rows_long_prefix(prefix):
    # 40 sequences x 8 heads: two CTAs per KV head, the second with one tile; 37 blocks
    # = 592 prefix keys end inside a 128-key step
    g = np.random.default_rng(prefix)
    w = _case(70 + prefix, prefix, g.integers(0, 300, 40).tolist(), 8, cache="fp16", qd="fp16")
    out, st = _cascade(w, prefix)
    assert st == pa.PA_OK, pa.pa_status_string(st)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"cascade, prefix {prefix} blocks")


def test_cascade_without_prefix_is_decode():
    w = _case(80, 0, [5, 16, 300, 1, 77], 4)
    out, st = _cascade(w, 0)
    assert st == pa.PA_OK
    rows, ref = oracle_step(w)
    compare(out, rows, ref, "prefix_blocks = 0")


def test_cascade_consecutive_calls_one_workspace():
    w = _case(81, 5, SUFFIXES, 8, cache="fp8")
    rows, ref = oracle_step(w)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    for prefix in (5, 2, 0, 5):      # any leading part of a shared prefix is itself shared
        out, st = _cascade(w, prefix, ws=ws)
        assert st == pa.PA_OK
        compare(out, rows, ref, f"call with prefix {prefix}")


def test_cascade_agrees_with_decode():
    w = _case(82, 6, SUFFIXES * 3, 6)
    out, st = _cascade(w, 6)
    assert st == pa.PA_OK
    ref_out = torch.empty_like(w.q[0])
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    pa.pa_decode(ref_out, w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables, w.seq_lens, w.scale, ws)
    torch.cuda.synchronize()
    diff = (out.float() - ref_out.float()).abs()
    assert diff.max().item() <= 1e-2 + 1e-2 * ref_out.float().abs().max().item()


def test_cascade_precondition_is_checked():
    w = _case(83, 4, [10, 20, 30], 4)
    # a table whose leading entry differs from sequence 0's
    tables = w.block_tables.clone()
    tables[1, 2] = tables[2, 4]           # a valid block, but not the shared one
    _, st = _cascade(w, 4, tables=tables)
    assert st == pa.PA_ERR_OUT_OF_RANGE
    # a sequence shorter than the prefix
    lens = w.seq_lens.clone()
    lens[2] = 4 * W.BLOCK_SIZE - 3
    _, st = _cascade(w, 4, lens=lens)
    assert st == pa.PA_ERR_OUT_OF_RANGE
    # the same workspace then serves a valid call
    out, st = _cascade(w, 4)
    assert st == pa.PA_OK
    rows, ref = oracle_step(w)
    compare(out, rows, ref, "after rejected calls")


def test_cascade_full_size_shared_prefix_sampled():
    w = W.make("shared-prefix", DEV)
    out, st = _cascade(w, w.shared_prefix_blocks)
    assert st == pa.PA_OK
    assert torch.isfinite(out.float()).all()
    lens = w.seq_lens.cpu().numpy()
    pick = sorted({0, 1, int(lens.argmax()), int(lens.argmin()), 77, w.num_seqs - 1})
    rows, ref = oracle_step(w, 0, pick)
    compare(out, rows, ref, "shared-prefix config, sampled rows")


# ---- the prefix cut into key segments (workspace with room for the extra partials) ----

def _split_ws(w):
    return pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads, shared_prefix=True)


@pytest.mark.parametrize("cache,qd", [("bf16", "bf16"), ("fp16", "fp16"), ("fp8", "bf16")])
@pytest.mark.parametrize("G", [1, 4, 8, 12])
@pytest.mark.parametrize("prefix", [24, 37, 130])
def test_cascade_split_prefix_matches_oracle(cache, qd, G, prefix):
    # 384, 592 and 2080 prefix keys: 3, 5 and 17 steps of 128 keys, the last two
    # ending inside a step; 17 steps over at most 16 segments gives segments of 2
    w = _case(90 + G + prefix, prefix, SUFFIXES, G, cache=cache, qd=qd)
    out, st = _cascade(w, prefix, ws=_split_ws(w))
    assert st == pa.PA_OK, pa.pa_status_string(st)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"split cascade {cache} G={G} prefix={prefix}")


def test_cascade_split_limited_by_workspace():
    # room for two extra partials per row only: three segments
    w = _case(95, 64, SUFFIXES, 4)
    base = pa.pa_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    rows = w.num_seqs * w.num_q_heads
    extra = 2 * rows * 128 * 4 + 256 + 2 * rows * 2 * 4 + 256
    ws = torch.zeros(base + extra, dtype=torch.uint8, device=DEV)
    out, st = _cascade(w, 64, ws=ws)
    assert st == pa.PA_OK
    rows_, ref = oracle_step(w)
    compare(out, rows_, ref, "split limited by workspace")


@pytest.mark.parametrize("bs,prefix", [(8, 75), (32, 20)])
def test_cascade_split_other_block_sizes(bs, prefix):
    lens = [prefix * bs + x for x in SUFFIXES]
    w = W.build_workload(name="cascade", seed=96 + bs, device=DEV, num_layers=1, seq_lens=lens,
                         q_lens=[1] * len(lens), num_q_heads=16, num_kv_heads=2, block_size=bs,
                         shared_prefix_blocks=prefix, write_new=False)
    out, st = _cascade(w, prefix, ws=_split_ws(w))
    assert st == pa.PA_OK
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"split cascade bs={bs}")


def test_cascade_split_long_prefix_sampled():
    # 32 sequences behind an 8192-token prompt: 8 tile-pair CTAs, the prefix cut into
    # segments until the prefix grid covers half the GPU
    w = W.make("shared-prefix-long", DEV)
    out, st = _cascade(w, w.shared_prefix_blocks, ws=_split_ws(w))
    assert st == pa.PA_OK
    assert torch.isfinite(out.float()).all()
    lens = w.seq_lens.cpu().numpy()
    pick = sorted({0, 1, int(lens.argmax()), int(lens.argmin()), w.num_seqs // 2, w.num_seqs - 1})
    rows, ref = oracle_step(w, 0, pick)
    compare(out, rows, ref, "long shared prefix, split, sampled rows")


# ---- more (sequence, KV head) units than resident combine CTAs: one warp merges a unit ----

@pytest.mark.parametrize("cache,qd,G", [("bf16", "bf16", 4), ("fp8", "bf16", 8), ("fp16", "fp16", 12)])
@pytest.mark.parametrize("prefix,split", [(6, False), (40, True)])
def test_cascade_many_units_warp_merge(cache, qd, G, prefix, split):
    # 96 sequences x 8 KV heads (x 2 head groups for G = 12): 768 or 1536 units, more
    # than two combine CTAs per SM; every suffix length class, the prefix whole (6
    # blocks) or cut into key segments (40 blocks = 640 keys with the split workspace)
    g = np.random.default_rng(prefix + G)
    suffixes = (SUFFIXES * 14)[:96]
    suffixes = [int(x) for x in g.permutation(suffixes)]
    w = _case(97 + G + prefix, prefix, suffixes, G, Hkv=8, cache=cache, qd=qd)
    assert w.num_seqs * w.num_kv_heads > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    out, st = _cascade(w, prefix, ws=_split_ws(w) if split else None)
    assert st == pa.PA_OK, pa.pa_status_string(st)
    pick = sorted({0, 1, 2, 3, 5, 6, 47, 94, 95} | {int(i) for i in g.choice(96, 6, replace=False)})
    rows, ref = oracle_step(w, 0, pick)
    compare(out, rows, ref, f"cascade warp merge {cache} G={G} prefix={prefix}")


def test_cascade_claimed_pieces_consecutive_calls():
    # units of 4 query heads over long private suffixes: the suffix decode hands out
    # its last pieces from the workspace counter, and the warp merge (more units than
    # combine CTAs) leaves the counter's base for the next call; three calls on one
    # workspace, then a plain decode and one more cascade, each against the oracle
    g = np.random.default_rng(7)
    suffixes = [int(x) for x in g.integers(1500, 2600, 96)]
    w = _case(131, 6, suffixes, 4, Hkv=8)
    assert w.num_seqs * w.num_kv_heads > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    pick = sorted({0, 1, 47, 94, 95} | {int(i) for i in g.choice(96, 5, replace=False)})
    rows, ref = oracle_step(w, 0, pick)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    for i in range(3):
        out, st = _cascade(w, 6, ws=ws)
        assert st == pa.PA_OK, pa.pa_status_string(st)
        compare(out, rows, ref, f"cascade call {i}")
    dec = torch.empty_like(w.q[0])
    pa.pa_decode(dec, w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables, w.seq_lens, w.scale, ws)
    torch.cuda.synchronize()
    compare(dec, rows, ref, "plain decode in between")
    out, st = _cascade(w, 6, ws=ws)
    assert st == pa.PA_OK
    compare(out, rows, ref, "cascade after the decode")
