"""GPU parity: the library's kernels, called through the C ABI, against the oracle
on the same seeded inputs.  Slot writes are compared byte for byte; attention
element by element within |err| <= 1e-2 + 1e-2 |ref|."""
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


def _case(seed, lens, G, Hkv=2, cache="bf16", qd="bf16", q_lens=None, prefix=0, extra=16, write_new=True):
    return W.build_workload(name="t", seed=seed, device=DEV, num_layers=1, seq_lens=lens,
                            q_lens=q_lens or [1] * len(lens), num_q_heads=G * Hkv, num_kv_heads=Hkv,
                            q_dtype=qd, cache_dtype=cache, extra_blocks=extra, write_new=write_new,
                            shared_prefix_blocks=prefix)


# ---------------------------------------------------------------- slot write

@pytest.mark.parametrize("cache,qd", [("bf16", "bf16"), ("fp16", "fp16"), ("fp8", "bf16"), ("fp8", "fp16")])
def test_reshape_bit_exact(cache, qd):
    w = _case(21, [5, 16, 17, 40, 300], 4, cache=cache, qd=qd)
    kc, vc = w.k_cache[0].clone(), w.v_cache[0].clone()
    ks = w.k_scale[0:1] if w.k_scale is not None else None
    vs = w.v_scale[0:1] if w.v_scale is not None else None
    pa.pa_reshape_and_cache(w.k_new[0], w.v_new[0], kc, vc, w.slot_mapping, ks, vs)
    torch.cuda.synchronize()
    ek, ev = oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), CODE[qd], raw(w.k_cache[0]),
                                      raw(w.v_cache[0]), CODE[cache], w.slot_mapping.cpu().numpy(),
                                      float(ks) if ks is not None else 1.0, float(vs) if vs is not None else 1.0)
    assert np.array_equal(raw(kc), ek) and np.array_equal(raw(vc), ev)


@pytest.mark.parametrize("scale", [1.0, 5.9 / 448, 2.0 ** -4, 1e-3, 0.37, 3e-6])
@pytest.mark.parametrize("src", ["bf16", "fp16"])
def test_reshape_fp8_every_16bit_value(scale, src):
    # every 16-bit pattern once (NaN, inf, subnormals, -0, values that saturate)
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    H = 4
    T = 65536 // (H * 128)
    x = bits.view(torch.bfloat16 if src == "bf16" else torch.float16).reshape(T, H, 128).to(DEV)
    y = x.flip(0).contiguous()
    nb = T // 16 + 2
    kc = torch.full((nb, H, 16, 128), 0x5A, dtype=torch.uint8, device=DEV)
    vc = kc.clone()
    slots = torch.randperm(nb * 16, generator=torch.Generator().manual_seed(3))[:T].to(DEV)
    ks = torch.tensor([scale], dtype=torch.float32, device=DEV)
    vs = torch.tensor([scale * 1.5], dtype=torch.float32, device=DEV)
    k0, v0 = raw(kc), raw(vc)
    pa.pa_reshape_and_cache(x, y, kc, vc, slots, ks, vs)
    torch.cuda.synchronize()
    ek, ev = oracle.reshape_and_cache(raw(x), raw(y), CODE[src], k0, v0, oracle.FP8_E4M3,
                                      slots.cpu().numpy(), float(ks), float(vs))
    gk, gv = raw(kc), raw(vc)
    mism = np.nonzero(gk.ravel() != ek.ravel())[0]
    assert mism.size == 0, [(hex(gk.ravel()[i]), hex(ek.ravel()[i])) for i in mism[:8]]
    assert np.array_equal(gv, ev)


def test_reshape_skips_negative_and_out_of_pool_slots():
    w = _case(22, [8, 9, 30], 4)
    kc, vc = w.k_cache[0].clone(), w.v_cache[0].clone()
    slots = w.slot_mapping.clone()
    slots[0] = -1
    slots[1] = w.num_blocks * 16 + 3
    pa.pa_reshape_and_cache(w.k_new[0], w.v_new[0], kc, vc, slots)
    torch.cuda.synchronize()
    sl = slots.cpu().numpy().copy()
    sl[1] = -1   # the oracle rejects an out-of-pool slot; the library skips it
    ek, _ = oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), oracle.BF16, raw(w.k_cache[0]),
                                     raw(w.v_cache[0]), oracle.BF16, sl)
    assert np.array_equal(raw(kc), ek)


# ---------------------------------------------------------------- decode

def test_tiny_config():
    w = W.tiny(DEV)
    out, kc, vc = gpu_step(w)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, "tiny")
    # the slot write happened exactly as the oracle's
    ek, ev = oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), oracle.BF16, raw(w.k_cache[0]),
                                      raw(w.v_cache[0]), oracle.BF16, w.slot_mapping.cpu().numpy())
    assert np.array_equal(raw(kc), ek) and np.array_equal(raw(vc), ev)


@pytest.mark.parametrize("G", [1, 4, 6, 8, 12])
@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("workers", [1, 2, 7, 0])
def test_decode_sweep(G, seed, workers):
    g = np.random.default_rng(500 + seed)
    lens = g.integers(1, 301, size=9).tolist() + [1, 16, 17]
    w = _case(seed, lens, G)
    out, _, _ = gpu_step(w, num_workers=workers)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"G={G} seed={seed} workers={workers}")


@pytest.mark.parametrize("cache,qd", [("fp16", "fp16"), ("fp8", "bf16"), ("fp8", "fp16")])
@pytest.mark.parametrize("workers", [3, 0])
def test_decode_other_dtypes(cache, qd, workers):
    w = _case(31, [1, 15, 16, 33, 200, 511], 4, Hkv=3, cache=cache, qd=qd)
    out, _, _ = gpu_step(w, num_workers=workers)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"{cache}/{qd}")


def test_decode_empty_sequences_give_zeros():
    w = _case(32, [0, 20, 0, 5], 4, write_new=False)
    out, _, _ = gpu_step(w)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    rows, ref = oracle_step(w, seqs=[1, 3])
    compare(out, rows, ref, "non-empty rows")


def test_decode_long_context_many_splits():
    w = _case(33, [32768, 5000, 3], 8, Hkv=1, write_new=False, extra=4)
    for workers in (1, 64, 0):
        out, _, _ = gpu_step(w, num_workers=workers)
        rows, ref = oracle_step(w)
        compare(out, rows, ref, f"workers={workers}")


def test_decode_placement_does_not_matter_bit_exact():
    w = _case(34, [3, 16, 33, 200, 129, 1000], 6, write_new=False, extra=40)
    a, _, _ = gpu_step(w)
    pi = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(9)).to(DEV)
    kc2 = torch.empty_like(w.k_cache[0])
    vc2 = torch.empty_like(w.v_cache[0])
    kc2[pi] = w.k_cache[0]
    vc2[pi] = w.v_cache[0]
    bt = w.block_tables
    bt2 = torch.where(bt >= 0, pi[bt.clamp(min=0).long()].int(), bt)
    b, _, _ = gpu_step(w, k_cache=kc2, v_cache=vc2, tables=bt2)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_decode_shared_prefix_equals_private_copies_bit_exact():
    w = _case(35, [40, 75, 33, 64, 100], 4, prefix=2, write_new=False, extra=4)
    a, _, _ = gpu_step(w)
    bt = w.block_tables.clone()
    prefix = bt[0, :2].clone()
    extra = []
    for s in range(1, w.num_seqs):
        for j in range(2):
            extra.append(int(prefix[j]))
            bt[s, j] = w.num_blocks + len(extra) - 1
    idx = torch.tensor(extra, device=DEV)
    kc2 = torch.cat([w.k_cache[0], w.k_cache[0][idx]])
    vc2 = torch.cat([w.v_cache[0], w.v_cache[0][idx]])
    b, _, _ = gpu_step(w, k_cache=kc2, v_cache=vc2, tables=bt)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_decode_v_equal_one_gives_one():
    w = _case(36, [1, 15, 16, 17, 290, 3000], 8, write_new=False)
    vc = torch.ones_like(w.v_cache[0])
    out, _, _ = gpu_step(w, v_cache=vc, num_workers=5)
    assert torch.allclose(out.float(), torch.ones_like(out, dtype=torch.float32), atol=8e-3, rtol=0)


def test_decode_one_hot_values_expose_every_block():
    lens = [5, 16, 37, 100, 255, 2047]
    w = _case(37, lens, 4, write_new=False)
    vc = torch.zeros_like(w.v_cache[0])
    for s, n in enumerate(lens):
        for j in range(-(-n // 16)):
            vc[int(w.block_tables[s, j]), :, :, j % 128] = 1.0
    q0 = torch.zeros_like(w.q[0])
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    for workers in (1, 3, 0):
        out = torch.empty_like(q0)
        pa.pa_decode(out, q0, w.k_cache[0], vc, w.block_tables, w.seq_lens, w.scale, ws, num_workers=workers)
        torch.cuda.synchronize()
        for s, n in enumerate(lens):
            exp = torch.zeros(128, dtype=torch.float64)
            for j in range(-(-n // 16)):
                exp[j % 128] += min(16, n - 16 * j) / n
            got = out[s].double().cpu()
            assert torch.allclose(got, exp.expand_as(got), atol=2e-3, rtol=4e-3), (s, workers)


def test_out_of_range_table_entry_is_recorded_not_faulted():
    w = _case(38, [40, 40], 4, write_new=False)
    bt = w.block_tables.clone()
    bt[1, 1] = w.num_blocks + 5
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(w.q[0])
    pa.pa_decode(out, w.q[0], w.k_cache[0], w.v_cache[0], bt, w.seq_lens, w.scale, ws)
    assert pa.pa_read_device_status(ws) == pa.PA_ERR_OUT_OF_RANGE
    rows, ref = oracle_step(w, seqs=[0])
    compare(out, rows, ref, "untouched sequence")
    assert pa.pa_read_device_status(ws) == pa.PA_OK   # cleared


def test_bounded_wait_times_out_and_context_survives():
    ws = pa.new_workspace(4, 8, 2)
    pa.pa_selftest_wait_timeout(ws, 2000)
    assert pa.pa_read_device_status(ws) == pa.PA_ERR_TIMEOUT
    w = W.tiny(DEV)
    out, _, _ = gpu_step(w, workspace=ws)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, "after timeout")


def test_workspace_needs_no_initialisation():
    w = _case(39, [3000, 10, 700], 8, write_new=False)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    for fill in (0xFF, 0x7F, 0x00):
        ws[256:].fill_(fill)          # scratch holds garbage (NaN patterns for 0xFF / 0x7F)
        out, _, _ = gpu_step(w, workspace=ws, num_workers=40)
        rows, ref = oracle_step(w)
        compare(out, rows, ref, f"scratch filled with {fill:#x}")


# ---------------------------------------------------------------- mixed batch

@pytest.mark.parametrize("cache,qd", [("bf16", "bf16"), ("fp16", "fp16"), ("fp8", "bf16")])
@pytest.mark.parametrize("G", [1, 4, 6, 8])
def test_mixed_small(cache, qd, G):
    lens = [30, 100, 64, 1, 77, 200, 19, 513]
    qls = [1, 20, 64, 1, 3, 130, 19, 2]
    w = _case(40 + G, lens, G, cache=cache, qd=qd, q_lens=qls)
    out, _, _ = gpu_step(w)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, f"mixed {cache} G={G}")


def test_mixed_decode_rows_only():
    w = _case(48, [10, 300, 45], 4, q_lens=[1, 1, 1])
    out = torch.empty_like(w.q[0])
    kc, vc = w.k_cache[0].clone(), w.v_cache[0].clone()
    pa.pa_reshape_and_cache(w.k_new[0], w.v_new[0], kc, vc, w.slot_mapping)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    pa.pa_mixed(out, w.q[0], w.query_start_loc, kc, vc, w.block_tables, w.seq_lens, 1, w.scale, ws)
    torch.cuda.synchronize()
    rows, ref = oracle_step(w)
    compare(out, rows, ref, "mixed decode-only")


def test_mixed_zero_length_rows_and_whole_prompt_chunk():
    lens = [64, 50, 33]
    qls = [0, 50, 1]          # no rows; a chunk that is the whole prompt; a decode row
    w = _case(49, lens, 8, Hkv=1, q_lens=qls)
    out, _, _ = gpu_step(w)
    rows, ref = oracle_step(w)
    compare(out, rows, ref, "zero-length + full prompt")


@pytest.mark.parametrize("bad", ["chunk_past_end", "decode_row_past_end"])
def test_mixed_rows_outside_q_are_recorded_not_faulted(bad):
    # query_start_loc naming rows past total_q: the kernels check every row range
    # against the size of q before touching it, record the error and skip the row
    lens, qls = [30, 100, 45], [1, 20, 1]
    w = _case(51, lens, 4, q_lens=qls, write_new=False)
    qsl = w.query_start_loc.clone()
    total_q = int(qsl[-1])
    if bad == "chunk_past_end":
        qsl[3] = total_q + 9          # sequence 2 becomes a chunk running 9 rows past the end of q
    else:
        qsl[2] = total_q + 3          # sequence 2's decode row is past the end of q (and
        qsl[3] = total_q + 4          # sequence 1's chunk with it)
    out = torch.zeros_like(w.q[0])
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    pa.pa_mixed(out, w.q[0], qsl, w.k_cache[0], w.v_cache[0], w.block_tables, w.seq_lens, 30, w.scale, ws)
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(ws) == pa.PA_ERR_OUT_OF_RANGE
    # the well-formed decode row of sequence 0 is still right
    rows, ref = oracle_step(w, seqs=[0])
    compare(out, rows, ref, "untouched decode row")


# ------------------------------------------------ claimed pieces (dynamic tail)

@pytest.mark.parametrize("workers", [4, 16, 40])
def test_claimed_pieces_many_calls_one_workspace(workers):
    # long ranges per worker: the last share of the blocks goes to pieces claimed from
    # the workspace counter; consecutive calls on one workspace keep numbering them right
    w = _case(60 + workers, [3000, 40, 1, 2500, 777, 64], 4, write_new=False)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads)
    rows, ref = oracle_step(w)
    outs = []
    for _ in range(4):
        out, _, _ = gpu_step(w, num_workers=workers, workspace=ws)
        compare(out, rows, ref, f"pieces, {workers} workers")
        outs.append(out)
    assert all(torch.equal(outs[0], o) for o in outs[1:])   # merged in slot order: reproducible


def test_claimed_pieces_after_a_timeout_and_other_calls():
    # a timed-out call, a plain decode and a mixed batch in between leave the counter usable
    # (units of 4 query heads: the ones that take claimed pieces)
    w = _case(64, [2000, 3000, 100], 4, write_new=False)
    ws = pa.new_workspace(16, 64, 8)
    pa.pa_selftest_wait_timeout(ws, 2000)
    assert pa.pa_read_device_status(ws) == pa.PA_ERR_TIMEOUT
    rows, ref = oracle_step(w)
    out, _, _ = gpu_step(w, num_workers=8, workspace=ws)
    compare(out, rows, ref, "after timeout")
    m = _case(65, [30, 100, 64], 4, q_lens=[1, 20, 64])
    mo, _, _ = gpu_step(m, workspace=ws)
    mrows, mref = oracle_step(m)
    compare(mo, mrows, mref, "mixed in between")
    out, _, _ = gpu_step(w, num_workers=8, workspace=ws)
    compare(out, rows, ref, "after mixed")
