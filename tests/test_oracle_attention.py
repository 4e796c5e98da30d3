"""Pins of the oracle's paged attention (decode and mixed) against things other
than itself: a dense library attention, closed forms, the pages' worked example
and the invariants the pages state."""
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_99_gb300 import workloads as W
from tests._dense import CODE, dense_kv, oracle_decode, raw, sdpa, values, workload_values

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _case(seed, lens, G, Hkv=2, cache="bf16", qd="bf16", extra=8, write_new=False, q_lens=None, prefix=0):
    return W.build_workload(name="t", seed=seed, device="cpu", num_layers=1, seq_lens=lens,
                            q_lens=q_lens or [1] * len(lens), num_q_heads=G * Hkv, num_kv_heads=Hkv,
                            q_dtype=qd, cache_dtype=cache, extra_blocks=extra, write_new=write_new,
                            shared_prefix_blocks=prefix)


def _dense_decode(w, layer=0):
    kc, vc = workload_values(w, layer)
    q = values(w.q[layer])
    tables = w.block_tables.numpy()
    out = np.zeros_like(q)
    for s, n in enumerate(w.seq_lens.tolist()):
        if n == 0:
            continue
        K, V = dense_kv(kc, vc, tables[s], n)
        out[s] = sdpa(q[s:s + 1], K, V, w.scale)[0]
    return out


# -- equality with dense attention (pins gather, grouping, softmax) ---------------

@pytest.mark.parametrize("G", [1, 4, 6, 8])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_decode_equals_dense_sdpa(G, seed):
    g = np.random.default_rng(100 + seed)
    lens = g.integers(1, 301, size=5).tolist()
    w = _case(seed, lens, G)
    got = oracle_decode(w)
    ref = _dense_decode(w)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("cache,qd", [("fp16", "fp16"), ("fp8", "bf16"), ("fp8", "fp16")])
def test_decode_equals_dense_other_dtypes(cache, qd):
    w = _case(11, [1, 17, 64, 250], 4, cache=cache, qd=qd)
    np.testing.assert_allclose(oracle_decode(w), _dense_decode(w), atol=1e-12, rtol=0)


def test_tiny_config_equals_dense():
    w = W.tiny("cpu")
    kc, vc = raw(w.k_cache[0]), raw(w.v_cache[0])
    kc, vc = oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), oracle.BF16, kc, vc, oracle.BF16,
                                      w.slot_mapping.numpy())
    got = oracle_decode(w, k_cache=kc, v_cache=vc)
    assert np.all(np.isfinite(got))
    # dense: the context read back from the pool plus the new token appended
    kv, vv = values(torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16)), \
        values(torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16))
    q = values(w.q[0])
    for s, n in enumerate(w.seq_lens.tolist()):
        K, V = dense_kv(kv, vv, w.block_tables[s].numpy(), n)
        np.testing.assert_array_equal(K[-1], values(w.k_new[0][s]))
        np.testing.assert_allclose(got[s], sdpa(q[s:s + 1], K, V, w.scale)[0], atol=1e-12, rtol=0)


def test_empty_sequence_yields_zeros():
    w = _case(3, [0, 20, 0, 5], 4)
    got = oracle_decode(w)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    np.testing.assert_allclose(got[[1, 3]], _dense_decode(w)[[1, 3]], atol=1e-12, rtol=0)


def test_bad_table_entry_is_an_error():
    w = _case(4, [40], 4)
    bt = w.block_tables.numpy().copy()
    bt[0, 1] = w.num_blocks  # out of the pool, inside the sequence
    with pytest.raises(ValueError):
        oracle_decode(w, tables=bt)
    bt = w.block_tables.numpy().copy()
    bt[0, 2] = -5            # the last needed block
    with pytest.raises(ValueError):
        oracle_decode(w, tables=bt)


# -- invariants the pages state ---------------------------------------------------

def test_physical_placement_is_irrelevant():
    # blocks "can live anywhere": relabel every physical block by a permutation
    w = _case(5, [3, 16, 33, 200, 129], 6, extra=20)
    kc, vc = raw(w.k_cache[0]), raw(w.v_cache[0])
    pi = np.random.default_rng(9).permutation(w.num_blocks)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[pi], vc2[pi] = kc, vc
    bt = w.block_tables.numpy()
    bt2 = np.where(bt >= 0, pi[np.clip(bt, 0, None)], -1).astype(np.int32)
    a = oracle_decode(w)
    b = oracle_decode(w, k_cache=kc2, v_cache=vc2, tables=bt2)
    assert np.array_equal(a, b)


def test_shared_prefix_equals_private_copies():
    w = _case(6, [40, 75, 33, 64], 4, prefix=2, extra=4)
    kc, vc = raw(w.k_cache[0]), raw(w.v_cache[0])
    bt = w.block_tables.numpy().copy()
    prefix = bt[0, :2].copy()
    assert all((bt[s, :2] == prefix).all() for s in range(4))
    # give every sequence but the first its own copy of the prefix blocks
    extra = []
    for s in range(1, 4):
        for j in range(2):
            extra.append(prefix[j])
            bt[s, j] = w.num_blocks + len(extra) - 1
    kc2 = np.concatenate([kc, kc[extra]])
    vc2 = np.concatenate([vc, vc[extra]])
    a = oracle_decode(w)
    b = oracle_decode(w, k_cache=kc2, v_cache=vc2, tables=bt)
    assert np.array_equal(a, b)


def test_sequences_do_not_attend_to_each_other():
    w = _case(7, [50, 50], 4, extra=0)
    kc, vc = raw(w.k_cache[0]).copy(), raw(w.v_cache[0]).copy()
    a = oracle_decode(w, k_cache=kc, v_cache=vc)
    own = w.block_tables[1, :4].numpy()
    kc[own] ^= 0x0100   # perturb sequence 1's blocks only
    vc[own] ^= 0x0100
    b = oracle_decode(w, k_cache=kc, v_cache=vc)
    assert np.array_equal(a[0], b[0]) and not np.array_equal(a[1], b[1])


def _worked_example():
    rows = {}
    with open(os.path.join(GOLDEN, "worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                p = line.split()
                rows[p[0]] = (int(p[1]), [int(x) for x in p[2:]])
    return rows


def test_pages_worked_example_shared_block():
    ex = _worked_example()
    (nA, tA), (nB, tB) = ex["A"], ex["B"]
    assert len(tA) == oracle.num_logical_blocks(nA) and oracle.last_block_fill(nA) == 6
    rng = np.random.default_rng(12)
    Hkv, G, d, nb = 1, 4, 128, 8
    kc = torch.randn(nb, Hkv, 16, d, generator=torch.Generator().manual_seed(1)).bfloat16()
    vc = torch.randn(nb, Hkv, 16, d, generator=torch.Generator().manual_seed(2)).bfloat16()
    q1 = torch.randn(1, G * Hkv, d, generator=torch.Generator().manual_seed(3)).bfloat16()
    q = raw(torch.cat([q1, q1, q1]))
    bt = np.full((3, 3), -1, np.int32)
    bt[0, :3] = tA
    bt[1, :1] = tB
    bt[2, :3] = tA
    lens = np.array([nA, nB, nB], np.int32)   # row 2: A read up to B's length
    out = oracle.decode(q, oracle.BF16, raw(kc), raw(vc), oracle.BF16, bt, lens, 128 ** -0.5)
    assert np.array_equal(out[1], out[2])     # B sees exactly A's first 16 tokens
    assert not np.array_equal(out[0], out[1])
    del rng


# -- closed forms -----------------------------------------------------------------

def _set_all(cache_bits, value_bits):
    c = cache_bits.copy()
    c[...] = value_bits
    return c


def test_v_equal_one_gives_one():
    w = _case(8, [1, 15, 16, 17, 290], 8)
    vc = _set_all(raw(w.v_cache[0]), 0x3F80)     # bf16 1.0
    got = oracle_decode(w, v_cache=vc)
    np.testing.assert_allclose(got, 1.0, atol=1e-14, rtol=0)


def test_zero_query_gives_mean_of_values():
    w = _case(9, [1, 7, 16, 45, 100], 4)
    q = np.zeros_like(raw(w.q[0]))
    got = oracle_decode(w, q=q)
    kc, vc = workload_values(w)
    for s, n in enumerate(w.seq_lens.tolist()):
        _, V = dense_kv(kc, vc, w.block_tables[s].numpy(), n)
        mean = V.mean(axis=0)                              # [Hkv, d]
        np.testing.assert_allclose(got[s], np.repeat(mean, 4, axis=0), atol=1e-13, rtol=0)


def test_dominant_key_selects_its_value():
    w = _case(10, [77], 1, Hkv=1)
    kc = raw(w.k_cache[0]).copy()
    qv = values(w.q[0])[0, 0]
    t = 37
    phys, off = int(w.block_tables[0, t // 16]), t % 16
    big = torch.from_numpy(40 * qv / np.linalg.norm(qv)).bfloat16()
    kc[phys, 0, off] = raw(big)
    got = oracle_decode(w, k_cache=kc)
    _, vv = workload_values(w)
    np.testing.assert_allclose(got[0, 0], vv[phys, 0, off], atol=1e-9, rtol=0)


def test_one_hot_values_expose_every_block():
    lens = [5, 16, 37, 100, 255]
    w = _case(13, lens, 4)
    vc = np.zeros_like(raw(w.v_cache[0]))
    for s, n in enumerate(lens):
        for j in range(oracle.num_logical_blocks(n)):
            vc[int(w.block_tables[s, j]), :, :, j % 128] = 0x3F80   # V = e_j for logical block j
    got = oracle_decode(w, q=np.zeros_like(raw(w.q[0])), v_cache=vc)
    for s, n in enumerate(lens):
        exp = np.zeros(128)
        for j in range(oracle.num_logical_blocks(n)):
            exp[j % 128] += min(16, n - 16 * j) / n
        np.testing.assert_allclose(got[s], np.tile(exp, (4 * 2, 1)), atol=1e-14, rtol=0)


# -- mixed batch -------------------------------------------------------------------

def _oracle_mixed(w, layer=0, k_cache=None, v_cache=None):
    return oracle.mixed(raw(w.q[layer]), CODE[w.q_dtype], w.query_start_loc.numpy(),
                        raw(w.k_cache[layer]) if k_cache is None else k_cache,
                        raw(w.v_cache[layer]) if v_cache is None else v_cache,
                        CODE[w.cache_dtype], w.block_tables.numpy(), w.seq_lens.numpy(), w.scale,
                        float(w.k_scale[layer]) if w.k_scale is not None else 1.0,
                        float(w.v_scale[layer]) if w.v_scale is not None else 1.0)


@pytest.mark.parametrize("cache", ["bf16", "fp8"])
def test_mixed_equals_dense_causal(cache):
    lens, qls = [30, 100, 64, 1, 77], [1, 20, 64, 1, 3]
    w = _case(14, lens, 4, cache=cache, q_lens=qls)
    got = _oracle_mixed(w)
    kc, vc = workload_values(w)
    q = values(w.q[0])
    qsl = w.query_start_loc.tolist()
    for s, (n, ql) in enumerate(zip(lens, qls)):
        K, V = dense_kv(kc, vc, w.block_tables[s].numpy(), n)
        pos = n - ql + np.arange(ql)
        mask = np.arange(n)[None, :] <= pos[:, None]            # query j sees keys 0..pos_j
        ref = sdpa(q[qsl[s]:qsl[s + 1]], K, V, w.scale, mask=mask)
        np.testing.assert_allclose(got[qsl[s]:qsl[s + 1]], ref, atol=1e-12, rtol=0)


def test_mixed_rows_equal_decode_of_prefix():
    lens, qls = [40, 90], [1, 25]
    w = _case(15, lens, 6, q_lens=qls)
    got = _oracle_mixed(w)
    qsl = w.query_start_loc.tolist()
    q = raw(w.q[0])
    for s, (n, ql) in enumerate(zip(lens, qls)):
        for j in range(ql):
            row = qsl[s] + j
            one = oracle.decode(q[row:row + 1], oracle.BF16, raw(w.k_cache[0]), raw(w.v_cache[0]), oracle.BF16,
                                w.block_tables[s:s + 1].numpy(), np.array([n - ql + j + 1], np.int32), w.scale)
            assert np.array_equal(one[0], got[row])


# -- slot write -------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_reshape_16bit_places_bits_and_leaves_the_rest(dtype):
    w = _case(16, [5, 16, 17, 40], 4, cache=dtype, qd=dtype, write_new=True)
    kc0, vc0 = raw(w.k_cache[0]), raw(w.v_cache[0])
    slots = w.slot_mapping.numpy()
    kc, vc = oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), CODE[dtype], kc0, vc0, CODE[dtype], slots)
    exp_k, exp_v = kc0.copy(), vc0.copy()
    for t, sl in enumerate(slots):
        exp_k[sl // 16, :, sl % 16, :] = raw(w.k_new[0][t])
        exp_v[sl // 16, :, sl % 16, :] = raw(w.v_new[0][t])
    assert np.array_equal(kc, exp_k) and np.array_equal(vc, exp_v)


def test_reshape_fp8_quantises_with_separate_scales():
    w = _case(17, [5, 16, 33], 4, cache="fp8", write_new=True)
    kc0, vc0 = raw(w.k_cache[0]), raw(w.v_cache[0])
    ks, vs = float(w.k_scale[0]), float(w.v_scale[0])
    assert ks != vs
    slots = w.slot_mapping.numpy()
    kc, vc = oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), oracle.BF16, kc0, vc0,
                                      oracle.FP8_E4M3, slots, ks, vs)
    changed = np.zeros(kc0.shape, bool)
    for t, sl in enumerate(slots):
        assert np.array_equal(kc[sl // 16, :, sl % 16], oracle.quantize(raw(w.k_new[0][t]), oracle.BF16, ks))
        assert np.array_equal(vc[sl // 16, :, sl % 16], oracle.quantize(raw(w.v_new[0][t]), oracle.BF16, vs))
        changed[sl // 16, :, sl % 16] = True
    assert np.array_equal(kc[~changed], kc0[~changed]) and np.array_equal(vc[~changed], vc0[~changed])


def test_reshape_skips_negative_slots_and_rejects_out_of_pool():
    w = _case(18, [8, 9], 4, write_new=True)
    kc0, vc0 = raw(w.k_cache[0]), raw(w.v_cache[0])
    slots = w.slot_mapping.numpy().copy()
    slots[0] = -1
    kc, vc = oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), oracle.BF16, kc0, vc0, oracle.BF16, slots)
    s1 = slots[1]
    mask = np.zeros(kc0.shape, bool)
    mask[s1 // 16, :, s1 % 16] = True
    assert np.array_equal(kc[~mask], kc0[~mask])
    slots[1] = w.num_blocks * 16
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), oracle.BF16, kc0, vc0, oracle.BF16, slots)


def test_write_then_decode_poisoned_pool_is_finite_and_dense():
    # every never-read slot holds NaN; the write fills the new tokens' slots
    w = _case(19, [1, 16, 17, 31, 150], 6, write_new=True)
    kc, vc = oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), oracle.BF16, raw(w.k_cache[0]),
                                      raw(w.v_cache[0]), oracle.BF16, w.slot_mapping.numpy())
    got = oracle_decode(w, k_cache=kc, v_cache=vc)
    assert np.all(np.isfinite(got))
    before = oracle_decode(w)
    assert np.all(np.isnan(before))   # without the write, the poisoned new slot is read


# -- other block sizes ("Basics of LLM Inference and vLLM Internals", s.11 question 3) ----

def _case_bs(seed, lens, G, bs, cache="bf16", q_lens=None, write_new=False):
    return W.build_workload(name="t", seed=seed, device="cpu", num_layers=1, seq_lens=lens,
                            q_lens=q_lens or [1] * len(lens), num_q_heads=G * 2, num_kv_heads=2,
                            cache_dtype=cache, extra_blocks=8, write_new=write_new, block_size=bs)


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("cache", ["bf16", "fp8"])
def test_decode_other_block_sizes_equal_dense(bs, cache):
    lens = [1, 7, 8, 9, 31, 32, 33, 150]
    w = _case_bs(40 + bs, lens, 4, bs, cache=cache)
    assert w.k_cache[0].shape[2] == bs
    got = oracle_decode(w)
    kc, vc = workload_values(w)
    q = values(w.q[0])
    tables = w.block_tables.numpy()
    for s, n in enumerate(lens):
        K, V = dense_kv(kc, vc, tables[s], n, block_size=bs)
        np.testing.assert_allclose(got[s], sdpa(q[s:s + 1], K, V, w.scale)[0], atol=1e-12, rtol=0)


@pytest.mark.parametrize("bs", [8, 32])
def test_mixed_other_block_sizes_equal_dense_causal(bs):
    lens, qls = [30, 100, 9, 77], [1, 41, 9, 3]
    w = _case_bs(50 + bs, lens, 4, bs, q_lens=qls)
    got = _oracle_mixed(w)
    kc, vc = workload_values(w)
    q = values(w.q[0])
    qsl = w.query_start_loc.tolist()
    for s, (n, ql) in enumerate(zip(lens, qls)):
        K, V = dense_kv(kc, vc, w.block_tables[s].numpy(), n, block_size=bs)
        pos = n - ql + np.arange(ql)
        mask = np.arange(n)[None, :] <= pos[:, None]
        ref = sdpa(q[qsl[s]:qsl[s + 1]], K, V, w.scale, mask=mask)
        np.testing.assert_allclose(got[qsl[s]:qsl[s + 1]], ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("bs", [8, 32])
def test_reshape_other_block_sizes_place_bits(bs):
    w = _case_bs(60 + bs, [5, 8, 9, 32, 33], 4, bs, write_new=True)
    kc0, vc0 = raw(w.k_cache[0]), raw(w.v_cache[0])
    slots = w.slot_mapping.numpy()
    kc, vc = oracle.reshape_and_cache(raw(w.k_new[0]), raw(w.v_new[0]), oracle.BF16, kc0, vc0, oracle.BF16, slots)
    exp_k, exp_v = kc0.copy(), vc0.copy()
    for t, sl in enumerate(slots):
        exp_k[sl // bs, :, sl % bs, :] = raw(w.k_new[0][t])
        exp_v[sl // bs, :, sl % bs, :] = raw(w.v_new[0][t])
    assert np.array_equal(kc, exp_k) and np.array_equal(vc, exp_v)


def test_block_size_does_not_change_the_result():
    # the same tokens stored in blocks of 8, 16 and 32 give the same float64 output
    lens = [5, 77, 40]
    base = _case_bs(70, lens, 4, 16)
    kb, vb = raw(base.k_cache[0]), raw(base.v_cache[0])
    bt0 = base.block_tables.numpy()
    outs = []
    for bs in (8, 16, 32):
        nb = sum(-(-n // bs) for n in lens)
        kc = np.zeros((nb, 2, bs, 128), kb.dtype)
        vc = np.zeros_like(kc)
        bt = np.full((len(lens), max(-(-n // bs) for n in lens)), -1, np.int32)
        nxt = 0
        for s, n in enumerate(lens):
            for j in range(-(-n // bs)):
                bt[s, j] = nxt
                nxt += 1
            for t in range(n):
                kc[bt[s, t // bs], :, t % bs] = kb[bt0[s, t // 16], :, t % 16]
                vc[bt[s, t // bs], :, t % bs] = vb[bt0[s, t // 16], :, t % 16]
        outs.append(oracle.decode(raw(base.q[0]), oracle.BF16, kc, vc, oracle.BF16, bt,
                                  np.array(lens, np.int32), base.scale))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[2], outs[1])
