"""Block copies (pa_copy_blocks) bit for bit, and copy-on-write end to end: a
forked sequence shares a partly filled block, gets a private copy from the pool,
writes its new token there, and both sequences decode to the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_99_gb300 as pa
from tests._dense import CODE, raw

pytestmark = pytest.mark.gpu
DEV = "cuda"
TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp8": torch.uint8}


def _caches(g, nb, hkv, cache):
    if cache == "fp8":
        # any e4m3 code but the two NaNs (S.1111.111)
        k = torch.randint(0, 256, (nb, hkv, 16, 128), generator=g, dtype=torch.uint8)
        v = torch.randint(0, 256, (nb, hkv, 16, 128), generator=g, dtype=torch.uint8)
        k[(k & 0x7F) == 0x7F] -= 1
        v[(v & 0x7F) == 0x7F] -= 1
    else:
        k = torch.randn(nb, hkv, 16, 128, generator=g).to(TORCH[cache])
        v = torch.randn(nb, hkv, 16, 128, generator=g).to(TORCH[cache])
    return k.to(DEV), v.to(DEV)


@pytest.mark.parametrize("cache,hkv", [("bf16", 2), ("fp16", 8), ("fp8", 8), ("fp8", 1)])
def test_copy_blocks_bit_exact(cache, hkv):
    g = torch.Generator().manual_seed(hkv)
    nb = 300
    k, v = _caches(g, nb, hkv, cache)
    perm = torch.randperm(nb, generator=g)
    src, dst = perm[:100].int(), perm[100:200].int()        # distinct, disjoint
    want_k, want_v = raw(k).copy(), raw(v).copy()
    want_k[dst.numpy()] = want_k[src.numpy()]
    want_v[dst.numpy()] = want_v[src.numpy()]
    pa.pa_copy_blocks(k, v, src.to(DEV), dst.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(raw(k), want_k) and np.array_equal(raw(v), want_v)


def test_copy_blocks_out_of_range_is_recorded():
    g = torch.Generator().manual_seed(9)
    k, v = _caches(g, 20, 2, "bf16")
    before_k = raw(k).copy()
    ws = pa.new_workspace(1, 8, 2)
    src = torch.tensor([3, 20, 5], dtype=torch.int32, device=DEV)
    dst = torch.tensor([7, 8, -1], dtype=torch.int32, device=DEV)
    pa.pa_copy_blocks(k, v, src, dst, workspace=ws)
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(ws) == pa.PA_ERR_OUT_OF_RANGE
    want = before_k.copy()
    want[7] = before_k[3]                  # only the valid pair was copied
    assert np.array_equal(raw(k), want)


@pytest.mark.parametrize("cache,qd", [("bf16", "bf16"), ("fp8", "bf16")])
def test_copy_on_write_fork_then_decode(cache, qd):
    g = torch.Generator().manual_seed(21)
    hkv, G, n = 2, 4, 40                   # 40 tokens: blocks 0, 1 full, block 2 holds 8
    pool = pa.BlockPool(64, 16)
    k, v = _caches(g, 64, hkv, "bf16" if cache != "fp8" else "fp8")
    ks = vs = None
    if cache == "fp8":
        ks = torch.tensor([0.02], device=DEV)
        vs = torch.tensor([0.03], device=DEV)
    a = pool.allocate(3)                   # sequence A
    pool.share(a)                          # B forks A: the same three blocks
    # B writes into its last block only: that one gets a private copy
    last, src, dst = pool.copy_on_write([a[2]])
    b = a[:2] + last
    assert src == [a[2]] and dst == last and last[0] not in a
    assert [pool.ref_count(x) for x in a] == [2, 2, 1] and pool.ref_count(last[0]) == 1
    pa.pa_copy_blocks(k, v, torch.tensor(src, dtype=torch.int32, device=DEV),
                      torch.tensor(dst, dtype=torch.int32, device=DEV))
    # B's new token (position 40) goes into its private block
    knew = torch.randn(1, hkv, 128, generator=g).to(TORCH[qd]).to(DEV)
    vnew = torch.randn(1, hkv, 128, generator=g).to(TORCH[qd]).to(DEV)
    slot = torch.tensor([b[2] * 16 + 8], dtype=torch.int64, device=DEV)
    pre_k, pre_v = raw(k).copy(), raw(v).copy()
    pa.pa_reshape_and_cache(knew, vnew, k, v, slot, ks, vs)
    tables = torch.tensor([a + [0], b + [0]], dtype=torch.int32, device=DEV)
    lens = torch.tensor([n, n + 1], dtype=torch.int32, device=DEV)
    q = torch.randn(2, hkv * G, 128, generator=g).to(TORCH[qd]).to(DEV)
    out = torch.empty_like(q)
    ws = pa.new_workspace(2, hkv * G, hkv)
    scale = 128 ** -0.5
    pa.pa_decode(out, q, k, v, tables, lens, scale, ws, ks, vs)
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(ws) == pa.PA_OK
    # A's blocks are untouched by B's write
    assert np.array_equal(raw(k)[a[2]], pre_k[a[2]]) and np.array_equal(raw(v)[a[2]], pre_v[a[2]])
    ek, ev = oracle.reshape_and_cache(raw(knew), raw(vnew), CODE[qd], pre_k, pre_v, CODE[cache],
                                      slot.cpu().numpy(), float(ks) if ks is not None else 1.0,
                                      float(vs) if vs is not None else 1.0)
    ref = oracle.decode(raw(q), CODE[qd], ek, ev, CODE[cache], tables.cpu().numpy(), lens.cpu().numpy(), scale,
                        float(ks) if ks is not None else 1.0, float(vs) if vs is not None else 1.0)
    got = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert np.all(err <= 1e-2 + 1e-2 * np.abs(ref)), err.max()
