"""The host block pool (pa_pool_*): pinned to the pages' numbers, then checked
against the plain model in oracle/block_pool.py on random operation sequences."""
import numpy as np
import pytest

import paged_kv_cache_99_gb300 as pa
from oracle.block_pool import PoolModel
from paged_kv_cache_99_gb300 import build_ext


@pytest.fixture(scope="module", autouse=True)
def _library_built():
    build_ext.build()        # host code: the pool needs no GPU


def _documents(seed=3, docs=10, n=5033):
    # synthetic documents of random words, no two starting alike
    g = np.random.default_rng(seed)
    out = []
    for d in range(docs):
        t = g.integers(0, 150_000, n).astype(np.int32)
        t[0] = 200_000 + d
        out.append(t)
    return out


def _three_passes(pool_alloc, pool_free, docs):
    res = []
    for order in (range(len(docs)), range(len(docs)), reversed(range(len(docs)))):
        total = 0
        for d in order:
            blocks, hit = pool_alloc(docs[d])
            total += hit
            pool_free(blocks)
        res.append(total)
    return res


def test_model_pinned_to_the_pages():
    # "Basics of LLM Inference and vLLM Internals", s.4: 21,520 tokens = 1,345 blocks, 1,344 usable
    assert -(-21_520 // 16) == 1345
    m = PoolModel(1345, 16)
    assert m.num_free == 1344
    # s.9 / s.10: ten ~5,000-token documents without shared prefixes, read forward, forward
    # again and backward: 0, 0 and 21,488 prefix-hit tokens (1,343 blocks)
    assert _three_passes(lambda t: m.allocate_prompt(t), m.free, _documents()) == [0, 0, 21_488]


def test_library_pool_pinned_to_the_pages():
    p = pa.BlockPool(1345, 16)
    assert p.num_free == 1344
    assert _three_passes(p.allocate_prompt, p.free, _documents()) == [0, 0, 21_488]
    assert p.num_free == 1344 and p.num_cached == 1343


def test_null_block_never_handed_out():
    p = pa.BlockPool(9, 16)
    got = p.allocate(8)
    assert sorted(got) == list(range(1, 9))
    with pytest.raises(RuntimeError):
        p.allocate(1)                      # the queue is empty; nothing changes
    assert p.num_free == 0
    p.free(got)
    assert p.num_free == 8


def test_bad_arguments():
    with pytest.raises(ValueError):
        pa.BlockPool(1, 16)
    p = pa.BlockPool(8, 16)
    (b,) = p.allocate(1)
    p.free([b])
    with pytest.raises(RuntimeError):
        p.free([b])                        # no longer in use
    with pytest.raises(RuntimeError):
        p.share([b])
    with pytest.raises(RuntimeError):
        p.free([0])                        # the null block
    assert p.num_free == 7


def _state(p, n):
    return [p.ref_count(i) for i in range(n)], p.num_free, p.num_cached


def _model_state(m, n):
    return list(m.ref[:n]), m.num_free, m.num_cached


@pytest.mark.parametrize("bs,seed", [(16, 1), (16, 2), (4, 3), (4, 4), (1, 5)])
def test_library_pool_matches_model(bs, seed):
    g = np.random.default_rng(seed)
    nblocks = 64
    p, m = pa.BlockPool(nblocks, bs), PoolModel(nblocks, bs)
    bases = [g.integers(0, 50, g.integers(1, 12 * bs)).astype(np.int32) for _ in range(4)]
    held = []                              # tables in use (lists of block ids, table order)
    for step in range(400):
        op = g.integers(0, 5)
        if op == 0:                        # a prompt, often sharing a base prompt's prefix
            base = bases[g.integers(0, len(bases))]
            cut = int(g.integers(0, base.size + 1))
            tail = g.integers(0, 50, g.integers(0, 3 * bs)).astype(np.int32)
            toks = np.concatenate([base[:cut], tail])
            key = int(g.integers(0, 2))
            want = m.allocate_prompt(toks.tolist(), key)
            if want is None:
                with pytest.raises(RuntimeError):
                    p.allocate_prompt(toks, key)
            else:
                got = p.allocate_prompt(toks, key)
                assert got == (want[0], want[1]), f"step {step}: prompt"
                if got[0]:
                    held.append(got[0])
        elif op == 1:                      # plain allocation
            n = int(g.integers(1, 6))
            want = m.allocate(n)
            if want is None:
                with pytest.raises(RuntimeError):
                    p.allocate(n)
            else:
                assert p.allocate(n) == want, f"step {step}: allocate"
                held.append(want)
        elif op == 2 and held:             # a table finishes
            t = held.pop(int(g.integers(0, len(held))))
            p.free(t)
            m.free(t)
        elif op == 3 and held:             # a fork aliases a table's leading blocks
            t = held[int(g.integers(0, len(held)))]
            k = int(g.integers(1, len(t) + 1))
            p.share(t[:k])
            m.share(t[:k])
            held.append(list(t[:k]))
        elif op == 4 and held:             # copy-on-write before writing a table's blocks
            i = int(g.integers(0, len(held)))
            want = m.copy_on_write(held[i])
            if want is None:
                with pytest.raises(RuntimeError):
                    p.copy_on_write(held[i])
            else:
                got = p.copy_on_write(held[i])
                assert got == (want[0], want[1], want[2]), f"step {step}: copy-on-write"
                held[i] = got[0]
        assert _state(p, nblocks) == _model_state(m, nblocks), f"step {step}: state"
    for t in held:
        p.free(t)
        m.free(t)
    assert p.num_free == m.num_free == nblocks - 1
