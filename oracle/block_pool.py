"""TEST INFRASTRUCTURE ONLY -- plain model of the block pool, for the tests.

Only tests/ may import this module.  It shares nothing with the library's pool
(paged_kv_cache_99_gb300/csrc/pool.cpp) and is written straight from the pages:

* "Basics of LLM Inference and vLLM Internals", s.4 "PagedAttention and Block
  Management": a pool of fixed-size blocks whose free ones wait in a queue;
  block 0 is reserved as the null block (21,520 tokens = 1,345 blocks of 16, of
  which 1,344 are usable); a physical block shared by several tables carries a
  reference count.
* s.5 "Prefix Caching": full blocks are identified by their parent's identity
  and their own tokens (plus extra keys), so only prefixes hit, in whole blocks,
  and the block holding the last token is recomputed; finished requests return
  their blocks to the free queue keeping their content, reuse takes the front,
  returns go to the back with a request's tail blocks first.
* "The Memory Trick Behind Fast LLM Serving", "The block pool": blocks are popped
  from the free queue when a request needs room.

Readings where the pages are silent (the library takes the same ones): a freed
block holding no registered content goes to the front of the queue; a block's
identity is the exact token sequence from the start of the prompt through it
(with extra_key), which is what the hash chain stands for, so this model has no
collisions by construction.
"""
from __future__ import annotations

from collections import deque


class PoolModel:
    def __init__(self, num_blocks: int, block_size: int = 16):
        assert num_blocks >= 2 and block_size >= 1
        self.bs = block_size
        self.queue = deque(range(1, num_blocks))   # front = left; block 0 is the null block
        self.ref = [0] * num_blocks
        self.key = [None] * num_blocks              # registered content of a block
        self.where = {}                             # content -> block

    # -- plain operations ----------------------------------------------------
    @property
    def num_free(self) -> int:
        return len(self.queue)

    @property
    def num_cached(self) -> int:
        return len(self.where)

    def _take(self) -> int:
        b = self.queue.popleft()
        if self.key[b] is not None:                 # its content is evicted
            del self.where[self.key[b]]
            self.key[b] = None
        self.ref[b] = 1
        return b

    def allocate(self, n: int):
        if n > len(self.queue):
            return None
        return [self._take() for _ in range(n)]

    def share(self, blocks):
        assert all(self.ref[b] > 0 for b in blocks)
        for b in blocks:
            self.ref[b] += 1

    def free(self, blocks):
        # blocks given in table order; the last one given is returned first
        for b in reversed(list(blocks)):
            self.ref[b] -= 1
            assert self.ref[b] >= 0
            if self.ref[b] == 0:
                if self.key[b] is not None:
                    self.queue.append(b)
                else:
                    self.queue.appendleft(b)

    # -- prefix caching ------------------------------------------------------
    def allocate_prompt(self, tokens, extra_key: int = 0):
        tokens = list(tokens)
        n, bs = len(tokens), self.bs
        nfull, nb = n // bs, -(-n // bs)
        keys = [(extra_key, tuple(tokens[:(i + 1) * bs])) for i in range(nfull)]
        hit = 0
        while hit < nfull and (hit + 1) * bs <= n - 1 and keys[hit] in self.where:
            hit += 1
        hit_blocks = [self.where[keys[i]] for i in range(hit)]
        free_hits = sum(1 for b in hit_blocks if self.ref[b] == 0)
        if nb - hit > len(self.queue) - free_hits:
            return None
        for b in hit_blocks:
            if self.ref[b] == 0:
                self.queue.remove(b)
            self.ref[b] += 1
        out = list(hit_blocks)
        for i in range(hit, nb):
            b = self._take()
            if i < nfull and keys[i] not in self.where:
                self.key[b] = keys[i]
                self.where[keys[i]] = b
            out.append(b)
        return out, hit * bs

    def copy_on_write(self, blocks):
        blocks = list(blocks)
        need = sum(1 for b in blocks if self.ref[b] > 1)
        if need > len(self.queue):
            return None
        src, dst = [], []
        for k, b in enumerate(blocks):
            if self.ref[b] > 1:
                nb = self._take()
                self.ref[b] -= 1
                src.append(b)
                dst.append(nb)
                blocks[k] = nb
        return blocks, src, dst
