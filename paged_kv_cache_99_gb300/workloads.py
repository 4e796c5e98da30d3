"""Seeded synthetic inputs for the paged attention path.

This module only draws inputs: sequence lengths, physical block placement,
block tables, slot mappings, K/V/q values and FP8 scales, and poisons every
cache slot the path must never read.  It holds none of the attention
arithmetic; the library, the tests and the benchmark all take their inputs
from here.

Structure (lengths, block permutation) is always drawn from a CPU generator, so
a given seed yields the same tables on every machine; values are drawn on the
device the workload is built for.

Named workloads (sizes as the pages' examples and the benchmark suite use them):

``tiny``            1 layer, 4 decode sequences of 7/16/30/45 cached tokens plus one
                    new token each (written by the slot write), H_q=8, H_kv=2,
                    pool of 64 blocks, bf16.
``qwen2.5-1.5b``    28 layers, H_q=12, H_kv=2 (28,672 B/token in bf16), batch 64,
                    seq_lens uniform in [512, 4096], one decode step.
``gqa40-8k``        40 layers, H_q=32, H_kv=8, fp16 KV (160 KiB/token), batch 40 at
                    exactly 8192 tokens.
``shared-prefix``   1 layer, H_q=32, H_kv=8, bf16, batch 128; every table starts with
                    the same 128 physical blocks (2048 tokens), then a private suffix
                    of uniform [0, 1000] tokens.  Nothing is written (a shared block
                    is read-only).
``mixed-fp8``       1 layer, H_q=64, H_kv=8, FP8-e4m3 KV with per-tensor scales
                    amax/448 of the bf16 source; 16 decode rows with log-normal
                    lengths (median 8192, sigma 1, capped at 32768) plus 2 prefill
                    chunks of 512 queries on 4096-token contexts; the slot write
                    stores all 1040 new tokens.
``mixed-bf16``      the same batch with a bf16 cache.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BLOCK_SIZE = 16
HEAD_DIM = 128

# NaN bit patterns written into every slot the path must never read.
POISON_BITS = {"bf16": 0x7FC0, "fp16": 0x7E00, "fp8": 0x7F}
TORCH_DTYPE = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp8": torch.uint8}
ELEM_BYTES = {"bf16": 2, "fp16": 2, "fp8": 1}


@dataclass
class Workload:
    name: str
    num_layers: int
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    q_dtype: str                      # "bf16" | "fp16"  (also the new K/V source type)
    cache_dtype: str                  # "bf16" | "fp16" | "fp8"
    seq_lens: torch.Tensor            # int32 [B]: cached tokens after this step's write
    query_start_loc: torch.Tensor     # int32 [B+1]: cumulative query rows
    block_tables: torch.Tensor        # int32 [B, max_blocks]; entries past a sequence's blocks = -1
    slot_mapping: torch.Tensor        # int64 [T]: slot of every new token (empty if nothing is written)
    q: torch.Tensor                   # [L, total_q, H_q, d]
    k_new: torch.Tensor               # [L, T, H_kv, d]
    v_new: torch.Tensor               # [L, T, H_kv, d]
    k_cache: list = field(default_factory=list)   # L x [num_blocks, H_kv, block_size, d]
    v_cache: list = field(default_factory=list)
    k_scale: torch.Tensor | None = None          # float32 [L] (FP8 only)
    v_scale: torch.Tensor | None = None
    scale: float = 1.0 / math.sqrt(HEAD_DIM)
    seed: int = 0
    shared_prefix_blocks: int = 0
    q_lens_host: list = field(default_factory=list)   # host copy: no device sync when read

    @property
    def total_q(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_new_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    @property
    def q_lens(self) -> list:
        return list(self.q_lens_host)

    @property
    def max_q_len(self) -> int:
        return max(self.q_lens) if self.num_seqs else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.num_seqs else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def is_decode_only(self) -> bool:
        return all(x == 1 for x in self.q_lens)


def _draw(shape, dtype: str, gen: torch.Generator, device) -> torch.Tensor:
    """N(0, 1) drawn in float32 and rounded to the storage type."""
    out = torch.empty(shape, dtype=torch.bfloat16 if dtype == "fp8" else TORCH_DTYPE[dtype], device=device)
    flat = out.view(-1)
    chunk = 1 << 26
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=gen, device=device, dtype=torch.float32).to(flat.dtype)
    return out


def _as_int16(bits: int) -> int:
    return bits - 0x10000 if bits >= 0x8000 else bits


def build_workload(*, name: str, seed: int, device, num_layers: int, seq_lens, q_lens,
                   num_q_heads: int, num_kv_heads: int, q_dtype: str = "bf16",
                   cache_dtype: str = "bf16", extra_blocks: int = 64,
                   shared_prefix_blocks: int = 0, pool_blocks: int | None = None,
                   write_new: bool = True, head_dim: int = HEAD_DIM,
                   block_size: int = BLOCK_SIZE, fp8_scale: str = "tensor") -> Workload:
    """Build a paged batch.

    seq_lens[s] counts the tokens in the cache after this step (context plus the
    q_lens[s] new tokens).  With ``write_new`` the new tokens' slots are left
    poisoned in the cache and must be filled by the slot write; otherwise the
    cache already holds them and nothing is written.
    """
    device = torch.device(device)
    seq_lens = [int(x) for x in seq_lens]
    q_lens = [int(x) for x in q_lens]
    B = len(seq_lens)
    assert len(q_lens) == B and all(q >= 0 for q in q_lens)
    assert not write_new or all(q <= n for q, n in zip(q_lens, seq_lens))
    assert num_q_heads % num_kv_heads == 0
    sgen = torch.Generator(device="cpu").manual_seed(seed)
    vgen = torch.Generator(device=device).manual_seed(seed + 7919)

    nblk = [-(-n // block_size) for n in seq_lens]
    P = shared_prefix_blocks
    assert all(nb >= P for nb in nblk), "every sequence must cover the shared prefix"
    needed = P + sum(nb - P for nb in nblk)
    num_blocks = pool_blocks if pool_blocks is not None else needed + extra_blocks
    assert num_blocks >= needed
    perm = torch.randperm(num_blocks, generator=sgen).tolist()
    max_blocks = max(1, max(nblk) if nblk else 1)
    tables = torch.full((B, max_blocks), -1, dtype=torch.int32)
    cursor = P
    for s in range(B):
        row = perm[:P] + perm[cursor:cursor + nblk[s] - P]
        cursor += nblk[s] - P
        if row:
            tables[s, :len(row)] = torch.tensor(row, dtype=torch.int32)
    assigned = set(perm[:cursor])

    # slots of the new tokens: position pos lives in block pos // bs at offset pos % bs
    slots = []
    for s in range(B):
        for j in range(q_lens[s] if write_new else 0):
            pos = seq_lens[s] - q_lens[s] + j
            slots.append(int(tables[s, pos // block_size]) * block_size + pos % block_size)
    slot_mapping = torch.tensor(slots if write_new else [], dtype=torch.int64)
    total_q = sum(q_lens)
    qsl = torch.zeros(B + 1, dtype=torch.int32)
    if B:
        qsl[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int32), 0)

    # never-read slots: tails of last blocks, unassigned blocks, and (before the
    # slot write) the new tokens' own slots
    tail_slots = []
    for s in range(B):
        n = seq_lens[s]
        if nblk[s] and n % block_size:
            base = int(tables[s, nblk[s] - 1]) * block_size
            tail_slots.extend(range(base + n % block_size, base + block_size))
    free_blocks = sorted(set(range(num_blocks)) - assigned)
    poison_slot_list = tail_slots + (slots if write_new else [])

    T = len(slot_mapping)
    src_dtype = q_dtype
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    k_cache, v_cache, k_scales, v_scales = [], [], [], []
    q = torch.empty((num_layers, total_q, num_q_heads, head_dim), dtype=TORCH_DTYPE[q_dtype], device=device)
    k_new = torch.empty((num_layers, T, num_kv_heads, head_dim), dtype=TORCH_DTYPE[src_dtype], device=device)
    v_new = torch.empty_like(k_new)
    ps = torch.tensor(poison_slot_list, dtype=torch.int64, device=device)
    fb = torch.tensor(free_blocks, dtype=torch.int64, device=device)
    for layer in range(num_layers):
        q[layer] = _draw(q.shape[1:], q_dtype, vgen, device)
        k_new[layer] = _draw(k_new.shape[1:], src_dtype, vgen, device)
        v_new[layer] = _draw(v_new.shape[1:], src_dtype, vgen, device)
        kc = _draw(shape, cache_dtype if cache_dtype != "fp8" else "bf16", vgen, device)
        vc = _draw(shape, cache_dtype if cache_dtype != "fp8" else "bf16", vgen, device)
        if cache_dtype == "fp8" and fp8_scale == "head":
            # heads of different magnitude (K of head h x 2^(h mod 4), V x 2^((h+1) mod 4)),
            # so that each head needs its own scale
            hk = 2.0 ** (torch.arange(num_kv_heads, device=device) % 4).float()
            hv = 2.0 ** ((torch.arange(num_kv_heads, device=device) + 1) % 4).float()
            kc = (kc.float() * hk.view(1, -1, 1, 1)).to(kc.dtype)
            vc = (vc.float() * hv.view(1, -1, 1, 1)).to(vc.dtype)
            k_new[layer] = (k_new[layer].float() * hk.view(1, -1, 1)).to(k_new.dtype)
            v_new[layer] = (v_new[layer].float() * hv.view(1, -1, 1)).to(v_new.dtype)
            # one scale per KV head: amax over that head's bf16 values destined for the cache
            def head_amax(c, new):
                m = c.abs().float().amax(dim=(0, 2, 3))
                return torch.maximum(m, new.abs().float().amax(dim=(0, 2))) if T else m
            ks = head_amax(kc, k_new[layer]) / 448.0
            vs = head_amax(vc, v_new[layer]) / 448.0
            kc = (kc.float() / ks.view(1, -1, 1, 1)).to(torch.float8_e4m3fn).view(torch.uint8)
            vc = (vc.float() / vs.view(1, -1, 1, 1)).to(torch.float8_e4m3fn).view(torch.uint8)
            k_scales.append(ks)
            v_scales.append(vs)
        elif cache_dtype == "fp8":
            # per-tensor scale: amax over every bf16 value destined for this cache
            ks = torch.maximum(kc.abs().max().float(), k_new[layer].abs().max().float() if T else
                               torch.zeros((), device=device)) / 448.0
            vs = torch.maximum(vc.abs().max().float(), v_new[layer].abs().max().float() if T else
                               torch.zeros((), device=device)) / 448.0
            kc = (kc.float() / ks).to(torch.float8_e4m3fn).view(torch.uint8)
            vc = (vc.float() / vs).to(torch.float8_e4m3fn).view(torch.uint8)
            k_scales.append(ks)
            v_scales.append(vs)
        for c in (kc, vc):
            _poison(c, cache_dtype, ps, fb, block_size)
        k_cache.append(kc)
        v_cache.append(vc)

    return Workload(
        name=name, num_layers=num_layers, num_seqs=B, num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
        num_blocks=num_blocks, q_dtype=q_dtype, cache_dtype=cache_dtype,
        seq_lens=torch.tensor(seq_lens, dtype=torch.int32).to(device),
        query_start_loc=qsl.to(device), block_tables=tables.to(device),
        slot_mapping=slot_mapping.to(device), q=q, k_new=k_new, v_new=v_new,
        k_cache=k_cache, v_cache=v_cache,
        k_scale=torch.stack(k_scales).float() if k_scales else None,
        v_scale=torch.stack(v_scales).float() if v_scales else None,
        seed=seed, shared_prefix_blocks=P, q_lens_host=list(q_lens))


def _poison(cache: torch.Tensor, dtype: str, slots: torch.Tensor, free_blocks: torch.Tensor,
            block_size: int) -> None:
    """Write NaN bits into the given slots (all heads) and into whole free blocks."""
    raw = cache if dtype == "fp8" else cache.view(torch.int16)
    val = POISON_BITS["fp8"] if dtype == "fp8" else _as_int16(POISON_BITS[dtype])
    if free_blocks.numel():
        raw[free_blocks] = val
    if slots.numel():
        raw[slots // block_size, :, slots % block_size, :] = val


def poison_value(dtype: str) -> int:
    return POISON_BITS[dtype]


# -- the named workloads ---------------------------------------------------------

def tiny(device, seed: int = 1001, block_size: int = BLOCK_SIZE) -> Workload:
    ctx = [7, 16, 30, 45]
    return build_workload(name="tiny", seed=seed, device=device, num_layers=1,
                          seq_lens=[c + 1 for c in ctx], q_lens=[1] * 4, num_q_heads=8,
                          num_kv_heads=2, pool_blocks=64 * BLOCK_SIZE // block_size, block_size=block_size)


def qwen25_15b(device, seed: int = 1002, num_layers: int = 28, batch: int = 64,
               block_size: int = BLOCK_SIZE) -> Workload:
    g = torch.Generator(device="cpu").manual_seed(seed)
    lens = torch.randint(512, 4097, (batch,), generator=g).tolist()
    return build_workload(name="qwen2.5-1.5b", seed=seed, device=device, num_layers=num_layers,
                          seq_lens=lens, q_lens=[1] * batch, num_q_heads=12, num_kv_heads=2,
                          block_size=block_size)


def gqa40_8k(device, seed: int = 1003, num_layers: int = 40, batch: int = 40,
             seq_len: int = 8192, block_size: int = BLOCK_SIZE) -> Workload:
    return build_workload(name="gqa40-8k", seed=seed, device=device, num_layers=num_layers,
                          seq_lens=[seq_len] * batch, q_lens=[1] * batch, num_q_heads=32,
                          num_kv_heads=8, q_dtype="fp16", cache_dtype="fp16", extra_blocks=64,
                          block_size=block_size)


def shared_prefix(device, seed: int = 1004, batch: int = 128, prefix_tokens: int = 2048,
                  max_suffix: int = 1000, block_size: int = BLOCK_SIZE) -> Workload:
    # the prefix is prefix_tokens / block_size aliased blocks (128 of 16 tokens by default)
    assert prefix_tokens % block_size == 0
    g = torch.Generator(device="cpu").manual_seed(seed)
    suffix = torch.randint(0, max_suffix + 1, (batch,), generator=g).tolist()
    lens = [prefix_tokens + x for x in suffix]
    return build_workload(name="shared-prefix", seed=seed, device=device, num_layers=1,
                          seq_lens=lens, q_lens=[1] * batch, num_q_heads=32, num_kv_heads=8,
                          shared_prefix_blocks=prefix_tokens // block_size, write_new=False,
                          block_size=block_size)


def shared_prefix_long(device, seed: int = 1006, batch: int = 32, prefix_tokens: int = 8192,
                       max_suffix: int = 512, block_size: int = BLOCK_SIZE) -> Workload:
    # the other regime of a shared prefix: few sequences behind a long common prompt
    return shared_prefix(device, seed=seed, batch=batch, prefix_tokens=prefix_tokens, max_suffix=max_suffix,
                         block_size=block_size)


def shared_prefix_l2(device, seed: int = 1007, batch: int = 128, block_size: int = BLOCK_SIZE) -> Workload:
    # every sequence is the shared 2048-token prefix and nothing else: after its first
    # read the prefix is served from L2, so the decode's rate here is its L2 ceiling
    # for the shared-prefix batch's logical bytes
    return shared_prefix(device, seed=seed, batch=batch, prefix_tokens=2048, max_suffix=0, block_size=block_size)


def mixed_fp8(device, seed: int = 1005, num_decode: int = 16, num_chunks: int = 2,
              chunk_len: int = 512, chunk_ctx: int = 4096, median: int = 8192,
              sigma: float = 1.0, cap: int = 32768, block_size: int = BLOCK_SIZE,
              cache_dtype: str = "fp8", name: str = "mixed-fp8") -> Workload:
    g = torch.Generator(device="cpu").manual_seed(seed)
    z = torch.randn(num_decode, generator=g, dtype=torch.float64)
    dec = [int(min(cap, max(1, round(math.exp(math.log(median) + sigma * float(x)))))) for x in z]
    lens = dec + [chunk_ctx + chunk_len] * num_chunks
    qls = [1] * num_decode + [chunk_len] * num_chunks
    return build_workload(name=name, seed=seed, device=device, num_layers=1, seq_lens=lens,
                          q_lens=qls, num_q_heads=64, num_kv_heads=8, q_dtype="bf16",
                          cache_dtype=cache_dtype, block_size=block_size)


def mixed_bf16(device, seed: int = 1005, block_size: int = BLOCK_SIZE) -> Workload:
    # the mixed batch with a bf16 cache: the chunk kernel on 16-bit keys and values
    return mixed_fp8(device, seed=seed, block_size=block_size, cache_dtype="bf16", name="mixed-bf16")


NAMED = {
    "tiny": tiny,
    "qwen2.5-1.5b": qwen25_15b,
    "gqa40-8k": gqa40_8k,
    "shared-prefix": shared_prefix,
    "shared-prefix-long": shared_prefix_long,
    "shared-prefix-l2": shared_prefix_l2,
    "mixed-fp8": mixed_fp8,
    "mixed-bf16": mixed_bf16,
}


def make(name: str, device, **kw) -> Workload:
    return NAMED[name](device, **kw)
