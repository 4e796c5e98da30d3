"""Helpers for the GPU parity tests: run the library on a workload, run the
oracle on the same stored bits (optionally on a sample of sequences), compare."""
import numpy as np
import torch

import oracle
import paged_kv_cache_99_gb300 as pa
from paged_kv_cache_99_gb300 import workloads as W
from tests._dense import CODE, raw

# the attention tolerance the parity bar states: |gpu - ref| <= 1e-2 + 1e-2 |ref|
ATOL = 1e-2
RTOL = 1e-2


def gpu_step(w: W.Workload, layer: int = 0, num_workers: int = 0, k_cache=None, v_cache=None, tables=None,
             workspace=None):
    """Slot write (if the workload writes) then attention, on the GPU; returns (out, k_cache, v_cache)."""
    kc = (w.k_cache[layer] if k_cache is None else k_cache).clone()
    vc = (w.v_cache[layer] if v_cache is None else v_cache).clone()
    ks = w.k_scale[layer:layer + 1] if w.k_scale is not None else None
    vs = w.v_scale[layer:layer + 1] if w.v_scale is not None else None
    bt = w.block_tables if tables is None else tables
    if w.num_new_tokens:
        pa.pa_reshape_and_cache(w.k_new[layer], w.v_new[layer], kc, vc, w.slot_mapping, ks, vs)
    ws = pa.new_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads) if workspace is None else workspace
    out = torch.empty_like(w.q[layer])
    if w.is_decode_only:
        pa.pa_decode(out, w.q[layer], kc, vc, bt, w.seq_lens, w.scale, ws, ks, vs, num_workers=num_workers)
    else:
        pa.pa_mixed(out, w.q[layer], w.query_start_loc, kc, vc, bt, w.seq_lens, w.max_q_len, w.scale, ws, ks, vs)
    torch.cuda.synchronize()
    status = pa.pa_read_device_status(ws)
    assert status == pa.PA_OK, pa.pa_status_string(status)
    return out, kc, vc


def oracle_step(w: W.Workload, layer: int = 0, seqs=None):
    """Oracle slot write + attention for the given sequences (default: all).

    Only the blocks the chosen sequences reference are copied to the host; they
    are renumbered densely (placement does not change the result).  Returns
    (rows, out): the flattened query rows of those sequences and float64 outputs.
    """
    B = w.num_seqs
    seqs = list(range(B)) if seqs is None else list(seqs)
    qsl = w.query_start_loc.cpu().numpy()
    lens = w.seq_lens.cpu().numpy()
    tables = w.block_tables.cpu().numpy()
    need = []
    for s in seqs:
        nb = -(-int(lens[s]) // w.block_size)
        need.extend(int(x) for x in tables[s, :nb])
    uniq = sorted(set(need))
    remap = {b: i for i, b in enumerate(uniq)}
    idx = torch.tensor(uniq if uniq else [0], dtype=torch.int64, device=w.k_cache[layer].device)
    kc = raw(w.k_cache[layer].index_select(0, idx))
    vc = raw(w.v_cache[layer].index_select(0, idx))
    sub_tables = np.full((len(seqs), tables.shape[1]), -1, np.int32)
    for i, s in enumerate(seqs):
        nb = -(-int(lens[s]) // w.block_size)
        sub_tables[i, :nb] = [remap[int(x)] for x in tables[s, :nb]]
    rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in seqs]) if seqs else np.zeros(0, np.int64)
    sub_qsl = np.zeros(len(seqs) + 1, np.int32)
    sub_qsl[1:] = np.cumsum([qsl[s + 1] - qsl[s] for s in seqs])
    qbits = raw(w.q[layer][torch.as_tensor(rows, device=w.q.device)]) if len(rows) else \
        np.zeros((0, w.num_q_heads, w.head_dim), np.uint16)
    cd = CODE[w.cache_dtype]
    sub_lens = lens[seqs].astype(np.int32)

    def run(ks, vs):
        k, v = kc, vc
        if w.num_new_tokens:
            # the new tokens of the chosen sequences, with their slots renumbered
            slots = w.slot_mapping.cpu().numpy()
            tok_rows = rows  # new tokens are aligned with query rows when the workload writes
            new_slots = np.array([remap[int(slots[r]) // w.block_size] * w.block_size + int(slots[r]) % w.block_size
                                  for r in tok_rows], np.int64)
            tsel = torch.as_tensor(tok_rows, device=w.k_new.device)
            k, v = oracle.reshape_and_cache(raw(w.k_new[layer][tsel]), raw(w.v_new[layer][tsel]), CODE[w.q_dtype],
                                            k, v, cd, new_slots, ks, vs)
        if w.is_decode_only:
            return oracle.decode(qbits, CODE[w.q_dtype], k, v, cd, sub_tables, sub_lens, w.scale, ks, vs)
        return oracle.mixed(qbits, CODE[w.q_dtype], sub_qsl, k, v, cd, sub_tables, sub_lens, w.scale, ks, vs)

    if w.k_scale is None:
        return rows, run(1.0, 1.0)
    kscales = w.k_scale[layer].reshape(-1).tolist()
    vscales = w.v_scale[layer].reshape(-1).tolist()
    if len(kscales) == 1:
        return rows, run(kscales[0], vscales[0])
    # one scale per KV head: the outputs of KV head h's query heads depend on its
    # elements only, so run the oracle once per head with that head's scales
    G = w.num_q_heads // w.num_kv_heads
    out = None
    for h, (ks, vs) in enumerate(zip(kscales, vscales)):
        o = run(ks, vs)
        out = o if out is None else out
        out[:, h * G:(h + 1) * G] = o[:, h * G:(h + 1) * G]
    return rows, out


def compare(gpu_out: torch.Tensor, rows, ref: np.ndarray, what: str = ""):
    """Element-wise parity with the stated tolerance, plus an error-to-RMS guard."""
    got = gpu_out.float().cpu().numpy()[rows].astype(np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements outside tolerance, max err {err.max():.3e}"
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    # rounding of the probabilities and of the output is ~2^-9 relative per element; the
    # absolute term 1e-2 * rms (instead of 1e-2) still catches dropped or doubled blocks
    # when outputs are small, where the stated bound alone would not.  A row over a few
    # keys is not an average: its terms p_i V_i keep the size of V, they can cancel, and
    # the 16-bit rounding of p_i then errs by ~2^-9 of the terms, so the absolute term
    # takes the larger of the batch rms and the row's own rms
    row_rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True)) if ref.size else 0.0
    guard = err <= 1e-2 * np.abs(ref) + 1e-2 * np.maximum(rms, row_rms)
    assert guard.all(), f"{what}: max err {err.max():.3e} vs rms {rms:.3e}"
    return float(err.max(initial=0.0)), rms


def oracle_rows(w: W.Workload, layer: int, seqs, rows_per_seq: int = 6, seed: int = 0):
    """Oracle outputs for a sample of query rows of the chosen sequences.

    The oracle slot write is applied to the chosen sequences' new tokens; every
    sampled row (always the first and last of its sequence) is then the oracle
    decode of that one query over its causal prefix of pos + 1 tokens, which
    the oracle tests show equals the mixed-batch row exactly.
    """
    rng = np.random.default_rng(seed)
    qsl = w.query_start_loc.cpu().numpy()
    lens = w.seq_lens.cpu().numpy()
    tables = w.block_tables.cpu().numpy()
    need = sorted({int(x) for s in seqs for x in tables[s, :-(-int(lens[s]) // w.block_size)]})
    remap = {b: i for i, b in enumerate(need)}
    idx = torch.tensor(need, dtype=torch.int64, device=w.k_cache[layer].device)
    kc = raw(w.k_cache[layer].index_select(0, idx))
    vc = raw(w.v_cache[layer].index_select(0, idx))
    ks = float(w.k_scale[layer]) if w.k_scale is not None else 1.0
    vs = float(w.v_scale[layer]) if w.v_scale is not None else 1.0
    cd = CODE[w.cache_dtype]
    if w.num_new_tokens:
        slots = w.slot_mapping.cpu().numpy()
        toks = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in seqs])
        new_slots = np.array([remap[int(slots[r]) // w.block_size] * w.block_size + int(slots[r]) % w.block_size
                              for r in toks], np.int64)
        tsel = torch.as_tensor(toks, device=w.k_new.device)
        kc, vc = oracle.reshape_and_cache(raw(w.k_new[layer][tsel]), raw(w.v_new[layer][tsel]), CODE[w.q_dtype],
                                          kc, vc, cd, new_slots, ks, vs)
    rows, outs = [], []
    for s in seqs:
        ql, n = int(qsl[s + 1] - qsl[s]), int(lens[s])
        if ql == 0:
            continue
        js = sorted({0, ql - 1} | set(rng.choice(ql, min(ql, rows_per_seq), replace=False).tolist()))
        nb = -(-n // w.block_size)
        table = np.full((1, tables.shape[1]), -1, np.int32)
        table[0, :nb] = [remap[int(x)] for x in tables[s, :nb]]
        for j in js:
            r = int(qsl[s]) + j
            qb = raw(w.q[layer][r:r + 1])
            o = oracle.decode(qb, CODE[w.q_dtype], kc, vc, cd, table, np.array([n - ql + j + 1], np.int32),
                              w.scale, ks, vs)
            rows.append(r)
            outs.append(o[0])
    return np.array(rows, np.int64), np.stack(outs)
