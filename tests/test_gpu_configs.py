"""Parity at the full sizes of the benchmark workloads, in the launch
configuration the benchmark times (default worker count), on sampled outputs
the oracle computes one by one, plus properties that hold at any size."""
import numpy as np
import pytest
import torch

from paged_kv_cache_99_gb300 import workloads as W
from tests._gpu import compare, gpu_step, oracle_rows, oracle_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["qwen2.5-1.5b", "gqa40-8k", "shared-prefix", "mixed-fp8"])
def test_full_size_workload_sampled(name):
    w = W.make(name, "cuda")
    g = np.random.default_rng(11)
    lens = w.seq_lens.cpu().numpy()
    q_lens = np.array(w.q_lens)
    try:
        for layer in sorted({0, w.num_layers - 1}):
            out, _, _ = gpu_step(w, layer)
            assert torch.isfinite(out.float()).all(), f"{name}: non-finite output"
            dec = np.nonzero(q_lens == 1)[0]
            pick = set(g.choice(dec, min(4, dec.size), replace=False).tolist())
            pick |= {int(dec[lens[dec].argmax()]), int(dec[lens[dec].argmin()])}
            if w.is_decode_only:
                rows, ref = oracle_step(w, layer, sorted(pick))
            else:
                chunks = np.nonzero(q_lens > 1)[0].tolist()
                rows, ref = oracle_rows(w, layer, sorted(pick) + chunks, rows_per_seq=6)
            err, rms = compare(out, rows, ref, f"{name} layer {layer}")
            print(f"{name} layer {layer}: max err {err:.2e}, output rms {rms:.2e}, {len(rows)} rows checked")
    finally:
        del w
        torch.cuda.empty_cache()
