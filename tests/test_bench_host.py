"""Host-side pieces of the benchmark, on CPU: the algorithmic byte count, the
max-over-ranks timing reduction across two gloo ranks, the oracle arm, and the
rule that a DRAM-traffic record counts only for the kernel sources it was
taken on."""
import json
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_kv_cache_99_gb300 import workloads as W


def test_kv_bytes_tiny_and_per_token():
    w = W.tiny("cpu")
    assert bench.kv_read_bytes(w) == (8 + 17 + 31 + 46) * 2 * 2 * 128 * 2
    # Qwen2.5-1.5B shape: 28 layers x 1,024 B = 28,672 B per token, as the sizing formula gives
    w2 = W.qwen25_15b("cpu", num_layers=28, batch=2)
    assert bench.kv_read_bytes(w2) == int(w2.seq_lens.sum()) * 28672


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.reduce_max(1.5 + rank, world)
        bench.barrier(world)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_reference_arm_prints_contract_line(capsys):
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3",
                "--ref-step-seconds", "0.01"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


class _RecordingPa:
    """Stands in for the library: records which entry point each layer calls."""

    def __init__(self, log):
        self.log = log

    def __getattr__(self, name):
        def call(*args, **kwargs):
            self.log.append(name)
        return call


def test_step_hooks_wrap_each_layer_in_order():
    # the end-to-end step hangs its copies on these hooks: each layer's input wait
    # before its calls, its output copy after them
    w = W.qwen25_15b("cpu", num_layers=3, batch=2)
    log = []
    caches = [(w.k_cache[l], w.v_cache[l]) for l in range(w.num_layers)]
    outs = [torch.empty_like(w.q[l]) for l in range(w.num_layers)]
    bench.build_step(w, _RecordingPa(log), None, outs, caches,
                     before_layer=lambda l: log.append(f"before {l}"), after_layer=lambda l: log.append(f"after {l}"))
    want = []
    for l in range(3):
        want += [f"before {l}", "pa_decode_append", f"after {l}"]
    assert log == want
    # a mixed batch: slot write, then the mixed call, per layer
    wm = W.build_workload(name="m", seed=1, device="cpu", num_layers=2, seq_lens=[40, 90], q_lens=[1, 30],
                          num_q_heads=16, num_kv_heads=2)
    log.clear()
    bench.build_step(wm, _RecordingPa(log), None, [torch.empty_like(wm.q[l]) for l in range(2)],
                     [(wm.k_cache[l], wm.v_cache[l]) for l in range(2)])
    assert log == ["pa_reshape_and_cache", "pa_mixed"] * 2


def test_traffic_record_only_for_the_kernel_source_it_was_taken_on(tmp_path, monkeypatch):
    # a record counts only while the kernel's sources hash to the value it was taken on
    (tmp_path / "profiles").mkdir()
    rec = {"wl-a": {"kernel_hash": "1" * 16, "dram_bytes_per_launch": 123},
           "wl-b": {"kernel_hash": "0" * 16, "dram_bytes_per_launch": 456}}
    (tmp_path / "profiles" / "chunk_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel="decode": "1" * 16)
    assert bench.recorded_traffic("wl-a", "chunk") == 123
    assert bench.recorded_traffic("wl-b", "chunk") is None      # stale: taken on other sources
    assert bench.recorded_traffic("wl-c", "chunk") is None      # never recorded
    assert bench.recorded_traffic("wl-a", "decode") is None     # no decode record file here


def test_committed_traffic_records_name_their_sources():
    # every committed record carries the hash it was taken on and a positive byte count
    for kernel in ("decode", "chunk"):
        with open(os.path.join(bench.ROOT, "profiles", f"{kernel}_traffic.json")) as f:
            rec = json.load(f)
        for name, ent in rec.items():
            if name == "note":
                continue
            assert len(ent["kernel_hash"]) == 16 and ent["dram_bytes_per_launch"] > 0, (kernel, name)
