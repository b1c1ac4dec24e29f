"""Host-side logic of bench.py that needs no GPU: the cross-rank reduction of
the N > 1 path (two gloo ranks on CPU), the algorithmic byte / FLOP
accounting behind the reported KV-read GB/s and roofline, and the workload
config both arms print."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from gqa_mqa_mla_gb300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        worst = bench.reduce_max(ms, dist, torch.device("cpu"))
        q.put((rank, worst, bench.whole_job_gbps(1_000_000_000, worst, world)))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_reduce_max_and_whole_job_value_over_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, worst, gbps in got:
        assert worst == 15.0  # max over ranks
        assert gbps == pytest.approx(2 * 1e9 / 15e-3 / 1e9)  # both ranks' bytes / slowest time


def test_reduce_max_without_process_group_is_identity():
    assert bench.reduce_max(3.5) == 3.5


def test_gqa_algorithmic_bytes_and_intensity_follow_the_pages():
    # "MQA, GQA, and MLA", section 4: FLOPs ~ 2 h S d 2, bytes ~ 2 g S d bytes,
    # intensity ~ h / g for 2-byte elements: MHA ~1, GQA (g = h/8) ~8, MQA ~h.
    for h_kv, expect in [(64, 1.0), (8, 8.0), (1, 64.0)]:
        x = synth.gqa_inputs(batch=2, h_q=64, h_kv=h_kv, seq_lens=[300, 700], block_size=16,
                             dtype="bf16", device="cpu")
        kv_bytes = bench.gqa_bytes(x) - 2 * x.batch * x.h_q * x.d_head * 2
        assert kv_bytes == 1000 * h_kv * 128 * 2 * 2
        flops = 2 * x.h_q * 1000 * x.d_head * 2
        assert flops / kv_bytes == expect


def test_mla_algorithmic_bytes_and_flops():
    x = synth.mla_inputs(batch=2, seq_lens=[100, 28], block_size=64, device="cpu")
    assert bench.mla_bytes(x) == 2 * 128 * 576 * 2 + 128 * 576 * 2 + 2 * 128 * 512 * 2
    assert bench.mla_flops(x) == 128 * 128 * (2 * 576 + 2 * 512)


def test_workload_config_is_the_workload_only():
    """Both arms print bench.workload_config: shapes, cache layout and the L2
    note of the measured workload, and no choice of the implementation."""
    g = type("G", (), {"batch": 64, "h_q": 64, "h_kv": 8, "d_head": 128, "max_seq_len": 8192,
                       "block_size": 16})()
    cfg = bench.workload_config(["gqa", "mla"], g, type("M", (), {"batch": 32})())
    assert cfg["workload"] == f"{bench.GQA_WORKLOAD} + {bench.MLA_WORKLOAD}"
    assert cfg["gqa"] == {"h_q": 64, "h_kv": 8, "d_head": 128, "batch": 64, "seq_len": 8192,
                          "block_size": 16, "table": "permuted"}
    assert cfg["mla"] == {"heads": 128, "d_c": 512, "d_rope": 64, "batch": 32, "seq_len": 8192,
                          "block_size": 64, "table": "permuted"}
    flat = repr(cfg)
    assert "split" not in flat and "pairs" not in flat
    only_mla = bench.workload_config(["mla"], None, type("M", (), {"batch": 32})())
    assert only_mla["workload"] == bench.MLA_WORKLOAD and only_mla["gqa"] is None
