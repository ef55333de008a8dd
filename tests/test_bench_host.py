"""Host-side logic of bench.py without a GPU: algorithmic work counts and the
multi-rank aggregation (world size 2 over gloo on the CPU)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth


def test_decode_bytes_tiny_config_by_hand():
    wl = synth.make_workload("tiny_fp32_decode")
    # contexts 5+17+33+64 = 119 tokens; K and V rows of 2 heads x 64 fp32 = 512 B each
    kv = 119 * 2 * 512
    qo = 2 * 4 * 4 * 64 * 4
    pages = 1 + 2 + 3 + 4
    assert bench.decode_call_bytes(wl) == kv + qo + 4 * pages + 4 * 4
    assert bench.kv_bytes(wl) == kv


def test_prefill_flops_by_hand():
    spec = dict(kind="prefill", dtype="bf16", B=2, Hq=4, Hkv=2, hd=8, P=16, chunks=[3, 1], prefixes=[2, 0], seed=1)
    wl = synth.make_workload(spec)
    # request 0: rows see 3, 4, 5 keys; request 1: 1 key -> 13 pairs
    assert bench.prefill_flops(wl) == 4 * 8 * 4 * 13


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [10.0, 12.5][rank]
    m = bench.max_over_ranks(elapsed, world)
    rate = bench.whole_job_rate(256, m, world)
    q.put((rank, m, rate))
    dist.destroy_process_group()


def test_multi_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, m, rate in res:
        assert m == 12.5                          # the slowest rank's time
        assert rate == pytest.approx(2 * 256 / 12.5e-3)
