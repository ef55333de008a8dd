"""The decode step is capturable in a CUDA graph: no host synchronisation and no
allocation inside the calls.  A graph captured once for a batch-size bucket
replays correctly after the batch's q, new K/V, lengths and block tables are
replaced in place (qwen-engine README: decode batches captured per padded size
and replayed with fresh inputs)."""
import pytest
import torch

import oracle
import synth
from gpu_harness import GpuCase, as_f64
from paged_kv_gqa_08_gb300.step import run_step, write_rows

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]

BUCKET_MAX_CTX = 2048


def _load_into(run, wl):
    """Copy a workload's step inputs and cached rows into run's static buffers."""
    t = synth.to_torch(wl, "cuda")
    for k in ("q", "k_new", "v_new", "context_lens", "cu_seqlens_q", "block_tables", "q_norm_w", "k_norm_w"):
        if t.get(k) is not None:
            run.t[k].copy_(t[k])
    run.k_cache.fill_(float("nan"))
    run.v_cache.fill_(float("nan"))
    nh = max(int(wl.cu_hist[-1]), 1)
    write_rows(run.desc, t["hist_k"], t["hist_v"], t["cu_hist"], t["hist_lens"], t["block_tables"],
               wl.max_pages_per_seq, torch.empty(nh, dtype=torch.int32, device="cuda"),
               torch.empty(nh, dtype=torch.int64, device="cuda"), run.k_cache, run.v_cache)


def test_decode_step_replays_from_a_cuda_graph_with_new_inputs():
    spec = dict(synth.CONFIGS["qwen3_0p6b_decode"], B=16, num_pages=2200, max_pages_per_seq=BUCKET_MAX_CTX // 16)
    wl1 = synth.make_workload(spec, seed=101)
    wl2 = synth.make_workload(spec, seed=202)
    run = GpuCase(wl1)

    def step():
        t = run.t
        run_step(run.desc, "decode", run.bufs, t["q"], t["k_new"], t["v_new"], t["cu_seqlens_q"], t["context_lens"],
                 t["block_tables"], run.k_cache, run.v_cache, wl1.scale, wl1.max_pages_per_seq, BUCKET_MAX_CTX, 1)

    step()                                   # first call outside capture (plans, attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        # undo the eager step's cache write so the replay starts from wl1's state
        _load_into(run, wl1)
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for wl in (wl1, wl2, wl1):
        _load_into(run, wl)
        g.replay()
        torch.cuda.synchronize()
        ok, err, bound = oracle.within_tolerance(as_f64(run.bufs.out[: wl.batch]), oracle.reference_step(wl)["o"],
                                                 wl.dtype)
        assert ok, (wl.seed, err, bound)


def test_planned_prefill_step_replays_from_a_cuda_graph_with_new_lengths():
    # Same bucket (batch, tokens, cache), different prefix lengths: the device
    # planner re-plans on every replay, so the split pattern follows the data.
    base = dict(kind="prefill", dtype="bf16", B=3, Hq=16, Hkv=8, hd=128, P=16, chunks=[150, 1, 40], norm=True,
                num_pages=1200, max_pages_per_seq=6000 // 16)
    wl1 = synth.make_workload(dict(base, prefixes=[5000, 20, 300]), seed=11)
    wl2 = synth.make_workload(dict(base, prefixes=[64, 5900, 4000]), seed=12)
    max_ctx = 6000
    run = GpuCase(wl1)
    assert run.bufs.workspace is not None

    def step():
        t = run.t
        run_step(run.desc, "prefill", run.bufs, t["q"], t["k_new"], t["v_new"], t["cu_seqlens_q"],
                 t["context_lens"], t["block_tables"], run.k_cache, run.v_cache, wl1.scale, wl1.max_pages_per_seq,
                 max_ctx, 150, t["q_norm_w"], t["k_norm_w"], wl1.eps, wl1.rope_theta)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _load_into(run, wl1)
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    plans = []
    for wl in (wl1, wl2, wl1):
        _load_into(run, wl)
        g.replay()
        torch.cuda.synchronize()
        plans.append(run.bufs.workspace[:16].view(torch.int32).tolist())
        ok, err, bound = oracle.within_tolerance(as_f64(run.bufs.out[: wl.num_new_tokens]),
                                                 oracle.reference_step(wl)["o"], wl.dtype)
        assert ok, (wl.seed, err, bound)
    assert plans[0] == plans[2]
