"""Decode graphs captured per padded batch size and replayed with fewer live
requests (nano-vLLM learning note, ModelRunner.capture_cudagraph listing:
one graph per batch size 1, 2, 4, 8, 16, 32, 48, 64, ...; its fixed-size
input buffers start zeroed, so the rows past the live batch have length 0;
qwen-engine README: decode replayed from CUDA graphs).

For every bucket, the step is captured once with the library's two decode
forms (slot mapping + KV write + pa_decode, and the fused pa_decode_kv_write),
then replayed with new inputs in which only the first `live` rows are
requests and the rest are padding (context length 0, block-table entries that
are not page ids, NaN queries).  The live rows must match the oracle, the
padding rows' outputs and the cache outside the live rows' new slots must be
untouched, the fused form must report slot -1 for the padding rows, and no
device flag may be raised.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_harness import GpuCase, as_f64, storage
from paged_kv_gqa_08_gb300 import pa_decode_kv_write, pa_read_device_errors
from paged_kv_gqa_08_gb300.step import alloc_step_buffers, run_step, write_rows

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]

BUCKETS = [1, 2, 4, 8, 16, 32, 48, 64]
LIVE = {1: 1, 2: 1, 4: 3, 8: 5, 16: 11, 32: 21, 48: 33, 64: 40}
MAX_CTX = 608                       # bucket bound on context lengths
PAGES_PER_SEQ = MAX_CTX // 16
SENTINEL = 3.0                      # value left in the padding rows' outputs
NOT_A_PAGE = -7                     # block-table entries of padding rows


def _spec(bucket):
    return dict(synth.CONFIGS["qwen3_0p6b_decode"], B=bucket, L_range=(16, MAX_CTX),
                num_pages=bucket * PAGES_PER_SEQ + 8, max_pages_per_seq=PAGES_PER_SEQ)


def _load(run, wl, live):
    """Put workload `wl` into the captured buffers with rows >= live as padding."""
    t = synth.to_torch(wl, "cuda")
    run.k_cache.fill_(float("nan"))
    run.v_cache.fill_(float("nan"))
    nh = max(int(wl.cu_hist[-1]), 1)
    write_rows(run.desc, t["hist_k"], t["hist_v"], t["cu_hist"], t["hist_lens"], t["block_tables"],
               wl.max_pages_per_seq, torch.empty(nh, dtype=torch.int32, device="cuda"),
               torch.empty(nh, dtype=torch.int64, device="cuda"), run.k_cache, run.v_cache)
    for k in ("q", "k_new", "v_new", "context_lens", "cu_seqlens_q", "block_tables"):
        run.t[k].copy_(t[k])
    run.t["context_lens"][live:] = 0
    run.t["block_tables"][live:] = NOT_A_PAGE
    run.t["q"][live:] = float("nan")
    run.bufs.out.fill_(SENTINEL)
    run.bufs.slots.fill_(12345)


def _expected(wl, live):
    """The oracle's cache and outputs when only the first `live` rows are requests."""
    k_cache = wl.poison_storage(wl.cache_shape())
    v_cache = wl.poison_storage(wl.cache_shape())
    _, hist_slots = oracle.slot_mapping(wl.block_tables, wl.hist_lens, wl.cu_hist, wl.page_size)
    oracle.kv_write(wl.hist_k, wl.hist_v, hist_slots, k_cache, v_cache)
    _, slots = oracle.slot_mapping(wl.block_tables[:live], wl.context_lens[:live], wl.cu_seqlens_q[:live + 1],
                                   wl.page_size)
    oracle.kv_write(wl.k_new[:live], wl.v_new[:live], slots, k_cache, v_cache)
    o, _ = oracle.decode(wl.q, k_cache, v_cache, wl.block_tables, wl.context_lens, wl.scale, wl.dtype,
                         requests=range(live))
    return k_cache, v_cache, slots, o


def _capture(step):
    step()                                  # plans and kernel attributes outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("fused", [False, True], ids=["pa_decode", "pa_decode_kv_write"])
@pytest.mark.parametrize("bucket", BUCKETS)
def test_bucket_graph_replays_a_padded_batch(bucket, fused):
    wl_a = synth.make_workload(_spec(bucket), seed=500 + bucket)
    wl_b = synth.make_workload(_spec(bucket), seed=900 + bucket)
    run = GpuCase(wl_a)
    desc, t = run.desc, run.t
    run.bufs = alloc_step_buffers(desc, "decode", bucket, bucket, MAX_CTX, "cuda")  # sized for the bucket
    row = wl_a.num_kv_heads * wl_a.head_dim

    def step():
        if fused:
            pa_decode_kv_write(desc, t["q"], t["k_new"], row, t["v_new"], row, bucket, run.k_cache, run.v_cache,
                               t["block_tables"], PAGES_PER_SEQ, t["context_lens"], MAX_CTX, wl_a.scale,
                               run.bufs.max_ctas, run.bufs.slots, run.bufs.out, run.bufs.workspace)
        else:
            run_step(desc, "decode", run.bufs, t["q"], t["k_new"], t["v_new"], t["cu_seqlens_q"],
                     t["context_lens"], t["block_tables"], run.k_cache, run.v_cache, wl_a.scale, PAGES_PER_SEQ,
                     MAX_CTX, 1)

    _load(run, wl_a, bucket)
    g = _capture(step)
    pa_read_device_errors(reset=True)
    # a padded batch with new inputs, then the full bucket again
    for wl, live in ((wl_b, LIVE[bucket]), (wl_a, bucket)):
        _load(run, wl, live)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        k_exp, v_exp, slots, o_exp = _expected(wl, live)
        ok, err, bound = oracle.within_tolerance(as_f64(run.bufs.out[:live]), o_exp, wl.dtype)
        assert ok, (bucket, live, err, bound)
        assert torch.all(run.bufs.out[live:] == SENTINEL), "padding rows' outputs were written"
        assert np.array_equal(storage(run.k_cache), k_exp), "k cache differs from the oracle's"
        assert np.array_equal(storage(run.v_cache), v_exp), "v cache differs from the oracle's"
        got_slots = run.bufs.slots[:bucket].cpu().numpy()
        assert np.array_equal(got_slots[:live], slots)
        assert np.all(got_slots[live:] == -1)
        assert pa_read_device_errors(reset=True) == 0
