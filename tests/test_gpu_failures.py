"""Failure detection on the GPU without faulting it: the bounded-wait path,
the metadata validator, and host-side argument errors."""
import time

import pytest
import torch

import oracle
import synth
from gpu_harness import GpuCase, as_f64
from paged_kv_gqa_08_gb300 import (PA_DEVERR_TIMEOUT, pa_read_device_errors, pa_selftest_bounded_wait,
                                   pa_validate_metadata)

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]


def test_bounded_wait_gives_up_flags_and_leaves_context_usable():
    pa_read_device_errors(reset=True)
    t0 = time.perf_counter()
    pa_selftest_bounded_wait(200)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    assert 0.15 < el < 10.0
    assert pa_read_device_errors(reset=True) & PA_DEVERR_TIMEOUT
    # the context still runs real work correctly
    wl = synth.make_workload("tiny_fp32_decode")
    out = GpuCase(wl).step()
    torch.cuda.synchronize()
    ok, err, bound = oracle.within_tolerance(as_f64(out[: wl.batch]), oracle.reference_step(wl)["o"], wl.dtype)
    assert ok, (err, bound)
    assert pa_read_device_errors(reset=True) == 0


def test_validate_metadata_counts_problems():
    wl = synth.make_workload("qwen3_0p6b_chunked_prefill")
    run = GpuCase(wl)
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (run.desc, wl.batch)
    pa_validate_metadata(*args, run.t["cu_seqlens_q"], run.t["context_lens"], run.t["block_tables"],
                         wl.max_pages_per_seq, wl.max_context_len, cnt)
    torch.cuda.synchronize()
    assert int(cnt.item()) == 0
    bt = run.t["block_tables"].clone()
    bt[3, 0] = -5
    bt[6, 1] = wl.num_pages
    ctx = run.t["context_lens"].clone()
    ctx[2] = -1
    ctx[5] = 0          # a padding row: not a problem
    bt[5] = -9          # (its block-table row is never looked at)
    cu = run.t["cu_seqlens_q"].clone()
    pa_validate_metadata(*args, cu, ctx, bt, wl.max_pages_per_seq, wl.max_context_len, cnt)
    torch.cuda.synchronize()
    assert int(cnt.item()) == 3
