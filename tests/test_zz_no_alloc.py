"""pa_decode_no_alloc, the decode entry point for callers that cannot
allocate device memory (a plugin handed only its buffers, a framework that
forbids allocation at that point, a process whose allocator owns the device
heap).  It must give pa_decode's results from the library's fixed
scratch, call after call, and refuse batches too large for that scratch.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import oracle
import synth
from gpu_harness import GpuCase, as_f64
from paged_kv_gqa_08_gb300 import PA_BF16, PA_ERR_WORKSPACE, PA_OK, cache_desc, load_library, pa_read_device_errors

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]


def _call(lib, run, wl, out, batch=None, max_ctx=None):
    """pa_decode_no_alloc straight through the C ABI."""
    return lib.pa_decode_no_alloc(
        ctypes.byref(run.desc), run.t["q"].data_ptr(), wl.batch if batch is None else batch,
        run.k_cache.data_ptr(), run.v_cache.data_ptr(), run.t["block_tables"].data_ptr(), wl.max_pages_per_seq,
        run.t["context_lens"].data_ptr(), wl.max_context_len if max_ctx is None else max_ctx, wl.scale, 0,
        out.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", ["qwen3_0p6b_decode", "qwen3_8b_decode", "tiny_fp32_decode"])
def test_no_alloc_matches_pa_decode_on_two_calls_in_a_row(name):
    lib = load_library()
    wl = synth.make_workload(name)
    run = GpuCase(wl)
    ref = as_f64(run.step()[: wl.batch])          # pa_decode with a caller workspace
    pa_read_device_errors(reset=True)
    for _ in range(2):                              # the second call reuses the scratch as the first left it
        out = torch.full_like(run.bufs.out, float("nan"))
        assert _call(lib, run, wl, out) == PA_OK
        torch.cuda.synchronize()
        ok, err, bound = oracle.within_tolerance(as_f64(out[: wl.batch]), ref, wl.dtype)
        assert ok, (err, bound)
    assert pa_read_device_errors(reset=True) == 0


def test_no_alloc_rejects_a_batch_larger_than_its_scratch():
    lib = load_library()
    wl = synth.make_workload("qwen3_0p6b_decode", B=4)
    run = GpuCase(wl)
    out = torch.empty_like(run.bufs.out)
    # 4096 requests of 64 q-heads x 128 need far more than 16 MiB of partials;
    # the call is refused on the host before anything is enqueued
    big = cache_desc(64, 8, 128, 16, wl.num_pages, PA_BF16)
    st = lib.pa_decode_no_alloc(ctypes.byref(big), run.t["q"].data_ptr(), 4096, run.k_cache.data_ptr(),
                                run.v_cache.data_ptr(), run.t["block_tables"].data_ptr(), wl.max_pages_per_seq,
                                run.t["context_lens"].data_ptr(), wl.max_context_len, wl.scale, 0,
                                out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == PA_ERR_WORKSPACE
