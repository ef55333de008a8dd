"""pa_decode_no_alloc, the decode entry point for callers that cannot
allocate device memory (a plugin handed only its buffers, a framework that
forbids allocation at that point, a process whose allocator owns the device
heap).  It must give the oracle's results (and pa_decode's) from the
library's fixed scratch, call after call, and refuse batches too large for
that scratch.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import pytest
import torch

import oracle
import synth
from gpu_harness import GpuCase, as_f64
from paged_kv_gqa_08_gb300 import PA_BF16, PA_ERR_WORKSPACE, PA_OK, cache_desc, load_library, pa_read_device_errors

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _call(lib, run, wl, out, batch=None, max_ctx=None):
    """pa_decode_no_alloc straight through the C ABI."""
    return lib.pa_decode_no_alloc(
        ctypes.byref(run.desc), run.t["q"].data_ptr(), wl.batch if batch is None else batch,
        run.k_cache.data_ptr(), run.v_cache.data_ptr(), run.t["block_tables"].data_ptr(), wl.max_pages_per_seq,
        run.t["context_lens"].data_ptr(), wl.max_context_len if max_ctx is None else max_ctx, wl.scale, 0,
        out.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", ["qwen3_0p6b_decode", "qwen3_8b_decode", "long_context_decode", "tiny_fp32_decode"])
def test_no_alloc_matches_oracle_and_pa_decode_on_two_calls_in_a_row(name):
    lib = load_library()
    wl = synth.make_workload(name)
    run = GpuCase(wl)
    with_ws = as_f64(run.step()[: wl.batch])       # the step's KV write, then pa_decode with a caller workspace
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl)["o"]
    pa_read_device_errors(reset=True)
    for _ in range(2):                              # the second call reuses the scratch as the first left it
        out = torch.full_like(run.bufs.out, float("nan"))
        assert _call(lib, run, wl, out) == PA_OK
        torch.cuda.synchronize()
        got = as_f64(out[: wl.batch])
        ok, err, bound = oracle.within_tolerance(got, ref, wl.dtype)
        assert ok, ("oracle", err, bound)
        ok, err, bound = oracle.within_tolerance(got, with_ws, wl.dtype)
        assert ok, ("pa_decode", err, bound)
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


_FIRST_CALL_CHILD = textwrap.dedent("""
    import ctypes, sys
    sys.path[:0] = [{root!r}, {tests!r}]
    import torch, oracle, synth
    from gpu_harness import GpuCase, as_f64
    from paged_kv_gqa_08_gb300 import PA_OK, load_library
    lib = load_library()
    wl = synth.make_workload("qwen3_8b_decode", B=6)
    run = GpuCase(wl)
    run.step()
    torch.cuda.synchronize()
    out = torch.full_like(run.bufs.out, float("nan"))
    st = lib.pa_decode_no_alloc(ctypes.byref(run.desc), run.t["q"].data_ptr(), wl.batch, run.k_cache.data_ptr(),
                                run.v_cache.data_ptr(), run.t["block_tables"].data_ptr(), wl.max_pages_per_seq,
                                run.t["context_lens"].data_ptr(), wl.max_context_len, wl.scale, 0, out.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    assert st == PA_OK, st
    torch.cuda.synchronize()
    ok, err, bound = oracle.within_tolerance(as_f64(out[: wl.batch]), oracle.reference_step(wl)["o"], wl.dtype)
    assert ok, (err, bound)
    print("first call ok", err)
""")


def test_no_alloc_first_call_in_a_fresh_process_with_lazy_module_loading():
    # With lazy module loading the fixed scratch is placed in device memory by
    # the first call's address lookup; that first call must succeed and be right.
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY")
    code = _FIRST_CALL_CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "first call ok" in r.stdout
