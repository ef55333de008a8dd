"""pa_decode_kv_write: the step's KV write fused into decode.  The cache must
equal the oracle's bit for bit (new rows included), the reported slots must be
the oracle's slot mapping, and the outputs must match the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_harness import GpuCase, as_f64, storage
from paged_kv_gqa_08_gb300 import PA_DEVERR_BAD_LENGTH, pa_decode, pa_decode_kv_write, pa_read_device_errors

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]


def _bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _fused(run, wl, max_ctas=0, ctx=None):
    t = run.t
    row = wl.num_kv_heads * wl.head_dim
    slots = torch.full((wl.batch,), -7, dtype=torch.int64, device="cuda")
    out = torch.full_like(run.bufs.out, float("nan"))
    pa_decode_kv_write(run.desc, t["q"], t["k_new"], row, t["v_new"], row, wl.batch, run.k_cache, run.v_cache,
                       t["block_tables"], wl.max_pages_per_seq, t["context_lens"] if ctx is None else ctx,
                       wl.max_context_len, wl.scale, max_ctas, slots, out, run.bufs.workspace)
    torch.cuda.synchronize()
    return out, slots


def _check_all(run, wl, out, slots):
    ref = oracle.reference_step(wl)
    ok, err, bound = oracle.within_tolerance(as_f64(out[: wl.batch]), ref["o"], wl.dtype)
    assert ok, (err, bound)
    assert np.array_equal(slots.cpu().numpy(), ref["slots"])
    assert np.array_equal(_bits(storage(run.k_cache)), _bits(ref["k_cache"]))
    assert np.array_equal(_bits(storage(run.v_cache)), _bits(ref["v_cache"]))


@pytest.mark.parametrize("name", ["tiny_fp32_decode", "qwen3_0p6b_decode", "qwen3_8b_decode", "long_context_decode"])
def test_fused_decode_configs(name):
    wl = synth.make_workload(name)
    run = GpuCase(wl)                        # cache holds the history only
    pa_read_device_errors(reset=True)
    out, slots = _fused(run, wl)
    _check_all(run, wl, out, slots)
    assert pa_read_device_errors(reset=True) == 0


SMALL = [
    ("f32", 4, 2, 64, 16, [1, 15, 16, 17, 100]),
    ("bf16", 24, 8, 128, 16, [1, 2, 77, 500]),
    ("bf16", 32, 4, 128, 256, [255, 256, 257, 3000]),
    ("bf16", 4, 4, 64, 16, [9, 200, 31]),
    ("bf16", 48, 8, 128, 16, [300, 45, 1]),         # G = 6
    ("bf16", 28, 4, 128, 32, [130, 7]),             # G = 7
]


@pytest.mark.parametrize("case", SMALL, ids=[f"{c[0]}-hq{c[1]}-hkv{c[2]}-d{c[3]}-p{c[4]}" for c in SMALL])
@pytest.mark.parametrize("max_ctas", [0, 1, 3])
def test_fused_decode_small_shapes(case, max_ctas):
    dtype, Hq, Hkv, hd, P, lens = case
    wl = synth.make_workload(dict(kind="decode", dtype=dtype, B=len(lens), Hq=Hq, Hkv=Hkv, hd=hd, P=P,
                                  context_lens=lens, seed=sum(lens) + 5))
    run = GpuCase(wl, max_ctas=max_ctas)
    out, slots = _fused(run, wl, max_ctas)
    _check_all(run, wl, out, slots)


def test_fused_decode_reports_skipped_requests():
    wl = synth.make_workload("qwen3_0p6b_decode", B=6)
    run = GpuCase(wl)
    pa_read_device_errors(reset=True)
    ctx = run.t["context_lens"].clone()
    ctx[3] = -2         # bad metadata: skipped and flagged
    ctx[1] = 0          # a padding row: skipped, slot -1, no flag of its own
    out, slots = _fused(run, wl, ctx=ctx)
    assert pa_read_device_errors(reset=True) == PA_DEVERR_BAD_LENGTH
    s = slots.cpu().numpy()
    ref = oracle.reference_step(wl)
    assert s[3] == -1 and s[1] == -1
    good = [0, 2, 4, 5]
    assert np.array_equal(s[good], ref["slots"][good])
    ok, err, bound = oracle.within_tolerance(as_f64(out[good]), ref["o"][good], wl.dtype)
    assert ok, (err, bound)


@pytest.mark.parametrize("B", [512, 513, 1100])
def test_decode_batches_on_both_sides_of_the_in_kernel_plan_limit(B):
    """Up to 512 requests every decode CTA computes the batch's chunk prefix
    sums itself; beyond that a plan kernel computes them first.  On both sides
    of the limit: the fused call against the oracle (cache bit for bit), then
    pa_decode with a padding row (skipped, no flag) and a bad length (skipped,
    flagged) among the requests."""
    wl = synth.make_workload(dict(kind="decode", dtype="bf16", B=B, Hq=16, Hkv=8, hd=128, P=16, L_range=(1, 96),
                                  seed=B + 3))
    run = GpuCase(wl)
    pa_read_device_errors(reset=True)
    out, slots = _fused(run, wl)
    _check_all(run, wl, out, slots)
    assert pa_read_device_errors(reset=True) == 0
    ref = oracle.reference_step(wl)
    ctx = run.t["context_lens"].clone()
    ctx[B - 2] = 0
    ctx[7] = -1
    out2 = torch.full_like(run.bufs.out, 7.0)
    pa_decode(run.desc, run.t["q"], wl.batch, run.k_cache, run.v_cache, run.t["block_tables"], wl.max_pages_per_seq,
              ctx, wl.max_context_len, wl.scale, 0, out2, run.bufs.workspace)
    torch.cuda.synchronize()
    assert pa_read_device_errors(reset=True) == PA_DEVERR_BAD_LENGTH
    good = [b for b in range(B) if b not in (7, B - 2)]
    ok, err, bound = oracle.within_tolerance(as_f64(out2[good]), ref["o"][good], wl.dtype)
    assert ok, (err, bound)
    assert torch.all(out2[B - 2] == 7.0) and torch.all(out2[7] == 7.0)


@pytest.mark.parametrize("name", ["qwen3_0p6b_decode", "long_context_decode"])
def test_fused_decode_with_inputs_and_out_in_pinned_host_memory(name):
    # Pinned host memory is mapped into the device's address space: the
    # kernels read q and the new K / V rows and write the output (decode
    # kernel and merge) there directly, as the end-to-end benchmark does.
    wl = synth.make_workload(name)
    run = GpuCase(wl)
    t = run.t
    row = wl.num_kv_heads * wl.head_dim
    q_host, k_host, v_host = (t[k].cpu().pin_memory() for k in ("q", "k_new", "v_new"))
    out_host = torch.full(tuple(run.bufs.out.shape), float("nan"), dtype=run.bufs.out.dtype).pin_memory()
    slots = torch.full((wl.batch,), -7, dtype=torch.int64, device="cuda")
    pa_read_device_errors(reset=True)
    pa_decode_kv_write(run.desc, q_host, k_host, row, v_host, row, wl.batch, run.k_cache, run.v_cache,
                       t["block_tables"], wl.max_pages_per_seq, t["context_lens"], wl.max_context_len, wl.scale, 0,
                       slots, out_host, run.bufs.workspace)
    torch.cuda.synchronize()
    _check_all(run, wl, out_host, slots)
    assert pa_read_device_errors(reset=True) == 0


def test_unfused_decode_with_q_and_out_in_pinned_host_memory():
    # pa_decode on the tensor-core path: q read and the output written (decode
    # kernel and merge) in pinned host memory, after the KV write on the device
    from paged_kv_gqa_08_gb300 import pa_decode
    wl = synth.make_workload("qwen3_8b_decode")
    run = GpuCase(wl)
    run.step()                                   # writes the new rows (and decodes) on the device
    torch.cuda.synchronize()
    q_host = run.t["q"].cpu().pin_memory()
    out_host = torch.full(tuple(run.bufs.out.shape), float("nan"), dtype=run.bufs.out.dtype).pin_memory()
    pa_read_device_errors(reset=True)
    pa_decode(run.desc, q_host, wl.batch, run.k_cache, run.v_cache, run.t["block_tables"], wl.max_pages_per_seq,
              run.t["context_lens"], wl.max_context_len, wl.scale, 0, out_host, run.bufs.workspace)
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl)
    ok, err, bound = oracle.within_tolerance(as_f64(out_host[: wl.batch]), ref["o"], wl.dtype)
    assert ok, (err, bound)
    assert pa_read_device_errors(reset=True) == 0


def test_decode_output_only_16_byte_aligned():
    """pa_decode and pa_decode_kv_write with output rows 16 bytes past a
    32-byte boundary give the bytes of the same call with an aligned output."""
    wl = synth.make_workload("qwen3_0p6b_decode", B=24)
    run = GpuCase(wl)
    _fused(run, wl)  # the new rows are in the cache from here on: both calls below see the same keys
    shape = tuple(run.bufs.out.shape)
    row = wl.num_kv_heads * wl.head_dim
    slots = torch.empty(wl.batch, dtype=torch.int64, device="cuda")

    def call(fused, out):
        if fused:  # writing the new rows again stores the same bytes
            pa_decode_kv_write(run.desc, run.t["q"], run.t["k_new"], row, run.t["v_new"], row, wl.batch, run.k_cache,
                               run.v_cache, run.t["block_tables"], wl.max_pages_per_seq, run.t["context_lens"],
                               wl.max_context_len, wl.scale, 0, slots, out, run.bufs.workspace)
        else:
            pa_decode(run.desc, run.t["q"], wl.batch, run.k_cache, run.v_cache, run.t["block_tables"],
                      wl.max_pages_per_seq, run.t["context_lens"], wl.max_context_len, wl.scale, 0, out,
                      run.bufs.workspace)
        torch.cuda.synchronize()

    for fused in (True, False):
        aligned = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
        call(fused, aligned)
        buf = torch.zeros(run.bufs.out.numel() + 8, dtype=torch.bfloat16, device="cuda")
        out = buf[8:].view(shape)
        assert out.data_ptr() % 32 == 16
        call(fused, out)
        assert torch.equal(out[:wl.batch].view(torch.int16), aligned[:wl.batch].view(torch.int16)), fused
        assert torch.all(buf[:8].view(torch.int16) == 0)
    assert pa_read_device_errors(reset=True) == 0
