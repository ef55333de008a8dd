"""GPU parity of batched GQA decode (split-KV + LSE merge) against the oracle."""
import pytest
import torch

import oracle
import synth
from gpu_harness import GpuCase, as_f64
from paged_kv_gqa_08_gb300 import (PA_DEVERR_BAD_LENGTH, PA_DEVERR_BAD_PAGE, pa_decode, pa_decode_workspace_size,
                                   pa_read_device_errors)

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]


def _check(out, ref, dtype):
    ok, err, bound = oracle.within_tolerance(as_f64(out), ref, dtype)
    assert ok, f"max abs err {err:.3e} > bound {bound:.3e}"
    return err


@pytest.mark.parametrize("name", ["tiny_fp32_decode", "qwen3_0p6b_decode", "qwen3_8b_decode", "long_context_decode"])
def test_decode_configs_match_oracle(name):
    wl = synth.make_workload(name)
    pa_read_device_errors(reset=True)
    run = GpuCase(wl)
    out = run.step()
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl)
    _check(out[: wl.batch], ref["o"], wl.dtype)
    assert pa_read_device_errors(reset=True) == 0


SMALL = [
    # dtype, Hq, Hkv, hd, P, context lens
    ("f32", 4, 2, 64, 16, [1, 15, 16, 17, 100]),
    ("f32", 8, 8, 128, 32, [3, 64, 65, 300]),
    ("f32", 6, 2, 64, 16, [40, 7]),
    ("bf16", 8, 8, 128, 16, [1, 2, 16, 17, 1000, 2049]),
    ("bf16", 16, 8, 128, 256, [255, 256, 257, 3000]),
    ("bf16", 24, 8, 128, 16, [77, 500]),           # G = 3
    ("bf16", 32, 4, 128, 64, [33, 129, 900]),       # G = 8
    ("bf16", 20, 4, 128, 16, [5, 700]),             # G = 5
    ("bf16", 4, 4, 64, 16, [9, 200, 31]),           # G = 1, head_dim 64
    ("bf16", 16, 2, 64, 128, [1, 1000]),            # G = 8, head_dim 64
    ("bf16", 2, 1, 128, 16, [50, 51]),              # one kv head
    ("bf16", 48, 8, 128, 16, [300, 45, 1]),         # G = 6 (heads padded to 8 in the reduction)
    ("bf16", 28, 4, 128, 32, [130, 7]),             # G = 7
    ("bf16", 12, 2, 64, 16, [66, 500]),             # G = 6, head_dim 64
    ("f32", 14, 2, 64, 16, [20, 90]),               # G = 7
    ("f32", 24, 4, 128, 16, [64, 3]),               # G = 6, head_dim 128
    ("bf16", 64, 8, 128, 16, [1, 333, 2000]),       # the largest head set: 8 kv-heads x G = 8
    ("f32", 64, 8, 64, 32, [90, 7]),                # the same in fp32, head_dim 64
]


@pytest.mark.parametrize("case", SMALL, ids=[f"{c[0]}-hq{c[1]}-hkv{c[2]}-d{c[3]}-p{c[4]}" for c in SMALL])
@pytest.mark.parametrize("max_ctas", [0, 1, 5])
def test_decode_small_shapes(case, max_ctas):
    dtype, Hq, Hkv, hd, P, lens = case
    spec = dict(kind="decode", dtype=dtype, B=len(lens), Hq=Hq, Hkv=Hkv, hd=hd, P=P, context_lens=lens, seed=sum(lens))
    wl = synth.make_workload(spec)
    run = GpuCase(wl, max_ctas=max_ctas)
    out = run.step()
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl)
    _check(out[: wl.batch], ref["o"], wl.dtype)
    assert pa_read_device_errors(reset=True) == 0


def test_decode_split_plans_agree():
    wl = synth.make_workload("qwen3_8b_decode", B=12)
    ref = oracle.reference_step(wl)
    outs = []
    for max_ctas in (1, 3, 0):
        run = GpuCase(wl, max_ctas=max_ctas)
        outs.append(run.step().clone())
    torch.cuda.synchronize()
    for o in outs:
        _check(o[: wl.batch], ref["o"], wl.dtype)


def test_decode_page_permutation_is_bitwise_invariant():
    wl = synth.make_workload("qwen3_0p6b_decode", B=24)
    run = GpuCase(wl)
    out1 = run.step().clone()
    perm = torch.randperm(wl.num_pages, device="cuda")
    kc2 = torch.empty_like(run.k_cache)
    vc2 = torch.empty_like(run.v_cache)
    kc2[perm] = run.k_cache
    vc2[perm] = run.v_cache
    bt2 = perm[run.t["block_tables"].long()].to(torch.int32)
    out2 = torch.empty_like(out1)
    pa_decode(run.desc, run.t["q"], wl.batch, kc2, vc2, bt2, wl.max_pages_per_seq, run.t["context_lens"],
              wl.max_context_len, wl.scale, 0, out2, run.bufs.workspace)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_decode_flags_bad_metadata_and_keeps_other_requests_right():
    wl = synth.make_workload("qwen3_0p6b_decode", B=6)
    ref = oracle.reference_step(wl)
    run = GpuCase(wl)
    run.step()
    torch.cuda.synchronize()
    pa_read_device_errors(reset=True)
    # request 2: an out-of-range page id; request 4: a negative context length;
    # request 1: a padding row (length 0), skipped without a flag
    bt = run.t["block_tables"].clone()
    bt[2, 0] = 10 ** 6
    ctx = run.t["context_lens"].clone()
    ctx[4] = -3
    ctx[1] = 0
    out = torch.full_like(run.bufs.out, 7.0)
    pa_decode(run.desc, run.t["q"], wl.batch, run.k_cache, run.v_cache, bt, wl.max_pages_per_seq, ctx,
              wl.max_context_len, wl.scale, 0, out, run.bufs.workspace)
    torch.cuda.synchronize()
    flags = pa_read_device_errors(reset=True)
    assert flags & PA_DEVERR_BAD_PAGE and flags & PA_DEVERR_BAD_LENGTH
    good = [0, 3, 5]
    _check(out[good], ref["o"][good], wl.dtype)
    assert torch.all(out[4] == 7.0)          # skipped request: output untouched
    assert torch.all(out[1] == 7.0)          # padding row: output untouched
    # a padding row alone raises nothing
    bt = run.t["block_tables"].clone()
    bt[1] = -7
    pa_decode(run.desc, run.t["q"], wl.batch, run.k_cache, run.v_cache, bt, wl.max_pages_per_seq, ctx.clamp(min=0),
              wl.max_context_len, wl.scale, 0, out, run.bufs.workspace)
    torch.cuda.synchronize()
    assert pa_read_device_errors(reset=True) == 0


def test_decode_zero_batch_is_a_no_op():
    wl = synth.make_workload("tiny_fp32_decode")
    run = GpuCase(wl)
    pa_decode(run.desc, run.t["q"], 0, run.k_cache, run.v_cache, run.t["block_tables"], wl.max_pages_per_seq,
              run.t["context_lens"], wl.max_context_len, wl.scale, 0, run.bufs.out, run.bufs.workspace)
    torch.cuda.synchronize()


def test_decode_workspace_too_small_is_rejected():
    from paged_kv_gqa_08_gb300 import PA_ERR_WORKSPACE, PagedAttnError
    wl = synth.make_workload("tiny_fp32_decode")
    run = GpuCase(wl)
    need = pa_decode_workspace_size(run.desc, wl.batch, wl.max_context_len, 0)
    assert need > 0
    with pytest.raises(PagedAttnError) as e:
        pa_decode(run.desc, run.t["q"], wl.batch, run.k_cache, run.v_cache, run.t["block_tables"],
                  wl.max_pages_per_seq, run.t["context_lens"], wl.max_context_len, wl.scale, 0, run.bufs.out,
                  run.bufs.workspace, need - 256)
    assert e.value.status == PA_ERR_WORKSPACE
