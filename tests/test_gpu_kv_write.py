"""GPU parity of the slot mapping and the KV write (bit-exact), and of the
fused q/k RMSNorm + RoPE (within two bf16 units in the last place)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_harness import GpuCase, storage

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]


def _close_on_unit_scale(got: np.ndarray, ref: np.ndarray, dtype: str) -> None:
    """Normed + rotated values [..., head_dim]: |got - ref| <= 3 units in the
    last place (bf16; 16 for fp32) of the rotation pair's norm, at least 1.

    The GPU normalises and rotates in fp32, the oracle in float64.  The two
    inputs of a rotation pair are each rounded to the dtype after x*r and after
    *w, so they may differ by one unit at their own magnitude; the rotation
    combines them with |cos|, |sin| <= 1 (two units) and rounds once more (one
    unit).  Both inputs are bounded by the pair's norm, which the rotation keeps,
    so that norm sets the scale -- not the output, which can cancel towards 0."""
    g, r = oracle.widen(got, dtype), oracle.widen(ref, dtype)
    half = r.shape[-1] // 2
    pair = np.sqrt(r[..., :half] ** 2 + r[..., half:] ** 2)
    pair = np.concatenate([pair, pair], axis=-1)
    mant, units = (7, 3) if dtype == "bf16" else (23, 16)
    scale = np.maximum(pair, 1.0)
    ulp = np.exp2(np.floor(np.log2(scale)) - mant)
    bad = np.abs(g - r) > units * ulp
    assert not np.any(bad), f"{int(bad.sum())} values off by up to {float(np.max(np.abs(g - r))):.3e}"


def _bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a


@pytest.mark.parametrize("name", synth.CONFIG_ORDER + ["prefill_2k"])
def test_step_slot_mapping_and_cache_write(name):
    wl = synth.make_workload(name)
    run = GpuCase(wl)
    run.step()
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl, with_attention=False)
    n = wl.num_new_tokens
    # slot mapping: exact
    assert np.array_equal(run.bufs.positions[:n].cpu().numpy(), ref["positions"])
    assert np.array_equal(run.bufs.slots[:n].cpu().numpy(), ref["slots"])
    _, hist_slots = oracle.slot_mapping(wl.block_tables, wl.hist_lens, wl.cu_hist, wl.page_size)
    assert np.array_equal(run.hist_slots[: len(hist_slots)].cpu().numpy(), hist_slots)
    kc, vc = storage(run.k_cache), storage(run.v_cache)
    # V is a pure copy everywhere; poison (NaN) bits of never-written slots match too
    assert np.array_equal(_bits(vc), _bits(ref["v_cache"]))
    if wl.q_norm_w is None:
        assert np.array_equal(_bits(kc), _bits(ref["k_cache"]))
        return
    # k of the new tokens went through RMSNorm + RoPE: compare those rows on
    # the scale of the normalised values, everything else bit for bit
    flat_g = kc.reshape(-1, wl.num_kv_heads * wl.head_dim)
    flat_r = ref["k_cache"].reshape(-1, wl.num_kv_heads * wl.head_dim)
    new = ref["slots"]
    mask = np.ones(flat_g.shape[0], bool)
    mask[new] = False
    assert np.array_equal(flat_g[mask], flat_r[mask])
    _close_on_unit_scale(flat_g[new].reshape(len(new), wl.num_kv_heads, wl.head_dim),
                         flat_r[new].reshape(len(new), wl.num_kv_heads, wl.head_dim), wl.dtype)
    _close_on_unit_scale(storage(run.bufs.q_out[:n]), ref["q"], wl.dtype)


def test_kv_write_skips_minus_one_and_flags_bad_slots():
    from paged_kv_gqa_08_gb300 import (PA_DEVERR_BAD_SLOT, cache_desc, PA_BF16, pa_kv_write,
                                       pa_read_device_errors)
    pa_read_device_errors(reset=True)
    dev = "cuda"
    desc = cache_desc(4, 2, 64, 16, 4, PA_BF16)
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    k = torch.randn(5, 2, 64, device=dev).to(torch.bfloat16)
    v = torch.randn(5, 2, 64, device=dev).to(torch.bfloat16)
    slots = torch.tensor([3, -1, 63, 64, 0], dtype=torch.int64, device=dev)   # 64 is out of range
    pa_kv_write(desc, k, 128, v, 128, 5, slots, kc, vc)
    torch.cuda.synchronize()
    fk = kc.view(64, 128)
    assert torch.equal(fk[3], k[0].view(-1)) and torch.equal(fk[63], k[2].view(-1)) and torch.equal(fk[0], k[4].view(-1))
    untouched = [s for s in range(64) if s not in (0, 3, 63)]
    assert torch.count_nonzero(fk[untouched]) == 0
    assert pa_read_device_errors(reset=True) & PA_DEVERR_BAD_SLOT


def test_kv_write_from_fused_qkv_rows():
    # k and v as strided views into one [N, (Hq + 2 Hkv) * hd] projection output
    from paged_kv_gqa_08_gb300 import cache_desc, PA_BF16, pa_kv_write
    dev = "cuda"
    Hq, Hkv, hd, N = 16, 8, 128, 37
    qkv = torch.randn(N, (Hq + 2 * Hkv) * hd, device=dev).to(torch.bfloat16)
    k = qkv[:, Hq * hd:(Hq + Hkv) * hd]
    v = qkv[:, (Hq + Hkv) * hd:]
    desc = cache_desc(Hq, Hkv, hd, 16, 8, PA_BF16)
    kc = torch.zeros(8, 16, Hkv, hd, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    slots = torch.randperm(128, device=dev)[:N].to(torch.int64)
    pa_kv_write(desc, k, qkv.stride(0), v, qkv.stride(0), N, slots, kc, vc)
    torch.cuda.synchronize()
    assert torch.equal(kc.view(128, -1)[slots], k)
    assert torch.equal(vc.view(128, -1)[slots], v)


def _two_writes(wl, edit=None):
    """The step's write part as pa_slot_mapping + pa_qk_norm_rope_kv_write and
    as pa_prefill_qk_norm_rope_kv_write, on two copies of the same state."""
    from paged_kv_gqa_08_gb300 import (pa_prefill_qk_norm_rope_kv_write, pa_qk_norm_rope_kv_write,
                                       pa_read_device_errors, pa_slot_mapping)
    runs, flags = [GpuCase(wl), GpuCase(wl)], []
    n = wl.num_new_tokens
    for k, run in enumerate(runs):
        t = run.t
        if edit is not None:
            edit(t)
        run.bufs.positions.fill_(-5)
        run.bufs.slots.fill_(-5)
        pa_read_device_errors(reset=True)
        if k == 0:
            pa_slot_mapping(run.desc, wl.batch, t["cu_seqlens_q"], t["context_lens"], t["block_tables"],
                            wl.max_pages_per_seq, n, run.bufs.positions, run.bufs.slots)
            pa_qk_norm_rope_kv_write(run.desc, t["q"], t["q"].stride(0), t["k_new"], t["k_new"].stride(0), t["v_new"],
                                     t["v_new"].stride(0), n, run.bufs.positions, t["q_norm_w"], t["k_norm_w"],
                                     wl.eps, wl.rope_theta, run.bufs.slots, run.bufs.q_out, run.k_cache, run.v_cache)
        else:
            pa_prefill_qk_norm_rope_kv_write(run.desc, t["q"], t["q"].stride(0), t["k_new"], t["k_new"].stride(0),
                                             t["v_new"], t["v_new"].stride(0), n, t["cu_seqlens_q"], wl.batch,
                                             t["context_lens"], t["block_tables"], wl.max_pages_per_seq,
                                             t["q_norm_w"], t["k_norm_w"], wl.eps, wl.rope_theta, run.bufs.q_out,
                                             run.k_cache, run.v_cache, run.bufs.positions, run.bufs.slots)
        torch.cuda.synchronize()
        flags.append(pa_read_device_errors(reset=True))
    a, b = runs
    assert flags[0] == flags[1]
    assert torch.equal(a.bufs.positions[:n], b.bufs.positions[:n])
    assert torch.equal(a.bufs.slots[:n], b.bufs.slots[:n])
    assert torch.equal(a.bufs.q_out[:n].view(torch.int16), b.bufs.q_out[:n].view(torch.int16))
    assert np.array_equal(_bits(storage(a.k_cache)), _bits(storage(b.k_cache)))
    assert np.array_equal(_bits(storage(a.v_cache)), _bits(storage(b.v_cache)))
    return flags[1]


@pytest.mark.parametrize("name", ["qwen3_0p6b_chunked_prefill", "prefill_2k"])
def test_prefill_write_in_one_kernel_equals_slot_mapping_then_norm_rope(name):
    assert _two_writes(synth.make_workload(name)) == 0


def test_prefill_write_in_one_kernel_padding_rows_and_bad_pages():
    from paged_kv_gqa_08_gb300 import PA_DEVERR_BAD_PAGE
    spec = dict(kind="prefill", dtype="bf16", B=5, Hq=16, Hkv=8, hd=128, P=16, chunks=[7, 40, 1, 33, 2],
                prefixes=[0, 300, 64, 17, 5], norm=True, seed=13)
    wl = synth.make_workload(spec)

    def edit(t):
        t["context_lens"][2] = 0                                # a padding row: position 0, slot -1, no flag
        t["block_tables"][3, 1] = wl.num_pages + 9              # a page past the cache: slot -1, flagged
    assert _two_writes(wl, edit) == PA_DEVERR_BAD_PAGE
