"""GPU parity of chunked prefill (norm + rope + KV write + attention) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_harness import GpuCase, as_f64
from paged_kv_gqa_08_gb300 import (pa_kv_write, pa_prefill_qk_norm_rope_kv_write, pa_prefill_varlen,
                                   pa_prefill_workspace_size, pa_read_device_errors, pa_slot_mapping)

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("cuda_lib")]


def _check(out, ref, dtype):
    ok, err, bound = oracle.within_tolerance(as_f64(out), ref, dtype)
    assert ok, f"max abs err {err:.3e} > bound {bound:.3e}"
    return err


@pytest.mark.parametrize("name", ["qwen3_0p6b_chunked_prefill", "prefill_2k"])
def test_prefill_configs_match_oracle(name):
    wl = synth.make_workload(name)
    pa_read_device_errors(reset=True)
    run = GpuCase(wl)
    out = run.step()
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl)
    _check(out[: wl.num_new_tokens], ref["o"], wl.dtype)
    assert pa_read_device_errors(reset=True) == 0


def test_workspace_sized_for_the_largest_batch_serves_a_smaller_call():
    """The planned-prefill workspace size never shrinks as the token bound
    grows, so one workspace sized for the largest batch (here 16k tokens, a
    batch that would not split) serves the mixed chunked-prefill step."""
    wl = synth.make_workload("qwen3_0p6b_chunked_prefill")
    run = GpuCase(wl)
    sizes = [pa_prefill_workspace_size(run.desc, wl.batch, 2048, n, 8192) for n in (64, 1218, 4096, 16384)]
    assert sizes[0] > 0 and all(a <= b for a, b in zip(sizes, sizes[1:])), sizes
    run.bufs.workspace = torch.empty(sizes[-1], dtype=torch.uint8, device="cuda")
    pa_read_device_errors(reset=True)
    out = run.step()
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl)
    _check(out[: wl.num_new_tokens], ref["o"], wl.dtype)
    assert pa_read_device_errors(reset=True) == 0


SMALL = [
    # dtype, Hq, Hkv, hd, P, chunks, prefixes, norm
    ("bf16", 16, 8, 128, 16, [1, 7, 63, 64, 65, 129, 300], [0, 5, 127, 128, 200, 1000, 33], True),
    ("bf16", 16, 8, 128, 256, [130, 1, 64], [0, 257, 700], False),
    ("bf16", 8, 8, 128, 16, [200, 3], [50, 0], True),           # G = 1
    ("bf16", 16, 4, 128, 32, [37, 90], [11, 300], True),        # G = 4
    ("bf16", 32, 4, 128, 16, [17, 40], [160, 2], False),        # G = 8
    ("bf16", 24, 8, 128, 16, [45, 12], [9, 130], True),         # G = 3
    ("bf16", 20, 4, 128, 64, [30, 26], [64, 1], False),         # G = 5
    ("bf16", 48, 8, 128, 16, [40, 9], [100, 0], True),          # G = 6 (21-token q-tiles, 126 rows)
    ("bf16", 28, 4, 128, 32, [25, 70], [5, 200], False),        # G = 7 (18-token q-tiles)
    ("bf16", 8, 4, 64, 16, [20, 5], [40, 0], True),             # head_dim 64 (CUDA-core kernel)
    ("f32", 4, 2, 64, 16, [1, 9, 33], [0, 16, 5], True),
    ("f32", 8, 4, 128, 32, [70, 2], [0, 100], False),
    ("bf16", 64, 8, 128, 16, [70, 5, 130], [33, 300, 0], True),   # the largest head set: 8 kv-heads x G = 8
    ("bf16", 64, 8, 64, 16, [40, 3], [9, 120], False),             # the same with head_dim 64 (CUDA cores)
]


@pytest.mark.parametrize("case", SMALL, ids=[f"{c[0]}-hq{c[1]}-hkv{c[2]}-d{c[3]}-p{c[4]}-{'norm' if c[7] else 'plain'}"
                                             for c in SMALL])
def test_prefill_small_shapes(case):
    dtype, Hq, Hkv, hd, P, chunks, prefixes, norm = case
    spec = dict(kind="prefill", dtype=dtype, B=len(chunks), Hq=Hq, Hkv=Hkv, hd=hd, P=P, chunks=chunks,
                prefixes=prefixes, norm=norm, seed=sum(chunks) + 7)
    wl = synth.make_workload(spec)
    run = GpuCase(wl)
    out = run.step()
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl)
    _check(out[: wl.num_new_tokens], ref["o"], wl.dtype)
    assert pa_read_device_errors(reset=True) == 0


def test_prefill_with_length_one_chunks_matches_decode():
    wl = synth.make_workload("qwen3_0p6b_decode", B=16)
    run = GpuCase(wl)
    out_dec = run.step().clone()
    out_pf = torch.empty_like(out_dec)
    pa_prefill_varlen(run.desc, run.t["q"], run.t["cu_seqlens_q"], wl.batch, 1, wl.batch, run.k_cache, run.v_cache,
                      run.t["block_tables"], wl.max_pages_per_seq, run.t["context_lens"], wl.max_context_len,
                      wl.scale, out_pf)
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl)
    _check(out_dec[: wl.batch], ref["o"], wl.dtype)
    _check(out_pf[: wl.batch], ref["o"], wl.dtype)


def test_prefill_empty_requests_in_batch():
    # requests with no new tokens are skipped; the others are unaffected
    spec = dict(kind="prefill", dtype="bf16", B=4, Hq=16, Hkv=8, hd=128, P=16, chunks=[0, 40, 0, 3],
                prefixes=[10, 20, 0, 64], norm=True, seed=99)
    wl = synth.make_workload(spec)
    run = GpuCase(wl)
    out = run.step()
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl)
    _check(out[: wl.num_new_tokens], ref["o"], wl.dtype)


def test_mixed_decode_rows_and_prefill_chunks_in_one_launch():
    # decode requests are chunks of length 1 in the same varlen batch as real chunks
    spec = dict(kind="prefill", dtype="bf16", B=6, Hq=32, Hkv=8, hd=128, P=16, chunks=[1, 300, 1, 1, 77, 1],
                prefixes=[900, 0, 45, 2047, 129, 3], norm=True, seed=21)
    wl = synth.make_workload(spec)
    run = GpuCase(wl)
    out = run.step()
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl)
    _check(out[: wl.num_new_tokens], ref["o"], wl.dtype)


def _plan_header(run):
    """{CTAs per kv-head, split pairs, part size, q-tile pairs} of the last planned call."""
    return run.bufs.workspace[:16].view(torch.int32).tolist()


def test_planned_and_unplanned_launches_agree_on_the_mixed_chunk_batch():
    wl = synth.make_workload("qwen3_0p6b_chunked_prefill")
    ref = oracle.reference_step(wl)
    pa_read_device_errors(reset=True)
    plain = GpuCase(wl, plan_prefill=False)
    assert plain.bufs.workspace is None
    out_plain = plain.step().clone()
    planned = GpuCase(wl)
    out_planned = planned.step()
    torch.cuda.synchronize()
    units, splits, tau, pairs = _plan_header(planned)
    assert pairs == 14 and splits > 0 and units > pairs and tau >= 2
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        # the planner's scoring on a 152-SM GB300: parts of 31 key tiles, the
        # fastest size measured for this batch -- the four 33-36-tile pairs of
        # the 512-token chunk over 4096 and the two 32-tile single q-tiles are
        # cut in two
        assert (units, splits, tau) == (20, 6, 31)
    _check(out_plain[: wl.num_new_tokens], ref["o"], wl.dtype)
    _check(out_planned[: wl.num_new_tokens], ref["o"], wl.dtype)
    assert pa_read_device_errors(reset=True) == 0


LONG = [
    # Hq, Hkv, P, chunks, prefixes: few q-tile pairs over long prefixes, so the
    # planner cuts each pair's keys into many parts
    (16, 8, 16, [200], [20000]),
    (32, 4, 32, [1, 90, 1], [9000, 15000, 31]),    # G = 8; single-row tiles
    (8, 8, 16, [130, 1], [12000, 6000]),           # G = 1
]


@pytest.mark.parametrize("case", LONG, ids=[f"hq{c[0]}-hkv{c[1]}-chunks{len(c[3])}" for c in LONG])
def test_split_key_ranges_match_oracle(case):
    Hq, Hkv, P, chunks, prefixes = case
    spec = dict(kind="prefill", dtype="bf16", B=len(chunks), Hq=Hq, Hkv=Hkv, hd=128, P=P, chunks=chunks,
                prefixes=prefixes, norm=True, seed=sum(prefixes) % 1000 + 3)
    wl = synth.make_workload(spec)
    pa_read_device_errors(reset=True)
    run = GpuCase(wl)
    out = run.step()
    torch.cuda.synchronize()
    units, splits, tau, pairs = _plan_header(run)
    assert splits > 0 and units > pairs
    ref = oracle.reference_step(wl)
    _check(out[: wl.num_new_tokens], ref["o"], wl.dtype)
    assert pa_read_device_errors(reset=True) == 0


def test_planned_prefill_with_empty_requests_and_tiny_workload():
    spec = dict(kind="prefill", dtype="bf16", B=5, Hq=16, Hkv=8, hd=128, P=16, chunks=[0, 3, 0, 1, 0],
                prefixes=[10, 5000, 0, 1, 7], norm=True, seed=5)
    wl = synth.make_workload(spec)
    pa_read_device_errors(reset=True)
    run = GpuCase(wl)
    out = run.step()
    torch.cuda.synchronize()
    assert _plan_header(run)[3] == 2          # only the two non-empty requests have pairs
    ref = oracle.reference_step(wl)
    _check(out[: wl.num_new_tokens], ref["o"], wl.dtype)
    assert pa_read_device_errors(reset=True) == 0


# Random batches through the planned launch: group sizes 1-8, page sizes 16-256,
# chunk and prefix mixes that make the planner split some pairs (few pairs over
# long prefixes) and not others; every case against the oracle.
RANDOM_CASES = 12


@pytest.mark.parametrize("seed", range(RANDOM_CASES))
def test_random_planned_batches_match_oracle(seed):
    rng = np.random.default_rng(1000 + seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8]))
    P = int(rng.choice([16, 32, 64, 256]))
    B = int(rng.integers(1, 6))
    chunks = [int(c) for c in rng.choice([1, 3, 17, 64, 100, 250], size=B)]
    prefixes = [int(x) for x in rng.integers(0, 3000, size=B)]
    spec = dict(kind="prefill", dtype="bf16", B=B, Hq=Hkv * G, Hkv=Hkv, hd=128, P=P, chunks=chunks,
                prefixes=prefixes, norm=bool(seed % 2), seed=seed + 50)
    wl = synth.make_workload(spec)
    pa_read_device_errors(reset=True)
    run = GpuCase(wl)
    out = run.step()
    torch.cuda.synchronize()
    ref = oracle.reference_step(wl)
    _check(out[: wl.num_new_tokens], ref["o"], wl.dtype)
    assert pa_read_device_errors(reset=True) == 0


@pytest.mark.parametrize("planned", [True, False], ids=["planned", "unplanned"])
def test_prefill_padding_rows_are_skipped(planned):
    # Requests 1 and 3 become padding rows (context length 0, block-table rows
    # that hold no page id): their output rows stay untouched, no flag is
    # raised, and the other requests are unaffected.
    spec = dict(kind="prefill", dtype="bf16", B=4, Hq=16, Hkv=8, hd=128, P=16, chunks=[20, 5, 30, 7],
                prefixes=[100, 40, 0, 300], norm=False, seed=31)
    wl = synth.make_workload(spec)
    run = GpuCase(wl, plan_prefill=planned)
    run.step()
    torch.cuda.synchronize()
    pa_read_device_errors(reset=True)
    ctx = run.t["context_lens"].clone()
    bt = run.t["block_tables"].clone()
    for b in (1, 3):
        ctx[b] = 0
        bt[b] = -7
    out = torch.full_like(run.bufs.out, 3.0)
    pa_prefill_varlen(run.desc, run.t["q"], run.t["cu_seqlens_q"], wl.batch, wl.max_new_len, wl.num_new_tokens,
                      run.k_cache, run.v_cache, bt, wl.max_pages_per_seq, ctx, wl.max_context_len, wl.scale, out,
                      run.bufs.workspace)
    torch.cuda.synchronize()
    assert pa_read_device_errors(reset=True) == 0
    cu = wl.cu_seqlens_q
    rows = {b: list(range(cu[b], cu[b + 1])) for b in range(wl.batch)}
    ref = oracle.reference_step(wl, requests=[0, 2])
    _check(out[rows[0] + rows[2]], ref["o"], wl.dtype)
    assert torch.all(out[rows[1] + rows[3]] == 3.0)


PERMUTED = {
    "mixed_chunks": "qwen3_0p6b_chunked_prefill",
    "split_key_ranges": dict(kind="prefill", dtype="bf16", B=3, Hq=32, Hkv=4, hd=128, P=32, chunks=[1, 90, 1],
                             prefixes=[9000, 15000, 31], norm=True, seed=77),
}


@pytest.mark.parametrize("planned", [True, False], ids=["planned", "unplanned"])
@pytest.mark.parametrize("case", sorted(PERMUTED))
def test_prefill_page_permutation_is_bitwise_invariant(case, planned):
    # Moving every page to another physical id (and rewriting the block
    # tables to match) changes no output bit: the work split and the order
    # of the arithmetic depend on logical positions only.
    wl = synth.make_workload(PERMUTED[case])
    run = GpuCase(wl, plan_prefill=planned)
    out1 = run.step().clone()
    if planned:
        assert _plan_header(run)[1] > 0 or case == "mixed_chunks"
    g = torch.Generator(device="cuda").manual_seed(5)
    perm = torch.randperm(wl.num_pages, device="cuda", generator=g)
    kc2 = torch.empty_like(run.k_cache)
    vc2 = torch.empty_like(run.v_cache)
    kc2[perm] = run.k_cache
    vc2[perm] = run.v_cache
    bt2 = perm[run.t["block_tables"].long()].to(torch.int32)
    q = run.bufs.q_out if wl.q_norm_w is not None else run.t["q"]
    out2 = torch.full_like(out1, float("nan"))
    pa_prefill_varlen(run.desc, q, run.t["cu_seqlens_q"], wl.batch, wl.max_new_len, wl.num_new_tokens, kc2, vc2, bt2,
                      wl.max_pages_per_seq, run.t["context_lens"], wl.max_context_len, wl.scale, out2,
                      run.bufs.workspace)
    torch.cuda.synchronize()
    n = wl.num_new_tokens
    assert torch.equal(out1[:n].view(torch.int16), out2[:n].view(torch.int16))
    assert pa_read_device_errors(reset=True) == 0


def _separate_calls(run):
    """The prefill step as the calls pa_prefill_step is defined by, one after another."""
    wl, t, b = run.wl, run.t, run.bufs
    n = wl.num_new_tokens
    if t["q_norm_w"] is not None:
        pa_prefill_qk_norm_rope_kv_write(run.desc, t["q"], t["q"].stride(0), t["k_new"], t["k_new"].stride(0),
                                         t["v_new"], t["v_new"].stride(0), n, t["cu_seqlens_q"], wl.batch,
                                         t["context_lens"], t["block_tables"], wl.max_pages_per_seq, t["q_norm_w"],
                                         t["k_norm_w"], wl.eps, wl.rope_theta, b.q_out, run.k_cache, run.v_cache,
                                         b.positions, b.slots)
        qa = b.q_out
    else:
        pa_slot_mapping(run.desc, wl.batch, t["cu_seqlens_q"], t["context_lens"], t["block_tables"],
                        wl.max_pages_per_seq, n, b.positions, b.slots)
        pa_kv_write(run.desc, t["k_new"], t["k_new"].stride(0), t["v_new"], t["v_new"].stride(0), n, b.slots,
                    run.k_cache, run.v_cache)
        qa = t["q"]
    pa_prefill_varlen(run.desc, qa, t["cu_seqlens_q"], wl.batch, max(wl.max_new_len, 1), n, run.k_cache, run.v_cache,
                      t["block_tables"], wl.max_pages_per_seq, t["context_lens"], max(wl.max_context_len, 1),
                      wl.scale, b.out, b.workspace)
    return b.out


STEP_CASES = [
    ("qwen3_0p6b_chunked_prefill", True),
    ("qwen3_0p6b_chunked_prefill", False),
    ("prefill_2k", True),
    (dict(kind="prefill", dtype="bf16", B=4, Hq=16, Hkv=4, hd=128, P=16, chunks=[300, 1, 45, 129],
          prefixes=[2000, 70, 0, 513], norm=False, seed=41), True),          # plain: slot mapping + KV write
    (dict(kind="prefill", dtype="f32", B=3, Hq=4, Hkv=2, hd=64, P=16, chunks=[1, 9, 33],
          prefixes=[0, 16, 5], norm=True, seed=50), True),                   # CUDA-core attention
]


@pytest.mark.parametrize("case", STEP_CASES, ids=[f"{c[0] if isinstance(c[0], str) else c[0]['dtype'] + '-' + ('norm' if c[0]['norm'] else 'plain')}-{'planned' if c[1] else 'unplanned'}" for c in STEP_CASES])
def test_prefill_step_equals_the_separate_calls(case):
    """pa_prefill_step (its planner beside the write kernel) gives exactly the
    cache, positions, slots, q_out and output of the separate calls."""
    name, planned = case
    wl = synth.make_workload(name)
    runs = [GpuCase(wl, plan_prefill=planned), GpuCase(wl, plan_prefill=planned)]
    outs = []
    for k, run in enumerate(runs):
        run.bufs.out.fill_(0)
        run.bufs.positions.fill_(-5)
        run.bufs.slots.fill_(-5)
        pa_read_device_errors(reset=True)
        outs.append(run.step() if k == 0 else _separate_calls(run))
        torch.cuda.synchronize()
        assert pa_read_device_errors(reset=True) == 0
    a, b = runs
    n = wl.num_new_tokens

    def bits(x):
        return x.contiguous().view(-1).view(torch.int16 if x.dtype == torch.bfloat16 else torch.int32)
    assert torch.equal(bits(outs[0]), bits(outs[1]))
    assert torch.equal(a.bufs.positions[:n], b.bufs.positions[:n])
    assert torch.equal(a.bufs.slots[:n], b.bufs.slots[:n])
    if wl.q_norm_w is not None:
        assert torch.equal(bits(a.bufs.q_out[:n]), bits(b.bufs.q_out[:n]))
    assert torch.equal(bits(a.k_cache), bits(b.k_cache)) and torch.equal(bits(a.v_cache), bits(b.v_cache))
    _check(outs[0][:n], oracle.reference_step(wl)["o"], wl.dtype)


@pytest.mark.parametrize("planned", [True, False])
def test_prefill_output_only_16_byte_aligned(planned):
    """An output whose rows start 16 bytes past a 32-byte boundary: the TMA
    stores of whole-token rows and the threads' own stores of ragged rows give
    the bytes of an aligned output."""
    spec = dict(kind="prefill", dtype="bf16", B=3, Hq=16, Hkv=8, hd=128, P=16, chunks=[128, 77, 300],
                prefixes=[0, 500, 64], norm=False, seed=77)
    wl = synth.make_workload(spec)
    run = GpuCase(wl, plan_prefill=planned)
    n = wl.num_new_tokens
    aligned = run.step()[:n].clone()
    torch.cuda.synchronize()
    shape = tuple(run.bufs.out.shape)
    buf = torch.zeros(run.bufs.out.numel() + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(shape)
    assert out.data_ptr() % 32 == 16
    pa_prefill_varlen(run.desc, run.t["q"], run.t["cu_seqlens_q"], wl.batch, wl.max_new_len, n, run.k_cache,
                      run.v_cache, run.t["block_tables"], wl.max_pages_per_seq, run.t["context_lens"],
                      wl.max_context_len, wl.scale, out, run.bufs.workspace)
    torch.cuda.synchronize()
    assert torch.equal(out[:n].view(torch.int16), aligned.view(torch.int16))
    assert torch.all(buf[:8].view(torch.int16) == 0)
    assert pa_read_device_errors(reset=True) == 0


@pytest.mark.parametrize("graph", [False, True])
def test_prefill_step_never_reads_the_cache_before_the_write(graph):
    """pa_prefill_step's planner starts beside the KV-write kernel; the
    attention must still read the cache only after the write.  Before every
    one of 20 steps the new tokens' cache slots are poisoned with NaN (a
    kernel on the same stream): each step's output must equal the first one
    bit for bit, eagerly and replayed from a CUDA graph."""
    wl = synth.make_workload("qwen3_0p6b_chunked_prefill")
    run = GpuCase(wl)
    n = wl.num_new_tokens
    ref = run.step()[:n].clone()
    torch.cuda.synchronize()
    slots = run.bufs.slots[:n].clone()
    slots = slots[slots >= 0]
    rows = wl.num_kv_heads * wl.head_dim
    kc, vc = run.k_cache.view(-1, rows), run.v_cache.view(-1, rows)

    def body():
        kc.index_fill_(0, slots, float("nan"))
        vc.index_fill_(0, slots, float("nan"))
        run.step()

    if graph:
        body()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=s):
            body()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
    for _ in range(20):
        run.bufs.out.fill_(0)
        g.replay() if graph else body()
        torch.cuda.synchronize()
        assert torch.equal(run.bufs.out[:n].view(torch.int16), ref.view(torch.int16))
    assert pa_read_device_errors(reset=True) == 0


@pytest.mark.parametrize("planned", [True, False])
def test_prefill_step_with_a_padding_row_equals_the_separate_calls(planned):
    """A padding row (context length 0) inside pa_prefill_step: its tokens get
    position 0 and slot -1, its output rows stay untouched, no flag is raised,
    and everything equals the separate calls bit for bit."""
    spec = dict(kind="prefill", dtype="bf16", B=4, Hq=16, Hkv=8, hd=128, P=16, chunks=[40, 9, 130, 3],
                prefixes=[100, 0, 257, 31], norm=True, seed=91)
    wl = synth.make_workload(spec)
    runs = [GpuCase(wl, plan_prefill=planned), GpuCase(wl, plan_prefill=planned)]
    n = wl.num_new_tokens
    pad = 1
    outs = []
    for k, run in enumerate(runs):
        run.t["context_lens"][pad] = 0
        run.bufs.out.fill_(7.0)
        run.bufs.positions.fill_(-5)
        run.bufs.slots.fill_(-5)
        pa_read_device_errors(reset=True)
        outs.append(run.step() if k == 0 else _separate_calls(run))
        torch.cuda.synchronize()
        assert pa_read_device_errors(reset=True) == 0
    a, b = runs
    s0, s1 = int(wl.cu_seqlens_q[pad]), int(wl.cu_seqlens_q[pad + 1])
    assert torch.all(outs[0][s0:s1] == 7.0)
    assert torch.all(a.bufs.positions[s0:s1] == 0) and torch.all(a.bufs.slots[s0:s1] == -1)
    assert torch.equal(outs[0][:n].view(torch.int16), outs[1][:n].view(torch.int16))
    assert torch.equal(a.bufs.positions[:n], b.bufs.positions[:n])
    assert torch.equal(a.bufs.slots[:n], b.bufs.slots[:n])
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), b.v_cache.view(torch.int16))
