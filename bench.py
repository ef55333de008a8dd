#!/usr/bin/env python3
"""Benchmark of libpagedattn on one GB300 (or N replicas, one per GPU).

A step is one pass of the attention hot path over one batch:
  decode (headline, the Qwen3-0.6B-shaped batch: 256 requests, 16 q / 8 kv
  heads, head_dim 128, page size 16, contexts 128..2048): split-KV decode
  attention with the slot mapping and KV write of the 256 new tokens folded
  in (pa_decode_kv_write) + merge;
  prefill (secondary): slot mapping, q/k RMSNorm + RoPE + KV write, chunked
  prefill attention over the paged prefix.
value = algorithmic HBM bytes of the decode step / step time (GB/s), summed
over ranks.  Inputs are synthetic and seeded (synth/), the KV cache (1.1 GB)
is larger than L2, so no L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
import os

# The CPU baseline is the float64 oracle with every core of this process's
# affinity available to BLAS; the thread count is set before numpy loads and
# recorded with the result.
HOST_CORES = len(os.sched_getaffinity(0))
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(HOST_CORES))
BLAS_THREADS = os.environ["OPENBLAS_NUM_THREADS"]

import argparse
import ctypes
import hashlib
import json
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from paged_kv_gqa_08_gb300 import PA_BF16, PA_F32, build as pa_build, cache_desc, load_library  # noqa: E402
from paged_kv_gqa_08_gb300 import pa_decode, pa_prefill_varlen, pa_read_device_errors  # noqa: E402
from paged_kv_gqa_08_gb300.step import alloc_step_buffers, write_rows  # noqa: E402

METRIC = "paged GQA decode HBM GB/s (% of peak) & attn tok/s; prefill TFLOP/s vs peak"
UNIT = "GB/s"
HEADLINE = "qwen3_0p6b_decode"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------
def decode_call_bytes(wl) -> int:
    """HBM bytes one pa_decode call must move: K and V of every context token,
    q and o, the used block-table entries and the context lengths."""
    e = wl.elem_bytes
    kv = int(wl.context_lens.astype(np.int64).sum()) * 2 * wl.num_kv_heads * wl.head_dim * e
    qo = 2 * wl.batch * wl.num_q_heads * wl.head_dim * e
    pages = int(((wl.context_lens.astype(np.int64) + wl.page_size - 1) // wl.page_size).sum())
    return kv + qo + 4 * pages + 4 * wl.batch


def kv_bytes(wl) -> int:
    return int(wl.context_lens.astype(np.int64).sum()) * 2 * wl.num_kv_heads * wl.head_dim * wl.elem_bytes


def write_bytes(wl) -> int:
    """Slot mapping + KV write (+ q/k norm-rope) of the step's new tokens."""
    n, e = wl.num_new_tokens, wl.elem_bytes
    row = wl.num_kv_heads * wl.head_dim * e
    b = 4 * n * row + 8 * n                              # read k, v; write k, v; read slots
    b += 4 * (2 * wl.batch + 1) + 4 * n + 12 * n         # metadata in, positions + slots out
    if wl.q_norm_w is not None:
        b += 2 * n * wl.num_q_heads * wl.head_dim * e     # read q, write q_out
    return b


def fused_write_bytes(wl) -> int:
    """The KV write inside pa_decode_kv_write: read the new k, v rows, write them
    into the cache, write the slot of each request."""
    row = wl.num_kv_heads * wl.head_dim * wl.elem_bytes
    return 4 * wl.batch * row + 8 * wl.batch


def prefill_flops(wl) -> int:
    """4 * head_dim * Hq * (unmasked query-key pairs): QK^T plus PV."""
    pairs = 0
    for pre, n in zip(wl.hist_lens.astype(np.int64), wl.new_lens.astype(np.int64)):
        pairs += n * pre + n * (n + 1) // 2
    return int(4 * wl.head_dim * wl.num_q_heads * pairs)


def prefill_call_bytes(wl) -> int:
    e = wl.elem_bytes
    return kv_bytes(wl) + 2 * wl.num_new_tokens * wl.num_q_heads * wl.head_dim * e


def describe(wl) -> str:
    lens = wl.context_lens
    if wl.kind == "decode":
        return (f"{wl.name}: {wl.batch} requests x 1 new token, {wl.num_q_heads} q / {wl.num_kv_heads} kv heads, "
                f"head_dim {wl.head_dim}, page {wl.page_size}, contexts {lens.min()}..{lens.max()}, {wl.dtype}")
    return (f"{wl.name}: {wl.batch} requests, chunks {wl.new_lens.tolist()}, prefixes "
            f"{wl.hist_lens.min()}..{wl.hist_lens.max()}, {wl.num_q_heads} q / {wl.num_kv_heads} kv heads, "
            f"head_dim {wl.head_dim}, page {wl.page_size}, {wl.dtype}")


# ---------------------------------------------------------------------------
# peaks, clocks, profiles
# ---------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


_REASONS = [(0x1, "gpu_idle"), (0x2, "applications_clocks_setting"), (0x4, "sw_power_cap"), (0x8, "hw_slowdown"),
            (0x10, "sync_boost"), (0x20, "sw_thermal_slowdown"), (0x40, "hw_thermal_slowdown"),
            (0x80, "hw_power_brake_slowdown"), (0x100, "display_clock_setting")]


class ClockSampler:
    """Samples the SM clock and clock-event reasons through NVML while running."""

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            ok = False
            try:
                bus = torch.cuda.get_device_properties(device_index)
                busid = f"{bus.pci_domain_id:08x}:{bus.pci_bus_id:02x}:{bus.pci_device_id:02x}.0".encode()
                ok = nvml.nvmlDeviceGetHandleByPciBusId_v2(busid, ctypes.byref(h)) == 0
            except Exception:
                ok = False
            if not ok and nvml.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(h)) != 0:
                return
            self._nvml, self._handle = nvml, h
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
        except OSError:
            self._nvml = None

    def _read(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, ctypes.byref(clk)) == 0:
            self.samples.append(int(clk.value))
        fn = getattr(self._nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self._nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        if fn(self._handle, ctypes.byref(rs)) == 0:
            self.reasons |= int(rs.value)

    def _run(self):
        while not self._stop.is_set():
            self._read()
            time.sleep(self.period)

    def __enter__(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            self._read()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"], "samples": 0}
        names = [n for bit, n in _REASONS if self.reasons & bit]
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(self.samples)}


def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_gqa_08_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(key: str, src_files) -> object:
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source is unchanged since it was captured; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[key]
        if e.get("source_sha256_16") != kernel_source_hash(src_files):
            return None
        return int(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# device setup and timing
# ---------------------------------------------------------------------------
class Device:
    def __init__(self, wl, dev, max_ctas=0, fused=False):
        self.wl = wl
        self.dev = dev
        self.fused = fused and wl.kind == "decode"   # KV write fused into decode (pa_decode_kv_write)
        self.t = synth.to_torch(wl, dev)
        self.desc = cache_desc(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, wl.num_pages,
                               PA_F32 if wl.dtype == "f32" else PA_BF16)
        dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
        self.k_cache = torch.full(wl.cache_shape(), float("nan"), dtype=dt, device=dev)
        self.v_cache = torch.full(wl.cache_shape(), float("nan"), dtype=dt, device=dev)
        nh = max(int(wl.cu_hist[-1]), 1)
        write_rows(self.desc, self.t["hist_k"], self.t["hist_v"], self.t["cu_hist"], self.t["hist_lens"],
                   self.t["block_tables"], wl.max_pages_per_seq, torch.empty(nh, dtype=torch.int32, device=dev),
                   torch.empty(nh, dtype=torch.int64, device=dev), self.k_cache, self.v_cache)
        self.t["hist_k"] = self.t["hist_v"] = None
        self.bufs = alloc_step_buffers(self.desc, wl.kind, wl.num_new_tokens, wl.batch, wl.max_context_len, dev,
                                       norm=wl.q_norm_w is not None, max_ctas=max_ctas,
                                       max_seqlen_q=max(wl.max_new_len, 1))
        torch.cuda.synchronize()

    def write_part(self):
        """Slot mapping + (norm/rope +) KV write: everything before attention."""
        wl, t, b = self.wl, self.t, self.bufs
        from paged_kv_gqa_08_gb300 import pa_kv_write, pa_prefill_qk_norm_rope_kv_write, pa_slot_mapping
        n = wl.num_new_tokens
        if self.fused:
            return
        if wl.q_norm_w is not None:
            # slot mapping, q/k norm and rotary, KV write: one kernel
            q = t["q"]
            pa_prefill_qk_norm_rope_kv_write(self.desc, q, q.stride(0), t["k_new"], t["k_new"].stride(0), t["v_new"],
                                             t["v_new"].stride(0), n, t["cu_seqlens_q"], wl.batch, t["context_lens"],
                                             t["block_tables"], wl.max_pages_per_seq, t["q_norm_w"], t["k_norm_w"],
                                             wl.eps, wl.rope_theta, b.q_out, self.k_cache, self.v_cache,
                                             b.positions, b.slots)
        else:
            pa_slot_mapping(self.desc, wl.batch, t["cu_seqlens_q"], t["context_lens"], t["block_tables"],
                            wl.max_pages_per_seq, n, b.positions, b.slots)
            pa_kv_write(self.desc, t["k_new"], t["k_new"].stride(0), t["v_new"], t["v_new"].stride(0), n, b.slots,
                        self.k_cache, self.v_cache)

    def prefill_step(self):
        """The whole prefill step in one call (pa_prefill_step: the write part,
        then the planned attention, its planner beside the write kernel)."""
        wl, t, b = self.wl, self.t, self.bufs
        from paged_kv_gqa_08_gb300 import pa_prefill_step
        q = t["q"]
        pa_prefill_step(self.desc, q, q.stride(0), t["k_new"], t["k_new"].stride(0), t["v_new"], t["v_new"].stride(0),
                        wl.num_new_tokens, t["cu_seqlens_q"], wl.batch, wl.max_new_len, t["context_lens"],
                        wl.max_context_len, t["block_tables"], wl.max_pages_per_seq, t["q_norm_w"], t["k_norm_w"],
                        wl.eps or 0.0, wl.rope_theta or 0.0, wl.scale, b.q_out, self.k_cache, self.v_cache,
                        b.positions, b.slots, b.out, b.workspace)

    def attn_part(self):
        wl, t, b = self.wl, self.t, self.bufs
        q = b.q_out if wl.q_norm_w is not None else t["q"]
        if self.fused:
            from paged_kv_gqa_08_gb300 import pa_decode_kv_write
            row = wl.num_kv_heads * wl.head_dim
            pa_decode_kv_write(self.desc, q, t["k_new"], row, t["v_new"], row, wl.batch, self.k_cache, self.v_cache,
                               t["block_tables"], wl.max_pages_per_seq, t["context_lens"], wl.max_context_len,
                               wl.scale, b.max_ctas, b.slots, b.out, b.workspace)
        elif wl.kind == "decode":
            pa_decode(self.desc, q, wl.batch, self.k_cache, self.v_cache, t["block_tables"], wl.max_pages_per_seq,
                      t["context_lens"], wl.max_context_len, wl.scale, b.max_ctas, b.out, b.workspace)
        else:
            pa_prefill_varlen(self.desc, q, t["cu_seqlens_q"], wl.batch, wl.max_new_len, wl.num_new_tokens,
                              self.k_cache, self.v_cache, t["block_tables"], wl.max_pages_per_seq,
                              t["context_lens"], wl.max_context_len, wl.scale, b.out, b.workspace)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest of the ranks' values (the timing rule: the slowest rank)."""
    if world == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, elapsed_ms_max: float, world: int) -> float:
    """Units per second of the whole job: every rank's units over the slowest rank's time."""
    return world * units_per_rank / (elapsed_ms_max * 1e-3)


def time_device_steps(d: Device, steps: int, warmup: int, world: int, clocks: ClockSampler = None):
    """Warm up, then time exactly `steps` steps; per-step events split the
    write part from the attention call."""
    for _ in range(warmup):
        d.write_part()
        d.attn_part()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    ctx = clocks if clocks is not None else _Null()
    with ctx:
        start.record()
        for k in range(steps):
            ev[k][0].record()
            d.write_part()
            ev[k][1].record()
            d.attn_part()
            ev[k][2].record()
        end.record()
        torch.cuda.synchronize()
    barrier(world)
    total_ms = start.elapsed_time(end)
    attn_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    write_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    return max_over_ranks(total_ms, world), attn_ms, write_ms


def capture_graph(body):
    """Capture `body` (after one eager run, so every plan is cached) into a CUDA graph."""
    body()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        body()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def time_graph_steps(d: Device, steps: int, warmup: int, world: int, clocks=None):
    """The whole step as one CUDA graph, replayed back to back."""
    g = capture_graph(lambda: (d.write_part(), d.attn_part()))
    for _ in range(warmup):
        g.replay()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    ctx = clocks if clocks is not None else _Null()
    with ctx:
        start.record()
        for _ in range(steps):
            g.replay()
        end.record()
        torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(start.elapsed_time(end), world)


def flush_l2(buf: torch.Tensor) -> None:
    """Overwrite a buffer larger than L2, then read it back, so that L2 holds
    none of the step's data and no dirty lines whose write-back would land in
    the timed region."""
    buf.zero_()
    buf.view(torch.int64).sum()


def time_graph_parts(d: Device, steps: int, warmup: int, flush=None, warm_s: float = 0.0):
    """The write part and the attention call as two CUDA graphs, L2 flushed
    before every step when `flush` (a buffer larger than L2) is given; CUDA
    events around each replay.  Warm-up: `warmup` steps, continued until
    `warm_s` seconds of replays have passed.  Returns mean (step, write,
    attention) ms."""
    gw = capture_graph(d.write_part)
    ga = capture_graph(d.attn_part)

    def warm_step():
        if flush is not None:
            flush_l2(flush)
        gw.replay()
        ga.replay()

    for _ in range(warmup):
        warm_step()
    torch.cuda.synchronize()
    t_end = time.perf_counter() + warm_s
    while time.perf_counter() < t_end:
        for _ in range(10):
            warm_step()
        torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    torch.cuda.synchronize()
    for k in range(steps):
        if flush is not None:
            flush_l2(flush)
        ev[k][0].record()
        gw.replay()
        ev[k][1].record()
        ga.replay()
        ev[k][2].record()
    torch.cuda.synchronize()
    write_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    attn_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    return write_ms + attn_ms, write_ms, attn_ms


def time_graph_whole(body, steps: int, warmup: int, flush=None):
    """`body` as one CUDA graph, L2 flushed before every replay when `flush` is
    given; CUDA events around each replay.  Returns the mean ms."""
    g = capture_graph(body)
    for _ in range(warmup):
        if flush is not None:
            flush_l2(flush)
        g.replay()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for k in range(steps):
        if flush is not None:
            flush_l2(flush)
        ev[k][0].record()
        g.replay()
        ev[k][1].record()
    torch.cuda.synchronize()
    return sum(e[0].elapsed_time(e[1]) for e in ev) / steps


def step_percentiles(d: Device, n: int = 100):
    """p10 / p50 / p90 of single graph-replayed steps (CUDA events around each
    replay), taken after the timed region."""
    g = capture_graph(lambda: (d.write_part(), d.attn_part()))
    for _ in range(5):
        g.replay()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        g.replay()
        b.record()
    torch.cuda.synchronize()
    t = np.sort(np.array([a.elapsed_time(b) for a, b in ev]))
    return {"p10": float(t[int(0.1 * (n - 1))]), "p50": float(t[int(0.5 * (n - 1))]), "p90": float(t[int(0.9 * (n - 1))]),
            "replays": n}


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def time_e2e(d: Device, steps: int, warmup: int, world: int):
    """Same step through host buffers.  Every step moves its inputs from pinned
    host memory to the GPU and its output back: the metadata by one
    host-to-device copy (one pinned buffer of 256-byte aligned views, mirrored
    on the device), while q and the new K / V rows are read and the output
    written by the kernels themselves in pinned host memory (mapped into the
    device's address space), so those transfers overlap the KV-cache streaming.
    Returns (ms for all steps, h2d bytes per step, d2h bytes per step, whether
    the host-side output equals the device-side one)."""
    wl, t = d.wl, d.t
    dev_out = d.bufs.out.clone()             # the device-buffer result of the same inputs
    attn_ref = d.bufs.out
    names = ["context_lens", "cu_seqlens_q", "block_tables"]
    mapped = ["q", "k_new", "v_new"]
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += (t[k].numel() * t[k].element_size() + 255) // 256 * 256
    dev_buf = torch.empty(total, dtype=torch.uint8, device=t["q"].device)
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    saved = {k: t[k] for k in names + mapped}
    for k in names:
        nb = t[k].numel() * t[k].element_size()
        view = dev_buf[offs[k]:offs[k] + nb].view(t[k].dtype).view(t[k].shape)
        view.copy_(t[k])
        host_buf[offs[k]:offs[k] + nb].copy_(t[k].contiguous().view(-1).view(torch.uint8).cpu())
        t[k] = view
    for k in mapped:
        t[k] = t[k].cpu().pin_memory()
    n = wl.num_new_tokens
    out_host = torch.empty(tuple(d.bufs.out.shape), dtype=d.bufs.out.dtype).pin_memory()
    d.bufs.out = out_host
    h2d = sum(saved[k].numel() * saved[k].element_size() for k in names + mapped)
    d2h = out_host[:n].numel() * out_host.element_size()

    def body():
        dev_buf.copy_(host_buf, non_blocking=True)
        d.write_part()
        d.attn_part()

    # the copy in, the step writing its output to the host: one graph launch
    # and one host sync per step
    g = capture_graph(body)

    def one():
        g.replay()
        torch.cuda.current_stream().synchronize()

    for _ in range(warmup):
        one()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    el = time.perf_counter() - t0
    barrier(world)
    same = bool(torch.equal(out_host[:n], dev_out[:n].cpu()))
    d.bufs.out = attn_ref
    t.update(saved)
    return max_over_ranks(el * 1e3, world), h2d, d2h, same


# ---------------------------------------------------------------------------
# the float64 oracle as the CPU baseline / reference arm
# ---------------------------------------------------------------------------
def oracle_setup(wl):
    import oracle
    k_cache = wl.poison_storage(wl.cache_shape())
    v_cache = wl.poison_storage(wl.cache_shape())
    _, hist_slots = oracle.slot_mapping(wl.block_tables, wl.hist_lens, wl.cu_hist, wl.page_size)
    oracle.kv_write(wl.hist_k, wl.hist_v, hist_slots, k_cache, v_cache)
    return k_cache, v_cache


def oracle_step(wl, k_cache, v_cache, reqs):
    """The oracle's decode step for the requests `reqs`: slots, KV write, attention."""
    import oracle
    _, slots = oracle.slot_mapping(wl.block_tables, wl.context_lens, wl.cu_seqlens_q, wl.page_size)
    r = np.asarray(reqs)
    oracle.kv_write(wl.k_new[r], wl.v_new[r], slots[r], k_cache, v_cache)
    oracle.decode(wl.q, k_cache, v_cache, wl.block_tables, wl.context_lens, wl.scale, wl.dtype, requests=reqs)


def sample_bytes(wl, reqs) -> int:
    e = wl.elem_bytes
    sub = wl.context_lens[np.asarray(reqs)].astype(np.int64)
    row = wl.num_kv_heads * wl.head_dim * e
    return int(sub.sum()) * 2 * row + len(reqs) * (2 * wl.num_q_heads * wl.head_dim * e + 4 * row)


def cpu_baseline(wl, budget_s: float = 15.0):
    k_cache, v_cache = oracle_setup(wl)
    reqs = list(range(wl.batch))
    done_bytes, passes = 0, 0
    t0 = time.perf_counter()
    while True:
        oracle_step(wl, k_cache, v_cache, reqs)
        done_bytes += sample_bytes(wl, reqs)
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s or passes >= 3:
            break
    return {"value": done_bytes / el / 1e9, "unit": UNIT, "cores": HOST_CORES, "kind": "oracle",
            "blas_threads": BLAS_THREADS,
            "sample": f"{passes} pass(es) of the float64 oracle's decode step (slot mapping, KV write, "
                      f"attention) over all {wl.batch} requests of {wl.name}, {HOST_CORES} host cores available "
                      f"to BLAS (OPENBLAS/OMP threads {BLAS_THREADS}), {el:.1f} s"}


def headline_config(wl, world: int) -> dict:
    """The headline workload's config, the same on both arms."""
    return {"workload": describe(wl), "step": "slot mapping and KV write fused into split-KV decode "
            "(pa_decode_kv_write) + LSE merge, launched as one CUDA graph",
            "global_batch": world * wl.batch, "kv_bytes_per_step": kv_bytes(wl),
            "algorithmic_bytes_per_step": decode_call_bytes(wl) + fused_write_bytes(wl),
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (KV cache 1.1 GB > 129 MB L2); no flush"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = synth.make_workload(HEADLINE)
    k_cache, v_cache = oracle_setup(wl)
    # size each step's sample so the whole run stays within about two minutes
    t0 = time.perf_counter()
    oracle_step(wl, k_cache, v_cache, [0])
    one = max(time.perf_counter() - t0, 1e-3)
    per_step = 120.0 / max(1, args.steps + args.warmup)
    n_req = int(max(1, min(wl.batch, per_step / one)))
    rng = np.random.default_rng(123)
    for _ in range(args.warmup):
        oracle_step(wl, k_cache, v_cache, sorted(rng.choice(wl.batch, n_req, replace=False).tolist()))
    tot_bytes = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        reqs = sorted(rng.choice(wl.batch, n_req, replace=False).tolist())
        oracle_step(wl, k_cache, v_cache, reqs)
        tot_bytes += sample_bytes(wl, reqs)
    el = time.perf_counter() - t0
    value = tot_bytes / el / 1e9
    sample = (f"each step: {n_req} of the {wl.batch} requests of {wl.name} (random) through the float64 oracle "
              f"(slot mapping, KV write, attention), {HOST_CORES} host "
              f"cores available to BLAS (OPENBLAS/OMP threads {BLAS_THREADS})")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, synth/)",
            "config": headline_config(wl, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": HOST_CORES, "kind": "oracle",
                             "blas_threads": BLAS_THREADS, "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def run_case(spec: str):
    """Profiling helper: set up the first B requests of a workload and run three
    steps through the C ABI (no timing), e.g. --case decode:qwen3_8b_decode:16;
    kind "fused" runs the decode step as pa_decode_kv_write, a prefill step is
    one pa_prefill_step call."""
    kind, name, nreq = spec.split(":")
    nreq = int(nreq)
    fused = kind == "fused"
    if fused:
        kind = "decode"
    c = synth.CONFIGS[name]
    if nreq == c["B"]:
        wl = synth.make_workload(name)
    elif kind == "prefill":
        extra = {"prefixes": c["prefixes"][:nreq]} if "prefixes" in c else {}
        wl = synth.make_workload(name, B=nreq, chunks=c["chunks"][:nreq], **extra)
    else:
        wl = synth.make_workload(name, B=nreq)
    pa_build.build()
    load_library()
    d = Device(wl, "cuda:0", fused=fused)
    for _ in range(3):
        if wl.kind == "prefill":
            d.prefill_step()
        else:
            d.write_part()
            d.attn_part()
    torch.cuda.synchronize()
    print(json.dumps({"case": spec, "workload": describe(wl), "kv_bytes": kv_bytes(wl),
                      "decode_bytes": decode_call_bytes(wl) if wl.kind == "decode" else None,
                      "prefill_flops": prefill_flops(wl) if wl.kind == "prefill" else None}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="headline only (no prefill / other configs)")
    ap.add_argument("--case", help="profiling helper KIND:CONFIG:B (see run_case); runs 3 steps and exits")
    args = ap.parse_args()
    if args.case:
        run_case(args.case)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, rank, world)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    pa_build.build()
    load_library()
    pa_read_device_errors(reset=True)
    hbm_peak, tc_peak, tc_sustained, peak_src = load_peaks()

    # ---------------- headline: decode step ----------------
    wl = synth.make_workload(HEADLINE)
    # the same step with separate slot-mapping / KV-write / decode calls, for comparison
    du = Device(wl, dev)
    unfused_ms = time_graph_steps(du, args.steps, args.warmup, world) / args.steps
    del du
    torch.cuda.empty_cache()
    d = Device(wl, dev, fused=True)
    clocks = ClockSampler(local)
    # per-call CUDA events (eager launches) give the kernel-level roofline numbers
    eager_total_ms, attn_ms, write_ms = time_device_steps(d, args.steps, args.warmup, world)
    # the timed steps: the whole step replayed as one CUDA graph
    total_ms = time_graph_steps(d, args.steps, args.warmup, world, clocks)
    ms = total_ms / args.steps
    step_bytes = decode_call_bytes(wl) + fused_write_bytes(wl)
    value = whole_job_rate(step_bytes, ms, world) / 1e9
    tok_s = whole_job_rate(wl.batch, ms, world)
    dec_bytes = step_bytes
    achieved = dec_bytes / (attn_ms * 1e-3) / 1e9
    traffic = profiled_traffic("decode_qwen3_0p6b", ["decode.cu", "pa_common.cuh"])
    e2e_ms, h2d, d2h, e2e_same = time_e2e(d, max(20, args.steps // 5), args.warmup, world)
    e2e_step_ms = e2e_ms / max(20, args.steps // 5)
    from paged_kv_gqa_08_gb300 import pa_decode_plan_info
    n_parts, _ = pa_decode_plan_info(d.desc, wl.batch, wl.max_context_len, 0)
    # per step: the split-KV decode with the KV write, the merge (if split), and a
    # plan kernel before them beyond 512 requests (include/pagedattn.h, pa_decode)
    launches = args.steps * (1 + (1 if n_parts > 1 else 0) + (1 if wl.batch > 512 else 0))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "accumulate": "f32", "data": "synthetic (seeded, synth/)",
        "config": headline_config(wl, world),
        "attn_tok_per_s": tok_s,
        "hbm_frac_of_step": value / world / hbm_peak,
        "roofline": {"kernel": "pa_decode_kv_write (split-KV decode with the KV write, planned in-kernel, + merge)",
                     "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "traffic": traffic, "peak_source": f"hbm_gbs of {peak_src}",
                     "algorithmic_bytes_per_launch": dec_bytes, "launch_ms": attn_ms},
        "write_part_ms": write_ms,
        "eager_ms_per_step": eager_total_ms / args.steps,
        "unfused_ms_per_step": unfused_ms,
        "e2e": {"value": world * step_bytes / (e2e_step_ms * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_step_ms,
                "transfers": "metadata by one pinned host-to-device copy per step; q and the new K/V rows "
                             "read and the output written by the kernels in pinned host memory",
                "output_matches_device_run": e2e_same},
        "gpu_launches": launches,
        "decode_partitions": n_parts,
        "clocks": clocks.summary(),
        "step_ms_percentiles": step_percentiles(d),
    }
    del d
    torch.cuda.empty_cache()

    # ---------------- secondary: prefill and the other decode shapes ----------------
    if not args.no_extra:
        extra = {"timing": "each config's KV-write part and attention call replayed as two CUDA graphs with CUDA "
                           "events around each replay, after at least 0.2 s of warm-up replays (the GPU idles "
                           "while a config's inputs are generated on the host); prefill configs also as the whole "
                           "step (pa_prefill_step) in one graph, which is their ms_per_step; prefill configs (KV "
                           "fits in L2): L2 flushed before every step (512 MiB overwritten, then read back); "
                           "decode configs with KV > 512 MiB: no flush"}
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        for name, steps in (("qwen3_0p6b_chunked_prefill", 100), ("prefill_2k", 20)):
            w = synth.make_workload(name)
            dd = Device(w, dev)
            parts_ms, w_ms, a_ms = time_graph_parts(dd, steps, 5, flush, warm_s=0.2)
            step_ms = time_graph_whole(dd.prefill_step, steps, 5, flush)
            fl = prefill_flops(w)
            tflops = fl / (a_ms * 1e-3) / 1e12
            rt = max(fl / (tc_peak * 1e12), prefill_call_bytes(w) / (hbm_peak * 1e9))
            extra[name] = {"workload": describe(w), "ms_per_step": step_ms,
                           "step_launch": "pa_prefill_step as one CUDA graph (write kernel; planner beside it; "
                                          "attention; merge)",
                           "parts_ms_per_step": parts_ms, "prefill_ms": a_ms,
                           "launch": "planned (pa_prefill_varlen with workspace: plan, attention, merge)",
                           "write_ms": w_ms, "flops": fl, "tflops": tflops, "tok_per_s": w.num_new_tokens / (step_ms * 1e-3),
                           "roofline": {"bound": "tensor", "achieved": tflops, "peak": tc_peak, "unit": "TFLOP/s",
                                        "frac": tflops / tc_peak, "peak_source": f"bf16_tflops of {peak_src}",
                                        "roofline_ms": rt * 1e3, "frac_of_roofline_time": rt * 1e3 / a_ms}}
            del dd
            torch.cuda.empty_cache()
        for name in ("qwen3_8b_decode", "long_context_decode", "tiny_fp32_decode"):
            w = synth.make_workload(name)
            dd = Device(w, dev)
            step_ms, w_ms, a_ms = time_graph_parts(dd, 100, 5, None if kv_bytes(w) > (512 << 20) else flush,
                                                   warm_s=0.2)
            b = decode_call_bytes(w)
            extra[name] = {"workload": describe(w), "ms_per_step": step_ms, "decode_ms": a_ms, "write_ms": w_ms,
                           "decode_gbs": b / (a_ms * 1e-3) / 1e9, "hbm_frac": b / (a_ms * 1e-3) / 1e9 / hbm_peak,
                           "attn_tok_per_s": w.batch / (step_ms * 1e-3)}
            del dd
            torch.cuda.empty_cache()
        del flush
        line["secondary"] = extra
    line["device_error_flags"] = pa_read_device_errors(reset=True)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(synth.make_workload(HEADLINE))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
