"""Device-side setup shared by the GPU parity tests.

Uploads a seeded workload, fills a NaN-poisoned cache with the workload's
already-cached rows through the library (slot mapping + KV write), and runs
one step through the C ABI.  Nothing here computes attention.
"""
from __future__ import annotations

import numpy as np
import torch

import synth
from paged_kv_gqa_08_gb300 import PA_BF16, PA_F32, cache_desc
from paged_kv_gqa_08_gb300.step import alloc_step_buffers, run_step, write_rows


def torch_dtype(wl) -> torch.dtype:
    return torch.float32 if wl.dtype == "f32" else torch.bfloat16


def desc_of(wl):
    return cache_desc(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, wl.num_pages,
                      PA_F32 if wl.dtype == "f32" else PA_BF16)


def storage(t: torch.Tensor) -> np.ndarray:
    """Tensor -> numpy storage format of the oracle (bf16 as uint16 bits)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class GpuCase:
    """All device state of one workload."""

    def __init__(self, wl, device: str = "cuda", max_ctas: int = 0, cache_fill: float = float("nan"),
                 plan_prefill: bool = True):
        self.wl = wl
        self.device = device
        self.t = synth.to_torch(wl, device)
        self.desc = desc_of(wl)
        dt = torch_dtype(wl)
        self.k_cache = torch.full(wl.cache_shape(), cache_fill, dtype=dt, device=device)
        self.v_cache = torch.full(wl.cache_shape(), cache_fill, dtype=dt, device=device)
        nh = int(wl.cu_hist[-1])
        self.hist_pos = torch.empty(max(nh, 1), dtype=torch.int32, device=device)
        self.hist_slots = torch.empty(max(nh, 1), dtype=torch.int64, device=device)
        write_rows(self.desc, self.t["hist_k"], self.t["hist_v"], self.t["cu_hist"], self.t["hist_lens"],
                   self.t["block_tables"], wl.max_pages_per_seq, self.hist_pos, self.hist_slots,
                   self.k_cache, self.v_cache)
        self.bufs = alloc_step_buffers(self.desc, wl.kind, wl.num_new_tokens, wl.batch,
                                       max(wl.max_context_len, 1), device, norm=wl.q_norm_w is not None,
                                       max_ctas=max_ctas, max_seqlen_q=max(wl.max_new_len, 1),
                                       plan_prefill=plan_prefill)

    def step(self) -> torch.Tensor:
        wl, t = self.wl, self.t
        return run_step(self.desc, wl.kind, self.bufs, t["q"], t["k_new"], t["v_new"], t["cu_seqlens_q"],
                        t["context_lens"], t["block_tables"], self.k_cache, self.v_cache, wl.scale,
                        wl.max_pages_per_seq, max(wl.max_context_len, 1), max(wl.max_new_len, 1),
                        t["q_norm_w"], t["k_norm_w"], wl.eps or 0.0, wl.rope_theta or 0.0)
