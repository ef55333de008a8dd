"""One attention-layer step over a paged KV cache, through the C ABI.

The order is the nano-vLLM learning note's (Qwen3Attention.forward and
Attention.forward listings): positions and slots of the step's new tokens,
optional per-head q/k RMSNorm + rotary, the KV write, then decode or
chunked-prefill attention over the cache.  This module only allocates buffers
and sequences calls; every value is computed by libpagedattn's kernels.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

from . import (pa_decode, pa_decode_workspace_size, pa_kv_write, pa_prefill_qk_norm_rope_kv_write, pa_prefill_step,
               pa_prefill_workspace_size, pa_slot_mapping)


@dataclasses.dataclass
class StepBuffers:
    positions: torch.Tensor            # int32 [N]
    slots: torch.Tensor                # int64 [N]
    out: torch.Tensor                  # [N, Hq, hd]
    q_out: Optional[torch.Tensor]      # [N, Hq, hd] normed + rotated q (when norm weights are used)
    workspace: Optional[torch.Tensor]  # decode split-KV / planned-prefill workspace (bytes)
    max_ctas: int = 0


def torch_dtype(desc) -> torch.dtype:
    return torch.float32 if desc.dtype == 0 else torch.bfloat16


def alloc_step_buffers(desc, kind: str, num_tokens: int, batch: int, max_context_len: int, device,
                       norm: bool = False, max_ctas: int = 0, max_seqlen_q: Optional[int] = None,
                       plan_prefill: bool = True) -> StepBuffers:
    """Buffers of one step.  A prefill step gets the planned-launch workspace
    unless ``plan_prefill`` is False (or the shape is never planned); it is
    sized for chunks up to ``max_seqlen_q`` tokens (default: ``num_tokens``)."""
    dt = torch_dtype(desc)
    n = max(num_tokens, 1)
    positions = torch.empty(n, dtype=torch.int32, device=device)
    slots = torch.empty(n, dtype=torch.int64, device=device)
    out = torch.empty(n, desc.num_q_heads, desc.head_dim, dtype=dt, device=device)
    q_out = torch.empty_like(out) if norm else None
    ws = None
    if kind == "decode":
        nbytes = pa_decode_workspace_size(desc, batch, max_context_len, max_ctas)
        if nbytes == 0:
            raise RuntimeError("pa_decode_workspace_size returned 0 (unsupported shape or no device)")
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    elif plan_prefill and num_tokens > 0:
        nbytes = pa_prefill_workspace_size(desc, batch, max_seqlen_q or num_tokens, num_tokens, max_context_len)
        if nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return StepBuffers(positions, slots, out, q_out, ws, max_ctas)


def write_rows(desc, k_rows, v_rows, cu_rows, lens, block_tables, max_pages_per_seq, bufs_positions, bufs_slots,
               k_cache, v_cache, stream=None):
    """Store already-computed K/V rows (the last ``cu_rows`` segment of each of
    ``lens[b]`` tokens) into their slots: slot mapping then KV write."""
    n = k_rows.shape[0]
    batch = lens.shape[0]
    if n == 0:
        return
    pa_slot_mapping(desc, batch, cu_rows, lens, block_tables, max_pages_per_seq, n, bufs_positions, bufs_slots,
                    stream)
    row = desc.num_kv_heads * desc.head_dim
    pa_kv_write(desc, k_rows, row, v_rows, row, n, bufs_slots, k_cache, v_cache, stream)


def run_step(desc, kind: str, bufs: StepBuffers, q, k, v, cu_seqlens_q, context_lens, block_tables,
             k_cache, v_cache, scale: float, max_pages_per_seq: int, max_context_len: int, max_seqlen_q: int,
             q_norm_w=None, k_norm_w=None, eps: float = 0.0, rope_theta: float = 0.0, stream=None):
    """Run one step; returns ``bufs.out`` (the attention output of the new tokens)."""
    n = q.shape[0]
    batch = context_lens.shape[0]
    if kind != "decode":
        # the write part and the attention in one call, whose attention planner
        # runs beside the write kernel
        pa_prefill_step(desc, q, q.stride(0), k, k.stride(0), v, v.stride(0), n, cu_seqlens_q, batch, max_seqlen_q,
                        context_lens, max_context_len, block_tables, max_pages_per_seq, q_norm_w, k_norm_w, eps,
                        rope_theta, scale, bufs.q_out, k_cache, v_cache, bufs.positions, bufs.slots, bufs.out,
                        bufs.workspace, stream=stream)
        return bufs.out
    if q_norm_w is not None:
        # slot mapping, norm, rotary and KV write in one kernel
        pa_prefill_qk_norm_rope_kv_write(desc, q, q.stride(0), k, k.stride(0), v, v.stride(0), n, cu_seqlens_q,
                                         batch, context_lens, block_tables, max_pages_per_seq, q_norm_w, k_norm_w,
                                         eps, rope_theta, bufs.q_out, k_cache, v_cache, bufs.positions, bufs.slots,
                                         stream)
        qa = bufs.q_out
    else:
        pa_slot_mapping(desc, batch, cu_seqlens_q, context_lens, block_tables, max_pages_per_seq, n, bufs.positions,
                        bufs.slots, stream)
        pa_kv_write(desc, k, k.stride(0), v, v.stride(0), n, bufs.slots, k_cache, v_cache, stream)
        qa = q
    pa_decode(desc, qa, batch, k_cache, v_cache, block_tables, max_pages_per_seq, context_lens, max_context_len,
              scale, bufs.max_ctas, bufs.out, bufs.workspace, None, stream)
    return bufs.out
