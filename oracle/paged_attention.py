"""Plain float64 CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` may import this module.  It shares no code with
the CUDA library (no kernels, headers, helpers or tables) and never consumes a
value produced by it.

What it computes, and where the pages define it:

* slot mapping -- nano-vLLM learning note, ``prepare_decode`` listing: a
  request's token at logical position ``pos`` lives in physical slot
  ``block_table[pos // page_size] * page_size + pos % page_size``; the
  ``prepare_prefill`` listing gives the new tokens' positions as
  ``range(num_cached, num_cached + num_scheduled)``.
* KV write -- nano-vLLM learning note, ``store_kvcache_kernel`` listing: row t
  of k / v is copied to flat slot ``slot_mapping[t]`` of k_cache / v_cache;
  ``-1`` means "store nothing".
* Q/K RMSNorm -- nano-vLLM learning note, ``RMSNorm.rms_forward`` listing:
  statistics in floating point, the normalised value cast back to the input
  dtype *before* the multiply by the weight.
* RoPE -- nano-vLLM learning note, ``apply_rotary_emb`` and ``inv_freq``
  listings: half-split (x1 = first half, x2 = second half),
  ``y1 = x1 cos - x2 sin``, ``y2 = x2 cos + x1 sin``, frequencies
  ``theta ** (-2i / rotary_dim)``; absolute positions (qwen-inference-lab
  README, feature list).
* Order of the per-token steps -- nano-vLLM learning note,
  ``Qwen3Attention.forward`` listing: q_norm / k_norm, then rotary, then
  attention; ``Attention.forward`` listing: store the new K/V first, then
  attend, reading K/V from the cache when block tables are present.
* Attention -- the textbook definition over pages gathered into contiguous K/V,
  the shape of the qwen-inference-lab README's own path (it copies a
  request's pages into one contiguous tensor and runs SDPA on it).  q-head h reads kv-head ``h // (Hq // Hkv)`` (the
  ``Qwen3Attention.forward`` listing views q as [-1, num_heads, hd] and k, v
  as [-1, num_kv_heads, hd]).  Prefill row i of a request whose chunk starts
  after ``prefix`` cached tokens sees keys ``0 .. prefix + i``.
* Split-KV merge -- partial softmax results over disjoint key ranges combined
  by their log-sum-exp; the exact identity
  ``softmax over a union = weighted sum of per-range softmaxes``.

Storage formats: fp32 values are float32 arrays; bf16 values are uint16 bit
patterns.  Every function widens to float64 exactly and narrows with round to
nearest, ties to even.
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np

# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------


def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even).

    bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and float32's
    exponent range; below 2**-126 the spacing stays at 2**-133.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # x = m * 2**e with 0.5 <= |m| < 1
    e = np.maximum(e, -125)                  # 2**-126 = 0.5 * 2**-125
    quantum = np.ldexp(1.0, e - 8)
    r = np.rint(x / quantum) * quantum       # np.rint rounds half to even
    big = np.abs(r) >= 2.0 ** 128
    if np.any(big):
        r = np.where(big, np.copysign(np.inf, x), r)
    return np.where(np.isfinite(x), r, x)


def round_to_dtype(x, dtype: str) -> np.ndarray:
    """Round float64 values to the storage dtype's value set ("f64" = no-op)."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f64":
        return x
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        return round_to_bf16(x)
    raise ValueError(dtype)


def widen(a, dtype: str) -> np.ndarray:
    """Storage values -> float64 (exact)."""
    if dtype == "bf16":
        bits = np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    return np.asarray(a).astype(np.float64)


def narrow(x, dtype: str) -> np.ndarray:
    """float64 -> storage values (round to nearest, ties to even)."""
    r = round_to_dtype(x, dtype)
    if dtype == "bf16":
        return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    if dtype == "f32":
        return r.astype(np.float32)
    return r


# ---------------------------------------------------------------------------
# slot mapping and the KV write
# ---------------------------------------------------------------------------


def slot_mapping(block_tables, context_lens, cu_seqlens_q, page_size: int):
    """Positions and physical slots of each request's new tokens.

    Request b holds ``context_lens[b]`` tokens after this step, the last
    ``n_b = cu_seqlens_q[b+1] - cu_seqlens_q[b]`` of which are new; its new
    tokens sit at positions ``context_lens[b] - n_b + j`` (nano-vLLM learning
    note, ``prepare_prefill``: ``range(start, end)``; ``prepare_decode``: the
    single new token is at ``len(seq) - 1``).  Each position's slot is the
    page from the block table times the page size plus the offset in the page
    (``prepare_decode``: ``block_table[-1] * block_size +
    last_block_num_tokens - 1``).
    """
    bt = np.asarray(block_tables)
    ctx = np.asarray(context_lens, dtype=np.int64)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    n = int(cu[-1])
    positions = np.empty(n, dtype=np.int64)
    slots = np.empty(n, dtype=np.int64)
    for b in range(len(ctx)):
        start_pos = int(ctx[b]) - int(cu[b + 1] - cu[b])
        for j, t in enumerate(range(int(cu[b]), int(cu[b + 1]))):
            pos = start_pos + j
            page = int(bt[b, pos // page_size])
            positions[t] = pos
            slots[t] = page * page_size + pos % page_size
    return positions, slots


def kv_write(k, v, slots, k_cache, v_cache) -> None:
    """Copy row t of k / v into flat slot ``slots[t]`` of the caches, in place.

    nano-vLLM learning note, ``store_kvcache_kernel`` listing: one program
    per token; a slot of -1 stores nothing; the row is ``num_kv_heads *
    head_dim`` elements.  The copy is bitwise.
    """
    row = k_cache.shape[-2] * k_cache.shape[-1]
    kc = k_cache.reshape(-1, row)
    vc = v_cache.reshape(-1, row)
    kr = np.asarray(k).reshape(len(slots), row)
    vr = np.asarray(v).reshape(len(slots), row)
    for t, s in enumerate(np.asarray(slots, dtype=np.int64)):
        if s == -1:
            continue
        kc[s] = kr[t]
        vc[s] = vr[t]


# ---------------------------------------------------------------------------
# per-token Q/K normalisation and rotation
# ---------------------------------------------------------------------------


def rms_norm(x, w, eps: float, dtype: str) -> np.ndarray:
    """RMSNorm over the last axis (nano-vLLM learning note, ``rms_forward``).

    ``r = 1 / sqrt(mean(x**2) + eps)``; ``y = round(round(x * r) * w)`` where
    ``round`` narrows to the storage dtype: the listing casts ``x * r`` back
    to the input dtype before ``mul_(weight)``, and a bf16 multiply rounds its
    result.  Arguments and result are float64 arrays holding dtype values.
    """
    x = np.asarray(x, dtype=np.float64)
    var = np.mean(x * x, axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(var + eps)
    return round_to_dtype(round_to_dtype(x * r, dtype) * np.asarray(w, dtype=np.float64), dtype)


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """``1 / theta ** (2i / head_dim)`` for i < head_dim / 2 (``inv_freq`` listing)."""
    i = np.arange(0, head_dim, 2, dtype=np.float64)
    return 1.0 / np.power(float(theta), i / head_dim)


def rope(x, positions, theta: float, dtype: str) -> np.ndarray:
    """Half-split rotary embedding at absolute positions (``apply_rotary_emb``).

    ``x``: float64 [n, heads, hd]; ``positions``: [n].  Angles and the rotation
    are evaluated in float64 and the result narrowed to the storage dtype, as
    the listing casts back with ``.to(x.dtype)``.
    """
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_inv_freq(hd, theta)[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., : hd // 2], x[..., hd // 2:]
    y = np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)
    return round_to_dtype(y, dtype)


def qk_norm_rope(q, k, q_norm_w, k_norm_w, positions, eps: float, theta: float, dtype: str):
    """q_norm / k_norm then rotary on the new tokens (``Qwen3Attention.forward``).

    Storage in, storage out: q [n, Hq, hd], k [n, Hkv, hd].  V is not touched
    by either step.
    """
    qn = rms_norm(widen(q, dtype), widen(q_norm_w, dtype), eps, dtype)
    kn = rms_norm(widen(k, dtype), widen(k_norm_w, dtype), eps, dtype)
    return (narrow(rope(qn, positions, theta, dtype), dtype),
            narrow(rope(kn, positions, theta, dtype), dtype))


# ---------------------------------------------------------------------------
# attention over gathered pages
# ---------------------------------------------------------------------------


def gather_kv(k_cache, v_cache, block_table_row, length: int, dtype: str):
    """Contiguous float64 K, V [length, Hkv, hd] of one request.

    Pages ``block_table_row[0], block_table_row[1], ...`` hold logical tokens
    ``0..P-1, P..2P-1, ...``; only the first ``length`` rows are read, so no
    unwritten slot is ever touched.
    """
    P = k_cache.shape[1]
    n_pages = (length + P - 1) // P
    pages = np.asarray(block_table_row[:n_pages], dtype=np.int64)
    K = k_cache[pages].reshape(n_pages * P, *k_cache.shape[2:])[:length]
    V = v_cache[pages].reshape(n_pages * P, *v_cache.shape[2:])[:length]
    return widen(K, dtype), widen(V, dtype)


def attend(q, K, V, positions, scale: float, return_probs: bool = False):
    """Softmax attention of query rows over contiguous keys, with GQA grouping.

    ``q``: float64 [n, Hq, hd]; ``K``, ``V``: float64 [L, Hkv, hd];
    ``positions``: [n], query row i sees keys ``j <= positions[i]``.
    Returns ``o`` [n, Hq, hd] and ``lse`` [n, Hq] (natural log of the softmax
    denominator including the max), plus the probabilities [n, Hq, L] if asked.
    """
    q = np.asarray(q, dtype=np.float64)
    n, Hq, hd = q.shape
    L, Hkv, _ = K.shape
    G = Hq // Hkv
    pos = np.asarray(positions, dtype=np.int64)
    hidden = np.arange(L)[None, :] > pos[:, None]
    o = np.empty((n, Hq, hd))
    lse = np.empty((n, Hq))
    probs = np.empty((n, Hq, L)) if return_probs else None
    for h in range(Hq):
        kv = h // G
        s = scale * (q[:, h, :] @ K[:, kv, :].T)
        s[hidden] = -np.inf
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        den = p.sum(axis=1, keepdims=True)
        p = p / den
        o[:, h, :] = p @ V[:, kv, :]
        lse[:, h] = m[:, 0] + np.log(den[:, 0])
        if return_probs:
            probs[:, h, :] = p
    if return_probs:
        return o, lse, probs
    return o, lse


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, dtype: str,
           requests: Optional[Sequence[int]] = None):
    """Decode attention: one query per request over all its ``context_lens[b]`` keys.

    ``q``: storage [B, Hq, hd].  Returns float64 o [len(requests), Hq, hd] and
    lse.  ``context_lens`` counts the token written this step (nano-vLLM
    learning note, ``prepare_decode``: ``context_lens.append(len(seq))``).
    """
    reqs = range(len(context_lens)) if requests is None else requests
    outs, lses = [], []
    for b in reqs:
        L = int(context_lens[b])
        K, V = gather_kv(k_cache, v_cache, block_tables[b], L, dtype)
        o, lse = attend(widen(q[b: b + 1], dtype), K, V, [L - 1], scale)
        outs.append(o[0])
        lses.append(lse[0])
    return np.stack(outs), np.stack(lses)


def prefill(q, cu_seqlens_q, k_cache, v_cache, block_tables, context_lens, scale: float,
            dtype: str, requests: Optional[Sequence[int]] = None):
    """Chunked-prefill attention of packed new tokens over prefix + causal chunk.

    ``q``: storage [sum n_b, Hq, hd] packed by ``cu_seqlens_q`` (qwen-engine
    README, flat varlen prefill).  Request b's chunk holds the last ``n_b`` of
    its ``context_lens[b]`` tokens; its row i sits at position
    ``context_lens[b] - n_b + i`` and sees keys up to that position, all read
    back from the cache (``Attention.forward``: ``k, v = k_cache, v_cache``
    when block tables are given).  Returns float64 o for the rows of the
    selected requests, in packed order, and their lse.
    """
    reqs = range(len(context_lens)) if requests is None else requests
    outs, lses = [], []
    for b in reqs:
        s0, s1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        if s1 == s0:
            continue
        L = int(context_lens[b])
        K, V = gather_kv(k_cache, v_cache, block_tables[b], L, dtype)
        positions = np.arange(L - (s1 - s0), L)
        o, lse = attend(widen(q[s0:s1], dtype), K, V, positions, scale)
        outs.append(o)
        lses.append(lse)
    if not outs:
        return np.zeros((0,) + tuple(q.shape[1:])), np.zeros((0, q.shape[1]))
    return np.concatenate(outs), np.concatenate(lses)


# ---------------------------------------------------------------------------
# split-KV partials and their log-sum-exp merge
# ---------------------------------------------------------------------------


def decode_partials(q_row, K, V, bounds: Sequence[Tuple[int, int]], scale: float):
    """Per-range softmax results of one decode query over key ranges ``bounds``.

    Returns o_parts [S, Hq, hd] (each normalised over its own range) and
    lse_parts [S, Hq].
    """
    o_parts, lse_parts = [], []
    for lo, hi in bounds:
        o, lse = attend(q_row[None], K[lo:hi], V[lo:hi], [hi - lo - 1], scale)
        o_parts.append(o[0])
        lse_parts.append(lse[0])
    return np.stack(o_parts), np.stack(lse_parts)


def merge_partials(o_parts, lse_parts):
    """Combine per-range results: weights ``exp(lse_s - max_s lse_s)``."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0, keepdims=True)
    w = np.exp(lse_parts - m)
    o = (w[..., None] * o_parts).sum(axis=0) / w.sum(axis=0)[..., None]
    lse = m[0] + np.log(w.sum(axis=0))
    return o, lse


# ---------------------------------------------------------------------------
# comparison rule
# ---------------------------------------------------------------------------

FP32_ATOL = 1e-5
BF16_ATOL = 2e-2
BF16_REL_OF_MAX = 1e-2


def within_tolerance(got, ref, dtype: str):
    """(ok, max_abs_err, bound): fp32 max|err| <= 1e-5; bf16 max|err| <= 2e-2
    and <= 1e-2 * max|ref|."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return True, 0.0, 0.0
    err = float(np.max(np.abs(got - ref)))
    if dtype == "f32":
        bound = FP32_ATOL
    else:
        bound = min(BF16_ATOL, BF16_REL_OF_MAX * float(np.max(np.abs(ref))))
    return bool(np.isfinite(err) and err <= bound), err, bound


def reference_step(wl, requests: Optional[Sequence[int]] = None, with_attention: bool = True):
    """One whole step of a workload, computed by the oracle from the seeded inputs.

    Builds the cache from the history rows with the oracle's own slot mapping
    and KV write, applies the step's own norm/rotation (if the workload has
    norm weights) and KV write, then attends.  Returns a dict with the caches,
    the new tokens' positions / slots, the q actually attended (storage) and
    the float64 outputs of the selected requests (None when
    ``with_attention`` is False).
    """
    dt = wl.dtype
    k_cache = wl.poison_storage(wl.cache_shape())
    v_cache = wl.poison_storage(wl.cache_shape())
    _, hist_slots = slot_mapping(wl.block_tables, wl.hist_lens, wl.cu_hist, wl.page_size)
    kv_write(wl.hist_k, wl.hist_v, hist_slots, k_cache, v_cache)
    positions, slots = slot_mapping(wl.block_tables, wl.context_lens, wl.cu_seqlens_q, wl.page_size)
    q, k = wl.q, wl.k_new
    if wl.q_norm_w is not None:
        q, k = qk_norm_rope(wl.q, wl.k_new, wl.q_norm_w, wl.k_norm_w, positions,
                            wl.eps, wl.rope_theta, dt)
    kv_write(k, wl.v_new, slots, k_cache, v_cache)
    if not with_attention:
        o = lse = None
    elif wl.kind == "decode":
        o, lse = decode(q, k_cache, v_cache, wl.block_tables, wl.context_lens, wl.scale, dt, requests)
    else:
        o, lse = prefill(q, wl.cu_seqlens_q, k_cache, v_cache, wl.block_tables, wl.context_lens,
                         wl.scale, dt, requests)
    return dict(k_cache=k_cache, v_cache=v_cache, positions=positions, slots=slots,
                q=q, k=k, o=o, lse=lse)

