"""Seeded synthetic inputs shaped like the Qwen3 serving workloads on the pages.

The pages (the nano-vLLM learning note, the qwen-engine and qwen-inference-lab
READMEs) serve Qwen3-0.6B and Qwen3-8B; the only model facts the attention path
needs are head counts and head_dim.  No trained weights, prompts or datasets are
involved: every value here is drawn from ``numpy.random.default_rng(seed)``.

Draw order (fixed, so a config and a seed pin every value):
  1. context / chunk / prefix lengths
  2. the physical page permutation
  3. the already-cached ("history") K, then V, ~ N(0,1)
  4. this step's new k, then v, ~ N(0,1)
  5. q ~ N(0,1)
  6. the q-norm then k-norm weights, 1 + 0.1 N(0,1) (configs that norm only)

Floating values are cast once to the config dtype; those exact values feed both
the CUDA path and the oracle.  bf16 values are carried as uint16 bit patterns,
fp32 values as float32.

Layout decisions made here are the page allocator's, not the attention
method's: request b owns ceil(context_len_b / page_size) pages, taken in logical
order from a seeded permutation of the page ids; unused block-table entries and
unused pages point at / hold poison (NaN), and the last page id is a dedicated
poison page.  Nothing in this module computes a slot, a norm, a rotation or a
softmax.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import math
import os
from typing import Optional

import numpy as np

BF16_NAN_BITS = np.uint16(0x7FC0)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bits."""
    u = np.array(x, dtype=np.float32, copy=True).view(np.uint32)
    bias = u >> np.uint32(16)
    bias &= np.uint32(1)
    bias += np.uint32(0x7FFF)
    u += bias
    u >>= np.uint32(16)
    return u.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_storage(rng: np.random.Generator, shape, dtype: str, block: int = 1 << 22) -> np.ndarray:
    """Draw N(0,1) values of `shape` and store them in the config dtype.

    The array is cut into blocks of `block` values; one draw from `rng` gives
    each block its own seed, and the blocks are filled in parallel.  The values
    depend only on `rng`'s state, never on the thread count.
    """
    n = int(np.prod(shape))
    nb = max(1, -(-n // block))
    seeds = rng.integers(0, np.iinfo(np.int64).max, size=nb, dtype=np.int64)
    out = np.empty(n, dtype=np.float32 if dtype == "f32" else np.uint16)

    def fill(i: int) -> None:
        s, e = i * block, min(n, (i + 1) * block)
        x = np.random.default_rng(int(seeds[i])).standard_normal(e - s, dtype=np.float32)
        out[s:e] = x if dtype == "f32" else bf16_bits_from_f32(x)

    if nb == 1:
        fill(0)
    else:
        with cf.ThreadPoolExecutor(max_workers=min(nb, os.cpu_count() or 4)) as ex:
            list(ex.map(fill, range(nb)))
    return out.reshape(shape)


def _storage_from_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    return x.copy() if dtype == "f32" else bf16_bits_from_f32(x)


# ---------------------------------------------------------------------------
# The workloads.  Sizes follow the five benchmark configurations; "prefill_2k"
# is an added prefill-heavy case (8 chunks of 2048 new tokens over 2048 cached
# tokens) where the tensor cores, not launch and tail effects, set the time.
# ---------------------------------------------------------------------------
CONFIGS = {
    "tiny_fp32_decode": dict(
        kind="decode", dtype="f32", B=4, Hq=4, Hkv=2, hd=64, P=16,
        context_lens=[5, 17, 33, 64], num_pages=32, seed=0),
    "qwen3_0p6b_decode": dict(
        kind="decode", dtype="bf16", B=256, Hq=16, Hkv=8, hd=128, P=16,
        L_range=(128, 2048), seed=2),
    "qwen3_8b_decode": dict(
        kind="decode", dtype="bf16", B=64, Hq=32, Hkv=8, hd=128, P=256,
        L_range=(1024, 8192), seed=3),
    "qwen3_0p6b_chunked_prefill": dict(
        kind="prefill", dtype="bf16", B=8, Hq=16, Hkv=8, hd=128, P=16,
        chunks=[1, 32, 64, 512, 1, 32, 64, 512], prefix_range=(0, 4096),
        prefix_first=0, prefix_last=4096, norm=True, seed=4),
    "long_context_decode": dict(
        kind="decode", dtype="bf16", B=8, Hq=32, Hkv=8, hd=128, P=256,
        L_fixed=32768, seed=5),
    "prefill_2k": dict(
        kind="prefill", dtype="bf16", B=8, Hq=16, Hkv=8, hd=128, P=16,
        chunks=[2048] * 8, prefixes=[2048] * 8, norm=True, seed=6),
}

# The order in which the benchmark configurations are listed (1-based index).
CONFIG_ORDER = ["tiny_fp32_decode", "qwen3_0p6b_decode", "qwen3_8b_decode",
                "qwen3_0p6b_chunked_prefill", "long_context_decode"]


@dataclasses.dataclass
class Workload:
    name: str
    kind: str                 # "decode" or "prefill"
    dtype: str                # "f32" or "bf16"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    poison_page: int
    context_lens: np.ndarray  # int32 [B]  cached prefix + this step's tokens
    new_lens: np.ndarray      # int32 [B]  this step's tokens per request
    cu_seqlens_q: np.ndarray  # int32 [B+1]
    hist_lens: np.ndarray     # int32 [B]  tokens already in the cache
    cu_hist: np.ndarray       # int32 [B+1]
    block_tables: np.ndarray  # int32 [B, max_pages]
    hist_k: np.ndarray        # storage [sum(hist_lens), Hkv, hd], logical order
    hist_v: np.ndarray
    k_new: np.ndarray         # storage [sum(new_lens), Hkv, hd]
    v_new: np.ndarray
    q: np.ndarray             # storage [sum(new_lens), Hq, hd]
    q_norm_w: Optional[np.ndarray]
    k_norm_w: Optional[np.ndarray]
    eps: Optional[float]
    rope_theta: Optional[float]
    scale: float
    seed: int

    @property
    def batch(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_new_tokens(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.batch else 0

    @property
    def max_new_len(self) -> int:
        return int(self.new_lens.max()) if self.batch else 0

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def poison_storage(self, shape) -> np.ndarray:
        """An array of `shape` filled with NaN in the config's storage format."""
        if self.dtype == "f32":
            return np.full(shape, np.nan, dtype=np.float32)
        return np.full(shape, BF16_NAN_BITS, dtype=np.uint16)

    def cache_shape(self):
        return (self.num_pages, self.page_size, self.num_kv_heads, self.head_dim)


def make_workload(name_or_spec, seed: Optional[int] = None, **overrides) -> Workload:
    """Build a workload from a named config or a spec dict (see CONFIGS)."""
    if isinstance(name_or_spec, str):
        spec = dict(CONFIGS[name_or_spec])
        name = name_or_spec
    else:
        spec = dict(name_or_spec)
        name = spec.pop("name", "custom")
    spec.update(overrides)
    if seed is None:
        seed = spec.get("seed", 0)
    rng = np.random.default_rng(seed)

    kind, dtype = spec["kind"], spec["dtype"]
    B, Hq, Hkv, hd, P = spec["B"], spec["Hq"], spec["Hkv"], spec["hd"], spec["P"]

    # 1. lengths
    if kind == "decode":
        if "context_lens" in spec:
            ctx = np.asarray(spec["context_lens"], dtype=np.int64)
        elif "L_fixed" in spec:
            ctx = np.full(B, spec["L_fixed"], dtype=np.int64)
        else:
            lo, hi = spec["L_range"]
            ctx = rng.integers(lo, hi + 1, size=B, dtype=np.int64)
        new = np.ones(B, dtype=np.int64)
        hist = ctx - new
    else:
        new = np.asarray(spec["chunks"], dtype=np.int64)
        if "prefixes" in spec:
            hist = np.asarray(spec["prefixes"], dtype=np.int64)
        else:
            lo, hi = spec["prefix_range"]
            hist = rng.integers(lo, hi + 1, size=B, dtype=np.int64)
            if "prefix_first" in spec and B > 0:
                hist[0] = spec["prefix_first"]
            if "prefix_last" in spec and B > 1:
                hist[-1] = spec["prefix_last"]
        ctx = hist + new
    assert ctx.shape == (B,) and new.shape == (B,)

    # 2. pages: request b owns ceil(ctx_b / P) pages, in logical order
    npages = (ctx + P - 1) // P
    used = int(npages.sum())
    if spec.get("num_pages") is not None:
        Np = int(spec["num_pages"])
    else:
        Np = used + 1 + int(math.ceil(0.05 * used))
    if used > Np - 1:
        raise ValueError(f"{name}: {used} pages needed but only {Np - 1} usable")
    perm = rng.permutation(Np - 1).astype(np.int32)
    poison = Np - 1
    max_pages = int(spec.get("max_pages_per_seq", max(1, int(npages.max()) if B else 1)))
    bt = np.full((B, max_pages), poison, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, : npages[b]] = perm[off: off + npages[b]]
        off += int(npages[b])

    cu_q = np.zeros(B + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(new)
    cu_h = np.zeros(B + 1, dtype=np.int32)
    cu_h[1:] = np.cumsum(hist)

    # 3.-5. values
    n_hist, n_new = int(cu_h[-1]), int(cu_q[-1])
    hist_k = _normal_storage(rng, (n_hist, Hkv, hd), dtype)
    hist_v = _normal_storage(rng, (n_hist, Hkv, hd), dtype)
    k_new = _normal_storage(rng, (n_new, Hkv, hd), dtype)
    v_new = _normal_storage(rng, (n_new, Hkv, hd), dtype)
    q = _normal_storage(rng, (n_new, Hq, hd), dtype)

    # 6. norm weights
    q_w = k_w = None
    eps = theta = None
    if spec.get("norm", False):
        q_w = _storage_from_f32(1.0 + 0.1 * rng.standard_normal(hd), dtype)
        k_w = _storage_from_f32(1.0 + 0.1 * rng.standard_normal(hd), dtype)
        eps = float(spec.get("eps", 1e-6))
        theta = float(spec.get("rope_theta", 1e6))

    return Workload(
        name=name, kind=kind, dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv,
        head_dim=hd, page_size=P, num_pages=Np, poison_page=poison,
        context_lens=ctx.astype(np.int32), new_lens=new.astype(np.int32),
        cu_seqlens_q=cu_q, hist_lens=hist.astype(np.int32), cu_hist=cu_h,
        block_tables=bt, hist_k=hist_k, hist_v=hist_v, k_new=k_new, v_new=v_new,
        q=q, q_norm_w=q_w, k_norm_w=k_w, eps=eps, rope_theta=theta,
        scale=float(spec.get("scale", 1.0 / math.sqrt(hd))), seed=int(seed))


def to_torch(wl: Workload, device="cuda") -> dict:
    """The workload's arrays as torch tensors on `device` (bit-identical values).

    bf16 arrays travel as their uint16 bit patterns and are reinterpreted, so
    no value is rounded again on the way.
    """
    import torch

    def arr(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    out = {k: arr(getattr(wl, k)) for k in ("hist_k", "hist_v", "k_new", "v_new", "q", "q_norm_w", "k_norm_w",
                                             "context_lens", "new_lens", "cu_seqlens_q", "hist_lens", "cu_hist",
                                             "block_tables")}
    return out
