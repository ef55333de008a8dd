// Chunked-prefill attention on the CUDA cores: the path for fp32 caches and
// head_dim 64 (bf16 / head_dim 128 runs on the tcgen05 kernel).
//
// Semantics (nano-vLLM learning note, Attention.forward and prepare_prefill
// listings; qwen-engine README, flat varlen packing): packed row t of request
// b sits at position context_lens[b] - n_b + (t - cu_seqlens_q[b]) and attends
// to keys 0 .. that position, read from the cache through block_tables[b].
//
// One warp per (packed row, q-head); a lane owns head_dim / 32 elements; one
// key per step with a warp-wide dot-product reduction and an online softmax
// in base 2.  Simple and exact-order-of-keys; not the fast path.
#include <math.h>

#include <algorithm>

#include "pa_common.cuh"

namespace pa {
namespace {

struct SimtParams {
  const char* q;
  const int32_t* cu;
  const char* k_cache;
  const char* v_cache;
  const int32_t* bt;
  const int32_t* ctx;
  char* out;
  unsigned int* err;
  int64_t num_pages;
  int64_t num_tokens;
  int32_t B, Hq, Hkv, P, maxp, max_ctx;
  float scale_log2;
};

template <typename T>
PA_DEVINL float load_elem(const char* base, int64_t idx) {
  if constexpr (sizeof(T) == 2) {
    return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(base)[idx]);
  } else {
    return reinterpret_cast<const float*>(base)[idx];
  }
}

template <typename T>
PA_DEVINL void store_elem(char* base, int64_t idx, float v) {
  if constexpr (sizeof(T) == 2) {
    reinterpret_cast<uint16_t*>(base)[idx] = float_to_bf16_bits(v);
  } else {
    reinterpret_cast<float*>(base)[idx] = v;
  }
}

template <typename T, int HD>
__global__ void __launch_bounds__(128) prefill_simt_kernel(const SimtParams p) {
  constexpr int DL = HD / 32;
  const int64_t t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = blockIdx.y * 4 + warp;
  if (hq >= p.Hq) return;
  // request of packed row t: last b with cu[b] <= t
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int s0 = p.cu[b], s1 = p.cu[b + 1];
  if (t < s0 || t >= s1) return;  // malformed cu_seqlens: nothing to do
  const int L = p.ctx[b];
  const int n = s1 - s0;
  if (L == 0) return;  // a padding row
  if (n > L || L > p.max_ctx || static_cast<int64_t>(L) > static_cast<int64_t>(p.maxp) * p.P) {
    if (lane == 0) raise_flag(p.err, PA_DEVERR_BAD_LENGTH);
    return;
  }
  const int pos = L - n + static_cast<int>(t - s0);
  const int G = p.Hq / p.Hkv;
  const int kvh = hq / G;

  float q[DL], o[DL];
#pragma unroll
  for (int e = 0; e < DL; ++e) {
    q[e] = load_elem<T>(p.q, (t * p.Hq + hq) * HD + lane + 32 * e) * p.scale_log2;
    o[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int32_t* row = p.bt + static_cast<int64_t>(b) * p.maxp;
  for (int j = 0; j <= pos; ++j) {
    const int page = row[j / p.P];
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) raise_flag(p.err, PA_DEVERR_BAD_PAGE);
      continue;
    }
    const int64_t base = ((static_cast<int64_t>(page) * p.P + (j % p.P)) * p.Hkv + kvh) * HD;
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < DL; ++e) s += q[e] * load_elem<T>(p.k_cache, base + lane + 32 * e);
#pragma unroll
    for (int msk = 16; msk >= 1; msk >>= 1) s += __shfl_xor_sync(0xffffffffu, s, msk);
    const float m_new = fmaxf(m, s);
    const float alpha = exp2f(m - m_new);
    const float pj = exp2f(s - m_new);
    l = l * alpha + pj;
#pragma unroll
    for (int e = 0; e < DL; ++e) o[e] = o[e] * alpha + pj * load_elem<T>(p.v_cache, base + lane + 32 * e);
    m = m_new;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < DL; ++e) store_elem<T>(p.out, (t * p.Hq + hq) * HD + lane + 32 * e, o[e] * inv);
}

}  // namespace

cudaError_t launch_prefill_simt(const pa_cache_desc& d, const PrefillArgs& a, cudaStream_t s) {
  if (a.num_tokens == 0 || a.batch == 0) return cudaSuccess;
  SimtParams p{};
  p.q = static_cast<const char*>(a.q);
  p.cu = a.cu_seqlens_q;
  p.k_cache = static_cast<const char*>(a.k_cache);
  p.v_cache = static_cast<const char*>(a.v_cache);
  p.bt = a.block_tables;
  p.ctx = a.context_lens;
  p.out = static_cast<char*>(a.out);
  p.err = a.err;
  p.num_pages = d.num_pages;
  p.num_tokens = a.num_tokens;
  p.B = a.batch;
  p.Hq = d.num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.P = d.page_size;
  p.maxp = a.max_pages;
  p.max_ctx = a.max_context_len;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  const dim3 grid(static_cast<unsigned>(a.num_tokens), (d.num_q_heads + 3) / 4);
  if (d.dtype == PA_BF16) {
    if (d.head_dim == 128) prefill_simt_kernel<__nv_bfloat16, 128><<<grid, 128, 0, s>>>(p);
    else prefill_simt_kernel<__nv_bfloat16, 64><<<grid, 128, 0, s>>>(p);
  } else {
    if (d.head_dim == 128) prefill_simt_kernel<float, 128><<<grid, 128, 0, s>>>(p);
    else prefill_simt_kernel<float, 64><<<grid, 128, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace pa
