// The C ABI of libpagedattn: host-side argument validation, per-device
// caches, the device error word, and kernel dispatch.  Every entry point
// validates everything it can see on the host before enqueueing anything.
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "pa_internal.h"

namespace pa {

// Device-side error flags (PA_DEVERR_*); one word per device.
__device__ unsigned int g_device_error_flags;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
unsigned int* g_err_word[kMaxDevices];
thread_local int g_last_cuda_error = 0;

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pa_status check_desc(const pa_cache_desc* d) {
  if (!d) return PA_ERR_NULL;
  if (d->dtype != PA_F32 && d->dtype != PA_BF16) return PA_ERR_DTYPE;
  if (d->num_q_heads < 1 || d->num_kv_heads < 1 || d->head_dim < 1 || d->page_size < 1 || d->num_pages < 1)
    return PA_ERR_SHAPE;
  if (d->num_q_heads % d->num_kv_heads != 0) return PA_ERR_SHAPE;
  if (d->head_dim != 64 && d->head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(d->num_kv_heads) || d->num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
  if (d->num_q_heads / d->num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(d->page_size) || d->page_size < 16) return PA_ERR_UNSUPPORTED;
  if (d->num_pages > (int64_t(1) << 40) / d->page_size) return PA_ERR_SHAPE;
  return PA_OK;
}

int64_t row_elems(const pa_cache_desc* d) { return static_cast<int64_t>(d->num_kv_heads) * d->head_dim; }

// A row stride (elements) is usable when it covers the row and keeps 16-byte alignment.
bool stride_ok(const pa_cache_desc* d, int64_t stride, int64_t min_elems) {
  return stride >= min_elems && (stride * elem_bytes(d->dtype)) % 16 == 0;
}

// Called by every entry point once its arguments are validated, before it
// launches anything: fetches the device error word and clears a launch error
// left pending by earlier, unrelated CUDA calls, so that the error checked
// after our own launches is ours.
pa_status prepare(unsigned int** err) {
  (void)cudaGetLastError();
  cudaError_t e = device_error_word(err);
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // namespace

pa_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return PA_ERR_CUDA;
}

pa_status check_decode_args(const pa_cache_desc* d, const void* q, int32_t batch, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables, int32_t max_pages_per_seq,
                            const int32_t* context_lens, int32_t max_context_len, float scale, int32_t max_ctas,
                            const void* out) {
  pa_status st = check_desc(d);
  if (st != PA_OK) return st;
  if (batch < 0 || max_ctas < 0) return PA_ERR_SHAPE;
  if (batch == 0) return PA_OK;
  if (max_pages_per_seq < 1 || max_context_len < 1) return PA_ERR_SHAPE;
  if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_pages_per_seq) * d->page_size)
    return PA_ERR_SHAPE;
  if (!isfinite(scale)) return PA_ERR_SHAPE;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PA_ERR_ALIGN;
  return PA_OK;
}

cudaError_t current_device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_info[dev].device != dev) {
    DeviceInfo di;
    di.device = dev;
    if ((e = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
        cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&di.l2_bytes, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) return e;
    g_info[dev] = di;
  }
  *out = g_info[dev];
  return cudaSuccess;
}

cudaError_t device_error_word(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_word[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error_flags);
    if (e != cudaSuccess) return e;
    g_err_word[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_err_word[dev];
  return cudaSuccess;
}

}  // namespace pa

namespace pa {
namespace {

// Checks of pa_slot_mapping's arguments (batch > 0) and its parameters, the
// error word left to the caller.
pa_status slot_map_params(const pa_cache_desc* desc, int32_t batch, const int32_t* cu_seqlens_q,
                          const int32_t* context_lens, const int32_t* block_tables, int32_t max_pages_per_seq,
                          int64_t num_tokens, int32_t* positions, int64_t* slot_mapping, SlotMapParams* out) {
  if (!cu_seqlens_q || !context_lens || !block_tables) return PA_ERR_NULL;
  if (num_tokens > 0 && (!positions || !slot_mapping)) return PA_ERR_NULL;
  SlotMapParams& p = *out;
  p = SlotMapParams{};
  p.cu_seqlens_q = cu_seqlens_q;
  p.context_lens = context_lens;
  p.block_tables = block_tables;
  p.positions = positions;
  p.slots = slot_mapping;
  p.num_pages = desc->num_pages;
  p.num_tokens = num_tokens;
  p.batch = batch;
  p.page_size = desc->page_size;
  p.max_pages = max_pages_per_seq;
  return PA_OK;
}

// Checks of pa_kv_write's arguments (num_tokens > 0) and its parameters.
pa_status kv_write_params(const pa_cache_desc* desc, const void* k, int64_t k_row_stride, const void* v,
                          int64_t v_row_stride, int64_t num_tokens, const int64_t* slot_mapping, void* k_cache,
                          void* v_cache, KvWriteParams* out) {
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_NULL;
  const int64_t re = row_elems(desc);
  if (k_row_stride < re || v_row_stride < re) return PA_ERR_SHAPE;
  if (!stride_ok(desc, k_row_stride, re) || !stride_ok(desc, v_row_stride, re)) return PA_ERR_ALIGN;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
  const int E = elem_bytes(desc->dtype);
  KvWriteParams& p = *out;
  p = KvWriteParams{};
  p.k = static_cast<const char*>(k);
  p.v = static_cast<const char*>(v);
  p.k_stride_bytes = k_row_stride * E;
  p.v_stride_bytes = v_row_stride * E;
  p.n_tokens = num_tokens;
  p.slots = slot_mapping;
  p.k_cache = static_cast<char*>(k_cache);
  p.v_cache = static_cast<char*>(v_cache);
  p.num_slots = desc->num_pages * desc->page_size;
  p.row_bytes = static_cast<int32_t>(re * E);
  return PA_OK;
}

// The checks and parameters both norm / rotary entry points share; the
// position / slot source is filled in by the caller.
pa_status norm_rope_params(const pa_cache_desc* desc, const void* q, int64_t q_row_stride, const void* k,
                           int64_t k_row_stride, const void* v, int64_t v_row_stride, int64_t num_tokens,
                           const void* q_norm_w, const void* k_norm_w, float eps, float rope_theta, void* q_out,
                           void* k_cache, void* v_cache, NormRopeParams* out) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_tokens < 0 || num_tokens > 0x7fffffff) return PA_ERR_SHAPE;
  if (!q || !k || !v || !q_norm_w || !k_norm_w || !q_out || !k_cache || !v_cache) return PA_ERR_NULL;
  if (!(eps >= 0.f) || !isfinite(eps) || !(rope_theta > 1.f) || !isfinite(rope_theta)) return PA_ERR_SHAPE;
  const int64_t re = row_elems(desc);
  const int64_t qe = static_cast<int64_t>(desc->num_q_heads) * desc->head_dim;
  if (q_row_stride < qe || k_row_stride < re || v_row_stride < re) return PA_ERR_SHAPE;
  if (!stride_ok(desc, q_row_stride, qe) || !stride_ok(desc, k_row_stride, re) || !stride_ok(desc, v_row_stride, re))
    return PA_ERR_ALIGN;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_out) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(q_norm_w) || !aligned16(k_norm_w))
    return PA_ERR_ALIGN;
  if (q_out == q && q_row_stride != qe) return PA_ERR_SHAPE;
  NormRopeParams& p = *out;
  p = NormRopeParams{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.q_stride = q_row_stride;
  p.k_stride = k_row_stride;
  p.v_stride = v_row_stride;
  p.n_tokens = num_tokens;
  p.wq = q_norm_w;
  p.wk = k_norm_w;
  p.q_out = q_out;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.num_slots = desc->num_pages * desc->page_size;
  p.eps = eps;
  p.hq = desc->num_q_heads;
  p.hkv = desc->num_kv_heads;
  for (int i = 0; i < desc->head_dim / 2; ++i) {
    const double f = pow(static_cast<double>(rope_theta), -2.0 * i / desc->head_dim);
    p.inv_freq_hi[i] = static_cast<float>(f);
    p.inv_freq_lo[i] = static_cast<float>(f - static_cast<double>(p.inv_freq_hi[i]));
  }
  return PA_OK;
}

// Checks of pa_prefill_qk_norm_rope_kv_write's arguments (num_tokens > 0) and
// its parameters, the error word left to the caller.
pa_status prefill_norm_params(const pa_cache_desc* desc, const void* q, int64_t q_row_stride, const void* k,
                              int64_t k_row_stride, const void* v, int64_t v_row_stride, int64_t num_tokens,
                              const int32_t* cu_seqlens_q, int32_t batch, const int32_t* context_lens,
                              const int32_t* block_tables, int32_t max_pages_per_seq, const void* q_norm_w,
                              const void* k_norm_w, float eps, float rope_theta, void* q_out, void* k_cache,
                              void* v_cache, int32_t* positions_out, int64_t* slot_mapping_out, NormRopeParams* out) {
  if (batch == 0 || max_pages_per_seq < 1) return PA_ERR_SHAPE;  // tokens without requests, or no pages
  NormRopeParams& p = *out;
  pa_status st = norm_rope_params(desc, q, q_row_stride, k, k_row_stride, v, v_row_stride, num_tokens, q_norm_w,
                                  k_norm_w, eps, rope_theta, q_out, k_cache, v_cache, &p);
  if (st != PA_OK) return st;
  if (!cu_seqlens_q || !context_lens || !block_tables) return PA_ERR_NULL;
  p.cu = cu_seqlens_q;
  p.ctx = context_lens;
  p.bt = block_tables;
  p.batch = batch;
  p.maxp = max_pages_per_seq;
  p.page_size = desc->page_size;
  p.log2P = 0;
  while ((1 << p.log2P) < desc->page_size) ++p.log2P;
  p.num_pages = desc->num_pages;
  p.pos_out = positions_out;
  p.slots_out = slot_mapping_out;
  return PA_OK;
}

// Checks of pa_prefill_varlen's arguments and its launch arguments, the error
// word left to the caller; a->num_tokens == 0 when there is nothing to do.
pa_status prefill_args(const pa_cache_desc* desc, const void* q, const int32_t* cu_seqlens_q, int32_t batch,
                       int32_t max_seqlen_q, int64_t num_tokens, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int32_t max_pages_per_seq, const int32_t* context_lens,
                       int32_t max_context_len, float scale, void* out, void* workspace, size_t workspace_bytes,
                       PrefillArgs* a) {
  *a = PrefillArgs{};
  if (batch < 0 || num_tokens < 0 || max_seqlen_q < 0) return PA_ERR_SHAPE;
  if (batch == 0 || num_tokens == 0 || max_seqlen_q == 0) return num_tokens == 0 ? PA_OK : PA_ERR_SHAPE;
  if (num_tokens > 0x7fffffff) return PA_ERR_SHAPE;
  if (max_pages_per_seq < 1 || max_context_len < 1 || max_seqlen_q > max_context_len) return PA_ERR_SHAPE;
  if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_pages_per_seq) * desc->page_size)
    return PA_ERR_SHAPE;
  if (!isfinite(scale) || !(scale > 0.f)) return PA_ERR_SHAPE;
  if (!q || !cu_seqlens_q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PA_ERR_ALIGN;
  if (workspace) {
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_ALIGN;
    PrefillPlan plan;
    cudaError_t e = plan_prefill(*desc, batch, max_seqlen_q, num_tokens, max_context_len, &plan);
    if (e != cudaSuccess) return cuda_fail(e);
    if (plan.ws_bytes == 0) workspace = nullptr;  // this call is never planned
    else if (workspace_bytes < plan.ws_bytes) return PA_ERR_WORKSPACE;
  }
  a->q = q;
  a->cu_seqlens_q = cu_seqlens_q;
  a->k_cache = k_cache;
  a->v_cache = v_cache;
  a->block_tables = block_tables;
  a->context_lens = context_lens;
  a->out = out;
  a->num_tokens = num_tokens;
  a->batch = batch;
  a->max_seqlen_q = max_seqlen_q;
  a->max_pages = max_pages_per_seq;
  a->max_context_len = max_context_len;
  a->scale = scale;
  a->workspace = workspace;
  a->workspace_bytes = workspace_bytes;
  return PA_OK;
}

cudaError_t launch_prefill(const pa_cache_desc& d, const PrefillArgs& a, cudaStream_t s) {
  return d.dtype == PA_BF16 && d.head_dim == 128 ? launch_prefill_tc(d, a, s) : launch_prefill_simt(d, a, s);
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

pa_status pa_slot_mapping(const pa_cache_desc* desc, int32_t batch, const int32_t* cu_seqlens_q,
                          const int32_t* context_lens, const int32_t* block_tables, int32_t max_pages_per_seq,
                          int64_t num_tokens, int32_t* positions, int64_t* slot_mapping, pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (batch < 0 || num_tokens < 0 || max_pages_per_seq < 1) return PA_ERR_SHAPE;
  if (batch == 0) return num_tokens == 0 ? PA_OK : PA_ERR_SHAPE;
  SlotMapParams p;
  st = slot_map_params(desc, batch, cu_seqlens_q, context_lens, block_tables, max_pages_per_seq, num_tokens,
                       positions, slot_mapping, &p);
  if (st != PA_OK) return st;
  if ((st = prepare(&p.err)) != PA_OK) return st;
  cudaError_t e = launch_slot_mapping(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_kv_write(const pa_cache_desc* desc, const void* k, int64_t k_row_stride, const void* v,
                      int64_t v_row_stride, int64_t num_tokens, const int64_t* slot_mapping, void* k_cache,
                      void* v_cache, pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  KvWriteParams p;
  st = kv_write_params(desc, k, k_row_stride, v, v_row_stride, num_tokens, slot_mapping, k_cache, v_cache, &p);
  if (st != PA_OK) return st;
  if ((st = prepare(&p.err)) != PA_OK) return st;
  cudaError_t e = launch_kv_write(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_qk_norm_rope_kv_write(const pa_cache_desc* desc, const void* q, int64_t q_row_stride, const void* k,
                                   int64_t k_row_stride, const void* v, int64_t v_row_stride, int64_t num_tokens,
                                   const int32_t* positions, const void* q_norm_w, const void* k_norm_w, float eps,
                                   float rope_theta, const int64_t* slot_mapping, void* q_out, void* k_cache,
                                   void* v_cache, pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  NormRopeParams p;
  st = norm_rope_params(desc, q, q_row_stride, k, k_row_stride, v, v_row_stride, num_tokens, q_norm_w, k_norm_w, eps,
                        rope_theta, q_out, k_cache, v_cache, &p);
  if (st != PA_OK) return st;
  if (!positions || !slot_mapping) return PA_ERR_NULL;
  unsigned int* err = nullptr;
  if ((st = prepare(&err)) != PA_OK) return st;
  p.positions = positions;
  p.slots = slot_mapping;
  p.err = err;
  cudaError_t e = launch_norm_rope_kv_write(desc->dtype, desc->head_dim, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_prefill_qk_norm_rope_kv_write(const pa_cache_desc* desc, const void* q, int64_t q_row_stride,
                                           const void* k, int64_t k_row_stride, const void* v, int64_t v_row_stride,
                                           int64_t num_tokens, const int32_t* cu_seqlens_q, int32_t batch,
                                           const int32_t* context_lens, const int32_t* block_tables,
                                           int32_t max_pages_per_seq, const void* q_norm_w, const void* k_norm_w,
                                           float eps, float rope_theta, void* q_out, void* k_cache, void* v_cache,
                                           int32_t* positions_out, int64_t* slot_mapping_out, pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_tokens < 0 || batch < 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  NormRopeParams p;
  st = prefill_norm_params(desc, q, q_row_stride, k, k_row_stride, v, v_row_stride, num_tokens, cu_seqlens_q, batch,
                           context_lens, block_tables, max_pages_per_seq, q_norm_w, k_norm_w, eps, rope_theta, q_out,
                           k_cache, v_cache, positions_out, slot_mapping_out, &p);
  if (st != PA_OK) return st;
  if ((st = prepare(&p.err)) != PA_OK) return st;
  cudaError_t e = launch_norm_rope_kv_write(desc->dtype, desc->head_dim, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

size_t pa_decode_workspace_size(const pa_cache_desc* desc, int32_t batch, int32_t max_context_len,
                                int32_t max_ctas) {
  if (check_desc(desc) != PA_OK || batch < 1 || max_context_len < 1 || max_ctas < 0) return 0;
  DecodePlan pl;
  if (plan_decode(*desc, batch, max_context_len, max_ctas, &pl) != cudaSuccess) return 0;
  return pl.ws_bytes;
}

pa_status pa_decode_plan_info(const pa_cache_desc* desc, int32_t batch, int32_t max_context_len, int32_t max_ctas,
                              int32_t* num_partitions, int32_t* tokens_per_chunk) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (batch < 1 || max_context_len < 1 || max_ctas < 0) return PA_ERR_SHAPE;
  DecodePlan pl;
  cudaError_t e = plan_decode(*desc, batch, max_context_len, max_ctas, &pl);
  if (e == cudaErrorInvalidValue) return PA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return cuda_fail(e);
  if (num_partitions) *num_partitions = pl.n_ctas;
  if (tokens_per_chunk) *tokens_per_chunk = pl.tokens_per_chunk;
  return PA_OK;
}

pa_status pa_decode(const pa_cache_desc* desc, const void* q, int32_t batch, const void* k_cache,
                    const void* v_cache, const int32_t* block_tables, int32_t max_pages_per_seq,
                    const int32_t* context_lens, int32_t max_context_len, float scale, int32_t max_ctas, void* out,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  pa_status st = check_decode_args(desc, q, batch, k_cache, v_cache, block_tables, max_pages_per_seq, context_lens,
                                   max_context_len, scale, max_ctas, out);
  if (st != PA_OK || batch == 0) return st;
  if (!workspace) return PA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_ALIGN;
  unsigned int* err = nullptr;
  if ((st = prepare(&err)) != PA_OK) return st;
  DecodePlan pl;
  cudaError_t e = plan_decode(*desc, batch, max_context_len, max_ctas, &pl);
  if (e == cudaErrorInvalidValue) return PA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return cuda_fail(e);
  if (workspace_bytes < pl.ws_bytes) return PA_ERR_WORKSPACE;
  DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = out;
  a.workspace = workspace;
  a.err = err;
  a.batch = batch;
  a.max_pages = max_pages_per_seq;
  a.max_context_len = max_context_len;
  a.scale = scale;
  e = launch_decode(*desc, pl, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_decode_kv_write(const pa_cache_desc* desc, const void* q, const void* k_new, int64_t k_row_stride,
                             const void* v_new, int64_t v_row_stride, int32_t batch, void* k_cache, void* v_cache,
                             const int32_t* block_tables, int32_t max_pages_per_seq, const int32_t* context_lens,
                             int32_t max_context_len, float scale, int32_t max_ctas, int64_t* slot_mapping,
                             void* out, void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (batch < 0 || max_ctas < 0) return PA_ERR_SHAPE;
  if (batch == 0) return PA_OK;
  if (max_pages_per_seq < 1 || max_context_len < 1) return PA_ERR_SHAPE;
  if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_pages_per_seq) * desc->page_size)
    return PA_ERR_SHAPE;
  if (!isfinite(scale)) return PA_ERR_SHAPE;
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_NULL;
  const int64_t re = row_elems(desc);
  if (k_row_stride < re || v_row_stride < re) return PA_ERR_SHAPE;
  if (!stride_ok(desc, k_row_stride, re) || !stride_ok(desc, v_row_stride, re)) return PA_ERR_ALIGN;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(out))
    return PA_ERR_ALIGN;
  if (desc->num_pages * desc->page_size >= (int64_t(1) << 31)) return PA_ERR_UNSUPPORTED;
  if (!workspace) return PA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_ALIGN;
  unsigned int* err = nullptr;
  if ((st = prepare(&err)) != PA_OK) return st;
  DecodePlan pl;
  cudaError_t e = plan_decode(*desc, batch, max_context_len, max_ctas, &pl);
  if (e == cudaErrorInvalidValue) return PA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return cuda_fail(e);
  if (workspace_bytes < pl.ws_bytes) return PA_ERR_WORKSPACE;
  DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = out;
  a.workspace = workspace;
  a.err = err;
  a.batch = batch;
  a.max_pages = max_pages_per_seq;
  a.max_context_len = max_context_len;
  a.scale = scale;
  const int E = elem_bytes(desc->dtype);
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_new_stride_bytes = k_row_stride * E;
  a.v_new_stride_bytes = v_row_stride * E;
  a.slot_out = slot_mapping;
  e = launch_decode(*desc, pl, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_prefill_varlen(const pa_cache_desc* desc, const void* q, const int32_t* cu_seqlens_q, int32_t batch,
                            int32_t max_seqlen_q, int64_t num_tokens, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int32_t max_pages_per_seq, const int32_t* context_lens,
                            int32_t max_context_len, float scale, void* out, void* workspace,
                            size_t workspace_bytes, pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  PrefillArgs a;
  st = prefill_args(desc, q, cu_seqlens_q, batch, max_seqlen_q, num_tokens, k_cache, v_cache, block_tables,
                    max_pages_per_seq, context_lens, max_context_len, scale, out, workspace, workspace_bytes, &a);
  if (st != PA_OK || a.num_tokens == 0) return st;
  if ((st = prepare(&a.err)) != PA_OK) return st;
  cudaError_t e = launch_prefill(*desc, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_prefill_step(const pa_cache_desc* desc, const void* q, int64_t q_row_stride, const void* k,
                          int64_t k_row_stride, const void* v, int64_t v_row_stride, int64_t num_tokens,
                          const int32_t* cu_seqlens_q, int32_t batch, int32_t max_seqlen_q,
                          const int32_t* context_lens, int32_t max_context_len, const int32_t* block_tables,
                          int32_t max_pages_per_seq, const void* q_norm_w, const void* k_norm_w, float eps,
                          float rope_theta, float scale, void* q_out, void* k_cache, void* v_cache,
                          int32_t* positions_out, int64_t* slot_mapping_out, void* out, void* workspace,
                          size_t workspace_bytes, pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_tokens < 0 || batch < 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  const bool norm = q_norm_w != nullptr || k_norm_w != nullptr;
  // every argument of both parts is checked before anything is enqueued
  NormRopeParams np;
  SlotMapParams sp;
  KvWriteParams kp;
  if (norm) {
    st = prefill_norm_params(desc, q, q_row_stride, k, k_row_stride, v, v_row_stride, num_tokens, cu_seqlens_q,
                             batch, context_lens, block_tables, max_pages_per_seq, q_norm_w, k_norm_w, eps,
                             rope_theta, q_out, k_cache, v_cache, positions_out, slot_mapping_out, &np);
  } else {
    // attention reads q itself, so its rows must be packed
    if (q_row_stride != static_cast<int64_t>(desc->num_q_heads) * desc->head_dim) return PA_ERR_SHAPE;
    if (batch == 0 || max_pages_per_seq < 1) return PA_ERR_SHAPE;
    st = slot_map_params(desc, batch, cu_seqlens_q, context_lens, block_tables, max_pages_per_seq, num_tokens,
                         positions_out, slot_mapping_out, &sp);
    if (st == PA_OK)
      st = kv_write_params(desc, k, k_row_stride, v, v_row_stride, num_tokens, slot_mapping_out, k_cache, v_cache,
                           &kp);
  }
  if (st != PA_OK) return st;
  PrefillArgs a;
  st = prefill_args(desc, norm ? q_out : q, cu_seqlens_q, batch, max_seqlen_q, num_tokens, k_cache, v_cache,
                    block_tables, max_pages_per_seq, context_lens, max_context_len, scale, out, workspace,
                    workspace_bytes, &a);
  if (st != PA_OK) return st;
  unsigned int* err = nullptr;
  if ((st = prepare(&err)) != PA_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (norm) {
    np.err = err;
    e = launch_norm_rope_kv_write(desc->dtype, desc->head_dim, np, s);
  } else {
    sp.err = kp.err = err;
    e = launch_slot_mapping(sp, s);
    if (e == cudaSuccess) e = launch_kv_write(kp, s);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  a.err = err;
  a.planner_beside_write = true;
  e = launch_prefill(*desc, a, s);
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

size_t pa_prefill_workspace_size(const pa_cache_desc* desc, int32_t batch, int32_t max_seqlen_q,
                                 int64_t num_tokens, int32_t max_context_len) {
  if (check_desc(desc) != PA_OK || batch < 1 || max_seqlen_q < 1 || num_tokens < 1 || max_context_len < 1 ||
      max_seqlen_q > max_context_len || num_tokens > 0x7fffffff)
    return 0;
  PrefillPlan plan;
  if (plan_prefill(*desc, batch, max_seqlen_q, num_tokens, max_context_len, &plan) != cudaSuccess) return 0;
  return plan.ws_bytes;
}

pa_status pa_validate_metadata(const pa_cache_desc* desc, int32_t batch, const int32_t* cu_seqlens_q,
                               const int32_t* context_lens, const int32_t* block_tables, int32_t max_pages_per_seq,
                               int32_t max_context_len, int32_t* error_count, pa_stream_t stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (batch < 0 || max_pages_per_seq < 1 || max_context_len < 1) return PA_ERR_SHAPE;
  if (!error_count) return PA_ERR_NULL;
  if (batch > 0 && (!context_lens || !block_tables)) return PA_ERR_NULL;
  unsigned int* err = nullptr;
  if ((st = prepare(&err)) != PA_OK) return st;
  ValidateArgs a{};
  a.cu_seqlens_q = cu_seqlens_q;
  a.context_lens = context_lens;
  a.block_tables = block_tables;
  a.error_count = error_count;
  a.num_pages = desc->num_pages;
  a.batch = batch;
  a.max_pages = max_pages_per_seq;
  a.max_context_len = max_context_len;
  a.page_size = desc->page_size;
  cudaError_t e = launch_validate(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_selftest_bounded_wait(int32_t timeout_ms, pa_stream_t stream) {
  if (timeout_ms < 1 || timeout_ms > 10000) return PA_ERR_SHAPE;
  unsigned int* err = nullptr;
  pa_status st = prepare(&err);
  if (st != PA_OK) return st;
  cudaError_t e = launch_bounded_wait_selftest(err, timeout_ms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_read_device_errors(uint32_t* flags, int32_t reset) {
  if (!flags) return PA_ERR_NULL;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_error_flags, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e);
  *flags = v;
  if (reset) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_device_error_flags, &z, sizeof(z));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return PA_OK;
}

int32_t pa_last_cuda_error(void) { return g_last_cuda_error; }

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "a required pointer is NULL";
    case PA_ERR_DTYPE: return "unknown dtype";
    case PA_ERR_SHAPE: return "a count, size or stride is out of range";
    case PA_ERR_ALIGN: return "a pointer or row stride is not 16-byte aligned";
    case PA_ERR_UNSUPPORTED: return "shape outside the supported set";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_VALIDATION: return "metadata validation failed";
    case PA_ERR_CAPACITY: return "not enough free blocks";
  }
  return "unknown status";
}

int32_t pa_version(void) { return 200; }

}  // extern "C"
