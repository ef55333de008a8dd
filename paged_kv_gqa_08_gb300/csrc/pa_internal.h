// Internal interface between the C ABI (api.cu) and the kernel translation
// units.  Host-side C++ only; nothing here is exported.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pagedattn.h"

namespace pa {

// Cached properties of one device.
struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int max_smem_optin = 0;  // bytes per block with the opt-in attribute
  int cc_major = 0, cc_minor = 0;
  int l2_bytes = 0;        // L2 cache size
};
// Properties of the current device (queried once per device).
cudaError_t current_device_info(DeviceInfo* out);

// Address of the device error word on the current device.
cudaError_t device_error_word(unsigned int** out);

// Records `e` as the calling thread's last CUDA error (pa_last_cuda_error)
// and returns PA_ERR_CUDA; every entry point's PA_ERR_CUDA goes through it.
pa_status cuda_fail(cudaError_t e);

// Host-side checks shared by the decode entry points: the descriptor, the
// sizes, the scale and the pointers pa_decode takes (its workspace aside).
// PA_OK with batch == 0 means "nothing to do".
pa_status check_decode_args(const pa_cache_desc* d, const void* q, int32_t batch, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables, int32_t max_pages_per_seq,
                            const int32_t* context_lens, int32_t max_context_len, float scale, int32_t max_ctas,
                            const void* out);

inline int elem_bytes(int dtype) { return dtype == PA_F32 ? 4 : 2; }

// ---------------------------------------------------------------------------
// slot mapping / KV write / fused norm + rope + KV write
// ---------------------------------------------------------------------------
struct SlotMapParams {
  const int32_t* cu_seqlens_q;
  const int32_t* context_lens;
  const int32_t* block_tables;
  int32_t* positions;
  int64_t* slots;
  unsigned int* err;
  int64_t num_pages;
  int64_t num_tokens;
  int32_t batch, page_size, max_pages;
};
cudaError_t launch_slot_mapping(const SlotMapParams& p, cudaStream_t s);

struct KvWriteParams {
  const char* k;
  const char* v;
  int64_t k_stride_bytes, v_stride_bytes;
  int64_t n_tokens;
  const int64_t* slots;
  char* k_cache;
  char* v_cache;
  int64_t num_slots;
  int32_t row_bytes;
  unsigned int* err;
};
cudaError_t launch_kv_write(const KvWriteParams& p, cudaStream_t s);

struct NormRopeParams {
  const void* q;
  const void* k;
  const void* v;
  int64_t q_stride, k_stride, v_stride;  // elements
  int64_t n_tokens;
  const int32_t* positions;
  const void* wq;
  const void* wk;
  const int64_t* slots;
  void* q_out;
  void* k_cache;
  void* v_cache;
  int64_t num_slots;
  unsigned int* err;
  float eps;
  int32_t hq, hkv;
  // theta^(-2i/head_dim), computed on the host in double and passed as a
  // float plus the float nearest to the remainder
  float inv_freq_hi[64], inv_freq_lo[64];
  // positions == nullptr: each token's position and slot come from the varlen
  // metadata (as pa_slot_mapping computes them), optionally written out
  const int32_t* cu;
  const int32_t* ctx;
  const int32_t* bt;
  int32_t batch, maxp, page_size, log2P;
  int64_t num_pages;
  int32_t* pos_out;
  int64_t* slots_out;
};
cudaError_t launch_norm_rope_kv_write(int dtype, int head_dim, const NormRopeParams& p, cudaStream_t s);

// ---------------------------------------------------------------------------
// decode
// ---------------------------------------------------------------------------
struct DecodePlan {
  int nw = 0;            // consumer warps per CTA (= num_kv_heads)
  int tokens_per_chunk = 0;
  int chunk_bytes = 0;   // K (or V) bytes of one chunk in shared memory
  int row_pitch = 0;     // shared-memory bytes per token row of a chunk
  int stages = 0;
  int n_ctas = 0;        // partitions of the key space
  size_t smem_bytes = 0;
  // workspace layout (byte offsets)
  size_t ws_cs = 0, ws_cta_seq = 0, ws_lse = 0, ws_o = 0, ws_bytes = 0;
  // shared-memory layout (byte offsets)
  uint32_t off_bar = 0, off_meta = 0, off_p = 0, off_alpha = 0, off_ml = 0, off_abort = 0;
  uint32_t off_cs = 0;   // the batch's chunk prefix sums when each CTA plans for itself
  int p_row = 0;         // floats per token row of the probability tile
};
// Plan for the current device; returns cudaErrorInvalidValue for an
// unsupported shape.
cudaError_t plan_decode(const pa_cache_desc& d, int batch, int max_context_len, int max_ctas,
                        DecodePlan* out);

struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  void* workspace;
  unsigned int* err;
  int32_t batch, max_pages, max_context_len;
  float scale;
  // fused KV write of the step's new tokens (all null for plain decode)
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  int64_t k_new_stride_bytes = 0, v_new_stride_bytes = 0;
  int64_t* slot_out = nullptr;
};
cudaError_t launch_decode(const pa_cache_desc& d, const DecodePlan& plan, const DecodeArgs& a,
                          cudaStream_t s);

// Launch `fn` so that it may start while the stream's previous kernel runs
// (programmatic stream serialisation); the kernel calls pdl_wait() before it
// reads anything that kernel writes.
inline cudaError_t launch_after_previous(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                         void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// ---------------------------------------------------------------------------
// prefill
// ---------------------------------------------------------------------------
struct PrefillArgs {
  const void* q;
  const int32_t* cu_seqlens_q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  unsigned int* err;
  int64_t num_tokens;
  int32_t batch, max_seqlen_q, max_pages, max_context_len;
  float scale;
  // Caller workspace for the planned tensor-core launch (null: one CTA per
  // q-tile pair in grid order, no split).
  void* workspace = nullptr;
  size_t workspace_bytes = 0;
  // The stream's previous kernel is this library's KV write of the same step,
  // launched by the same call: it reads none of the metadata's producers'
  // output, so the planner may start beside it (and waits for it before it
  // exits, which the attention kernel's wait on the planner then covers).
  bool planner_beside_write = false;
};
// Workspace layout of the planned tensor-core prefill (byte offsets, each
// 256-aligned); ws_bytes == 0 when the call cannot be planned.
struct PrefillPlan {
  int32_t pair_cap, slot_cap, unit_cap, split_cap, n_sm;  // workspace layout capacities
  int32_t run_slot_cap, run_split_cap;  // this call: part slots the planner may use, split pairs it may form
  size_t off_hdr, off_pairs, off_units, off_splits, off_lse, off_o, ws_bytes;
};
cudaError_t plan_prefill(const pa_cache_desc& d, int32_t batch, int32_t max_seqlen_q, int64_t num_tokens,
                         int32_t max_context_len, PrefillPlan* out);
// CUDA-core kernel (any supported dtype / head_dim).
cudaError_t launch_prefill_simt(const pa_cache_desc& d, const PrefillArgs& a, cudaStream_t s);
// tcgen05 tensor-core kernel (bf16, head_dim 128).
cudaError_t launch_prefill_tc(const pa_cache_desc& d, const PrefillArgs& a, cudaStream_t s);

// ---------------------------------------------------------------------------
// metadata validation
// ---------------------------------------------------------------------------
struct ValidateArgs {
  const int32_t* cu_seqlens_q;
  const int32_t* context_lens;
  const int32_t* block_tables;
  int32_t* error_count;
  int64_t num_pages;
  int32_t batch, max_pages, max_context_len, page_size;
};
cudaError_t launch_validate(const ValidateArgs& a, cudaStream_t s);
cudaError_t launch_bounded_wait_selftest(unsigned int* err, int timeout_ms, cudaStream_t s);

}  // namespace pa
