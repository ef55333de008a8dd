// pa_decode_no_alloc: pa_decode for callers that cannot allocate device
// memory.  The pages have no counterpart of this call.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run decode: a plugin or embedding that is handed only its input
// and output buffers, code inside a framework that forbids allocations at that
// point, or a process whose memory manager owns the whole device heap.  pa_decode needs a caller-owned
// workspace for its split-KV partials; this variant takes that scratch from a
// fixed array inside the library instead.  The caller still passes q, the
// caches, the metadata and the output.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes
// (16 MiB); every device that loads the library holds it until the process
// exits.  Every call shares it and it keeps the last call's contents; nothing
// in it needs to start at zero (each call's plan kernel rewrites the metadata
// the decode and merge kernels read, and every partial is written before it is
// read), but calls that overlap on the GPU -- on two streams, or from two
// host threads -- race on it.
#include <cuda_runtime.h>
#include <math.h>

#include <mutex>

#include "pa_internal.h"

namespace pa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

// Device memory.  In host code this name is a host-side stand-in, not a device
// address: host code reaches the array only through the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device; looked up once
// per device, with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The same host-side checks as pa_decode, minus the workspace arguments.
pa_status check_args(const pa_cache_desc* d, const void* q, int32_t batch, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int32_t max_pages_per_seq, const int32_t* context_lens,
                     int32_t max_context_len, float scale, int32_t max_ctas, const void* out) {
  if (!d) return PA_ERR_NULL;
  if (d->dtype != PA_F32 && d->dtype != PA_BF16) return PA_ERR_DTYPE;
  if (d->num_q_heads < 1 || d->num_kv_heads < 1 || d->head_dim < 1 || d->page_size < 1 || d->num_pages < 1)
    return PA_ERR_SHAPE;
  if (d->num_q_heads % d->num_kv_heads != 0) return PA_ERR_SHAPE;
  if (d->head_dim != 64 && d->head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (!pow2(d->num_kv_heads) || d->num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
  if (d->num_q_heads / d->num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
  if (!pow2(d->page_size) || d->page_size < 16) return PA_ERR_UNSUPPORTED;
  if (d->num_pages > (int64_t(1) << 40) / d->page_size) return PA_ERR_SHAPE;
  if (batch < 0 || max_ctas < 0) return PA_ERR_SHAPE;
  if (batch == 0) return PA_OK;
  if (max_pages_per_seq < 1 || max_context_len < 1) return PA_ERR_SHAPE;
  if (static_cast<int64_t>(max_context_len) > static_cast<int64_t>(max_pages_per_seq) * d->page_size)
    return PA_ERR_SHAPE;
  if (!isfinite(scale)) return PA_ERR_SHAPE;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_NULL;
  if (!al16(q) || !al16(k_cache) || !al16(v_cache) || !al16(out)) return PA_ERR_ALIGN;
  return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_decode_no_alloc(const pa_cache_desc* desc, const void* q, int32_t batch,
                                        const void* k_cache, const void* v_cache, const int32_t* block_tables,
                                        int32_t max_pages_per_seq, const int32_t* context_lens,
                                        int32_t max_context_len, float scale, int32_t max_ctas, void* out,
                                        pa_stream_t stream) {
  pa_status st = check_args(desc, q, batch, k_cache, v_cache, block_tables, max_pages_per_seq, context_lens,
                            max_context_len, scale, max_ctas, out);
  if (st != PA_OK || batch == 0) return st;
  (void)cudaGetLastError();
  unsigned int* err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  DecodePlan pl;
  e = plan_decode(*desc, batch, max_context_len, max_ctas, &pl);
  if (e == cudaErrorInvalidValue) return PA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return PA_ERR_CUDA;
  if (pl.ws_bytes > kNoAllocScratchBytes) return PA_ERR_WORKSPACE;  // batch too large for the fixed scratch
  void* scratch = nullptr;
  e = scratch_address(&scratch);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = out;
  a.workspace = scratch;
  a.err = err;
  a.batch = batch;
  a.max_pages = max_pages_per_seq;
  a.max_context_len = max_context_len;
  a.scale = scale;
  e = launch_decode(*desc, pl, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
