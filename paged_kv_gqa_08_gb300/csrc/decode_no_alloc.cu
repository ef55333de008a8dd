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
// (16 MiB); every device that loads the library's code holds it until the
// process exits.  Under lazy module loading (CUDA_MODULE_LOADING=LAZY, the
// runtime's default) the array is placed in device memory only when its
// address is first looked up, which the first call of this entry point on
// each device does: make that call early, before the caller's memory manager
// takes the rest of the device heap and before any stream capture.  Later
// calls look up nothing and touch no allocator.  Every call shares it and it keeps the last call's contents; nothing
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

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_decode_no_alloc(const pa_cache_desc* desc, const void* q, int32_t batch,
                                        const void* k_cache, const void* v_cache, const int32_t* block_tables,
                                        int32_t max_pages_per_seq, const int32_t* context_lens,
                                        int32_t max_context_len, float scale, int32_t max_ctas, void* out,
                                        pa_stream_t stream) {
  pa_status st = check_decode_args(desc, q, batch, k_cache, v_cache, block_tables, max_pages_per_seq, context_lens,
                                   max_context_len, scale, max_ctas, out);
  if (st != PA_OK || batch == 0) return st;
  (void)cudaGetLastError();
  unsigned int* err = nullptr;
  cudaError_t e = device_error_word(&err);
  if (e != cudaSuccess) return cuda_fail(e);
  DecodePlan pl;
  e = plan_decode(*desc, batch, max_context_len, max_ctas, &pl);
  if (e == cudaErrorInvalidValue) return PA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return cuda_fail(e);
  if (pl.ws_bytes > kNoAllocScratchBytes) return PA_ERR_WORKSPACE;  // batch too large for the fixed scratch
  void* scratch = nullptr;
  e = scratch_address(&scratch);
  if (e != cudaSuccess) return cuda_fail(e);
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
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}
