// Opt-in device check of request metadata (block tables, lengths).
// Counts problems into a device word; never faults, never traps.
#include "pa_common.cuh"

namespace pa {
namespace {

__global__ void __launch_bounds__(128) validate_kernel(const ValidateArgs a) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.batch) return;
  int bad = 0;
  const int L = a.context_lens[b];
  if (L == 0) return;  // a padding row
  const int64_t by_pages = static_cast<int64_t>(a.max_pages) * a.page_size;
  const int64_t cap = a.max_context_len < by_pages ? a.max_context_len : by_pages;
  const bool len_ok = L >= 1 && L <= cap;
  if (!len_ok) ++bad;
  if (a.cu_seqlens_q) {
    const int n = a.cu_seqlens_q[b + 1] - a.cu_seqlens_q[b];
    if (n < 0 || (len_ok && n > L)) ++bad;
  }
  if (len_ok) {
    const int used = (L + a.page_size - 1) / a.page_size;
    const int32_t* row = a.block_tables + static_cast<int64_t>(b) * a.max_pages;
    for (int i = 0; i < used; ++i) {
      const int pg = row[i];
      if (pg < 0 || pg >= a.num_pages) ++bad;
    }
  }
  if (bad) atomicAdd(a.error_count, bad);
}

// One thread waits for an mbarrier phase that never completes; the bounded
// wait gives up after limit_ns and raises PA_DEVERR_TIMEOUT.
__global__ void bounded_wait_selftest_kernel(unsigned int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  mbar_wait_bounded(&bar, 0, &abort_flag, err, limit_ns);
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(unsigned int* err, int timeout_ms, cudaStream_t s) {
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(err, static_cast<uint64_t>(timeout_ms) * 1000000ull);
  return cudaGetLastError();
}

cudaError_t launch_validate(const ValidateArgs& a, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(a.error_count, 0, sizeof(int32_t), s);
  if (e != cudaSuccess || a.batch == 0) return e;
  validate_kernel<<<(a.batch + 127) / 128, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace pa
