// Batched GQA decode attention over a paged KV cache (sm_103a).
//
// Semantics (nano-vLLM learning note, Attention.forward and prepare_decode
// listings): each request's single query attends to all context_lens[b] keys
// of its block table, after this step's KV write.
//
// Design (HBM-bound):
//   * The keys of all requests are cut into chunks of T tokens (T divides the
//     page size, so a chunk lies inside one page and is one contiguous run of
//     T * Hkv * head_dim elements).  The global chunk list is split evenly
//     over the CTAs of one wave ("plan" kernel), so every SM streams the same
//     number of bytes whatever the length mix.  A request cut across CTAs
//     gets per-CTA (o, log2-sum-exp) partials, merged by a second kernel
//     (split-KV / flash-decoding).  The cut depends only on context_lens, so
//     results are bitwise independent of physical page ids.
//   * One producer warp issues 1-D bulk async copies (TMA engine) of each
//     chunk's K and V rows into a 3-stage shared-memory ring, with mbarrier
//     completion and an evict-first L2 hint.  Its 32 lanes look up block-table
//     entries for 32 chunks at a time.
//   * One consumer warp per kv-head reads its head's rows of the chunk, so
//     one K/V byte feeds all G q-heads of the group.  Two consumers:
//     - CUDA cores (fp32, or head_dim 64): each lane owns 16
//       bytes of a row; dot products use packed fp32x2 FMA, partial sums are
//       reduced with a halving butterfly of warp shuffles, the online
//       softmax runs in base 2 with the scale folded into q.
//     - tensor cores (bf16, head_dim 128, any group of up to 8): per 16-token
//       chunk, S = Q K^T and O += P V as mma.sync m16n8k16 with the group's
//       q-heads as the (zero-padded) 16 rows; K and V fragments come by
//       ldmatrix from stage rows padded by 16 bytes (each row its own copy),
//       so the loads are free of bank conflicts.  Far fewer instructions per
//       byte: the CUDA-core consumer is issue-bound from G = 4 on.
//   * Every wait is bounded (pa::mbar_wait_bounded): a kernel never hangs.
#include <math.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kTPL = 4;          // tokens per lane per chunk
constexpr int kStages = 3;       // shared-memory ring depth (CUDA-core consumers, up to two CTAs per SM)
constexpr int kStagesMma = 3;    // ring depth of the tensor-core consumers (one CTA per SM)
constexpr int kMmaTok = 16;      // tokens per chunk of the tensor-core consumers
constexpr int kPlanThreads = 1024;
constexpr int kInlinePlanMax = 512;  // batches the decode CTAs plan themselves (else a plan kernel runs first)
constexpr int kMergeThreads = 128;

__host__ __device__ constexpr int ilog2c(int x) { return x <= 1 ? 0 : 1 + ilog2c(x / 2); }
__host__ __device__ constexpr int pow2ceil(int x) { return x <= 1 ? 1 : 2 * pow2ceil((x + 1) / 2); }

template <typename T, int HD>
struct Geom {
  static constexpr int E = sizeof(T);
  static constexpr int DPL = 16 / E;      // elements a lane holds of one row
  static constexpr int NPR = DPL / 2;     // float2 pairs per lane
  static constexpr int LPR = HD / DPL;    // lanes covering one head row
  static constexpr int RPI = 32 / LPR;    // rows one warp instruction covers
  static constexpr int TOK = kTPL * RPI;  // tokens per chunk
  static constexpr int RB = HD * E;       // bytes of one head row
};

struct KParams {
  const char* q;
  const char* k_cache;
  const char* v_cache;
  const int32_t* bt;
  const int32_t* ctx;
  char* out;
  float* o_part;
  float* lse_part;
  int32_t* cs;       // [B+1] chunk prefix sums
  int32_t* cta_seq;  // [n_ctas] first request of each CTA
  unsigned int* err;
  int64_t num_pages;
  int32_t B, Hq, Hkv, P, maxp, max_ctx, n_ctas;
  int32_t log2P, log2T;
  int32_t row_bytes;    // Hkv * HD * E, one token of the cache
  int32_t row_pitch;    // shared-memory bytes per token row of a stage (row_bytes, + 16 for the MMA consumers)
  int32_t chunk_bytes;  // T * row_pitch
  uint32_t off_bar, off_meta, off_p, off_alpha, off_ml, off_abort;
  uint32_t off_cs;      // [kInlinePlanMax + 1] chunk prefix sums, then [32] warp totals (inline plan)
  int32_t inline_plan;  // 1: no plan kernel ran; every CTA computes the prefix sums itself
  int32_t p_row;        // floats per token row of the probability tile
  float scale_log2;     // softmax scale * log2(e)
  int32_t merge_w;      // warps per (request, q-head) in the merge kernel: 1, 2 or 4
  // Fused KV write (k_new != nullptr): the new token of request b is row b of
  // k_new / v_new; it is attended from there and stored into its cache slot
  // (position context_lens[b] - 1) by the CTA that owns the request's last chunk.
  const char* k_new;
  const char* v_new;
  int64_t k_new_stride, v_new_stride;  // bytes
  int64_t* slot_out;                   // optional: the slot written for request b
};

// First request whose chunks extend past chunk x0 (cs: the prefix sums).
__device__ __forceinline__ int first_request(const int32_t* cs, int B, int64_t x0) {
  int lo = 0, hi = B;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (cs[mid + 1] > x0) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// plan: chunk prefix sums and each CTA's first request
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const KParams p) {
  __shared__ int32_t warp_tot[kPlanThreads / 32];
  __shared__ int32_t carry;
  pdl_trigger();  // the decode kernel may start launching; it waits for this plan
  const int tid = threadIdx.x;
  const int T = 1 << p.log2T;
  const int cap = static_cast<int>(min(static_cast<int64_t>(p.max_ctx), static_cast<int64_t>(p.maxp) << p.log2P));
  if (tid == 0) carry = 0;
  cta_sync();
  for (int base = 0; base < p.B; base += kPlanThreads) {
    const int b = base + tid;
    int cnt = 0;
    if (b < p.B) {
      const int L = p.ctx[b];
      if (L >= 1 && L <= cap) {
        cnt = (L + T - 1) >> p.log2T;
      } else {
        // length 0 is a padding row: nothing is read, stored or written for it
        if (L != 0) raise_flag(p.err, PA_DEVERR_BAD_LENGTH);
        if (p.k_new != nullptr && p.slot_out) p.slot_out[b] = -1;
      }
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if ((tid & 31) >= o) x += y;
    }
    if ((tid & 31) == 31) warp_tot[tid >> 5] = x;
    cta_sync();
    if (tid < 32) {
      int w = warp_tot[tid];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (tid >= o) w += y;
      }
      warp_tot[tid] = w;
    }
    cta_sync();
    const int incl = x + ((tid >> 5) ? warp_tot[(tid >> 5) - 1] : 0) + carry;
    if (b < p.B) p.cs[b + 1] = incl;
    cta_sync();
    if (tid == kPlanThreads - 1) carry = incl;
    cta_sync();
  }
  if (tid == 0) p.cs[0] = 0;
  cta_sync();
  const int NC = carry;
  for (int c = tid; c < p.n_ctas; c += kPlanThreads)
    p.cta_seq[c] = first_request(p.cs, p.B, (static_cast<int64_t>(c) * NC) / p.n_ctas);
}

// The plan kernel's prefix sums, computed by every thread of a decode CTA into
// its shared memory (B <= kInlinePlanMax): each thread sums the chunk counts
// of a run of consecutive requests, the runs' totals are scanned across the
// CTA, then each thread writes its run's prefix sums.  CTA 0 also does the
// plan kernel's side work: it publishes the sums for the merge kernel, flags
// bad lengths and marks the slots of rows it skips.
__device__ __forceinline__ void plan_in_cta(const KParams& p, int32_t* cs_s, int32_t* warp_tot, bool first) {
  const int nthr = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = 1 << p.log2T;
  const int cap = static_cast<int>(min(static_cast<int64_t>(p.max_ctx), static_cast<int64_t>(p.maxp) << p.log2P));
  const int per = (p.B + nthr - 1) / nthr;
  const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
  int sum = 0;
  for (int b = b0; b < b1; ++b) {
    const int L = p.ctx[b];
    int cnt = 0;
    if (L >= 1 && L <= cap) {
      cnt = (L + T - 1) >> p.log2T;
    } else if (first) {
      // length 0 is a padding row: nothing is read, stored or written for it
      if (L != 0) raise_flag(p.err, PA_DEVERR_BAD_LENGTH);
      if (p.k_new != nullptr && p.slot_out) p.slot_out[b] = -1;
    }
    cs_s[b + 1] = cnt;
    sum += cnt;
  }
  int x = sum;  // inclusive scan of the runs' totals: within the warp, then over the warps
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  cta_sync();
  if (warp == 0) {
    int w = lane < (nthr >> 5) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_tot[lane] = w;
  }
  cta_sync();
  int run = x - sum + (warp ? warp_tot[warp - 1] : 0);
  for (int b = b0; b < b1; ++b) {
    run += cs_s[b + 1];
    cs_s[b + 1] = run;
  }
  if (tid == 0) cs_s[0] = 0;
  cta_sync();
  if (first)
    for (int b = tid; b <= p.B; b += nthr) p.cs[b] = cs_s[b];
}

// ---------------------------------------------------------------------------
// halving butterfly: reduce CUR values over the lanes of a row group, keeping
// half of the (partially summed) values per step.
// ---------------------------------------------------------------------------
template <int CUR, int M>
struct Butterfly {
  template <int N>
  static PA_DEVINL void run(float (&a)[N], int lane) {
    if constexpr (CUR >= 2) {
      constexpr int H = CUR / 2;
      const bool upper = (lane & M) != 0;
#pragma unroll
      for (int u = 0; u < H; ++u) {
        const float send = upper ? a[u] : a[u + H];
        const float keep = upper ? a[u + H] : a[u];
        a[u] = keep + __shfl_xor_sync(0xffffffffu, send, M);
      }
      if constexpr (M > 1) Butterfly<H, M / 2>::run(a, lane);
    } else {
      a[0] += __shfl_xor_sync(0xffffffffu, a[0], M);
      if constexpr (M > 1) Butterfly<1, M / 2>::run(a, lane);
    }
  }
};

// The halving levels of Butterfly alone (CUR values -> 1 over lane bits M,
// M/2, ...), for reducing a sub-array whose levels come first.
template <int CUR, int M>
struct Halve {
  template <int N>
  static PA_DEVINL void run(float (&a)[N], int lane) {
    if constexpr (CUR >= 2) {
      static_assert(M >= 1, "one lane bit per halving level");
      constexpr int H = CUR / 2;
      const bool upper = (lane & M) != 0;
#pragma unroll
      for (int u = 0; u < H; ++u) {
        const float send = upper ? a[u] : a[u + H];
        const float keep = upper ? a[u + H] : a[u];
        a[u] = keep + __shfl_xor_sync(0xffffffffu, send, M);
      }
      Halve<H, M / 2>::run(a, lane);
    }
  }
};

// Floats per token row of the probability tile: each probability is stored
// twice, (p, p), so that the PV products read ready-made fp32 pairs, and the
// row is padded to whole 16-byte vectors.
__host__ __device__ constexpr int p_row_floats(int G) { return 2 * (G <= 2 ? 2 : G <= 4 ? 4 : 8); }

template <typename T, int NPR>
PA_DEVINL void unpack16(const uint4 w, float2 (&f)[NPR]) {
  if constexpr (sizeof(T) == 2) {
    f[0] = bf16x2_to_float2(w.x);
    f[1] = bf16x2_to_float2(w.y);
    f[2] = bf16x2_to_float2(w.z);
    f[3] = bf16x2_to_float2(w.w);
  } else {
    f[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
    f[1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
  }
}

template <typename T, int NPR>
PA_DEVINL uint4 pack16(const float2 (&f)[NPR], float s) {
  uint4 w;
  if constexpr (sizeof(T) == 2) {
    w.x = pack_bf16x2(f[0].x * s, f[0].y * s);
    w.y = pack_bf16x2(f[1].x * s, f[1].y * s);
    w.z = pack_bf16x2(f[2].x * s, f[2].y * s);
    w.w = pack_bf16x2(f[3].x * s, f[3].y * s);
  } else {
    w.x = __float_as_uint(f[0].x * s);
    w.y = __float_as_uint(f[0].y * s);
    w.z = __float_as_uint(f[1].x * s);
    w.w = __float_as_uint(f[1].y * s);
  }
  return w;
}

// Time-only bounded wait used when draining copies after an abort.
PA_DEVINL void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// ---------------------------------------------------------------------------
// tensor-core consumer (bf16, head_dim 128, up to 8 q-heads per kv-head)
// ---------------------------------------------------------------------------
// mma.sync fragments (PTX ISA, m16n8k16 with .row.col): lane l is
// in row group gq = l / 4 and thread-in-group tq = l % 4.  A holds rows gq and
// gq + 8; B holds column gq; C holds rows gq (c0, c1) and gq + 8 (c2, c3) at
// columns 2 tq, 2 tq + 1.  Here the rows are the group's q-heads (G <= 8 of
// them, padded to 16 with zero rows), so only c0 / c1 of lanes with gq < G
// carry results.
PA_DEVINL void mma_16816(float (&d)[2], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  [[maybe_unused]] float x2, x3;  // rows gq + 8 (padding), discarded
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %10, %10};"
      : "+f"(d[0]), "+f"(d[1]), "=f"(x2), "=f"(x3)
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.f));
}

// 2^x on the special-function unit (PTX ex2.approx; x <= 0 here).
PA_DEVINL float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


// Four 8x8 b16 matrices from shared memory; lanes 8i .. 8i+7 give the row
// addresses of matrix i.  .trans delivers each matrix transposed.
PA_DEVINL void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

PA_DEVINL void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// The consumer warp of kv-head `warp` for the chunks [x0, x1) of CTA c: per
// 16-token chunk, S = Q K^T as 16 m16n8k16 MMAs in two chains (K^T fragments
// by ldmatrix from the padded stage rows), the online softmax in base 2 on
// the S fragments, and O += P V as 16 m16n8k16 MMAs (P straight from the S
// fragments, V fragments by transposed ldmatrix).  Same results contract as the CUDA-core
// consumer: whole requests to `out`, shares to the partial slots.
template <int G, int NS>
PA_DEVINL void mma_consumer(const KParams& p, unsigned char* smem, uint64_t* full, uint64_t* empty, const int4* meta,
                            volatile int* abort_flag, int x0, int x1, int c) {
  constexpr int RB = 256;  // bytes of one head row (128 bf16)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = warp;
  const int gq = lane >> 2, tq = lane & 3;
  const bool row_live = gq < G;
  const int lrow = lane & 7, lmat = lane >> 3;  // ldmatrix: this lane's row and matrix
  const uint32_t smem0 = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  uint32_t qa[8][2];  // A fragments of q for k-steps of 16 dims: dims 2tq.. and 2tq+8.. of row gq
  float o[16][2];     // O row gq, columns 8j + 2tq, 8j + 2tq + 1
  float m_run = -INFINITY, l_part = 0.f;
  int b = 0;
  uint4 nrow = make_uint4(0, 0, 0, 0);  // this head's piece of the request's new K (lanes 0-15) / V row

  for (int x = x0, it = 0; x < x1; ++x, ++it) {
    const int s = it % NS;
    if (!mbar_wait_bounded(&full[s], (it / NS) & 1, abort_flag, p.err)) break;
    const int4 md = meta[s];
    b = md.x;
    const int n = md.y, flags = md.z;

    if (flags & 1) {  // first chunk of this CTA's share of request b
      if ((flags & 16) && p.k_new != nullptr)  // the share ends the request: its new row, early
        nrow = *reinterpret_cast<const uint4*>(
            (lane < 16 ? p.k_new + static_cast<int64_t>(b) * p.k_new_stride
                       : p.v_new + static_cast<int64_t>(b) * p.v_new_stride) + h * RB + (lane & 15) * 16);
      const char* qrow = p.q + (static_cast<int64_t>(b) * p.Hq + h * G + (row_live ? gq : 0)) * RB;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qa[ks][0] = row_live ? *reinterpret_cast<const uint32_t*>(qrow + (ks * 16 + 2 * tq) * 2) : 0u;
        qa[ks][1] = row_live ? *reinterpret_cast<const uint32_t*>(qrow + (ks * 16 + 8 + 2 * tq) * 2) : 0u;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = 0.f;
      m_run = -INFINITY;
      l_part = 0.f;
    }

    unsigned char* kst = smem + static_cast<size_t>(s) * 2 * p.chunk_bytes + h * RB;
    unsigned char* vst = kst + p.chunk_bytes;
    if (md.w >= 0) {
      // fused KV write: this head's piece of the new row (row n - 1), read by
      // the consumer from k_new / v_new at the start of the share (not copied
      // by the producer, so they may be in pinned host memory), goes into the
      // stage for the products and to its slot
      const int64_t dst_off = static_cast<int64_t>(md.w) * p.row_bytes + h * RB;
      *reinterpret_cast<uint4*>((lane < 16 ? kst : vst) + (n - 1) * p.row_pitch + (lane & 15) * 16) = nrow;
      char* dst = const_cast<char*>(lane < 16 ? p.k_cache : p.v_cache) + dst_off + (lane & 15) * 16;
      stg16(dst, nrow);
    }
    if (n < kMmaTok) {
      // a ragged chunk: the V rows past its end meet probability 0 and must be
      // finite (they may hold another chunk's data or nothing yet)
      for (int r = n; r < kMmaTok; ++r)
        if (lane < 16) *reinterpret_cast<uint4*>(vst + r * p.row_pitch + lane * 16) = make_uint4(0, 0, 0, 0);
    }
    if (md.w >= 0 || n < kMmaTok) {
      // the fence orders these stores before the copies that refill the stage later
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }

    // S = Q K^T for the chunk's tokens 0-7 (s0) and 8-15 (s1): row gq, tokens
    // 2tq, 2tq + 1 (+ 8); two independent accumulator chains
    const uint32_t ka = smem0 + static_cast<uint32_t>(kst - smem) + lrow * p.row_pitch + lmat * 16;
    const uint32_t ka8 = ka + 8 * p.row_pitch;
    float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t bf[4], bg[4];
      ldsm_x4(bf, ka + kk * 64);
      ldsm_x4(bg, ka8 + kk * 64);
      mma_16816(s0, qa[2 * kk][0], qa[2 * kk][1], bf[0], bf[1]);
      mma_16816(s1, qa[2 * kk][0], qa[2 * kk][1], bg[0], bg[1]);
      mma_16816(s0, qa[2 * kk + 1][0], qa[2 * kk + 1][1], bf[2], bf[3]);
      mma_16816(s1, qa[2 * kk + 1][0], qa[2 * kk + 1][1], bg[2], bg[3]);
    }
    const int tk = 2 * tq;
    const float v0 = tk < n ? s0[0] * p.scale_log2 : -INFINITY;
    const float v1 = tk + 1 < n ? s0[1] * p.scale_log2 : -INFINITY;
    const float v2 = tk + 8 < n ? s1[0] * p.scale_log2 : -INFINITY;
    const float v3 = tk + 9 < n ? s1[1] * p.scale_log2 : -INFINITY;
    float mx = fmaxf(fmaxf(v0, v1), fmaxf(v2, v3));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = ex2_approx(m_run - m_use);
    const float p0 = ex2_approx(v0 - m_use), p1 = ex2_approx(v1 - m_use);
    const float p2 = ex2_approx(v2 - m_use), p3 = ex2_approx(v3 - m_use);
    l_part = l_part * alpha + ((p0 + p1) + (p2 + p3));
    if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= alpha;
        o[j][1] *= alpha;
      }
    }
    m_run = m_new;

    // O += P V (m16n8k16: k = the chunk's 16 tokens); matrices of the
    // transposed loads: tokens 0-7 / 8-15 x dims d .. d+7 / d+8 .. d+15
    const uint32_t pa0 = pack_bf16x2(p0, p1), pa2 = pack_bf16x2(p2, p3);
    const uint32_t va = smem0 + static_cast<uint32_t>(vst - smem) + (lrow + (lmat & 1) * 8) * p.row_pitch +
                        (lmat >> 1) * 16;
#pragma unroll
    for (int nn = 0; nn < 8; ++nn) {
      uint32_t bf[4];
      ldsm_x4_t(bf, va + nn * 32);
      mma_16816(o[2 * nn], pa0, pa2, bf[0], bf[1]);
      mma_16816(o[2 * nn + 1], pa0, pa2, bf[2], bf[3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    if (flags & 2) {  // last chunk of the share: write the result
      float l = l_part + __shfl_xor_sync(0xffffffffu, l_part, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if (row_live) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int hq = h * G + gq;
        if (flags & 4) {
          char* dst = p.out + (static_cast<int64_t>(b) * p.Hq + hq) * RB + tq * 4;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            *reinterpret_cast<uint32_t*>(dst + j * 16) = pack_bf16x2(o[j][0] * inv, o[j][1] * inv);
        } else {
          const int64_t slot = static_cast<int64_t>(c) + b;
          float* dst = p.o_part + (slot * p.Hq + hq) * 128 + 2 * tq;
#pragma unroll
          for (int j = 0; j < 16; ++j) *reinterpret_cast<float2*>(dst + 8 * j) = make_float2(o[j][0] * inv, o[j][1] * inv);
          if (tq == 0) p.lse_part[slot * p.Hq + hq] = l > 0.f ? m_run + log2f(l) : -INFINITY;
        }
      }
      __syncwarp();
    }
  }
}

// ---------------------------------------------------------------------------
// the split-KV decode kernel
// ---------------------------------------------------------------------------
// The bf16 head_dim-128 kernels run their products on the tensor cores (see
// the MMA consumer below); fp32 and head_dim 64 on the CUDA cores.
template <typename T, int HD, int G>
constexpr bool kUseMma = std::is_same<T, __nv_bfloat16>::value && HD == 128;

template <typename T, int HD, int G>
// Register cap: a 9-warp CTA is charged as 10 warps, so two CTAs per SM need
// at most 96 registers per thread (CUDA-core consumers, G <= 4); larger groups
// and the tensor-core consumers run one CTA per SM with a deeper ring.
__global__ void __launch_bounds__(9 * 32) __maxnreg__((G <= 4 && !kUseMma<T, HD, G>) ? 96 : 168)
    decode_kernel(const KParams p) {
  constexpr bool kMma = kUseMma<T, HD, G>;
  constexpr int kStages = kMma ? kStagesMma : ::pa::kStages;
  using Gm = Geom<T, HD>;
  constexpr int LPR = Gm::LPR, RPI = Gm::RPI, NPR = Gm::NPR;
  constexpr int V = G * kTPL;
  constexpr int VP = pow2ceil(V);
  constexpr int VF = VP >= LPR ? VP / LPR : 1;          // values a lane keeps
  constexpr int DUP = VP >= LPR ? 0 : ilog2c(LPR / VP);  // low lane bits holding copies
  constexpr int IBITS = ilog2c(kTPL / VF);               // lane bits carrying the token index
  constexpr int GP = VP / kTPL;                          // heads padded to a power of two
  constexpr int PR = p_row_floats(G);
  static_assert(VF <= kTPL, "a lane's values must share one head");
  static_assert(GP <= LPR, "the head levels of the reduction fit in a row's lanes");

  extern __shared__ __align__(128) unsigned char smem[];
  const int c = blockIdx.x;
  const int NW = p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int32_t* cs;  // [B+1] chunk prefix sums
  if (p.inline_plan) {
    int32_t* cs_s = reinterpret_cast<int32_t*>(smem + p.off_cs);
    plan_in_cta(p, cs_s, cs_s + kInlinePlanMax + 1, c == 0);
    cs = cs_s;
  } else {
    pdl_wait();  // the plan kernel's chunk sums and CTA starts are complete
    cs = p.cs;
  }
  pdl_trigger();  // the merge kernel may start launching; it waits for this grid
  const int NC = cs[p.B];
  const int x0 = static_cast<int>((static_cast<int64_t>(c) * NC) / p.n_ctas);
  const int x1 = static_cast<int>((static_cast<int64_t>(c + 1) * NC) / p.n_ctas);
  if (x0 >= x1) return;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* empty = full + kStages;
  int4* meta = reinterpret_cast<int4*>(smem + p.off_meta);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.off_abort);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  cta_sync();

  if (warp == NW) {
    // ------------------------------ producer ------------------------------
    const uint64_t pol = l2_policy_evict_first();
    const int tok = 1 << p.log2T;
    int b = p.inline_plan ? first_request(cs, p.B, x0) : p.cta_seq[c];
    int issued = 0;
    bool aborted = false;
    for (int xg = x0; xg < x1 && !aborted; xg += 32) {
      const int nvalid = min(32, x1 - xg);
      const int x = xg + lane;
      int my_b = b, n = 0, flags = 0, new_slot = -1;
      long long off = 0;
      if (lane < nvalid) {
        while (my_b < p.B - 1 && cs[my_b + 1] <= x) ++my_b;
        const int cb0 = cs[my_b], cb1 = cs[my_b + 1];
        const int jc = x - cb0;
        const int t0 = jc << p.log2T;
        n = min(tok, p.ctx[my_b] - t0);
        const int page = p.bt[static_cast<int64_t>(my_b) * p.maxp + (t0 >> p.log2P)];
        if (page < 0 || page >= p.num_pages) {
          raise_flag(p.err, PA_DEVERR_BAD_PAGE);
          n = 0;
        } else {
          off = ((static_cast<long long>(page) << p.log2P) + (t0 & (p.P - 1))) * p.row_bytes;
        }
        flags = ((x == x0 || jc == 0) ? 1 : 0) | ((x == x1 - 1 || x == cb1 - 1) ? 2 : 0) |
                ((cb0 >= x0 && cb1 <= x1) ? 4 : 0) | ((x == cb1 - 1) ? 8 : 0) | ((cb1 <= x1) ? 16 : 0);
        if (p.k_new != nullptr && (flags & 8) && n >= 1)
          new_slot = static_cast<int>(off / p.row_bytes) + n - 1;  // position context_len - 1
      }
      b = __shfl_sync(0xffffffffu, my_b, nvalid - 1);
      for (int u = 0; u < nvalid; ++u) {
        const int ub = __shfl_sync(0xffffffffu, my_b, u);
        const int un = __shfl_sync(0xffffffffu, n, u);
        const int uf = __shfl_sync(0xffffffffu, flags, u);
        const long long uoff = __shfl_sync(0xffffffffu, off, u);
        const int uslot = __shfl_sync(0xffffffffu, new_slot, u);
        int ok = 1;
        if (lane == 0) {
          const int it = xg - x0 + u;
          const int s = it % kStages;
          if (!mbar_wait_bounded(&empty[s], ((it / kStages) & 1) ^ 1, abort_flag, p.err)) {
            ok = 0;
          } else {
            meta[s] = make_int4(ub, un, uf, uslot);
            const uint32_t bytes = static_cast<uint32_t>(un) * static_cast<uint32_t>(p.row_bytes);
            // tensor-core consumers read the new token's row themselves
            const uint32_t copied = kMma && uslot >= 0 ? bytes - static_cast<uint32_t>(p.row_bytes) : bytes;
            mbar_arrive_expect_tx(&full[s], 2 * copied);
            unsigned char* dst = smem + static_cast<size_t>(s) * 2 * p.chunk_bytes;
            if constexpr (kMma) {
              // the row copies are issued by the whole warp below
              if (uslot >= 0 && p.slot_out) p.slot_out[ub] = uslot;
            } else if (uslot >= 0) {
              // the cached rows of the chunk, then the new token's row from k_new / v_new
              const uint32_t cached = bytes - p.row_bytes;
              if (cached) {
                bulk_g2s_hint(dst, p.k_cache + uoff, cached, &full[s], pol);
                bulk_g2s_hint(dst + p.chunk_bytes, p.v_cache + uoff, cached, &full[s], pol);
              }
              bulk_g2s(dst + cached, p.k_new + ub * p.k_new_stride, p.row_bytes, &full[s]);
              bulk_g2s(dst + p.chunk_bytes + cached, p.v_new + ub * p.v_new_stride, p.row_bytes, &full[s]);
              if (p.slot_out) p.slot_out[ub] = uslot;
            } else if (bytes) {
              bulk_g2s_hint(dst, p.k_cache + uoff, bytes, &full[s], pol);
              bulk_g2s_hint(dst + p.chunk_bytes, p.v_cache + uoff, bytes, &full[s], pol);
            }
            if (p.k_new != nullptr && (uf & 8) && uslot < 0 && p.slot_out) p.slot_out[ub] = -1;
            ++issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          aborted = true;
          break;
        }
        if constexpr (kMma) {
          // one copy per token row into rows of row_pitch bytes (the pad keeps
          // the MMA consumers' fragment loads free of bank conflicts): lane r
          // copies K row r, lane 16 + r V row r; the new token's row is read
          // by the consumers from k_new / v_new
          __syncwarp();
          const int s = (xg - x0 + u) % kStages;
          unsigned char* dst = smem + static_cast<size_t>(s) * 2 * p.chunk_bytes;
          const int r = lane & 15;
          const bool isv = lane >= 16;
          if (r < un && !(uslot >= 0 && r == un - 1)) {
            unsigned char* d = dst + (isv ? p.chunk_bytes : 0) + r * p.row_pitch;
            const char* src = (isv ? p.v_cache : p.k_cache) + uoff + static_cast<int64_t>(r) * p.row_bytes;
            bulk_g2s_hint(d, src, p.row_bytes, &full[s], pol);
          }
        }
      }
    }
    if (aborted && lane == 0) {
      // Copies already issued may still be landing: wait for them (time only).
      for (int it = max(0, issued - kStages); it < issued; ++it)
        drain_wait(&full[it % kStages], (it / kStages) & 1);
    }
    return;
  }

  // ------------------------------- consumers -------------------------------
  if constexpr (kMma) {
    mma_consumer<G, kStages>(p, smem, full, empty, meta, abort_flag, x0, x1, c);
    return;
  }
  const int h = warp;
  const int rs = lane / LPR, j = lane % LPR;
  const int vbase = (j >> DUP) * VF;
  const int g_l = vbase / kTPL;          // head of the lane's kept values
  const int i_l0 = vbase % kTPL;         // token index of its first kept value
  const bool writer = (j & ((1 << DUP) - 1)) == 0;
  const bool head_leader = writer && rs == 0 && (((j >> DUP) & ((1 << IBITS) - 1)) == 0) && g_l < G;
  float* p_tile = reinterpret_cast<float*>(smem + p.off_p) + warp * Gm::TOK * PR;
  float* alpha_s = reinterpret_cast<float*>(smem + p.off_alpha) + warp * 8;
  float* ml_s = reinterpret_cast<float*>(smem + p.off_ml) + warp * 16;

  float2 qf[G][NPR];
  float2 o[G][NPR];
  float m_run = -INFINITY, l_run = 0.f;

  for (int x = x0, it = 0; x < x1; ++x, ++it) {
    const int s = it % kStages;
    if (!mbar_wait_bounded(&full[s], (it / kStages) & 1, abort_flag, p.err)) break;
    const int4 md = meta[s];
    const int b = md.x, n = md.y, flags = md.z;

    if (flags & 1) {  // first chunk of this CTA's share of request b
      const char* qb = p.q + (static_cast<int64_t>(b) * p.Hq + h * G) * Gm::RB + j * 16;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float2 f[NPR];
        unpack16<T, NPR>(ldg16(qb + g * Gm::RB), f);
#pragma unroll
        for (int r = 0; r < NPR; ++r) {
          qf[g][r] = make_float2(f[r].x * p.scale_log2, f[r].y * p.scale_log2);
          o[g][r] = make_float2(0.f, 0.f);
        }
      }
      m_run = -INFINITY;
      l_run = 0.f;
    }

    const unsigned char* kbuf = smem + static_cast<size_t>(s) * 2 * p.chunk_bytes + h * Gm::RB + j * 16;
    const unsigned char* vbuf = kbuf + p.chunk_bytes;
    if (md.w >= 0) {
      // fused KV write: this head's 16-byte pieces of the new row go to its slot
      // (row slots of the warp take K and V in turn)
      const int64_t dst_off = static_cast<int64_t>(md.w) * p.row_bytes + h * Gm::RB + j * 16;
      const int src_off = (n - 1) * p.row_pitch;
      for (int part = rs; part < 2; part += RPI) {
        const unsigned char* src = (part == 0 ? kbuf : vbuf) + src_off;
        char* dst = const_cast<char*>(part == 0 ? p.k_cache : p.v_cache) + dst_off;
        stg16(dst, *reinterpret_cast<const uint4*>(src));
      }
    }

    // scores: partial dot products over this lane's 16 bytes of each row,
    // reduced over the row's lanes by a halving butterfly.  The score of
    // (head g, token i) is value g * kTPL + i, and the butterfly halves the
    // highest value bit first, so its first log2(GP) levels pair heads of one
    // token: they run per token, right after that token's products.
    float a[kTPL];
#pragma unroll
    for (int i = 0; i < kTPL; ++i) {
      const int t = i * RPI + rs;
      float2 kf[NPR];
      unpack16<T, NPR>(*reinterpret_cast<const uint4*>(kbuf + t * p.row_pitch), kf);
      float b[GP];
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        if (g < G) {
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int r = 0; r < NPR; ++r) acc = ffma2(qf[g][r], kf[r], acc);
          b[g] = acc.x + acc.y;
        } else {
          b[g] = 0.f;
        }
      }
      Halve<GP, LPR / 2>::run(b, lane);
      a[i] = b[0];
    }
    if constexpr (LPR / (2 * GP) >= 1) Butterfly<kTPL, LPR / (2 * GP)>::run(a, lane);

    // online softmax (base 2) for the lane's head
    float sc[VF];
    float mc = -INFINITY;
#pragma unroll
    for (int u = 0; u < VF; ++u) {
      const int t = (i_l0 + u) * RPI + rs;
      sc[u] = t < n ? a[u] : -INFINITY;
      mc = fmaxf(mc, sc[u]);
    }
#pragma unroll
    for (int k = 0; k < IBITS; ++k) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, 1 << (DUP + k)));
#pragma unroll
    for (int msk = LPR; msk < 32; msk <<= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, msk));
    const float m_new = fmaxf(m_run, mc);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = exp2f(m_run - m_use);
    float psum = 0.f;
#pragma unroll
    for (int u = 0; u < VF; ++u) {
      const float pv = exp2f(sc[u] - m_use);
      psum += pv;
      if (writer && g_l < G)
        *reinterpret_cast<float2*>(p_tile + ((i_l0 + u) * RPI + rs) * PR + 2 * g_l) = make_float2(pv, pv);
    }
    l_run = l_run * alpha + psum;
    m_run = m_new;
    if (head_leader) alpha_s[g_l] = alpha;
    __syncwarp();

    bool rescale = false;
    float al[G];
#pragma unroll
    for (int g4 = 0; g4 < G; g4 += 4) {
      const float4 a4 = *reinterpret_cast<const float4*>(alpha_s + g4);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
      for (int g = g4; g < G && g < g4 + 4; ++g) {
        al[g] = av[g - g4];
        rescale |= al[g] != 1.f;
      }
    }
    if (rescale) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int r = 0; r < NPR; ++r) o[g][r] = fmul2(o[g][r], make_float2(al[g], al[g]));
    }

    // o += p * V for this lane's 16 bytes of each row
#pragma unroll
    for (int i = 0; i < kTPL; ++i) {
      const int t = i * RPI + rs;
      if (t < n) {
        float2 vf[NPR];
        unpack16<T, NPR>(*reinterpret_cast<const uint4*>(vbuf + t * p.row_pitch), vf);
        const float4* prow = reinterpret_cast<const float4*>(p_tile + t * PR);
#pragma unroll
        for (int g2 = 0; g2 < G; g2 += 2) {
          const float4 pv2 = prow[g2 / 2];  // (p_g, p_g, p_g+1, p_g+1)
          const float2 pp0 = make_float2(pv2.x, pv2.y);
#pragma unroll
          for (int r = 0; r < NPR; ++r) o[g2][r] = ffma2(pp0, vf[r], o[g2][r]);
          if (g2 + 1 < G) {
            const float2 pp1 = make_float2(pv2.z, pv2.w);
#pragma unroll
            for (int r = 0; r < NPR; ++r) o[g2 + 1][r] = ffma2(pp1, vf[r], o[g2 + 1][r]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    if (flags & 2) {  // last chunk of the share: write the result
#pragma unroll
      for (int msk = LPR; msk < 32; msk <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int r = 0; r < NPR; ++r) {
            o[g][r].x += __shfl_xor_sync(0xffffffffu, o[g][r].x, msk);
            o[g][r].y += __shfl_xor_sync(0xffffffffu, o[g][r].y, msk);
          }
      float lt = l_run;
#pragma unroll
      for (int k = 0; k < IBITS; ++k) lt += __shfl_xor_sync(0xffffffffu, lt, 1 << (DUP + k));
#pragma unroll
      for (int msk = LPR; msk < 32; msk <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, msk);
      if (head_leader) {
        ml_s[2 * g_l] = m_run;
        ml_s[2 * g_l + 1] = lt;
      }
      __syncwarp();
      if (rs == 0) {
        const bool whole = (flags & 4) != 0;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float mg = ml_s[2 * g], lg = ml_s[2 * g + 1];
          const float inv = lg > 0.f ? 1.f / lg : 0.f;
          const int hq = h * G + g;
          if (whole) {
            char* dst = p.out + (static_cast<int64_t>(b) * p.Hq + hq) * Gm::RB + j * 16;
            stg16(dst, pack16<T, NPR>(o[g], inv));
          } else {
            const int64_t slot = static_cast<int64_t>(c) + b;
            float* dst = p.o_part + (slot * p.Hq + hq) * HD + j * Gm::DPL;
#pragma unroll
            for (int r = 0; r < NPR; r += 2)
              *reinterpret_cast<float4*>(dst + 2 * r) =
                  make_float4(o[g][r].x * inv, o[g][r].y * inv, o[g][r + 1].x * inv, o[g][r + 1].y * inv);
            if (j == 0) p.lse_part[slot * p.Hq + hq] = lg > 0.f ? mg + log2f(lg) : -INFINITY;
          }
        }
      }
      __syncwarp();
    }
  }
}

// ---------------------------------------------------------------------------
// log-sum-exp merge of the partials of requests cut across CTAs.  merge_w
// warps per (request, q-head): each takes a contiguous range of the partials,
// a lane owns HD/32 elements of the head, the partials' weights are computed
// one per lane and eight partials' loads are in flight together; the warps'
// sums meet in shared memory and are added in a fixed order.
// ---------------------------------------------------------------------------
template <typename T, int HD>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const KParams p) {
  constexpr int EL = HD / 32;  // elements per lane
  constexpr int NWARP = kMergeThreads / 32;
  __shared__ float red[NWARP][32][EL + 1];
  pdl_wait();                  // every partial of the decode grid is written
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = p.merge_w, item = warp / W, sub = warp - item * W;
  const int64_t u = static_cast<int64_t>(blockIdx.x) * (NWARP / W) + item;
  // The W warps of an item decide together; no warp leaves before the CTA
  // barrier below (merge_w, and so the barrier, is the same for every CTA).
  int b = 0, hq = 0, c0 = 0, parts = 0, NC = 0;
  bool active = u < static_cast<int64_t>(p.B) * p.Hq;
  if (active) {
    b = static_cast<int>(u / p.Hq);
    hq = static_cast<int>(u - static_cast<int64_t>(b) * p.Hq);
    NC = p.cs[p.B];
    const int cb0 = p.cs[b], cb1 = p.cs[b + 1];
    if (cb1 <= cb0) {
      active = false;
    } else {
      c0 = static_cast<int>(((static_cast<int64_t>(cb0) + 1) * p.n_ctas + NC - 1) / NC) - 1;
      const int c1 = static_cast<int>(((static_cast<int64_t>(cb1)) * p.n_ctas + NC - 1) / NC) - 1;
      parts = c1 - c0 + 1;
      active = c0 != c1;  // one CTA wrote the request whole
    }
  }
  // With more CTAs than chunks some CTAs between c0 and c1 own no chunk and
  // wrote no partial: only CTAs with a non-empty range take part.  With at
  // least as many chunks as CTAs every CTA has a range.
  const bool all_busy = NC >= p.n_ctas;
  auto start = [&](int c) { return (static_cast<int64_t>(c) * NC) / p.n_ctas; };
  auto busy = [&](int cc) { return all_busy || start(cc) < start(cc + 1); };
  auto lse_of = [&](int k) { return p.lse_part[(static_cast<int64_t>(c0 + k) + b) * p.Hq + hq]; };
  float acc[EL];
#pragma unroll
  for (int e = 0; e < EL; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (active) {
    float M = -INFINITY;
    for (int k = lane; k < parts; k += 32)
      if (busy(c0 + k)) M = fmaxf(M, lse_of(k));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const int per = (parts + W - 1) / W;
    const int k_begin = sub * per, k_end = min(parts, k_begin + per);
    if (M != -INFINITY) {
      for (int k0 = k_begin; k0 < k_end; k0 += 32) {
        const int k = k0 + lane;
        const float w_mine = k < k_end && busy(c0 + k) ? exp2f(lse_of(k) - M) : 0.f;
        const int kn = min(32, k_end - k0);
#pragma unroll 8
        for (int i = 0; i < kn; ++i) {
          const float w = __shfl_sync(0xffffffffu, w_mine, i);
          const int64_t slot = static_cast<int64_t>(c0 + k0 + i) + b;
          const float* src = p.o_part + (slot * p.Hq + hq) * HD + lane * EL;
          if (w != 0.f) {
            if constexpr (EL == 4) {
              const float4 ov = *reinterpret_cast<const float4*>(src);
              acc[0] += w * ov.x;
              acc[1] += w * ov.y;
              acc[2] += w * ov.z;
              acc[3] += w * ov.w;
            } else {
              const float2 ov = *reinterpret_cast<const float2*>(src);
              acc[0] += w * ov.x;
              acc[1] += w * ov.y;
            }
            wsum += w;
          }
        }
      }
    }
  }
  if (W > 1) {
#pragma unroll
    for (int e = 0; e < EL; ++e) red[warp][lane][e] = acc[e];
    red[warp][lane][EL] = wsum;
    cta_sync();
    if (sub != 0) return;
    for (int w2 = 1; w2 < W; ++w2) {
#pragma unroll
      for (int e = 0; e < EL; ++e) acc[e] += red[warp + w2][lane][e];
      wsum += red[warp + w2][lane][EL];
    }
  }
  if (!active) return;
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int64_t e0 = (static_cast<int64_t>(b) * p.Hq + hq) * HD + lane * EL;
  if constexpr (sizeof(T) == 2) {
    if constexpr (EL == 4) {
      *reinterpret_cast<uint2*>(p.out + e0 * 2) =
          make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
    } else {
      *reinterpret_cast<uint32_t*>(p.out + e0 * 2) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
  } else {
    if constexpr (EL == 4) {
      *reinterpret_cast<float4*>(p.out + e0 * 4) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    } else {
      *reinterpret_cast<float2*>(p.out + e0 * 4) = make_float2(acc[0] * inv, acc[1] * inv);
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct Fns {
  const void* main = nullptr;
  const void* merge = nullptr;
};

template <typename T, int HD>
Fns fns_for_g(int G) {
  switch (G) {
    case 1: return {reinterpret_cast<const void*>(decode_kernel<T, HD, 1>), reinterpret_cast<const void*>(decode_merge_kernel<T, HD>)};
    case 2: return {reinterpret_cast<const void*>(decode_kernel<T, HD, 2>), reinterpret_cast<const void*>(decode_merge_kernel<T, HD>)};
    case 3: return {reinterpret_cast<const void*>(decode_kernel<T, HD, 3>), reinterpret_cast<const void*>(decode_merge_kernel<T, HD>)};
    case 4: return {reinterpret_cast<const void*>(decode_kernel<T, HD, 4>), reinterpret_cast<const void*>(decode_merge_kernel<T, HD>)};
    case 5: return {reinterpret_cast<const void*>(decode_kernel<T, HD, 5>), reinterpret_cast<const void*>(decode_merge_kernel<T, HD>)};
    case 6: return {reinterpret_cast<const void*>(decode_kernel<T, HD, 6>), reinterpret_cast<const void*>(decode_merge_kernel<T, HD>)};
    case 7: return {reinterpret_cast<const void*>(decode_kernel<T, HD, 7>), reinterpret_cast<const void*>(decode_merge_kernel<T, HD>)};
    case 8: return {reinterpret_cast<const void*>(decode_kernel<T, HD, 8>), reinterpret_cast<const void*>(decode_merge_kernel<T, HD>)};
    default: return {};
  }
}

Fns get_fns(int dtype, int hd, int G) {
  if (dtype == PA_BF16) return hd == 128 ? fns_for_g<__nv_bfloat16, 128>(G) : fns_for_g<__nv_bfloat16, 64>(G);
  return hd == 128 ? fns_for_g<float, 128>(G) : fns_for_g<float, 64>(G);
}

// CTAs of one kernel instance that fit on an SM, cached per (device, kernel, smem).
struct OccKey {
  int device;
  const void* fn;
  int threads;
  size_t smem;
};
std::mutex g_occ_mu;
OccKey g_occ_keys[64];
int g_occ_vals[64];
int g_occ_n = 0;

cudaError_t ctas_per_sm(const DeviceInfo& di, const void* fn, int threads, size_t smem, int* out) {
  {
    std::lock_guard<std::mutex> lk(g_occ_mu);
    for (int i = 0; i < g_occ_n; ++i) {
      const OccKey& k = g_occ_keys[i];
      if (k.device == di.device && k.fn == fn && k.threads == threads && k.smem == smem) {
        *out = g_occ_vals[i];
        return cudaSuccess;
      }
    }
  }
  // The attribute is per kernel, not per launch: raise it to the device's
  // opt-in maximum so every plan's shared-memory size fits.
  cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
  if (e != cudaSuccess) return e;
  // Prefer the largest shared-memory carve-out so that several CTAs fit.
  e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  std::lock_guard<std::mutex> lk(g_occ_mu);
  if (g_occ_n < 64) {
    g_occ_keys[g_occ_n] = {di.device, fn, threads, smem};
    g_occ_vals[g_occ_n] = n;
    ++g_occ_n;
  }
  *out = n;
  return cudaSuccess;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool uses_mma(int dtype, int hd, int /*G*/) { return dtype == PA_BF16 && hd == 128; }

}  // namespace

cudaError_t plan_decode(const pa_cache_desc& d, int batch, int max_ctx, int max_ctas, DecodePlan* out) {
  DeviceInfo di;
  cudaError_t e = current_device_info(&di);
  if (e != cudaSuccess) return e;
  const int E = elem_bytes(d.dtype);
  const int G = d.num_q_heads / d.num_kv_heads;
  const Fns f = get_fns(d.dtype, d.head_dim, G);
  if (!f.main) return cudaErrorInvalidValue;
  const int dpl = 16 / E, lpr = d.head_dim / dpl, rpi = 32 / lpr;
  DecodePlan pl;
  pl.nw = d.num_kv_heads;
  pl.tokens_per_chunk = uses_mma(d.dtype, d.head_dim, G) ? kMmaTok : kTPL * rpi;
  const int row_bytes = d.num_kv_heads * d.head_dim * E;
  pl.row_pitch = uses_mma(d.dtype, d.head_dim, G) ? row_bytes + 16 : row_bytes;
  pl.chunk_bytes = pl.tokens_per_chunk * pl.row_pitch;
  const int stages = uses_mma(d.dtype, d.head_dim, G) ? kStagesMma : kStages;
  pl.stages = stages;
  size_t off = static_cast<size_t>(stages) * 2 * pl.chunk_bytes;
  pl.off_bar = static_cast<uint32_t>(off);
  off += 2 * stages * sizeof(uint64_t);
  pl.off_meta = static_cast<uint32_t>(align_up(off, 16));
  off = pl.off_meta + stages * 16;
  pl.off_abort = static_cast<uint32_t>(off);
  off += 16;
  pl.p_row = p_row_floats(G);
  pl.off_p = static_cast<uint32_t>(align_up(off, 16));
  off = pl.off_p + static_cast<size_t>(pl.nw) * pl.tokens_per_chunk * pl.p_row * 4;
  pl.off_alpha = static_cast<uint32_t>(align_up(off, 16));
  off = pl.off_alpha;
  off += static_cast<size_t>(pl.nw) * 8 * 4;
  pl.off_ml = static_cast<uint32_t>(off);
  off += static_cast<size_t>(pl.nw) * 16 * 4;
  // room for the batch's prefix sums (whatever the batch, so that the CTAs
  // per SM, and with them the plan, do not depend on it)
  pl.off_cs = static_cast<uint32_t>(align_up(off, 16));
  off = pl.off_cs + static_cast<size_t>(kInlinePlanMax + 1 + 32) * 4;
  pl.smem_bytes = align_up(off, 128);
  if (pl.smem_bytes > static_cast<size_t>(di.max_smem_optin)) return cudaErrorInvalidValue;
  int occ = 0;
  e = ctas_per_sm(di, f.main, (pl.nw + 1) * 32, pl.smem_bytes, &occ);
  if (e != cudaSuccess) return e;
  const int64_t chunks_upper =
      static_cast<int64_t>(batch) * ((max_ctx + pl.tokens_per_chunk - 1) / pl.tokens_per_chunk);
  int64_t n = static_cast<int64_t>(occ) * di.sm_count;
  if (max_ctas > 0) n = std::min<int64_t>(n, max_ctas);
  n = std::min<int64_t>(n, std::max<int64_t>(1, chunks_upper));
  pl.n_ctas = static_cast<int>(std::max<int64_t>(1, n));
  size_t w = 0;
  pl.ws_cs = w;
  w = align_up(w + static_cast<size_t>(batch + 1) * 4, 256);
  pl.ws_cta_seq = w;
  w = align_up(w + static_cast<size_t>(pl.n_ctas) * 4, 256);
  pl.ws_lse = w;
  const size_t slots = static_cast<size_t>(pl.n_ctas) + batch;
  w = align_up(w + slots * d.num_q_heads * 4, 256);
  pl.ws_o = w;
  w = align_up(w + slots * d.num_q_heads * d.head_dim * 4, 256);
  pl.ws_bytes = w;
  *out = pl;
  return cudaSuccess;
}

cudaError_t launch_decode(const pa_cache_desc& d, const DecodePlan& pl, const DecodeArgs& a, cudaStream_t s) {
  const int G = d.num_q_heads / d.num_kv_heads;
  const Fns f = get_fns(d.dtype, d.head_dim, G);
  if (!f.main) return cudaErrorInvalidValue;
  char* ws = static_cast<char*>(a.workspace);
  KParams p{};
  p.q = static_cast<const char*>(a.q);
  p.k_cache = static_cast<const char*>(a.k_cache);
  p.v_cache = static_cast<const char*>(a.v_cache);
  p.bt = a.block_tables;
  p.ctx = a.context_lens;
  p.out = static_cast<char*>(a.out);
  p.o_part = reinterpret_cast<float*>(ws + pl.ws_o);
  p.lse_part = reinterpret_cast<float*>(ws + pl.ws_lse);
  p.cs = reinterpret_cast<int32_t*>(ws + pl.ws_cs);
  p.cta_seq = reinterpret_cast<int32_t*>(ws + pl.ws_cta_seq);
  p.err = a.err;
  p.num_pages = d.num_pages;
  p.B = a.batch;
  p.Hq = d.num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.P = d.page_size;
  p.maxp = a.max_pages;
  p.max_ctx = a.max_context_len;
  p.n_ctas = pl.n_ctas;
  p.log2P = 0;
  while ((1 << p.log2P) < d.page_size) ++p.log2P;
  p.log2T = 0;
  while ((1 << p.log2T) < pl.tokens_per_chunk) ++p.log2T;
  p.row_bytes = d.num_kv_heads * d.head_dim * elem_bytes(d.dtype);
  p.row_pitch = pl.row_pitch;
  p.chunk_bytes = pl.chunk_bytes;
  p.off_bar = pl.off_bar;
  p.off_meta = pl.off_meta;
  p.off_p = pl.off_p;
  p.off_alpha = pl.off_alpha;
  p.off_ml = pl.off_ml;
  p.off_abort = pl.off_abort;
  p.off_cs = pl.off_cs;
  p.inline_plan = a.batch <= kInlinePlanMax ? 1 : 0;
  p.p_row = pl.p_row;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.k_new = static_cast<const char*>(a.k_new);
  p.v_new = static_cast<const char*>(a.v_new);
  p.k_new_stride = a.k_new_stride_bytes;
  p.v_new_stride = a.v_new_stride_bytes;
  p.slot_out = a.slot_out;

  // (plan ->) decode -> merge.  Up to kInlinePlanMax requests every decode CTA
  // computes the plan's prefix sums itself, which costs less than a kernel
  // boundary on the step's critical path; beyond, a plan kernel runs first.
  // The kernels after the first are launched to overlap their launch with the
  // kernel before them (each waits for it before reading its output).
  void* args[] = {&p};
  cudaError_t e;
  if (p.inline_plan) {
    e = cudaLaunchKernel(f.main, dim3(pl.n_ctas), dim3((pl.nw + 1) * 32), args, pl.smem_bytes, s);
  } else {
    decode_plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_after_previous(f.main, dim3(pl.n_ctas), dim3((pl.nw + 1) * 32), pl.smem_bytes, s, args);
  }
  if (e != cudaSuccess) return e;
  if (pl.n_ctas > 1) {
    // warps per (request, q-head): about one per 8 partials of a request when
    // the requests are equally long (CTAs per request / 8), at most 4
    const int per_req = pl.n_ctas / std::max(1, a.batch);
    p.merge_w = per_req >= 32 ? 4 : per_req >= 16 ? 2 : 1;
    const int64_t pairs = static_cast<int64_t>(a.batch) * d.num_q_heads;
    const int items = kMergeThreads / 32 / p.merge_w;
    const unsigned blocks = static_cast<unsigned>((pairs + items - 1) / items);
    e = launch_after_previous(f.merge, dim3(blocks), dim3(kMergeThreads), 0, s, args);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace pa
