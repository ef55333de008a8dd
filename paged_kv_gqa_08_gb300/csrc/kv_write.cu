// Slot mapping, KV scatter, and the fused per-head Q/K RMSNorm + RoPE + KV
// scatter (sm_103a).  All three are small, latency- or HBM-bound kernels.
#include <limits.h>
#include <math.h>

#include <algorithm>

#include "pa_common.cuh"

namespace pa {
namespace {

// ---------------------------------------------------------------------------
// slot mapping (nano-vLLM learning note, prepare_prefill / prepare_decode)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) slot_mapping_kernel(const SlotMapParams p) {
  const int b = blockIdx.x;
  const int s0 = p.cu_seqlens_q[b], s1 = p.cu_seqlens_q[b + 1];
  const int L = p.context_lens[b];
  const int n = s1 - s0;
  const int start = L - n;
  if (L == 0 && n >= 0 && s0 >= 0 && static_cast<int64_t>(s1) <= p.num_tokens) {
    // A padding row (length 0: a batch padded up to a fixed size): its tokens
    // are stored nowhere.
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
      p.positions[s0 + j] = 0;
      p.slots[s0 + j] = -1;
    }
    return;
  }
  const bool ok = n >= 0 && start >= 0 && s0 >= 0 && static_cast<int64_t>(s1) <= p.num_tokens &&
                  static_cast<int64_t>(L) <= static_cast<int64_t>(p.max_pages) * p.page_size;
  if (!ok) {
    if (threadIdx.x == 0) raise_flag(p.err, PA_DEVERR_BAD_LENGTH);
    // Leave well-formed rows of this request marked "store nothing".
    if (n > 0 && s0 >= 0 && static_cast<int64_t>(s1) <= p.num_tokens)
      for (int j = threadIdx.x; j < n; j += blockDim.x) {
        p.positions[s0 + j] = 0;
        p.slots[s0 + j] = -1;
      }
    return;
  }
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int pos = start + j;
    const int page = p.block_tables[static_cast<int64_t>(b) * p.max_pages + pos / p.page_size];
    int64_t slot = -1;
    if (page >= 0 && page < p.num_pages) {
      slot = static_cast<int64_t>(page) * p.page_size + pos % p.page_size;
    } else {
      raise_flag(p.err, PA_DEVERR_BAD_PAGE);
    }
    p.positions[s0 + j] = pos;
    p.slots[s0 + j] = slot;
  }
}

// ---------------------------------------------------------------------------
// KV scatter (nano-vLLM learning note, store_kvcache_kernel): 16-byte chunks,
// one thread per chunk of K and the same chunk of V.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) kv_write_kernel(const KvWriteParams p) {
  // the prefill planner of the same step may start beside this grid (it
  // reads none of its output and waits for it before it exits)
  pdl_trigger();
  const uint32_t cpr = static_cast<uint32_t>(p.row_bytes) >> 4;
  const int64_t total = p.n_tokens * cpr;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / cpr;
    const uint32_t ch = static_cast<uint32_t>(i - t * cpr);
    const int64_t slot = p.slots[t];
    if (slot < 0 || slot >= p.num_slots) {
      if (slot != -1 && ch == 0) raise_flag(p.err, PA_DEVERR_BAD_SLOT);
      continue;
    }
    const uint4 kw = ldg16(p.k + t * p.k_stride_bytes + ch * 16);
    const uint4 vw = ldg16(p.v + t * p.v_stride_bytes + ch * 16);
    stg16(p.k_cache + slot * p.row_bytes + ch * 16, kw);
    stg16(p.v_cache + slot * p.row_bytes + ch * 16, vw);
  }
}

// ---------------------------------------------------------------------------
// fused q/k RMSNorm + rotary + KV scatter.  One CTA (4 warps) per token.
// A group of LPH lanes handles one head: lane l owns elements
// [4l, 4l+4) of the first half and the same of the second half, so each lane
// holds both members of its rotation pairs.  Values are rounded to the storage
// type after the normalisation, after the weight and after the rotation (the
// casts of the Qwen3 norm and rotary in the nano-vLLM learning note); for bf16
// the element arithmetic runs on fp32 pairs (packed multiplies and FMAs, one
// two-lane conversion per rounding).
// ---------------------------------------------------------------------------
template <typename T>
struct Vec4;
template <>
struct Vec4<float> {
  static PA_DEVINL void load(const void* p, float (&x)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
  static PA_DEVINL void store(void* p, const float (&x)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  }
};
template <>
struct Vec4<__nv_bfloat16> {
  static PA_DEVINL void load(const void* p, float (&x)[4]) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    const float2 a = bf16x2_to_float2(v.x), b = bf16x2_to_float2(v.y);
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  }
  static PA_DEVINL void store(void* p, const float (&x)[4]) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
  }
};

// 2*pi as the float nearest to it plus the float nearest to the remainder
// (Cody and Waite's additive reduction, 1980), and the float nearest to 1/(2*pi).
constexpr float kTwoPiF1 = 6.28318548202514648f;
constexpr float kTwoPiF2 = -1.74845553146951609e-7f;
constexpr float kInvTwoPiF = 0.159154943091895336f;

// The rotation angle pos * f reduced into [-pi, pi], with f given as the float
// pair fh + fl.  pos * fh is split exactly into p1 + e1 (an FMA recovers the
// product's rounding error: Dekker's two-product); pos * fl is below 2^-24 of
// the angle, so one rounding of it is negligible.  The angle is then reduced
// by k = rint(pos * fh / (2 pi)) against the two-float 2 pi: each FMA's result
// is exact or within an ulp of a value below pi, so for angles up to ~2^17 rad
// (positions up to ~131k at frequency 1) the reduced angle is within a few
// 1e-7 rad of the exact one.
PA_DEVINL float reduce_angle(int pos, float fh, float fl) {
  const float pf = static_cast<float>(pos);  // exact below 2^24
  const float p1 = pf * fh;
  const float e1 = fmaf(pf, fh, -p1);
  const float e2 = pf * fl;
  const float k = rintf(p1 * kInvTwoPiF);
  const float r = fmaf(-k, kTwoPiF2, fmaf(-k, kTwoPiF1, p1));
  return r + (e1 + e2);
}

// Two bf16 products, each rounded once to bf16 (the exact product of two
// bf16 values fits in fp32, so this equals rounding the fp32 product).
PA_DEVINL uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Position and cache slot of new token t from the varlen metadata, as
// pa_slot_mapping computes them (nano-vLLM learning note, prepare_prefill
// listing): request b owns tokens cu[b] .. cu[b+1]-1, at positions
// context_lens[b] - n_b + j; a padding row (length 0) and an inconsistent
// request get position 0 and slot -1.  With `report` the flags and the
// optional outputs are written.
PA_DEVINL void map_token_of(const NormRopeParams& p, int64_t t, int b, int s0, int s1, int L, bool report, int& pos,
                             int64_t& slot) {
  const int n = s1 - s0, start = L - n;
  pos = 0;
  slot = -1;
  unsigned int flag = 0;
  if (s0 < 0 || t < s0 || t >= s1 || static_cast<int64_t>(s1) > p.n_tokens) {
    flag = PA_DEVERR_BAD_LENGTH;  // cu_seqlens_q does not cover the token
  } else if (L == 0) {
    // a padding row: stored nowhere
  } else if (start < 0 || static_cast<int64_t>(L) > static_cast<int64_t>(p.maxp) * p.page_size) {
    flag = PA_DEVERR_BAD_LENGTH;
  } else {
    pos = start + static_cast<int>(t - s0);
    const int page = p.bt[static_cast<int64_t>(b) * p.maxp + (pos >> p.log2P)];
    if (page >= 0 && page < p.num_pages)
      slot = static_cast<int64_t>(page) * p.page_size + (pos & (p.page_size - 1));
    else
      flag = PA_DEVERR_BAD_PAGE;
  }
  if (report) {
    if (flag) raise_flag(p.err, flag);
    if (p.pos_out) p.pos_out[t] = pos;
    if (p.slots_out) p.slots_out[t] = slot;
  }
}

// The same for any batch: the token's request by binary search over cu.
PA_DEVINL void map_token(const NormRopeParams& p, int64_t t, bool report, int& pos, int64_t& slot) {
  int lo = 0, hi = p.batch - 1;  // the last request whose tokens start at or before t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  map_token_of(p, t, lo, p.cu[lo], p.cu[lo + 1], p.ctx[lo], report, pos, slot);
}

constexpr int kNrThreads = 128;
constexpr int kNrCtasPerSm = 8;
constexpr int kNrMaxPerCta = 2048;

// Shared-memory bytes of one token's stage: its q, k and v rows.
__host__ __device__ constexpr int nr_stage_bytes(int hq, int hkv, int hd, int e) { return (hq + 2 * hkv) * hd * e; }

// A CTA walks the tokens t = blockIdx.x, blockIdx.x + gridDim.x, ...: one
// thread copies each token's q, k and v rows into a two-stage shared-memory
// ring with bulk async copies (TMA engine), two tokens ahead, so the rows of
// the next token stream in while the current one is normed and rotated.
// A group of LPH lanes handles one head: lane l owns elements [4l, 4l+4) of
// the first half and the same of the second half, so each lane holds both
// members of its rotation pairs.  Values are rounded to the storage type
// after the normalisation, after the weight and after the rotation (the
// casts of the Qwen3 norm and rotary in the nano-vLLM learning note); for
// bf16 the element arithmetic runs on fp32 pairs (packed multiplies and FMAs,
// one two-lane conversion per rounding).
template <typename T, int HD>
__global__ void __launch_bounds__(kNrThreads) norm_rope_kv_write_kernel(const NormRopeParams p) {
  constexpr int E = sizeof(T);
  constexpr int PE = 4;
  constexpr int LPH = HD / (2 * PE);  // lanes per head
  constexpr int HPW = 32 / LPH;       // heads per warp pass
  extern __shared__ __align__(128) unsigned char nr_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPH, l = lane % LPH;
  const int row_q = p.hq * HD * E, row_kv = p.hkv * HD * E;
  const int stage_bytes = row_q + 2 * row_kv;
  unsigned char* stages = nr_smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(nr_smem + 2 * stage_bytes);
  float* cs_s = reinterpret_cast<float*>(full + 2);   // [HD / 2]
  float* sn_s = cs_s + HD / 2;
  // the CTA's tokens' (position, slot) when they come from the metadata
  longlong2* meta_s = reinterpret_cast<longlong2*>(sn_s + HD / 2);
  __shared__ int abort_flag;
  pdl_trigger();  // as in kv_write_kernel: the prefill planner may start beside this grid

  const int64_t t0 = blockIdx.x, dt = gridDim.x;
  const int n_mine = static_cast<int>((p.n_tokens - t0 + dt - 1) / dt);  // tokens of this CTA
  auto issue = [&](int i) {  // thread 0: the copies of the CTA's i-th token into stage i & 1
    const int64_t t = t0 + i * dt;
    unsigned char* st = stages + (i & 1) * stage_bytes;
    mbar_arrive_expect_tx(&full[i & 1], static_cast<uint32_t>(stage_bytes));
    bulk_g2s(st, static_cast<const char*>(p.q) + t * p.q_stride * E, row_q, &full[i & 1]);
    bulk_g2s(st + row_q, static_cast<const char*>(p.k) + t * p.k_stride * E, row_kv, &full[i & 1]);
    bulk_g2s(st + row_q + row_kv, static_cast<const char*>(p.v) + t * p.v_stride * E, row_kv, &full[i & 1]);
  };
  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    abort_flag = 0;
    fence_mbar_init();
    if (n_mine > 0) issue(0);
    if (n_mine > 1) issue(1);
  }

  float wq_a[PE], wq_b[PE], wk_a[PE], wk_b[PE];
  Vec4<T>::load(static_cast<const T*>(p.wq) + l * PE, wq_a);
  Vec4<T>::load(static_cast<const T*>(p.wq) + HD / 2 + l * PE, wq_b);
  Vec4<T>::load(static_cast<const T*>(p.wk) + l * PE, wk_a);
  Vec4<T>::load(static_cast<const T*>(p.wk) + HD / 2 + l * PE, wk_b);
  // bf16: the weights as bf16 pairs for the packed multiply
  uint32_t wq_a2[PE / 2], wq_b2[PE / 2], wk_a2[PE / 2], wk_b2[PE / 2];
#pragma unroll
  for (int e2 = 0; e2 < PE / 2; ++e2) {
    wq_a2[e2] = pack_bf16x2(wq_a[2 * e2], wq_a[2 * e2 + 1]);
    wq_b2[e2] = pack_bf16x2(wq_b[2 * e2], wq_b[2 * e2 + 1]);
    wk_a2[e2] = pack_bf16x2(wk_a[2 * e2], wk_a[2 * e2 + 1]);
    wk_b2[e2] = pack_bf16x2(wk_b[2 * e2], wk_b[2 * e2 + 1]);
  }
  // a token's position and slot: from the inputs, or mapped from the varlen
  // metadata for all of the CTA's tokens at once by warp 1 (the mapping's
  // dependent loads overlap the first token's copies)
  const bool mapped = p.positions == nullptr;
  if (mapped && warp == 1) {
    if (p.batch < 32) {
      // up to 31 requests: their cu and lengths in the lanes, one load each,
      // so a token's request is a count of lanes, not a chain of loads
      const int cu_l = lane <= p.batch ? p.cu[lane] : INT_MAX;
      const int ctx_l = lane < p.batch ? p.ctx[lane] : 0;
      for (int k0 = 0; k0 < n_mine; k0 += 32) {
        const int k = k0 + lane;
        const int64_t t = t0 + static_cast<int64_t>(k) * dt;
        int b = -1;
#pragma unroll 1
        for (int j = 0; j < p.batch; ++j) b += __shfl_sync(0xffffffffu, cu_l, j) <= t;
        b = max(b, 0);
        const int s0 = __shfl_sync(0xffffffffu, cu_l, b), s1 = __shfl_sync(0xffffffffu, cu_l, b + 1);
        const int L = __shfl_sync(0xffffffffu, ctx_l, b);
        if (k < n_mine) {
          int pos;
          int64_t slot;
          map_token_of(p, t, b, s0, s1, L, true, pos, slot);
          meta_s[k] = make_longlong2(pos, slot);
        }
      }
    } else {
      for (int k = lane; k < n_mine; k += 32) {
        int pos;
        int64_t slot;
        map_token(p, t0 + k * dt, true, pos, slot);
        meta_s[k] = make_longlong2(pos, slot);
      }
    }
  }
  auto token_meta = [&](int i, int& pos, int64_t& slot) {
    if (mapped) {
      const longlong2 m = meta_s[i];
      pos = static_cast<int>(m.x);
      slot = m.y;
    } else {
      pos = p.positions[t0 + i * dt];
      slot = p.slots[t0 + i * dt];
    }
  };
  cta_sync();
  int pos_next = 0;
  int64_t slot_next = -1;
  if (n_mine > 0) token_meta(0, pos_next, slot_next);

  int done = 0;  // tokens finished (their stages consumed)
  for (int i = 0; i < n_mine; ++i) {
    const int64_t t = t0 + i * dt;
    const int pos = pos_next;
    const int64_t slot = slot_next;
    if (i + 1 < n_mine) token_meta(i + 1, pos_next, slot_next);  // the next token's, one token ahead
    const bool slot_ok = slot >= 0 && slot < p.num_slots;
    if (!slot_ok && slot != -1 && threadIdx.x == 0) raise_flag(p.err, PA_DEVERR_BAD_SLOT);
    // cos / sin of the token's HD/2 pair indices, one thread per pair: the
    // angle pos * theta^(-2i/HD) formed and reduced modulo 2*pi in two-float
    // arithmetic, then evaluated by the special-function unit
    if (threadIdx.x < HD / 2) {
      const float r = reduce_angle(pos, p.inv_freq_hi[threadIdx.x], p.inv_freq_lo[threadIdx.x]);
      float sv, cv;
      __sincosf(r, &sv, &cv);
      cs_s[threadIdx.x] = cv;
      sn_s[threadIdx.x] = sv;
    }
    const bool ok = mbar_wait_bounded(&full[i & 1], (i >> 1) & 1, &abort_flag, p.err);
    if (!__syncthreads_and(ok)) break;  // cos / sin written, every thread past its wait
    float cs[PE], sn[PE], nsn[PE];
#pragma unroll
    for (int e = 0; e < PE; ++e) {
      cs[e] = cs_s[l * PE + e];
      sn[e] = sn_s[l * PE + e];
      nsn[e] = -sn[e];
    }
    const unsigned char* st = stages + (i & 1) * stage_bytes;
    const int nheads = p.hq + p.hkv;
    for (int hh = warp * HPW + sub; hh - sub < nheads; hh += (kNrThreads / 32) * HPW) {
      const bool active = hh < nheads;
      const bool isq = hh < p.hq;
      const T* src = reinterpret_cast<const T*>(st) + static_cast<int64_t>(active ? hh : 0) * HD;
      float xa[PE] = {0.f, 0.f, 0.f, 0.f}, xb[PE] = {0.f, 0.f, 0.f, 0.f};
      if (active) {
        Vec4<T>::load(src + l * PE, xa);
        Vec4<T>::load(src + HD / 2 + l * PE, xb);
      }
      float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < PE; e += 2) {
        ss2 = ffma2(make_float2(xa[e], xa[e + 1]), make_float2(xa[e], xa[e + 1]), ss2);
        ss2 = ffma2(make_float2(xb[e], xb[e + 1]), make_float2(xb[e], xb[e + 1]), ss2);
      }
      float ss = ss2.x + ss2.y;
#pragma unroll
      for (int m = LPH / 2; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      if (!active) continue;
      const float r = rsqrtf(ss * (1.0f / HD) + p.eps);
      T* dst = isq ? static_cast<T*>(p.q_out) + (t * p.hq + hh) * HD
                   : static_cast<T*>(p.k_cache) + (slot * p.hkv + (hh - p.hq)) * HD;
      const bool store = isq || slot_ok;
      if constexpr (sizeof(T) == 2) {
        // y_a = n_a cos - n_b sin, y_b = n_b cos + n_a sin on fp32 pairs
        uint32_t wa[PE / 2], wb[PE / 2];
        const float2 r2 = make_float2(r, r);
#pragma unroll
        for (int e2 = 0; e2 < PE / 2; ++e2) {
          const int e = 2 * e2;
          const float2 ta = fmul2(make_float2(xa[e], xa[e + 1]), r2);
          const float2 tb = fmul2(make_float2(xb[e], xb[e + 1]), r2);
          const float2 na = bf16x2_to_float2(mul_bf16x2(pack_bf16x2(ta.x, ta.y), isq ? wq_a2[e2] : wk_a2[e2]));
          const float2 nb = bf16x2_to_float2(mul_bf16x2(pack_bf16x2(tb.x, tb.y), isq ? wq_b2[e2] : wk_b2[e2]));
          const float2 c2 = make_float2(cs[e], cs[e + 1]);
          const float2 ya = ffma2(nb, make_float2(nsn[e], nsn[e + 1]), fmul2(na, c2));
          const float2 yb = ffma2(nb, c2, fmul2(na, make_float2(sn[e], sn[e + 1])));
          wa[e2] = pack_bf16x2(ya.x, ya.y);
          wb[e2] = pack_bf16x2(yb.x, yb.y);
        }
        if (store) {
          *reinterpret_cast<uint2*>(dst + l * PE) = make_uint2(wa[0], wa[1]);
          *reinterpret_cast<uint2*>(dst + HD / 2 + l * PE) = make_uint2(wb[0], wb[1]);
        }
      } else {
        float ya[PE], yb[PE];
#pragma unroll
        for (int e = 0; e < PE; ++e) {
          const float na = round_to<T>(round_to<T>(xa[e] * r) * (isq ? wq_a[e] : wk_a[e]));
          const float nb = round_to<T>(round_to<T>(xb[e] * r) * (isq ? wq_b[e] : wk_b[e]));
          ya[e] = round_to<T>(na * cs[e] - nb * sn[e]);
          yb[e] = round_to<T>(nb * cs[e] + na * sn[e]);
        }
        if (store) {
          Vec4<T>::store(dst + l * PE, ya);
          Vec4<T>::store(dst + HD / 2 + l * PE, yb);
        }
      }
    }
    if (slot_ok) {  // the v row, unchanged, into its slot
      const unsigned char* vsrc = st + row_q + row_kv;
      char* vdst = static_cast<char*>(p.v_cache) + slot * row_kv;
      for (int ch = threadIdx.x; ch < row_kv / 16; ch += kNrThreads)
        stg16(vdst + ch * 16, *reinterpret_cast<const uint4*>(vsrc + ch * 16));
    }
    cta_sync();  // every thread is done with the stage and with cos / sin
    if (threadIdx.x == 0 && i + 2 < n_mine) issue(i + 2);
    done = i + 1;
  }
  if (threadIdx.x == 0) {
    // after an abort, copies issued for tokens not reached may still land:
    // wait for them (time only) before the CTA exits
    for (int i = done; i < n_mine && i < done + 2; ++i) {
      const uint64_t tw = global_timer_ns();
      while (!mbar_try_wait(&full[i & 1], (i >> 1) & 1) && global_timer_ns() - tw < kWaitLimitNs) {
      }
    }
  }
}

}  // namespace

cudaError_t launch_slot_mapping(const SlotMapParams& p, cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  slot_mapping_kernel<<<p.batch, 128, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_kv_write(const KvWriteParams& p, cudaStream_t s) {
  if (p.n_tokens == 0) return cudaSuccess;
  DeviceInfo di;
  cudaError_t e = current_device_info(&di);
  if (e != cudaSuccess) return e;
  const int64_t total = p.n_tokens * (p.row_bytes / 16);
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(di.sm_count) * 8);
  kv_write_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_norm_rope_kv_write(int dtype, int head_dim, const NormRopeParams& p, cudaStream_t s) {
  if (p.n_tokens == 0) return cudaSuccess;
  DeviceInfo di;
  cudaError_t e = current_device_info(&di);
  if (e != cudaSuccess) return e;
  const int es = dtype == PA_BF16 ? 2 : 4;
  // one wave of CTAs walking the tokens, with at most kNrMaxPerCta tokens
  // each (the mapped tokens' positions and slots are kept in shared memory)
  const int64_t wave = static_cast<int64_t>(di.sm_count) * kNrCtasPerSm;
  const unsigned grid = static_cast<unsigned>(
      std::max(std::min<int64_t>(p.n_tokens, wave), (p.n_tokens + kNrMaxPerCta - 1) / kNrMaxPerCta));
  const int64_t per_cta = (p.n_tokens + grid - 1) / grid;  // tokens of the busiest CTA
  const size_t smem = 2 * static_cast<size_t>(nr_stage_bytes(p.hq, p.hkv, head_dim, es)) + 2 * sizeof(uint64_t) +
                      head_dim * sizeof(float) + (p.positions == nullptr ? per_cta * sizeof(longlong2) : 0);
  if (smem > static_cast<size_t>(di.max_smem_optin)) return cudaErrorInvalidValue;
  const void* fn = dtype == PA_BF16
                       ? (head_dim == 128 ? reinterpret_cast<const void*>(norm_rope_kv_write_kernel<__nv_bfloat16, 128>)
                                          : reinterpret_cast<const void*>(norm_rope_kv_write_kernel<__nv_bfloat16, 64>))
                       : (head_dim == 128 ? reinterpret_cast<const void*>(norm_rope_kv_write_kernel<float, 128>)
                                          : reinterpret_cast<const void*>(norm_rope_kv_write_kernel<float, 64>));
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  void* args[] = {const_cast<NormRopeParams*>(&p)};
  e = cudaLaunchKernel(fn, dim3(grid), dim3(kNrThreads), args, smem, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pa
