// Chunked-prefill attention on the 5th-generation tensor cores (sm_103a):
// tcgen05.mma with fp32 accumulators in tensor memory, operands staged by TMA,
// bf16 inputs, head_dim 128.
//
// Semantics (nano-vLLM learning note, Attention.forward / prepare_prefill
// listings; qwen-engine README, flat varlen packing): row i of request b's
// chunk sits at position context_lens[b] - n_b + i and attends to keys
// 0 .. that position, all read from the paged cache.
//
// One CTA = (request, kv-head, pair of q-tiles).  A q-tile is 128 rows:
// TQ = 128 / G tokens x the G q-heads that share the kv-head, so each staged
// K/V tile feeds the whole GQA group, and it feeds both q-tiles of the pair
// (256 rows per K/V tile).
//   warp 0     TMA producer: both Q tiles once (3-D map), then per 128-key tile
//              the K and V rows gathered page by page with 16-row boxes
//              (single-row boxes for a ragged end, so no slot past the context
//              is read).
//   warp 1     allocates all 512 TMEM columns; lane 0 issues the MMAs:
//              S_g = Q_g K_j^T and O_g += P_g V_j for the two q-tiles g, in
//              the order PV_0(j), QK_0(j+1), PV_1(j), QK_1(j+1), so that each
//              softmax group has a PV and a QK of the other group to hide in.
//   warps 2-9  two softmax groups of 4 warps, one thread per row (= TMEM
//              lane): pass 1 reads S and takes the row max; O in TMEM is
//              rescaled only when a row max grows by more than 2^8; pass 2
//              reads S again, turns it into bf16 probabilities and writes them
//              back over S's first 64 columns, where the PV MMA reads its A
//              operand.  Finally O / l goes to global memory.
// TMEM: S_0 cols 0-127 (P_0 in 0-63), S_1 128-255 (P_1 in 128-191),
//       O_0 256-383, O_1 384-511.
// Every wait is bounded; a timeout raises PA_DEVERR_TIMEOUT and the CTA
// drains its copies and MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kBM = 128;                    // rows per q-tile
constexpr int kBN = 128;                    // keys per tile
constexpr int kHalfBytes = 128 * 128;       // 128 rows x 64 bf16 (one swizzle-atom column)
constexpr int kTileBytes = 2 * kHalfBytes;  // 128 rows x 128 bf16
constexpr int kThreads = 320;
constexpr int kBoxRows = 16;
constexpr uint32_t kTmemCols = 512;

constexpr int kOffQ = 0;                          // two q-tiles
constexpr int kOffK = kOffQ + 2 * kTileBytes;     // two K stages
constexpr int kOffV = kOffK + 2 * kTileBytes;     // two V stages
constexpr int kOffBar = kOffV + 2 * kTileBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;  // + slack to align the base to 1024

// kind::f16 instruction descriptor: D fp32, A and B bf16, M = 128, N = 128.
constexpr uint32_t kIdescQK = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                              ((uint32_t)(kBM >> 4) << 24);
constexpr uint32_t kIdescPV = kIdescQK | (1u << 16);  // B (= V) is MN-major

struct TcParams {
  CUtensorMap tm_q;    // q      [num_tokens, Hq, 128], box {64, G, TQ}
  CUtensorMap tm_k16;  // k_cache rows, box {64, 16}
  CUtensorMap tm_k1;   //                box {64, 1}
  CUtensorMap tm_v16;
  CUtensorMap tm_v1;
  const int32_t* cu;
  const int32_t* bt;
  const int32_t* ctx;
  char* out;
  unsigned int* err;
  int64_t num_pages;
  int32_t B, Hq, Hkv, G, TQ, P, log2P, maxp, max_ctx;
  float scale_log2;
};

// ---------------------------------------------------------------------------
// tcgen05 / TMA primitives
// ---------------------------------------------------------------------------
PA_DEVINL void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

PA_DEVINL void tma_load_3d(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

PA_DEVINL void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
PA_DEVINL void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
PA_DEVINL void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 descriptor version 1).
PA_DEVINL uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

PA_DEVINL void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

PA_DEVINL void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

#define PA_R32(r)                                                                                             \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), \
      "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),  \
      "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), \
      "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define PA_W32(r)                                                                                                 \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), \
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), \
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), \
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])

// 32 consecutive fp32 columns of this thread's TMEM lane.  The load and its
// wait sit in one asm statement, so the outputs are defined only after the
// asynchronous load has completed.
PA_DEVINL void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : PA_R32(r)
      : "r"(taddr)
      : "memory");
}

PA_DEVINL void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      PA_W32(r)
      : "memory");
}

PA_DEVINL void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

PA_DEVINL void drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
}


// O += A(TMEM) * B(smem): the A operand (probabilities) is read from tensor memory.
PA_DEVINL void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

// Load 32 columns without waiting; the registers are valid only after
// tmem_wait_ld32 on the same array, whose asm reads and rewrites them so the
// compiler cannot move any use above the wait.
PA_DEVINL void tmem_ld32_async(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : PA_R32(r)
      : "r"(taddr)
      : "memory");
}

#define PA_RW32(r)                                                                                              \
  "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), \
      "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]),  \
      "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), \
      "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])

PA_DEVINL void tmem_wait_ld32(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : PA_RW32(r)::"memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane.
PA_DEVINL void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// 2^x on the special-function unit (PTX ex2.approx; inputs here are <= 8).
PA_DEVINL float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  const int qp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s0 = p.cu[b], s1 = p.cu[b + 1];
  const int n = s1 - s0;
  if (2 * qp * p.TQ >= n) return;
  const int L = p.ctx[b];
  const int cap = min(p.max_ctx, p.maxp << p.log2P);
  if (s0 < 0 || L < n || L > cap) {
    if (threadIdx.x == 0) raise_flag(p.err, PA_DEVERR_BAD_LENGTH);
    return;
  }
  const int nq = (2 * qp + 1) * p.TQ < n ? 2 : 1;  // q-tiles of the pair with rows
  int rows[2], pos0[2], ntg[2];
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int qt = 2 * qp + g;
    rows[g] = g < nq ? min(p.TQ, n - qt * p.TQ) : 0;   // live tokens of the tile
    pos0[g] = L - n + qt * p.TQ;                       // position of its first token
    ntg[g] = g < nq ? (pos0[g] + rows[g] + kBN - 1) / kBN : 0;  // key tiles it needs
  }
  const int kv_len = pos0[nq - 1] + rows[nq - 1];
  const int nt = ntg[nq - 1];

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = bars + 3;
  uint64_t* k_empty = bars + 5;
  uint64_t* v_empty = bars + 7;
  uint64_t* s_full = bars + 9;    // per q-tile
  uint64_t* p_full = bars + 11;   // per q-tile
  uint64_t* pv_done = bars + 13;  // per q-tile
  uint64_t* o_final = bars + 15;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 16) + 1;

  // Rows never loaded must hold finite values: zero both Q tiles and both V stages.
  {
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < 2 * kTileBytes / 16; i += kThreads) {
      reinterpret_cast<uint4*>(smem + kOffQ)[i] = z;
      reinterpret_cast<uint4*>(smem + kOffV)[i] = z;
    }
  }
  fence_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 4);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(o_final, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------- TMA producer -------------------------------
    int issued_k = 0, issued_v = 0;
    bool ok = true;
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(nq * 2 * p.G * p.TQ * 128));
      for (int g = 0; g < nq; ++g) {
        const int z = s0 + (2 * qp + g) * p.TQ;
        tma_load_3d(smem + kOffQ + g * kTileBytes, &p.tm_q, 0, h * p.G, z, q_full);
        tma_load_3d(smem + kOffQ + g * kTileBytes + kHalfBytes, &p.tm_q, 64, h * p.G, z, q_full);
      }
    }
    const int64_t bt_row = static_cast<int64_t>(b) * p.maxp;
    const int box = lane >> 2, half = (lane >> 1) & 1, isv = lane & 1;
    const int x = h * 128 + half * 64;
    for (int j = 0; j < nt && ok; ++j) {
      const int st = j & 1;
      const uint32_t par = ((j >> 1) & 1) ^ 1;
      const int t0 = j * kBN;
      const int valid = min(kBN, kv_len - t0);
      const int nfull = valid / kBoxRows, rem = valid % kBoxRows;
      int y_full = -1, y_rem = -1;
      if (box < nfull) {
        const int key0 = t0 + box * kBoxRows;
        const int page = p.bt[bt_row + (key0 >> p.log2P)];
        if (page >= 0 && page < p.num_pages) y_full = (page << p.log2P) + (key0 & (p.P - 1));
        else raise_flag(p.err, PA_DEVERR_BAD_PAGE);
      }
      if (rem && lane < 4) {
        const int key0 = t0 + nfull * kBoxRows;
        const int page = p.bt[bt_row + (key0 >> p.log2P)];
        if (page >= 0 && page < p.num_pages) y_rem = (page << p.log2P) + (key0 & (p.P - 1));
        else raise_flag(p.err, PA_DEVERR_BAD_PAGE);
      }
      uint32_t mine = (y_full >= 0 ? kBoxRows * 128 : 0) + (y_rem >= 0 ? rem * 128 : 0);
      uint32_t kb = isv ? 0 : mine, vb = isv ? mine : 0;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        kb += __shfl_xor_sync(0xffffffffu, kb, o);
        vb += __shfl_xor_sync(0xffffffffu, vb, o);
      }
      int okk = 1;
      if (lane == 0) {
        okk = mbar_wait_bounded(&k_empty[st], par, abort_flag, p.err);
        if (okk) mbar_arrive_expect_tx(&k_full[st], kb);
      }
      ok = __shfl_sync(0xffffffffu, okk, 0) != 0;
      if (!ok) break;
      if (!isv) {
        unsigned char* dst = smem + kOffK + st * kTileBytes + half * kHalfBytes;
        if (y_full >= 0) tma_load_2d(dst + box * kBoxRows * 128, &p.tm_k16, x, y_full, &k_full[st]);
        if (y_rem >= 0)
          for (int r = 0; r < rem; ++r) tma_load_2d(dst + (nfull * kBoxRows + r) * 128, &p.tm_k1, x, y_rem + r, &k_full[st]);
      }
      ++issued_k;
      int okv = 1;
      if (lane == 0) {
        okv = mbar_wait_bounded(&v_empty[st], par, abort_flag, p.err);
        if (okv) mbar_arrive_expect_tx(&v_full[st], vb);
      }
      ok = __shfl_sync(0xffffffffu, okv, 0) != 0;
      if (!ok) break;
      if (isv) {
        unsigned char* dst = smem + kOffV + st * kTileBytes + half * kHalfBytes;
        if (y_full >= 0) tma_load_2d(dst + box * kBoxRows * 128, &p.tm_v16, x, y_full, &v_full[st]);
        if (y_rem >= 0)
          for (int r = 0; r < rem; ++r) tma_load_2d(dst + (nfull * kBoxRows + r) * 128, &p.tm_v1, x, y_rem + r, &v_full[st]);
      }
      ++issued_v;
    }
    if (!ok && lane == 0) {
      drain(q_full, 0);
      for (int j = max(0, issued_k - 2); j < issued_k; ++j) drain(&k_full[j & 1], (j >> 1) & 1);
      for (int j = max(0, issued_v - 2); j < issued_v; ++j) drain(&v_full[j & 1], (j >> 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------- MMA issuer -------------------------------
    if (lane == 0) {
      bool ok = mbar_wait_bounded(q_full, 0, abort_flag, p.err);
      const uint32_t aQ = smem_u32(smem + kOffQ);
      const uint32_t aK = smem_u32(smem + kOffK), aV = smem_u32(smem + kOffV);
      auto qk = [&](int g, int j) {
        const uint32_t qbase = aQ + g * kTileBytes, kbase = aK + (j & 1) * kTileBytes;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
          mma_bf16(tmem + g * 128, sdesc(qbase + off, 16, 1024), sdesc(kbase + off, 16, 1024), kIdescQK, k > 0);
        }
        mma_commit(&s_full[g]);
      };
      auto pv = [&](int g, int j) -> bool {
        if (!mbar_wait_bounded(&p_full[g], j & 1, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t vbase = aV + (j & 1) * kTileBytes;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_bf16_ts(tmem + 256 + g * 128, tmem + g * 128 + k * 8, sdesc(vbase + k * 16 * 128, kHalfBytes, 1024),
                      kIdescPV, (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(&pv_done[g]);
        return true;
      };
      if (ok) ok = mbar_wait_bounded(&k_full[0], 0, abort_flag, p.err);
      if (ok) {
        tc_fence_after();
        for (int g = 0; g < nq; ++g) qk(g, 0);
        mma_commit(&k_empty[0]);
      }
      for (int j = 0; j < nt && ok; ++j) {
        const bool more = j + 1 < nt;
        if (!(ok = mbar_wait_bounded(&v_full[j & 1], (j >> 1) & 1, abort_flag, p.err))) break;
        // q-tile 0: PV of tile j, then QK of tile j+1 (the tensor pipe runs them
        // in issue order, so QK overwrites S_0 only after PV has read P_0)
        if (j < ntg[0] && !(ok = pv(0, j))) break;
        if (more) {
          if (!(ok = mbar_wait_bounded(&k_full[(j + 1) & 1], ((j + 1) >> 1) & 1, abort_flag, p.err))) break;
          tc_fence_after();
          if (j + 1 < ntg[0]) qk(0, j + 1);
        }
        // q-tile 1
        if (j < ntg[1] && !(ok = pv(1, j))) break;
        if (more && j + 1 < ntg[1]) qk(1, j + 1);
        mma_commit(&v_empty[j & 1]);
        if (more) mma_commit(&k_empty[(j + 1) & 1]);
      }
      mma_commit(o_final);
      if (!ok) drain(o_final, 0);
    }
  } else {
    // ------------------------------- softmax groups -------------------------------
    const int g = (warp - 2) >> 2;
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t colS = g * 128, colO = 256 + g * 128;
    const int t = row / p.G, gg = row - (row / p.G) * p.G;
    const bool live = g < nq && row < p.TQ * p.G && t < rows[g];
    const int pos_r = pos0[g] + t;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntg[g]; ++j) {
      ok = mbar_wait_bounded(&s_full[g], j & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int key0 = j * kBN;
      const bool need_mask = key0 + kBN - 1 > pos0[g];
      // One TMEM round trip per tile: all 128 scores of the row are loaded
      // (four loads, one wait), the row max is taken over the raw scores (the
      // scale is positive, so it commutes with the max) with eight independent
      // accumulators, and the probabilities are computed from registers.
      uint32_t x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32_async(tmem + lane_off + colS + 32 * c, x + 32 * c);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_wait_ld32(x + 32 * c);
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < 128; ++e)
          if (key0 + e > pos_r) x[e] = __float_as_uint(-INFINITY);
      }
      float mx;
      {
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = __uint_as_float(x[e]);
#pragma unroll
        for (int e = 8; e < 128; ++e) m8[e & 7] = fmaxf(m8[e & 7], __uint_as_float(x[e]));
#pragma unroll
        for (int e = 0; e < 4; ++e) m8[e] = fmaxf(m8[e], m8[e + 4]);
        mx = fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])) * p.scale_log2;
      }
      if (__any_sync(0xffffffffu, mx > m_used + 8.f)) {
        const float m_new = fmaxf(m_used, mx);
        const float alpha = m_used == -INFINITY ? 0.f : ex2(m_used - m_new);
        if (j > 0) {
          ok = mbar_wait_bounded(&pv_done[g], (j - 1) & 1, abort_flag, p.err);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + colO + 32 * c, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tmem + lane_off + colO + 32 * c, o);
          }
          tmem_wait_st();
        }
        l *= alpha;
        m_used = m_new;
      }
      // probabilities as bf16, written over the first 64 columns of S (masked
      // scores are -inf and give exactly 0)
      const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
      float2 rs4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) rs4[e] = make_float2(0.f, 0.f);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p0 = ex2(fmaf(__uint_as_float(x[64 * hh + 2 * e]), p.scale_log2, neg_m));
          const float p1 = ex2(fmaf(__uint_as_float(x[64 * hh + 2 * e + 1]), p.scale_log2, neg_m));
          rs4[e & 3] = fadd2(rs4[e & 3], make_float2(p0, p1));
          w[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tmem + lane_off + colS + 32 * hh, w);
        tmem_st16(tmem + lane_off + colS + 32 * hh + 16, w + 16);
      }
      tmem_wait_st();
      const float2 rsum = fadd2(fadd2(rs4[0], rs4[1]), fadd2(rs4[2], rs4[3]));
      l += rsum.x + rsum.y;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[g]);
    }
    // epilogue: O / l to global memory
    if (g < nq) {
      if (ok) ok = mbar_wait_bounded(o_final, 0, abort_flag, p.err);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        char* dst = p.out + ((static_cast<int64_t>(s0) + (2 * qp + g) * p.TQ + t) * p.Hq + h * p.G + gg) * 256;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + colO + 32 * c, o);
          if (live) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[8 * q4 + 0]) * inv, __uint_as_float(o[8 * q4 + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv, __uint_as_float(o[8 * q4 + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv, __uint_as_float(o[8 * q4 + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv, __uint_as_float(o[8 * q4 + 7]) * inv);
              *reinterpret_cast<uint4*>(dst + c * 64 + q4 * 16) = w;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------
// host side: tensor maps and launch
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

bool encode(EncodeTiledFn fn, CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill_tc(const pa_cache_desc& d, const PrefillArgs& a, cudaStream_t s) {
  if (a.num_tokens == 0 || a.batch == 0) return cudaSuccess;
  // TMA coordinates are 32-bit: the cache rows must be addressable.
  if (d.num_pages * d.page_size >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  TcParams p;
  memset(&p, 0, sizeof(p));
  const int G = d.num_q_heads / d.num_kv_heads;
  const int TQ = kBM / G;
  {
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(d.num_q_heads), static_cast<cuuint64_t>(a.num_tokens)};
    const cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(d.num_q_heads) * 256};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(TQ)};
    if (!encode(fn, &p.tm_q, a.q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d.num_kv_heads) * 128,
                                static_cast<cuuint64_t>(d.num_pages) * d.page_size};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d.num_kv_heads) * 256};
    const cuuint32_t box16[2] = {64, kBoxRows}, box1[2] = {64, 1};
    if (!encode(fn, &p.tm_k16, a.k_cache, 2, dims, strides, box16) ||
        !encode(fn, &p.tm_k1, a.k_cache, 2, dims, strides, box1) ||
        !encode(fn, &p.tm_v16, a.v_cache, 2, dims, strides, box16) ||
        !encode(fn, &p.tm_v1, a.v_cache, 2, dims, strides, box1))
      return cudaErrorInvalidValue;
  }
  p.cu = a.cu_seqlens_q;
  p.bt = a.block_tables;
  p.ctx = a.context_lens;
  p.out = static_cast<char*>(a.out);
  p.err = a.err;
  p.num_pages = d.num_pages;
  p.B = a.batch;
  p.Hq = d.num_q_heads;
  p.Hkv = d.num_kv_heads;
  p.G = G;
  p.TQ = TQ;
  p.P = d.page_size;
  p.log2P = 0;
  while ((1 << p.log2P) < d.page_size) ++p.log2P;
  p.maxp = a.max_pages;
  p.max_ctx = a.max_context_len;
  p.scale_log2 = a.scale * 1.4426950408889634f;

  {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!done[dev]) {
      e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) return e;
      done[dev] = true;
    }
  }
  const int qtiles = (a.max_seqlen_q + TQ - 1) / TQ;
  const dim3 grid((qtiles + 1) / 2, d.num_kv_heads, a.batch);
  prefill_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
