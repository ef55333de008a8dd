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
//   warp 0     TMA producer of Q and K: both Q tiles once (3-D map) and K
//              tile 0 go out during the CTA's setup, then per 128-key tile
//              the K rows gathered page by page with 16-row boxes
//              (single-row boxes for a ragged end, so no slot past the context
//              is read); block-table entries are read one tile ahead.
//   warp 10    TMA producer of V, the same way; K and V run ahead of the MMAs
//              independently, each as far as its own two stages allow.
//   warp 1     allocates all 512 TMEM columns; lane 0 issues the MMAs:
//              S_g = Q_g K_j^T and O_g += P_g V_j for the two q-tiles g, in
//              the order PV_0(j), QK_0(j+1), PV_1(j), QK_1(j+1), so that each
//              softmax group has a PV and a QK of the other group to hide in.
//   warps 2-9  two softmax groups of 4 warps, one thread per row (= TMEM
//              lane): a tile's 128 scores come into registers in one TMEM
//              round trip, the row max is taken, O in TMEM is rescaled only
//              when a row max grows by more than 2^8, and the bf16
//              probabilities are written back over S's first 64 columns,
//              where the PV MMA reads its A operand.  Finally O / l goes to
//              global memory.
// TMEM: S_0 cols 0-127 (P_0 in 0-63), S_1 128-255 (P_1 in 128-191),
//       O_0 256-383, O_1 384-511.
// Every wait is bounded; a timeout raises PA_DEVERR_TIMEOUT and the CTA
// drains its copies and MMAs, frees its TMEM and returns.
//
// Planned launch (the caller gives a workspace): a one-CTA planner kernel
// turns the pairs into units, cutting long key ranges into parts and listing
// the units longest first; a CTA then runs one (unit, kv-head), a part writes
// O / l and the row log-sum-exp in fp32, and a merge kernel combines the
// parts of each split pair (flash-decoding's split-KV rule, applied to
// prefill rows).
#include <cuda.h>
#include <limits.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kBM = 128;                    // rows per q-tile
constexpr int kBN = 128;                    // keys per tile
constexpr int kHalfBytes = 128 * 128;       // 128 rows x 64 bf16 (one swizzle-atom column)
constexpr int kTileBytes = 2 * kHalfBytes;  // 128 rows x 128 bf16
constexpr int kThreads = 352;  // warp 0 K copies, 1 MMA, 2-9 softmax, 10 V copies
constexpr int kVWarp = 10;
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
  int64_t num_pages, num_tokens;
  int32_t B, Hq, Hkv, G, TQ, P, log2P, maxp, max_ctx;
  float scale_log2;
  // Planned launch (all null without a workspace): CTA x of the 1-D grid runs
  // kv-head x % Hkv of unit x / Hkv, units[u] = {request, q-tile pair,
  // first key tile | (end key tile << 16), partial slot or -1}.  A unit with a
  // slot covers part of its pair's keys and writes O / l and the base-2
  // log-sum-exp of each row to o_part / lse_part for the merge kernel.
  const int4* units;
  const int32_t* n_units;
  float* o_part;    // [slot][Hkv][2 q-tiles][128 rows][128]
  float* lse_part;  // [slot][Hkv][2 q-tiles][128 rows]
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

  int h, b, qp, j_lo = 0, j_hi = 1 << 30, slot = -1;
  if (p.units) {
    pdl_wait();     // the planner's unit list is complete
    pdl_trigger();  // the merge kernel may start launching; it waits for this grid
    const int u = static_cast<int>(blockIdx.x) / p.Hkv;
    h = static_cast<int>(blockIdx.x) - u * p.Hkv;
    if (u >= *p.n_units) return;
    const int4 ud = p.units[u];
    b = ud.x;
    qp = ud.y;
    j_lo = ud.z & 0xffff;
    j_hi = static_cast<int>(static_cast<uint32_t>(ud.z) >> 16);
    slot = ud.w;
  } else {
    h = blockIdx.y;
    b = blockIdx.z;
    qp = blockIdx.x;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s0 = p.cu[b], s1 = p.cu[b + 1];
  const int n = s1 - s0;
  if (2 * qp * p.TQ >= n) return;
  const int L = p.ctx[b];
  const int cap = static_cast<int>(min(static_cast<int64_t>(p.max_ctx), static_cast<int64_t>(p.maxp) << p.log2P));
  if (L == 0 && s0 >= 0 && s1 <= p.num_tokens) return;  // a padding row
  if (s0 < 0 || s1 > p.num_tokens || L < n || L > cap) {
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
  // This unit's key tiles: [j_lo, j_hi) of the pair's [0, ntg).  ntl[g] is the
  // number q-tile g processes; local tile index jl = j - j_lo.
  const int kv_len = pos0[nq - 1] + rows[nq - 1];
  j_hi = min(j_hi, ntg[nq - 1]);
  const int nt = j_hi - j_lo;
  if (nt <= 0) return;
  int ntl[2];
#pragma unroll
  for (int g = 0; g < 2; ++g) ntl[g] = max(0, min(j_hi, ntg[g]) - j_lo);

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

  // Producer lane geometry.  Block-table entries are read one tile ahead: the
  // loads for tile j + 1 are issued before tile j's stage waits, so their
  // latency is hidden behind them; tile 0's are read before the setup below.
  // kNoPage marks an entry the lane does not need.
  const bool producer = warp == 0 || warp == kVWarp;
  const bool vrole = warp == kVWarp;
  const int64_t bt_row = static_cast<int64_t>(b) * p.maxp;
  const int box = lane >> 2, half = (lane >> 1) & 1, isv = lane & 1;
  const int x = h * 128 + half * 64;
  constexpr int kNoPage = INT_MIN;
  auto load_pages = [&](int jj, int& pg_full, int& pg_rem) {
    const int t0 = (j_lo + jj) * kBN;
    const int valid = min(kBN, kv_len - t0);
    const int nfull = valid / kBoxRows, rem = valid % kBoxRows;
    pg_full = box < nfull ? p.bt[bt_row + ((t0 + box * kBoxRows) >> p.log2P)] : kNoPage;
    pg_rem = rem && lane < 4 ? p.bt[bt_row + ((t0 + nfull * kBoxRows) >> p.log2P)] : kNoPage;
  };
  int pf_next = kNoPage, pr_next = kNoPage;
  if (producer) load_pages(0, pf_next, pr_next);

  // V rows past the last key are never loaded but meet a probability of 0 in
  // the PV products, so they must hold finite values: zero both V stages.  Q
  // needs nothing (and is loaded during this setup): a q-tile in use is always
  // a whole TMA box, and an unused one is never read.
  {
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < 2 * kTileBytes / 16; i += kThreads)
      reinterpret_cast<uint4*>(smem + kOffV)[i] = z;
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
    // both Q tiles, issued before the setup barrier so that their latency overlaps it
    mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(nq * 2 * p.G * p.TQ * 128));
    for (int g = 0; g < nq; ++g) {
      const int z = s0 + (2 * qp + g) * p.TQ;
      tma_load_3d(smem + kOffQ + g * kTileBytes, &p.tm_q, 0, h * p.G, z, q_full);
      tma_load_3d(smem + kOffQ + g * kTileBytes + kHalfBytes, &p.tm_q, 64, h * p.G, z, q_full);
    }
  }

  // One K or V tile (by the role of the calling producer warp): page ids ->
  // rows of the cache, the stage's byte count, then one TMA box per lane.
  // False when the stage wait ran out.
  auto issue_tile = [&](int j, int pf, int pr) -> bool {
    const int st = j & 1;
    const uint32_t par = ((j >> 1) & 1) ^ 1;
    const int t0 = (j_lo + j) * kBN;
    const int valid = min(kBN, kv_len - t0);
    const int nfull = valid / kBoxRows, rem = valid % kBoxRows;
    int y_full = -1, y_rem = -1;
    if (pf != kNoPage) {
      const int key0 = t0 + box * kBoxRows;
      if (pf >= 0 && pf < p.num_pages) y_full = (pf << p.log2P) + (key0 & (p.P - 1));
      else raise_flag(p.err, PA_DEVERR_BAD_PAGE);
    }
    if (pr != kNoPage) {
      const int key0 = t0 + nfull * kBoxRows;
      if (pr >= 0 && pr < p.num_pages) y_rem = (pr << p.log2P) + (key0 & (p.P - 1));
      else raise_flag(p.err, PA_DEVERR_BAD_PAGE);
    }
    uint32_t mine = (y_full >= 0 ? kBoxRows * 128 : 0) + (y_rem >= 0 ? rem * 128 : 0);
    uint32_t bytes = (isv != 0) == vrole ? mine : 0;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
    uint64_t* full = vrole ? &v_full[st] : &k_full[st];
    int okw = 1;
    if (lane == 0) {
      okw = mbar_wait_bounded(vrole ? &v_empty[st] : &k_empty[st], par, abort_flag, p.err);
      if (okw) mbar_arrive_expect_tx(full, bytes);
    }
    if (__shfl_sync(0xffffffffu, okw, 0) == 0) return false;
    if ((isv != 0) == vrole) {
      unsigned char* dst = smem + (vrole ? kOffV : kOffK) + st * kTileBytes + half * kHalfBytes;
      const CUtensorMap* m16 = vrole ? &p.tm_v16 : &p.tm_k16;
      const CUtensorMap* m1 = vrole ? &p.tm_v1 : &p.tm_k1;
      if (y_full >= 0) tma_load_2d(dst + box * kBoxRows * 128, m16, x, y_full, full);
      if (y_rem >= 0)
        for (int r = 0; r < rem; ++r) tma_load_2d(dst + (nfull * kBoxRows + r) * 128, m1, x, y_rem + r, full);
    }
    return true;
  };
  // K tile 0 goes out before the setup barrier as well (the K region is not
  // zeroed, and a stage's first wait passes at once)
  int k_first = 0;
  if (warp == 0) {
    __syncwarp();  // lane 0's barrier initialisation is visible to the warp
    const int pf = pf_next, pr = pr_next;
    if (nt > 1) load_pages(1, pf_next, pr_next);
    if (issue_tile(0, pf, pr)) k_first = 1;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0 || warp == kVWarp) {
    // ------------------------------- TMA producers -------------------------------
    // warp 0 copies Q and the K tiles, warp kVWarp the V tiles; each runs ahead
    // as far as its own stages allow
    int issued = vrole ? 0 : k_first;
    bool ok = vrole || k_first == 1;
    for (int j = issued; j < nt && ok; ++j) {
      const int pf = pf_next, pr = pr_next;
      if (j + 1 < nt) load_pages(j + 1, pf_next, pr_next);
      ok = issue_tile(j, pf, pr);
      if (ok) ++issued;
    }
    if (!ok && lane == 0) {
      if (!vrole) drain(q_full, 0);
      uint64_t* full = vrole ? v_full : k_full;
      for (int j = max(0, issued - 2); j < issued; ++j) drain(&full[j & 1], (j >> 1) & 1);
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
        for (int g = 0; g < nq; ++g)
          if (ntl[g] > 0) qk(g, 0);
        mma_commit(&k_empty[0]);
      }
      for (int j = 0; j < nt && ok; ++j) {
        const bool more = j + 1 < nt;
        if (!(ok = mbar_wait_bounded(&v_full[j & 1], (j >> 1) & 1, abort_flag, p.err))) break;
        // q-tile 0: PV of tile j, then QK of tile j+1 (the tensor pipe runs them
        // in issue order, so QK overwrites S_0 only after PV has read P_0)
        if (j < ntl[0] && !(ok = pv(0, j))) break;
        if (more) {
          if (!(ok = mbar_wait_bounded(&k_full[(j + 1) & 1], ((j + 1) >> 1) & 1, abort_flag, p.err))) break;
          tc_fence_after();
          if (j + 1 < ntl[0]) qk(0, j + 1);
        }
        // q-tile 1
        if (j < ntl[1] && !(ok = pv(1, j))) break;
        if (more && j + 1 < ntl[1]) qk(1, j + 1);
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
    for (int j = 0; j < ntl[g]; ++j) {
      ok = mbar_wait_bounded(&s_full[g], j & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int key0 = (j_lo + j) * kBN;
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
          const float2 t = ffma2(make_float2(__uint_as_float(x[64 * hh + 2 * e]), __uint_as_float(x[64 * hh + 2 * e + 1])),
                                 make_float2(p.scale_log2, p.scale_log2), make_float2(neg_m, neg_m));
          const float p0 = ex2(t.x);
          const float p1 = ex2(t.y);
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
    // epilogue: O / l to global memory, or this part's partial result
    if (g < nq && slot >= 0) {
      if (ok) ok = mbar_wait_bounded(o_final, 0, abort_flag, p.err);
      const int64_t prow = ((static_cast<int64_t>(slot) * p.Hkv + h) * 2 + g) * kBM + row;
      if (__all_sync(0xffffffffu, ok)) {
        if (ntl[g] > 0) {
          tc_fence_after();
          const float inv = l > 0.f ? 1.f / l : 0.f;
          float* dstp = p.o_part + prow * 128;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + colO + 32 * c, o);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              *reinterpret_cast<float4*>(dstp + 32 * c + 4 * q4) =
                  make_float4(__uint_as_float(o[4 * q4]) * inv, __uint_as_float(o[4 * q4 + 1]) * inv,
                              __uint_as_float(o[4 * q4 + 2]) * inv, __uint_as_float(o[4 * q4 + 3]) * inv);
          }
          p.lse_part[prow] = l > 0.f ? m_used + __log2f(l) : -INFINITY;
        } else {
          p.lse_part[prow] = -INFINITY;  // no key tile of this part reaches q-tile g
        }
      }
    } else if (g < nq) {
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
  cta_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------
// planner: q-tile pairs -> units (split long key ranges, longest first)
// ---------------------------------------------------------------------------
// A CTA of the attention kernel runs one unit.  Without a plan the units are
// the q-tile pairs themselves in grid order, so a batch whose pairs fill less
// than a wave, or whose last wave holds its longest pairs, waits on its
// longest pair.  The planner (one CTA, on the device, so the launch needs no
// host copy of the lengths and can be captured in a graph) lists the pairs
// with their key-tile counts nt, chooses a part size tau, cuts every pair
// with nt > tau into ceil(nt / tau) near-equal key ranges, and writes the
// units sorted by length, longest first, so that the hardware block
// scheduler, which starts CTAs in index order as SMs free up, approximates
// longest-processing-time-first list scheduling.
//
// tau minimises an estimate of the makespan in units of one key tile of one
// CTA: a unit costs its length + 1 (prologue, epilogue) + 1 more when it is a
// part (partial store, merge); with U CTAs of largest cost c_max and mean
// load A = total cost / SMs, the estimate is min(ceil(U / SMs) * c_max,
// A + c_max) (the waves bound and the list-scheduling bound).  Splitting is
// considered only while the pairs fill at most four waves; beyond that the
// ordering alone keeps the tail short.
constexpr int kPlanThreads = 1024;
constexpr int kPlanBuckets = 2048;   // unit lengths >= 2047 tiles share the last bucket
constexpr int kPlanSmemPairs = 2048; // pairs kept in shared memory (the rest are re-read from the workspace)
constexpr int kPlanCandidates = 32;  // one per warp
constexpr int kSplitWaves = 4;
constexpr int kMaxSlots = 65535;     // slot counts are scanned in 16 bits

struct PlanParams {
  const int32_t* cu;
  const int32_t* ctx;
  unsigned int* err;
  int4* pairs;   // [pair_cap] {request, pair, nt, 0}
  int4* units;   // [pair_cap + slot_cap]
  int4* splits;  // [split_cap] {request, pair, first slot, parts}
  int32_t* hdr;  // {units, split pairs, tau, pairs}
  int64_t num_tokens;
  int32_t B, TQ, Hkv, n_sm, max_seqlen_q, cap_ctx, pair_cap, slot_cap, split_cap;
};

// Exclusive prefix sum over the CTA (blockDim.x a multiple of 32, <= 1024).
template <typename T>
PA_DEVINL T block_scan_excl(T v, T* sh, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  cta_sync();
  if (warp == 0) {
    T w = lane < nw ? sh[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh[lane] = w;
  }
  cta_sync();
  const T r = (warp > 0 ? sh[warp - 1] : T(0)) + x - v;
  *total = sh[nw - 1];
  cta_sync();
  return r;
}

PA_DEVINL int parts_of(int nt, int tau) { return (nt + tau - 1) / tau; }

// A pair of nt key tiles cut into `parts` ranges: the first nt % parts ranges
// hold one tile more than the others (lengths base + 1 and base).
__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(const PlanParams q) {
  __shared__ unsigned long long sh_scan[32];
  __shared__ int cursor[kPlanBuckets];
  __shared__ int4 sh_pairs[kPlanSmemPairs];
  __shared__ float cand_est[kPlanCandidates];
  __shared__ int cand_tau[kPlanCandidates];
  __shared__ int sh_max_nt, sh_tau;
  pdl_trigger();  // the attention kernel may start launching; it waits for this plan
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) sh_max_nt = 0;
  for (int i = tid; i < kPlanBuckets; i += kPlanThreads) cursor[i] = 0;

  // 1. the q-tile pairs of every request and their key-tile counts
  unsigned long long carry = 0;
  int max_nt = 0;
  for (int base = 0; base < q.B; base += kPlanThreads) {
    const int b = base + tid;
    int np = 0, n = 0, L = 0;
    if (b < q.B) {
      const int s0 = q.cu[b], s1 = q.cu[b + 1];
      n = s1 - s0;
      L = q.ctx[b];
      const bool padding = L == 0 && s0 >= 0 && n >= 0 && s1 <= q.num_tokens;
      if (padding)
        np = 0;
      else if (s0 < 0 || n < 0 || s1 > q.num_tokens || n > q.max_seqlen_q || L < n || L > q.cap_ctx)
        raise_flag(q.err, PA_DEVERR_BAD_LENGTH);
      else
        np = ((n + q.TQ - 1) / q.TQ + 1) / 2;
    }
    unsigned long long tot;
    const unsigned long long off = carry + block_scan_excl<unsigned long long>(np, sh_scan, &tot);
    for (int k = 0; k < np; ++k) {
      const int nt = (L - n + min((2 * k + 2) * q.TQ, n) + kBN - 1) / kBN;
      const int4 pr = make_int4(b, k, nt, 0);
      if (off + k < static_cast<unsigned long long>(q.pair_cap)) q.pairs[off + k] = pr;
      if (off + k < kPlanSmemPairs) sh_pairs[off + k] = pr;
      max_nt = max(max_nt, nt);
    }
    carry += tot;
  }
  if (max_nt > 0) atomicMax(&sh_max_nt, max_nt);
  if (carry > static_cast<unsigned long long>(q.pair_cap)) {  // lengths disagree with the workspace's sizes
    if (tid == 0) {
      raise_flag(q.err, PA_DEVERR_BAD_LENGTH);
      q.hdr[0] = q.hdr[1] = q.hdr[2] = q.hdr[3] = 0;
    }
    return;
  }
  const int n_pairs = static_cast<int>(carry);
  cta_sync();
  max_nt = sh_max_nt;
  auto pair_at = [&](int i) -> int4 { return i < kPlanSmemPairs ? sh_pairs[i] : q.pairs[i]; };

  // 2. the part size: one candidate per warp, from max_nt (no split) down to 2
  int tau = max(max_nt, 1);
  if (n_pairs > 0 && max_nt > 2 && q.slot_cap > 1 &&
      static_cast<int64_t>(n_pairs) * q.Hkv <= static_cast<int64_t>(kSplitWaves) * q.n_sm) {
    const int n_cand = min(kPlanCandidates, max_nt - 1);
    if (warp < n_cand) {
      const int c = warp;
      const int t_c = max_nt <= kPlanCandidates
                          ? max_nt - c
                          : max(2, static_cast<int>(ceilf(max_nt * exp2f(-log2f(0.5f * max_nt) * c / (n_cand - 1)))));
      int units = 0, slots = 0, work = 0, cmax = 0;
      for (int i = lane; i < n_pairs; i += 32) {
        const int nt = pair_at(i).z;
        const int parts = parts_of(nt, t_c);
        const int split = parts > 1;
        units += parts;
        slots += split ? parts : 0;
        work += nt + parts * (1 + split);
        cmax = max(cmax, (nt + parts - 1) / parts + 1 + split);
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        units += __shfl_xor_sync(0xffffffffu, units, o);
        slots += __shfl_xor_sync(0xffffffffu, slots, o);
        work += __shfl_xor_sync(0xffffffffu, work, o);
        cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
      }
      if (lane == 0) {
        const float ctas = static_cast<float>(units) * q.Hkv;
        const float waves = ceilf(ctas / q.n_sm);
        const float mean = static_cast<float>(work) * q.Hkv / q.n_sm;
        cand_est[c] = slots > q.slot_cap ? INFINITY : fminf(waves * cmax, mean + cmax);
        cand_tau[c] = t_c;
      }
    }
    cta_sync();
    if (warp == 0) {
      // arg-min; ties go to the lower index (the larger part size)
      float e = lane < n_cand ? cand_est[lane] : INFINITY;
      int c = lane;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float e2 = __shfl_xor_sync(0xffffffffu, e, o);
        const int c2 = __shfl_xor_sync(0xffffffffu, c, o);
        if (e2 < e || (e2 == e && c2 < c)) {
          e = e2;
          c = c2;
        }
      }
      if (lane == 0) sh_tau = e < INFINITY ? cand_tau[c] : max_nt;  // candidate 0 (no split) is always finite
    }
    cta_sync();
    tau = sh_tau;
  }

  // 3. histogram of unit lengths, then bucket cursors in descending length order
  for (int i = tid; i < n_pairs; i += kPlanThreads) {
    const int nt = pair_at(i).z;
    const int parts = parts_of(nt, tau), base = nt / parts, rem = nt - base * parts;
    if (rem) atomicAdd(&cursor[min(base + 1, kPlanBuckets - 1)], rem);
    if (parts > rem) atomicAdd(&cursor[min(base, kPlanBuckets - 1)], parts - rem);
  }
  cta_sync();
  {
    static_assert(kPlanBuckets == 2 * kPlanThreads, "two buckets per thread");
    const int hi = kPlanBuckets - 1 - 2 * tid, lo = hi - 1;
    const int c_hi = cursor[hi], c_lo = cursor[lo];
    unsigned long long tot;
    const int ex = static_cast<int>(block_scan_excl<unsigned long long>(c_hi + c_lo, sh_scan, &tot));
    cursor[hi] = ex;
    cursor[lo] = ex + c_hi;
    cta_sync();
  }

  // 4. units, partial slots and the split list; one scan of
  //    units (bits 0-31) | slots (32-47) | split pairs (48-63)
  unsigned long long acc = 0;
  for (int b0 = 0; b0 < n_pairs; b0 += kPlanThreads) {
    const int i = b0 + tid;
    int4 pr = make_int4(0, 0, 0, 0);
    int parts = 0;
    if (i < n_pairs) {
      pr = pair_at(i);
      parts = parts_of(pr.z, tau);
    }
    const int split = parts > 1;
    const unsigned long long mine = static_cast<unsigned long long>(parts) |
                                    (static_cast<unsigned long long>(split ? parts : 0) << 32) |
                                    (static_cast<unsigned long long>(split) << 48);
    unsigned long long tot;
    const unsigned long long before = acc + block_scan_excl<unsigned long long>(mine, sh_scan, &tot);
    if (parts > 0) {
      const int slot0 = static_cast<int>((before >> 32) & 0xffff), si = static_cast<int>(before >> 48);
      const int base = pr.z / parts, rem = pr.z - base * parts;
      const int p_hi = rem ? atomicAdd(&cursor[min(base + 1, kPlanBuckets - 1)], rem) : 0;
      const int p_lo = parts > rem ? atomicAdd(&cursor[min(base, kPlanBuckets - 1)], parts - rem) : 0;
      for (int k = 0; k < parts; ++k) {
        const int j0 = k * base + min(k, rem);
        const int j1 = j0 + base + (k < rem);
        const int pos = k < rem ? p_hi + k : p_lo + (k - rem);
        q.units[pos] = make_int4(pr.x, pr.y, j0 | (j1 << 16), split ? slot0 + k : -1);
      }
      if (split) q.splits[si] = make_int4(pr.x, pr.y, slot0, parts);
    }
    acc += tot;
  }
  if (tid == 0) {
    q.hdr[0] = static_cast<int>(acc & 0xffffffffu);
    q.hdr[1] = static_cast<int>(acc >> 48);
    q.hdr[2] = tau;
    q.hdr[3] = n_pairs;
  }
}

// ---------------------------------------------------------------------------
// merge of split pairs: O = sum_k 2^(lse_k - M) O_k / sum_k 2^(lse_k - M)
// ---------------------------------------------------------------------------
constexpr int kMergeThreads = 256;                     // 8 warps = 8 rows per CTA
constexpr int kMergeRowBlocks = 2 * kBM / (kMergeThreads / 32);

struct MergeParams {
  const int32_t* cu;
  const int4* splits;
  const int32_t* hdr;
  const float* o_part;
  const float* lse_part;
  char* out;
  int32_t Hq, Hkv, G, TQ;
};

// CTA = (8 rows of a split pair, kv-head); a warp per row, 4 dims per lane.
// The parts' log-sum-exps are loaded one per lane and reduced by shuffles;
// the O loads of four parts are in flight together.
__global__ void __launch_bounds__(kMergeThreads) prefill_merge_kernel(const MergeParams m) {
  pdl_wait();  // every part of the attention grid is written
  const int si = blockIdx.x / kMergeRowBlocks, h = blockIdx.y;
  if (si >= m.hdr[1]) return;
  const int4 sp = m.splits[si];
  const int b = sp.x, qp = sp.y, slot0 = sp.z, parts = sp.w;
  const int s0 = m.cu[b], n = m.cu[b + 1] - s0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (blockIdx.x % kMergeRowBlocks) * (kMergeThreads / 32) + warp;  // row of the pair, 0..255
  const int g = r / kBM, row = r % kBM;
  const int t = row / m.G, gg = row - t * m.G;
  const int tok = (2 * qp + g) * m.TQ + t;
  if (tok >= n) return;
  const int64_t slot_stride = static_cast<int64_t>(m.Hkv) * 2 * kBM;  // rows per slot
  const int64_t r0 = (static_cast<int64_t>(slot0) * m.Hkv + h) * 2 * kBM + r;
  float mx = -INFINITY;
  for (int k = lane; k < parts; k += 32) mx = fmaxf(mx, m.lse_part[r0 + k * slot_stride]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  for (int k0 = 0; k0 < parts; k0 += 32) {
    const int k = k0 + lane;
    const float lse = k < parts ? m.lse_part[r0 + k * slot_stride] : -INFINITY;
    const float w_mine = lse == -INFINITY ? 0.f : exp2f(lse - mx);
    const int kn = min(32, parts - k0);
#pragma unroll 4
    for (int i = 0; i < kn; ++i) {
      const float w = __shfl_sync(0xffffffffu, w_mine, i);
      const float4 o =
          *reinterpret_cast<const float4*>(m.o_part + (r0 + (k0 + i) * slot_stride) * 128 + 4 * lane);
      if (w != 0.f) {
        acc.x = fmaf(w, o.x, acc.x);
        acc.y = fmaf(w, o.y, acc.y);
        acc.z = fmaf(w, o.z, acc.z);
        acc.w = fmaf(w, o.w, acc.w);
        wsum += w;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint2 v;
  v.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  v.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(m.out + ((static_cast<int64_t>(s0) + tok) * m.Hq + h * m.G + gg) * 256 + 8 * lane) = v;
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

cudaError_t plan_prefill(const pa_cache_desc& d, int32_t batch, int32_t max_seqlen_q, int64_t num_tokens,
                         int32_t max_context_len, PrefillPlan* out) {
  memset(out, 0, sizeof(*out));
  // Only the tensor-core path is planned; unit descriptors hold key tiles in 16 bits.
  if (d.dtype != PA_BF16 || d.head_dim != 128) return cudaSuccess;
  if ((static_cast<int64_t>(max_context_len) + kBN - 1) / kBN > 0xffff) return cudaSuccess;
  if (batch < 1 || max_seqlen_q < 1 || num_tokens < 1) return cudaSuccess;
  DeviceInfo di;
  cudaError_t e = current_device_info(&di);
  if (e != cudaSuccess) return e;
  const int G = d.num_q_heads / d.num_kv_heads, TQ = kBM / G;
  const int64_t pmax = ((max_seqlen_q + TQ - 1) / TQ + 1) / 2;
  const int64_t pair_cap = std::min<int64_t>(batch * pmax, num_tokens / (2 * TQ) + batch);
  if (pair_cap > (1 << 30)) return cudaSuccess;
  PrefillPlan& pl = *out;
  pl.n_sm = di.sm_count;
  pl.pair_cap = static_cast<int32_t>(pair_cap);
  // Layout capacities: they grow with the bounds only, so a workspace sized
  // for the largest call serves every smaller one.
  pl.slot_cap = std::min(kMaxSlots, (kSplitWaves * di.sm_count + d.num_kv_heads - 1) / d.num_kv_heads);
  pl.split_cap = pl.slot_cap / 2;
  pl.unit_cap = pl.pair_cap + pl.slot_cap;
  // This call: the planner splits only while the pairs fill at most
  // kSplitWaves waves, and there are at least num_tokens / (2 TQ) pairs, so
  // when those alone fill more nothing is split and no merge is launched.  A
  // split pair is one of the pairs, so at most pair_cap of them: the merge grid
  // is sized by that bound too (its CTAs past the planner's count exit at once,
  // but still cost a launch).
  const bool no_split = num_tokens / (2 * TQ) * d.num_kv_heads > static_cast<int64_t>(kSplitWaves) * di.sm_count;
  pl.run_slot_cap = no_split ? 0 : pl.slot_cap;
  pl.run_split_cap = no_split ? 0 : static_cast<int32_t>(std::min<int64_t>(pl.split_cap, pair_cap));
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t off = 0;
  pl.off_hdr = off;
  off = up(off + 4 * sizeof(int32_t));
  pl.off_pairs = off;
  off = up(off + static_cast<size_t>(pl.pair_cap) * sizeof(int4));
  pl.off_units = off;
  off = up(off + static_cast<size_t>(pl.unit_cap) * sizeof(int4));
  pl.off_splits = off;
  off = up(off + static_cast<size_t>(std::max(pl.split_cap, 1)) * sizeof(int4));
  const size_t rows = static_cast<size_t>(pl.slot_cap) * d.num_kv_heads * 2 * kBM;
  pl.off_lse = off;
  off = up(off + rows * sizeof(float));
  pl.off_o = off;
  off = up(off + rows * 128 * sizeof(float));
  pl.ws_bytes = off;
  return cudaSuccess;
}

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
  p.num_tokens = a.num_tokens;
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
  if (!a.workspace) {
    const int qtiles = (a.max_seqlen_q + TQ - 1) / TQ;
    const dim3 grid((qtiles + 1) / 2, d.num_kv_heads, a.batch);
    prefill_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
  }

  // planned launch: planner -> attention units -> merge of split pairs
  PrefillPlan pl;
  cudaError_t e = plan_prefill(d, a.batch, a.max_seqlen_q, a.num_tokens, a.max_context_len, &pl);
  if (e != cudaSuccess) return e;
  if (pl.ws_bytes == 0 || a.workspace_bytes < pl.ws_bytes) return cudaErrorInvalidValue;
  char* ws = static_cast<char*>(a.workspace);
  PlanParams q;
  q.cu = a.cu_seqlens_q;
  q.ctx = a.context_lens;
  q.err = a.err;
  q.pairs = reinterpret_cast<int4*>(ws + pl.off_pairs);
  q.units = reinterpret_cast<int4*>(ws + pl.off_units);
  q.splits = reinterpret_cast<int4*>(ws + pl.off_splits);
  q.hdr = reinterpret_cast<int32_t*>(ws + pl.off_hdr);
  q.num_tokens = a.num_tokens;
  q.B = a.batch;
  q.TQ = TQ;
  q.Hkv = d.num_kv_heads;
  q.n_sm = pl.n_sm;
  q.max_seqlen_q = a.max_seqlen_q;
  q.cap_ctx = static_cast<int32_t>(std::min<int64_t>(a.max_context_len, int64_t(a.max_pages) << p.log2P));
  q.pair_cap = pl.pair_cap;
  q.slot_cap = pl.run_slot_cap;
  q.split_cap = pl.run_split_cap;
  prefill_plan_kernel<<<1, kPlanThreads, 0, s>>>(q);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  p.units = q.units;
  p.n_units = q.hdr;
  p.lse_part = reinterpret_cast<float*>(ws + pl.off_lse);
  p.o_part = reinterpret_cast<float*>(ws + pl.off_o);
  {
    void* args[] = {&p};
    e = launch_after_previous(reinterpret_cast<const void*>(prefill_tc_kernel),
                              dim3(static_cast<unsigned>(pl.pair_cap + pl.run_slot_cap) * d.num_kv_heads),
                              dim3(kThreads), kSmemBytes, s,
                              args);
    if (e != cudaSuccess) return e;
  }

  if (pl.run_split_cap > 0) {
    MergeParams m;
    m.cu = a.cu_seqlens_q;
    m.splits = q.splits;
    m.hdr = q.hdr;
    m.o_part = p.o_part;
    m.lse_part = p.lse_part;
    m.out = p.out;
    m.Hq = d.num_q_heads;
    m.Hkv = d.num_kv_heads;
    m.G = G;
    m.TQ = TQ;
    void* args[] = {&m};
    e = launch_after_previous(reinterpret_cast<const void*>(prefill_merge_kernel),
                              dim3(pl.run_split_cap * kMergeRowBlocks, d.num_kv_heads), dim3(kMergeThreads), 0, s,
                              args);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pa
