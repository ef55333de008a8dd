// Chunked-prefill attention on the 5th-generation tensor cores (sm_103a):
// tcgen05.mma with fp32 accumulators in tensor memory, operands staged by TMA,
// bf16 inputs, head_dim 128.
//
// Semantics (nano-vLLM learning note, Attention.forward / prepare_prefill
// listings; qwen-engine README, flat varlen packing): row i of request b's
// chunk sits at position context_lens[b] - n_b + i and attends to keys
// 0 .. that position, all read from the paged cache.
//
// Work item = (q-tile pair of a request, kv-head, range of 128-key tiles).  A
// q-tile is 128 rows: TQ = 128 / G tokens x the G q-heads that share the
// kv-head, so each staged K/V tile feeds the whole GQA group.  A pair with
// two q-tiles runs in pair mode: each K/V tile feeds both (256 rows).  A
// pair with one q-tile (a short chunk) runs in split mode: its key tiles
// alternate between the two softmax groups, each keeping its own O and row
// statistics, and the first group merges the two halves at the end.
//
// Planned launch (the caller gives a workspace): a one-CTA planner kernel
// lists the pairs, cuts long key ranges into parts and lists the units
// longest first; the attention kernel is persistent -- one CTA per SM takes
// items (unit x kv-head) from a shared counter as it frees up -- and a part
// writes O / l and the row log-sum-exp in fp32 for a merge kernel that
// combines the parts of each split pair (flash-decoding's split-KV rule,
// applied to prefill rows).  Without a workspace, each CTA runs its own
// pair's item with all its keys.  Launched by the prefill step right after its
// KV-write kernel, the planner starts beside that kernel (it reads only the
// varlen metadata) and waits for it before it exits.
//
// Warp roles (12 warps):
//   warps 0-7  two softmax groups of 4 warps, one thread per row (= TMEM
//              lane): a tile's 128 scores come into registers in one TMEM
//              round trip, the row max is taken, O in TMEM is rescaled only
//              when a row max grows by more than 2^8, and the bf16
//              probabilities are written back over S's first 64 columns,
//              where the PV MMA reads its A operand.  At an item's end O / l
//              goes to global memory (O is released to the next item as soon
//              as it is in registers): a warp whose 32 rows are whole tokens
//              stages them in shared memory and lane 0 issues TMA stores, so
//              the warp does not wait on its stores; other rows are stored
//              by their threads.
//   warp 8     TMA producer of Q and K: an item's Q tiles (3-D map), then
//              per 128-key tile the K rows gathered page by page with 16-row
//              boxes (single-row boxes for a ragged end, so no slot past the
//              context is read); block-table entries are read one tile ahead.
//   warp 9     TMA producer of V, the same way; K and V run ahead of the MMAs
//              independently in two-stage rings that continue across items.
//   warp 10    allocates all 512 TMEM columns; lane 0 issues the MMAs:
//              S_g = Q K^T and O_g += P_g V for the two groups, in the order
//              PV_0, QK_0 of the next step, PV_1, QK_1 of the next step, so
//              that each softmax group has a PV and a QK of the other group
//              to hide in.
//   warp 11    work scheduler: takes the next item when the CTA's current
//              item has all its K tiles issued, and hands it to the others
//              through a two-slot ring in shared memory.
// The softmax warpgroups run with 200 registers, the warpgroup of warps 8-11
// with 104 (setmaxnreg; the launch gives 168 to every thread).
// TMEM: S_0 cols 0-127 (P_0 in 0-63), S_1 128-255 (P_1 in 128-191),
//       O_0 256-383, O_1 384-511.
// Every wait is bounded; a timeout raises PA_DEVERR_TIMEOUT and the CTA
// drains its copies and MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <limits.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kBM = 128;                    // rows per q-tile
constexpr int kBN = 128;                    // keys per tile
constexpr int kHalfBytes = 128 * 128;       // 128 rows x 64 bf16 (one swizzle-atom column)
constexpr int kTileBytes = 2 * kHalfBytes;  // 128 rows x 128 bf16
// warps 0-3 softmax group 0, 4-7 softmax group 1, 8 Q and K copies, 9 V copies,
// 10 MMA issuer, 11 work scheduler
constexpr int kThreads = 384;
constexpr int kKWarp = 8, kVWarp = 9, kMmaWarp = 10, kSchedWarp = 11;
constexpr int kItemConsumers = 11;  // warps that take each work item: the copies, the MMA issuer, 8 softmax
// Per-thread registers: at launch (the kernel must be built with exactly this
// many; the host checks), and after the warpgroups rebalance.
constexpr int kLaunchRegs = 168, kSoftmaxRegs = 200, kRoleRegs = 104;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kRoleRegs <= kThreads * kLaunchRegs,
              "the rebalanced registers fit in the launch allocation");
constexpr int kBoxRows = 16;
constexpr uint32_t kTmemCols = 512;

constexpr int kOffQ = 0;                          // two q-tiles
constexpr int kOffK = kOffQ + 2 * kTileBytes;     // two K stages
constexpr int kOffV = kOffK + 2 * kTileBytes;     // two V stages
constexpr int kStageBytes = 32 * 128;             // a softmax warp's 32 rows x 128 bytes on their way out
constexpr int kOffStage = kOffV + 2 * kTileBytes; // eight softmax warps' output staging (1024-aligned)
constexpr int kOffBar = kOffStage + 8 * kStageBytes;  // 26 mbarriers
// indices of the mbarriers in their table (pairs are [2], one per stage or group)
constexpr int kBarItemFull = 0, kBarItemEmpty = 2, kBarQFull = 4, kBarQEmpty = 5, kBarKFull = 6, kBarKEmpty = 8,
              kBarVFull = 10, kBarVEmpty = 12, kBarSFull = 14, kBarPFull = 16, kBarPvDone = 18, kBarOFree = 20,
              kBarMlFull = 22, kBarMlEmpty = 23, kBarMmaDone = 24, kBarSchedGo = 25;
constexpr int kOffItem = kOffBar + 256;           // two work items
constexpr int kOffMl = kOffItem + 256;            // 128 (max, sum) rows handed between the softmax groups
constexpr int kOffMisc = kOffMl + 128 * 8;        // TMEM base address, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
static_assert(kSmemBytes <= 232448, "within the 227 KB a CTA may use");
static_assert(kOffStage % 1024 == 0, "128-byte-swizzled staging starts on a 1024-byte boundary");

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
  CUtensorMap tm_o;    // out    [num_tokens, Hq, 128], box {64, G, 32 / G}: one softmax warp's rows
  int32_t o_tma;       // 1: tm_o is valid (G a power of two, so a warp's 32 rows are whole tokens)
  const int32_t* cu;
  const int32_t* bt;
  const int32_t* ctx;
  char* out;
  unsigned int* err;
  int64_t num_pages, num_tokens;
  int32_t B, Hq, Hkv, G, TQ, P, log2P, maxp, max_ctx;
  float scale_log2;
  // Planned launch (all null without a workspace): the CTAs take work items
  // k = unit * Hkv + kv-head from *counter, units[u] = {request, q-tile pair,
  // first key tile | (end key tile << 16), partial slot or -1}.  A unit with a
  // slot covers part of its pair's keys and writes O / l and the base-2
  // log-sum-exp of each row to o_part / lse_part for the merge kernel.
  const int4* units;
  const int32_t* n_units;
  int32_t* counter;  // next item to hand out (zeroed by the planner)
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

// Shared -> global copy of a 3-D box (bulk async-group of the issuing thread).
PA_DEVINL void tma_store_3d(const CUtensorMap* tm, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}

PA_DEVINL void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
PA_DEVINL void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
PA_DEVINL void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

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
// One (unit, kv-head) of work, as the scheduler warp hands it to the others.
struct Item {
  int32_t valid;    // 0: no more work for this CTA
  int32_t b, h, qp; // request, kv-head, q-tile pair
  int32_t j_lo, nt; // key tiles [j_lo, j_lo + nt)
  int32_t slot;     // partial-result slot of a split pair, or -1
  int32_t s0;       // the request's first packed row
  int32_t nq;       // q-tiles of the pair with rows (1 or 2)
  int32_t split;    // 1: one q-tile whose key tiles alternate between the two softmax groups
  int32_t c[2];     // key tiles softmax group g processes
  int32_t qt[2];    // q-tile of the pair (0 or 1) group g works on
  int32_t rows[2];  // live tokens of that q-tile
  int32_t pos0[2];  // position of its first token
  int32_t kv_len;   // keys the pair needs (last token's position + 1)
  int32_t pad[5];
};
static_assert(sizeof(Item) == 96, "two items fit their shared-memory slot");

// The work of pair qp of request b for kv-head h over key tiles [j_lo, j_hi).
// False when there is none (a padding row, an empty range, a pair without
// rows) or the request's lengths are inconsistent (flagged).
PA_DEVINL bool make_item(const TcParams& p, int b, int qp, int h, int j_lo, int j_hi, int slot, Item& it) {
  const int s0 = p.cu[b], s1 = p.cu[b + 1];
  const int n = s1 - s0;
  const int L = p.ctx[b];
  if (L == 0 && s0 >= 0 && s1 <= p.num_tokens) return false;  // a padding row
  const int cap = static_cast<int>(min(static_cast<int64_t>(p.max_ctx), static_cast<int64_t>(p.maxp) << p.log2P));
  if (s0 < 0 || s1 > p.num_tokens || n < 0 || L < n || L > cap) {
    raise_flag(p.err, PA_DEVERR_BAD_LENGTH);
    return false;
  }
  if (2 * qp * p.TQ >= n) return false;
  const int nq = (2 * qp + 1) * p.TQ < n ? 2 : 1;
  int rows[2], pos0[2], ntg[2];
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int qt = 2 * qp + g;
    rows[g] = g < nq ? min(p.TQ, n - qt * p.TQ) : 0;
    pos0[g] = L - n + qt * p.TQ;
    ntg[g] = g < nq ? (pos0[g] + rows[g] + kBN - 1) / kBN : 0;
  }
  j_hi = min(j_hi, ntg[nq - 1]);
  const int nt = j_hi - j_lo;
  if (nt <= 0) return false;
  it.valid = 1;
  it.b = b;
  it.h = h;
  it.qp = qp;
  it.j_lo = j_lo;
  it.nt = nt;
  it.slot = slot;
  it.s0 = s0;
  it.nq = nq;
  it.split = nq == 1;
  it.kv_len = pos0[nq - 1] + rows[nq - 1];
  if (it.split) {
    it.c[0] = (nt + 1) / 2;
    it.c[1] = nt / 2;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      it.qt[g] = 0;
      it.rows[g] = rows[0];
      it.pos0[g] = pos0[0];
    }
  } else {
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      it.c[g] = max(0, min(j_hi, ntg[g]) - j_lo);
      it.qt[g] = g;
      it.rows[g] = rows[g];
      it.pos0[g] = pos0[g];
    }
  }
  return true;
}

// Wait (lane 0) for work item i, copy it to every lane and release its slot.
// False when the wait ran out.
PA_DEVINL bool take_item(Item* items, uint64_t* item_full, uint64_t* item_empty, int i, volatile int* abort_flag,
                         unsigned int* err, Item& it) {
  const int s = i & 1;
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(&item_full[s], (i >> 1) & 1, abort_flag, err);
  if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
  it = items[s];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&item_empty[s]);
  return true;
}

// The same for a role that runs on one lane (the MMA issuer).
PA_DEVINL bool take_item_lane(Item* items, uint64_t* item_full, uint64_t* item_empty, int i,
                              volatile int* abort_flag, unsigned int* err, Item& it) {
  const int s = i & 1;
  if (!mbar_wait_bounded(&item_full[s], (i >> 1) & 1, abort_flag, err)) return false;
  it = items[s];
  mbar_arrive(&item_empty[s]);
  return true;
}



// mbarrier helpers on 32-bit shared-memory addresses (the MMA issuer names its
// barriers as base + 8 * index, so no 64-bit pointers stay live).
PA_DEVINL bool try_wait_a(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

PA_DEVINL bool wait_a(uint32_t bar, uint32_t parity, volatile int* abort, unsigned int* err) {
  if (try_wait_a(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (try_wait_a(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        raise_flag(err, PA_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

PA_DEVINL void commit_a(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// The 8 MMAs (k = 16 dims each) of S = Q K^T for one 128 x 128 tile, and of
// O (+)= P V with P from tensor memory.  An operand descriptor is passed as
// its low 32 bits (address >> 4 and leading offset), the high half being the
// same for every operand here (stride 1024, descriptor version, 128-byte
// swizzle); the k-th operand is the tile's low half plus its address offset >> 4.
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);

PA_DEVINL uint32_t desc_lo(uint32_t saddr, uint32_t lbo) { return ((saddr & 0x3FFFFu) >> 4) | ((lbo >> 4) << 16); }

PA_DEVINL void mma_ss(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "mov.b64 da, {%1, %5};\n\t"
      "mov.b64 db, {%2, %5};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(acc), "n"(kDescHi)
      : "memory");
}

PA_DEVINL void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "mov.b64 db, {%2, %5};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(acc), "n"(kDescHi)
      : "memory");
}

PA_DEVINL void issue_qk(uint32_t d_s, uint32_t a_lo, uint32_t b_lo) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t off = ((k >> 2) * kHalfBytes + (k & 3) * 32) >> 4;
    mma_ss(d_s, a_lo + off, b_lo + off, kIdescQK, k > 0);
  }
}

PA_DEVINL void issue_pv(uint32_t d_o, uint32_t a_p, uint32_t v_lo, bool first) {
#pragma unroll
  for (int k = 0; k < 8; ++k)
    mma_ts(d_o, a_p + k * 8, v_lo + ((k * 16 * 128) >> 4), kIdescPV, (!first || k > 0) ? 1u : 0u);
}

// 32-byte global stores (one whole sector per lane).
PA_DEVINL void stg32(void* ptr, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4, uint32_t a5,
                     uint32_t a6, uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(a0), "r"(a1), "r"(a2),
               "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

// O columns [32 * Q0, 32 * Q0 + N) of a row to global memory, scaled by a:
// fp32 into the part's slot row, or bf16 into the output row when the row is
// live (all indices known at compile time, so `o` stays in registers).
template <int Q0, int N>
PA_DEVINL void store_cols(const uint32_t (&o)[N], float a, bool part, bool live, float* part_row, char* out_row,
                          bool out32) {
  auto f = [&](int e) { return __uint_as_float(o[e]) * a; };
  if (part) {
    float* dstp = part_row + 32 * Q0;
#pragma unroll
    for (int q8 = 0; q8 < N / 8; ++q8)
      stg32(dstp + 8 * q8, __float_as_uint(f(8 * q8)), __float_as_uint(f(8 * q8 + 1)), __float_as_uint(f(8 * q8 + 2)),
            __float_as_uint(f(8 * q8 + 3)), __float_as_uint(f(8 * q8 + 4)), __float_as_uint(f(8 * q8 + 5)),
            __float_as_uint(f(8 * q8 + 6)), __float_as_uint(f(8 * q8 + 7)));
  } else if (live) {
#pragma unroll
    for (int q16 = 0; q16 < N / 16; ++q16) {
      const int e = 16 * q16;
      const uint32_t w0 = pack_bf16x2(f(e), f(e + 1)), w1 = pack_bf16x2(f(e + 2), f(e + 3));
      const uint32_t w2 = pack_bf16x2(f(e + 4), f(e + 5)), w3 = pack_bf16x2(f(e + 6), f(e + 7));
      const uint32_t w4 = pack_bf16x2(f(e + 8), f(e + 9)), w5 = pack_bf16x2(f(e + 10), f(e + 11));
      const uint32_t w6 = pack_bf16x2(f(e + 12), f(e + 13)), w7 = pack_bf16x2(f(e + 14), f(e + 15));
      char* dst = out_row + Q0 * 64 + q16 * 32;
      if (out32) {
        stg32(dst, w0, w1, w2, w3, w4, w5, w6, w7);
      } else {  // an output only 16-byte aligned
        stg16(dst, make_uint4(w0, w1, w2, w3));
        stg16(dst + 16, make_uint4(w4, w5, w6, w7));
      }
    }
  }
}

// A softmax warp's 32 output rows (whole tokens: G q-heads each), scaled by
// a and rounded to bf16, through its 4 KB staging buffer and two TMA stores
// of half a row each.  Chunk c (16 bytes) of row r sits at chunk c ^ (r & 7)
// of the row's 128 bytes -- the 128-byte swizzle the tensor map names, so
// neither these writes nor the TMA engine's reads meet a bank conflict.  The
// warp does not wait for the global writes; before it refills the buffer,
// lane 0 (whose bulk groups these are) waits until the previous store has
// read it.
PA_DEVINL void store_rows_tma(const uint32_t (&o)[128], float a, uint32_t stage, const CUtensorMap* tm, int y,
                              int z, int lane, bool& pending) {
  auto f = [&](int e) { return __uint_as_float(o[e]) * a; };
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (pending) {
      if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      __syncwarp();
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int e = 64 * h + 8 * c;
      const uint32_t addr = stage + static_cast<uint32_t>(lane * 128 + ((c ^ (lane & 7)) << 4));
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pack_bf16x2(f(e), f(e + 1))),
                   "r"(pack_bf16x2(f(e + 2), f(e + 3))), "r"(pack_bf16x2(f(e + 4), f(e + 5))),
                   "r"(pack_bf16x2(f(e + 6), f(e + 7)))
                   : "memory");
    }
    fence_async_smem();  // the rows are visible to the TMA engine
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tm, stage, 64 * h, y, z);
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    pending = true;
  }
}

struct SoftmaxArgs {
  const CUtensorMap* tm_o;  // output rows by TMA (null: by the threads' own stores)
  char* out;
  bool out32;  // out is 32-byte aligned (whole-sector stores)
  float* o_part;
  float* lse_part;
  unsigned int* err;
  int32_t Hq, Hkv, G, TQ;
  float scale_log2;
};

// The two softmax warpgroups (warps 0-7).  A function of its own, entered
// after the warpgroups' register rebalance, so that it is compiled for the
// larger register budget.
__device__ __noinline__ void softmax_role(const SoftmaxArgs p, unsigned char* smem, uint32_t tmem, int warp,
                                          int lane) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* item_full = bars + kBarItemFull;
  uint64_t* item_empty = bars + kBarItemEmpty;
  uint64_t* s_full = bars + kBarSFull;
  uint64_t* p_full = bars + kBarPFull;
  uint64_t* pv_done = bars + kBarPvDone;
  uint64_t* o_free = bars + kBarOFree;
  uint64_t* ml_full = bars + kBarMlFull;
  uint64_t* ml_empty = bars + kBarMlEmpty;
  Item* items = reinterpret_cast<Item*>(smem + kOffItem);
  float2* ml = reinterpret_cast<float2*>(smem + kOffMl);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc) + 1;
  // ------------------------------- softmax groups -------------------------------
  // Group g (warps 4g .. 4g+3) owns S_g / O_g; a thread owns one row (TMEM
  // lane).  Pair mode: group g works on q-tile g with all its key tiles.
  // Split mode (one q-tile): both groups work on q-tile 0, group g on the
  // item's key tiles g, g+2, g+4, ...; group 0's epilogue merges the two
  // partial results (the split-KV rule within one CTA).
  const int g = warp >> 2;
  const int wq = warp & 3;  // TMEM lane quarter this warp may access
  const int row = wq * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t colS = g * 128, colO = 256 + g * 128;
  const int t_r = row / p.G, gg = row - (row / p.G) * p.G;
  const uint32_t stage = smem_u32(smem + kOffStage + warp * kStageBytes);
  bool tma_pending = false;  // this warp has output stores in flight
  int sc = 0;          // S tiles this group has consumed
  int pc[2] = {0, 0};  // PVs issued per group before the current item
  int ms = 0;          // split-mode items done
  bool ok = true;
  for (int i = 0; ok; ++i) {
    Item it;
    if (!take_item(items, item_full, item_empty, i, abort_flag, p.err, it)) {
      ok = false;
      break;
    }
    if (!it.valid) break;
    const int c0 = it.c[0], c1 = it.c[1];
    const int c = g ? c1 : c0;
    const int p0 = g ? it.pos0[1] : it.pos0[0];
    const int qtg = g ? it.qt[1] : it.qt[0];
    const int pos_r = p0 + t_r;
    const bool live = row < p.TQ * p.G && t_r < (g ? it.rows[1] : it.rows[0]);
    const int j_lo = it.j_lo, split = it.split, slot = it.slot, hh_kv = it.h;
    const int it_qp = it.qp, it_s0 = it.s0;
    float m_used = -INFINITY, l = 0.f;
    for (int s = 0; s < c; ++s) {
      ok = mbar_wait_bounded(&s_full[g], sc & 1, abort_flag, p.err);
      ++sc;
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int key0 = (j_lo + (split ? 2 * s + g : s)) * kBN;
      const bool need_mask = key0 + kBN - 1 > p0;
      // One TMEM round trip per tile: all 128 scores of the row are loaded
      // (four loads, one wait), the row max is taken over the raw scores (the
      // scale is positive, so it commutes with the max) with eight independent
      // accumulators, and the probabilities are computed from registers.
      uint32_t x[128];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32_async(tmem + lane_off + colS + 32 * q, x + 32 * q);
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_wait_ld32(x + 32 * q);
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
        if (s > 0) {
          // rescale O_g once the previous PV into it has completed
          ok = mbar_wait_bounded(&pv_done[g], (pc[g] + s - 1) & 1, abort_flag, p.err);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + colO + 32 * q, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tmem + lane_off + colO + 32 * q, o);
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
          const float2 tv = ffma2(make_float2(__uint_as_float(x[64 * hh + 2 * e]), __uint_as_float(x[64 * hh + 2 * e + 1])),
                                  make_float2(p.scale_log2, p.scale_log2), make_float2(neg_m, neg_m));
          const float p0v = ex2(tv.x);
          const float p1v = ex2(tv.y);
          rs4[e & 3] = fadd2(rs4[e & 3], make_float2(p0v, p1v));
          w[e] = pack_bf16x2(p0v, p1v);
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
    if (!ok) break;
    const int last_pv0 = pc[0] + c0 - 1, last_pv1 = pc[1] + c1 - 1;  // running indices
    pc[0] += c0;
    pc[1] += c1;
    const int qt = 2 * it_qp + qtg;  // q-tile index in the request
    const int64_t prow = ((static_cast<int64_t>(slot) * p.Hkv + hh_kv) * 2 + qtg) * kBM + row;
    char* dst = p.out + ((static_cast<int64_t>(it_s0) + qt * p.TQ + t_r) * p.Hq + hh_kv * p.G + gg) * 256;
    if (!split) {
      // ------------- pair mode epilogue: this group's q-tile -------------
      if (c > 0) {
        ok = mbar_wait_bounded(&pv_done[g], (g ? last_pv1 : last_pv0) & 1, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the whole row in one TMEM round trip; O_g is free for the next item
        // as soon as it is in registers
        uint32_t o[128];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32_async(tmem + lane_off + colO + 32 * q, o + 32 * q);
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_wait_ld32(o + 32 * q);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&o_free[g]);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        if (p.tm_o != nullptr && slot < 0 && __all_sync(0xffffffffu, live))
          store_rows_tma(o, inv, stage, p.tm_o, hh_kv * p.G, it_s0 + qt * p.TQ + wq * 32 / p.G, lane, tma_pending);
        else
          store_cols<0>(o, inv, slot >= 0, live, p.o_part + prow * 128, dst, p.out32);
        if (slot >= 0) p.lse_part[prow] = l > 0.f ? m_used + __log2f(l) : -INFINITY;
      } else if (slot >= 0) {
        p.lse_part[prow] = -INFINITY;  // no key tile of this part reaches the q-tile
      }
    } else if (g == 1) {
      // ------------- split mode: group 1 hands its row statistics over -------------
      if (ms > 0) {
        ok = mbar_wait_bounded(ml_empty, (ms - 1) & 1, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
      }
      ml[row] = make_float2(m_used, l);
      __syncwarp();
      if (lane == 0) mbar_arrive(ml_full);
      ++ms;
    } else {
      // ------------- split mode: group 0 merges both halves of the keys -------------
      ok = mbar_wait_bounded(&pv_done[0], last_pv0 & 1, abort_flag, p.err) &&
           mbar_wait_bounded(ml_full, ms & 1, abort_flag, p.err) &&
           (c1 == 0 || mbar_wait_bounded(&pv_done[1], last_pv1 & 1, abort_flag, p.err));
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float2 m1 = ml[row];
      const float mm = fmaxf(m_used, m1.x);
      const float w0 = m_used == -INFINITY ? 0.f : ex2(m_used - mm);
      const float w1 = m1.x == -INFINITY ? 0.f : ex2(m1.x - mm);
      const float lsum = w0 * l + w1 * m1.y;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      const float a0 = w0 * inv, a1 = w1 * inv;
      const bool two = c1 > 0;
      // half a row of each O per TMEM round trip (the other group's O only
      // when it ran: otherwise it holds an earlier item's values)
      // a quarter row of each O per TMEM round trip (the other group's O only
      // when it ran: otherwise it holds an earlier item's values)
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t o[32];
        if (two) {
          uint32_t o1[32];
          tmem_ld32_async(tmem + lane_off + 256 + 32 * q, o);
          tmem_ld32_async(tmem + lane_off + 384 + 32 * q, o1);
          tmem_wait_ld32(o);
          tmem_wait_ld32(o1);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            o[e] = __float_as_uint(fmaf(__uint_as_float(o[e]), a0, __uint_as_float(o1[e]) * a1));
        } else {
          tmem_ld32(tmem + lane_off + 256 + 32 * q, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a0);
        }
        store_cols<0>(o, 1.f, slot >= 0, live, p.o_part + prow * 128 + 32 * q, dst + 64 * q, p.out32);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(ml_empty);
        mbar_arrive(&o_free[0]);
        if (two) mbar_arrive(&o_free[1]);
      }
      if (slot >= 0) p.lse_part[prow] = lsum > 0.f ? mm + __log2f(lsum) : -INFINITY;
      ++ms;
    }
  }
  // the output stores have completed (and read their staging) before the CTA exits
  if (tma_pending && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (p.units) {
    pdl_trigger();  // the merge kernel may start launching; it waits for this grid
  } else {
    // one pair per CTA: a pair without rows leaves at once (the same for every thread)
    const int b = blockIdx.z;
    if (2 * static_cast<int>(blockIdx.x) * p.TQ >= p.cu[b + 1] - p.cu[b]) return;
  }

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* item_full = bars + kBarItemFull;    // [2] scheduler -> all roles
  uint64_t* item_empty = bars + kBarItemEmpty;   // [2] all roles -> scheduler
  uint64_t* q_full = bars + kBarQFull;       // the item's Q tiles landed
  uint64_t* q_empty = bars + kBarQEmpty;      // the item's last QK is done
  uint64_t* k_full = bars + kBarKFull;       // [2] K stages
  uint64_t* k_empty = bars + kBarKEmpty;
  uint64_t* v_full = bars + kBarVFull;      // [2] V stages
  uint64_t* v_empty = bars + kBarVEmpty;
  uint64_t* s_full = bars + kBarSFull;      // [2] per softmax group: S = Q K^T in TMEM
  uint64_t* p_full = bars + kBarPFull;      // [2] probabilities written
  uint64_t* pv_done = bars + kBarPvDone;     // [2] a PV of the group completed
  uint64_t* o_free = bars + kBarOFree;      // [2] O of the group read out by the epilogue
  uint64_t* ml_full = bars + kBarMlFull;     // group 1's (max, sum) rows handed to group 0
  uint64_t* ml_empty = bars + kBarMlEmpty;    // group 0 has read them
  uint64_t* mma_done = bars + kBarMmaDone;    // every MMA of the CTA completed
  uint64_t* sched_go = bars + kBarSchedGo;    // the current item's K tiles are all issued
  Item* items = reinterpret_cast<Item*>(smem + kOffItem);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc) + 1;

  // V rows past the last key of a tile meet a probability of 0 in the PV
  // products, so they must hold finite values: both V stages start zeroed and
  // the V producer zeroes the rows a ragged tile leaves unloaded.
  {
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < 2 * kTileBytes / 16; i += kThreads)
      reinterpret_cast<uint4*>(smem + kOffV)[i] = z;
  }
  fence_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&item_full[s], 1);
      mbar_init(&item_empty[s], kItemConsumers);
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 4);
      mbar_init(&pv_done[s], 1);
      mbar_init(&o_free[s], 4);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(ml_full, 4);
    mbar_init(ml_empty, 4);
    mbar_init(mma_done, 1);
    mbar_init(sched_go, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // Registers: the launch gives every thread kLaunchRegs; the copy, MMA and
  // scheduler warpgroup hands most of its share to the two softmax
  // warpgroups (the sum stays within the launch's allocation).
  if (warp < kKWarp) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    SoftmaxArgs sa;
    sa.tm_o = p.o_tma ? &p.tm_o : nullptr;
    sa.out = p.out;
    sa.out32 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
    sa.o_part = p.o_part;
    sa.lse_part = p.lse_part;
    sa.err = p.err;
    sa.Hq = p.Hq;
    sa.Hkv = p.Hkv;
    sa.G = p.G;
    sa.TQ = p.TQ;
    sa.scale_log2 = p.scale_log2;
    softmax_role(sa, smem, tmem, warp, lane);
    tc_fence_before();
    cta_sync();  // pairs with the other warpgroup's barrier before the TMEM is freed
    return;
  }
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRoleRegs));
  if (warp == kSchedWarp) {
    // ------------------------------- work scheduler -------------------------------
    // Planned launch: items k = unit * Hkv + kv-head are taken from a shared
    // counter, so a CTA that finishes early takes the next one (the units are
    // listed longest first).  Otherwise the CTA's own pair is its one item.
    if (lane == 0) {
      if (p.units) pdl_wait();  // the planner's unit list and counter are ready
      const int total = p.units ? *p.n_units * p.Hkv : 1;
      int pub = 0, k_own = 0;
      for (;;) {
        Item it;
        it.valid = 0;
        // Take the next item only when this CTA is about to need it (its
        // previous item's K tiles are all issued), so that the items, listed
        // longest first, go to the CTAs that free up first.
        if (pub > 0) {
          const uint64_t tg = global_timer_ns();
          bool okg = true;
          while (!mbar_try_wait(sched_go, (pub - 1) & 1)) {
            __nanosleep(64);
            if (*abort_flag || global_timer_ns() - tg > kWaitLimitNs) {
              if (!*abort_flag) raise_flag(p.err, PA_DEVERR_TIMEOUT);
              *abort_flag = 1;
              okg = false;
              break;
            }
          }
          if (!okg) break;
        }
        const int k = p.units ? atomicAdd(p.counter, 1) : k_own++;
        const bool last = k >= total;
        if (!last) {
          int b, qp, h, jl, jh, sl;
          if (p.units) {
            const int u = k / p.Hkv;
            h = k - u * p.Hkv;
            const int4 ud = p.units[u];
            b = ud.x;
            qp = ud.y;
            jl = ud.z & 0xffff;
            jh = static_cast<int>(static_cast<uint32_t>(ud.z) >> 16);
            sl = ud.w;
          } else {
            b = blockIdx.z;
            h = blockIdx.y;
            qp = blockIdx.x;
            jl = 0;
            jh = 1 << 30;
            sl = -1;
          }
          if (!make_item(p, b, qp, h, jl, jh, sl, it)) continue;
        }
        const int s = pub & 1;
        // the slot frees when every role has taken the item two back: poll
        // slowly, so as not to take issue slots from the softmax warps
        const uint32_t par = ((pub >> 1) & 1) ^ 1;
        const uint64_t tw = global_timer_ns();
        bool okw = true;
        while (!mbar_try_wait(&item_empty[s], par)) {
          __nanosleep(500);
          if (*abort_flag || global_timer_ns() - tw > kWaitLimitNs) {
            if (!*abort_flag) raise_flag(p.err, PA_DEVERR_TIMEOUT);
            *abort_flag = 1;
            okw = false;
            break;
          }
        }
        if (!okw) break;
        items[s] = it;
        mbar_arrive(&item_full[s]);  // release: the item's fields are visible to its waiters
        ++pub;
        if (last) break;
      }
    }
    __syncwarp();
  } else if (warp == kKWarp || warp == kVWarp) {
    // ------------------------------- TMA producers -------------------------------
    // Warp kKWarp copies each item's Q tiles and its K tiles, warp kVWarp its V
    // tiles, each into its own two-stage ring that runs on across items.
    const bool vrole = warp == kVWarp;
    const int box = lane >> 2, half = (lane >> 1) & 1, isv = lane & 1;
    uint64_t* full = vrole ? v_full : k_full;
    uint64_t* empty = vrole ? v_empty : k_empty;
    const CUtensorMap* m16 = vrole ? &p.tm_v16 : &p.tm_k16;
    const CUtensorMap* m1 = vrole ? &p.tm_v1 : &p.tm_k1;
    constexpr int kNoPage = INT_MIN;
    int kc = 0;  // tiles issued into this ring
    int nq_issued = 0;  // items whose Q tiles were issued
    bool ok = true;
    for (int i = 0; ok; ++i) {
      Item it;
      if (!take_item(items, item_full, item_empty, i, abort_flag, p.err, it)) {
        ok = false;
        break;
      }
      if (!it.valid) break;
      const int64_t bt_row = static_cast<int64_t>(it.b) * p.maxp;
      const int x = it.h * 128 + half * 64;
      // Block-table entries of tile t: lane `box` reads the page of its 16-row
      // box, lanes 0-3 the page of a ragged end.
      auto load_pages = [&](int t, int& pg_full, int& pg_rem) {
        const int t0 = (it.j_lo + t) * kBN;
        const int valid = min(kBN, it.kv_len - t0);
        const int nfull = valid / kBoxRows, rem = valid % kBoxRows;
        pg_full = box < nfull ? p.bt[bt_row + ((t0 + box * kBoxRows) >> p.log2P)] : kNoPage;
        pg_rem = rem && lane < 4 ? p.bt[bt_row + ((t0 + nfull * kBoxRows) >> p.log2P)] : kNoPage;
      };
      int pf_next = kNoPage, pr_next = kNoPage;
      load_pages(0, pf_next, pr_next);
      if (!vrole) {
        // the item's Q tiles, once the previous item's last QK has read Q
        int okq = 1;
        if (lane == 0) {
          okq = i == 0 || mbar_wait_bounded(q_empty, (i - 1) & 1, abort_flag, p.err);
          if (okq) {
            ++nq_issued;
            mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(it.nq * p.G * p.TQ * 256));
            for (int g = 0; g < it.nq; ++g) {
              const int z = it.s0 + (2 * it.qp + g) * p.TQ;
              tma_load_3d(smem + kOffQ + g * kTileBytes, &p.tm_q, 0, it.h * p.G, z, q_full);
              tma_load_3d(smem + kOffQ + g * kTileBytes + kHalfBytes, &p.tm_q, 64, it.h * p.G, z, q_full);
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, okq, 0)) {
          ok = false;
          break;
        }
      }
      for (int t = 0; t < it.nt; ++t) {
        const int pf = pf_next, pr = pr_next;
        if (t + 1 < it.nt) load_pages(t + 1, pf_next, pr_next);  // one tile ahead
        const int st = kc & 1;
        const int t0 = (it.j_lo + t) * kBN;
        const int valid = min(kBN, it.kv_len - t0);
        const int nfull = valid / kBoxRows, rem = valid % kBoxRows;
        int y_full = -1, y_rem = -1;
        if (pf != kNoPage) {
          if (pf >= 0 && pf < p.num_pages) y_full = (pf << p.log2P) + ((t0 + box * kBoxRows) & (p.P - 1));
          else raise_flag(p.err, PA_DEVERR_BAD_PAGE);
        }
        if (pr != kNoPage) {
          if (pr >= 0 && pr < p.num_pages) y_rem = (pr << p.log2P) + ((t0 + nfull * kBoxRows) & (p.P - 1));
          else raise_flag(p.err, PA_DEVERR_BAD_PAGE);
        }
        const uint32_t mine = (y_full >= 0 ? kBoxRows * 128 : 0) + (y_rem >= 0 ? rem * 128 : 0);
        uint32_t bytes = (isv != 0) == vrole ? mine : 0;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
        int okw = 1;
        if (lane == 0) okw = mbar_wait_bounded(&empty[st], ((kc >> 1) & 1) ^ 1, abort_flag, p.err);
        if (!__shfl_sync(0xffffffffu, okw, 0)) {
          ok = false;
          break;
        }
        unsigned char* stage = smem + (vrole ? kOffV : kOffK) + st * kTileBytes;
        if (vrole && valid < kBN) {
          // a ragged tile: zero the rows it leaves unloaded (they may hold
          // another request's values), before the copies are counted
          const int chunks = (kBN - valid) * 16;
          for (int c = lane; c < chunks; c += 32) {
            const int r = valid + (c >> 4), ch = c & 15;
            *reinterpret_cast<uint4*>(stage + (ch >> 3) * kHalfBytes + r * 128 + (ch & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
          __syncwarp();
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[st], bytes);
        __syncwarp();
        if ((isv != 0) == vrole) {
          unsigned char* dst = stage + half * kHalfBytes;
          if (y_full >= 0) tma_load_2d(dst + box * kBoxRows * 128, m16, x, y_full, &full[st]);
          if (y_rem >= 0)
            for (int r = 0; r < rem; ++r) tma_load_2d(dst + (nfull * kBoxRows + r) * 128, m1, x, y_rem + r, &full[st]);
        }
        ++kc;
      }
      if (!ok) break;
      if (!vrole) {
        __syncwarp();
        if (lane == 0) mbar_arrive(sched_go);  // the scheduler may take the next item
      }
    }
    if (!ok && lane == 0) {
      // copies may still be landing: wait for them (time only) before the CTA exits
      if (!vrole && nq_issued > 0) drain(q_full, (nq_issued - 1) & 1);
      for (int j = max(0, kc - 2); j < kc; ++j) drain(&full[j & 1], (j >> 1) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------- MMA issuer -------------------------------
    if (lane == 0) {
      // low descriptor halves of the two Q tiles and the K / V stages; an MMA's
      // operand is its tile's plus the address offset >> 4 (the 14-bit address
      // field never carries: shared addresses are < 256 KB)
      const uint32_t dQ0 = desc_lo(smem_u32(smem + kOffQ), 16);
      const uint32_t dQ1 = desc_lo(smem_u32(smem + kOffQ + kTileBytes), 16);
      const uint32_t dK0 = desc_lo(smem_u32(smem + kOffK), 16);
      const uint32_t dK1 = desc_lo(smem_u32(smem + kOffK + kTileBytes), 16);
      const uint32_t dV0 = desc_lo(smem_u32(smem + kOffV), kHalfBytes);
      const uint32_t dV1 = desc_lo(smem_u32(smem + kOffV + kTileBytes), kHalfBytes);
      const uint32_t bar0 = smem_u32(bars);
      int kc = 0;          // K/V tiles consumed before this item (both rings advance alike)
      int pc0 = 0, pc1 = 0;  // PVs issued per group
      int ow0 = 0, ow1 = 0;  // items whose O_g has been written
      bool ok = true;
      for (int i = 0; ok; ++i) {
        Item it;
        if (!take_item_lane(items, item_full, item_empty, i, abort_flag, p.err, it)) break;
        if (!it.valid) break;
        if (!(ok = mbar_wait_bounded(q_full, i & 1, abort_flag, p.err))) break;
        tc_fence_after();
        const int c0 = it.c[0], c1 = it.c[1];
        int qk_left = c0 + c1;  // the item's last QK releases the Q tiles
        // ring stage and phase of the item's tile t
        auto st_of = [&](int t) { return (kc + t) & 1; };
        auto ph_of = [&](int t) { return static_cast<uint32_t>(((kc + t) >> 1) & 1); };
        // barrier i of the table at the top of the kernel
        auto bar = [&](int idx) { return bar0 + 8u * static_cast<uint32_t>(idx); };
        auto wait_k = [&](int t) {
          const bool r = wait_a(bar(kBarKFull + st_of(t)), ph_of(t), abort_flag, p.err);
          tc_fence_after();
          return r;
        };
        auto wait_v = [&](int t) { return wait_a(bar(kBarVFull + st_of(t)), ph_of(t), abort_flag, p.err); };
        auto rel_k = [&](int t) { commit_a(bar(kBarKEmpty + st_of(t))); };
        auto rel_v = [&](int t) { commit_a(bar(kBarVEmpty + st_of(t))); };
        // S_g = Q K_t^T into TMEM columns g * 128
        auto qk = [&](int g, uint32_t dq, int t) {
          issue_qk(tmem + g * 128, dq, st_of(t) ? dK1 : dK0);
          commit_a(bar(kBarSFull + g));
          if (--qk_left == 0) commit_a(bar(kBarQEmpty));
        };
        // O_g (+)= P_g V_t once the group's probabilities are written; the
        // item's first PV overwrites O_g after the previous item's epilogue read it
        auto pv0 = [&](int t, bool first) -> bool {
          if (!wait_a(bar(kBarPFull), pc0 & 1, abort_flag, p.err)) return false;
          if (first) {
            if (ow0 > 0 && !wait_a(bar(kBarOFree), (ow0 - 1) & 1, abort_flag, p.err)) return false;
            ++ow0;
          }
          tc_fence_after();
          issue_pv(tmem + 256, tmem, st_of(t) ? dV1 : dV0, first);
          commit_a(bar(kBarPvDone));
          ++pc0;
          return true;
        };
        auto pv1 = [&](int t, bool first) -> bool {
          if (!wait_a(bar(kBarPFull + 1), pc1 & 1, abort_flag, p.err)) return false;
          if (first) {
            if (ow1 > 0 && !wait_a(bar(kBarOFree + 1), (ow1 - 1) & 1, abort_flag, p.err)) return false;
            ++ow1;
          }
          tc_fence_after();
          issue_pv(tmem + 384, tmem + 128, st_of(t) ? dV1 : dV0, first);
          commit_a(bar(kBarPvDone + 1));
          ++pc1;
          return true;
        };
        // Order per step: PV_0, QK_0 of the next step, PV_1, QK_1 of the next
        // step -- each softmax group has a PV and a QK of the other group to
        // hide in, and QK_g overwrites S_g only after PV_g read P_g (one
        // thread's MMAs execute in issue order).
        if (!it.split) {
          // pair mode: tile s feeds q-tile 0 (its first c0 tiles) and q-tile 1 (all c1 = nt)
          if ((ok = wait_k(0))) {
            if (c0 > 0) qk(0, dQ0, 0);
            qk(1, dQ1, 0);
            rel_k(0);
          }
          for (int s = 0; s < c1 && ok; ++s) {
            const bool more = s + 1 < c1;
            if (!(ok = wait_v(s))) break;
            if (s < c0 && !(ok = pv0(s, s == 0))) break;
            if (more) {
              if (!(ok = wait_k(s + 1))) break;
              if (s + 1 < c0) qk(0, dQ0, s + 1);
            }
            if (!(ok = pv1(s, s == 0))) break;
            rel_v(s);
            if (more) {
              qk(1, dQ1, s + 1);
              rel_k(s + 1);
            }
          }
        } else {
          // split mode: q-tile 0 only; group 0 takes the item's tiles 0, 2, 4, ...,
          // group 1 tiles 1, 3, 5, ...
          if ((ok = wait_k(0))) {
            qk(0, dQ0, 0);
            rel_k(0);
          }
          if (ok && c1 > 0 && (ok = wait_k(1))) {
            qk(1, dQ0, 1);
            rel_k(1);
          }
          for (int s = 0; s < c0 && ok; ++s) {
            const int ta = 2 * s, tb = 2 * s + 1;
            if (!(ok = wait_v(ta))) break;
            if (!(ok = pv0(ta, s == 0))) break;
            rel_v(ta);
            if (s + 1 < c0) {
              if (!(ok = wait_k(ta + 2))) break;
              qk(0, dQ0, ta + 2);
              rel_k(ta + 2);
            }
            if (s < c1) {
              if (!(ok = wait_v(tb))) break;
              if (!(ok = pv1(tb, s == 0))) break;
              rel_v(tb);
              if (s + 1 < c1) {
                if (!(ok = wait_k(tb + 2))) break;
                qk(1, dQ0, tb + 2);
                rel_k(tb + 2);
              }
            }
          }
        }
        kc += it.nt;
      }
      // every MMA has completed before the tensor memory is freed
      mma_commit(mma_done);
      drain(mma_done, 0);
    }
    __syncwarp();
  }

  tc_fence_before();
  cta_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------
// planner: q-tile pairs -> units (split long key ranges, longest first)
// ---------------------------------------------------------------------------
// Without a plan each CTA of the attention kernel runs one q-tile pair in
// grid order, so a batch whose pairs fill less than a wave, or whose last
// wave holds its longest pairs, waits on its longest pair.  The planner (one
// CTA, on the device, so the launch needs no host copy of the lengths and can
// be captured in a graph) lists the pairs with their key-tile counts nt,
// chooses a part size tau, cuts every pair with nt > tau into ceil(nt / tau)
// near-equal key ranges, and writes the units sorted by cost, longest first.
// The persistent attention kernel takes (unit, kv-head) items from a shared
// counter in that order whenever a CTA frees up: longest-processing-time-
// first list scheduling.
//
// tau is chosen among 32 candidates by the makespan of their items dealt to
// the SMs longest first in snake order, in units of one key tile of a q-tile
// pair (unit_cost).  Splitting is considered only while the pairs fill at
// most four waves; beyond that the ordering alone keeps the tail short.
constexpr int kPlanThreads = 1024;
constexpr int kPlanBuckets = 2048;   // unit lengths >= 2047 tiles share the last bucket
constexpr int kPlanSmemPairs = 2048; // pairs kept in shared memory (the rest are re-read from the workspace)
constexpr int kPlanCandidates = 32;  // one per warp
constexpr int kScoreBuckets = 64;    // cost buckets per candidate when scoring it
constexpr int kSplitWaves = 4;
constexpr int kMaxSlots = 65535;     // slot counts are scanned in 16 bits

struct PlanParams {
  const int32_t* cu;
  const int32_t* ctx;
  unsigned int* err;
  int4* pairs;   // [pair_cap] {request, pair, nt, q-tiles with rows}
  int4* units;   // [pair_cap + slot_cap]
  int4* splits;  // [split_cap] {request, pair, first slot, parts}
  int32_t* hdr;  // {units, split pairs, tau, pairs, work counter}
  int64_t num_tokens;
  int64_t kv_block_tokens;  // context tokens whose K and V fill a third of L2 (0: order by cost alone)
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

// floor(a / b) for 0 <= a < 2^24 and b >= 1, given inv_b ~ 1 / b: the float
// quotient is within one of the true one and is corrected.
PA_DEVINL int div_near(int a, int b, float inv_b) {
  int d = __float2int_rz(static_cast<float>(a) * inv_b);
  if (d * b > a) --d;
  else if ((d + 1) * b <= a) ++d;
  return d;
}

// Dynamic shared memory of the planner: per candidate, item counts and cost
// sums of its cost buckets and a difference array over the SMs.
inline size_t plan_dyn_bytes(int n_sm) {
  return static_cast<size_t>(2 * kPlanCandidates * kScoreBuckets + kPlanCandidates * (n_sm + 1)) * sizeof(int);
}

// Estimated time of a unit of `len` key tiles in steps of the attention
// kernel (one step: a 128-key tile of a q-tile pair): a single q-tile's key
// tiles alternate between the two softmax groups and take about 0.7 step
// each (two new K/V tiles per step); the hand-over between items costs about
// three steps, a part two more (its fp32 partial result, its share of the
// merge).
PA_DEVINL int unit_cost(int len, int nq, int part) {
  return (nq == 2 ? len : (7 * len + 9) / 10) + 3 + 2 * part;
}
PA_DEVINL int cost_bucket(int len, int nq, int part) { return min(unit_cost(len, nq, part), kPlanBuckets - 1); }

// Order of the units.  When the pairs fill more than kSplitWaves waves (no
// split) and their requests' K and V do not fit in L2 together, the requests
// are taken in blocks whose K and V fill about a third of L2, longest first
// within a block: longest first over the whole batch would run every
// request's pairs at once and read their K / V tiles back from DRAM several
// times.  Buckets are handed out from the highest index down.
constexpr int kMaxKvBlocks = 8;
constexpr int kBlockBuckets = kPlanBuckets / kMaxKvBlocks;
PA_DEVINL int order_bucket(int len, int nq, int part, int blk, bool blocked) {
  return blocked ? (kMaxKvBlocks - 1 - blk) * kBlockBuckets + min(unit_cost(len, nq, part), kBlockBuckets - 1)
                 : cost_bucket(len, nq, part);
}

// A pair of nt key tiles cut into `parts` ranges: the first nt % parts ranges
// hold one tile more than the others (lengths base + 1 and base).
template <bool kScore>
__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(const PlanParams q) {
  extern __shared__ int plan_dyn[];  // candidate scoring: see plan_dyn_bytes
  __shared__ unsigned long long sh_scan[32];
  __shared__ int cursor[kPlanBuckets];
  __shared__ int4 sh_pairs[kPlanSmemPairs];
  __shared__ float cand_est[kPlanCandidates];
  __shared__ int cand_tau[kPlanCandidates];
  __shared__ int sh_max_nt;
  pdl_trigger();  // the attention kernel may start launching; it waits for this plan
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) sh_max_nt = 0;
  for (int i = tid; i < kPlanBuckets; i += kPlanThreads) cursor[i] = 0;

  // 1. the q-tile pairs of every request and their key-tile counts; a pair's
  //    .w holds its q-tiles with rows (bits 0-7) and its request's K/V block
  //    (bits 8-15: context tokens of the requests before it / kv_block_tokens)
  unsigned long long carry = 0, carry_l = 0;
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
    unsigned long long tot, tot_l;
    const unsigned long long off = carry + block_scan_excl<unsigned long long>(np, sh_scan, &tot);
    const unsigned long long l_before =
        carry_l + block_scan_excl<unsigned long long>(np > 0 ? static_cast<unsigned long long>(L) : 0ull, sh_scan,
                                                      &tot_l);
    const int blk = q.kv_block_tokens > 0
                        ? static_cast<int>(min(l_before / static_cast<unsigned long long>(q.kv_block_tokens),
                                               static_cast<unsigned long long>(kMaxKvBlocks - 1)))
                        : 0;
    for (int k = 0; k < np; ++k) {
      const int nt = (L - n + min((2 * k + 2) * q.TQ, n) + kBN - 1) / kBN;
      const int4 pr = make_int4(b, k, nt, ((2 * k + 1) * q.TQ < n ? 2 : 1) | (blk << 8));
      if (off + k < static_cast<unsigned long long>(q.pair_cap)) q.pairs[off + k] = pr;
      if (off + k < kPlanSmemPairs) sh_pairs[off + k] = pr;
      max_nt = max(max_nt, nt);
    }
    carry += tot;
    carry_l += tot_l;
  }
  if (max_nt > 0) atomicMax(&sh_max_nt, max_nt);
  if (carry > static_cast<unsigned long long>(q.pair_cap)) {  // lengths disagree with the workspace's sizes
    if (tid == 0) {
      raise_flag(q.err, PA_DEVERR_BAD_LENGTH);
      q.hdr[0] = q.hdr[1] = q.hdr[2] = q.hdr[3] = q.hdr[4] = 0;
    }
    pdl_wait();  // the KV write beside which it may run has completed
    return;
  }
  const int n_pairs = static_cast<int>(carry);
  const bool blocked = q.kv_block_tokens > 0 && carry_l > static_cast<unsigned long long>(q.kv_block_tokens) &&
                       static_cast<int64_t>(n_pairs) * q.Hkv > static_cast<int64_t>(kSplitWaves) * q.n_sm;
  cta_sync();
  max_nt = sh_max_nt;
  auto pair_at = [&](int i) -> int4 { return i < kPlanSmemPairs ? sh_pairs[i] : q.pairs[i]; };

  // 2. the part size: one candidate per warp -- the 16 sizes from max_nt (no
  //    split) down, each of which splits exactly the pairs longer than it, then
  //    16 geometric steps down to 2 -- scored by the makespan of its items
  //    dealt to the SMs longest first in snake order (SM 0, 1, .., n-1, then
  //    n-1, .., 0, ...), which is close to the list schedule that the
  //    persistent kernel's work counter produces from the longest-first list.
  int tau = max(max_nt, 1);
  if (kScore && n_pairs > 0 && max_nt > 2 && q.slot_cap > 1 &&
      static_cast<int64_t>(n_pairs) * q.Hkv <= static_cast<int64_t>(kSplitWaves) * q.n_sm) {
    const int c = warp;
    int t_c;
    if (c < kPlanCandidates / 2) {
      t_c = max(2, max_nt - c);
    } else {
      const int t0 = max(2, max_nt - kPlanCandidates / 2);
      const float f = static_cast<float>(c - kPlanCandidates / 2 + 1) / (kPlanCandidates / 2);
      t_c = max(2, static_cast<int>(ceilf(t0 * exp2f(-log2f(0.5f * t0) * f))));
    }
    // this candidate's item costs, in 64 buckets of `w` cost units
    int* cnt = plan_dyn + c * kScoreBuckets;
    float* sum = reinterpret_cast<float*>(plan_dyn + kPlanCandidates * kScoreBuckets) + c * kScoreBuckets;
    float* diff = reinterpret_cast<float*>(plan_dyn + 2 * kPlanCandidates * kScoreBuckets) + c * (q.n_sm + 1);
    const int w = (unit_cost(t_c, 2, 1) + kScoreBuckets) / kScoreBuckets;
    const float inv_t = 1.f / t_c, inv_w = 1.f / w, inv_m = 1.f / q.n_sm;
    for (int k = lane; k < kScoreBuckets; k += 32) {
      cnt[k] = 0;
      sum[k] = 0.f;
    }
    for (int k = lane; k <= q.n_sm; k += 32) diff[k] = 0.f;
    __syncwarp();
    int slots = 0;
    for (int i = lane; i < n_pairs; i += 32) {
      const int4 pr = pair_at(i);
      const int nt = pr.z, nq = pr.w & 0xff;
      const int parts = div_near(nt + t_c - 1, t_c, inv_t);
      const int split = parts > 1;
      const int base = div_near(nt, parts, 1.f / parts), rem = nt - base * parts;
      slots += split ? parts : 0;
      if (rem) {
        const int cu = unit_cost(base + 1, nq, split);
        const int bk = min(div_near(cu, w, inv_w), kScoreBuckets - 1);
        atomicAdd(&cnt[bk], rem * q.Hkv);
        atomicAdd(&sum[bk], static_cast<float>(rem * q.Hkv) * cu);
      }
      if (parts > rem) {
        const int cu = unit_cost(base, nq, split);
        const int bk = min(div_near(cu, w, inv_w), kScoreBuckets - 1);
        atomicAdd(&cnt[bk], (parts - rem) * q.Hkv);
        atomicAdd(&sum[bk], static_cast<float>((parts - rem) * q.Hkv) * cu);
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) slots += __shfl_xor_sync(0xffffffffu, slots, o);
    __syncwarp();
    // deal: lane k owns buckets 63 - k and 31 - k (descending cost order);
    // the items of a bucket take the next positions of the deal, each worth
    // the bucket's mean cost, as a difference array over the SMs plus whole
    // rounds that reach every SM
    const int M = q.n_sm;
    int n_a = cnt[kScoreBuckets - 1 - lane], n_b = cnt[kScoreBuckets / 2 - 1 - lane];
    int pos_a = n_a, pos_b = n_b;  // inclusive scans, then exclusive
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ya = __shfl_up_sync(0xffffffffu, pos_a, o), yb = __shfl_up_sync(0xffffffffu, pos_b, o);
      if (lane >= o) {
        pos_a += ya;
        pos_b += yb;
      }
    }
    const int total_a = __shfl_sync(0xffffffffu, pos_a, 31);
    pos_a -= n_a;
    pos_b += total_a - n_b;
    float rounds = 0.f;
    auto deal = [&](int p0, int n, float cost) {
      const int p1 = p0 + n;
      while (p0 < p1) {
        const int layer = div_near(p0, M, inv_m), s0 = p0 - layer * M;
        const int e = min(p1 - layer * M, M);  // end of this layer's part
        if (s0 == 0 && e == M) {
          const int full = div_near(p1 - p0, M, inv_m);  // whole rounds
          rounds += cost * full;
          p0 += full * M;
          continue;
        }
        const int lo = (layer & 1) ? M - e : s0, hi = (layer & 1) ? M - s0 : e;
        atomicAdd(&diff[lo], cost);
        atomicAdd(&diff[hi], -cost);
        p0 = layer * M + e;
      }
    };
    if (n_a > 0) deal(pos_a, n_a, sum[kScoreBuckets - 1 - lane] / n_a);
    if (n_b > 0) deal(pos_b, n_b, sum[kScoreBuckets / 2 - 1 - lane] / n_b);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) rounds += __shfl_xor_sync(0xffffffffu, rounds, o);
    __syncwarp();
    // loads: prefix sums of the difference array, contiguous runs per lane
    const int per = (M + 31) / 32, m0 = min(M, lane * per), m1 = min(M, m0 + per);
    float run = 0.f, best = 0.f;
    for (int m = m0; m < m1; ++m) run += diff[m];
    float pre = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, pre, o);
      if (lane >= o) pre += y;
    }
    run = pre - run;  // load before this lane's first SM
    for (int m = m0; m < m1; ++m) {
      run += diff[m];
      best = fmaxf(best, run);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, o));
    if (lane == 0) {
      cand_est[c] = slots > q.slot_cap ? INFINITY : best + rounds;
      cand_tau[c] = t_c;
    }
    cta_sync();
    // every warp takes the arg-min; ties go to the lower index (the larger
    // part size); candidate 0 (no split) is always finite
    float e = cand_est[lane];
    int cc = lane;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float e2 = __shfl_xor_sync(0xffffffffu, e, o);
      const int c2 = __shfl_xor_sync(0xffffffffu, cc, o);
      if (e2 < e || (e2 == e && c2 < cc)) {
        e = e2;
        cc = c2;
      }
    }
    tau = e < INFINITY ? cand_tau[cc] : max_nt;
  }

  // 3. histogram of unit costs, then bucket cursors in descending cost order
  for (int i = tid; i < n_pairs; i += kPlanThreads) {
    const int4 pr = pair_at(i);
    const int nt = pr.z, nq = pr.w & 0xff, blk = pr.w >> 8;
    const int parts = parts_of(nt, tau), base = nt / parts, rem = nt - base * parts, split = parts > 1;
    if (rem) atomicAdd(&cursor[order_bucket(base + 1, nq, split, blk, blocked)], rem);
    if (parts > rem) atomicAdd(&cursor[order_bucket(base, nq, split, blk, blocked)], parts - rem);
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
      const int nq = pr.w & 0xff, blk = pr.w >> 8;
      const int p_hi = rem ? atomicAdd(&cursor[order_bucket(base + 1, nq, split, blk, blocked)], rem) : 0;
      const int p_lo =
          parts > rem ? atomicAdd(&cursor[order_bucket(base, nq, split, blk, blocked)], parts - rem) : 0;
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
    q.hdr[4] = 0;  // the attention kernel's work counter
  }
  pdl_wait();  // the KV write beside which it may run has completed
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
    // output rows by TMA when a softmax warp's 32 rows are whole tokens
    if ((G & (G - 1)) == 0) {
      const cuuint32_t obox[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(32 / G)};
      if (!encode(fn, &p.tm_o, a.out, 3, dims, strides, obox)) return cudaErrorInvalidValue;
      p.o_tma = 1;
    }
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
      // The warpgroups' register rebalance assumes the launch allocation; a
      // build with another register count would make the softmax warpgroups
      // wait for registers that are never released, so it is not launched.
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, prefill_tc_kernel);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidKernelImage;
      e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess) return e;
      int n_sm = 0;
      if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
      e = cudaFuncSetAttribute(prefill_plan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(plan_dyn_bytes(n_sm)));
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
  {
    // context tokens whose K and V (all kv-heads) fill a third of L2
    DeviceInfo di;
    if ((e = current_device_info(&di)) != cudaSuccess) return e;
    const int64_t kv_per_token = static_cast<int64_t>(d.num_kv_heads) * 128 * 2 * 2;
    q.kv_block_tokens = di.l2_bytes > 0 ? std::max<int64_t>(1, di.l2_bytes / 3 / kv_per_token) : 0;
  }
  q.max_seqlen_q = a.max_seqlen_q;
  q.cap_ctx = static_cast<int32_t>(std::min<int64_t>(a.max_context_len, int64_t(a.max_pages) << p.log2P));
  q.pair_cap = pl.pair_cap;
  q.slot_cap = pl.run_slot_cap;
  q.split_cap = pl.run_split_cap;
  // part sizes are scored only when the call may split (when its tokens
  // alone make pairs that fill more than kSplitWaves waves it may not)
  // The planner reads only the varlen metadata.  Behind the same call's KV
  // write (which writes none of it) it is launched to run beside that kernel;
  // it waits for it before it exits, so the attention kernel's wait on the
  // planner is a wait on both.  Otherwise it starts after the previous kernel.
  {
    void* args[] = {&q};
    const void* fn = q.slot_cap > 1 ? reinterpret_cast<const void*>(prefill_plan_kernel<true>)
                                    : reinterpret_cast<const void*>(prefill_plan_kernel<false>);
    const size_t dyn = q.slot_cap > 1 ? plan_dyn_bytes(pl.n_sm) : 0;
    if (a.planner_beside_write)
      e = launch_after_previous(fn, dim3(1), dim3(kPlanThreads), dyn, s, args);
    else
      e = cudaLaunchKernel(fn, dim3(1), dim3(kPlanThreads), args, dyn, s);
    if (e != cudaSuccess) return e;
  }

  p.units = q.units;
  p.n_units = q.hdr;
  p.counter = q.hdr + 4;
  p.lse_part = reinterpret_cast<float*>(ws + pl.off_lse);
  p.o_part = reinterpret_cast<float*>(ws + pl.off_o);
  {
    // persistent: one CTA per SM (at most one per possible item), each taking
    // items until the list is exhausted
    const int64_t items = static_cast<int64_t>(pl.pair_cap + pl.run_slot_cap) * d.num_kv_heads;
    const unsigned ctas = static_cast<unsigned>(std::min<int64_t>(pl.n_sm, items));
    void* args[] = {&p};
    e = launch_after_previous(reinterpret_cast<const void*>(prefill_tc_kernel), dim3(ctas), dim3(kThreads),
                              kSmemBytes, s, args);
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
