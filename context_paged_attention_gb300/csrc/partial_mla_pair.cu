// cp_paged_attn_partial, MLA path: one work item per two-CTA cluster, the two
// CTAs split by role, on the tcgen05 tensor cores.
//
// MLA's one latent KV head is striped like a GQA head (mstar PR #1124
// "Context / Sequence Parallel 1/5", description: MLA's one latent head
// included; copy_slots indexes the token axis): partner p's stripe slot k is
// logical position k * P + p at physical slot k % (page_size / P) of page
// k / (page_size / P).  All 128 query heads of a token share the latent
// rows, so a partner's partial is a dense contraction with M = 128 heads:
//   S = Q K^T   (K = the 576 latent + rope values of each key row)
//   O += P V    (V = the first 512 values of the same rows)
//
// Why two CTAs: O alone (128 x 512 fp32) fills all 512 columns of an SM's
// tensor memory, so one CTA can neither keep Q there nor double-buffer S.
// The cluster therefore splits the work by role, with the same key tiles:
//   * CTA 0 (scores) holds Q in tensor memory as the A operand of S (columns
//     128..415, two bf16 a column) and two 64-column S buffers (0 and 64).
//     Warp 5 streams 64-key tiles of whole latent rows (9 column blocks of
//     64 values, 128-byte swizzle) by TMA into a ring of 24 KB units (3
//     column blocks each); warp 4 issues a tile's 36 S MMAs (N = 64 keys, A
//     from tensor memory, so only K is read from shared memory) a unit at a
//     time as the units land and the S buffer is free; warps 0-3 (thread =
//     head = TMEM lane) read S, run the online softmax (running max raised
//     only when it grows by more than 8 in log2 units, so a rescale is rare
//     and every probability stays <= 2^8), write their rows of P as bf16
//     into a per-warp staging slot and send the slot to CTA 1 with one bulk
//     copy, the row's rescale factor with an asynchronous store, both counted
//     in bytes on CTA 1's barrier.
//   * CTA 1 (values) holds O in all 512 columns.  Warp 5 streams the value
//     part of the same tiles (8 column blocks) into a 2-tile ring, each tile
//     once CTA 0 reports that its rows landed there (so CTA 1's copies find
//     them in L2 instead of racing CTA 0's to HBM); warp 4 waits for each
//     value tile and issues P V (two N = 256 MMAs per 16 keys) and, through a
//     multicast commit, tells CTA 0 when a P buffer may be overwritten; warps
//     0-3 rescale their O row when CTA 0 raised the max, zero the value rows
//     of keys outside the stripe (waiting for that tile only then), and at
//     the end of an item normalise O and write it out.  Those warps can run
//     up to three tiles ahead of the MMAs, so their "O ready" and "P V done"
//     barriers form a ring of four tiles (a parity wait stays unambiguous).
// O is normalised by the sum of the bf16-rounded probabilities (an exact
// convex combination of the values); the LSE keeps the fp32 sum.
//
// Work: every (token, partner) stripe is an item; the grid is persistent
// (one cluster per two SMs).  Each CTA plans the same way: the stripes are
// ranked longest first, stripes longer than max(total / clusters, 16 tiles)
// are cut into near-equal pieces, and item i goes to cluster i mod C in a
// snake order (C-1 .. 0 on odd rounds), which balances about as well as a
// greedy longest-first queue without any shared counter.  Pieces of a cut
// stripe write normalised partials to workspace slots; the last to finish
// (a ticket) merges them.  Too many stripes to rank in shared memory: items
// are whole stripes in dispatch order.
//
// Fused calls over pages of 64 slots (P * page_size / P = 64) take another
// grouping.  The P partners hold the 64 slots of a logical page as P runs of
// page_size / P rows at the same page id of their pools, so one 4-D TMA box
// -- 64 values x page_size / P rows x P partners x the unit's column blocks
// -- brings a unit of the whole logical page into a 64-key tile (row r =
// partner r / (page_size / P), slot r % (page_size / P); the placement,
// interleave included, says which position each row holds).  An item is
// then a token, its tiles are its logical pages, and the online softmax runs
// over every partner's keys at once: the exact merge of the partner partials
// happens tile by tile inside it, and the kernel writes the token's final
// output.  With page runs of 16 rows this needs a quarter of the TMA boxes
// of the per-partner tiles, and the copy engines, not the boxes, set the
// pace.  The clusters split the sequence of all tiles into contiguous
// ranges of equal cost, a token start counted as kItemCostTiles tiles; a
// token that straddles a boundary is cut, its pieces go to workspace slots,
// and a follow-up kernel (mla_merge_pieces_kernel) merges them with the
// optional extra partial.
//
// Every wait is bounded; one that runs out raises the abort flag of both
// CTAs, which ends their other waits, and the call reports
// CPATTN_DEV_TC_TIMEOUT (that item's output is not written).
#include <cuda.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "split_combine.cuh"
#include "tc05.cuh"

namespace cpattn {

namespace {

constexpr int kHeads = 128;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kKB = kDqk / 64;       // 9 column blocks of a latent row
constexpr int kVB = kDv / 64;        // 8 column blocks of its value part
constexpr int kTile = 64;            // keys per tile
constexpr int kBlk = kTile * 128;    // one column block of a tile (8 KB)
constexpr int kVStage = kVB * kBlk;  // 64 KB
constexpr int kUBlk = 3;             // CTA 0: column blocks of a ring unit (24 KB, one TMA box)
constexpr int kUnitsK = kKB / kUBlk;  // units of a tile
constexpr int kKUnits = 8;            // CTA 0: ring of units (2.7 tiles)
constexpr uint32_t kKUnit = kUBlk * kBlk;
static_assert(kKB % kUBlk == 0, "whole units a tile");
constexpr int kVStages = 2;           // CTA 1: tiles of value rows in flight
constexpr int kVUB = kVB;             // CTA 1: column blocks of a value unit (a whole tile's, 64 KB:
                                      // measured faster than two 32 KB halves with their own barriers)
constexpr int kVUnits = kVB / kVUB;   // value units of a tile
constexpr int kVRing = kVStages * kVUnits;
constexpr uint32_t kVUnit = kVUB * kBlk;
static_assert(kVB % kVUB == 0 && kVUB % 4 == 0, "whole units a tile, N = 256 a unit");
constexpr int kLandRing = 16;        // CTA 1's "K tile landed on CTA 0" barriers
constexpr int kPBuf = kHeads * 128;  // P of one tile: 128 rows x 64 bf16
constexpr int kPBufs = 3;            // CTA 1: P buffers (the softmax runs up to 3 tiles ahead of P V)
// CTA 1: barriers a tile for "O ready for the tile's P V" and "P V done".  The
// epilogue warps wait for P V only now and then (a rescale, an item's end),
// and may run up to kPBufs tiles ahead of the MMAs (their one per-tile wait
// is for P, which needs the P V kPBufs tiles back done), so a parity wait is
// unambiguous only with a ring of more than kPBufs barriers.
constexpr int kTileRing = 4;
static_assert(kTileRing > kPBufs, "parity waits on the tile ring");
constexpr int kThreads = 192;
constexpr int kWMma = 4;
constexpr int kWLoad = 5;
constexpr int kMinChunkTiles = 16;   // cut pieces hold at least 1024 keys
constexpr int kItemCostTiles = 16;   // grouped plans: what starting a token costs a cluster, in tiles
constexpr int kSortMax = 512;        // stripes ranked in shared memory
constexpr int kItemsBytes = 4096;    // per-cluster item list (stripes), or the token tables (grouped)
constexpr int kGroupMaxTokens = kItemsBytes / 8 - 1;  // grouped plans: pre[T + 1] and sbase[T] ints
static_assert(kGroupMaxTokens == kMlaGroupMaxTokens, "grouped token limit shared with the planner");
constexpr uint32_t kQCol = 128;      // CTA 0: S buffers at columns 0 and 64, Q at 128..415
constexpr int kMergeUnroll = 8;

// shared-memory map (offsets from a 1024-byte aligned base), the same in both CTAs
constexpr uint32_t OFF_P = kVStages * kVStage;                   // CTA 1: P buffers [kPBufs]
constexpr uint32_t OFF_ALPHA = OFF_P + kPBufs * kPBuf;           // CTA 1: [kPBufs][128] rescale factors
constexpr uint32_t OFF_FIN = OFF_ALPHA + kPBufs * kHeads * 4;    // CTA 1: [128] (1 / sum, LSE)
constexpr uint32_t OFF_SCR = (OFF_FIN + kHeads * 8 + 1023u) & ~1023u;  // CTA 1: output staging, merge scratch
constexpr uint32_t OFF_PSTAGE = kKUnits * kKUnit;               // CTA 0: P rows of the 4 softmax warps
constexpr uint32_t kPSlot = 32 * 128;                            //   (4 KB each) on their way to CTA 1
constexpr uint32_t kAreaK = OFF_PSTAGE + 4 * kPSlot;              // CTA 0's part of the map
constexpr uint32_t kScrMin = 2 * kHeads * 128;                    // CTA 1: store_rows' two staging chunks
constexpr uint32_t kAreaV = OFF_SCR + kScrMin;                     // CTA 1's part, with the least scratch
constexpr uint32_t kStageArea = ((kAreaK > kAreaV ? kAreaK : kAreaV) + 1023u) & ~1023u;
constexpr int kScrFloats = static_cast<int>((kStageArea - OFF_SCR) / 4);
// barriers (arrival counts in brackets)
enum : int {
  B_KFULL = 0,                      // x8 CTA 0 [1 + bytes (TMA) | 32 copy lanes]: unit landed
  B_KEMPTY = B_KFULL + kKUnits,     // x8 CTA 0 [commit]: the S MMAs that read the unit done
  B_SFULL = B_KEMPTY + kKUnits,     // x2 CTA 0 [commit]: S written
  B_SEMPTY = B_SFULL + 2,           // x2 CTA 0 [4 softmax warps]: S read
  B_QFULL = B_SEMPTY + 2,           // CTA 0 [4 softmax warps]: the item's Q in tensor memory
  B_QEMPTY = B_QFULL + 1,           // CTA 0 [commit]: the item's last S done
  B_PEMPTY = B_QEMPTY + 1,          // x3 CTA 0 [multicast commit from CTA 1]: P V of the buffer done
  B_FINEMPTY = B_PEMPTY + kPBufs,   // CTA 0 [4 remote arrivals]: CTA 1 read the item's row scales
  B_VFULL = B_FINEMPTY + 1,         // x4 CTA 1 [1 + bytes | 32]: value unit landed
  B_VEMPTY = B_VFULL + kVRing,      // x4 CTA 1 [commit]: the P V MMAs that read the unit done
  B_PFULL = B_VEMPTY + kVRing,      // x3 CTA 1 [1 + bytes of CTA 0's copies]: P and rescale factors landed
  B_READY = B_PFULL + kPBufs,       // x4 CTA 1 [4 epilogue warps]: O rescaled, V rows fixed
  B_PVDONE = B_READY + kTileRing,   // x4 CTA 1 [commit]: P V done
  B_FINFULL = B_PVDONE + kTileRing,         // CTA 1 [1 + bytes of CTA 0's asynchronous stores]: the item's row scales and LSEs
  B_DRAIN = B_FINFULL + 1,          // both [commit]: the MMA thread's last MMAs done
  B_EPSYNC = B_DRAIN + 1,           // CTA 1 [128 epilogue threads]: their group barrier (merges)
  B_KLAND = B_EPSYNC + 1,           // x16 CTA 1 [1 remote arrival]: the tile's rows reached CTA 0 (so they sit in L2)
  B_MERGE = B_KLAND + kLandRing,    // x2 CTA 1 [1 + bytes]: a batch of partial rows landed (merges of cut items)
  kBars = B_MERGE + 2
};
constexpr uint32_t OFF_BAR = kStageArea;
constexpr uint32_t OFF_MISC = OFF_BAR + kBars * 8;  // [0] TMEM base, [1] abort, [2] items (-1: on the fly) / first token, [3] tiles
struct MlaItem {
  int t, p, b;           // token, partner, row (-1: no row)
  int k_begin, k_end;    // stripe slots of this item
  int slot;              // workspace slot of a cut stripe's piece, or -1
  int slot_base, npieces;
};
constexpr int kMaxOwn = kItemsBytes / static_cast<int>(sizeof(MlaItem));  // items one cluster keeps in its list
constexpr uint32_t OFF_ITEMS = OFF_MISC + 32;
constexpr size_t kSmemBytes = 1024 + OFF_ITEMS + kItemsBytes;
static_assert(OFF_SCR + kScrMin <= kStageArea && kScrFloats * 4 >= static_cast<int>(kScrMin),
              "CTA 1 map exceeds the stage area");
static_assert(kSmemBytes + 64 <= 232448, "shared memory per CTA");

// The epilogue warps of CTA 1 (threads 0..127) as a merge group.  Their
// barrier is an mbarrier with a bounded wait rather than bar.sync, so that a
// warp that gave up after a timeout cannot leave the others waiting forever.
struct EpGroup {
  __device__ static int tid() { return threadIdx.x; }
  __device__ static int size() { return kHeads; }
  __device__ static void sync() {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t mb = tc05::smem_addr(reinterpret_cast<uint8_t*>(
                            (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023))) +
                        OFF_BAR + B_EPSYNC * 8;
    uint64_t state;
    asm volatile("mbarrier.arrive.shared::cta.b64 %0, [%1];\n" : "=l"(state) : "r"(mb) : "memory");
    for (uint32_t it = 0; it < (1u << 22); ++it) {
      uint32_t done;
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(mb), "l"(state)
          : "memory");
      if (done) return;
    }
  }
};

__device__ __forceinline__ void arrive_local(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void cp_arrive_noinc(uint32_t mbar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp16_zero(uint32_t dst, const void* any_gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, 0;\n" ::"r"(dst), "l"(any_gmem) : "memory");
}

// Bounded wait for the phase of parity `parity`; gives up when the abort
// flag is raised.  kCluster: the phase is completed by another CTA's release
// (acquire at cluster scope).
template <bool kCluster>
__device__ __forceinline__ bool pwait(uint32_t mbar, uint32_t parity, const volatile int* abort_flag) {
  for (uint32_t it = 0; it < (1u << 22); ++it) {
    uint32_t done;
    if constexpr (kCluster) {
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
          " selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(mbar), "r"(parity)
          : "memory");
    } else {
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(mbar), "r"(parity)
          : "memory");
    }
    if (done) return true;
    if ((it & 63u) == 63u && *abort_flag) return false;
  }
  return false;
}

// A whole warp waits: lane 0 polls (one shared-memory probe at a time, not
// 32), the verdict goes to every lane, and __syncwarp orders the other lanes'
// later accesses after lane 0's acquire.  One verdict for the warp, so no lane
// leaves a loop that its warp-mates stay in.
template <bool kCluster>
__device__ __forceinline__ bool wwait(uint32_t mbar, uint32_t parity, const volatile int* abort_flag) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = pwait<kCluster>(mbar, parity, abort_flag) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Token, partner, row and stripe length of stripe s = token * P + partner.
struct StripeGeo {
  int t, p, b, n;
};
__device__ __forceinline__ StripeGeo stripe_geo(const PartialArgs& a, int t, int p, bool may_report) {
  StripeGeo g{t, p, -1, 0};
  if (t < 0) return g;
  if (a.qo_indptr != nullptr) {
    if (t < __ldg(a.qo_indptr + a.num_rows)) g.b = find_row(a.qo_indptr, a.num_rows, t);
  } else if (t < a.num_rows) {
    g.b = t;
  }
  if (g.b >= 0) {
    int L = __ldg(a.kv_len + g.b);
    if (L > a.max_kv_len) {
      if (may_report && p == 0) report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
      L = a.max_kv_len;
    }
    g.n = stripe_len(max(L, 0), p, a.P, a.interleave);
  }
  return g;
}

// The plan (all threads of the CTA; both CTAs of a cluster compute the same
// one).  `tmp` is shared memory free until the first tile lands.
__device__ void mla_plan(const PartialArgs& a, int C, int c, int* tmp, int* misc, MlaItem* items) {
  const int S = a.num_tokens * a.P;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* tiles = tmp;            // [S] tiles of each stripe
  int* ns = tiles + S;         // [S] stripe lengths
  int* order = ns + S;         // [S] stripes, longest first
  int* pre = order + S;        // [S + 1] first item of each ranked stripe
  int* sbase = pre + S + 1;    // [S] first workspace slot of each ranked stripe (cut stripes only)
  int part = 0;
  for (int s = tid; s < S; s += blockDim.x) {
    const StripeGeo g = stripe_geo(a, s / a.P, s % a.P, true);
    ns[s] = g.n;
    tiles[s] = (g.n + kTile - 1) / kTile;
    part += tiles[s];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) atomicAdd(misc + 3, part);
  __syncthreads();
  const int W = misc[3];
  const int chunk = max((W + C - 1) / C, kMinChunkTiles);
  for (int s = tid; s < S; s += blockDim.x) {
    const int ts = tiles[s];
    int r = 0;
    for (int s2 = 0; s2 < S; ++s2) {
      const int t2 = tiles[s2];
      r += (t2 > ts) || (t2 == ts && s2 < s);
    }
    order[r] = s;
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (S + 31) / 32;
    const int i0 = min(S, lane * per), i1 = min(S, i0 + per);
    int sp = 0, ss = 0;
    for (int i = i0; i < i1; ++i) {
      const int pc = max(1, (tiles[order[i]] + chunk - 1) / chunk);
      sp += pc;
      ss += pc > 1 ? pc : 0;
    }
    int ip = sp, is = ss;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, ip, o), v = __shfl_up_sync(0xffffffffu, is, o);
      if (lane >= o) {
        ip += u;
        is += v;
      }
    }
    int ep = ip - sp, es = is - ss;
    for (int i = i0; i < i1; ++i) {
      const int pc = max(1, (tiles[order[i]] + chunk - 1) / chunk);
      pre[i] = ep;
      sbase[i] = es;
      ep += pc;
      es += pc > 1 ? pc : 0;
    }
    if (lane == 31) pre[S] = ip;
  }
  __syncthreads();
  if (tid == 0) {
    const int N = pre[S];
    int n = 0;
    for (int k = 0; n < kMaxOwn; ++k) {
      const int idx = k * C + ((k & 1) ? C - 1 - c : c);
      if (idx >= N) break;
      int lo = 0, hi = S - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= idx) lo = mid; else hi = mid - 1;
      }
      const int s = order[lo];
      const int pc = pre[lo + 1] - pre[lo];
      const int piece = idx - pre[lo];
      const StripeGeo g = stripe_geo(a, s / a.P, s % a.P, false);
      const int tl = tiles[s];
      const int base = tl / pc, rem = tl % pc;
      const int st = piece * base + min(piece, rem);
      const int cnt = base + (piece < rem ? 1 : 0);
      MlaItem it;
      it.t = g.t;
      it.p = g.p;
      it.b = g.b;
      it.k_begin = st * kTile;
      it.k_end = min(ns[s], (st + cnt) * kTile);
      it.slot = pc > 1 ? sbase[lo] + piece : -1;
      it.slot_base = sbase[lo];
      it.npieces = pc;
      if (it.slot >= a.max_chunks) {  // the workspace bound makes this impossible; never write past it
        report(a.dev_status, CPATTN_DEV_BAD_INDPTR);
        it.t = -1;
      }
      items[n++] = it;
    }
    misc[2] = n;
  }
  __syncthreads();
}

// Item k of cluster c: from the plan's list, or (too many stripes to rank)
// stripe k * C + (snake c) in dispatch order, whole.
__device__ __forceinline__ bool get_item(const PartialArgs& a, int k, int C, int c, int n_items, const MlaItem* items,
                                         MlaItem& it) {
  if (n_items >= 0) {
    if (k >= n_items) return false;
    it = items[k];
    return true;
  }
  const int S = a.num_tokens * a.P;
  const int idx = k * C + ((k & 1) ? C - 1 - c : c);
  if (idx >= S) return false;
  const int z = idx / a.P, p = idx - z * a.P;
  int t = z;
  if (a.qo_indptr == nullptr && a.row_order != nullptr) {
    t = __ldg(a.row_order + z);
    if (t < 0 || t >= a.num_rows) {
      if (p == 0) report(a.dev_status, CPATTN_DEV_BAD_INDPTR);
      t = -1;
    }
  }
  const StripeGeo g = stripe_geo(a, t, p, true);
  it.t = g.t;
  it.p = g.p;
  it.b = g.b;
  it.k_begin = 0;
  it.k_end = g.n;
  it.slot = -1;
  it.slot_base = -1;
  it.npieces = 1;
  return true;
}

// Pool row of stripe slot k of the item (-1 if its page is rejected; reported when `rep`).
__device__ __forceinline__ int64_t pool_row(const PartialArgs& a, const MlaItem& it, int k, int pb0, int npg,
                                            bool rep) {
  const int jj = page_of_slot(a, k);
  if (jj >= npg) {
    if (rep) report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
    return -1;
  }
  const int pg = __ldg(a.page_indices + pb0 + jj);
  if (pg < 0 || pg >= a.num_pages) {
    if (rep) report(a.dev_status, CPATTN_DEV_PAGE_OUT_OF_RANGE);
    return -1;
  }
  return (static_cast<int64_t>(it.p) * a.num_pages + pg) * a.ps_l + (k - jj * a.ps_l);
}

// ---- grouped tiles (fused calls, logical pages of 64 slots) ----------------

// Keys of token t's row (clamped to max_kv_len; 0 for tokens of no row).
__device__ __forceinline__ int token_len(const PartialArgs& a, int t, int* b_out, bool may_report) {
  const StripeGeo g = stripe_geo(a, t, 0, may_report);
  *b_out = g.b;
  if (g.b < 0) return 0;
  int L = __ldg(a.kv_len + g.b);
  if (L > a.max_kv_len) L = a.max_kv_len;
  return max(L, 0);
}

// Cluster whose range of the W tiles holds tile x (ranges [c W / C, (c + 1) W / C)).
__device__ __forceinline__ int tile_cluster(int64_t x, int64_t W, int C) {
  return static_cast<int>(((x + 1) * C + W - 1) / W) - 1;
}

// The grouped plan (all threads; both CTAs compute the same one).  Token t
// with n > 0 pages spans kItemCostTiles + n positions of a sequence of all
// tokens -- a token's start (its Q load, its output store) costs a cluster
// about as much as that many tiles, so a cluster whose range starts a token
// inside it gets that many fewer pages -- and its pages sit at the last n of
// them.  pre[t] = first position of token t, pre[T] = W; sbase[t] = first
// workspace slot of a cut token (the pieces of cut tokens numbered in token
// order).  The W positions go to Ce = min(C, ceil(pages / 16)) clusters in
// equal contiguous ranges (clusters from Ce on get none).  misc[3] = W,
// misc[4] = Ce, misc[2] = first token of cluster c.
__device__ void mla_plan_group(const PartialArgs& a, int C, int c, int* pre, int* sbase, int* misc) {
  const int T = a.num_tokens;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (warp == 0) {
    const int per = (T + 31) / 32;
    const int i0 = min(T, lane * per), i1 = min(T, i0 + per);
    int sp = 0, sr = 0;  // positions, pages
    for (int t = i0; t < i1; ++t) {
      int b;
      const int n = (token_len(a, t, &b, true) + kTile - 1) / kTile;
      sr += n;
      sp += n > 0 ? n + kItemCostTiles : 0;
    }
    int ip = sp;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, ip, o);
      if (lane >= o) ip += u;
    }
    int ep = ip - sp;
    for (int t = i0; t < i1; ++t) {
      int b;
      pre[t] = ep;
      const int n = (token_len(a, t, &b, false) + kTile - 1) / kTile;
      ep += n > 0 ? n + kItemCostTiles : 0;
    }
    if (lane == 31) pre[T] = ip;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sr += __shfl_xor_sync(0xffffffffu, sr, o);
    __syncwarp();
    // workspace slots of cut tokens (pieces in token order)
    const int64_t W = pre[T];
    {
      const int64_t cap = (static_cast<int64_t>(sr) + kMinChunkTiles - 1) / kMinChunkTiles;
      if (cap < C) C = static_cast<int>(cap);
    }
    if (C < 1) C = 1;
    int ss = 0;
    for (int t = i0; t < i1; ++t) {
      const int n = pre[t + 1] - pre[t];
      const int pcs =
          n > 0 && W > 0 ? tile_cluster(pre[t + 1] - 1, W, C) - tile_cluster(pre[t] + kItemCostTiles, W, C) + 1 : 1;
      ss += pcs > 1 ? pcs : 0;
    }
    int is = ss;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, is, o);
      if (lane >= o) is += u;
    }
    int es = is - ss;
    for (int t = i0; t < i1; ++t) {
      const int n = pre[t + 1] - pre[t];
      const int pcs =
          n > 0 && W > 0 ? tile_cluster(pre[t + 1] - 1, W, C) - tile_cluster(pre[t] + kItemCostTiles, W, C) + 1 : 1;
      sbase[t] = es;
      es += pcs > 1 ? pcs : 0;
    }
    __syncwarp();
    if (lane == 0) {
      misc[3] = pre[T];
      misc[4] = C;
      // first token whose tiles reach into this cluster's range
      const int64_t s0 = static_cast<int64_t>(c) * W / C;
      int lo = 0, hi = T;  // first t with pre[t + 1] > s0
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid + 1] > s0) hi = mid; else lo = mid + 1;
      }
      misc[2] = lo;
    }
  }
  __syncthreads();
}

// Item k of cluster c in the grouped plan: token t_first + k, the part of its
// pages inside the cluster's range (k_begin / k_end in positions of the row;
// none when the range holds only the token's start cost).
__device__ __forceinline__ bool get_item_group(const PartialArgs& a, int k, int C, int c, const int* pre,
                                               const int* sbase, int64_t W, int t_first, MlaItem& it) {
  const int t = t_first + k;
  if (t >= a.num_tokens || W == 0 || c >= C) return false;
  const int64_t s0 = static_cast<int64_t>(c) * W / C, s1 = static_cast<int64_t>(c + 1) * W / C;
  if (pre[t] >= s1) return false;
  int b;
  const int L = token_len(a, t, &b, false);
  const int64_t pt0 = pre[t], pt1 = pre[t + 1];
  const int64_t f0 = pt1 > pt0 ? pt0 + kItemCostTiles : pt0;  // position of the token's first page
  const int64_t lo = f0 > s0 ? f0 : s0, hi = pt1 < s1 ? pt1 : s1;
  it.t = t;
  it.p = 0;
  it.b = b;
  it.k_begin = 0;
  it.k_end = 0;
  if (hi > lo) {  // else: a token of no pages (written by the zero pass), or only its start cost here
    it.k_begin = static_cast<int>(lo - f0) * kTile;
    it.k_end = min(L, static_cast<int>(hi - f0) * kTile);
  }
  const int n = pre[t + 1] - pre[t];
  const int c0 = n > 0 ? tile_cluster(f0, W, C) : c;
  const int pcs = n > 0 ? tile_cluster(pre[t + 1] - 1, W, C) - c0 + 1 : 1;
  it.npieces = pcs;
  it.slot_base = sbase[t];
  it.slot = pcs > 1 ? sbase[t] + (c - c0) : -1;
  if (it.slot >= a.max_chunks) {  // the workspace bound makes this impossible; never write past it
    if (threadIdx.x == 0) report(a.dev_status, CPATTN_DEV_BAD_INDPTR);
    it.t = -1;
  }
  return true;
}

// Row of the page pool where logical page (k_begin / 64 + j) of the item
// starts in every partner's pool (page id * page_size / P), or -1 (past the
// table, rejected page; reported when `rep`).
__device__ __forceinline__ int group_page_row(const PartialArgs& a, const MlaItem& it, int j, int pb0, int npg,
                                              bool rep) {
  const int jj = it.k_begin / kTile + j;
  if (jj >= npg) {
    if (rep) report(a.dev_status, CPATTN_DEV_POS_PAST_TABLE);
    return -1;
  }
  const int pg = __ldg(a.page_indices + pb0 + jj);
  if (pg < 0 || pg >= a.num_pages) {
    if (rep) report(a.dev_status, CPATTN_DEV_PAGE_OUT_OF_RANGE);
    return -1;
  }
  return pg * a.ps_l;
}

// Page-table words behind the key mask of tile j, read a tile before the
// mask is needed (tile_mask_from takes the decision then), so the table's
// latency hides behind the previous tile.  Grouped tiles: the logical page
// (same word in every lane); per-partner tiles: the pages of keys lane and
// 32 + lane.  -2: no word (past the item or the table).
struct MaskWords {
  int pa, pb;
};
template <bool kGroup>
__device__ __forceinline__ MaskWords tile_mask_words(const PartialArgs& a, const MlaItem& it, int j, int pb0, int npg,
                                                     int lane) {
  MaskWords w{-2, -2};
  if constexpr (kGroup) {
    const int jj = it.k_begin / kTile + j;
    if (jj < npg) w.pa = __ldg(a.page_indices + pb0 + jj);
  } else {
    const int ka = it.k_begin + j * kTile + lane, kb = ka + 32;
    if (ka < it.k_end) {
      const int jj = page_of_slot(a, ka);
      if (jj < npg) w.pa = __ldg(a.page_indices + pb0 + jj);
    }
    if (kb < it.k_end) {
      const int jj = page_of_slot(a, kb);
      if (jj < npg) w.pb = __ldg(a.page_indices + pb0 + jj);
    }
  }
  return w;
}
// Key mask of tile j (one bit a key, every lane gets it) from the words read
// before: a key holds data when its page is accepted and its position lies
// inside the item.  Grouped tile row r is partner p = r / ps_l's physical
// slot l = r % ps_l of the logical page, at in-page offset
// (l / I) * I * P + p * I + l % I (I = 1: l * P + p).
template <bool kGroup>
__device__ __forceinline__ uint64_t tile_mask_from(const PartialArgs& a, const MlaItem& it, int j, MaskWords w,
                                                   int lane) {
  auto page_ok = [&](int pg) { return pg >= 0 && pg < a.num_pages; };
  if constexpr (kGroup) {
    if (!page_ok(w.pa)) return 0ull;
    const int base = it.k_begin + j * kTile;
    if (base + kTile <= it.k_end) return ~0ull;  // the rows hold positions base .. base + 63
    const int I = a.interleave;
    auto pos_of = [&](int r) {
      const int p = r / a.ps_l, l = r - (r / a.ps_l) * a.ps_l;
      return base + (l / I) * I * a.P + p * I + (l % I);
    };
    const uint32_t lo = __ballot_sync(0xffffffffu, pos_of(lane) < it.k_end);
    const uint32_t hi = __ballot_sync(0xffffffffu, pos_of(lane + 32) < it.k_end);
    return static_cast<uint64_t>(lo) | (static_cast<uint64_t>(hi) << 32);
  } else {
    const uint32_t lo = __ballot_sync(0xffffffffu, page_ok(w.pa)), hi = __ballot_sync(0xffffffffu, page_ok(w.pb));
    return static_cast<uint64_t>(lo) | (static_cast<uint64_t>(hi) << 32);
  }
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, int x, int y, int z, int w, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];\n" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(mbar)
      : "memory");
}

// Copies of column blocks kb0 .. kb0 + nb - 1 of grouped tile j into dst
// (8 KB a block), by the calling lane: one 4-D box (64 values x ps_l rows x
// P partners x nb blocks; the map's box holds nb blocks); page_row from
// group_page_row (-1: nothing copied).
__device__ __forceinline__ void load_unit_group(const CUtensorMap* tmap, uint32_t dst, int kb0, int nb, uint32_t full,
                                                int page_row) {
  tc05::mbar_arrive_expect_tx(full, page_row >= 0 ? nb * kBlk : 0);
  if (page_row >= 0) tma_load_4d(dst, tmap, 0, page_row, 0, kb0, full);
}

// Pool rows of the page runs of tile j (TMA path): lane r < kTile / box_rows
// looks up run r (-1: past the item or a rejected page, reported), so a tile
// costs one round trip to the page table.
__device__ __forceinline__ int tile_run_row(const PartialArgs& a, const MlaItem& it, int j, int pb0, int npg,
                                            int box_rows, int lane) {
  const int kr = it.k_begin + j * kTile + lane * box_rows;
  if (lane >= kTile / box_rows || kr >= it.k_end) return -1;
  return static_cast<int>(pool_row(a, it, kr, pb0, npg, true));
}

// Copies of column blocks kb0 .. kb0 + nb - 1 of a per-partner tile by TMA
// boxes of box_rows rows: lane r issues run r's boxes (run_row: its pool row
// from tile_run_row, -1: not copied), lane 0 counts the bytes (run_bytes a
// block, all runs) on `full`.  The whole warp calls.
__device__ __forceinline__ void load_unit_runs(const CUtensorMap* tmap, uint32_t dst, int kb0, int nb, uint32_t full,
                                               int run_row, uint32_t run_bytes, int box_rows, int lane) {
  if (lane == 0) tc05::mbar_arrive_expect_tx(full, nb * run_bytes);
  if (run_row >= 0)
    for (int kb = 0; kb < nb; ++kb)
      tc05::tma_load_2d(dst + kb * kBlk + lane * box_rows * 128, tmap, (kb0 + kb) * 64, run_row, full);
}

// Copy path (no TMA): source rows of keys lane and 32 + lane of tile j
// (nullptr: no data).
__device__ __forceinline__ void cp_tile_rows(const PartialArgs& a, const MlaItem& it, int j, int pb0, int npg, int lane,
                                             const uint8_t*& r0, const uint8_t*& r1) {
  const uint8_t* pool = static_cast<const uint8_t*>(a.pool_k);
  const int ka = it.k_begin + j * kTile + lane, kb = ka + 32;
  r0 = nullptr;
  r1 = nullptr;
  if (ka < it.k_end) {
    const int64_t row = pool_row(a, it, ka, pb0, npg, true);
    if (row >= 0) r0 = pool + row * (kDqk * 2);
  }
  if (kb < it.k_end) {
    const int64_t row = pool_row(a, it, kb, pb0, npg, true);
    if (row >= 0) r1 = pool + row * (kDqk * 2);
  }
}

// Copy path: column blocks kb0 .. kb0 + nb - 1 of the tile by 16-byte
// cp.async copies of the whole warp (zero fill for keys without data),
// counted on `full` (32 arrivals).
__device__ __forceinline__ void cp_tile_blocks(uint32_t dst, int kb0, int nb, const uint8_t* r0, const uint8_t* r1,
                                               const void* any_gmem, uint32_t full, int lane) {
  const int nch = nb * 8;  // 16-byte chunks of a key row
  for (int idx = lane; idx < kTile * nch; idx += 32) {
    const int key = idx / nch, ch = idx - key * nch;
    const uintptr_t s0 = __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(r0), key & 31);
    const uintptr_t s1 = __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(r1), key & 31);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(key < 32 ? s0 : s1);
    const uint32_t d = dst + (ch >> 3) * kBlk + tc05::sw128(key, ch & 7);
    if (src != nullptr) cp16(d, src + (kb0 * 8 + ch) * 16);
    else cp16_zero(d, any_gmem);
  }
  cp_arrive_noinc(full);
}

}  // namespace

template <bool kTma, bool kGroup>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_pair_kernel(const PartialArgs a, const __grid_constant__ CUtensorMap tmap,
                    const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_out,
                    const __grid_constant__ CUtensorMap tmap_ws, int box_rows) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = tc05::smem_addr(base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = tc05::cluster_rank();  // 0: scores, 1: values
  const uint32_t peer = rank ^ 1u;
  const int C = gridDim.x / 2, c = blockIdx.x / 2;
  int* misc = reinterpret_cast<int*>(base + OFF_MISC);
  volatile int* abort_flag = misc + 1;
  MlaItem* items = reinterpret_cast<MlaItem*>(base + OFF_ITEMS);
  auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + static_cast<uint32_t>(i) * 8u; };
  auto raise_abort = [&]() {
    *abort_flag = 1;
    tc05::st_cluster_u32(tc05::mapa(sb + OFF_MISC + 4, peer), 1u);
    report(a.dev_status, CPATTN_DEV_TC_TIMEOUT);
  };

  // the merge of cut tokens (grouped plans) may be scheduled already; it
  // waits for this grid's completion before it reads anything
  if (tid == 0) pdl_trigger();
  pdl_wait();  // every input may come from the kernels before this one
  // ---- plan, barriers, tensor memory
  if (tid == 0) {
    misc[1] = 0;
    misc[2] = -1;
    misc[3] = 0;
    misc[4] = C;
  }
  __syncthreads();
  int* g_pre = reinterpret_cast<int*>(base + OFF_ITEMS);  // grouped plans: [kGroupMaxTokens + 1]
  int* g_sbase = g_pre + (kGroupMaxTokens + 1);            //                [kGroupMaxTokens]
  if constexpr (kGroup) {
    mla_plan_group(a, C, c, g_pre, g_sbase, misc);
  } else {
    const int S = a.num_tokens * a.P;
    if (S <= kSortMax && S + 2 * C <= kMaxOwn * C) mla_plan(a, C, c, reinterpret_cast<int*>(base), misc, items);
  }
  if (tid == 0) {
    const uint32_t load_arrivals = kTma ? 1u : 32u;
    for (int i = 0; i < kKUnits; ++i) {
      tc05::mbar_init(bar(B_KFULL + i), load_arrivals);
      tc05::mbar_init(bar(B_KEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc05::mbar_init(bar(B_SFULL + i), 1);
      tc05::mbar_init(bar(B_SEMPTY + i), 4);
    }
    for (int i = 0; i < kTileRing; ++i) {
      tc05::mbar_init(bar(B_READY + i), 4);
      tc05::mbar_init(bar(B_PVDONE + i), 1);
    }
    for (int i = 0; i < kPBufs; ++i) {
      tc05::mbar_init(bar(B_PEMPTY + i), 1);
      tc05::mbar_init(bar(B_PFULL + i), 1);
    }
    for (int i = 0; i < kVRing; ++i) {
      tc05::mbar_init(bar(B_VFULL + i), load_arrivals);
      tc05::mbar_init(bar(B_VEMPTY + i), 1);
    }
    tc05::mbar_init(bar(B_QFULL), 4);
    tc05::mbar_init(bar(B_QEMPTY), 1);
    tc05::mbar_init(bar(B_FINEMPTY), 4);
    tc05::mbar_init(bar(B_FINFULL), 1);
    tc05::mbar_init(bar(B_DRAIN), 1);
    tc05::mbar_init(bar(B_EPSYNC), kHeads);
    tc05::mbar_init(bar(B_MERGE), 1);
    tc05::mbar_init(bar(B_MERGE + 1), 1);
    for (int i = 0; i < kLandRing; ++i) tc05::mbar_init(bar(B_KLAND + i), 1);
    tc05::mbar_init_fence();
  }
  if (warp == 0) tc05::tmem_alloc(tc05::smem_addr(misc), 512);
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  tc05::cluster_sync();  // the peer's barriers exist before any remote arrival
  const uint32_t tbase = static_cast<uint32_t>(misc[0]);
  const int n_items = misc[2];
  const int64_t g_W = misc[3];
  const int g_C = misc[4];  // grouped plans: clusters with a range
  auto item = [&](int k, MlaItem& it) {
    if constexpr (kGroup) return get_item_group(a, k, g_C, c, g_pre, g_sbase, g_W, n_items, it);
    else return get_item(a, k, C, c, n_items, items, it);
  };
  auto mask_words = [&](const MlaItem& it, int j, int pb0, int npg) {
    return tile_mask_words<kGroup>(a, it, j, pb0, npg, lane);
  };
  auto ntiles = [](const MlaItem& it) {
    return it.t >= 0 && it.k_end > it.k_begin ? (it.k_end - it.k_begin + kTile - 1) / kTile : 0;
  };
  bool ok = true;

  if (warp == kWLoad) {
    // ---- loader (both CTAs).  CTA 0: whole latent rows in units of kUBlk
    // column blocks into a ring of kKUnits units (a unit is free again once
    // the S MMAs that read it are done).  CTA 1: the value part of the same
    // tiles into a ring of kVRing units of kVUB column blocks.  The ring constants are
    // compile-time per role: this warp shares its scheduler with a softmax
    // warp, so every instruction it issues per unit counts.
    auto run = [&](auto kU_, auto kUB_, auto kR_, auto kBytes_, int b_full, int b_empty, const CUtensorMap* map4) {
      constexpr int kU = decltype(kU_)::value, kUB = decltype(kUB_)::value, kR = decltype(kR_)::value;
      constexpr uint32_t kBytes = decltype(kBytes_)::value;
      int g = 0, q = 0, issued = 0;  // tiles, next unit's slot, units issued
      uint32_t par = 0;              // parity of the slot's next use
      for (int k = 0; ok; ++k) {
        MlaItem it;
        if (!item(k, it)) break;
        const int nt = ntiles(it);
        if (nt == 0) continue;
        const int pb0 = __ldg(a.page_indptr + it.b), npg = __ldg(a.page_indptr + it.b + 1) - pb0;
        // page rows of the next tile are looked up while the stage it goes to is still busy
        auto rows_of = [&](int jt) { return kTma ? tile_run_row(a, it, jt, pb0, npg, box_rows, lane) : -1; };
        // grouped plans: lane l holds the page row of tile j0 + l of the current
        // batch of 32 tiles, and the next batch is read while this one is used
        auto batch_of = [&](int j0) { return j0 + lane < nt ? group_page_row(a, it, j0 + lane, pb0, npg, true) : -1; };
        int cur_rows = 0, next_rows = 0;
        if constexpr (kGroup) {
          cur_rows = batch_of(0);
          next_rows = batch_of(32);
        } else {
          (void)cur_rows;
          (void)next_rows;
        }
        int run_row = kGroup ? 0 : rows_of(0);
        for (int j = 0; j < nt; ++j, ++g) {
          if constexpr (kGroup) {
            if (j > 0 && (j & 31) == 0) {
              cur_rows = next_rows;
              next_rows = batch_of(j + 32);
            }
            run_row = __shfl_sync(0xffffffffu, cur_rows, j & 31);
          }
          // CTA 1 copies a tile's value rows once CTA 0 has the whole rows:
          // they are in L2 by then, and CTA 1's copies do not race CTA 0's to HBM
          if (rank == 1) ok = wwait<true>(bar(B_KLAND + g % kLandRing), (g / kLandRing) & 1, abort_flag);
          if (!ok) break;
          int nu = 0;  // units of this tile issued
          if constexpr (kTma) {
            // per-partner tiles: lane r < kTile / box_rows copies run r; grouped
            // tiles: lane 0 copies the unit with one 4-D box
            uint32_t run_bytes = 0;
            if constexpr (!kGroup)
              run_bytes = __popc(__ballot_sync(0xffffffffu, run_row >= 0)) * static_cast<uint32_t>(box_rows) * 128u;
            else
              (void)run_bytes;
            int qq = q;
            uint32_t pp = par;
            if constexpr (kGroup) {
              // lane 0 alone: no warp-wide step a unit
              if (lane == 0) {
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                  if (!pwait<false>(bar(b_empty + qq), pp ^ 1u, abort_flag)) break;
                  load_unit_group(map4, sb + qq * kBytes, u * kUB, kUB, bar(b_full + qq), run_row);
                  ++nu;
                  if (++qq == kR) {
                    qq = 0;
                    pp ^= 1u;
                  }
                }
              }
              nu = __shfl_sync(0xffffffffu, nu, 0);
            } else {
#pragma unroll
              for (int u = 0; u < kU; ++u) {
                if (!wwait<false>(bar(b_empty + qq), pp ^ 1u, abort_flag)) break;
                load_unit_runs(&tmap, sb + qq * kBytes, u * kUB, kUB, bar(b_full + qq), run_row, run_bytes, box_rows,
                               lane);
                ++nu;
                if (++qq == kR) {
                  qq = 0;
                  pp ^= 1u;
                }
              }
            }
          } else {
            const uint8_t* r0;
            const uint8_t* r1;
            cp_tile_rows(a, it, j, pb0, npg, lane, r0, r1);
            int qq = q;
            uint32_t pp = par;
            for (int u = 0; u < kU; ++u) {
              if (!wwait<false>(bar(b_empty + qq), pp ^ 1u, abort_flag)) break;
              cp_tile_blocks(sb + qq * kBytes, u * kUB, kUB, r0, r1, a.pool_k, bar(b_full + qq), lane);
              ++nu;
              if (++qq == kR) {
                qq = 0;
                pp ^= 1u;
              }
            }
          }
          issued += nu;
          ok = nu == kU;
          if (!ok) break;
          q += kU;
          if (q >= kR) {
            q -= kR;
            par ^= 1u;
          }
          if (!kGroup && j + 1 < nt) run_row = rows_of(j + 1);
        }
      }
      if (!ok) raise_abort();
      if (*abort_flag) {
        // nothing may land after the CTA exits: wait (bounded) for the last copies issued into each slot
        for (int n2 = max(0, issued - kR); n2 < issued; ++n2) {
          const uint32_t mb = bar(b_full + n2 % kR), par2 = (n2 / kR) & 1;
          for (uint32_t i = 0; i < (1u << 20); ++i) {
            uint32_t done;
            asm volatile(
                "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                : "=r"(done)
                : "r"(mb), "r"(par2)
                : "memory");
            if (done) break;
          }
        }
      }
    };
    if (rank == 0)
      run(std::integral_constant<int, kUnitsK>{}, std::integral_constant<int, kUBlk>{},
          std::integral_constant<int, kKUnits>{}, std::integral_constant<uint32_t, kKUnit>{}, B_KFULL, B_KEMPTY, &tmap);
    else
      run(std::integral_constant<int, kVUnits>{}, std::integral_constant<int, kVUB>{},
          std::integral_constant<int, kVRing>{}, std::integral_constant<uint32_t, kVUnit>{}, B_VFULL, B_VEMPTY, &tmap_v);
  } else if (rank == 0 && warp == kWMma) {
    // ---- CTA 0, MMA warp (one elected lane issues): S = Q K^T of each tile, Q from tensor memory
    const uint32_t id_s = tc05::idesc_bf16(128, kTile, false, false);
    const uint32_t r_kland = tc05::mapa(bar(B_KLAND), 1);
    int g = 0, qi = 0, kq = 0;  // kq, kpar: ring slot of the next tile's first unit and its use parity
    uint32_t kpar = 0;
    for (int k = 0; ok; ++k) {
      MlaItem it;
      if (!item(k, it)) break;
      const int nt = ntiles(it);
      if (nt == 0) continue;
      ok = wwait<false>(bar(B_QFULL), qi & 1, abort_flag);
      for (int j = 0; j < nt && ok; ++j, ++g) {
        const int sbuf = g & 1;
        ok = wwait<false>(bar(B_SEMPTY + sbuf), ((g >> 1) & 1) ^ 1, abort_flag);
        if (!ok) break;
        bool fail = false;
        if (tc05::elect_one()) {
          // unit u of the tile sits in ring slot kq + u (mod kKUnits); its 12
          // MMAs go as soon as it landed, and a commit frees the slot
          const uint32_t dcol = tbase + sbuf * kTile;
          int q = kq;
          uint32_t par = kpar;
#pragma unroll
          for (int u = 0; u < kUnitsK; ++u) {
            if (!pwait<false>(bar(B_KFULL + q), par, abort_flag)) {
              fail = true;
              break;
            }
            // the tile's last unit landed, so all its rows sit in L2: CTA 1 may
            // copy their value part (a signal only, nothing to publish)
            if (u == kUnitsK - 1) tc05::mbar_arrive_remote_relaxed(r_kland + (g % kLandRing) * 8);
            if constexpr (!kTma) tc05::fence_smem_to_async();  // the unit came through cp.async
            tc05::fence_after_sync();
#pragma unroll
            for (int b = 0; b < kUBlk; ++b) {
              const uint64_t dk = tc05::desc_k128(sb + q * kKUnit + b * kBlk);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const int ks = (u * kUBlk + b) * 4 + kk;
                tc05::mma_ts(dcol, tbase + kQCol + ks * 8, tc05::desc_add(dk, kk * 32), id_s, ks > 0);
              }
            }
            tc05::commit(bar(B_KEMPTY + q));
            if (++q == kKUnits) {
              q = 0;
              par ^= 1u;
            }
          }
          if (!fail) tc05::commit(bar(B_SFULL + sbuf));
        }
        ok = __ballot_sync(0xffffffffu, fail) == 0u;
        kq += kUnitsK;
        if (kq >= kKUnits) {
          kq -= kKUnits;
          kpar ^= 1u;
        }
      }
      if (!ok) break;
      if (tc05::elect_one()) tc05::commit(bar(B_QEMPTY));
      __syncwarp();
      ++qi;
    }
    if (!ok) raise_abort();
    if (tc05::elect_one()) {
      tc05::commit(bar(B_DRAIN));
      tc05::mbar_wait(bar(B_DRAIN), 0, 1u << 20);
    }
    __syncwarp();
  } else if (rank == 0 && warp < 4) {
    // ---- CTA 0, warps 0-3: Q into tensor memory, online softmax, P to CTA 1
    const float sl = a.scale * kLog2e;
    const uint32_t my_lane = tc05::taddr(tbase, warp * 32, 0);
    const uint32_t r_p = tc05::mapa(sb + OFF_P, 1), r_alpha = tc05::mapa(sb + OFF_ALPHA, 1);
    const uint32_t r_fin = tc05::mapa(sb + OFF_FIN, 1);
    const uint32_t r_pfull = tc05::mapa(bar(B_PFULL), 1), r_finfull = tc05::mapa(bar(B_FINFULL), 1);
    const uint32_t pst = sb + OFF_PSTAGE + tid * 128;  // this row's place in the warp's staging slot
    int g = 0, qi = 0, prev_t = -1;
    for (int k = 0; ok; ++k) {
      MlaItem it;
      if (!item(k, it)) break;
      const int nt = ntiles(it);
      if (nt == 0) continue;
      const int pb0 = __ldg(a.page_indptr + it.b), npg = __ldg(a.page_indptr + it.b + 1) - pb0;
      // Q row (token it.t, head tid) -> columns 128..415 of lane tid, once the previous item's S is done
      ok = wwait<false>(bar(B_QEMPTY), (qi & 1) ^ 1, abort_flag);
      if (!ok) break;
      tc05::fence_after_sync();
      if (it.t != prev_t) {
        // coalesced: a lane loads 16-byte chunk (lane & 7) of rows 4 i + lane / 8
        // of its warp's 32 (four whole 128-byte lines an instruction), a
        // 64-value column block at a time through the warp's P staging slot,
        // where thread r then reads its row's block for tcgen05.st
        if (lane == 0) tc05::bulk_wait_read();  // the slot's last P copy has read it
        __syncwarp();
        const uint8_t* qrows =
            static_cast<const uint8_t*>(a.q) + (static_cast<int64_t>(it.t) * a.num_q_heads + warp * 32) * (kDqk * 2);
        uint8_t* slot = base + OFF_PSTAGE + warp * kPSlot;
        const int lr8 = lane >> 3, lc = lane & 7;
        constexpr int kGrp = 3;  // column blocks whose loads are in flight together
#pragma unroll
        for (int g0 = 0; g0 < kKB; g0 += kGrp) {
          uint4 u[kGrp][8];
#pragma unroll
          for (int b = 0; b < kGrp; ++b)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (g0 + b < kKB)
                u[b][i] =
                    __ldg(reinterpret_cast<const uint4*>(qrows + (4 * i + lr8) * (kDqk * 2) + (g0 + b) * 128 + lc * 16));
#pragma unroll
          for (int b = 0; b < kGrp; ++b) {
            if (g0 + b >= kKB) break;
#pragma unroll
            for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4*>(slot + tc05::sw128(4 * i + lr8, lc)) = u[b][i];
            __syncwarp();
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 v = *reinterpret_cast<const uint4*>(slot + tc05::sw128(lane, c));
              w[4 * c] = v.x;
              w[4 * c + 1] = v.y;
              w[4 * c + 2] = v.z;
              w[4 * c + 3] = v.w;
            }
            __syncwarp();  // the slot is rewritten for the next block
            tc05::st_x16_u32(my_lane + kQCol + (g0 + b) * 32, *reinterpret_cast<uint32_t(*)[16]>(w));
            tc05::st_x16_u32(my_lane + kQCol + (g0 + b) * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(w + 16));
          }
        }
        tc05::st_wait();
        prev_t = it.t;
      }
      tc05::fence_before_sync();
      __syncwarp();
      if (lane == 0) arrive_local(bar(B_QFULL));
      // the next item's Q row goes into L2 some eight tiles before this item ends
      int next_t = -1;
      {
        MlaItem nx;
        if (item(k + 1, nx) && nx.t >= 0 && nx.t != it.t) next_t = nx.t;
      }
      const int j_pf = nt > 8 ? nt - 8 : 0;
      float m = -INFINITY, l = 0.f, lr = 0.f;
      MaskWords next_words = mask_words(it, 0, pb0, npg);
      for (int j = 0; j < nt; ++j, ++g) {
        const int sbuf = g & 1;
        if (j == j_pf && next_t >= 0) {
          const char* q2 = static_cast<const char*>(a.q) + (static_cast<int64_t>(next_t) * a.num_q_heads + tid) * (kDqk * 2);
#pragma unroll
          for (int ln = 0; ln < (kDqk * 2) / 128; ++ln) asm volatile("prefetch.global.L2 [%0];\n" ::"l"(q2 + ln * 128));
        }
        const MaskWords words = next_words;
        if (j + 1 < nt) next_words = mask_words(it, j + 1, pb0, npg);
        ok = wwait<false>(bar(B_SFULL + sbuf), (g >> 1) & 1, abort_flag);
        if (!ok) break;
        tc05::fence_after_sync();
        float sv[kTile];
        {
          float v0[16], v1[16], v2[16], v3[16];
          tc05::ld_x16(my_lane + sbuf * kTile, v0);
          tc05::ld_x16(my_lane + sbuf * kTile + 16, v1);
          tc05::ld_x16(my_lane + sbuf * kTile + 32, v2);
          tc05::ld_x16(my_lane + sbuf * kTile + 48, v3);
          tc05::ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            sv[e] = v0[e];
            sv[16 + e] = v1[e];
            sv[32 + e] = v2[e];
            sv[48 + e] = v3[e];
          }
        }
        tc05::fence_before_sync();
        __syncwarp();
        if (lane == 0) arrive_local(bar(B_SEMPTY + sbuf));
        // keys without data: -inf (so their probability is 0); the running max
        // is kept in log2 units, the scores stay unscaled
        const uint64_t vmask = tile_mask_from<kGroup>(a, it, j, words, lane);
        if (vmask != ~0ull) {
#pragma unroll
          for (int e = 0; e < kTile; ++e) sv[e] = ((vmask >> e) & 1ull) ? sv[e] : -INFINITY;
        }
        float mx[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) mx[e] = fmaxf(fmaxf(sv[e], sv[16 + e]), fmaxf(sv[32 + e], sv[48 + e]));
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
          for (int e = 0; e < w; ++e) mx[e] = fmaxf(mx[e], mx[e + w]);
        const float bm = mx[0] * sl;
        float alpha = 1.f;
        if (bm > m + 8.f) {
          alpha = m == -INFINITY ? 0.f : exp2f(m - bm);
          l *= alpha;
          lr *= alpha;
          m = bm;
        }
        // The row of P (bf16, 128-byte swizzle) goes to this warp's staging
        // slot, once the slot's previous copy has read it; the slot then
        // travels to P buffer `sbuf` of CTA 1 as one bulk copy, and the rescale
        // factor by an asynchronous store, both counted in bytes on CTA 1's
        // barrier.  The buffer is free once its P V two tiles back is done.
        if (lane == 0) tc05::bulk_wait_read();
        __syncwarp();
        {
          // p = 2^(s * scale * log2 e - m): one FMA and one ex2 a key (a key
          // at -inf gives 0; while every key so far is masked m is -inf and
          // every p is 0); four partial sums of p and of bf16(p) each
          const float nm = m == -INFINITY ? 0.f : -m;
          float ls[4] = {0.f, 0.f, 0.f, 0.f}, lrs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t pk[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const int e = 8 * cc + 2 * e2;
              const float p0 = ex2_approx(fmaf(sv[e], sl, nm));
              const float p1 = ex2_approx(fmaf(sv[e + 1], sl, nm));
              ls[e2] += p0 + p1;
              __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
              pk[e2] = *reinterpret_cast<uint32_t*>(&pb);
              lrs[e2] += __uint_as_float(pk[e2] << 16) + __uint_as_float(pk[e2] & 0xffff0000u);
            }
            tc05::st_shared_v4(pst + ((cc ^ (tid & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
          }
          l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
          lr += (lrs[0] + lrs[1]) + (lrs[2] + lrs[3]);
        }
        tc05::fence_smem_to_async();  // the copy engine reads what these threads wrote
        const int pq = g % kPBufs;
        ok = wwait<true>(bar(B_PEMPTY + pq), ((g / kPBufs) & 1) ^ 1, abort_flag);
        if (!ok) break;
        const uint32_t pfull = r_pfull + pq * 8;
        tc05::st_async_b32(r_alpha + (pq * kHeads + tid) * 4, __float_as_uint(alpha), pfull);
        if (lane == 0) {
          tc05::bulk_s2cluster(r_p + pq * kPBuf + warp * kPSlot, sb + OFF_PSTAGE + warp * kPSlot, kPSlot, pfull);
          tc05::bulk_commit();
        }
      }
      if (!ok) break;
      // the item's row scale and LSE to CTA 1, once it read the previous item's
      ok = wwait<true>(bar(B_FINEMPTY), (qi & 1) ^ 1, abort_flag);
      if (!ok) break;
      const float inv = lr > 0.f ? 1.f / lr : 0.f;
      const float lse = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      // an asynchronous store counted in bytes on CTA 1's barrier: no
      // cluster-scope release, which would wait for this CTA's copies in flight
      tc05::st_async_v2(r_fin + tid * 8, __float_as_uint(inv), __float_as_uint(lse), r_finfull);
      ++qi;
    }
    if (!ok) raise_abort();
    if (lane == 0) tc05::bulk_wait_all();  // the staging slot stays until its last copy is done
    __syncwarp();
  } else if (warp == kWMma) {
    // ---- CTA 1, MMA warp (one elected lane issues): O += P V
    const uint32_t id_pv = tc05::idesc_bf16(128, 256, false, true);
    int g = 0;
    for (int k = 0; ok; ++k) {
      MlaItem it;
      if (!item(k, it)) break;
      const int nt = ntiles(it);
      for (int j = 0; j < nt; ++j, ++g) {
        const int pbuf = g % kTileRing;
        ok = wwait<false>(bar(B_READY + pbuf), (g / kTileRing) & 1, abort_flag);
        if (!ok) break;
        bool fail = false;
        if (tc05::elect_one()) {
          tc05::fence_after_sync();
          const uint64_t dp = tc05::desc_k128(sb + OFF_P + (g % kPBufs) * kPBuf);
          // value unit h (columns 64 kVUB h ..) of the tile: its MMAs go as
          // soon as it landed, and a commit frees its ring slot
#pragma unroll
          for (int h = 0; h < kVUnits; ++h) {
            const int n = g * kVUnits + h, vq = n % kVRing;
            if (!pwait<false>(bar(B_VFULL + vq), (n / kVRing) & 1, abort_flag)) {
              fail = true;
              break;
            }
            if constexpr (!kTma) tc05::fence_smem_to_async();  // the unit came through cp.async
            tc05::fence_after_sync();
            const uint64_t dv = tc05::desc_mn128(sb + vq * kVUnit, kBlk);
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks) {
              const uint64_t ad = tc05::desc_add(dp, ks * 32);
              const uint64_t bd = tc05::desc_add(dv, ks * 16 * 128);
#pragma unroll
              for (int c = 0; c < kVUB / 4; ++c)
                tc05::mma_ss(tbase + (h * kVUB + 4 * c) * 64, ad, tc05::desc_add(bd, 4 * c * kBlk), id_pv,
                             j > 0 || ks > 0);
            }
            tc05::commit(bar(B_VEMPTY + vq));
          }
          if (!fail) {
            tc05::commit(bar(B_PVDONE + pbuf));
            tc05::commit_multicast(bar(B_PEMPTY + g % kPBufs), 0x1);
          }
        }
        ok = __ballot_sync(0xffffffffu, fail) == 0u;
        if (!ok) break;
      }
    }
    if (!ok) raise_abort();
    if (tc05::elect_one()) {
      tc05::commit(bar(B_DRAIN));
      tc05::mbar_wait(bar(B_DRAIN), 0, 1u << 20);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ---- CTA 1, warps 0-3: value-row fixes, O rescales, the normalised output
    const uint32_t my_lane = tc05::taddr(tbase, warp * 32, 0);
    const uint32_t r_finempty = tc05::mapa(bar(B_FINEMPTY), 0);
    const float* alpha_s = reinterpret_cast<const float*>(base + OFF_ALPHA);
    const float2* fin_s = reinterpret_cast<const float2*>(base + OFF_FIN);
    float* scratch = reinterpret_cast<float*>(base + OFF_SCR);
    // grouped plans: per token (slot of its first piece, pieces; 1: whole)
    int32_t* rec = a.ws_cnt + static_cast<int64_t>(a.num_tokens) * a.P;
    // O (tensor memory, this thread's row = head tid) times wo, plus we times
    // row tid of ext when given, into the 128 rows at dst0 (a row every 512
    // elements; fp32, or bf16 rounded to nearest even).  Staged through shared
    // memory in 128-byte chunks of every row, so that eight threads store each
    // line.  All epilogue threads call.
    // With `map` (grouped plans), each staged chunk leaves by a TMA store of
    // the box at column ch * cols, row y0; else by the threads' stores.
    auto store_rows_t = [&](auto bf16_c, void* dst0, const CUtensorMap* map, int y0, float wo, float we,
                            const float* ext) {
      constexpr bool kB = decltype(bf16_c)::value;
      constexpr int cols = kB ? 64 : 32, nch = kDv / cols, esz = kB ? 2 : 4;
      // the next chunk's tensor-memory loads (and extra rows) are in flight
      // while this chunk goes out
      float v[cols];
      float4 xe[cols / 4];
      auto fetch = [&](int ch) {
#pragma unroll
        for (int q = 0; q < cols / 16; ++q)
          tc05::ld_x16(my_lane + ch * cols + 16 * q, *reinterpret_cast<float(*)[16]>(v + 16 * q));
        if (ext != nullptr) {
#pragma unroll
          for (int e = 0; e < cols / 4; ++e)
            xe[e] = __ldg(reinterpret_cast<const float4*>(ext + static_cast<int64_t>(tid) * kDv + ch * cols) + e);
        }
      };
      fetch(0);
#pragma unroll 1
      for (int ch = 0; ch < nch; ++ch) {
        uint8_t* buf = base + OFF_SCR + (ch & 1) * (kHeads * 128);
        tc05::ld_wait();
        uint32_t wds[32];
#pragma unroll
        for (int e = 0; e < cols; ++e) v[e] *= wo;
        if (ext != nullptr) {
#pragma unroll
          for (int e = 0; e < cols / 4; ++e) {
            v[4 * e] = fmaf(we, xe[e].x, v[4 * e]);
            v[4 * e + 1] = fmaf(we, xe[e].y, v[4 * e + 1]);
            v[4 * e + 2] = fmaf(we, xe[e].z, v[4 * e + 2]);
            v[4 * e + 3] = fmaf(we, xe[e].w, v[4 * e + 3]);
          }
        }
        if constexpr (kB) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
            wds[e] = *reinterpret_cast<uint32_t*>(&h);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) wds[e] = __float_as_uint(v[e]);
        }
        if (ch + 1 < nch) fetch(ch + 1);  // the values are in wds: the next chunk's loads go now
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(buf + tc05::sw128(tid, q)) =
              make_uint4(wds[4 * q], wds[4 * q + 1], wds[4 * q + 2], wds[4 * q + 3]);
        if (map != nullptr) {
          tc05::fence_smem_to_async();  // the copy engine reads what these threads wrote
          // the previous chunk's store has read its buffer (written again next chunk)
          if (tid == 0) tc05::bulk_wait_read();
          EpGroup::sync();
          if (tid == 0) {
            tc05::tma_store_2d(map, tc05::smem_addr(buf), ch * cols, y0);
            tc05::bulk_commit();
          }
          continue;
        }
        EpGroup::sync();
        // all eight loads first: the stores could alias them for all the
        // compiler knows, so interleaving would wait out each load in turn
        uint4 vals[8];
#pragma unroll
        for (int i2 = 0; i2 < 8; ++i2) {
          const int x = i2 * kHeads + tid, row = x >> 3, q = x & 7;
          vals[i2] = *reinterpret_cast<const uint4*>(buf + tc05::sw128(row, q));
        }
#pragma unroll
        for (int i2 = 0; i2 < 8; ++i2) {
          const int x = i2 * kHeads + tid, row = x >> 3, q = x & 7;
          *reinterpret_cast<uint4*>(static_cast<char*>(dst0) + static_cast<int64_t>(row) * kDv * esz + ch * 128 + q * 16) =
              vals[i2];
        }
      }
    };
    auto store_rows = [&](void* dst0, bool to_bf16, float wo, float we, const float* ext) {
      if (to_bf16) store_rows_t(std::true_type{}, dst0, nullptr, 0, wo, we, ext);
      else store_rows_t(std::false_type{}, dst0, nullptr, 0, wo, we, ext);
    };
    // the same by TMA stores: rows y0 .. y0 + 127 of the map's tensor; the
    // staging buffers are free again on return
    auto store_rows_tma = [&](const CUtensorMap* map, int y0, bool to_bf16, float wo, float we, const float* ext) {
      if (to_bf16) store_rows_t(std::true_type{}, nullptr, map, y0, wo, we, ext);
      else store_rows_t(std::false_type{}, nullptr, map, y0, wo, we, ext);
      if (tid == 0) tc05::bulk_wait_read();
      EpGroup::sync();
    };
    // Exact merge of E partials of all 128 rows (the LSE merge of lse_merge):
    // entry e < E0 is workspace slot sl0 + e (rows contiguous), entry E0 (when
    // ext_o is given) the extra partial.  Each thread forms its row's weights;
    // then batches of R rows of every entry come into shared memory by bulk
    // copies (two batches in flight) and the weighted rows go to row r of
    // dst0 (a row every 512 elements, fp32 or bf16) with coalesced stores; the
    // row's LSE to put_lse.  The staging area is the merge scratch, or, for the
    // cluster's last item (no tile of it or after it still in flight), the
    // value stages and P buffers too: the copies' latency sets the pace, so the
    // batches should be large.  Returns false (nothing done) when the entries
    // do not fit.  All epilogue threads call.
    int merge_phase = 0;  // batches issued on B_MERGE so far (parity tracking)
    auto merge_bulk = [&](int E0, int64_t sl0, const float* ext_o, const float* ext_lse, void* dst0, bool to_bf16,
                          bool wide, auto put_lse) -> bool {
      const uint32_t area = wide ? 0u : OFF_SCR;
      const uint32_t area_bytes = wide ? OFF_ALPHA : static_cast<uint32_t>(kScrFloats) * 4u;
      const int E = E0 + (ext_o != nullptr ? 1 : 0);
      float* wt = reinterpret_cast<float*>(base + area);  // [E][128]
      const uint32_t wt_bytes = static_cast<uint32_t>((E * kHeads * 4 + 1023) & ~1023);
      if (wt_bytes >= area_bytes) return false;
      const uint32_t avail = area_bytes - wt_bytes;
      const int R = static_cast<int>(avail / 2 / (static_cast<uint32_t>(E) * kDv * 4));
      if (R < 1) return false;
      {
        // weights of row tid
        float mx = -INFINITY;
        for (int e = 0; e < E; ++e) {
          const float l = e < E0 ? __ldcg(a.ws_lse + (sl0 + e) * kHeads + tid) : __ldg(ext_lse + tid);
          wt[e * kHeads + tid] = l;
          mx = fmaxf(mx, l);
        }
        float sum = 0.f;
        for (int e = 0; e < E; ++e) {
          const float l = wt[e * kHeads + tid];
          sum += (mx == -INFINITY || l == -INFINITY) ? 0.f : expf(l - mx);
        }
        const float inv = sum == 0.f ? 0.f : 1.f / sum;
        for (int e = 0; e < E; ++e) {
          const float l = wt[e * kHeads + tid];
          wt[e * kHeads + tid] = (sum == 0.f || l == -INFINITY) ? 0.f : expf(l - mx) * inv;
        }
        put_lse(tid, sum == 0.f ? -INFINITY : mx + logf(sum));
      }
      uint8_t* buf0 = base + area + wt_bytes;
      const uint32_t buf_bytes = static_cast<uint32_t>(E) * R * kDv * 4;
      const int nbatch = (kHeads + R - 1) / R;
      auto issue = [&](int k) {
        const uint32_t mb = bar(B_MERGE + ((merge_phase + k) & 1));  // batch k's barrier (as waited below)
        const int r0 = k * R, nr = min(R, kHeads - r0);
        const uint32_t dst = tc05::smem_addr(buf0 + (k & 1) * buf_bytes);
        tc05::mbar_arrive_expect_tx(mb, static_cast<uint32_t>(E * nr) * kDv * 4);
        for (int e = 0; e < E; ++e) {
          const float* src = e < E0 ? a.ws_o + ((sl0 + e) * kHeads + r0) * kDv : ext_o + static_cast<int64_t>(r0) * kDv;
          asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                           dst + e * nr * kDv * 4),
                       "l"(src), "r"(nr * kDv * 4), "r"(mb)
                       : "memory");
        }
      };
      EpGroup::sync();  // weights in place; the staging area is free
      if (tid == 0) {
        // the partial rows were written by other CTAs' plain stores, published
        // by the ticket; the copies read them through the async proxy
        asm volatile("fence.proxy.async;\n" ::: "memory");
        issue(0);
        if (nbatch > 1) issue(1);
      }
      bool okm = true;
      for (int k = 0; k < nbatch; ++k) {
        const int ph = merge_phase + k;  // batch k is phase (ph >> 1) of barrier ph & 1
        okm = okm && wwait<false>(bar(B_MERGE + (ph & 1)), (ph >> 1) & 1, abort_flag);
        const int r0 = k * R, nr = min(R, kHeads - r0);
        const float4* bf = reinterpret_cast<const float4*>(buf0 + (k & 1) * buf_bytes);
        if (okm) {
          // thread tid owns column group c4 = tid of every row (kDv / 4 ==
          // kHeads).  Two rows at a time, their loads (four entries each)
          // all issued before any arithmetic and the stores after: the stores
          // could alias the loads for all the compiler knows, so it keeps this
          // order, and the 4 warps alone cannot hide shared-memory latency.
          static_assert(kDv / 4 == kHeads, "one column group a thread");
          const int c4 = tid;
          for (int rr0 = 0; rr0 < nr; rr0 += 2) {
            float4 acc[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int e0 = 0; e0 < E; e0 += 4) {
              float w[2][4];
              float4 v[2][4];
#pragma unroll
              for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  w[r][e] = 0.f;
                  if (rr0 + r < nr && e0 + e < E) {
                    w[r][e] = wt[(e0 + e) * kHeads + r0 + rr0 + r];
                    v[r][e] = bf[((e0 + e) * nr + rr0 + r) * (kDv / 4) + c4];
                  }
                }
#pragma unroll
              for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  if (w[r][e] == 0.f) continue;  // empty entries' rows never enter the sum
                  acc[r].x = fmaf(w[r][e], v[r][e].x, acc[r].x);
                  acc[r].y = fmaf(w[r][e], v[r][e].y, acc[r].y);
                  acc[r].z = fmaf(w[r][e], v[r][e].z, acc[r].z);
                  acc[r].w = fmaf(w[r][e], v[r][e].w, acc[r].w);
                }
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              if (rr0 + r >= nr) break;
              const int64_t oi = static_cast<int64_t>(r0 + rr0 + r) * kDv + c4 * 4;
              if (to_bf16) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(acc[r].x, acc[r].y),
                               hi = __floats2bfloat162_rn(acc[r].z, acc[r].w);
                *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(dst0) + oi) =
                    make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
              } else {
                *reinterpret_cast<float4*>(static_cast<float*>(dst0) + oi) = acc[r];
              }
            }
          }
        }
        EpGroup::sync();  // buffer k & 1 consumed
        if (tid == 0 && okm && k + 2 < nbatch) issue(k + 2);
      }
      merge_phase += nbatch;
      if (!okm) {
        ok = false;
        // nothing may land after the CTA exits: wait (bounded) for the batches in flight
        if (tid == 0)
          for (int k = max(0, nbatch - 2); k < nbatch; ++k) {
            const int ph = merge_phase - nbatch + k;
            tc05::mbar_wait(bar(B_MERGE + (ph & 1)), (ph >> 1) & 1, 1u << 20);
          }
      }
      return true;
    };
    int g = 0, fi = 0;
    if constexpr (kGroup) {
      // tokens without pages (padding tokens, rows of no keys): the extra
      // partial alone, or 0 / -inf; cluster c takes tokens c, c + C, ...
      for (int t = c; t < a.num_tokens; t += C) {
        if (g_pre[t + 1] != g_pre[t]) continue;
        if (tid == 0) {
          rec[2 * t] = 0;
          rec[2 * t + 1] = 1;
        }
        const int64_t row = static_cast<int64_t>(t) * kHeads + tid;
        const bool has_e = a.extra_lse != nullptr;
        const float le = has_e ? __ldg(a.extra_lse + row) : -INFINITY;
        for (int e = 0; e < kDv; e += 4) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (has_e && le != -INFINITY) v = __ldg(reinterpret_cast<const float4*>(a.extra_o + row * kDv + e));
          if (a.out_bf16) {
            __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + row * kDv + e) =
                make_uint2(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1));
          } else {
            *reinterpret_cast<float4*>(static_cast<float*>(a.out) + row * kDv + e) = v;
          }
        }
        if (a.lse_out != nullptr) a.lse_out[row] = le;
      }
    }
    for (int k = 0; ok; ++k) {
      MlaItem it;
      if (!item(k, it)) break;
      if (it.t < 0) continue;
      const int nt = ntiles(it);
      const int64_t orow = (static_cast<int64_t>(it.p) * a.num_tokens + it.t) * a.num_q_heads + tid;
      if (kGroup && nt == 0) continue;  // the zero pass wrote it
      if (nt == 0) {  // empty stripe (or a token of no row): 0 / -inf
        float4* d4 = reinterpret_cast<float4*>(a.o_part + orow * kDv);
        for (int e = 0; e < kDv / 4; ++e) d4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        a.lse_part[lse_slot(a, it.p, it.t, tid)] = -INFINITY;
        if (a.fused) pair_finish<kMergeUnroll, EpGroup>(a, it.t, 0, kHeads, kDv, scratch, kScrFloats);
        continue;
      }
      const int pb0 = __ldg(a.page_indptr + it.b), npg = __ldg(a.page_indptr + it.b + 1) - pb0;
      MaskWords next_words = mask_words(it, 0, pb0, npg);
      for (int j = 0; j < nt; ++j, ++g) {
        const int pbuf = g % kTileRing, vs = g % kVStages;
        const MaskWords words = next_words;
        if (j + 1 < nt) next_words = mask_words(it, j + 1, pb0, npg);
        // P and the rescale factors arrive by bulk copies from CTA 0 (bytes counted)
        const int pq = g % kPBufs;
        if (tid == 0) tc05::mbar_arrive_expect_tx(bar(B_PFULL + pq), kPBuf + kHeads * 4);
        ok = wwait<true>(bar(B_PFULL + pq), (g / kPBufs) & 1, abort_flag);
        if (!ok) break;
        const uint64_t vmask = tile_mask_from<kGroup>(a, it, j, words, lane);
        tc05::fence_smem_to_async();  // the tensor core reads P next
        const float alpha = alpha_s[pq * kHeads + tid];
        if (kTma && vmask != ~0ull) {
          // value rows of keys without data (past the item, rejected pages, runs
          // not copied): zero, once the tile's units landed (they sit together,
          // stage vs of the ring); the MMA warp waits for them by itself.  This
          // warp may be ahead of the MMAs: the P V two tiles back first (its
          // units then landed), so that the parity waits below are unambiguous.
          if (g >= kVStages)
            ok = wwait<false>(bar(B_PVDONE + (g - kVStages) % kTileRing), ((g - kVStages) / kTileRing) & 1,
                              abort_flag);
          for (int h = 0; h < kVUnits && ok; ++h) {
            const int n = g * kVUnits + h;
            ok = wwait<false>(bar(B_VFULL + n % kVRing), (n / kVRing) & 1, abort_flag);
          }
          if (!ok) break;
          uint8_t* st = base + vs * kVStage;
          for (int idx = tid; idx < kTile * kVB * 8; idx += 128) {
            const int key = idx / (kVB * 8);
            if ((vmask >> key) & 1ull) continue;
            const int ch = idx - key * (kVB * 8);
            *reinterpret_cast<uint4*>(st + (ch >> 3) * kBlk + tc05::sw128(key, ch & 7)) = make_uint4(0u, 0u, 0u, 0u);
          }
          tc05::fence_smem_to_async();
        }
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O (all 512 columns) of the rows whose max rose, after the previous P V
          ok = wwait<false>(bar(B_PVDONE + (g - 1) % kTileRing), ((g - 1) / kTileRing) & 1, abort_flag);
          if (!ok) break;
          tc05::fence_after_sync();
#pragma unroll 1
          for (int col = 0; col < kDv; col += 32) {
            float v[16], w[16];
            tc05::ld_x16(my_lane + col, v);
            tc05::ld_x16(my_lane + col + 16, w);
            tc05::ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              v[e] *= alpha;
              w[e] *= alpha;
            }
            tc05::st_x16(my_lane + col, v);
            tc05::st_x16(my_lane + col + 16, w);
          }
          tc05::st_wait();
        }
        tc05::fence_before_sync();
        __syncwarp();
        if (lane == 0) arrive_local(bar(B_READY + pbuf));
      }
      if (!ok) break;
      // ---- epilogue of the item: O / sum -> o_part (whole stripe) or the piece's workspace slot
      if (tid == 0) tc05::mbar_arrive_expect_tx(bar(B_FINFULL), kHeads * 8);
      ok = wwait<true>(bar(B_FINFULL), fi & 1, abort_flag);
      if (!ok) break;
      const float2 f = fin_s[tid];
      __syncwarp();
      if (lane == 0) tc05::mbar_arrive_remote(r_finempty);
      ok = wwait<false>(bar(B_PVDONE + (g - 1) % kTileRing), ((g - 1) / kTileRing) & 1, abort_flag);
      if (!ok) break;
      tc05::fence_after_sync();
      ++fi;
      if (kGroup && it.slot < 0) {
        // a whole token: its final output, merged with the extra partial if given
        const int64_t row = static_cast<int64_t>(it.t) * kHeads + tid;
        float wo = f.x, we = 0.f, lse = f.y;
        if (a.extra_lse != nullptr) {
          const float le = __ldg(a.extra_lse + row);
          const float M = fmaxf(f.y, le);
          const float w1 = f.y == -INFINITY ? 0.f : expf(f.y - M), w2 = le == -INFINITY ? 0.f : expf(le - M);
          const float sum = w1 + w2;
          wo = sum > 0.f ? f.x * (w1 / sum) : 0.f;
          we = sum > 0.f ? w2 / sum : 0.f;
          lse = sum > 0.f ? M + logf(sum) : -INFINITY;
        }
        store_rows_tma(&tmap_out, it.t * kHeads, a.out_bf16 != 0, wo, we,
                       a.extra_lse != nullptr ? a.extra_o + static_cast<int64_t>(it.t) * kHeads * kDv : nullptr);
        tc05::fence_before_sync();
        if (a.lse_out != nullptr) a.lse_out[row] = lse;
        if (tid == 0) {
          rec[2 * it.t] = 0;
          rec[2 * it.t + 1] = 1;
        }
        continue;
      }
      if (kGroup) {
        // a piece of a cut token: its normalised partial to its workspace
        // slot; the merge kernel that follows combines the pieces (and the
        // extra partial) into the token's final output
        store_rows_tma(&tmap_ws, it.slot * kHeads, false, f.x, 0.f, nullptr);
        tc05::fence_before_sync();
        a.ws_lse[static_cast<int64_t>(it.slot) * kHeads + tid] = f.y;
        if (tid == 0) {
          rec[2 * it.t] = it.slot_base;
          rec[2 * it.t + 1] = it.npieces;
        }
        continue;
      }
      float* dst0 = it.slot < 0 ? a.o_part + (orow - tid) * kDv : a.ws_o + static_cast<int64_t>(it.slot) * kHeads * kDv;
      store_rows(dst0, false, f.x, 0.f, nullptr);
      tc05::fence_before_sync();
      if (it.slot < 0) {
        a.lse_part[lse_slot(a, it.p, it.t, tid)] = f.y;
      } else {
        a.ws_lse[static_cast<int64_t>(it.slot) * kHeads + tid] = f.y;
        // the last piece of the stripe to finish merges the pieces into o_part
        const int64_t s_idx = static_cast<int64_t>(it.t) * a.P + it.p;
        if (!take_ticket<EpGroup>(a.ws_cnt + s_idx, it.npieces)) continue;
        const int64_t sl0 = it.slot_base;
        const int64_t prow0 = (static_cast<int64_t>(it.p) * a.num_tokens + it.t) * a.num_q_heads;
        MlaItem nx;
        const bool wide = !item(k + 1, nx);
        if (!merge_bulk(it.npieces, sl0, nullptr, nullptr, a.o_part + prow0 * kDv, false, wide,
                        [&](int r, float lv) { a.lse_part[lse_slot(a, it.p, it.t, r)] = lv; }))
        merge_rows<kMergeUnroll, EpGroup>(
            kHeads, it.npieces, kDv, [&](int r, int e) { return __ldcg(a.ws_lse + (sl0 + e) * kHeads + r); },
            [&](int r, int e) { return a.ws_o + ((sl0 + e) * kHeads + r) * kDv; },
            [&](int r, int d, float4 v) {
              const int64_t o = (static_cast<int64_t>(it.p) * a.num_tokens + it.t) * a.num_q_heads + r;
              *reinterpret_cast<float4*>(a.o_part + o * kDv + d) = v;
            },
            [&](int r, float lv) { a.lse_part[lse_slot(a, it.p, it.t, r)] = lv; }, scratch, kScrFloats);
        if (tid == 0) a.ws_cnt[s_idx] = 0;
      }
      if (a.fused) pair_finish<kMergeUnroll, EpGroup>(a, it.t, 0, kHeads, kDv, scratch, kScrFloats);
    }
    if (tid == 0) tc05::bulk_wait_all();  // the TMA stores are done before the CTA exits
    if (!ok) raise_abort();
  }

  // ---- teardown: every MMA done, tensor memory freed, and neither CTA exits
  // while the other may still write into it
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  if (warp == 0) tc05::tmem_dealloc(tbase, 512);
  tc05::cluster_sync();
}

// Grouped plans: the exact merge of the pieces of each cut token (and the
// extra partial, when given) into its final output and LSE.  Block (t, rb)
// takes rows 4 rb .. 4 rb + 3 of token t, a warp a row: lane e holds the
// weight of piece e (32 at a time), lane l accumulates 16-byte columns
// l + 32 i of the row, with the loads of four pieces in flight.  The
// token's record (slot of its first piece, pieces) comes from the partial
// kernel, which this grid follows on the stream (it may start early and
// waits here for that grid to finish).
constexpr int kMergeRows = 4;
__global__ void __launch_bounds__(128) mla_merge_pieces_kernel(const PartialArgs a, int ws_slots) {
  pdl_wait();
  const int t = blockIdx.x, lane = threadIdx.x & 31;
  const int r = blockIdx.y * kMergeRows + (threadIdx.x >> 5);
  const int32_t* rec = a.ws_cnt + static_cast<int64_t>(a.num_tokens) * a.P;
  const int npieces = __ldcg(rec + 2 * t + 1);
  const int64_t sl0 = __ldcg(rec + 2 * t), trow = static_cast<int64_t>(t) * kHeads + r;
  // written whole by the partial kernel; or a record that kernel did not
  // write (it gave up on a wait): never read outside the slots
  if (npieces <= 1 || sl0 < 0 || sl0 + npieces > ws_slots) return;
  const bool has_e = a.extra_lse != nullptr;
  const int E = npieces + (has_e ? 1 : 0);
  auto lse_of = [&](int e) {
    return e < npieces ? __ldcg(a.ws_lse + (sl0 + e) * kHeads + r) : __ldg(a.extra_lse + trow);
  };
  auto row_of = [&](int e) {
    return reinterpret_cast<const float4*>(e < npieces ? a.ws_o + ((sl0 + e) * kHeads + r) * kDv
                                                       : a.extra_o + trow * kDv);
  };
  float mx = -INFINITY;
  for (int e = lane; e < E; e += 32) mx = fmaxf(mx, lse_of(e));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  for (int e = lane; e < E; e += 32) {
    const float l = lse_of(e);
    sum += (mx == -INFINITY || l == -INFINITY) ? 0.f : expf(l - mx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < E; c0 += 32) {
    // lane e: the weight of piece c0 + e (0 for an empty one, whose row is never read)
    float w_l = 0.f;
    if (c0 + lane < E) {
      const float l = lse_of(c0 + lane);
      w_l = (sum > 0.f && l != -INFINITY) ? expf(l - mx) * inv : 0.f;
    }
    const int ne = min(32, E - c0);
    for (int e0 = 0; e0 < ne; e0 += 4) {
      float w[4];
      float4 v[4][4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        w[b] = __shfl_sync(0xffffffffu, w_l, (e0 + b) & 31);
        if (e0 + b >= ne) w[b] = 0.f;
        if (w[b] != 0.f) {
          const float4* src = row_of(c0 + e0 + b);
#pragma unroll
          for (int i = 0; i < 4; ++i) v[b][i] = __ldcg(src + lane + 32 * i);
        }
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (w[b] == 0.f) continue;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i].x = fmaf(w[b], v[b][i].x, acc[i].x);
          acc[i].y = fmaf(w[b], v[b][i].y, acc[i].y);
          acc[i].z = fmaf(w[b], v[b][i].z, acc[i].z);
          acc[i].w = fmaf(w[b], v[b][i].w, acc[i].w);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t oi = trow * kDv + (lane + 32 * i) * 4;
    if (a.out_bf16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x, acc[i].y), hi = __floats2bfloat162_rn(acc[i].z, acc[i].w);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + oi) =
          make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(a.out) + oi) = acc[i];
    }
  }
  if (lane == 0 && a.lse_out != nullptr) a.lse_out[trow] = sum > 0.f ? mx + logf(sum) : -INFINITY;
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 2-D bf16 view [rows][576] with 1152-byte rows, 64-column boxes of `box_rows` rows, 128-byte swizzle.
bool encode_rows(CUtensorMap* map, const void* ptr, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || rows == 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDqk * 2)};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 view [P][num_pages * ps_l][576] of an MLA pool: boxes of 64
// values x ps_l rows x P partners (a logical page of every partner), 128-byte swizzle.
bool encode_pages(CUtensorMap* map, const void* ptr, int P, uint64_t rows_per_partner, uint32_t ps_l, uint32_t nblk) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || rows_per_partner == 0) return false;
  // dims: 64 values of a column block, rows of a partner's pool, partners,
  // column blocks (128 bytes apart); a box is nblk blocks of a logical page
  const cuuint64_t dims[4] = {64u, rows_per_partner, static_cast<cuuint64_t>(P), static_cast<cuuint64_t>(kKB)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kDqk * 2), rows_per_partner * kDqk * 2, 128u};
  const cuuint32_t box[4] = {64u, ps_l, static_cast<cuuint32_t>(P), nblk};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows of 512 values (fp32, or bf16) written as boxes of 128 rows x 128
// bytes (the epilogue's staged chunks, 128-byte swizzle).
bool encode_out(CUtensorMap* map, void* ptr, uint64_t rows, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr || rows == 0 || ptr == nullptr) return false;
  const uint32_t esz = bf16 ? 2u : 4u;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDv), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDv) * esz};
  const cuuint32_t box[2] = {128u / esz, 128u};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// SMs of the current device (0 if unknown).
int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

}  // namespace

int mla_max_clusters() {
  const int sms = device_sms();
  return sms >= 2 ? sms / 2 : 76;
}

int mla_ws_slots(int P, int interleave, int num_tokens, int max_kv_len, int grouped) {
  const int64_t by_clusters = 2LL * mla_max_clusters();
  // Pieces of cut stripes: a stripe of n tiles is cut only when n exceeds the
  // chunk max(total / C, 16 tiles), into at most 2 n / chunk pieces, so all
  // pieces together number at most 2 C; and at most ceil(n / 16) per stripe.
  int64_t n = 0;
  const int max_stripe_tiles = (max_stripe_len(max_kv_len, P, interleave) + kTile - 1) / kTile;
  if (max_stripe_tiles > kMinChunkTiles) {
    const int64_t per = (max_stripe_tiles + kMinChunkTiles - 1) / kMinChunkTiles;
    const int64_t by_stripes = static_cast<int64_t>(num_tokens) * P * per;
    n = by_stripes < by_clusters ? by_stripes : by_clusters;
  }
  if (grouped) {
    // Pieces of cut tokens: Ce - 1 range boundaries, each cutting at most one
    // token, so at most 2 (Ce - 1) <= 2 C pieces; and Ce <= W / 16, W <= T x
    // the tiles of the longest row.  (The per-stripe bound stays covered: the
    // kernel falls back to per-partner tiles if it cannot describe the pool.)
    const int64_t max_tiles = (static_cast<int64_t>(max_kv_len) + kTile - 1) / kTile;
    const int64_t by_tiles = 2 * ((static_cast<int64_t>(num_tokens) * max_tiles + kMinChunkTiles - 1) / kMinChunkTiles);
    const int64_t g = by_tiles < by_clusters ? by_tiles : by_clusters;
    if (g >= 2 && g > n) n = g;
  }
  return static_cast<int>(n);
}

int launch_mla_partial(const PartialArgs& a, cudaStream_t s, cudaError_t* err) {
  if (a.num_q_heads != kHeads || a.head_dim != kDqk || a.head_dim_v != kDv || a.num_kv_heads != 1)
    return CPATTN_ERR_UNSUPPORTED_SHAPE;
  const int64_t pool_rows = static_cast<int64_t>(a.P) * a.num_pages * a.ps_l;
  if (pool_rows >= (int64_t{1} << 31)) return CPATTN_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap map, map_v, map_out, map_ws;
  std::memset(&map, 0, sizeof(map));
  std::memset(&map_v, 0, sizeof(map_v));
  std::memset(&map_out, 0, sizeof(map_out));
  std::memset(&map_ws, 0, sizeof(map_ws));
  // fused calls over logical pages of 64 slots: tiles are whole logical
  // pages, one 4-D box per ring unit (the per-partner partials are merged
  // inside the online softmax)
  const uint64_t rows_pp = static_cast<uint64_t>(a.num_pages) * a.ps_l;
  // (outputs of whole tokens and the pieces of cut ones leave by TMA stores)
  const int ws_slots = mla_ws_slots(a.P, a.interleave, a.num_tokens, a.max_kv_len, 1);
  const bool group = a.fused && a.page_size == kTile && a.num_tokens <= kGroupMaxTokens &&
                     encode_pages(&map, a.pool_k, a.P, rows_pp, a.ps_l, kUBlk) &&
                     encode_pages(&map_v, a.pool_k, a.P, rows_pp, a.ps_l, kVUB) &&
                     encode_out(&map_out, a.out, static_cast<uint64_t>(a.num_tokens) * kHeads, a.out_bf16 != 0) &&
                     (ws_slots == 0 || encode_out(&map_ws, a.ws_o, static_cast<uint64_t>(ws_slots) * kHeads, false));
  // per-partner tiles: TMA when every 64-key tile is a whole number of page
  // runs of >= 8 rows (so each box lands on a 1024-byte boundary of the
  // 128-byte swizzle pattern), or lies inside one page run
  int box_rows = 0;
  if (a.ps_l >= 8 && a.ps_l <= kTile && kTile % a.ps_l == 0) box_rows = a.ps_l;
  else if (a.ps_l % kTile == 0) box_rows = kTile;
  const bool tma = group || (box_rows > 0 && encode_rows(&map, a.pool_k, static_cast<uint64_t>(pool_rows), box_rows));
  auto kern = group ? mla_pair_kernel<true, true> : (tma ? mla_pair_kernel<true, false> : mla_pair_kernel<false, false>);
  const int variant = group ? 2 : (tma ? 1 : 0);
  static std::atomic<int> smem_set[3][64];
  *err = ensure_smem(kern, kSmemBytes, smem_set[variant]);
  if (*err != cudaSuccess) return CPATTN_ERR_CUDA;
  // persistent grid: as many clusters as fit (one CTA per SM)
  static std::atomic<int> fit[3][64];
  int dev = 0;
  cudaGetDevice(&dev);
  int C = fit[variant][dev & 63].load(std::memory_order_relaxed);
  if (C <= 0) {
    C = mla_max_clusters();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * C, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0 && n < C) C = n;
    cudaGetLastError();  // a failed query leaves no error behind
    fit[variant][dev & 63].store(C, std::memory_order_relaxed);
  }
  *err = launch_pdl(kern, dim3(2 * C, 1, 1), dim3(kThreads, 1, 1), kSmemBytes, s, a, map, map_v, map_out, map_ws,
                    box_rows);
  if (*err != cudaSuccess) return CPATTN_ERR_CUDA;
  if (group && a.num_tokens > 0) {
    // the cut tokens' merge, launched to overlap the partial kernel's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.num_tokens), kHeads / kMergeRows, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    *err = cudaLaunchKernelEx(&cfg, mla_merge_pieces_kernel, a, ws_slots);
    if (*err != cudaSuccess) return CPATTN_ERR_CUDA;
  }
  return CPATTN_OK;
}

}  // namespace cpattn
