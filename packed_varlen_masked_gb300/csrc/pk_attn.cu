// Packed mixed-mask variable-length attention forward for GB300 (sm_103a).
//
// What it computes is the operation of "[RFC]: HunyuanImage 3.0 deployment"
// (Proposed Change, P0 "Packed Attention for Multi-Request Batching" and its
// "Attention mask challenge" bullet): attention over sequences packed back to
// back by cu_seqlens, each with the generalized causal mask (text causal,
// image tokens also seeing their whole own segment), with grouped-query
// heads.  The host planner turns the mask into a per-token key limit and a
// list of 128-row query tiles, each visiting a prefix of 128-key tiles that
// are either fully visible (no mask math) or partial (per-element compare).
// Queries and keys are bf16, or FP8 E4M3 (F8: S = Q K^T on kind::f8f6f4,
// one dequantisation scale each folded into the softmax scale).  Values and
// P enter the P V product in fp16 (the values converted from bf16 by a
// kernel before the launch), or, with V8, both in E4M3 (the values
// transposed by a kernel before the launch).  The output is bf16.
//
// Kernel organisation (one persistent CTA per SM, 12 warps).  The CTA runs
// its work items' query heads ("units") one after another; a unit is a
// 128-row query tile streaming the key/value tiles of its sequence.
//   warp 0      TMA producer of the query tiles (double buffered) and of a
//               ring of key tiles; warp 2: TMA producer of a ring of value
//               tiles (128-byte swizzled boxes, one per 64 columns of the
//               head dimension; ring depths in Cfg).
//   warp 1      allocates the 512 TMEM columns; one thread issues every
//               S(t) = Q K(t)^T (both operands K-major in shared memory).
//   warp 3      one thread issues every O += P(t) V(t) (P read from TMEM, V
//               MN-major in shared memory).  A tcgen05.mma costs its issuing
//               thread a large part of the product's own time, and two
//               issuers in different warps work concurrently.
//   warps 4-7   softmax: thread r owns row r of S, P and O in TMEM.  Online
//               softmax in base 2 with a lazily moved running maximum, P
//               written as fp16 pairs; at the end of a unit it hands the
//               row's (m, l) to the epilogue and goes on to the next unit.
//   warps 8-11  epilogue: after a unit's last P V, moves O out of TMEM
//               (freeing it for the next unit), writes O / l as bf16 (whole
//               128-byte row segments per warp store) and the natural-log
//               LSE.
// Registers: the one-thread roles give theirs up (setmaxnreg) to the
// softmax, whose exponential loop keeps a whole 128-column row of scores
// and its 64 fp16 pairs live, and to the epilogue, which holds a row of O.
// PAIR (opt-in, bf16 with D = 128): a cluster of two CTAs on an SM pair
// computes two query tiles as M = 256 products (tcgen05 cta_group::2); the
// rank-0 CTA's producers and issuers serve both, each CTA holding half of
// every key and value tile, and both CTAs run their rows' softmax and
// epilogue.
// SHARE (the default where every work item has two query heads):
// a cluster of two CTAs on neighbouring SMs runs each item with one query
// head per CTA.  Both stream the same key/value tiles through rings of the
// same shape; each CTA's producers copy half of every tile (one 64-column
// box, or for one-box tiles 64 of the rows) into the shared memory
// of both CTAs (TMA multicast), and a ring stage is refilled only after both
// CTAs' products have read it (each MMA issuer's commit arrives on the
// stage's empty barrier in both CTAs).  Everything else is the one-CTA
// kernel, per CTA.
// TMEM columns: S double buffer [0,256), P double buffer [256,384), O
// [384,384+D).  Because S(t) and P(t) live in different columns and both are
// double buffered, the S issuer computes S(t+2) as soon as the softmax has
// read S(t), and the tensor pipe runs S(t+2) and P(t-1)V(t-1) while the
// softmax works on tile t.
//
// Every mbarrier wait is bounded in time; on expiry the kernel records
// PK_ERR_TIMEOUT, raises a CTA-local abort flag so the other roles stop, lets
// in-flight copies and MMAs land, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "pk_internal.h"
#include "attn_common.cuh"
#include "sync.cuh"
#include "tmem_ops.cuh"

namespace pk {
namespace dev {

constexpr int kThreads = 384;
// Registers per thread after setmaxnreg: warps 0-3, 4-7 and 8-11.  A CTA is
// launched with kThreads x kRegsLaunch registers (the most __launch_bounds__
// allows at one CTA per SM); the three shares must fit in that, or the
// increases would wait forever.  The host checks the compiled count before
// the first launch.
constexpr int kRegsMma = 64, kRegsSoftmax = 240, kRegsEpi = 200;
constexpr int kRegsLaunch = 65536 / kThreads / 8 * 8;  // 168
static_assert(128 * (kRegsMma + kRegsSoftmax + kRegsEpi) <= kThreads * kRegsLaunch,
              "register split exceeds the CTA's allocation");
constexpr uint32_t kTmemCols = 512;
// Lanes that write one output row together in the epilogue (16-byte chunks).
constexpr int kStoreGroup = 8;
// F8: queries and keys are FP8 E4M3 (one byte per element), values bf16.
// PAIR: the SM-pair kernel (bf16, D = 128): a cluster of two CTAs computes
// M = 256 products; each CTA holds its own 128 query rows, half of every key
// tile (64 rows) and half of every value tile (64 of the D columns).
// SHARE: head-pair clusters; each CTA copies half of every key and value
// tile into both CTAs (see the file comment).
template <int D, bool F8 = false, bool V8 = false, bool PAIR = false, bool SHARE = false>
struct Cfg {
  // Query/key tiles: rows in boxes of 128-byte rows (64 bf16 or 128 FP8
  // elements); value tiles: 128 rows of D fp16 in 64-column boxes.
  static constexpr int kQKElemsPerBox = F8 ? 128 : 64;
  static constexpr int kQKBoxes = D / kQKElemsPerBox;
  static constexpr int kQKTileBytes = 128 * D * (F8 ? 1 : 2);  // a query tile
  static constexpr int kKRows = PAIR ? 64 : 128;               // key rows per CTA and tile
  static constexpr int kKBoxBytes = kKRows * 128;
  static constexpr int kKTileBytes = kKRows * D * (F8 ? 1 : 2);
  // V8: E4M3 values, transposed (one 128-byte row of keys per head-dimension
  // index), one box per tile; PAIR: one 64-column box (this CTA's half);
  // else fp16 values in 64-column boxes.
  static constexpr int kVBoxes = (V8 || PAIR) ? 1 : D / 64;
  static constexpr int kVTileBytes = PAIR ? 128 * 64 * 2 : 128 * D * (V8 ? 1 : 2);
  // Rings: two query tiles (the next unit's loads during this one), and key
  // and value tiles.  Shared memory stays above half an SM, so exactly one
  // CTA (and one 512-column TMEM allocation) lives on each SM.  In head-pair
  // clusters a stage waits for the slower CTA of the two: there bf16 at
  // D = 128 takes two key and three value stages (0.5 to 1.5 % faster than
  // three and two) and FP8 queries/keys five key stages of 16 KB and three
  // value stages (0.3 to 1 % faster than four and three); D = 64 keeps the
  // one-CTA kernel's four and four.
  static constexpr int kKStages =
      SHARE ? (D == 64 ? 4 : (F8 ? 5 : 2)) : PAIR ? 7 : (F8 ? 4 : (D == 128 ? 3 : 4));
  static constexpr int kVStages =
      SHARE ? (D == 64 ? 4 : 3) : PAIR ? 3 : (V8 ? 4 : (F8 ? 3 : (D == 128 ? 2 : 4)));
  // TMEM columns: S double buffer, P double buffer (16-bit pairs), O.
  static constexpr uint32_t kColS0 = 0;    // S(t) in [128*(t%2), +128)
  static constexpr uint32_t kColP0 = 256;  // P(t) in [256 + 64*(t%2), +64)
  static constexpr uint32_t kColO = 384;   // O in [384, 384 + D)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kQKTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kKTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * kVTileBytes;
  static_assert(!F8 || D == 128, "FP8 queries/keys need head_dim 128");
  static_assert(!V8 || F8, "E4M3 values come with E4M3 queries and keys");
  static_assert(!PAIR || (D == 128 && !F8), "the SM-pair kernel is bf16 with head_dim 128");
  static_assert(!SHARE || (!V8 && !PAIR), "head-pair clusters: 16-bit values, one CTA per head");
  // SHARE: rows per key and value copy.  Two-box tiles (bf16 keys and the
  // values at D = 128) split by boxes, each CTA copying one whole box;
  // one-box tiles (FP8 keys, D = 64) split by rows, 64 each.
  static constexpr int kShareKRows = kQKBoxes == 1 ? 64 : 128;
  static constexpr int kShareVRows = kVBoxes == 1 ? 64 : 128;
  // Arrivals of the softmax (S buffer free, P ready) and the epilogue (O
  // free): one per thread of the CTA's warpgroup, or, in the pair kernel,
  // of both CTAs' warpgroups (on the rank-0 CTA's barrier).
  static constexpr uint32_t kGroupArrivals = PAIR ? 256 : 128;
  // barrier indices
  static constexpr int kQFull = 0, kQEmpty = 2;  // [2] each
  static constexpr int kKFull = 4, kKEmpty = kKFull + kKStages;
  static constexpr int kVFull = kKEmpty + kKStages, kVEmpty = kVFull + kVStages;
  static constexpr int kSFull = kVEmpty + kVStages;  // [2]
  static constexpr int kSFree = kSFull + 2;          // [2]
  static constexpr int kPReady = kSFree + 2;         // [2]
  static constexpr int kPvDone = kPReady + 2;        // [2]
  static constexpr int kOFree = kPvDone + 2;
  static constexpr int kMmaDone = kOFree + 1;  // [2]: one per MMA issuer
  static constexpr int kLmFull = kMmaDone + 2;   // a unit's row (m, l) handed over
  static constexpr int kLmFree = kLmFull + 1;    // ... and taken by the epilogue
  static constexpr int kNumBars = kLmFree + 1;
  static constexpr int kOffLm = (kOffBar + kNumBars * 8 + 15) / 16 * 16;  // float2 [128]
  static constexpr int kOffMisc = kOffLm + 128 * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kSmemBytes > 114 * 1024, "one CTA per SM");
  static_assert(kColO + D <= 512, "TMEM budget");
};

// A unit of work is one query head of a work item: a 128-row query tile that
// streams the key/value tiles of its sequence.  A CTA on its own runs the
// heads of each of its items back to back, so the second head's keys and
// values come from L2.  Every role walks the same unit sequence.
// In the pair kernel the items come in (rank 0, rank 1) pairs and each CTA
// walks its own item of every pair (stride 2).  In a head-pair cluster each
// CTA runs one query head of every item (fixed slot: its cluster rank).
struct UnitIter {
  const pk_work_item* items;
  int it, end, slot, stride, rank;
  bool fixed;
  pk_work_item w;
  __device__ UnitIter(const pk_work_item* items_, int beg, int end_, int stride_ = 1,
                      int rank_ = 0, int fixed_slot = -1)
      : items(items_), it(beg), end(end_), slot(fixed_slot < 0 ? 0 : fixed_slot),
        stride(stride_), rank(rank_), fixed(fixed_slot >= 0) {
    if (it < end) w = items[it * stride + rank];
  }
  __device__ bool valid() const { return it < end; }
  __device__ int head() const { return slot ? w.hq1 : w.hq0; }
  __device__ void next() {
    if (!fixed) {
      if (slot == 0 && w.hq1 >= 0) {
        slot = 1;
        return;
      }
      slot = 0;
    }
    if (++it < end) w = items[it * stride + rank];
  }
};

// The unit iterator of a role: the pair kernel's stride and rank, or a
// head-pair cluster's fixed slot.
template <bool PAIR, bool SHARE>
__device__ __forceinline__ UnitIter role_units(const KernelParams& p, int beg, int end,
                                               uint32_t pair_rank) {
  return UnitIter(p.items, beg, end, PAIR ? 2 : 1, PAIR ? (int)pair_rank : 0,
                  SHARE ? (int)cluster_rank() : -1);
}

// Q/K producer (one thread): per unit its query tile (double buffered), then
// the ring of key tiles.  Keys and values are re-read by the other query
// heads of the group and by neighbouring query tiles, so they are kept in L2
// (evict-last); a query tile is read once (evict-first).
template <int D, bool F8, bool V8, bool PAIR, bool SHARE>
__device__ void producer_qk_role(const KernelParams& p, const CUtensorMap* tm_q,
                                 const CUtensorMap* tm_k, uint32_t sbase, int beg, int end,
                                 const WaitCtl& wc) {
  using C = Cfg<D, F8, V8, PAIR, SHARE>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * (uint32_t)i; };
  const uint64_t keep = l2_policy_evict_last(), stream = l2_policy_evict_first();
  uint32_t g = 0, u = 0, k_armed = 0, q_armed = 0;
  bool ok = true;
  constexpr int kCtas = PAIR ? 2 : 1;  // pair: this (rank-0) thread loads both CTAs' tiles
  const int srank = SHARE ? (int)cluster_rank() : 0;  // the key box or rows this CTA copies
  for (UnitIter ui = role_units<PAIR, SHARE>(p, beg, end, 0); ui.valid() && ok; ui.next(), ++u) {
    const pk_work_item& w = ui.w;
    const uint32_t qb = u & 1u;
    if (!(ok = mbar_wait(bar(C::kQEmpty + qb), ((u >> 1) & 1u) ^ 1u, wc))) break;
    mbar_arrive_expect_tx(bar(C::kQFull + qb), kCtas * C::kQKTileBytes);
    ++q_armed;
    if constexpr (PAIR) {
      // rank r's query rows into rank r's buffer (a partner without rows
      // reloads the leader's), completing on this CTA's barrier
      const int q1 = p.items[ui.it * 2 + 1].q_start;
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int h = 0; h < C::kQKBoxes; ++h)
          tma_load_3d_pair(map_to_rank(sbase + C::kOffQ + qb * C::kQKTileBytes + h * kBoxBytes, r),
                           tm_q, bar(C::kQFull + qb), h * C::kQKElemsPerBox, ui.head(),
                           r ? q1 : w.q_start, stream);
    } else {
#pragma unroll
      for (int h = 0; h < C::kQKBoxes; ++h)
        tma_load_3d_hint(sbase + C::kOffQ + qb * C::kQKTileBytes + h * kBoxBytes, tm_q,
                         bar(C::kQFull + qb), h * C::kQKElemsPerBox, ui.head(), w.q_start, stream);
    }
    for (int j = 0; j < w.n_kt; ++j, ++g) {
      const uint32_t st = g % C::kKStages, ph = (g / C::kKStages) & 1u;
      if (!(ok = mbar_wait(bar(C::kKEmpty + st), ph ^ 1u, wc))) break;
      mbar_arrive_expect_tx(bar(C::kKFull + st), kCtas * C::kKTileBytes);
      ++k_armed;
      if constexpr (SHARE) {  // this CTA's half of the tile, into both CTAs
        if constexpr (C::kQKBoxes == 2)
          tma_load_3d_mc(sbase + C::kOffK + st * C::kKTileBytes + srank * C::kKBoxBytes, tm_k,
                         bar(C::kKFull + st), srank * C::kQKElemsPerBox, w.hkv,
                         key_tile_row(p, w, j), (uint16_t)3, keep);
        else
          tma_load_3d_mc(sbase + C::kOffK + st * C::kKTileBytes + srank * 64 * 128, tm_k,
                         bar(C::kKFull + st), 0, w.hkv, key_tile_row(p, w, j) + srank * 64,
                         (uint16_t)3, keep);
      } else if constexpr (PAIR) {  // key rows [64 r, 64 r + 64) of the tile to rank r
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int h = 0; h < C::kQKBoxes; ++h)
            tma_load_3d_pair(
                map_to_rank(sbase + C::kOffK + st * C::kKTileBytes + h * C::kKBoxBytes, r), tm_k,
                bar(C::kKFull + st), h * C::kQKElemsPerBox, w.hkv,
                key_tile_row(p, w, j) + r * C::kKRows, keep);
      } else {
#pragma unroll
        for (int h = 0; h < C::kQKBoxes; ++h)
          tma_load_3d_hint(sbase + C::kOffK + st * C::kKTileBytes + h * C::kKBoxBytes, tm_k,
                           bar(C::kKFull + st), h * C::kQKElemsPerBox, w.hkv,
                           key_tile_row(p, w, j), keep);
      }
    }
  }
  // Every copy issued must land before the CTA may exit.  After a normal run
  // the consumers have waited for them all and these waits pass at once;
  // after an abort (this thread's or a consumer's) they may be in flight.
  // The last kKStages armings of the ring (and the last two of Q) are the
  // only ones that can be open, each the most recent arming of its stage.
  // Head-pair cluster: a stage's phase completes only with the other CTA's
  // half too (see mbar_wait_cluster_drain).
  for (uint32_t k = 1; k <= (uint32_t)C::kKStages && k <= k_armed; ++k) {
    const uint32_t i = k_armed - k;
    if constexpr (SHARE)
      mbar_wait_cluster_drain(bar(C::kKFull + i % C::kKStages), (i / C::kKStages) & 1u, wc);
    else
      mbar_wait_drain(bar(C::kKFull + i % C::kKStages), (i / C::kKStages) & 1u, wc);
  }
  for (uint32_t k = 1; k <= 2u && k <= q_armed; ++k) {
    const uint32_t i = q_armed - k;
    mbar_wait_drain(bar(C::kQFull + (i & 1u)), (i >> 1) & 1u, wc);
  }
  // Head-pair cluster: the other CTA's last commits (arrivals on this CTA's
  // empty barriers) land before this CTA may exit.
  if constexpr (SHARE) {
    for (uint32_t k = 1; k <= (uint32_t)C::kKStages && k <= k_armed; ++k) {
      const uint32_t i = k_armed - k;
      mbar_wait_cluster_drain(bar(C::kKEmpty + i % C::kKStages), (i / C::kKStages) & 1u, wc);
    }
  }
}

// V producer (one thread of another warp): the ring of value tiles, so that
// a value tile waiting for its stage never holds back the next key tile.
template <int D, bool F8, bool V8, bool PAIR, bool SHARE>
__device__ void producer_v_role(const KernelParams& p, const CUtensorMap* tm_v, uint32_t sbase,
                                int beg, int end, const WaitCtl& wc) {
  using C = Cfg<D, F8, V8, PAIR, SHARE>;
  constexpr int kCtas = PAIR ? 2 : 1;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * (uint32_t)i; };
  const uint64_t keep = l2_policy_evict_last();
  uint32_t g = 0, v_armed = 0;
  bool ok = true;
  const int srank = SHARE ? (int)cluster_rank() : 0;  // the value box this CTA copies
  for (UnitIter ui = role_units<PAIR, SHARE>(p, beg, end, 0); ui.valid() && ok; ui.next()) {
    const pk_work_item& w = ui.w;
    for (int j = 0; j < w.n_kt; ++j, ++g) {
      const uint32_t st = g % C::kVStages, ph = (g / C::kVStages) & 1u;
      if (!(ok = mbar_wait(bar(C::kVEmpty + st), ph ^ 1u, wc))) break;
      mbar_arrive_expect_tx(bar(C::kVFull + st), kCtas * C::kVTileBytes);
      ++v_armed;
      if constexpr (SHARE) {  // this CTA's half of the tile, into both CTAs
        if constexpr (C::kVBoxes == 2)
          tma_load_3d_mc(sbase + C::kOffV + st * C::kVTileBytes + srank * kBoxBytes, tm_v,
                         bar(C::kVFull + st), srank * 64, w.hkv, key_tile_row(p, w, j),
                         (uint16_t)3, keep);
        else
          tma_load_3d_mc(sbase + C::kOffV + st * C::kVTileBytes + srank * 64 * 128, tm_v,
                         bar(C::kVFull + st), 0, w.hkv, key_tile_row(p, w, j) + srank * 64,
                         (uint16_t)3, keep);
      } else if constexpr (PAIR) {  // value columns [64 r, 64 r + 64) to rank r
#pragma unroll
        for (int r = 0; r < 2; ++r)
          tma_load_3d_pair(map_to_rank(sbase + C::kOffV + st * C::kVTileBytes, r), tm_v,
                           bar(C::kVFull + st), r * 64, w.hkv, key_tile_row(p, w, j), keep);
      } else if constexpr (V8) {  // (key, head-dimension index, head) view of the transposed copy
        const int row = p.v8_row ? p.v8_row[ui.it] + j * 128 : key_tile_row(p, w, j);
        tma_load_3d_hint(sbase + C::kOffV + st * C::kVTileBytes, tm_v, bar(C::kVFull + st), row,
                         0, w.hkv, keep);
      } else {
#pragma unroll
        for (int h = 0; h < C::kVBoxes; ++h)
          tma_load_3d_hint(sbase + C::kOffV + st * C::kVTileBytes + h * kBoxBytes, tm_v,
                           bar(C::kVFull + st), h * 64, w.hkv, key_tile_row(p, w, j), keep);
      }
    }
  }
  for (uint32_t k = 1; k <= (uint32_t)C::kVStages && k <= v_armed; ++k) {  // as above
    const uint32_t i = v_armed - k;
    if constexpr (SHARE)
      mbar_wait_cluster_drain(bar(C::kVFull + i % C::kVStages), (i / C::kVStages) & 1u, wc);
    else
      mbar_wait_drain(bar(C::kVFull + i % C::kVStages), (i / C::kVStages) & 1u, wc);
  }
  if constexpr (SHARE) {
    for (uint32_t k = 1; k <= (uint32_t)C::kVStages && k <= v_armed; ++k) {
      const uint32_t i = v_armed - k;
      mbar_wait_cluster_drain(bar(C::kVEmpty + i % C::kVStages), (i / C::kVStages) & 1u, wc);
    }
  }
}

// MMA issue is split between two threads (a tcgen05.mma costs its issuing
// thread about as long as a third of the 128x128x16 product itself, and two
// threads of different warps issue concurrently).  Key tile t of the CTA's
// stream (t counts across units) computes S(t) into S buffer t%2; after the
// softmax has written P(t) into P buffer t%2, O += P(t) V(t).
//
// S issuer (warp 1): S(t) needs K(t) loaded and S buffer t%2 released by the
// softmax of tile t-2, so it runs up to two tiles ahead of the softmax and
// the tensor pipe computes S(t+2) while the softmax works on tile t.
template <int D, bool F8, bool V8, bool PAIR, bool SHARE>
__device__ void mma_s_role(const KernelParams& p, uint32_t sbase, uint32_t tmem, int beg,
                           int end, const WaitCtl& wc) {
  using C = Cfg<D, F8, V8, PAIR, SHARE>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * (uint32_t)i; };
  const uint64_t q_desc0 = sdesc(sbase + C::kOffQ, 16, 1024);
  const uint64_t k_desc0 = sdesc(sbase + C::kOffK, 16, 1024);
  constexpr uint64_t kQTileDesc = (uint64_t)(C::kQKTileBytes >> 4);
  constexpr uint64_t kKTileDesc = (uint64_t)(C::kKTileBytes >> 4);
  uint32_t t = 0, u = 0;
  bool ok = true;
  for (UnitIter ui = role_units<PAIR, SHARE>(p, beg, end, 0); ui.valid() && ok; ui.next(), ++u) {
    const uint32_t n = (uint32_t)ui.w.n_kt, qb = u & 1u;
    if (!(ok = mbar_wait(bar(C::kQFull + qb), (u >> 1) & 1u, wc))) break;
    for (uint32_t j = 0; j < n; ++j, ++t) {
      const uint32_t kst = t % C::kKStages, b = t & 1u;
      if (!(ok = mbar_wait(bar(C::kKFull + kst), (t / C::kKStages) & 1u, wc))) break;
      if (t >= 2 && !(ok = mbar_wait(bar(C::kSFree + b), ((t >> 1) - 1u) & 1u, wc))) break;
      tc_fence_after();
      if constexpr (PAIR) {  // both CTAs' softmax wait for S; the buffers are this CTA's
        issue_qk_pair<D>(tmem + C::kColS0 + b * 128u, q_desc0 + qb * kQTileDesc,
                         k_desc0 + kst * kKTileDesc);
        tc_commit_pair(bar(C::kSFull + b), 3);
        tc_commit_pair(bar(C::kKEmpty + kst), 1);
        if (j + 1 == n) tc_commit_pair(bar(C::kQEmpty + qb), 1);
      } else {
        issue_qk<D, F8>(tmem + C::kColS0 + b * 128u, q_desc0 + qb * kQTileDesc,
                        k_desc0 + kst * kKTileDesc);
        tc_commit(bar(C::kSFull + b));
        if constexpr (SHARE)  // both CTAs' producers refill this stage
          tc_commit_mc(bar(C::kKEmpty + kst), 3);
        else
          tc_commit(bar(C::kKEmpty + kst));
        if (j + 1 == n) tc_commit(bar(C::kQEmpty + qb));  // last use of this Q buffer
      }
    }
  }
  // Every MMA this thread issued must finish before TMEM is released.
  if constexpr (PAIR)
    tc_commit_pair(bar(C::kMmaDone + 0), 1);
  else
    tc_commit(bar(C::kMmaDone + 0));
  mbar_wait_drain(bar(C::kMmaDone + 0), 0, wc);
}

// P V issuer (warp 3): O (+)= P(t) V(t) needs V(t) loaded and P(t) written;
// a unit's first product overwrites O, after the previous unit's O was read.
template <int D, bool F8, bool V8, bool PAIR, bool SHARE>
__device__ void mma_pv_role(const KernelParams& p, uint32_t sbase, uint32_t tmem, int beg,
                            int end, const WaitCtl& wc) {
  using C = Cfg<D, F8, V8, PAIR, SHARE>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * (uint32_t)i; };
  // fp16 values: MN-major, 64-column boxes kBoxBytes apart; E4M3 values:
  // K-major (transposed copy)
  const uint64_t v_desc0 = sdesc(sbase + C::kOffV, V8 ? 16u : (uint32_t)kBoxBytes, 1024);
  constexpr uint64_t kTileDesc = (uint64_t)(C::kVTileBytes >> 4);
  uint32_t t = 0, u = 0;
  bool ok = true;
  for (UnitIter ui = role_units<PAIR, SHARE>(p, beg, end, 0); ui.valid() && ok; ui.next(), ++u) {
    const uint32_t n = (uint32_t)ui.w.n_kt;
    for (uint32_t j = 0; j < n; ++j, ++t) {
      const uint32_t vst = t % C::kVStages, b = t & 1u;
      if (!(ok = mbar_wait(bar(C::kVFull + vst), (t / C::kVStages) & 1u, wc))) break;
      if (!(ok = mbar_wait(bar(C::kPReady + b), (t >> 1) & 1u, wc))) break;
      if (j == 0 && !(ok = mbar_wait(bar(C::kOFree), (u & 1u) ^ 1u, wc))) break;
      tc_fence_after();
      if constexpr (PAIR) {  // both CTAs' softmax and epilogue wait for P V
        issue_pv_pair<D>(tmem + C::kColO, tmem + C::kColP0 + b * 64u, v_desc0 + vst * kTileDesc,
                         j > 0);
        tc_commit_pair(bar(C::kPvDone + b), 3);
        tc_commit_pair(bar(C::kVEmpty + vst), 1);
      } else {
        if constexpr (V8)
          issue_pv_f8<D>(tmem + C::kColO, tmem + C::kColP0 + b * 64u, v_desc0 + vst * kTileDesc,
                         j > 0);
        else
          issue_pv<D>(tmem + C::kColO, tmem + C::kColP0 + b * 64u, v_desc0 + vst * kTileDesc,
                      j > 0);
        tc_commit(bar(C::kPvDone + b));
        if constexpr (SHARE)
          tc_commit_mc(bar(C::kVEmpty + vst), 3);
        else
          tc_commit(bar(C::kVEmpty + vst));
      }
    }
  }
  if constexpr (PAIR)
    tc_commit_pair(bar(C::kMmaDone + 1), 1);
  else
    tc_commit(bar(C::kMmaDone + 1));
  mbar_wait_drain(bar(C::kMmaDone + 1), 0, wc);
}

// An arrival of a softmax or epilogue thread on an MMA-side barrier: this
// CTA's, or in the pair kernel's rank-1 CTA the rank-0 CTA's.  The rank-1
// arrival is relaxed: what it announces (S or O read out of this CTA's TMEM,
// or P written into it) has completed before it (every TMEM load and store
// here is fused with its wait), and the products that follow only touch
// TMEM.
template <bool PAIR>
__device__ __forceinline__ void group_arrive(uint32_t bar, uint32_t rank) {
  if (PAIR && rank != 0)
    mbar_arrive_cluster_relaxed(map_to_rank(bar, 0));
  else
    mbar_arrive(bar);
}

// Softmax warpgroup (warps 4-7): thread r owns row r of S, P and O in TMEM.
template <int D, bool F8, bool V8, bool PAIR, bool SHARE>
__device__ void softmax_role(const KernelParams& p, uint32_t sbase, uint8_t* sgen, uint32_t tmem,
                             int beg, int end, const WaitCtl& wc) {
  using C = Cfg<D, F8, V8, PAIR, SHARE>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * (uint32_t)i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;  // TMEM lane quadrant this warp may access
  const int r = quad * 32 + lane;
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  const uint32_t tO = tmem + lane_base + C::kColO;
  const float sl2 = p.scale_log2;
  uint32_t g = 0, u = 0;
  bool ok = true;
  bool s_ready = false;  // S(t) of the next tile already seen complete
  float2* lm = reinterpret_cast<float2*>(sgen + C::kOffLm);
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  for (UnitIter ui = role_units<PAIR, SHARE>(p, beg, end, rank); ui.valid() && ok;
       ui.next(), ++u) {
    const pk_work_item& w = ui.w;
    const bool valid = r < w.q_rows;
    // (a pair's rank-1 item may have no rows: its rows see no key)
    const int lim = w.q_rows > 0 ? p.kv_limit[w.q_start + (valid ? r : w.q_rows - 1)] : -1;
    float m_used = -INFINITY, l = 0.f;
    for (int j = 0; j < w.n_kt; ++j) {
      const uint32_t t = g + (uint32_t)j, b = t & 1u;
      const uint32_t tS = tmem + lane_base + C::kColS0 + b * 128u;
      const uint32_t tP = tmem + lane_base + C::kColP0 + b * 64u;
      if (!s_ready) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kSFull + b), (t >> 1) & 1u, wc));
        if (!ok) break;
      }
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld_x128(tS, sr);
      // S buffer b may now take S(t+2).
      tc_fence_before();
      group_arrive<PAIR>(bar(C::kSFree + b), rank);
      if (j >= w.n_full) {  // partial tile: keys past this row's limit are -inf
        const int nvis = lim - j * 128 + 1;
#pragma unroll
        for (int c = 0; c < 128; ++c) sr[c] = c < nvis ? sr[c] : 0xff800000u;
      }
      // P buffer b last held P(t-2); test early whether its product has
      // been read, so the barrier latency hides under the exponentials.
      const uint32_t tpp = t - 2u;
      const bool p_free = t < 2 || mbar_test_wait(bar(C::kPvDone + b), (tpp >> 1) & 1u);
      // Likewise whether S(t+1) has landed (S(t+3) cannot complete before
      // this softmax frees S(t+1)'s buffer, so a yes stays valid).
      const bool s_next = mbar_test_wait(bar(C::kSFull + (b ^ 1u)), ((t + 1u) >> 1) & 1u);
      // p = 2^(s*scale*log2e - m) as fp16 pairs for the tensor cores, the
      // row sum l in fp32.  After a unit's first tile, the exponentials use
      // the running maximum m_used as it stands.  Every p is non-negative, so
      // none can pass 2^kRescaleLog2 unless the tile's sum does: only then is
      // the tile maximum computed, and if it passes m_used + kRescaleLog2
      // the row takes it, rescales O and l, and recomputes the tile from the
      // scores still in registers.  P, O and l keep their relative
      // precision at any scale, so the only limits on the threshold are
      // range: p <= 2^15 fits fp16 P, and O <= L * 2^15 * max|v|.
      // V8: P as E4M3 codes, four keys per TMEM column (32 columns).
      uint32_t pp[V8 ? 32 : 64];
      float acc[8];
      auto exp_pass = [&](float neg) {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        if constexpr (V8) {
#pragma unroll
          for (int c = 0; c < 128; c += 4) {
            float a0, a1, a2, a3;
            fma2(a0, a1, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]), sl2, sl2, neg, neg);
            fma2(a2, a3, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]), sl2, sl2, neg, neg);
            const float p0 = ex2(a0), p1 = ex2(a1), p2 = ex2(a2), p3 = ex2(a3);
            pp[c >> 2] = pack_e4m3x4(p0, p1, p2, p3);
            const int q = (c >> 2) & 1;
            acc2(acc[4 * q], acc[4 * q + 1], p0, p1);
            acc2(acc[4 * q + 2], acc[4 * q + 3], p2, p3);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 128; c += 2) {
            float a0, a1;
            fma2(a0, a1, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]), sl2, sl2, neg, neg);
            const float p0 = ex2(a0), p1 = ex2(a1);
            pp[c >> 1] = pack_f16x2(p0, p1);
            const int q = (c >> 1) & 3;
            acc2(acc[2 * q], acc[2 * q + 1], p0, p1);
          }
        }
      };
      auto row_max = [&]() {
        float mc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mc[i] = fmaxf(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]));
#pragma unroll
        for (int b0 = 16; b0 < 128; b0 += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i)
            mc[i] = max3(mc[i], __uint_as_float(sr[b0 + 2 * i]), __uint_as_float(sr[b0 + 2 * i + 1]));
        return max3(max3(mc[0], mc[1], mc[2]), max3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7])) * sl2;
      };
      // E4M3 P (largest finite 448) lets the maximum lag by 8 at most.
      constexpr float kLag = V8 ? 8.0f : kRescaleLog2;
      constexpr float kRescaleSum = V8 ? 256.0f : 32768.0f;  // 2^kLag
      if (j == 0) m_used = row_max();
      // The rare rescale path takes a second trip through this one copy of
      // the exponential loop (a second inlined copy measured slower).
      unsigned votes;
      for (int pass = 0;; ++pass) {
        // A row that sees no key of its range keeps m_used = -inf and p = 0.
        exp_pass(m_used == -INFINITY ? 0.0f : -m_used);
        if (pass == 1) break;
        const float tile_sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        // One warp vote for: a possible rescale (bit 0), P buffer still busy
        // (bit 1), next S not yet seen (bit 2).
        votes = __reduce_or_sync(
            0xffffffffu, (!(tile_sum <= kRescaleSum) ? 1u : 0u) | (p_free ? 0u : 2u) | (s_next ? 0u : 4u));
        if (!(votes & 1u)) break;
        // Rare: some row's maximum may have outgrown m_used.
        const float m_tile = row_max();
        const bool need = m_tile > m_used + kLag;
        if (!__any_sync(0xffffffffu, need)) break;
        // O must hold P(t-1) V(t-1) before it is rescaled (j > 0 here: the
        // first tile's maximum is exact).
        const uint32_t tp = t - 1u;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kPvDone + (tp & 1u)), (tp >> 1) & 1u, wc));
        if (!ok) break;
        tc_fence_after();
        const float f = need ? ex2(m_used - m_tile) : 1.0f;
        if (need) {
          m_used = m_tile;
          l *= f;
        }
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld_x32(tO + (uint32_t)c0, o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f);
          tmem_st_x32(tO + (uint32_t)c0, o);
        }
      }
      if (!ok) break;
      s_ready = (votes & 4u) == 0u;
      l += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      if (votes & 2u) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kPvDone + b), (tpp >> 1) & 1u, wc));
        if (!ok) break;
      }
      tc_fence_after();
      if constexpr (V8)
        tmem_st_x32(tP, pp);
      else
        tmem_st_x64(tP, pp);
      tc_fence_before();
      group_arrive<PAIR>(bar(C::kPReady + b), rank);
    }
    if (!ok) break;
    // Hand the unit's row statistics to the epilogue warps, once they have
    // taken the previous unit's.
    if (u > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kLmFree), (u - 1u) & 1u, wc));
      if (!ok) break;
    }
    lm[r] = make_float2(m_used, l);
    mbar_arrive(bar(C::kLmFull));
    g += (uint32_t)w.n_kt;
  }
}

// Epilogue warpgroup (warps 8-11): thread r owns row r of O in TMEM.  Per
// unit it takes (m, l) from the softmax, waits for the unit's last P V,
// moves O into registers and frees it for the next unit's first product,
// then writes O / l as bf16 and the natural-log LSE.
template <int D, bool F8, bool V8, bool PAIR, bool SHARE>
__device__ void epilogue_role(const KernelParams& p, uint32_t sbase, uint8_t* sgen,
                              uint32_t tmem, int beg, int end, const WaitCtl& wc) {
  using C = Cfg<D, F8, V8, PAIR, SHARE>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * (uint32_t)i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const uint32_t tO = tmem + ((uint32_t)(quad * 32) << 16) + C::kColO;
  const float2* lm = reinterpret_cast<const float2*>(sgen + C::kOffLm);
  uint32_t g = 0, u = 0;
  bool ok = true;
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  for (UnitIter ui = role_units<PAIR, SHARE>(p, beg, end, rank); ui.valid() && ok;
       ui.next(), ++u) {
    const pk_work_item& w = ui.w;
    const int h = ui.head();
    if (!(ok = __all_sync(0xffffffffu, mbar_wait_sleep(bar(C::kLmFull), u & 1u, wc)))) break;
    const float2 ml = lm[r];
    mbar_arrive(bar(C::kLmFree));
    const uint32_t tl = g + (uint32_t)w.n_kt - 1u;  // the unit's last product
    ok = __all_sync(0xffffffffu, mbar_wait_sleep(bar(C::kPvDone + (tl & 1u)), (tl >> 1) & 1u, wc));
    if (!ok) break;
    tc_fence_after();
    uint32_t o[D];
    if constexpr (D == 128) {
      tmem_ld_x128(tO, o);
    } else {
      uint32_t (&o0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&o[0]);
      uint32_t (&o1)[32] = *reinterpret_cast<uint32_t (*)[32]>(&o[32]);
      tmem_ld_x32(tO, o0);
      tmem_ld_x32(tO + 32u, o1);
    }
    tc_fence_before();
    group_arrive<PAIR>(bar(C::kOFree), rank);
    const float l = ml.y;
    // a row without keys writes zeros; E4M3 values carry their scale
    const float inv_l = l > 0.f ? p.v_scale / l : 0.f;
    // The thread's row as bf16: N = D/8 chunks of 16 bytes (4 words each).
    constexpr int N = D / 8;
    constexpr int G = kStoreGroup < N ? kStoreGroup : N;
    uint32_t pk[D / 2];
#pragma unroll
    for (int c = 0; c < D / 2; ++c) {
      float x0, x1;
      mul2(x0, x1, __uint_as_float(o[2 * c]), __uint_as_float(o[2 * c + 1]), inv_l, inv_l);
      pk[c] = pack_bf16x2(x0, x1);
    }
    // Transpose G x G blocks of chunks within each group of G lanes (rows):
    // stage m swaps bit m of (lane, chunk) for every chunk (a chunk whose
    // bits differ moves to lane l ^ m, slot s ^ m), so afterwards lane l
    // holds, in slot B*G + k, chunk B*G + l of its group's row k.
    const int lid = lane & (G - 1);
#pragma unroll
    for (int m = 1; m < G; m <<= 1) {
      const bool hi = (lid & m) != 0;
#pragma unroll
      for (int s0 = 0; s0 < N; ++s0) {
        if (s0 & m) continue;
        const int s1 = s0 | m;
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
          const uint32_t send = hi ? pk[4 * s0 + wd] : pk[4 * s1 + wd];
          const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, m);
          if (hi)
            pk[4 * s0 + wd] = recv;
          else
            pk[4 * s1 + wd] = recv;
        }
      }
    }
    // Store (B, k): the G lanes of a group write G * 16 contiguous bytes of
    // one row, chunks B*G .. B*G + G - 1 (32 / G rows per warp instruction).
    const int row0 = quad * 32 + (lane / G) * G;
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const int row = row0 + k;
      if (row < w.q_rows) {
        uint8_t* dst = p.out + (((size_t)(w.q_start + row) * (size_t)p.hq + (size_t)h) * D) * 2 +
                       (size_t)lid * 16;
#pragma unroll
        for (int B = 0; B < N / G; ++B) {
          const int s = B * G + k;
          *reinterpret_cast<uint4*>(dst + (size_t)B * G * 16) =
              make_uint4(pk[4 * s], pk[4 * s + 1], pk[4 * s + 2], pk[4 * s + 3]);
        }
      }
    }
    if (r < w.q_rows)
      p.lse[(size_t)h * (size_t)p.T + (size_t)(w.q_start + r)] =
          l > 0.f ? (ml.x + __log2f(l)) * 0.69314718055994530942f : -INFINITY;
    g += (uint32_t)w.n_kt;
  }
}

// Values bf16 -> fp16, before the attention launch, into the caller's
// workspace (rows at the same offsets as in v; v16 may be v itself).  P
// enters the P V product as fp16 (11 significant bits, against bf16's 8), and
// the product takes both operands in one format.  bf16 values in [2^-14,
// 2^16) convert exactly; smaller ones round to fp16 subnormals (absolute
// error <= 2^-25); magnitudes of 2^16 and beyond saturate to 65504 and the
// launch reports PK_ERR_RANGE.  The work is a list of 128-row blocks:
// `blocks` holds (block, rows holding keys) pairs, the block's other rows
// zeroed (they are read only as masked keys, where 0 * P must stay 0 even if
// the pool holds garbage there); with `blocks` null, blocks 0, 1, ... of
// rows [0, rows).  Every thread moves 16 bytes per step, four steps in
// flight.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 x, float& amax) {
  uint4 y;
  y.x = bf16x2_to_f16x2(x.x, amax);
  y.y = bf16x2_to_f16x2(x.y, amax);
  y.z = bf16x2_to_f16x2(x.z, amax);
  y.w = bf16x2_to_f16x2(x.w, amax);
  return y;
}

__global__ void __launch_bounds__(512) pk_v_to_f16_kernel(const uint4* v, uint4* v16,
                                                          const int32_t* __restrict__ blocks,
                                                          int32_t num_blocks, int32_t rows,
                                                          int32_t pieces_per_row,
                                                          int32_t* status) {
  constexpr int kStep = 512;
  float amax = 0.f;
  for (int32_t i = blockIdx.x; i < num_blocks; i += gridDim.x) {
    const int32_t blk = blocks ? blocks[2 * i] : i;
    const int32_t nvalid = blocks ? blocks[2 * i + 1] : min(128, rows - blk * 128);
    const size_t base = (size_t)blk * 128 * pieces_per_row;
    const int32_t n = nvalid * pieces_per_row;
    int32_t k = threadIdx.x;
    for (; k + 3 * kStep < n; k += 4 * kStep) {
      uint4 x[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) x[c] = v[base + k + c * kStep];
#pragma unroll
      for (int c = 0; c < 4; ++c) v16[base + k + c * kStep] = bf16x8_to_f16x8(x[c], amax);
    }
    for (; k < n; k += kStep) v16[base + k] = bf16x8_to_f16x8(v[base + k], amax);
    if (blocks) {
      const int32_t n_all = 128 * pieces_per_row;
      for (k = n + threadIdx.x; k < n_all; k += kStep) v16[base + k] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (!(amax < 65520.0f) && status) atomicCAS(status, 0, (int32_t)PK_ERR_RANGE);
}

// E4M3 values [Tk][H][D] -> the transposed copy [H][D][rows_t] bytes that
// the all-E4M3 P V product reads K-major (one row of keys per head-dimension
// index).  Work items are (chunk, head) pairs; a chunk (source row, copy
// row, rows holding keys n, rows written m; n <= m <= 128, the copy row and
// m multiples of 16) moves source rows [src, src + n) to copy rows
// [dst, dst + n) and writes zeros to copy rows [dst + n, dst + m).  Each
// item goes through a shared-memory tile: 16-byte loads along the head
// dimension, 16-byte stores along the keys.
__global__ void __launch_bounds__(256) pk_v8_transpose_kernel(const uint8_t* v8, uint8_t* vt,
                                                              const int32_t* __restrict__ chunks,
                                                              int32_t num_chunks, int32_t H,
                                                              int32_t D, int32_t rows_t) {
  __shared__ uint32_t tile[128][33];  // [key][head-dim word] (D <= 128), padded
  for (int32_t i = blockIdx.x; i < num_chunks * H; i += gridDim.x) {
    const int32_t ci = i / H, h = i - ci * H;
    const int32_t src = chunks[4 * ci], dst = chunks[4 * ci + 1];
    const int32_t n = chunks[4 * ci + 2], m = chunks[4 * ci + 3];
    const int32_t pieces = D / 16;  // 16-byte pieces per key
    for (int32_t e = threadIdx.x; e < 128 * pieces; e += 256) {
      const int32_t k = e / pieces, c = e - k * pieces;
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (k < n)
        x = *reinterpret_cast<const uint4*>(v8 + ((size_t)(src + k) * H + h) * D + (size_t)c * 16);
      tile[k][4 * c + 0] = x.x;
      tile[k][4 * c + 1] = x.y;
      tile[k][4 * c + 2] = x.z;
      tile[k][4 * c + 3] = x.w;
    }
    __syncthreads();
    for (int32_t e = threadIdx.x; e < D * 8; e += 256) {  // (head-dim index, 16 keys)
      const int32_t dd = e >> 3, k0 = (e & 7) * 16;
      if (k0 >= m) continue;
      uint32_t w[4];
#pragma unroll
      for (int32_t q = 0; q < 4; ++q) {
        uint32_t word = 0;
#pragma unroll
        for (int32_t b = 0; b < 4; ++b)
          word |= ((tile[k0 + 4 * q + b][dd >> 2] >> (8 * (dd & 3))) & 0xffu) << (8 * b);
        w[q] = word;
      }
      *reinterpret_cast<uint4*>(vt + ((size_t)h * D + dd) * rows_t + dst + k0) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
  }
}

template <int D, bool F8, bool V8, bool PAIR, bool SHARE>
__global__ void __launch_bounds__(kThreads, 1)
    pk_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const KernelParams p) {
  using C = Cfg<D, F8, V8, PAIR, SHARE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1 KB alignment
  uint8_t* sgen = smem_raw + (sbase - raw);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sgen + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + C::kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * (uint32_t)i; };
  // Pair kernel: CTA rank 0 of each cluster loads both CTAs' tiles and issues
  // the M = 256 products; both CTAs run their rows' softmax and epilogue.
  const uint32_t rank = PAIR ? cluster_rank() : 0u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kQFull + s), 1);
      mbar_init(bar(C::kQEmpty + s), 1);
      mbar_init(bar(C::kSFull + s), 1);
      mbar_init(bar(C::kSFree + s), C::kGroupArrivals);
      mbar_init(bar(C::kPReady + s), C::kGroupArrivals);
      mbar_init(bar(C::kPvDone + s), 1);
    }
    // SHARE: a ring stage is empty once both CTAs' products have read it.
    constexpr uint32_t kEmptyArrivals = SHARE ? 2 : 1;
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(bar(C::kKFull + s), 1);
      mbar_init(bar(C::kKEmpty + s), kEmptyArrivals);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(bar(C::kVFull + s), 1);
      mbar_init(bar(C::kVEmpty + s), kEmptyArrivals);
    }
    mbar_init(bar(C::kOFree), C::kGroupArrivals);
    mbar_init(bar(C::kMmaDone + 0), 1);
    mbar_init(bar(C::kMmaDone + 1), 1);
    mbar_init(bar(C::kLmFull), 128);
    mbar_init(bar(C::kLmFree), 128);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    if constexpr (PAIR) {  // one allocation for the pair: the same columns in both CTAs
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_holder)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_holder)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  // Clusters: both CTAs' barriers exist before either CTA's copies or
  // arrivals reach them.
  if constexpr (PAIR || SHARE) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int unit_set = (PAIR || SHARE) ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int beg = p.cta_offsets[unit_set], end = p.cta_offsets[unit_set + 1];
  const WaitCtl wc{abort_flag, p.status, p.wait_limit_ns};

  if (warp < 4) {
    // Producers and MMA issuers: one thread each, few registers (idle in the
    // pair's rank-1 CTA).
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsMma));
    if (rank == 0) {
      if (warp == 0) {
        if (lane == 0) producer_qk_role<D, F8, V8, PAIR, SHARE>(p, &tm_q, &tm_k, sbase, beg, end, wc);
      } else if (warp == 1) {
        if (lane == 0) mma_s_role<D, F8, V8, PAIR, SHARE>(p, sbase, tmem, beg, end, wc);
      } else if (warp == 2) {
        if (lane == 0) producer_v_role<D, F8, V8, PAIR, SHARE>(p, &tm_v, sbase, beg, end, wc);
      } else {
        if (lane == 0) mma_pv_role<D, F8, V8, PAIR, SHARE>(p, sbase, tmem, beg, end, wc);
      }
    }
    __syncwarp();
  } else if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    softmax_role<D, F8, V8, PAIR, SHARE>(p, sbase, sgen, tmem, beg, end, wc);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
    epilogue_role<D, F8, V8, PAIR, SHARE>(p, sbase, sgen, tmem, beg, end, wc);
  }

  tc_fence_before();
  __syncthreads();
  // Pair: the rank-0 CTA's products read and write both CTAs' shared and
  // tensor memory, and its copies land in both; it leaves this barrier only
  // after its issuers and producers have drained them, and neither CTA
  // frees TMEM or exits before that.  Head-pair cluster: each CTA's copies
  // land in both CTAs; neither exits before the other has drained.
  if constexpr (PAIR || SHARE) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(kTmemCols)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(kTmemCols)
                   : "memory");
  }
}

// One CTA waits on a barrier that nothing arrives at; the bounded wait must
// give up, record PK_ERR_TIMEOUT and return.
__global__ void pk_wait_timeout_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar_storage;
  __shared__ int abort_flag;
  const uint32_t bar = smem_u32(&bar_storage);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl wc{&abort_flag, status, limit_ns};
    mbar_wait(bar, 0, wc);
  }
  __syncthreads();
}

}  // namespace dev
}  // namespace pk

namespace {

std::atomic<uint64_t> g_wait_limit_ns{4000000000ull};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qres;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &qres) == cudaSuccess &&
        qres == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

// (d, H, T) view of a [T][H][d] tensor of 2-byte (bf16, fp16) or 1-byte
// (FP8) elements, boxes of 128 bytes x 1 head x 128 rows with 128-byte
// swizzle; rows past T read as zeros.
bool make_map(CUtensorMap* m, const void* base, int H, int T, int D, CUtensorMapDataType dt,
              int box_rows = 128) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t eb = dt == CU_TENSOR_MAP_DATA_TYPE_UINT8 ? 1 : 2;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)D * eb, (cuuint64_t)H * D * eb};
  const cuuint32_t box[3] = {(cuuint32_t)(128 / eb), 1, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// (key, head-dimension index, head) view of the transposed E4M3 value copy
// [H][D][rows_t] bytes: boxes of 128 keys (128 bytes) x D x 1 head with
// 128-byte swizzle; keys past rows_t read as zeros.
bool make_map_v8t(CUtensorMap* m, const void* base, int H, int rows_t, int D) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)rows_t, (cuuint64_t)D, (cuuint64_t)H};
  const cuuint64_t strides[2] = {(cuuint64_t)rows_t, (cuuint64_t)D * rows_t};
  const cuuint32_t box[3] = {128, (cuuint32_t)D, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Device capability check and SM count, cached per device ordinal.
pk_status check_device(int* sm_count = nullptr) {
  static std::mutex mu;
  static int cap_state[64];  // 0 unknown, 1 ok, 2 unsupported
  static int sms[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return PK_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(mu);
  if (cap_state[dev] == 0) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return PK_ERR_CUDA;
    }
    sms[dev] = n;
    cap_state[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  if (sm_count) *sm_count = sms[dev];
  return cap_state[dev] == 1 ? PK_OK : PK_ERR_UNSUPPORTED;
}

// The value rows the plan's kernel reads, bf16 -> fp16 into v16 (which may
// be v itself: the conversion is elementwise, in place).  Contiguous keys:
// rows [0, v_conv_rows) converted, rows no sequence owns zeroed (a key tile
// overhanging the last sequence reads them, masked, and 0 * P must stay 0).
// Paged keys: the pool blocks the block table lists, rows past each block's
// keys zeroed.
pk_status convert_values(const pk_plan* plan, const void* v, void* v16, int sm_count,
                         cudaStream_t stream, int32_t* dev_status) {
  const size_t row_bytes = (size_t)plan->hkv * plan->head_dim * 2;
  const int32_t pieces_per_row = (int32_t)(row_bytes / 16);
  const int32_t* list = nullptr;
  int32_t nblocks = 0, rows = plan->Tk;
  if (plan->paged) {
    list = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(plan->dev) +
                                            plan->layout.vblk_off);
    nblocks = (int32_t)(plan->v_blocks.size() / 2);
  } else {
    rows = plan->v_conv_rows;
    nblocks = (rows + 127) / 128;
    if (plan->Tk > rows &&
        cudaMemsetAsync(static_cast<uint8_t*>(v16) + (size_t)rows * row_bytes, 0,
                        (size_t)(plan->Tk - rows) * row_bytes, stream) != cudaSuccess) {
      cudaGetLastError();
      return PK_ERR_CUDA;
    }
  }
  if (nblocks == 0) return PK_OK;
  const int grid = std::min(nblocks, 4 * std::max(sm_count, 1));
  pk::dev::pk_v_to_f16_kernel<<<grid, 512, 0, stream>>>(static_cast<const uint4*>(v),
                                                         static_cast<uint4*>(v16), list, nblocks,
                                                         rows, pieces_per_row, dev_status);
  if (cudaGetLastError() != cudaSuccess) return PK_ERR_CUDA;
  return PK_OK;
}

// scale: the softmax scale of the scores as the MMA computes them (for FP8
// queries/keys it includes their dequantisation scales).
// The transposed E4M3 copy of the value rows the plan reads (see
// pk_v8_transpose_kernel and the plan's chunk list), into vt.
pk_status transpose_values(const pk_plan* plan, const void* v8, void* vt, int sm_count,
                           cudaStream_t stream) {
  const int32_t nchunks = (int32_t)(plan->v8_chunks.size() / 4);
  if (nchunks == 0) return PK_OK;
  const int32_t* list = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(plan->dev) +
                                                         plan->layout.v8chunk_off);
  const int grid = std::min(nchunks * plan->hkv, 8 * std::max(sm_count, 1));
  pk::dev::pk_v8_transpose_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint8_t*>(v8), static_cast<uint8_t*>(vt), list, nchunks, plan->hkv,
      plan->head_dim, plan->v8_rows);
  if (cudaGetLastError() != cudaSuccess) return PK_ERR_CUDA;
  return PK_OK;
}

// v16: the fp16 values (the workspace convert_values has filled), or with V8
// the transposed E4M3 copy (transpose_values).
template <int D, bool F8, bool V8, bool PAIR = false, bool SHARE = false>
pk_status launch(const pk_plan* plan, const void* q, const void* k, const void* v16, void* out,
                 float* lse, float scale, cudaStream_t stream, int32_t* dev_status,
                 float v_scale = 1.0f) {
  using C = pk::dev::Cfg<D, F8, V8, PAIR, SHARE>;
  auto kernel = pk::dev::pk_attn_fwd_kernel<D, F8, V8, PAIR, SHARE>;
  CUtensorMap tq, tk, tv;
  const CUtensorMapDataType qk_dt =
      F8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map(&tq, q, plan->hq, plan->T, D, qk_dt) ||
      !make_map(&tk, k, plan->hkv, plan->Tk, D, qk_dt, SHARE ? C::kShareKRows : C::kKRows) ||
      !(V8 ? make_map_v8t(&tv, v16, plan->hkv, plan->v8_rows, D)
           : make_map(&tv, v16, plan->hkv, plan->Tk, D, CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      SHARE ? C::kShareVRows : 128)))
    return PK_ERR_CUDA;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  // The warpgroups' register split draws on the CTA's launch allocation: a
  // build whose kernel was compiled with fewer registers per thread must
  // not launch (its setmaxnreg increases could never be granted).
  static std::atomic<int> regs_state{0};  // 0 unknown, 1 fits, 2 does not
  if (regs_state.load() == 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) {
      cudaGetLastError();
      return PK_ERR_CUDA;
    }
    regs_state.store(fa.numRegs >= pk::dev::kRegsLaunch && fa.maxThreadsPerBlock >= pk::dev::kThreads
                         ? 1 : 2);
  }
  if (regs_state.load() != 1) return PK_ERR_UNSUPPORTED;
  const uint8_t* img = static_cast<const uint8_t*>(plan->dev);
  pk::dev::KernelParams kp;
  kp.items = reinterpret_cast<const pk_work_item*>(
      img + (PAIR ? plan->layout.pitems_off
                  : SHARE ? plan->layout.sitems_off : plan->layout.items_off));
  kp.cta_offsets = reinterpret_cast<const int32_t*>(
      img + (PAIR ? plan->layout.pcta_off_off
                  : SHARE ? plan->layout.scta_off_off : plan->layout.cta_off_off));
  kp.kv_limit = reinterpret_cast<const int32_t*>(img + plan->layout.kvlim_off);
  kp.block_table =
      plan->paged ? reinterpret_cast<const int32_t*>(img + plan->layout.table_off) : nullptr;
  kp.v8_row = V8 && !plan->paged
                  ? reinterpret_cast<const int32_t*>(img + plan->layout.v8row_off) : nullptr;
  kp.out = static_cast<uint8_t*>(out);
  kp.lse = lse;
  kp.status = dev_status;
  kp.T = plan->T;
  kp.hq = plan->hq;
  kp.scale_log2 = scale * 1.4426950408889634f;
  kp.v_scale = v_scale;
  kp.wait_limit_ns = g_wait_limit_ns.load();
  if constexpr (PAIR || SHARE) {
    // clusters of two CTAs on neighbouring SMs
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim =
        dim3(2u * (unsigned)(PAIR ? plan->num_clusters : plan->num_share_clusters));
    cfg.blockDim = dim3(pk::dev::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, kp) != cudaSuccess) {
      cudaGetLastError();
      return PK_ERR_CUDA;
    }
    return PK_OK;
  }
  kernel<<<plan->num_ctas, pk::dev::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, kp);
  if (cudaGetLastError() != cudaSuccess) return PK_ERR_CUDA;
  return PK_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace

namespace pk {
uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }
}  // namespace pk

extern "C" {

void pk_set_wait_timeout_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : 1); }

}  // extern "C"

namespace {

// Argument checks shared by the entry points.  check_plan: PK_OK with
// *nothing = true when the plan has no work.
pk_status check_plan(const pk_plan* plan, bool* nothing) {
  *nothing = false;
  if (plan == nullptr) return PK_ERR_INVALID_ARG;
  if (plan->T == 0 || plan->items.empty()) {
    *nothing = true;
    return PK_OK;
  }
  if (plan->dev == nullptr) return PK_ERR_NOT_UPLOADED;
  if (plan->Tk <= 0) return PK_ERR_INVALID_ARG;  // queries need a key/value tensor to map
  return PK_OK;
}

// A value tensor and a workspace (the fp16 copy) of the plan's size.
pk_status check_values(const pk_plan* plan, const void* v, const void* workspace,
                       size_t workspace_bytes, bool e4m3_transposed = false) {
  if (!v || !workspace) return PK_ERR_INVALID_ARG;
  if (workspace_bytes < (e4m3_transposed ? pk_attn_workspace_bytes_fp8_pv(plan)
                                         : pk_attn_workspace_bytes(plan)))
    return PK_ERR_INVALID_ARG;
  if (!aligned16(v) || !aligned16(workspace)) return PK_ERR_ALIGNMENT;
  return PK_OK;
}

// Queries, keys, the outputs and the scale.
pk_status check_attn(const void* q, const void* k, const void* out, const float* lse, float scale) {
  if (!(scale > 0.f) || !std::isfinite(scale)) return PK_ERR_INVALID_ARG;
  if (!q || !k || !out || !lse) return PK_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return PK_ERR_ALIGNMENT;
  return PK_OK;
}

}  // namespace

extern "C" {

pk_status pk_attn_convert_values(const pk_plan* plan, const void* v, void* workspace,
                                 size_t workspace_bytes, pk_stream_t stream,
                                 int32_t* dev_status) {
  bool nothing = false;
  pk_status st = check_plan(plan, &nothing);
  if (st != PK_OK || nothing) return st;
  if ((st = check_values(plan, v, workspace, workspace_bytes)) != PK_OK) return st;
  int sms = 0;
  if ((st = check_device(&sms)) != PK_OK) return st;
  return convert_values(plan, v, workspace, sms, reinterpret_cast<cudaStream_t>(stream),
                        dev_status);
}

pk_status pk_attn_fwd_converted(const pk_plan* plan, const void* q, const void* k,
                                const void* v16, void* out, float* lse, float scale,
                                pk_stream_t stream, int32_t* dev_status) {
  if (plan == nullptr || !(scale > 0.f) || !std::isfinite(scale)) return PK_ERR_INVALID_ARG;
  bool nothing = false;
  pk_status st = check_plan(plan, &nothing);
  if (st != PK_OK || nothing) return st;
  if ((st = check_attn(q, k, out, lse, scale)) != PK_OK ||
      (st = check_values(plan, v16, v16, pk_attn_workspace_bytes(plan))) != PK_OK)
    return st;
  if ((st = check_device()) != PK_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (plan->head_dim == 128) {
    if (plan->use_pairs && plan->num_clusters > 0)  // pk_plan_set_sm_pairs
      return launch<128, false, false, true>(plan, q, k, v16, out, lse, scale, s, dev_status);
    if (plan->use_share && plan->num_share_clusters > 0)  // pk_plan_set_kv_share
      return launch<128, false, false, false, true>(plan, q, k, v16, out, lse, scale, s,
                                                    dev_status);
    return launch<128, false, false>(plan, q, k, v16, out, lse, scale, s, dev_status);
  }
  if (plan->head_dim == 64) {
    if (plan->use_share && plan->num_share_clusters > 0)  // pk_plan_set_kv_share
      return launch<64, false, false, false, true>(plan, q, k, v16, out, lse, scale, s,
                                                   dev_status);
    return launch<64, false, false>(plan, q, k, v16, out, lse, scale, s, dev_status);
  }
  return PK_ERR_UNSUPPORTED;
}

pk_status pk_attn_fwd(const pk_plan* plan, const void* q, const void* k, const void* v,
                      void* out, float* lse, float scale, void* workspace, size_t workspace_bytes,
                      pk_stream_t stream, int32_t* dev_status) {
  if (plan == nullptr || !(scale > 0.f) || !std::isfinite(scale)) return PK_ERR_INVALID_ARG;
  bool nothing = false;
  pk_status st = check_plan(plan, &nothing);
  if (st != PK_OK || nothing) return st;
  if ((st = check_attn(q, k, out, lse, scale)) != PK_OK ||
      (st = check_values(plan, v, workspace, workspace_bytes)) != PK_OK)
    return st;
  if ((st = pk_attn_convert_values(plan, v, workspace, workspace_bytes, stream, dev_status)) !=
      PK_OK)
    return st;
  return pk_attn_fwd_converted(plan, q, k, workspace, out, lse, scale, stream, dev_status);
}

}  // extern "C"

// Scratch of pk_attn_fwd_noalloc: a file-scope device array, so that callers
// who cannot allocate device memory still have room for the fp16 copy of the
// values.  Every device that loads the library holds it until the process
// exits.  In host code its name is only a stand-in: the device address comes
// from cudaGetSymbolAddress, taken once per device (with that device current)
// and cached.
static constexpr size_t kStaticScratchBytes = size_t(64) << 20;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

namespace {

void* static_scratch_address() {
  static std::mutex mu;
  static void* addr[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_static_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = a;
  }
  return addr[dev];
}

}  // namespace

extern "C" {

pk_status pk_attn_fwd_noalloc(const pk_plan* plan, const void* q, const void* k, const void* v,
                              void* out, float* lse, float scale, pk_stream_t stream,
                              int32_t* dev_status) {
  if (plan == nullptr) return PK_ERR_INVALID_ARG;
  if (pk_attn_workspace_bytes(plan) > kStaticScratchBytes) return PK_ERR_TOO_LARGE;
  bool nothing = false;
  pk_status st = check_plan(plan, &nothing);
  if (st != PK_OK || nothing) return st;
  if ((st = check_device()) != PK_OK) return st;
  void* scratch = static_scratch_address();
  if (scratch == nullptr) return PK_ERR_CUDA;
  return pk_attn_fwd(plan, q, k, v, out, lse, scale, scratch, kStaticScratchBytes, stream,
                     dev_status);
}

pk_status pk_attn_fwd_fp8(const pk_plan* plan, const void* q8, float q_scale, const void* k8,
                          float k_scale, const void* v, void* out, float* lse, float scale,
                          void* workspace, size_t workspace_bytes, pk_stream_t stream,
                          int32_t* dev_status) {
  if (plan == nullptr) return PK_ERR_INVALID_ARG;
  const float s_all = scale * q_scale * k_scale;
  if (!(scale > 0.f) || !(q_scale > 0.f) || !(k_scale > 0.f) || !std::isfinite(s_all) ||
      !(s_all > 0.f))
    return PK_ERR_INVALID_ARG;
  if (plan->head_dim != 128) return PK_ERR_UNSUPPORTED;
  bool nothing = false;
  pk_status st = check_plan(plan, &nothing);
  if (st != PK_OK || nothing) return st;
  if ((st = check_attn(q8, k8, out, lse, s_all)) != PK_OK ||
      (st = check_values(plan, v, workspace, workspace_bytes)) != PK_OK)
    return st;
  if ((st = pk_attn_convert_values(plan, v, workspace, workspace_bytes, stream, dev_status)) !=
      PK_OK)
    return st;
  if ((st = check_device()) != PK_OK) return st;
  if (plan->use_share && plan->num_share_clusters > 0)  // pk_plan_set_kv_share
    return launch<128, true, false, false, true>(plan, q8, k8, workspace, out, lse, s_all,
                                                 reinterpret_cast<cudaStream_t>(stream),
                                                 dev_status);
  return launch<128, true, false>(plan, q8, k8, workspace, out, lse, s_all,
                           reinterpret_cast<cudaStream_t>(stream), dev_status);
}

pk_status pk_attn_fwd_fp8_pv(const pk_plan* plan, const void* q8, float q_scale, const void* k8,
                             float k_scale, const void* v8, float v_scale, void* out, float* lse,
                             float scale, void* workspace, size_t workspace_bytes,
                             pk_stream_t stream, int32_t* dev_status) {
  if (plan == nullptr) return PK_ERR_INVALID_ARG;
  const float s_all = scale * q_scale * k_scale;
  if (!(scale > 0.f) || !(q_scale > 0.f) || !(k_scale > 0.f) || !std::isfinite(s_all) ||
      !(s_all > 0.f) || !(v_scale > 0.f) || !std::isfinite(v_scale))
    return PK_ERR_INVALID_ARG;
  if (plan->head_dim != 128) return PK_ERR_UNSUPPORTED;
  bool nothing = false;
  pk_status st = check_plan(plan, &nothing);
  if (st != PK_OK || nothing) return st;
  if ((st = check_attn(q8, k8, out, lse, s_all)) != PK_OK ||
      (st = check_values(plan, v8, workspace, workspace_bytes, true)) != PK_OK)
    return st;
  int sms = 0;
  if ((st = check_device(&sms)) != PK_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = transpose_values(plan, v8, workspace, sms, s)) != PK_OK) return st;
  return launch<128, true, true>(plan, q8, k8, workspace, out, lse, s_all, s, dev_status, v_scale);
}

pk_status pk_attn_fwd_host(const pk_plan* plan, const void* q_host, const void* k_host,
                           const void* v_host, void* out_host, float* lse_host, void* q_dev,
                           void* k_dev, void* v_dev, void* out_dev, float* lse_dev, float scale,
                           pk_stream_t stream, int32_t* dev_status) {
  if (plan == nullptr) return PK_ERR_INVALID_ARG;
  if (plan->T == 0) return PK_OK;
  if (!q_host || !k_host || !v_host || !out_host || !lse_host) return PK_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t T = (size_t)plan->T, Tk = (size_t)plan->Tk, d = (size_t)plan->head_dim;
  const size_t qb = T * plan->hq * d * 2, kvb = Tk * plan->hkv * d * 2;
  const size_t lb = T * plan->hq * sizeof(float);
  if (!q_dev || !k_dev || !v_dev || !out_dev || !lse_dev) return PK_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(q_dev, q_host, qb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(k_dev, k_host, kvb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(v_dev, v_host, kvb, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  // v_dev is library staging: the values are converted to fp16 in place.
  pk_status st = pk_attn_fwd(plan, q_dev, k_dev, v_dev, out_dev, lse_dev, scale, v_dev, kvb,
                             stream, dev_status);
  if (st != PK_OK) return st;
  if (cudaMemcpyAsync(out_host, out_dev, qb, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(lse_host, lse_dev, lb, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  return PK_OK;
}

pk_status pk_debug_wait_timeout(int32_t* dev_status, uint64_t timeout_ns, pk_stream_t stream) {
  if (dev_status == nullptr) return PK_ERR_INVALID_ARG;
  pk_status st = check_device();
  if (st != PK_OK) return st;
  pk::dev::pk_wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      dev_status, timeout_ns ? timeout_ns : 1);
  if (cudaGetLastError() != cudaSuccess) return PK_ERR_CUDA;
  return PK_OK;
}

}  // extern "C"
