// Internal definitions shared by the host planner and the CUDA launcher.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "pk.h"

namespace pk {

constexpr int kTileQ = 128;   // query rows per tile (tcgen05 M)
constexpr int kTileK = 128;   // keys per tile (tcgen05 N of S = Q K^T)
constexpr size_t kImageAlign = 256;

static_assert(sizeof(pk_work_item) == 32, "work item is 32 bytes");

constexpr int kKeyBlock = 128;  // rows per block of a paged key/value pool

struct PlanImageLayout {
  size_t items_off = 0;    // pk_work_item[num_items], CTA-ordered
  size_t cta_off_off = 0;  // int32[num_ctas + 1]
  size_t kvlim_off = 0;    // int32[Tq]: last visible key index of the row's key range, -1 none
  size_t table_off = 0;    // int32[num_seqs * blocks_per_seq] when keys are paged
  size_t vblk_off = 0;     // int32[v_blocks.size()]: (pool block, valid rows) the kernel reads
  size_t pitems_off = 0;   // pk_work_item[2 * num_pairs]: SM-pair items, cluster-ordered
  size_t pcta_off_off = 0; // int32[num_clusters + 1]
  size_t sitems_off = 0;   // pk_work_item[num_items]: head-pair cluster items, cluster-ordered
  size_t scta_off_off = 0; // int32[num_share_clusters + 1]
  size_t v8chunk_off = 0;  // int32[v8_chunks.size()]: the E4M3 value transpose's chunks
  size_t v8row_off = 0;    // int32[num_items] (contiguous keys): row of an item's first
                           // key tile in the transposed E4M3 value copy
  size_t bytes = 0;
};

// Upper bound of every device-side wait (pk_set_wait_timeout_ns).
uint64_t wait_limit_ns();

}  // namespace pk

struct pk_plan {
  int32_t T = 0;          // query rows (Tq)
  int32_t Tk = 0;         // rows of the key/value tensors (contiguous keys or pool)
  bool paged = false;     // keys/values read through the block table
  int32_t blocks_per_seq = 0;
  std::vector<int32_t> block_table;
  int32_t num_seqs = 0;
  int32_t hq = 0, hkv = 0, head_dim = 0;
  int32_t num_ctas = 0;
  int32_t num_full_tiles = 0, num_partial_tiles = 0;
  int64_t visible_pairs = 0;    // per query head, over the whole pack
  double useful_flops = 0.0;    // 4 d per visible pair and query head of this plan's items
  std::vector<int32_t> cu_q;    // [num_seqs + 1] query rows of each sequence
  int32_t shard_rank = 0, shard_ranks = 1;  // pk_plan_shard: this plan's share
  std::vector<int32_t> kv_limit;           // [Tq] last visible key of the row's key range, -1 none
  // Value rows the attention kernel reads, for their conversion to fp16:
  // contiguous keys, rows [0, v_conv_rows) (rows [v_conv_rows, Tk) no
  // sequence owns are zeroed in the copy); paged keys, (pool block, rows of
  // it holding keys) pairs, the block's other rows zeroed in the copy.
  int32_t v_conv_rows = 0;
  std::vector<int32_t> v_blocks;
  // The transposed E4M3 value copy (pk_attn_fwd_fp8_pv), [hkv][d][v8_rows]
  // bytes: (source row, copy row, rows holding keys, rows written) chunks of
  // at most 128 rows.  Contiguous keys: sequence s's keys start at copy row
  // v8_seq_row[s], its key count rounded up to 16 rows after the previous
  // sequence's (a tensor copy may only start on a 16-byte boundary), written
  // with zeros past the keys.  Paged keys: pool rows as they are, every
  // referenced block written whole.
  int32_t v8_rows = 0;
  std::vector<int32_t> v8_chunks;
  std::vector<int32_t> ck;          // contiguous keys: [num_seqs + 1] key row starts
  std::vector<int32_t> v8_seq_row;  // contiguous keys: [num_seqs]
  std::vector<pk_work_item> items;         // CTA-ordered
  std::vector<int32_t> cta_offsets;        // [num_ctas + 1]
  // The same work for SM pairs (head_dim 128, bf16 queries and keys): one
  // query head of two query tiles that read the same key/value tiles (same
  // first key row, key/value head and query head) per pair, run by a cluster
  // of two CTAs as M = 256 products; the pair visits the larger key-tile
  // count (the other rows see the extra tiles fully masked).  Stored as
  // consecutive (rank 0, rank 1) items with hq1 = -1; a pair without a
  // partner gets a rank-1 item with no rows.  Scheduled longest first over
  // num_clusters = num_ctas / 2 clusters.
  int32_t num_clusters = 0;
  bool use_pairs = false;                  // pk_plan_set_sm_pairs
  std::vector<pk_work_item> pair_items;    // [2 * num_pairs], cluster-ordered
  std::vector<int32_t> pair_cta_offsets;   // [num_clusters + 1], in pairs
  // The same items for head-pair clusters (every item with two query
  // heads): a cluster of two CTAs on neighbouring SMs runs each of
  // its items with one query head per CTA, the two CTAs streaming the same
  // key/value tiles, each copying half of every tile into both.  Scheduled
  // longest first over num_share_clusters = num_ctas / 2 clusters; the
  // default kernel at head_dim 128 wherever the schedule exists, opt-in at
  // 64 (pk_plan_set_kv_share).
  int32_t num_share_clusters = 0;
  bool use_share = false;
  std::vector<pk_work_item> share_items;   // [num_items], cluster-ordered
  std::vector<int32_t> share_offsets;      // [num_share_clusters + 1]
  pk::PlanImageLayout layout;
  std::vector<uint8_t> image;              // host copy of the device image
  void* dev = nullptr;                     // caller's buffer after upload
};
