// Host planner: descriptor validation, per-row key limit, tile
// classification and the longest-work-first persistent schedule.
//
// The mask of "[RFC]: HunyuanImage 3.0 deployment" (Proposed Change, P0
// "Attention mask challenge"; "Model structure", item 1) lets position x of a
// sequence see position y iff y <= x, or x and y share x's IMAGE segment.
// Because an image segment starts at or before x, the union of the causal
// prefix and the own segment is itself a prefix of the sequence: x sees
// exactly positions [0, lim(x)] with
//     lim(x) = x                      for a text token,
//     lim(x) = (end of x's segment)-1 for an image token.
// lim never decreases along a sequence and lim(x) >= x.  A query row sees the
// prefix of its key range up to lim(x) (none if the range starts after it),
// stored as an index into the range.  The page's "block-sparse mask" option
// then becomes a per-tile classification over 128 x 128 tiles:
//   skipped  : no row of the query tile sees any key of the key tile
//              (never enumerated: the visited key tiles are a prefix),
//   full     : every valid row sees every key of the tile (no mask math),
//   partial  : anything else (per-element compare against kv_limit).
#include <algorithm>
#include <cstring>
#include <memory>
#include <new>
#include <numeric>
#include <queue>
#include <map>
#include <array>
#include <vector>

#include <cuda_runtime_api.h>

#include "pk_internal.h"

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Relative cost of a work item for the longest-processing-time schedule:
// one unit per visited key tile and query head (the CTA runs the item's two
// heads one after the other), masked tiles a little dearer, and a fixed
// per-head cost (query load, pipeline fill, epilogue).
double item_cost(const pk_work_item& w) {
  const double per_head = w.n_full * 1.0 + (w.n_kt - w.n_full) * 1.3 + 3.0;
  return w.hq1 >= 0 ? 2.0 * per_head : per_head;
}

// Longest-processing-time-first: indices sorted by decreasing cost (ties
// keep their order, so items streaming the same keys/values start side by
// side), each given to the least-loaded of `bins` bins.
std::vector<std::vector<int32_t>> lpt_schedule(const std::vector<double>& cost, int32_t bins) {
  const int32_t n = static_cast<int32_t>(cost.size());
  std::vector<int32_t> order(n);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return cost[a] > cost[b]; });
  std::vector<std::vector<int32_t>> per(bins);
  using Load = std::pair<double, int32_t>;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int32_t c = 0; c < bins; ++c) heap.push({0.0, c});
  for (int32_t idx : order) {
    Load l = heap.top();
    heap.pop();
    per[l.second].push_back(idx);
    l.first += cost[idx];
    heap.push(l);
  }
  return per;
}

// Validation of the general layout; fills seg_first[s] (first segment of s)
// and seq_len[s] (positions covered by its segments).
pk_status validate_layout(const pk_layout& L, int32_t hq, int32_t hkv, int32_t d,
                          std::vector<int32_t>& seg_first, std::vector<int32_t>& seq_len) {
  const int32_t S = L.num_seqs;
  if (S < 0 || L.num_segs < 0 || L.cu_seqlens_q == nullptr || L.cu_seqlens_k == nullptr)
    return PK_ERR_INVALID_ARG;
  if (L.num_segs > 0 && L.segs == nullptr) return PK_ERR_INVALID_ARG;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return PK_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PK_ERR_UNSUPPORTED;
  const int32_t* cq = L.cu_seqlens_q;
  const int32_t* ck = L.cu_seqlens_k;
  if (cq[0] != 0 || ck[0] != 0) return PK_ERR_INVALID_ARG;
  for (int32_t s = 0; s < S; ++s)
    if (cq[s + 1] < cq[s] || ck[s + 1] < ck[s]) return PK_ERR_INVALID_ARG;
  // Rows are addressed with int32 and tiles may overhang the end by 127.
  if (cq[S] > INT32_MAX - 2 * pk::kTileQ || L.num_kv_rows > INT32_MAX - 2 * pk::kTileK ||
      L.num_kv_rows < 0)
    return PK_ERR_INVALID_ARG;
  seg_first.assign(S, -1);
  seq_len.assign(S, 0);
  int32_t prev = -1;
  for (int32_t g = 0; g < L.num_segs; ++g) {
    const pk_seq_segment& sg = L.segs[g];
    if (sg.seq < 0 || sg.seq >= S || sg.seq < prev) return PK_ERR_INVALID_ARG;
    if (sg.len <= 0 || (sg.type != PK_TEXT && sg.type != PK_IMAGE)) return PK_ERR_INVALID_ARG;
    if (sg.start != seq_len[sg.seq] || sg.len > INT32_MAX / 2 - seq_len[sg.seq])
      return PK_ERR_INVALID_ARG;
    if (seg_first[sg.seq] < 0) seg_first[sg.seq] = g;
    seq_len[sg.seq] += sg.len;
    prev = sg.seq;
  }
  for (int32_t s = 0; s < S; ++s) {
    const int32_t q0 = L.q_pos0 ? L.q_pos0[s] : 0, k0 = L.k_pos0 ? L.k_pos0[s] : 0;
    const int32_t nq = cq[s + 1] - cq[s], nk = ck[s + 1] - ck[s];
    if (q0 < 0 || k0 < 0 || q0 > seq_len[s] - nq || k0 > seq_len[s] - nk) return PK_ERR_INVALID_ARG;
  }
  if (L.block_table != nullptr) {
    if (L.blocks_per_seq <= 0 || L.num_kv_rows % pk::kKeyBlock) return PK_ERR_INVALID_ARG;
    const int32_t pool_blocks = L.num_kv_rows / pk::kKeyBlock;
    for (int32_t s = 0; s < S; ++s) {
      const int32_t k0 = L.k_pos0 ? L.k_pos0[s] : 0, nk = ck[s + 1] - ck[s];
      if (nk == 0) continue;
      if (k0 % pk::kKeyBlock) return PK_ERR_INVALID_ARG;
      const int32_t b0 = k0 / pk::kKeyBlock, nb = (nk + pk::kKeyBlock - 1) / pk::kKeyBlock;
      if (b0 + nb > L.blocks_per_seq) return PK_ERR_INVALID_ARG;
      for (int32_t b = b0; b < b0 + nb; ++b) {
        const int32_t pb = L.block_table[(size_t)s * L.blocks_per_seq + b];
        if (pb < 0 || pb >= pool_blocks) return PK_ERR_INVALID_ARG;
      }
    }
    for (int32_t s = 0; s < S; ++s)
      if (ck[s + 1] == ck[s] && cq[s + 1] > cq[s]) {
        // rows without keys read table entry 0 (all masked): it must be valid
        if (S == 0 || L.block_table[0] < 0 || L.block_table[0] >= pool_blocks)
          return PK_ERR_INVALID_ARG;
      }
  } else if (L.num_kv_rows < ck[S]) {
    return PK_ERR_INVALID_ARG;
  }
  if (cq[S] > 0 && L.num_kv_rows == 0) return PK_ERR_INVALID_ARG;  // no key tensor to read
  return PK_OK;
}

// num_ctas 0: the current device's SM count.
pk_status resolve_num_ctas(int32_t* num_ctas) {
  if (*num_ctas < 0) return PK_ERR_INVALID_ARG;
  if (*num_ctas == 0) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0) {
      cudaGetLastError();
      return PK_ERR_CUDA;
    }
    *num_ctas = sms;
  }
  return PK_OK;
}

// SM-pair items (see pk_plan::pair_items): each item's query heads are
// taken one at a time (a pair item is one head of two query tiles, the work
// of one two-head item, so the 76 clusters get as fine a schedule as the
// 152 CTAs), and the one-head items that read the same key and value tiles
// form a group; within it, ordered by key-tile count (then first row),
// neighbours pair up, so a pair's two tiles visit about as many key tiles (a
// text tile that sees one key tile is not paired with an image tile that
// sees the whole segment).  The pairs, in the order of their groups' first
// items, are scheduled longest first over `clusters` clusters.
void schedule_pairs(pk_plan* p, const std::vector<pk_work_item>& items, int32_t clusters) {
  p->pair_items.clear();
  p->pair_cta_offsets.clear();
  p->num_clusters = 0;
  if (p->head_dim != 128 || clusters < 1 || items.empty()) return;
  using Key = std::array<int32_t, 4>;
  std::map<Key, int32_t> group_of;
  std::vector<std::vector<pk_work_item>> groups;
  for (const pk_work_item& w0 : items) {
    for (int hs = 0; hs < 2; ++hs) {  // one query head per pair item (finer schedule)
      if (hs == 1 && w0.hq1 < 0) break;
      pk_work_item w = w0;
      w.hq0 = hs ? w0.hq1 : w0.hq0;
      w.hq1 = -1;
      const Key k{w.kv_start, w.hkv, w.hq0, w.hq1};
      auto it = group_of.find(k);
      if (it == group_of.end()) {
        group_of[k] = static_cast<int32_t>(groups.size());
        groups.push_back({w});
      } else {
        groups[it->second].push_back(w);
      }
    }
  }
  std::vector<std::array<pk_work_item, 2>> pairs;
  for (std::vector<pk_work_item>& g : groups) {
    std::stable_sort(g.begin(), g.end(), [](const pk_work_item& a, const pk_work_item& b) {
      return a.n_kt != b.n_kt ? a.n_kt < b.n_kt : a.q_start < b.q_start;
    });
    for (size_t i = 0; i < g.size(); i += 2) {
      std::array<pk_work_item, 2> pr{g[i], g[i]};
      if (i + 1 < g.size()) {
        pr[1] = g[i + 1];
        pr[0].n_kt = pr[1].n_kt = std::max(g[i].n_kt, g[i + 1].n_kt);
        pr[0].n_full = pr[1].n_full = std::min(g[i].n_full, g[i + 1].n_full);
      } else {
        pr[1].q_rows = 0;  // no partner: no rows (its loads read the leader's rows)
      }
      pairs.push_back(pr);
    }
  }
  const int32_t n_pairs = static_cast<int32_t>(pairs.size());
  const int32_t grid = std::min<int32_t>(clusters, n_pairs);
  p->num_clusters = grid;
  std::vector<double> cost(n_pairs);
  for (int32_t i = 0; i < n_pairs; ++i) cost[i] = item_cost(pairs[i][0]);
  const std::vector<std::vector<int32_t>> per = lpt_schedule(cost, grid);
  p->pair_cta_offsets.assign(grid + 1, 0);
  p->pair_items.reserve(2 * static_cast<size_t>(n_pairs));
  for (int32_t c = 0; c < grid; ++c) {
    for (int32_t idx : per[c]) {
      p->pair_items.push_back(pairs[idx][0]);
      p->pair_items.push_back(pairs[idx][1]);
    }
    p->pair_cta_offsets[c + 1] = static_cast<int32_t>(p->pair_items.size() / 2);
  }
}

// Head-pair cluster items (see pk_plan::share_items): the plan's items as
// they are, each run by one cluster (a query head per CTA), scheduled
// longest first over `clusters` clusters.  None unless every item has two
// query heads.
void schedule_share(pk_plan* p, const std::vector<pk_work_item>& items, int32_t clusters) {
  p->share_items.clear();
  p->share_offsets.clear();
  p->num_share_clusters = 0;
  p->use_share = false;
  if (clusters < 1 || items.empty()) return;
  for (const pk_work_item& w : items)
    if (w.hq1 < 0) return;
  const int32_t n = static_cast<int32_t>(items.size());
  const int32_t grid = std::min<int32_t>(clusters, n);
  std::vector<double> cost(n);
  for (int32_t i = 0; i < n; ++i) cost[i] = item_cost(items[i]);
  const std::vector<std::vector<int32_t>> per = lpt_schedule(cost, grid);
  p->share_offsets.assign(grid + 1, 0);
  p->share_items.reserve(n);
  for (int32_t c = 0; c < grid; ++c) {
    for (int32_t idx : per[c]) p->share_items.push_back(items[idx]);
    p->share_offsets[c + 1] = static_cast<int32_t>(p->share_items.size());
  }
  p->num_share_clusters = grid;
  // On by default at head_dim 128, where the clusters' saved L2 reads buy
  // clock under the power limit; at 64 (half the bytes per tile) they
  // measured 1.7% slower than one CTA per SM, so they are opt-in there.
  p->use_share = p->head_dim == 128;
}

// Longest-processing-time-first schedule of `items` over `num_ctas` CTAs
// (and over num_ctas / 2 SM pairs or head-pair clusters), then the plan's
// device image.
void schedule_and_image(pk_plan* p, std::vector<pk_work_item> items, int32_t num_ctas) {
  const int32_t Tq = p->T;
  // The plan's own work: tiles visited and useful FLOPs (4 d per visible
  // (query, key) pair and query head of its items).
  p->num_full_tiles = p->num_partial_tiles = 0;
  double pairs_x_heads = 0.0;
  for (const pk_work_item& w : items) {
    p->num_full_tiles += w.n_full;
    p->num_partial_tiles += w.n_kt - w.n_full;
    int64_t pairs = 0;
    for (int32_t r = 0; r < w.q_rows; ++r) pairs += p->kv_limit[w.q_start + r] + 1;
    pairs_x_heads += static_cast<double>(pairs) * (w.hq1 >= 0 ? 2 : 1);
  }
  p->useful_flops = 4.0 * p->head_dim * pairs_x_heads;
  const int32_t n_items = static_cast<int32_t>(items.size());
  const int32_t grid = std::min<int32_t>(num_ctas, n_items);
  p->num_ctas = grid;
  std::vector<double> cost(n_items);
  for (int32_t i = 0; i < n_items; ++i) cost[i] = item_cost(items[i]);
  const std::vector<std::vector<int32_t>> per_cta = lpt_schedule(cost, grid);
  p->cta_offsets.assign(grid + 1, 0);
  p->items.reserve(n_items);
  for (int32_t c = 0; c < grid; ++c) {
    for (int32_t idx : per_cta[c]) p->items.push_back(items[idx]);
    p->cta_offsets[c + 1] = static_cast<int32_t>(p->items.size());
  }
  schedule_pairs(p, items, num_ctas / 2);
  schedule_share(p, items, num_ctas / 2);

  // Device image.
  pk::PlanImageLayout& IL = p->layout;
  IL.items_off = 0;
  IL.cta_off_off = align_up(IL.items_off + sizeof(pk_work_item) * n_items, pk::kImageAlign);
  IL.kvlim_off = align_up(IL.cta_off_off + sizeof(int32_t) * (grid + 1), pk::kImageAlign);
  IL.table_off = align_up(IL.kvlim_off + sizeof(int32_t) * static_cast<size_t>(Tq), pk::kImageAlign);
  IL.vblk_off = align_up(IL.table_off + sizeof(int32_t) * p->block_table.size(), pk::kImageAlign);
  IL.pitems_off = align_up(IL.vblk_off + sizeof(int32_t) * p->v_blocks.size(), pk::kImageAlign);
  IL.pcta_off_off =
      align_up(IL.pitems_off + sizeof(pk_work_item) * p->pair_items.size(), pk::kImageAlign);
  IL.sitems_off = align_up(IL.pcta_off_off + sizeof(int32_t) * p->pair_cta_offsets.size(),
                           pk::kImageAlign);
  IL.scta_off_off =
      align_up(IL.sitems_off + sizeof(pk_work_item) * p->share_items.size(), pk::kImageAlign);
  IL.v8chunk_off = align_up(IL.scta_off_off + sizeof(int32_t) * p->share_offsets.size(),
                            pk::kImageAlign);
  IL.v8row_off = align_up(IL.v8chunk_off + sizeof(int32_t) * p->v8_chunks.size(), pk::kImageAlign);
  // Contiguous keys: an item's key tiles sit in the E4M3 value copy at the
  // copy row of its sequence (the last sequence whose keys start at the
  // item's first key row: the non-empty one among equal starts).
  std::vector<int32_t> v8_row;
  if (!p->paged) {
    v8_row.resize(n_items);
    for (int32_t i = 0; i < n_items; ++i) {
      const int32_t s = static_cast<int32_t>(
          std::upper_bound(p->ck.begin(), p->ck.end(), p->items[i].kv_start) - p->ck.begin()) - 1;
      v8_row[i] = (s >= 0 && s < p->num_seqs) ? p->v8_seq_row[s] : 0;
    }
  }
  IL.bytes = align_up(IL.v8row_off + sizeof(int32_t) * v8_row.size(), pk::kImageAlign);
  p->image.assign(IL.bytes, 0);
  if (n_items)
    std::memcpy(p->image.data() + IL.items_off, p->items.data(), sizeof(pk_work_item) * n_items);
  std::memcpy(p->image.data() + IL.cta_off_off, p->cta_offsets.data(), sizeof(int32_t) * (grid + 1));
  if (Tq)
    std::memcpy(p->image.data() + IL.kvlim_off, p->kv_limit.data(), sizeof(int32_t) * Tq);
  if (!p->block_table.empty())
    std::memcpy(p->image.data() + IL.table_off, p->block_table.data(),
                sizeof(int32_t) * p->block_table.size());
  if (!p->v_blocks.empty())
    std::memcpy(p->image.data() + IL.vblk_off, p->v_blocks.data(),
                sizeof(int32_t) * p->v_blocks.size());
  if (!p->pair_items.empty()) {
    std::memcpy(p->image.data() + IL.pitems_off, p->pair_items.data(),
                sizeof(pk_work_item) * p->pair_items.size());
    std::memcpy(p->image.data() + IL.pcta_off_off, p->pair_cta_offsets.data(),
                sizeof(int32_t) * p->pair_cta_offsets.size());
  }
  if (!p->share_items.empty()) {
    std::memcpy(p->image.data() + IL.sitems_off, p->share_items.data(),
                sizeof(pk_work_item) * p->share_items.size());
    std::memcpy(p->image.data() + IL.scta_off_off, p->share_offsets.data(),
                sizeof(int32_t) * p->share_offsets.size());
  }
  if (!p->v8_chunks.empty())
    std::memcpy(p->image.data() + IL.v8chunk_off, p->v8_chunks.data(),
                sizeof(int32_t) * p->v8_chunks.size());
  if (!v8_row.empty())
    std::memcpy(p->image.data() + IL.v8row_off, v8_row.data(), sizeof(int32_t) * v8_row.size());
}

pk_status build_plan(const pk_layout& L, int32_t hq, int32_t hkv, int32_t d, int32_t num_ctas,
                     pk_plan** out) {
  if (out == nullptr) return PK_ERR_INVALID_ARG;
  *out = nullptr;
  std::vector<int32_t> seg_first, seq_len;
  pk_status st = validate_layout(L, hq, hkv, d, seg_first, seq_len);
  if (st != PK_OK) return st;
  if ((st = resolve_num_ctas(&num_ctas)) != PK_OK) return st;

  // Owned here until the plan is complete (the vectors below may throw).
  std::unique_ptr<pk_plan> owner(new pk_plan());
  pk_plan* p = owner.get();
  const int32_t S = L.num_seqs;
  const int32_t* cq = L.cu_seqlens_q;
  const int32_t* ck = L.cu_seqlens_k;
  const int32_t Tq = cq[S];
  p->T = Tq;
  p->Tk = L.num_kv_rows;
  p->paged = L.block_table != nullptr;
  p->blocks_per_seq = p->paged ? L.blocks_per_seq : 0;
  if (p->paged)
    p->block_table.assign(L.block_table, L.block_table + (size_t)S * L.blocks_per_seq);
  p->num_seqs = S;
  p->hq = hq;
  p->hkv = hkv;
  p->head_dim = d;

  // Per query row: last visible key of its sequence's key range, as an
  // index into that range (-1: the row sees none of it).  The key limit of
  // position x is x for text and the end of x's segment minus one for image.
  p->kv_limit.assign(Tq, -1);
  for (int32_t s = 0; s < S; ++s) {
    const int32_t nq = cq[s + 1] - cq[s], nk = ck[s + 1] - ck[s];
    if (nq == 0) continue;
    const int32_t q0 = L.q_pos0 ? L.q_pos0[s] : 0, k0 = L.k_pos0 ? L.k_pos0[s] : 0;
    int32_t g = seg_first[s];
    for (int32_t i = 0; i < nq; ++i) {
      const int32_t x = q0 + i;
      while (L.segs[g].start + L.segs[g].len <= x) ++g;
      const int32_t lim_pos =
          L.segs[g].type == PK_IMAGE ? L.segs[g].start + L.segs[g].len - 1 : x;
      const int32_t rel = std::min(lim_pos, k0 + nk - 1) - k0;
      p->kv_limit[cq[s] + i] = rel < 0 ? -1 : rel;
      p->visible_pairs += rel < 0 ? 0 : rel + 1;
    }
  }

  // Value rows the kernel reads (converted to fp16 before each launch).  For
  // paged keys: each referenced pool block with the rows of it that hold
  // keys (the rest of the block is read only as masked keys, and zeroed in
  // the copy); a tile of rows without keys reads table entry 0's block.
  if (p->paged) {
    std::vector<int32_t> valid(static_cast<size_t>(L.num_kv_rows / pk::kKeyBlock), -1);
    bool keyless_rows = false;
    for (int32_t s = 0; s < S; ++s) {
      const int32_t nk = ck[s + 1] - ck[s];
      if (nk == 0) {
        keyless_rows = keyless_rows || cq[s + 1] > cq[s];
        continue;
      }
      const int32_t k0 = L.k_pos0 ? L.k_pos0[s] : 0;
      const int32_t b0 = k0 / pk::kKeyBlock, nb = (nk + pk::kKeyBlock - 1) / pk::kKeyBlock;
      for (int32_t bb = b0; bb < b0 + nb; ++bb) {
        const int32_t pb = L.block_table[(size_t)s * L.blocks_per_seq + bb];
        const int32_t rows = std::min(pk::kKeyBlock, k0 + nk - bb * pk::kKeyBlock);
        valid[pb] = std::max(valid[pb], rows);
      }
    }
    if (keyless_rows) valid[L.block_table[0]] = std::max(valid[L.block_table[0]], 0);
    for (size_t i = 0; i < valid.size(); ++i)
      if (valid[i] >= 0) {
        p->v_blocks.push_back(static_cast<int32_t>(i));
        p->v_blocks.push_back(valid[i]);
        const int32_t row = static_cast<int32_t>(i) * pk::kKeyBlock;
        p->v8_chunks.insert(p->v8_chunks.end(), {row, row, valid[i], pk::kKeyBlock});
      }
    p->v8_rows = (p->Tk + 15) / 16 * 16;
  } else {
    p->v_conv_rows = ck[S];
    p->ck.assign(ck, ck + S + 1);
    p->v8_seq_row.assign(S, 0);
    int32_t row = 0;
    for (int32_t s = 0; s < S; ++s) {
      const int32_t nk = ck[s + 1] - ck[s];
      p->v8_seq_row[s] = row;
      for (int32_t c = 0; c < nk; c += pk::kKeyBlock) {
        const int32_t n = std::min(pk::kKeyBlock, nk - c);
        p->v8_chunks.insert(p->v8_chunks.end(), {ck[s] + c, row + c, n, (n + 15) / 16 * 16});
      }
      row += (nk + 15) / 16 * 16;
    }
    if (row == 0) {  // no keys at all: one tile of zeros for the masked reads
      p->v8_chunks.insert(p->v8_chunks.end(), {0, 0, 0, pk::kKeyBlock});
      row = pk::kKeyBlock;
    }
    p->v8_rows = row;
  }

  // Work items: every 128-row query tile x key/value head x query-head pair,
  // listed key/value head by key/value head within each sequence.  The
  // schedule keeps this order among items of equal cost, so the CTAs running
  // side by side stream the same keys and values (one head's, not all of a
  // sequence's), which then stay in L2: on the mixed-resolution pack that
  // takes 10% off the DRAM reads.
  std::vector<pk_work_item> items;
  const int32_t group = hq / hkv;
  const int32_t pairs = (group + 1) / 2;
  for (int32_t s = 0; s < S; ++s) {
    const int32_t b = cq[s], e = cq[s + 1];
    const int32_t k0 = L.k_pos0 ? L.k_pos0[s] : 0;
    for (int32_t g = 0; g < hkv; ++g) {
      for (int32_t r0 = b; r0 < e; r0 += pk::kTileQ) {
        const int32_t rows = std::min(pk::kTileQ, e - r0);
        const int32_t lim_first = p->kv_limit[r0];
        const int32_t lim_last = p->kv_limit[r0 + rows - 1];
        pk_work_item w{};
        w.q_start = r0;
        w.q_rows = rows;
        // An empty key range (every row masked) still reads one key tile: for
        // paged keys point it at table entry 0, a validated block.
        const bool no_keys = ck[s + 1] == ck[s];
        w.kv_start = p->paged ? (no_keys ? 0 : s * L.blocks_per_seq + k0 / pk::kKeyBlock) : ck[s];
        // A tile whose rows see no key still visits key tile 0 (all masked),
        // so every row's output and LSE are written by the same path.
        w.n_kt = lim_last < 0 ? 1 : lim_last / pk::kTileK + 1;
        w.n_full = std::min(w.n_kt, lim_first < 0 ? 0 : (lim_first + 1) / pk::kTileK);
        w.hkv = g;
        for (int32_t pr = 0; pr < pairs; ++pr) {
          w.hq0 = g * group + 2 * pr;
          w.hq1 = (2 * pr + 1 < group) ? w.hq0 + 1 : -1;
          items.push_back(w);
        }
      }
    }
  }

  p->cu_q.assign(cq, cq + S + 1);
  schedule_and_image(p, std::move(items), num_ctas);
  *out = owner.release();
  return PK_OK;
}

// One rank's share of a plan: the plan's work units, a (sequence, key/value
// head) pair each (all query tiles and query heads of one sequence that read
// one key/value head), go to ranks longest first, each to the least-loaded
// rank (the items' cost model), which every rank computes identically; the
// rank keeps its units' items and schedules them over its own CTAs.  The
// host data the kernel reads (key limits, block table, value rows) is the
// full plan's, so the rank's kernel runs on the full tensors and writes only
// its rows and heads of out and lse.
pk_status build_shard(const pk_plan* full, int32_t rank, int32_t num_ranks, int32_t num_ctas,
                      pk_plan** out) {
  if (out == nullptr) return PK_ERR_INVALID_ARG;
  *out = nullptr;
  if (full == nullptr || num_ranks < 1 || rank < 0 || rank >= num_ranks) return PK_ERR_INVALID_ARG;
  pk_status st = resolve_num_ctas(&num_ctas);
  if (st != PK_OK) return st;
  // units in (sequence, key/value head) order
  const int64_t n_units = static_cast<int64_t>(full->num_seqs) * full->hkv;
  std::vector<double> cost(n_units, 0.0);
  std::vector<int64_t> unit_of(full->items.size());
  for (size_t i = 0; i < full->items.size(); ++i) {
    const pk_work_item& w = full->items[i];
    const int32_t s =
        static_cast<int32_t>(std::upper_bound(full->cu_q.begin(), full->cu_q.end(), w.q_start) -
                             full->cu_q.begin()) - 1;
    unit_of[i] = static_cast<int64_t>(s) * full->hkv + w.hkv;
    cost[unit_of[i]] += item_cost(w);
  }
  std::vector<int64_t> order(n_units);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](int64_t a, int64_t b) { return cost[a] > cost[b]; });
  std::vector<int32_t> owner_of(n_units, -1);
  using Load = std::pair<double, int32_t>;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int32_t r = 0; r < num_ranks; ++r) heap.push({0.0, r});
  for (int64_t u : order) {
    if (cost[u] == 0.0) continue;  // no items
    Load l = heap.top();
    heap.pop();
    owner_of[u] = l.second;
    l.first += cost[u];
    heap.push(l);
  }
  std::unique_ptr<pk_plan> owner(new pk_plan());
  pk_plan* p = owner.get();
  p->T = full->T;
  p->Tk = full->Tk;
  p->paged = full->paged;
  p->blocks_per_seq = full->blocks_per_seq;
  p->block_table = full->block_table;
  p->num_seqs = full->num_seqs;
  p->hq = full->hq;
  p->hkv = full->hkv;
  p->head_dim = full->head_dim;
  p->visible_pairs = full->visible_pairs;
  p->kv_limit = full->kv_limit;
  p->v_conv_rows = full->v_conv_rows;
  p->v_blocks = full->v_blocks;
  p->v8_rows = full->v8_rows;
  p->v8_chunks = full->v8_chunks;
  p->ck = full->ck;
  p->v8_seq_row = full->v8_seq_row;
  p->cu_q = full->cu_q;
  p->shard_rank = rank;
  p->shard_ranks = num_ranks;
  std::vector<pk_work_item> items;
  for (size_t i = 0; i < full->items.size(); ++i)
    if (owner_of[unit_of[i]] == rank) items.push_back(full->items[i]);
  schedule_and_image(p, std::move(items), num_ctas);
  *out = owner.release();
  return PK_OK;
}

// The C entry points never let a C++ exception out: a failed host
// allocation is PK_ERR_OUT_OF_MEMORY.
template <typename F>
pk_status guarded(F&& f) {
  try {
    return f();
  } catch (const std::bad_alloc&) {
    return PK_ERR_OUT_OF_MEMORY;
  } catch (...) {
    return PK_ERR_INVALID_ARG;
  }
}

// pk_plan_create's work: global (packed-stream) segments to the
// per-sequence form of the general layout, then the planner.
pk_status create_from_global_segments(const int32_t* cu, int32_t num_seqs, const pk_segment* segs,
                                      int32_t num_segs, int32_t hq, int32_t hkv, int32_t d,
                                      int32_t num_ctas, pk_plan** out) {
  if (out == nullptr) return PK_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_seqs < 0 || num_segs < 0 || cu == nullptr || (num_segs > 0 && segs == nullptr))
    return PK_ERR_INVALID_ARG;
  if (cu[0] != 0) return PK_ERR_INVALID_ARG;
  for (int32_t s = 0; s < num_seqs; ++s)
    if (cu[s + 1] < cu[s]) return PK_ERR_INVALID_ARG;
  // Global segments -> per-sequence segments: each must tile its sequence.
  std::vector<pk_seq_segment> ss;
  ss.reserve(num_segs);
  int32_t g = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t pos = cu[s];
    while (pos < cu[s + 1]) {
      if (g >= num_segs) return PK_ERR_INVALID_ARG;
      const pk_segment& sg = segs[g];
      if (sg.start != pos || sg.len <= 0 || sg.len > cu[s + 1] - pos) return PK_ERR_INVALID_ARG;
      if (sg.type != PK_TEXT && sg.type != PK_IMAGE) return PK_ERR_INVALID_ARG;
      ss.push_back(pk_seq_segment{s, pos - cu[s], sg.len, sg.type});
      pos += sg.len;
      ++g;
    }
  }
  if (g != num_segs) return PK_ERR_INVALID_ARG;
  pk_layout L{};
  L.num_seqs = num_seqs;
  L.cu_seqlens_q = cu;
  L.cu_seqlens_k = cu;
  L.segs = ss.data();
  L.num_segs = static_cast<int32_t>(ss.size());
  L.num_kv_rows = cu[num_seqs];
  return build_plan(L, hq, hkv, d, num_ctas, out);
}

}  // namespace

extern "C" {

const char* pk_status_string(pk_status st) {
  switch (st) {
    case PK_OK: return "ok";
    case PK_ERR_INVALID_ARG: return "invalid argument";
    case PK_ERR_UNSUPPORTED: return "unsupported configuration";
    case PK_ERR_ALIGNMENT: return "misaligned tensor";
    case PK_ERR_CUDA: return "CUDA error";
    case PK_ERR_TIMEOUT: return "device wait timed out";
    case PK_ERR_DEVICE_CHECK: return "device consistency check failed";
    case PK_ERR_NOT_UPLOADED: return "plan not uploaded";
    case PK_ERR_OUT_OF_MEMORY: return "host memory allocation failed";
    case PK_ERR_RANGE: return "a value of magnitude >= 2^16 is outside the fp16 P V product's range";
    case PK_ERR_TOO_LARGE:
      return "the plan's values need more than the 64 MiB static scratch of pk_attn_fwd_noalloc";
  }
  return "unknown status";
}

pk_status pk_plan_create_layout(const pk_layout* layout, int32_t hq, int32_t hkv,
                                int32_t head_dim, int32_t num_ctas, pk_plan** out) {
  if (out) *out = nullptr;
  if (layout == nullptr) return PK_ERR_INVALID_ARG;
  return guarded([&] { return build_plan(*layout, hq, hkv, head_dim, num_ctas, out); });
}

pk_status pk_plan_create(const int32_t* cu, int32_t num_seqs, const pk_segment* segs,
                         int32_t num_segs, int32_t hq, int32_t hkv, int32_t d, int32_t num_ctas,
                         pk_plan** out) {
  return guarded([&] {
    return create_from_global_segments(cu, num_seqs, segs, num_segs, hq, hkv, d, num_ctas, out);
  });
}

pk_status pk_plan_shard(const pk_plan* full, int32_t rank, int32_t num_ranks, int32_t num_ctas,
                        pk_plan** out) {
  if (out) *out = nullptr;
  return guarded([&] { return build_shard(full, rank, num_ranks, num_ctas, out); });
}

size_t pk_plan_device_bytes(const pk_plan* p) { return p ? p->layout.bytes : 0; }

size_t pk_attn_workspace_bytes(const pk_plan* p) {
  return p ? static_cast<size_t>(p->Tk) * p->hkv * p->head_dim * 2 : 0;
}

size_t pk_attn_workspace_bytes_fp8_pv(const pk_plan* p) {
  return p ? static_cast<size_t>(p->v8_rows) * p->hkv * p->head_dim : 0;
}

pk_status pk_plan_upload(pk_plan* p, void* dev_buf, size_t bytes, pk_stream_t stream) {
  if (p == nullptr || dev_buf == nullptr) return PK_ERR_INVALID_ARG;
  if (bytes < p->layout.bytes) return PK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(dev_buf) % pk::kImageAlign) return PK_ERR_ALIGNMENT;
  if (cudaMemcpyAsync(dev_buf, p->image.data(), p->layout.bytes, cudaMemcpyHostToDevice,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  p->dev = dev_buf;
  return PK_OK;
}

void pk_plan_destroy(pk_plan* p) { delete p; }

double pk_plan_useful_flops(const pk_plan* p) { return p ? p->useful_flops : 0.0; }

pk_status pk_plan_get_info(const pk_plan* p, pk_plan_info* info) {
  if (p == nullptr || info == nullptr) return PK_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  info->total_tokens = p->T;
  info->num_seqs = p->num_seqs;
  info->hq = p->hq;
  info->hkv = p->hkv;
  info->head_dim = p->head_dim;
  info->num_items = static_cast<int32_t>(p->items.size());
  info->num_ctas = p->num_ctas;
  info->num_full_tiles = p->num_full_tiles;
  info->num_partial_tiles = p->num_partial_tiles;
  info->kv_rows = p->Tk;
  info->visible_pairs = p->visible_pairs;
  info->useful_flops = pk_plan_useful_flops(p);
  return PK_OK;
}

pk_status pk_plan_get_kv_limit(const pk_plan* p, int32_t* out, int64_t n) {
  if (p == nullptr || (out == nullptr && p->T > 0) || n < p->T) return PK_ERR_INVALID_ARG;
  if (p->T) std::memcpy(out, p->kv_limit.data(), sizeof(int32_t) * p->T);
  return PK_OK;
}

pk_status pk_plan_set_sm_pairs(pk_plan* p, int32_t enable) {
  if (p == nullptr) return PK_ERR_INVALID_ARG;
  if (enable && p->num_clusters == 0) return PK_ERR_UNSUPPORTED;
  p->use_pairs = enable != 0;
  return PK_OK;
}

pk_status pk_plan_set_kv_share(pk_plan* p, int32_t enable) {
  if (p == nullptr) return PK_ERR_INVALID_ARG;
  if (enable && p->num_share_clusters == 0) return PK_ERR_UNSUPPORTED;
  p->use_share = enable != 0;
  return PK_OK;
}

int32_t pk_plan_kv_share(const pk_plan* p) {
  return (p != nullptr && p->use_share && p->num_share_clusters > 0) ? 1 : 0;
}

pk_status pk_plan_get_share(const pk_plan* p, int32_t* num_clusters, pk_work_item* items,
                            int64_t n_items, int32_t* cluster_offsets, int64_t n_offsets) {
  if (p == nullptr || num_clusters == nullptr) return PK_ERR_INVALID_ARG;
  *num_clusters = p->num_share_clusters;
  if (items == nullptr && cluster_offsets == nullptr) return PK_OK;
  const int64_t ni = static_cast<int64_t>(p->share_items.size());
  if (items == nullptr || cluster_offsets == nullptr || n_items < ni ||
      n_offsets < static_cast<int64_t>(p->share_offsets.size()))
    return PK_ERR_INVALID_ARG;
  if (ni) std::memcpy(items, p->share_items.data(), sizeof(pk_work_item) * ni);
  if (!p->share_offsets.empty())
    std::memcpy(cluster_offsets, p->share_offsets.data(),
                sizeof(int32_t) * p->share_offsets.size());
  return PK_OK;
}

pk_status pk_plan_get_pairs(const pk_plan* p, int32_t* num_pairs, int32_t* num_clusters,
                            pk_work_item* items, int64_t n_items, int32_t* cluster_offsets,
                            int64_t n_offsets) {
  if (p == nullptr || num_pairs == nullptr || num_clusters == nullptr) return PK_ERR_INVALID_ARG;
  const int64_t ni = static_cast<int64_t>(p->pair_items.size());
  *num_pairs = static_cast<int32_t>(ni / 2);
  *num_clusters = p->num_clusters;
  if (items == nullptr && cluster_offsets == nullptr) return PK_OK;
  if (items == nullptr || cluster_offsets == nullptr || n_items < ni ||
      n_offsets < static_cast<int64_t>(p->pair_cta_offsets.size()))
    return PK_ERR_INVALID_ARG;
  if (ni) std::memcpy(items, p->pair_items.data(), sizeof(pk_work_item) * ni);
  if (!p->pair_cta_offsets.empty())
    std::memcpy(cluster_offsets, p->pair_cta_offsets.data(),
                sizeof(int32_t) * p->pair_cta_offsets.size());
  return PK_OK;
}

pk_status pk_plan_get_items(const pk_plan* p, pk_work_item* items, int64_t n_items,
                            int32_t* cta_offsets, int64_t n_offsets) {
  if (p == nullptr) return PK_ERR_INVALID_ARG;
  const int64_t ni = static_cast<int64_t>(p->items.size());
  if (n_items < ni || n_offsets < p->num_ctas + 1) return PK_ERR_INVALID_ARG;
  if ((ni && items == nullptr) || cta_offsets == nullptr) return PK_ERR_INVALID_ARG;
  if (ni) std::memcpy(items, p->items.data(), sizeof(pk_work_item) * ni);
  std::memcpy(cta_offsets, p->cta_offsets.data(), sizeof(int32_t) * (p->num_ctas + 1));
  return PK_OK;
}

}  // extern "C"
