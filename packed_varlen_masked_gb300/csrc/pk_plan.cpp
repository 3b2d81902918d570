// Host planner: descriptor validation, per-token key limit, tile
// classification and the longest-work-first persistent schedule.
//
// The mask of "[RFC]: HunyuanImage 3.0 deployment" (Proposed Change, P0
// "Attention mask challenge"; "Model structure", item 1) lets query i of a
// sequence see key j iff j <= i, or i and j share i's IMAGE segment.  Because
// an image segment starts at or before i, the union of the causal prefix and
// the own segment is itself a prefix of the sequence: row i sees exactly keys
// [seq_start, kv_limit[i]] with
//     kv_limit[i] = i                      for a text token,
//     kv_limit[i] = (end of i's segment)-1 for an image token.
// kv_limit never decreases along a sequence and kv_limit[i] >= i, so every
// row sees at least the sequence's first key.  The page's "block-sparse mask"
// option then becomes a per-tile classification over 128 x 128 tiles:
//   skipped  : no row of the query tile sees any key of the key tile
//              (never enumerated: the visited key tiles are a prefix),
//   full     : every valid row sees every key of the tile (no mask math),
//   partial  : anything else (per-element compare against kv_limit).
#include <algorithm>
#include <cstring>
#include <new>
#include <numeric>
#include <queue>
#include <vector>

#include <cuda_runtime_api.h>

#include "pk_internal.h"

namespace {

pk_status validate(const int32_t* cu, int32_t num_seqs, const pk_segment* segs,
                   int32_t num_segs, int32_t hq, int32_t hkv, int32_t d) {
  if (num_seqs < 0 || num_segs < 0 || cu == nullptr) return PK_ERR_INVALID_ARG;
  if (num_segs > 0 && segs == nullptr) return PK_ERR_INVALID_ARG;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return PK_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PK_ERR_UNSUPPORTED;
  if (cu[0] != 0) return PK_ERR_INVALID_ARG;
  for (int32_t s = 0; s < num_seqs; ++s)
    if (cu[s + 1] < cu[s]) return PK_ERR_INVALID_ARG;
  // Tokens are addressed with int32 and tiles may overhang the end by 127.
  if (cu[num_seqs] > INT32_MAX - 2 * pk::kTileQ) return PK_ERR_INVALID_ARG;
  int32_t g = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t pos = cu[s];
    while (pos < cu[s + 1]) {
      if (g >= num_segs) return PK_ERR_INVALID_ARG;
      const pk_segment& sg = segs[g];
      if (sg.start != pos || sg.len <= 0) return PK_ERR_INVALID_ARG;
      if (sg.type != PK_TEXT && sg.type != PK_IMAGE) return PK_ERR_INVALID_ARG;
      if (sg.len > cu[s + 1] - pos) return PK_ERR_INVALID_ARG;
      pos += sg.len;
      ++g;
    }
  }
  if (g != num_segs) return PK_ERR_INVALID_ARG;
  return PK_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Relative cost of a work item for the longest-processing-time schedule:
// one unit per visited key tile, masked tiles a little dearer, a fixed
// per-item cost (query loads, pipeline fill, epilogue), and single-slot items
// doing half of the tensor work.
double item_cost(const pk_work_item& w) {
  double c = w.n_full * 1.0 + (w.n_kt - w.n_full) * 1.3 + 3.0;
  return w.hq1 >= 0 ? c : 0.55 * c;
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
  }
  return "unknown status";
}

pk_status pk_plan_create(const int32_t* cu, int32_t num_seqs,
                         const pk_segment* segs, int32_t num_segs, int32_t hq,
                         int32_t hkv, int32_t d, int32_t num_ctas,
                         pk_plan** out) {
  if (out == nullptr) return PK_ERR_INVALID_ARG;
  *out = nullptr;
  pk_status st = validate(cu, num_seqs, segs, num_segs, hq, hkv, d);
  if (st != PK_OK) return st;
  if (num_ctas < 0) return PK_ERR_INVALID_ARG;
  if (num_ctas == 0) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0) {
      cudaGetLastError();
      return PK_ERR_CUDA;
    }
    num_ctas = sms;
  }

  pk_plan* p = new (std::nothrow) pk_plan();
  if (p == nullptr) return PK_ERR_INVALID_ARG;
  const int32_t T = cu[num_seqs];
  p->T = T;
  p->num_seqs = num_seqs;
  p->hq = hq;
  p->hkv = hkv;
  p->head_dim = d;

  // Per-token key limit (global index of the last visible key).
  p->kv_limit.resize(T);
  for (int32_t g = 0; g < num_segs; ++g) {
    const pk_segment& sg = segs[g];
    for (int32_t t = sg.start; t < sg.start + sg.len; ++t)
      p->kv_limit[t] = sg.type == PK_IMAGE ? sg.start + sg.len - 1 : t;
  }

  // Work items: every 128-row query tile x key/value head x query-head pair.
  std::vector<pk_work_item> items;
  const int32_t group = hq / hkv;
  const int32_t pairs = (group + 1) / 2;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t b = cu[s], e = cu[s + 1];
    for (int32_t t = b; t < e; ++t) p->visible_pairs += p->kv_limit[t] - b + 1;
    for (int32_t q0 = b; q0 < e; q0 += pk::kTileQ) {
      const int32_t rows = std::min(pk::kTileQ, e - q0);
      const int32_t lim_first = p->kv_limit[q0];
      const int32_t lim_last = p->kv_limit[q0 + rows - 1];
      pk_work_item w{};
      w.q_start = q0;
      w.q_rows = rows;
      w.kv_start = b;
      w.n_kt = (lim_last - b) / pk::kTileK + 1;
      w.n_full = std::min(w.n_kt, (lim_first - b + 1) / pk::kTileK);
      for (int32_t g = 0; g < hkv; ++g) {
        for (int32_t pr = 0; pr < pairs; ++pr) {
          w.hkv = g;
          w.hq0 = g * group + 2 * pr;
          w.hq1 = (2 * pr + 1 < group) ? w.hq0 + 1 : -1;
          items.push_back(w);
          p->num_full_tiles += w.n_full;
          p->num_partial_tiles += w.n_kt - w.n_full;
        }
      }
    }
  }

  // Longest-processing-time-first: sort by cost (ties keep pack order so
  // items streaming the same keys/values start side by side), then give each
  // item to the least-loaded CTA.
  const int32_t n_items = static_cast<int32_t>(items.size());
  const int32_t grid = std::min<int32_t>(num_ctas, n_items);
  p->num_ctas = grid;
  std::vector<int32_t> order(n_items);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b2) {
    return item_cost(items[a]) > item_cost(items[b2]);
  });
  std::vector<std::vector<int32_t>> per_cta(grid);
  using Load = std::pair<double, int32_t>;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int32_t c = 0; c < grid; ++c) heap.push({0.0, c});
  for (int32_t idx : order) {
    Load l = heap.top();
    heap.pop();
    per_cta[l.second].push_back(idx);
    l.first += item_cost(items[idx]);
    heap.push(l);
  }
  p->cta_offsets.assign(grid + 1, 0);
  p->items.reserve(n_items);
  for (int32_t c = 0; c < grid; ++c) {
    for (int32_t idx : per_cta[c]) p->items.push_back(items[idx]);
    p->cta_offsets[c + 1] = static_cast<int32_t>(p->items.size());
  }

  // Device image.
  pk::PlanImageLayout& L = p->layout;
  L.items_off = 0;
  L.cta_off_off = align_up(L.items_off + sizeof(pk_work_item) * n_items, pk::kImageAlign);
  L.kvlim_off = align_up(L.cta_off_off + sizeof(int32_t) * (grid + 1), pk::kImageAlign);
  L.bytes = align_up(L.kvlim_off + sizeof(int32_t) * static_cast<size_t>(T), pk::kImageAlign);
  p->image.assign(L.bytes, 0);
  if (n_items)
    std::memcpy(p->image.data() + L.items_off, p->items.data(), sizeof(pk_work_item) * n_items);
  std::memcpy(p->image.data() + L.cta_off_off, p->cta_offsets.data(), sizeof(int32_t) * (grid + 1));
  if (T)
    std::memcpy(p->image.data() + L.kvlim_off, p->kv_limit.data(), sizeof(int32_t) * T);

  *out = p;
  return PK_OK;
}

size_t pk_plan_device_bytes(const pk_plan* p) { return p ? p->layout.bytes : 0; }

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

double pk_plan_useful_flops(const pk_plan* p) {
  return p ? 4.0 * p->head_dim * p->hq * static_cast<double>(p->visible_pairs) : 0.0;
}

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
  info->visible_pairs = p->visible_pairs;
  info->useful_flops = pk_plan_useful_flops(p);
  return PK_OK;
}

pk_status pk_plan_get_kv_limit(const pk_plan* p, int32_t* out, int64_t n) {
  if (p == nullptr || (out == nullptr && p->T > 0) || n < p->T) return PK_ERR_INVALID_ARG;
  if (p->T) std::memcpy(out, p->kv_limit.data(), sizeof(int32_t) * p->T);
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
