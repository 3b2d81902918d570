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

struct PlanImageLayout {
  size_t items_off = 0;    // pk_work_item[num_items], CTA-ordered
  size_t cta_off_off = 0;  // int32[num_ctas + 1]
  size_t kvlim_off = 0;    // int32[T]
  size_t bytes = 0;
};

}  // namespace pk

struct pk_plan {
  int32_t T = 0;
  int32_t num_seqs = 0;
  int32_t hq = 0, hkv = 0, head_dim = 0;
  int32_t num_ctas = 0;
  int32_t num_full_tiles = 0, num_partial_tiles = 0;
  int64_t visible_pairs = 0;
  std::vector<int32_t> kv_limit;           // [T] global index of last visible key
  std::vector<pk_work_item> items;         // CTA-ordered
  std::vector<int32_t> cta_offsets;        // [num_ctas + 1]
  pk::PlanImageLayout layout;
  std::vector<uint8_t> image;              // host copy of the device image
  void* dev = nullptr;                     // caller's buffer after upload
};
