// Merge of partial attention results by their log-sum-exp.
//
// Ring attention ("Parallelism Acceleration Guide", Ring Attention) splits
// the keys of a sequence into blocks that visit the queries one step at a
// time; every step yields, per query row and head, the softmax-weighted
// output over that key block and the natural-log LSE of its scores.  The
// attention over the union of disjoint key blocks follows from the parts
// alone:
//   lse = ln sum_c exp(lse_c)
//   out = sum_c exp(lse_c - lse) * o_c
// A part whose row saw no key (lse_c = -inf) contributes nothing; a row
// that no part saw gets out = 0 and lse = -inf.
//
// HBM-bound streaming.  The common case (up to four bf16 or fp32 parts,
// head dim >= 64) runs a staged kernel: one CTA per SM, one producer warp
// that moves chunks of consecutive rows of every part into a ring of shared
// memory stages with bulk asynchronous copies (and the rows' LSEs with
// 4-byte asynchronous copies) completing on the stage's mbarrier, and twelve
// consumer warps (three per SM sub-partition, to hide the arithmetic's
// latencies) that merge a stage and write the result with 16-byte stores.
// Up to ~200 KB per SM are in flight, which is what HBM3e needs.  Every
// other case (more parts, smaller head dims) runs a register kernel: a row's
// d values in 16-byte chunks, one per thread, so a warp covers 32 / (d / 8)
// whole rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "pk_internal.h"
#include "sync.cuh"

namespace pk {
namespace merge {

constexpr int kMaxParts = 16;
constexpr int kThreads = 256;

struct Params {
  const uint8_t* o[kMaxParts];
  const float* lse[kMaxParts];
  int32_t f32[kMaxParts];  // part dtype: 1 fp32, 0 bf16
  int32_t num_parts;
  int32_t T, H, d;
  int64_t rows;            // T * H
  uint8_t* out;
  int32_t out_f32;
  float* lse_out;
  int32_t* status;         // device status word for a timed-out wait, may be null
  uint64_t wait_ns;
  // staged kernel: stage layout (bytes), set on the host from the parts' types
  int32_t st_bytes, n_stages, lse_off;
  int32_t part_off[kMaxParts];
};

__device__ __forceinline__ void load8(const uint8_t* base, bool f32, int64_t elem, float (&x)[8]) {
  if (f32) {
    const float4* p = reinterpret_cast<const float4*>(base + elem * 4);
    const float4 a = p[0], b = p[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(base + elem * 2);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

__device__ __forceinline__ void store8(uint8_t* base, bool f32, int64_t elem, const float (&x)[8]) {
  if (f32) {
    float4* p = reinterpret_cast<float4*>(base + elem * 4);
    p[0] = make_float4(x[0], x[1], x[2], x[3]);
    p[1] = make_float4(x[4], x[5], x[6], x[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(base + elem * 2) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Register kernel.  NP: compile-time bound on the parts (the runtime count
// is <= NP), so the per-row work is exactly the parts present.
template <int NP>
__global__ void __launch_bounds__(kThreads) lse_merge_kernel(const Params p) {
  const int lane = threadIdx.x & 31;
  const int tpr = p.d >> 3;            // threads per row (divides 32)
  const int rpw = 32 / tpr;            // rows per warp
  const int sub = lane / tpr, chunk = lane - sub * tpr;
  const uint32_t warps = gridDim.x * (kThreads / 32);
  const uint32_t gw = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  const uint32_t rows = (uint32_t)p.rows, H = (uint32_t)p.H;
  constexpr float kLog2e = 1.4426950408889634f;
  for (uint32_t base = gw * rpw; base < rows; base += warps * rpw) {
    // Every lane of the warp runs the same trip count (base is warp-uniform).
    const uint32_t row = base + sub;
    const bool valid = row < rows;
    const uint32_t t = valid ? row / H : 0u;
    const uint32_t h = valid ? row - t * H : 0u;
    const size_t li = (size_t)h * (size_t)p.T + t;
    const size_t elem = (size_t)row * (size_t)p.d + (size_t)(chunk * 8);
    float w[NP], m = -INFINITY;
    bool nan = false;
#pragma unroll
    for (int c = 0; c < NP; ++c) {
      w[c] = (valid && c < p.num_parts) ? p.lse[c][li] : -INFINITY;
      nan |= w[c] != w[c];
      m = fmaxf(m, w[c]);
    }
    if (nan) m = __int_as_float(0x7fc00000);  // a NaN LSE poisons the row
    float x[NP][8];
#pragma unroll
    for (int c = 0; c < NP; ++c) {  // all loads first, then the arithmetic
      w[c] = m > -INFINITY ? exp2f((w[c] - m) * kLog2e) : 0.f;  // 0: empty part
      if (w[c] > 0.f) load8(p.o[c], p.f32[c] != 0, elem, x[c]);
    }
    float acc[8], wsum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int c = 0; c < NP; ++c) {
      if (w[c] > 0.f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(w[c], x[c][i], acc[i]);
        wsum += w[c];
      }
    }
    if (m > -INFINITY) {
      const float inv = 1.0f / wsum;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] *= inv;
    } else if (nan) {
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = m;
    }
    if (valid) store8(p.out, p.out_f32 != 0, elem, acc);
    // The LSE output may alias a part's LSE: every lane of the row has read
    // it before one lane writes it.
    __syncwarp();
    if (valid && chunk == 0) p.lse_out[li] = m > -INFINITY ? m + logf(wsum) : m;
  }
}

// ---------------------------------------------------------------------------
// Staged kernel (up to 4 parts, bf16 or fp32 each, d in {64, 128, 256}).
// Rows per stage: 48 at d = 128 (96 at 64, 24 at 256), so the twelve
// consumer warps each take the same share of a stage; a bf16 part's rows
// are 12 KB of a stage, an fp32 part's 24 KB.
constexpr int kChunkBytes = 12288;
constexpr int kBulkConsumerWarps = 12;
constexpr int kBulkThreads = 32 * (1 + kBulkConsumerWarps);
constexpr int kMaxStages = 16;
constexpr int kStageBudget = 200 * 1024;
// Shared memory after the stages: full and empty barriers of kMaxStages
// stages, abort flag, issued count.
constexpr int kBulkTail = 2 * kMaxStages * 8 + 16;

// 2^x on the SFU (relative error ~2^-22): weights of parts whose LSE lies
// below the row maximum.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Stage layout when the parts' element types are known at compile time:
// bit c of kMask set means part c is fp32 (its rows of a chunk take twice
// the bytes of bf16 rows); the parts' rows one after another, then the LSEs.
template <int NP, int kMask>
struct StageLayout {
  __host__ __device__ static constexpr int part_bytes(int c) { return ((kMask >> c) & 1) ? 2 * kChunkBytes : kChunkBytes; }
  __host__ __device__ static constexpr int part_off(int c) {
    int o = 0;
    for (int i = 0; i < c; ++i) o += part_bytes(i);
    return o;
  }
  static constexpr int kLseOff = part_off(NP);
  static constexpr int kStBytes = (kLseOff + NP * (kChunkBytes / 128) * 4 + 127) & ~127;
  static constexpr int kStagesFit = kStageBudget / kStBytes;
  static constexpr int kStages = kStagesFit < kMaxStages ? kStagesFit : kMaxStages;
  static constexpr int kSmem = kStages * kStBytes + kBulkTail;
  static_assert(kStages >= 2 && kSmem <= 227 * 1024, "shared memory budget");
};

// kMask >= 0: the parts' element types (bit c: part c is fp32) are known at
// compile time, and so are the stage layout and every element size;
// kMask < 0: they come from Params.
template <int NP, bool kOutF32, int kMask>
__global__ void __launch_bounds__(kBulkThreads, 1) lse_merge_bulk_kernel(const Params p) {
  using namespace pk::dev;
  constexpr bool kFixed = kMask >= 0;
  using BL = StageLayout<NP, kFixed ? kMask : 0>;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t n_stages = kFixed ? (uint32_t)BL::kStages : (uint32_t)p.n_stages;
  const uint32_t st_bytes = kFixed ? (uint32_t)BL::kStBytes : (uint32_t)p.st_bytes;
  const uint32_t off_bar = n_stages * st_bytes;
  auto is_f32 = [&](int c) { return kFixed ? ((kMask >> c) & 1) != 0 : p.f32[c] != 0; };
  auto stage_o = [&](uint32_t s, int c) {
    return s * st_bytes + (kFixed ? (uint32_t)BL::part_off(c) : (uint32_t)p.part_off[c]);
  };
  auto stage_l = [&](uint32_t s, int c) {
    return s * st_bytes + (kFixed ? (uint32_t)BL::kLseOff : (uint32_t)p.lse_off) +
           (uint32_t)c * (kChunkBytes / 128) * 4u;
  };
  auto full = [&](uint32_t s) { return sbase + off_bar + 8u * s; };
  auto empty = [&](uint32_t s) { return sbase + off_bar + 8u * ((uint32_t)kMaxStages + s); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + off_bar + 2 * kMaxStages * 8);
  uint32_t* issued_count = reinterpret_cast<uint32_t*>(smem + off_bar + 2 * kMaxStages * 8 + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rpc = kChunkBytes / (2 * p.d);    // rows per chunk
  const uint32_t rows = (uint32_t)p.rows, H = (uint32_t)p.H;
  const uint32_t nchunks = (rows + rpc - 1) / rpc;
  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < n_stages; ++s) {
      mbar_init(full(s), 1 + 32);  // expect_tx arrival + every producer lane's LSE copies
      mbar_init(empty(s), kBulkConsumerWarps);
    }
    *abort_flag = 0;
    *issued_count = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const WaitCtl wc{abort_flag, p.status, p.wait_ns};
  const int np = p.num_parts;

  if (warp == 0) {
    // Producer warp: lane 0 moves the outputs, every lane some of the LSEs.
    uint32_t i = 0;
    for (uint32_t k = blockIdx.x; k < nchunks; k += gridDim.x, ++i) {
      const uint32_t s = i % n_stages;
      const uint32_t n = i / n_stages;
      if (n > 0 && !__all_sync(0xffffffffu, mbar_wait(empty(s), (n - 1) & 1u, wc))) break;
      const uint32_t r0 = k * rpc;
      const uint32_t nr = rows - r0 < rpc ? rows - r0 : rpc;
      if (lane == 0) {
        const uint32_t row_elems = nr * (uint32_t)p.d;
        uint32_t total = 0;
#pragma unroll
        for (int c = 0; c < NP; ++c)
          if (c < np) total += row_elems * (is_f32(c) ? 4u : 2u);
        mbar_arrive_expect_tx(full(s), total);
#pragma unroll
        for (int c = 0; c < NP; ++c)
          if (c < np) {
            const uint32_t eb = is_f32(c) ? 4u : 2u;
            bulk_g2s(sbase + stage_o(s, c), p.o[c] + (size_t)r0 * (size_t)p.d * eb,
                     row_elems * eb, full(s));
          }
      }
      for (uint32_t r = lane; r < nr; r += 32) {
        const uint32_t row = r0 + r, t = row / H, h = row - t * H;
        const size_t li = (size_t)h * (size_t)p.T + t;
#pragma unroll
        for (int c = 0; c < NP; ++c)
          if (c < np) cp_async4(sbase + stage_l(s, c) + 4u * r, p.lse[c] + li);
      }
      cp_async_arrive(full(s));
    }
    if (lane == 0) *issued_count = i;
  } else {
    // Consumer warps: merge the rows of a stage.  A thread takes 16 values
    // of a row, the 8 at chunk * 8 and the 8 at d / 2 + chunk * 8, so each
    // 16-byte shared load and global store of a warp is contiguous; the
    // per-row work (weights, reciprocal, LSE) is shared by d / 16 lanes.
    const int cw = warp - 1;
    const int tpr = p.d >> 4, rpw = 32 / tpr;
    const int sub = lane / tpr, chunk = lane - sub * tpr;
    const uint32_t half = (uint32_t)p.d >> 1;
    constexpr float kLog2e = 1.4426950408889634f;
    uint32_t i = 0;
    for (uint32_t k = blockIdx.x; k < nchunks; k += gridDim.x, ++i) {
      const uint32_t s = i % n_stages;
      if (!__all_sync(0xffffffffu, mbar_wait(full(s), (i / n_stages) & 1u, wc))) break;
      const uint32_t r0 = k * rpc;
      const uint32_t nr = rows - r0 < rpc ? rows - r0 : rpc;
      for (uint32_t rb = (uint32_t)(cw * rpw); rb < nr; rb += (uint32_t)(kBulkConsumerWarps * rpw)) {
        const uint32_t r = rb + (uint32_t)sub;  // rb is warp-uniform
        const bool valid = r < nr;
        float w[NP], m = -INFINITY;
        bool nan = false;
#pragma unroll
        for (int c = 0; c < NP; ++c) {
          w[c] = (valid && c < np) ? *reinterpret_cast<const float*>(smem + stage_l(s, c) + 4u * r)
                                   : -INFINITY;
          nan |= w[c] != w[c];
          m = fmaxf(m, w[c]);
        }
        if (nan) m = __int_as_float(0x7fc00000);
        float acc[16], wsum = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.f;
        const uint32_t e_off = r * (uint32_t)p.d + (uint32_t)chunk * 8u;  // element offset
#pragma unroll
        for (int c = 0; c < NP; ++c) {
          w[c] = m > -INFINITY ? ex2_approx((w[c] - m) * kLog2e) : 0.f;
          if (w[c] > 0.f) {
            if (is_f32(c)) {
              const float4* src = reinterpret_cast<const float4*>(smem + stage_o(s, c) + e_off * 4u);
              const float4* src2 = reinterpret_cast<const float4*>(smem + stage_o(s, c) + (e_off + half) * 4u);
              const float4 x[4] = {src[0], src[1], src2[0], src2[1]};
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                acc[4 * q4 + 0] = fmaf(w[c], x[q4].x, acc[4 * q4 + 0]);
                acc[4 * q4 + 1] = fmaf(w[c], x[q4].y, acc[4 * q4 + 1]);
                acc[4 * q4 + 2] = fmaf(w[c], x[q4].z, acc[4 * q4 + 2]);
                acc[4 * q4 + 3] = fmaf(w[c], x[q4].w, acc[4 * q4 + 3]);
              }
            } else {
              const uint8_t* src = smem + stage_o(s, c) + e_off * 2u;
              const uint4 u0 = *reinterpret_cast<const uint4*>(src);
              const uint4 u1 = *reinterpret_cast<const uint4*>(src + half * 2u);
              const uint32_t b[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                acc[2 * e] = fmaf(w[c], __uint_as_float(b[e] << 16), acc[2 * e]);
                acc[2 * e + 1] = fmaf(w[c], __uint_as_float(b[e] & 0xffff0000u), acc[2 * e + 1]);
              }
            }
            wsum += w[c];
          }
        }
        if (m > -INFINITY) {
          const float inv = __fdividef(1.0f, wsum);  // wsum in [1, NP]
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] *= inv;
        } else if (nan) {
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] = m;
        }
        const uint32_t row = r0 + r;
        if (valid) {
          const size_t e0 = (size_t)row * (size_t)p.d + (size_t)chunk * 8;
          store8(p.out, kOutF32, e0, *reinterpret_cast<const float(*)[8]>(acc));
          store8(p.out, kOutF32, e0 + half, *reinterpret_cast<const float(*)[8]>(acc + 8));
        }
        if (valid && chunk == 0) {
          const uint32_t t = row / H, h = row - t * H;
          p.lse_out[(size_t)h * (size_t)p.T + t] = m > -INFINITY ? m + __logf(wsum) : m;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(s));
    }
  }
  __syncthreads();
  // On a timeout some copies may still be in flight into this CTA's shared
  // memory: wait (bounded) for every stage's latest use before exiting.
  if (threadIdx.x == 0 && *abort_flag) {
    const uint32_t n = *issued_count;
    const uint32_t first = n > n_stages ? n - n_stages : 0u;
    for (uint32_t j = first; j < n; ++j)
      mbar_wait_drain(full(j % n_stages), (j / n_stages) & 1u, wc);
  }
}

int sm_count() {
  static std::mutex mu;
  static int cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

// One wave of persistent blocks: as many as fit on every SM at once.
template <int NP>
pk_status launch_regs(const Params& p, int64_t rows, int sms, cudaStream_t st) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lse_merge_kernel<NP>, kThreads, 0) !=
          cudaSuccess || per_sm <= 0) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  const int64_t rows_per_block = (int64_t)(kThreads / 32) * (32 / (p.d / 8));
  const int64_t need = (rows + rows_per_block - 1) / rows_per_block;
  const int64_t cap = (int64_t)sms * per_sm;
  lse_merge_kernel<NP><<<(int)(need < cap ? need : cap), kThreads, 0, st>>>(p);
  if (cudaGetLastError() != cudaSuccess) return PK_ERR_CUDA;
  return PK_OK;
}

// Stage layout from the parts' element types: each part's rows of a chunk
// (bf16 or fp32) one after another, then every part's LSEs.
template <int NP, bool kOutF32, int kMask>
pk_status launch_bulk(Params p, int64_t rows, int sms, cudaStream_t st) {
  const int rpc = kChunkBytes / (2 * p.d);
  int smem = StageLayout<NP, kMask >= 0 ? kMask : 0>::kSmem;
  if (kMask < 0) {
    int off = 0;
    for (int c = 0; c < p.num_parts; ++c) {
      p.part_off[c] = off;
      off += rpc * p.d * (p.f32[c] ? 4 : 2);
    }
    p.lse_off = off;
    p.st_bytes = (off + p.num_parts * (kChunkBytes / 128) * 4 + 127) & ~127;
    p.n_stages = kStageBudget / p.st_bytes;
    if (p.n_stages > kMaxStages) p.n_stages = kMaxStages;
    if (p.n_stages < 2) return PK_ERR_UNSUPPORTED;
    smem = p.n_stages * p.st_bytes + kBulkTail;
  }
  auto kern = lse_merge_bulk_kernel<NP, kOutF32, kMask>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  const int64_t chunks = (rows + rpc - 1) / rpc;
  kern<<<(int)(chunks < sms ? chunks : sms), kBulkThreads, smem, st>>>(p);
  if (cudaGetLastError() != cudaSuccess) return PK_ERR_CUDA;
  return PK_OK;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

}  // namespace merge
}  // namespace pk

extern "C" pk_status pk_lse_merge(const pk_merge_part* parts, int32_t num_parts, int32_t T,
                                  int32_t H, int32_t d, void* out, int32_t out_dtype,
                                  float* lse_out, pk_stream_t stream, int32_t* dev_status) {
  using namespace pk::merge;
  if (parts == nullptr || num_parts < 1 || T < 0 || H <= 0 || out == nullptr || lse_out == nullptr)
    return PK_ERR_INVALID_ARG;
  if (num_parts > kMaxParts) return PK_ERR_UNSUPPORTED;
  if (d <= 0 || d % 8 != 0 || 32 % (d / 8) != 0) return PK_ERR_UNSUPPORTED;
  if (out_dtype != PK_DTYPE_BF16 && out_dtype != PK_DTYPE_F32) return PK_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(lse_out, 4)) return PK_ERR_ALIGNMENT;
  Params p{};
  for (int c = 0; c < num_parts; ++c) {
    if (parts[c].o == nullptr || parts[c].lse == nullptr) return PK_ERR_INVALID_ARG;
    if (parts[c].dtype != PK_DTYPE_BF16 && parts[c].dtype != PK_DTYPE_F32) return PK_ERR_INVALID_ARG;
    if (!aligned(parts[c].o, 16) || !aligned(parts[c].lse, 4)) return PK_ERR_ALIGNMENT;
    p.o[c] = static_cast<const uint8_t*>(parts[c].o);
    p.lse[c] = parts[c].lse;
    p.f32[c] = parts[c].dtype == PK_DTYPE_F32;
  }
  const int64_t rows = (int64_t)T * H;
  if (rows == 0) return PK_OK;
  if (rows > (int64_t)INT32_MAX - 1024) return PK_ERR_INVALID_ARG;  // 32-bit row index
  p.num_parts = num_parts;
  p.T = T;
  p.H = H;
  p.d = d;
  p.rows = rows;
  p.out = static_cast<uint8_t*>(out);
  p.out_f32 = out_dtype == PK_DTYPE_F32;
  p.lse_out = lse_out;
  p.status = dev_status;
  p.wait_ns = pk::wait_limit_ns();
  const int sms = sm_count();
  if (sms <= 0) return PK_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (d >= 64 && num_parts <= 4) {
    const bool f = p.out_f32 != 0;
    bool bf16 = true;
    for (int c = 0; c < num_parts; ++c) bf16 = bf16 && !p.f32[c];
    if (bf16) {
      if (num_parts == 1) return f ? launch_bulk<1, true, 0>(p, rows, sms, st) : launch_bulk<1, false, 0>(p, rows, sms, st);
      if (num_parts == 2) return f ? launch_bulk<2, true, 0>(p, rows, sms, st) : launch_bulk<2, false, 0>(p, rows, sms, st);
      return f ? launch_bulk<4, true, 0>(p, rows, sms, st) : launch_bulk<4, false, 0>(p, rows, sms, st);
    }
    // A ring step: a running fp32 accumulator folded with one bf16 block.
    if (num_parts == 2 && p.f32[0] && !p.f32[1] && f) return launch_bulk<2, true, 1>(p, rows, sms, st);
    if (num_parts <= 2) return f ? launch_bulk<2, true, -1>(p, rows, sms, st) : launch_bulk<2, false, -1>(p, rows, sms, st);
    return f ? launch_bulk<4, true, -1>(p, rows, sms, st) : launch_bulk<4, false, -1>(p, rows, sms, st);
  }
  if (num_parts <= 2) return launch_regs<2>(p, rows, sms, st);
  if (num_parts <= 4) return launch_regs<4>(p, rows, sms, st);
  if (num_parts <= 8) return launch_regs<8>(p, rows, sms, st);
  return launch_regs<16>(p, rows, sms, st);
}
