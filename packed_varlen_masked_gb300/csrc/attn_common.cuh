// Device helpers shared by the attention kernels: tcgen05 instruction and
// shared-memory descriptors, MMA issue, TMA copies with L2 policies, the
// packed fp32 / bf16 arithmetic of the softmax, and the launch parameters.
#pragma once
#include <cuda.h>
#include <cstdint>

#include "pk_internal.h"

namespace pk {
namespace dev {

constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 bf16
// Growth of a row's maximum (log2 units) tolerated before O and l are
// rescaled: exponentials run against a stale maximum while it lags by less,
// so p <= 2^15, within fp16's largest finite value (65504).
constexpr float kRescaleLog2 = 15.0f;


// Instruction descriptors of tcgen05.mma kind::f16 (dense, f32 accumulate,
// bf16 A and B): bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16),
// 10-12 B format (1 = bf16), 15/16 A/B major (0 = K-major, 1 = MN-major),
// 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The same for fp16 A and B (format code 0 in bits 7-9 and 10-12).
__host__ __device__ constexpr uint32_t make_idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// kind::f8f6f4 with A and B both FP8 E4M3 (format code 0 in bits 7-9 and
// 10-12), f32 accumulate, both K-major.
__host__ __device__ constexpr uint32_t make_idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor (tcgen05 form): start address, leading and
// stride byte offsets (all >> 4), version 1 at bit 46, 128-byte swizzle (2)
// at bits 61-63.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// A 3-D tensor copy into shared memory, completing on barrier `bar`, with an
// L2 eviction-priority policy (from createpolicy).
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int c0, int c1, int c2,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// D(tmem) (+)= A(smem desc) * B(smem desc)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D(tmem) (+)= A(smem desc) * B(smem desc), FP8 operands.
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem desc), FP8 operands.
__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem desc)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Packed pair arithmetic: (d0, d1) = (a0, a1) * (b0, b1) + (c0, c1).
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
// (d0, d1) = (a0, a1) * (b0, b1)
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// (d0, d1) += (a0, a1)
__device__ __forceinline__ void acc2(float& d0, float& d1, float a0, float a1) {
  asm("{\n\t.reg .b64 ra, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rd, {%0, %1};\n\t"
      "add.rn.f32x2 rd, rd, ra;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}
// {lo -> bits 0-15, hi -> bits 16-31}, round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// The same packing into fp16 (finite inputs up to 65504 stay finite).
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Four floats as E4M3 codes (round to nearest even, saturating at 448),
// x0 in bits 0-7 ... x3 in bits 24-31.
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}
// A bf16 pair to an fp16 pair (round to nearest even, saturating at 65504),
// keeping the running maximum magnitude for the range check.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x, float& amax) {
  const float lo = __uint_as_float(x << 16), hi = __uint_as_float(x & 0xffff0000u);
  amax = max3(amax, fabsf(lo), fabsf(hi));
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

struct KernelParams {
  const pk_work_item* items;
  const int32_t* cta_offsets;
  const int32_t* kv_limit;       // per query row: last visible key of its range, -1 none
  const int32_t* block_table;    // paged keys: physical 128-row block of each key tile; else null
  const int32_t* v8_row;         // E4M3 values, contiguous keys: per item, the row of its first
                                 // key tile in the transposed copy (a multiple of 16); else null
  uint8_t* out;   // bf16 [T][hq][D]
  float* lse;     // [hq][T]
  int32_t* status;
  int32_t T;
  int32_t hq;
  float scale_log2;  // softmax scale * log2(e)
  float v_scale;     // dequantisation scale of E4M3 values (1 otherwise)
  uint64_t wait_limit_ns;
};

// First key/value row of key tile j of a work item: contiguous keys start
// at kv_start; paged keys take the block of the item's key range from the
// block table (blocks are one key tile, 128 rows).
__device__ __forceinline__ int key_tile_row(const KernelParams& p, const pk_work_item& w, int j) {
  return p.block_table ? p.block_table[w.kv_start + j] * 128 : w.kv_start + j * 128;
}

// S(tmem) = Q K^T over the head dimension: MMAs of 128x128 and K = 16
// (bf16) or 32 (FP8) elements, i.e. 32 bytes of every row per step.  Both
// tiles are K-major with 128-byte swizzle: row r of a box sits at r*128
// bytes, 8-row groups 1024 bytes apart; the k-th step starts 32*(k%4) bytes
// into box k/4.  q_desc / k_desc describe the tiles' first byte; a step only
// adds its byte offset / 16 to the start-address field.
template <int D, bool F8 = false>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = F8 ? make_idesc_e4m3(128, 128) : make_idesc(128, 128, false);
  constexpr int kSteps = F8 ? D / 32 : D / 16;
#pragma unroll
  for (int kk = 0; kk < kSteps; ++kk) {
    const uint64_t off = (uint64_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
    if (F8)
      mma_ss_f8(d_tmem, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
    else
      mma_ss(d_tmem, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// ---- SM pairs (cta_group::2): a cluster of two CTAs on an SM pair -------
// Tensor copy into the same shared-memory offset `dst` of every CTA of the
// cluster in `mask` (bit r: CTA rank r), each completing its bytes on the
// barrier at offset `bar` in that CTA.
__device__ __forceinline__ void tma_load_3d_mc(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                               int c0, int c1, int c2, uint16_t mask,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".multicast::cluster.L2::cache_hint [%0], [%1, {%4, %5, %6}], [%2], %3, %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "h"(mask), "r"(c0), "r"(c1), "r"(c2),
      "l"(policy)
      : "memory");
}
// Commit of this thread's (one-CTA) MMAs to the barrier at offset `bar` in
// every CTA of the cluster in `mask`.
__device__ __forceinline__ void tc_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(mask)
      : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
// The shared::cluster address of this CTA's shared address `saddr` in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Relaxed arrival on a barrier of another CTA of the cluster: it orders no
// memory operation, so the caller first completes what the arrival stands
// for (its TMEM loads and stores).  A release at cluster scope would cost a
// cluster-wide memory barrier per arrival.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Commit of this thread's pair MMAs to the barrier at `bar` in the CTAs of
// `mask` (bit r: CTA rank r).
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(mask)
      : "memory");
}
// Tensor copy into `dst` (a shared::cluster address: this CTA's or the
// peer's buffer), completing on this CTA's barrier `bar`.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}
// S = Q K^T over the pair, M = 256: each CTA holds its 128 query rows
// (K-major SW128, 64-column boxes of 128 rows) and half of the key tile (64
// rows per box, so its boxes are 8 KB apart); each CTA's TMEM gets its rows.
template <int D>
__device__ __forceinline__ void issue_qk_pair(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = make_idesc(256, 128, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t oq = (uint64_t)(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
    const uint64_t ok = (uint64_t)(((kk >> 2) * (kBoxBytes / 2) + (kk & 3) * 32) >> 4);
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(q_desc + oq), "l"(k_desc + ok), "r"(idesc), "r"(kk > 0 ? 1u : 0u)
        : "memory");
  }
}
// O += P V over the pair: P (fp16) from each CTA's TMEM rows; each CTA holds
// the values of 64 of the D columns (one MN-major SW128 box of 128 keys).
template <int D>
__device__ __forceinline__ void issue_pv_pair(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                              bool accumulate) {
  constexpr uint32_t idesc = make_idesc_f16(256, D, true);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(p_tmem + (uint32_t)kk * 8u), "l"(v_desc + (uint64_t)(kk * (2048 >> 4))), "r"(idesc),
        "r"((accumulate || kk > 0) ? 1u : 0u)
        : "memory");
}

// O(tmem) (+)= P V: 8 MMAs of 128 x D x 16, fp16 operands.  P (fp16 pairs)
// is read from TMEM, 8 columns per 16 keys.  V is MN-major with 128-byte swizzle: 16 keys
// span 2048 bytes, and the second 64-column box (D = 128) is 16384 bytes on.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                         bool accumulate) {
  constexpr uint32_t idesc = make_idesc_f16(128, D, true);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts(d_tmem, p_tmem + (uint32_t)kk * 8u, v_desc + (uint64_t)(kk * (2048 >> 4)), idesc,
           (accumulate || kk > 0) ? 1u : 0u);
}

// O(tmem) (+)= P V with E4M3 P and values: 4 MMAs of 128 x D x 32 on
// kind::f8f6f4.  P is read from TMEM, four keys per column (8 columns per
// 32 keys); the value tile is K-major with 128-byte swizzle (one 128-byte
// row of keys per head-dimension index), the k-th step 32 bytes along it.
template <int D>
__device__ __forceinline__ void issue_pv_f8(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                            bool accumulate) {
  constexpr uint32_t idesc = make_idesc_e4m3(128, D);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_ts_f8(d_tmem, p_tmem + (uint32_t)kk * 8u, v_desc + (uint64_t)((kk * 32) >> 4), idesc,
              (accumulate || kk > 0) ? 1u : 0u);
}

}  // namespace dev
}  // namespace pk
