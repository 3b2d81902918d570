// Host-buffer pipeline: successive attention steps whose inputs live in host
// memory, with each step's host -> device copy, kernel and device -> host
// copy on three streams, so one step's copies overlap the neighbouring
// steps' kernels.  Device memory is the caller's: num_slots sets of
// q/k/v/out/lse buffers, used round robin.  Events order the three stages
// of a step and keep a slot's buffers from being overwritten while an
// earlier step still reads them.
#include <cuda_runtime.h>

#include <new>
#include <vector>

#include "pk_internal.h"

struct pk_pipeline {
  const pk_plan* plan = nullptr;
  std::vector<pk_dev_slot> slots;
  cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
  std::vector<cudaEvent_t> ev_in, ev_comp, ev_out;  // per slot: stage done
  std::vector<bool> used;                            // slot has run a step
  int64_t steps = 0;
};

namespace {

void release(pk_pipeline* p) {
  if (p == nullptr) return;
  for (cudaStream_t s : {p->s_in, p->s_comp, p->s_out})
    if (s) cudaStreamSynchronize(s);
  for (auto* v : {&p->ev_in, &p->ev_comp, &p->ev_out})
    for (cudaEvent_t e : *v)
      if (e) cudaEventDestroy(e);
  for (cudaStream_t s : {p->s_in, p->s_comp, p->s_out})
    if (s) cudaStreamDestroy(s);
  cudaGetLastError();
  delete p;
}

}  // namespace

extern "C" {

pk_status pk_pipeline_create(const pk_plan* plan, const pk_dev_slot* slots, int32_t num_slots,
                             pk_pipeline** out) {
  if (out == nullptr) return PK_ERR_INVALID_ARG;
  *out = nullptr;
  if (plan == nullptr || slots == nullptr || num_slots < 1 || num_slots > 8)
    return PK_ERR_INVALID_ARG;
  for (int32_t i = 0; i < num_slots; ++i) {
    const pk_dev_slot& s = slots[i];
    if (!s.q || !s.k || !s.v || !s.out || !s.lse) return PK_ERR_INVALID_ARG;
  }
  pk_pipeline* p = new (std::nothrow) pk_pipeline();
  if (p == nullptr) return PK_ERR_OUT_OF_MEMORY;
  try {
    p->plan = plan;
    p->slots.assign(slots, slots + num_slots);
    p->ev_in.assign(num_slots, nullptr);
    p->ev_comp.assign(num_slots, nullptr);
    p->ev_out.assign(num_slots, nullptr);
    p->used.assign(num_slots, false);
  } catch (...) {  // no C++ exception crosses the C boundary
    delete p;
    return PK_ERR_OUT_OF_MEMORY;
  }
  bool ok = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->s_comp, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking) == cudaSuccess;
  for (int32_t i = 0; ok && i < num_slots; ++i)
    ok = cudaEventCreateWithFlags(&p->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->ev_comp[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->ev_out[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    release(p);
    return PK_ERR_CUDA;
  }
  *out = p;
  return PK_OK;
}

pk_status pk_pipeline_submit(pk_pipeline* p, const void* q_host, const void* k_host,
                             const void* v_host, void* out_host, float* lse_host, float scale,
                             int32_t* dev_status) {
  if (p == nullptr || !q_host || !k_host || !v_host || !out_host || !lse_host)
    return PK_ERR_INVALID_ARG;
  const pk_plan* plan = p->plan;
  const size_t T = (size_t)plan->T, Tk = (size_t)plan->Tk, d = (size_t)plan->head_dim;
  const size_t qb = T * plan->hq * d * 2, kvb = Tk * plan->hkv * d * 2;
  const size_t lb = T * plan->hq * sizeof(float);
  const int32_t n = (int32_t)p->slots.size();
  const int32_t i = (int32_t)(p->steps % n);
  const pk_dev_slot& s = p->slots[i];
  const bool reuse = p->used[i];
  // Copy in once the slot's previous kernel has read its inputs.
  if ((reuse && cudaStreamWaitEvent(p->s_in, p->ev_comp[i], 0) != cudaSuccess) ||
      cudaMemcpyAsync(s.q, q_host, qb, cudaMemcpyHostToDevice, p->s_in) != cudaSuccess ||
      cudaMemcpyAsync(s.k, k_host, kvb, cudaMemcpyHostToDevice, p->s_in) != cudaSuccess ||
      cudaMemcpyAsync(s.v, v_host, kvb, cudaMemcpyHostToDevice, p->s_in) != cudaSuccess ||
      cudaEventRecord(p->ev_in[i], p->s_in) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  // Compute once the inputs are in and the slot's previous outputs are out.
  if (cudaStreamWaitEvent(p->s_comp, p->ev_in[i], 0) != cudaSuccess ||
      (reuse && cudaStreamWaitEvent(p->s_comp, p->ev_out[i], 0) != cudaSuccess)) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  // The slot's v is this launch's workspace: its values become fp16 in place.
  pk_status st = pk_attn_fwd(plan, s.q, s.k, s.v, s.out, s.lse, scale, s.v, kvb,
                             reinterpret_cast<pk_stream_t>(p->s_comp), dev_status);
  if (st != PK_OK) return st;
  if (cudaEventRecord(p->ev_comp[i], p->s_comp) != cudaSuccess ||
      cudaStreamWaitEvent(p->s_out, p->ev_comp[i], 0) != cudaSuccess ||
      cudaMemcpyAsync(out_host, s.out, qb, cudaMemcpyDeviceToHost, p->s_out) != cudaSuccess ||
      cudaMemcpyAsync(lse_host, s.lse, lb, cudaMemcpyDeviceToHost, p->s_out) != cudaSuccess ||
      cudaEventRecord(p->ev_out[i], p->s_out) != cudaSuccess) {
    cudaGetLastError();
    return PK_ERR_CUDA;
  }
  p->used[i] = true;
  ++p->steps;
  return PK_OK;
}

pk_status pk_pipeline_sync(pk_pipeline* p) {
  if (p == nullptr) return PK_ERR_INVALID_ARG;
  for (cudaStream_t s : {p->s_in, p->s_comp, p->s_out})
    if (cudaStreamSynchronize(s) != cudaSuccess) {
      cudaGetLastError();
      return PK_ERR_CUDA;
    }
  return PK_OK;
}

pk_stream_t pk_pipeline_stream(const pk_pipeline* p, int32_t which) {
  if (p == nullptr) return nullptr;
  const cudaStream_t s = which == 0 ? p->s_in : which == 1 ? p->s_comp : which == 2 ? p->s_out
                                                                                     : nullptr;
  return reinterpret_cast<pk_stream_t>(s);
}

void pk_pipeline_destroy(pk_pipeline* p) { release(p); }

}  // extern "C"
