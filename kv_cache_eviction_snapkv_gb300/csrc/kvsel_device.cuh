// Device helpers shared by the libkvsel kernels.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "kvsel_internal.h"

namespace kvsel {

// First device-side error wins; later ones are dropped.
__device__ __forceinline__ void record_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

// 2^x with the hardware approximation (relative error about 2^-22); -inf -> +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float load_elem(const void* base, int64_t i, int dtype) {
  if (dtype == KVSEL_BF16)
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
  return reinterpret_cast<const float*>(base)[i];
}

__device__ __forceinline__ bool finite_f(float x) { return fabsf(x) <= 3.402823466e38f; }

// Debug builds (-DKVSEL_DEBUG) check the index arithmetic of the gathers and
// output writes against the bounds the host passed: a failed check records
// KVSEL_ERR_BAD_INDEX and the access is skipped. Release builds compile the
// checks away (the condition is not evaluated).
__device__ __forceinline__ bool debug_in_bounds(bool ok, int* status) {
  if (!ok) record_status(status, KVSEL_ERR_BAD_INDEX);
  return ok;
}
#ifdef KVSEL_DEBUG
#define KVSEL_IN_BOUNDS(cond, status) (::kvsel::debug_in_bounds((cond), (status)))
#else
#define KVSEL_IN_BOUNDS(cond, status) true
#endif

// Largest s in [0, n) with base_of(s) <= key (arrays sorted by base, base_of(0) <= key).
template <typename F>
__device__ __forceinline__ int upper_find(int n, int key, F base_of) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (base_of(mid) <= key) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Decode a scoring work item into (layer, scored sequence, head, chunk).
struct ItemPos {
  int layer, s, h, c;
  int inst;  // global instance id
};

__device__ __forceinline__ ItemPos decode_item(const ScoreArgs& a, int item) {
  ItemPos p;
  p.layer = item / a.items_per_layer;
  int rem = item - p.layer * a.items_per_layer;
  const SeqDesc* sq = a.seqs;
  p.s = upper_find(a.n_scored, rem, [&](int i) { return sq[i].item_base; });
  int local = rem - sq[p.s].item_base;
  int nc = sq[p.s].n_chunks;
  p.h = local / nc;
  p.c = local - p.h * nc;
  p.inst = p.layer * a.inst_per_layer + sq[p.s].inst_base + p.h;
  return p;
}

}  // namespace kvsel
