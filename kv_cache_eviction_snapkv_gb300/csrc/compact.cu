// Gather of the kept K/V rows into the compacted cache.
//
// Method: page "SnapKV: choosing the KV cache of a long prompt with an
// observation window", section "Computing one full selection from Q and K"
// (从 Q 和 K 开始算一次完整选择): K and V are gathered with one and the same
// index list, per head; a prompt shorter than the budget is kept whole.
//
// One output row is D * elem_bytes contiguous bytes; the (sequence, slot,
// head) rows of one sequence are contiguous in the output, so consecutive
// threads write consecutive vectors (coalesced), and each source row is one
// contiguous segment of K (and of V). Every index is checked against the
// sequence length before the read: an index outside [0, L) records
// KVSEL_ERR_BAD_INDEX and that row is not written.
#include "kvsel_device.cuh"

namespace kvsel {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

template <int VW> struct Vec;
template <> struct Vec<16> { using T = uint4; };
template <> struct Vec<8> { using T = uint2; };
template <> struct Vec<4> { using T = uint32_t; };
template <> struct Vec<2> { using T = uint16_t; };

template <int VW>
__global__ void __launch_bounds__(kThreads) compact_kernel(CompactArgs a) {
  using V = typename Vec<VW>::T;
  const uint32_t vpr = (uint32_t)(a.row_bytes / VW);  // vectors per row
  const int n_pairs = a.layers * a.S;
  for (int ls = blockIdx.y; ls < n_pairs; ls += gridDim.y) {
    const int layer = ls / a.S, b = ls - layer * a.S;
    const SeqDesc sd = a.seqs[b];
    const uint32_t n_out = (uint32_t)min(sd.len, a.C);
    const uint32_t total = n_out * (uint32_t)a.H * vpr;
    const int64_t out_row0 = ((int64_t)layer * a.T_out + sd.out_off) * a.H;
    const int64_t src_tok0 = (int64_t)layer * a.T + sd.tok_off;
    const int32_t* idx = a.idx + out_row0;
    const char* kb = reinterpret_cast<const char*>(a.k);
    const char* vb = reinterpret_cast<const char*>(a.v);
    char* okb = reinterpret_cast<char*>(a.out_k) + out_row0 * a.row_bytes;
    char* ovb = reinterpret_cast<char*>(a.out_v) + out_row0 * a.row_bytes;
    const uint32_t step = gridDim.x * kThreads;
    for (uint32_t e0 = blockIdx.x * kThreads + threadIdx.x; e0 < total; e0 += step * kUnroll) {
      V kv[kUnroll], vv[kUnroll];
      bool ok[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t e = e0 + u * step;
        ok[u] = false;
        if (e < total) {
          const uint32_t row = e / vpr, v = e - row * vpr;   // row = slot * H + head
          const uint32_t s = row / (uint32_t)a.H, h = row - s * (uint32_t)a.H;
          const int32_t j = __ldg(idx + row);
          if (j >= 0 && j < sd.len) {
            const int64_t src =
                ((src_tok0 + j) * a.kv_H + h / a.kv_div) * a.row_bytes + (int64_t)v * VW;
            kv[u] = __ldcs(reinterpret_cast<const V*>(kb + src));
            vv[u] = __ldcs(reinterpret_cast<const V*>(vb + src));
            ok[u] = true;
          } else {
            record_status(a.status, KVSEL_ERR_BAD_INDEX);
          }
          (void)s;
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t e = e0 + u * step;
        if (ok[u] && KVSEL_IN_BOUNDS(out_row0 + e / vpr < (layer + 1) * a.T_out * a.H,
                                              a.status)) {
          const int64_t dst = (int64_t)e * VW;
          __stcs(reinterpret_cast<V*>(okb + dst), kv[u]);
          __stcs(reinterpret_cast<V*>(ovb + dst), vv[u]);
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_compact(const CompactArgs& a) {
  if (a.layers == 0 || a.S == 0 || a.max_rows == 0) return cudaSuccess;
  auto aligned = [&](int vw) {
    if (a.row_bytes % vw) return false;
    for (const void* p : {a.k, a.v, (const void*)a.out_k, (const void*)a.out_v})
      if (reinterpret_cast<uintptr_t>(p) % vw) return false;
    return true;
  };
  const int vw = aligned(16) ? 16 : aligned(8) ? 8 : aligned(4) ? 4 : 2;
  const int64_t vecs = a.max_rows * (a.row_bytes / vw);
  int64_t gx = (vecs + (int64_t)kThreads * kUnroll - 1) / ((int64_t)kThreads * kUnroll);
  const int64_t pairs = (int64_t)a.layers * a.S;
  // enough blocks in flight for the whole GPU, without a huge grid per pair
  const int64_t cap = (int64_t)a.sm_count * 64;
  if (gx * pairs > cap) gx = (cap + pairs - 1) / pairs;
  if (gx < 1) gx = 1;
  if (gx > 65535 * 1024) gx = 65535 * 1024;
  const unsigned gy = (unsigned)(pairs < 65535 ? pairs : 65535);
  dim3 grid((unsigned)gx, gy);
  switch (vw) {
    case 16: compact_kernel<16><<<grid, kThreads, 0, a.stream>>>(a); break;
    case 8: compact_kernel<8><<<grid, kThreads, 0, a.stream>>>(a); break;
    case 4: compact_kernel<4><<<grid, kThreads, 0, a.stream>>>(a); break;
    default: compact_kernel<2><<<grid, kThreads, 0, a.stream>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace kvsel
