// Decode-side consumer of a compacted cache: one future query per (layer,
// sequence, query head) attends to the sequence's cache rows followed by its
// g appended rows.
//
// Method: page "SnapKV: choosing the KV cache of a long prompt with an
// observation window", section "Why deleting positions changes the output"
// (删除位置为什么会改变输出): the query's softmax over the rows it reads, its
// value sum, and the probability mass m that the full cache gives the kept
// rows, m = exp(lse over the kept rows - lse over all rows); section "The
// current prefill still reads the full K/V" (当前 prefill 仍读完整 K/V，压缩缓存
// 服务后续 decode): the cache holds min(L, C) + g rows once g generated tokens
// are appended; section "Computing one full selection from Q and K", last
// paragraph: a single query is unchanged by permuting K and V rows together,
// so the compacted rows are read in their stored order.
//
// Split over rows (flash-decoding): a CTA takes up to 512 rows of one
// (layer, sequence, query head); eight lanes share a row (each D/8 dimensions,
// so a row's 2*D*eb bytes of K and V are read as coalesced 16-byte vectors),
// four rows per lane group per step with one online-softmax rescale per four
// rows; the CTA writes one partial (max, sum, D weighted values) in base-2
// units. A second kernel merges an instance's partials into the output and the
// natural-log lse. HBM-bound: the algorithmic bytes are the K and V rows read
// once per query head (plus q and the output).
#include <cmath>

#include "kvsel_device.cuh"

namespace kvsel {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kRowsPerStep = kDecWarps * 16;      // 4 lane groups x 4 rows per warp

template <typename T, int E>
struct RowSlice {
  static constexpr int kVecs = E * (int)sizeof(T) / 16;
  uint4 raw[kVecs];
  __device__ __forceinline__ void load(const T* p) {
    const uint4* s = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int i = 0; i < kVecs; ++i) raw[i] = __ldcs(s + i);
  }
  __device__ __forceinline__ float at(int e) const {
    if constexpr (sizeof(T) == 2) {
      const uint32_t w = reinterpret_cast<const uint32_t*>(raw)[e >> 1];
      return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
    } else {
      return reinterpret_cast<const float*>(raw)[e];
    }
  }
};

__device__ __forceinline__ const DecSeq& find_seq(const DecodeArgs& a, int rem) {
  return a.seqs[upper_find(a.S, rem, [&](int i) { return a.seqs[i].item_base; })];
}

// Pointer to row j of (layer, sequence, kv head): cache rows first, then the
// appended ones.
template <typename T>
__device__ __forceinline__ const T* row_ptr(const DecodeArgs& a, const T* cache, const T* app,
                                           int layer, const DecSeq& sq, int kvh, int j) {
  // debug builds: row j of the instance lies in its cache rows or its g
  // appended rows (else the cache's first row of the layer is read instead)
  if (!KVSEL_IN_BOUNDS(j >= 0 && j < sq.n_rows + a.g && sq.row_off + sq.n_rows <= a.T &&
                           kvh < a.Hkv, a.status))
    return cache + (int64_t)layer * a.T * a.Hkv * a.D;
  if (j < sq.n_rows)
    return cache + (((int64_t)layer * a.T + sq.row_off + j) * a.Hkv + kvh) * a.D;
  const int64_t r = (int64_t)layer * a.S * a.g + (int64_t)sq.index * a.g + (j - sq.n_rows);
  return app + (r * a.Hkv + kvh) * a.D;
}

template <typename T, int E>
__global__ void __launch_bounds__(kDecThreads) decode_partial_kernel(const __grid_constant__ DecodeArgs a) {
  __shared__ float wm[kDecWarps], wl[kDecWarps];
  __shared__ float wo[kDecWarps][8 * E];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 3, sub = lane & 7;
  const int item = blockIdx.x;
  const int layer = item / a.items_per_layer;
  const int rem = item - layer * a.items_per_layer;
  const DecSeq& sq = find_seq(a, rem);
  const int local = rem - sq.item_base;
  const int h = local / sq.n_chunks, c = local - h * sq.n_chunks;
  const int kvh = h / (a.H / a.Hkv);
  const int n_total = sq.n_rows + a.g;
  const int r_begin = c * a.chunk_rows, r_end = min(n_total, r_begin + a.chunk_rows);
  const T* kc = reinterpret_cast<const T*>(a.k);
  const T* vc = reinterpret_cast<const T*>(a.v);
  const T* kn = reinterpret_cast<const T*>(a.k_new);
  const T* vn = reinterpret_cast<const T*>(a.v_new);

  float qv[E];
  {
    const T* qp = reinterpret_cast<const T*>(a.q) +
                  (((int64_t)layer * a.S + sq.index) * a.H + h) * a.D + sub * E;
    RowSlice<T, E> qs;
    qs.load(qp);
#pragma unroll
    for (int e = 0; e < E; ++e) qv[e] = qs.at(e) * a.scale_log2;
  }
  float m = -INFINITY, l = 0.f, o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;

  // warp-uniform trips (the shuffles need every lane); a lane group whose
  // rows are all past the end contributes nothing
  for (int wb = r_begin + warp * 16; wb < r_end; wb += kRowsPerStep) {
    const int r0 = wb + grp * 4;
    RowSlice<T, E> kr[4], vr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = min(r0 + i, r_end - 1);   // rows past the end repeat the last (masked below)
      kr[i].load(row_ptr(a, kc, kn, layer, sq, kvh, j) + sub * E);
      vr[i].load(row_ptr(a, vc, vn, layer, sq, kvh, j) + sub * E);
    }
    float s[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) d = fmaf(qv[e], kr[i].at(e), d);
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      d += __shfl_xor_sync(0xffffffffu, d, 2);
      d += __shfl_xor_sync(0xffffffffu, d, 4);
      s[i] = r0 + i < r_end ? d : -INFINITY;
    }
    const float mx = fmaxf(fmaxf(m, fmaxf(s[0], s[1])), fmaxf(s[2], s[3]));
    if (mx != -INFINITY) {
      const float sc = ex2(m - mx);         // m = -inf: 0
      float p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = ex2(s[i] - mx);
      l = fmaf(l, sc, (p[0] + p[1]) + (p[2] + p[3]));
#pragma unroll
      for (int e = 0; e < E; ++e) {
        float acc = o[e] * sc;
#pragma unroll
        for (int i = 0; i < 4; ++i) acc = fmaf(p[i], vr[i].at(e), acc);
        o[e] = acc;
      }
      m = mx;
    }
  }
  // merge the warp's four lane groups (lanes sub, sub + 8, sub + 16, sub + 24)
#pragma unroll
  for (int off = 8; off <= 16; off <<= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float lo = __shfl_xor_sync(0xffffffffu, l, off);
    const float mx = fmaxf(m, mo);
    const float f = mx == -INFINITY ? 0.f : ex2(m - mx);
    const float fo = mx == -INFINITY ? 0.f : ex2(mo - mx);
    l = l * f + lo * fo;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = o[e] * f + __shfl_xor_sync(0xffffffffu, o[e], off) * fo;
    m = mx;
  }
  if (lane < 8) {
#pragma unroll
    for (int e = 0; e < E; ++e) wo[warp][sub * E + e] = o[e];
    if (lane == 0) {
      wm[warp] = m;
      wl[warp] = l;
    }
  }
  __syncthreads();
  float* part = a.part + (int64_t)item * (2 + a.D);
  float mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) mx = fmaxf(mx, wm[w]);
  for (int d = tid; d < a.D; d += kDecThreads) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w)
      if (wm[w] != -INFINITY) acc = fmaf(wo[w][d], ex2(wm[w] - mx), acc);
    part[2 + d] = acc;
  }
  if (tid == 0) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w)
      if (wm[w] != -INFINITY) sum = fmaf(wl[w], ex2(wm[w] - mx), sum);
    part[0] = mx;
    part[1] = sum;
  }
}

// One block per (layer, sequence, query head): merges its chunks' partials.
__global__ void __launch_bounds__(128) decode_combine_kernel(const __grid_constant__ DecodeArgs a) {
  const int inst = blockIdx.x;                 // (layer * S + b) * H + h
  const int h = inst % a.H;
  const int lb = inst / a.H;
  const int b = lb % a.S, layer = lb / a.S;
  const DecSeq& sq = a.seqs[b];
  const int64_t first = (int64_t)layer * a.items_per_layer + sq.item_base + (int64_t)h * sq.n_chunks;
  const float* part = a.part + first * (2 + a.D);
  float mx = -INFINITY;
  for (int c = 0; c < sq.n_chunks; ++c) mx = fmaxf(mx, part[(int64_t)c * (2 + a.D)]);
  float sum = 0.f;
  for (int c = 0; c < sq.n_chunks; ++c) {
    const float* pc = part + (int64_t)c * (2 + a.D);
    sum = fmaf(pc[1], ex2(pc[0] - mx), sum);
  }
  const float inv = 1.f / sum;
  bool bad = !(sum > 0.f) || !finite_f(sum) || !finite_f(mx);
  for (int d = threadIdx.x; d < a.D; d += blockDim.x) {
    float acc = 0.f;
    for (int c = 0; c < sq.n_chunks; ++c) {
      const float* pc = part + (int64_t)c * (2 + a.D);
      acc = fmaf(pc[2 + d], ex2(pc[0] - mx), acc);
    }
    const float v = acc * inv;
    bad |= !finite_f(v);
    if (KVSEL_IN_BOUNDS(inst < a.layers * a.S * a.H, a.status)) a.out[(int64_t)inst * a.D + d] = v;
  }
  if (threadIdx.x == 0 && a.lse) a.lse[inst] = (mx + log2f(sum)) * 0.6931471805599453f;
  if (bad) record_status(a.status, KVSEL_ERR_NONFINITE);
}

// Retained mass and output error per instance: one warp each.
__global__ void __launch_bounds__(256) decode_quality_kernel(QualityArgs a) {
  const int64_t inst = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (inst >= a.n) return;
  float ss = 0.f;
  for (int d = lane; d < a.D; d += 32) {
    const float diff = a.out_full[inst * a.D + d] - a.out_keep[inst * a.D + d];
    ss = fmaf(diff, diff, ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if (lane == 0) {
    a.mass[inst] = expf(a.lse_keep[inst] - a.lse_full[inst]);
    a.err[inst] = sqrtf(ss);
  }
}

template <typename T, int E>
cudaError_t launch_partial(const DecodeArgs& a, int64_t items) {
  decode_partial_kernel<T, E><<<(unsigned)items, kDecThreads, 0, a.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

int decode_chunk_rows() { return 512; }

bool decode_supported(int dtype, int D) {
  return (dtype == KVSEL_BF16 || dtype == KVSEL_F32) && (D == 64 || D == 128);
}

cudaError_t launch_decode(const DecodeArgs& a) {
  const int64_t items = (int64_t)a.layers * a.items_per_layer;
  if (items == 0) return cudaSuccess;
  cudaError_t e;
  if (a.dtype == KVSEL_BF16)
    e = a.D == 128 ? launch_partial<__nv_bfloat16, 16>(a, items)
                   : launch_partial<__nv_bfloat16, 8>(a, items);
  else
    e = a.D == 128 ? launch_partial<float, 16>(a, items) : launch_partial<float, 8>(a, items);
  if (e) return e;
  const int64_t insts = (int64_t)a.layers * a.S * a.H;
  decode_combine_kernel<<<(unsigned)insts, 128, 0, a.stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode_quality(const QualityArgs& a) {
  if (a.n == 0) return cudaSuccess;
  decode_quality_kernel<<<(unsigned)((a.n + 7) / 8), 256, 0, a.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvsel
