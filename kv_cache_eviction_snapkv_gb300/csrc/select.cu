// Pooling of the prefix votes and the per-head top-(C - W) selection.
//
// Method: page "SnapKV: choosing the KV cache of a long prompt with an
// observation window", section "Pooling turns a peak into a neighbourhood
// preference" (池化把一个峰值扩展成邻域偏好): odd width k, stride 1, zero
// padding over the prefix votes only; the average divides by k even at the
// edges; max pooling takes the largest in-range neighbour. Then the C - W
// prefix positions with the highest pooled score are kept, ties going to the
// smaller position (the order key (-score, j) of the section "Computing one
// full selection from Q and K", 从 Q 和 K 开始算一次完整选择), and the window
// P..L-1 is appended.
//
// Selection per (layer, sequence, head), one CTA: scores map to order-keeping
// 32-bit keys; three histogram passes (11 + 11 + 10 bits) find the key T of
// the (C - W)-th largest score and how many keys equal to T are needed; an
// emit pass in position order takes every key > T and the first ones == T
// (smaller positions first); an on-chip bitonic sort of (~key, position)
// orders the kept positions by (-score, position).
#include "kvsel_device.cuh"

namespace kvsel {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBins = 2048;

// Order-keeping key: larger float -> larger key; -0 == +0; NaN lowest.
__device__ __forceinline__ uint32_t score_key(float v, int* status) {
  if (v != v) {
    record_status(status, KVSEL_ERR_NONFINITE);
    return 0u;
  }
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Pooled score of prefix position j from the votes s[0..P) of one instance.
__device__ __forceinline__ float pool_at(const float* s, int j, int P, int pool_kind,
                                         int pool_k) {
  const int R = pool_k >> 1;
  const int lo = max(0, j - R), hi = min(P - 1, j + R);
  if (pool_kind == KVSEL_POOL_AVG) {
    float acc = 0.f;
    for (int i = lo; i <= hi; ++i) acc += s[i];
    return acc / (float)pool_k;
  }
  float m = s[lo];
  for (int i = lo + 1; i <= hi; ++i) m = fmaxf(m, s[i]);
  return m;
}

// kvsel_score's pooling: one block per (layer, head, sequence).
__global__ void __launch_bounds__(256) pool_kernel(PoolArgs a) {
  const int inst = blockIdx.x;                 // ((layer * H) + h) * n_seqs + b
  const int b = inst % a.n_seqs;
  const int lh = inst / a.n_seqs;              // layer * H + h
  const SeqDesc sd = a.seqs[b];
  const int64_t base = (int64_t)lh * a.T + sd.tok_off;
  const int P = sd.len - a.W;
  for (int j = threadIdx.x; j < sd.len; j += blockDim.x)
    a.pooled[base + j] = j < P ? pool_at(a.votes + base, j, P, a.pool_kind, a.pool_k) : 0.f;
}

constexpr uint32_t kNoBin = 0xFFFFFFFFu;

// Warp-aggregated histogram increment (all 32 lanes call it; kNoBin = skip).
__device__ __forceinline__ void add_bin(uint32_t* hist, uint32_t bin, int lane) {
  const unsigned peers = __match_any_sync(0xffffffffu, bin);
  if (bin != kNoBin && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

// Warp 0 finds the bin holding the krem-th largest key among the counted ones.
// Writes (bin, count strictly above that bin) to out[0], out[1].
__device__ void find_bin(const uint32_t* hist, int nbins, uint32_t krem, uint32_t* out) {
  const int lane = threadIdx.x & 31;
  const int per = nbins / 32;
  const int lo = lane * per;
  uint32_t mine = 0;
  for (int i = 0; i < per; ++i) mine += hist[lo + i];
  uint32_t incl = mine;  // sum over lanes >= this lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t t = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += t;
  }
  const uint32_t above = incl - mine;
  if (above < krem && krem <= incl) {
    uint32_t acc = above;
    for (int i = per - 1; i >= 0; --i) {
      const uint32_t c = hist[lo + i];
      if (acc + c >= krem) {
        out[0] = (uint32_t)(lo + i);
        out[1] = acc;
        break;
      }
      acc += c;
    }
  }
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectArgs a, int n2) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(smem + kBins * 4);
  __shared__ uint32_t found[2];
  __shared__ uint32_t warp_eq[kSelWarps];
  __shared__ uint32_t n_sel;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int inst = blockIdx.x;                 // ((layer * S) + b) * H + h
  const int h = inst % a.H;
  const int lb = inst / a.H;
  const int b = lb % a.n_seqs;
  const int layer = lb / a.n_seqs;
  const SeqDesc sd = a.seqs[b];
  const int L = sd.len;
  int32_t* out = a.out_idx + ((int64_t)layer * a.T_out + sd.out_off) * a.H + h;

  if (L < a.C) {  // bypass: keep everything in order
    for (int s = tid; s < L; s += kSelThreads) out[(int64_t)s * a.H] = s;
    return;
  }
  const int P = L - a.W;
  const uint32_t k = (uint32_t)(a.C - a.W);
  const int64_t plane = ((int64_t)layer * a.H + h) * a.T + sd.tok_off;
  const float* src = a.scores + plane;
  const float* sc = src;  // the scores the passes read

  // Pass 1 (with pooling when inline): histogram of the top 11 key bits.
  for (int i = tid; i < kBins; i += kSelThreads) hist[i] = 0;
  __syncthreads();
  float* pl = a.pooled_ws + plane;
  for (int base = 0; base < P; base += kSelThreads) {
    const int j = base + tid;
    uint32_t bin = kNoBin;
    if (j < P) {
      float v;
      if (a.pool_inline) {
        v = pool_at(src, j, P, a.pool_kind, a.pool_k);
        pl[j] = v;
      } else {
        v = src[j];
      }
      bin = score_key(v, a.status) >> 21;
    }
    add_bin(hist, bin, lane);
  }
  if (a.pool_inline) sc = pl;
  __syncthreads();
  if (warp == 0) find_bin(hist, kBins, k, found);
  __syncthreads();
  const uint32_t d1 = found[0];
  uint32_t krem = k - found[1];

  // Pass 2: next 11 bits among keys whose top 11 bits are d1.
  for (int i = tid; i < kBins; i += kSelThreads) hist[i] = 0;
  __syncthreads();
  for (int base = 0; base < P; base += kSelThreads) {
    const int j = base + tid;
    uint32_t bin = kNoBin;
    if (j < P) {
      const uint32_t key = score_key(sc[j], a.status);
      if ((key >> 21) == d1) bin = (key >> 10) & 0x7FFu;
    }
    add_bin(hist, bin, lane);
  }
  __syncthreads();
  if (warp == 0) find_bin(hist, kBins, krem, found);
  __syncthreads();
  const uint32_t d2 = found[0];
  krem -= found[1];

  // Pass 3: last 10 bits among keys whose top 22 bits are (d1, d2).
  const uint32_t top22 = (d1 << 11) | d2;
  for (int i = tid; i < 1024; i += kSelThreads) hist[i] = 0;
  __syncthreads();
  for (int base = 0; base < P; base += kSelThreads) {
    const int j = base + tid;
    uint32_t bin = kNoBin;
    if (j < P) {
      const uint32_t key = score_key(sc[j], a.status);
      if ((key >> 10) == top22) bin = key & 0x3FFu;
    }
    add_bin(hist, bin, lane);
  }
  __syncthreads();
  if (warp == 0) find_bin(hist, 1024, krem, found);
  __syncthreads();
  const uint32_t thr = (top22 << 10) | found[0];
  const uint32_t need_eq = krem - found[1];  // keys == thr to keep, smallest positions first

  // Emit pass in position order.
  if (tid == 0) n_sel = 0;
  uint32_t eq_base = 0;
  __syncthreads();
  for (int base = 0; base < P; base += kSelThreads) {
    const int j = base + tid;
    const uint32_t key = j < P ? score_key(sc[j], a.status) : 0u;
    const bool gt = j < P && key > thr;
    const bool eq = j < P && key == thr;
    const uint32_t bal = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) warp_eq[warp] = __popc(bal);
    __syncthreads();
    uint32_t before = eq_base, total = 0;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
      const uint32_t c = warp_eq[w];
      if (w < warp) before += c;
      total += c;
    }
    before += __popc(bal & ((1u << lane) - 1u));
    if (gt || (eq && before < need_eq)) {
      const uint32_t pos = atomicAdd(&n_sel, 1u);
      keys[pos] = ((unsigned long long)(~key) << 32) | (uint32_t)j;
    }
    eq_base += total;
    __syncthreads();
  }
  for (int i = (int)k + tid; i < n2; i += kSelThreads) keys[i] = ~0ull;
  __syncthreads();

  // Bitonic sort ascending: larger score first, then smaller position.
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < (n2 >> 1); i += kSelThreads) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const unsigned long long x = keys[lo], y = keys[hi];
        if ((x > y) == up) {
          keys[lo] = y;
          keys[hi] = x;
        }
      }
      __syncthreads();
    }
  }
  for (int s = tid; s < (int)k; s += kSelThreads)
    out[(int64_t)s * a.H] = (int32_t)(keys[s] & 0xFFFFFFFFull);
  for (int w = tid; w < a.W; w += kSelThreads) out[(int64_t)(k + w) * a.H] = P + w;
}

}  // namespace

cudaError_t launch_pool(const PoolArgs& a) {
  const int64_t blocks = (int64_t)a.layers * a.H * a.n_seqs;
  if (blocks == 0) return cudaSuccess;
  pool_kernel<<<(unsigned)blocks, 256, 0, a.stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_select(const SelectArgs& a) {
  const int64_t blocks = (int64_t)a.layers * a.n_seqs * a.H;
  if (blocks == 0) return cudaSuccess;
  int n2 = 1;
  while (n2 < a.C - a.W) n2 <<= 1;
  if (n2 < 2) n2 = 2;
  const size_t smem = kBins * 4 + (size_t)n2 * 8;
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e) return e;
  select_kernel<<<(unsigned)blocks, kSelThreads, smem, a.stream>>>(a, n2);
  return cudaGetLastError();
}

}  // namespace kvsel
