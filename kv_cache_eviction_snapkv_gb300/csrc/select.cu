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
#include <algorithm>

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

// Histogram increment from all 32 lanes (kNoBin = skip): one add of the
// lane count when the whole warp shares a bin, else one add per lane.
__device__ __forceinline__ void add_bin(uint32_t* hist, uint32_t bin, int lane) {
  const uint32_t b0 = __shfl_sync(0xffffffffu, bin, 0);
  if (__all_sync(0xffffffffu, bin == b0)) {
    if (lane == 0 && b0 != kNoBin) atomicAdd(&hist[b0], 32u);
  } else if (bin != kNoBin) {
    atomicAdd(&hist[bin], 1u);
  }
}

// All threads of the block: find the bin holding the krem-th largest key
// among the counted ones; thread t owns bins [t*nb/NT, (t+1)*nb/NT). Writes
// (bin, count strictly above that bin) to out[0], out[1]. `wsum` is scratch
// for kSelWarps values. Ends with a barrier.
__device__ void find_bin_block(const uint32_t* hist, int nb, uint32_t krem, uint32_t* out,
                               uint32_t* wsum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = nb / kSelThreads;           // 4 or 2
  const int lo = tid * per;
  uint32_t mine = 0;
  for (int i = 0; i < per; ++i) mine += hist[lo + i];
  // suffix sums: bins owned by threads with a larger index come first
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += t;
  }
  if (lane == 0) wsum[warp] = incl;           // the warp's total
  __syncthreads();
  uint32_t later = 0;
  for (int w = warp + 1; w < kSelWarps; ++w) later += wsum[w];
  incl += later;
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
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Cluster plumbing: CTA rank, cluster barrier, distributed shared memory
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of `p` (this CTA's shared memory) in the shared window of CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p)), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}

__device__ __forceinline__ void dsmem_add_u32(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t dsmem_ld_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void dsmem_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Ascending bitonic sort of n = nt * R u64 keys by the first nt threads of the
// block, R per thread (thread t holds positions t*R .. t*R+R-1): strides below
// R in registers, below 32R by warp shuffles, the rest through shared memory.
// Every thread of the block calls it (the barriers need them all).
// ---------------------------------------------------------------------------

template <int R>
__device__ void bitonic_sort_blocked(unsigned long long* buf, int nt) {
  const int tid = threadIdx.x;
  const bool mine = tid < nt;
  const int n = nt * R;
  const int base = tid * R;
  unsigned long long v[R];
#pragma unroll
  for (int r = 0; r < R; ++r) v[r] = mine ? buf[base + r] : 0ull;
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32 * R) {
        if (mine) {
#pragma unroll
          for (int r = 0; r < R; ++r) buf[base + r] = v[r];
        }
        __syncthreads();
        for (int i = tid; i < n / 2; i += blockDim.x) {
          const int lo = 2 * i - (i & (stride - 1));
          const int hi = lo + stride;
          const bool up = (lo & size) == 0;
          const unsigned long long x = buf[lo], y = buf[hi];
          if ((x > y) == up) {
            buf[lo] = y;
            buf[hi] = x;
          }
        }
        __syncthreads();
        if (mine) {
#pragma unroll
          for (int r = 0; r < R; ++r) v[r] = buf[base + r];
        }
      } else if (mine) {
        if (stride >= R) {
          const int lx = stride / R;  // partner lane distance
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[r], lx);
            const int e = base + r;
            const bool up = (e & size) == 0;
            const bool lower = (e & stride) == 0;
            const unsigned long long mn = v[r] < o ? v[r] : o, mx = v[r] < o ? o : v[r];
            v[r] = (lower == up) ? mn : mx;
          }
        } else {
          // dispatch to a compile-time stride so the array is indexed statically
#pragma unroll
          for (int cs = R / 2; cs >= 1; cs >>= 1) {
            if (cs == stride) {
#pragma unroll
              for (int r = 0; r < R; ++r) {
                if ((r & cs) == 0) {
                  const bool up = ((base + r) & size) == 0;
                  if ((v[r] > v[r | cs]) == up) {
                    const unsigned long long t = v[r];
                    v[r] = v[r | cs];
                    v[r | cs] = t;
                  }
                }
              }
            }
          }
        }
      }
    }
  }
  if (mine) {
#pragma unroll
    for (int r = 0; r < R; ++r) buf[base + r] = v[r];
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// The selection kernel: one cluster of CS CTAs per (layer, sequence, head).
// CTA `rank` owns prefix positions [rank * NT*E, (rank+1) * NT*E) and keeps
// their keys in registers (position j = slice start + i*NT + tid for
// i < E). Histograms are summed in the leader (rank 0) through distributed
// shared memory; the leader sorts the kept keys and writes the output.
// ---------------------------------------------------------------------------

struct SelShared {
  uint32_t hist[kBins];        // this CTA's histogram
  uint32_t res[2];             // leader: (bin, count above)
  uint32_t cnt[kSelMaxCluster][2];  // leader: per rank (greater, equal) counts
  uint32_t warp_cnt[kSelWarps][2];
  uint32_t wsum[kSelWarps];
};

// Pooled score at stage position c of a zero-padded stage (s[c - R] ..
// s[c + R] are in bounds): sum in increasing position order, then / k
// (adding the zero pads leaves the sum unchanged); or the max.
template <int K>
__device__ __forceinline__ float pool_fixed(const float* s, int c, int kind) {
  constexpr int R = K / 2;
  if (kind == KVSEL_POOL_AVG) {
    float acc = 0.f;
#pragma unroll
    for (int d = -R; d <= R; ++d) acc += s[c + d];
    return acc / (float)K;
  }
  float m = s[c - R];
#pragma unroll
  for (int d = -R + 1; d <= R; ++d) m = fmaxf(m, s[c + d]);
  return m;
}

__device__ __forceinline__ float pool_any(const float* s, int c, int kind, int k) {
  switch (k) {
    case 1: return s[c];
    case 3: return pool_fixed<3>(s, c, kind);
    case 5: return pool_fixed<5>(s, c, kind);
    case 7: return pool_fixed<7>(s, c, kind);
    case 9: return pool_fixed<9>(s, c, kind);
    default: {
      const int R = k >> 1;
      if (kind == KVSEL_POOL_AVG) {
        float acc = 0.f;
        for (int d = -R; d <= R; ++d) acc += s[c + d];
        return acc / (float)k;
      }
      float m = s[c - R];
      for (int d = -R + 1; d <= R; ++d) m = fmaxf(m, s[c + d]);
      return m;
    }
  }
}

constexpr int kMaxE = 32;  // slice positions per thread of one CTA

// Variants that sort more than 8192 kept keys (R >= 16) need at least 139 KiB
// of shared memory, so they run one CTA per SM: they take the registers of two
// and keep twice as many gathered rows in flight.
template <int R> constexpr int kSelCtasPerSm = R >= 16 ? 1 : 2;
static_assert(kMaxE * kSelWarps <= kSelThreads && kMaxE * kSelWarps <= kBins,
              "the straddling slice's (row, warp) counts fit one per thread in the histogram");
template <int R> constexpr int kGatherU = R >= 16 ? 8 : 4;

template <int VW> struct CopyVec;
template <> struct CopyVec<16> { using T = uint4; };
template <> struct CopyVec<8> { using T = uint2; };
template <> struct CopyVec<4> { using T = uint32_t; };
template <> struct CopyVec<2> { using T = uint16_t; };

// Bounds of one instance's gather (checked in debug builds): source
// positions in [0, src_len) of its sequence, output rows before dst_end.
struct GatherBounds {
  int src_len;
  int64_t dst_end;
};

// Copies the instance's kept K and V rows (slot s <- position idx(s)) into
// out_K / out_V with VW-byte vectors, several rows in flight per thread.
template <int VW, int kU, typename IdxOf>
__device__ __forceinline__ void gather_rows(const SelectArgs& a, int n_rows, int64_t src_tok0,
                                            int64_t dst_row0, int h, GatherBounds gb,
                                            IdxOf idx_of) {
  using V = typename CopyVec<VW>::T;
  const int vpr = (int)(a.row_bytes / VW);
  const int total = n_rows * vpr;
  const char* kb = reinterpret_cast<const char*>(a.k);
  const char* vb = reinterpret_cast<const char*>(a.v);
  char* okb = reinterpret_cast<char*>(a.out_k);
  char* ovb = reinterpret_cast<char*>(a.out_v);
  (void)gb;
  for (int e0 = threadIdx.x; e0 < total; e0 += kSelThreads * kU) {
    V kv[kU], vv[kU];
    bool go[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * kSelThreads;
      go[u] = false;
      if (e < total) {
        const int s = e / vpr, vi = e - s * vpr;
        const int j = idx_of(s);
        go[u] = KVSEL_IN_BOUNDS(j >= 0 && j < gb.src_len && dst_row0 + s < gb.dst_end,
                                a.status);
        if (go[u]) {
          const int64_t src =
              ((src_tok0 + j) * a.kv_H + h / a.kv_div) * a.row_bytes + (int64_t)vi * VW;
          kv[u] = __ldcs(reinterpret_cast<const V*>(kb + src));
          vv[u] = __ldcs(reinterpret_cast<const V*>(vb + src));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * kSelThreads;
      if (go[u]) {
        const int s = e / vpr, vi = e - s * vpr;
        const int64_t dst = ((dst_row0 + s) * a.H + h) * a.row_bytes + (int64_t)vi * VW;
        __stcs(reinterpret_cast<V*>(okb + dst), kv[u]);
        __stcs(reinterpret_cast<V*>(ovb + dst), vv[u]);
      }
    }
  }
}

// kU rows of K and of V in flight per thread (8 where the kernel runs one
// CTA per SM and has the registers for it).
template <int kU, typename IdxOf>
__device__ __forceinline__ void gather_any(const SelectArgs& a, int n_rows, int64_t src_tok0,
                                           int64_t dst_row0, int h, GatherBounds gb,
                                           IdxOf idx_of) {
  switch (a.vec_bytes) {
    case 16: gather_rows<16, kU>(a, n_rows, src_tok0, dst_row0, h, gb, idx_of); break;
    case 8: gather_rows<8, kU>(a, n_rows, src_tok0, dst_row0, h, gb, idx_of); break;
    case 4: gather_rows<4, kU>(a, n_rows, src_tok0, dst_row0, h, gb, idx_of); break;
    default: gather_rows<2, kU>(a, n_rows, src_tok0, dst_row0, h, gb, idx_of); break;
  }
}

// ---------------------------------------------------------------------------
// Ascending sort of n = 512 * R u64 keys in `buf`: runs of 128 keys are
// sorted by the warps in registers and shuffles (bitonic, each lane holding 4
// consecutive keys), then rounds of merges double the sorted runs, each
// thread placing R consecutive outputs found by a merge-path search. During
// the merges key e sits at e + e / 16 (one 8-byte gap per 128 bytes), so the
// lanes' R-strided accesses spread over the banks. `tmp` and `buf` both hold
// n * 17 / 16 keys; the result ends in `buf`, unskewed. Every thread of the
// block calls it.
// ---------------------------------------------------------------------------

__device__ __forceinline__ int skw(int e) { return e + (e >> 4); }

template <int R>
__device__ void sort_runs_merge(unsigned long long* buf, unsigned long long* tmp) {
  constexpr int kPer = 4;                  // keys per lane in the run sort
  constexpr int kRun = 32 * kPer;
  constexpr int n = kSelThreads * R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int run = warp; run < n / kRun; run += kSelWarps) {
    const int base = run * kRun + lane * kPer;
    unsigned long long v[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) v[r] = buf[base + r];
#pragma unroll
    for (int size = 2; size <= kRun; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        if (stride >= kPer) {
          const int lx = stride / kPer;  // partner lane distance
#pragma unroll
          for (int r = 0; r < kPer; ++r) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[r], lx);
            const int e = lane * kPer + r;  // index within the run
            const bool up = size == kRun || (e & size) == 0;
            const bool lower = (e & stride) == 0;
            const unsigned long long mn = v[r] < o ? v[r] : o, mx = v[r] < o ? o : v[r];
            v[r] = (lower == up) ? mn : mx;
          }
        } else {
#pragma unroll
          for (int r = 0; r < kPer; ++r) {
            if ((r & stride) == 0) {
              const int e = lane * kPer + r;
              const bool up = size == kRun || (e & size) == 0;
              if ((v[r] > v[r | stride]) == up) {
                const unsigned long long t = v[r];
                v[r] = v[r | stride];
                v[r | stride] = t;
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kPer; ++r) tmp[skw(base + r)] = v[r];
  }
  __syncthreads();
  unsigned long long* src = tmp;
  unsigned long long* dst = buf;
  for (int len = kRun; len < n; len <<= 1) {
    const int out0 = tid * R;
    const int pbase = out0 / (2 * len) * (2 * len);
    const int d = out0 - pbase;
    // i = how many of the first d outputs come from A = [pbase, pbase + len)
    // (keys are distinct except the padding, and A wins ties: a stable merge)
    int lo = d > len ? d - len : 0, hi = d < len ? d : len;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (src[skw(pbase + mid)] <= src[skw(pbase + len + d - mid - 1)]) lo = mid + 1;
      else hi = mid;
    }
    int i = lo, j = d - lo;
#pragma unroll 4
    for (int r = 0; r < R; ++r) {
      const unsigned long long x = i < len ? src[skw(pbase + i)] : ~0ull;
      const unsigned long long y = j < len ? src[skw(pbase + len + j)] : ~0ull;
      const bool take_a = j >= len || (i < len && x <= y);
      dst[skw(out0 + r)] = take_a ? x : y;
      i += take_a;
      j += !take_a;
    }
    __syncthreads();
    unsigned long long* t = src;
    src = dst;
    dst = t;
  }
  // unskew into buf (through registers when the result is in buf itself)
  unsigned long long v[R];
#pragma unroll
  for (int r = 0; r < R; ++r) v[r] = src[skw(tid + r * kSelThreads)];
  __syncthreads();
#pragma unroll
  for (int r = 0; r < R; ++r) buf[tid + r * kSelThreads] = v[r];
  __syncthreads();
}

// Key pass for pooling width K <= 9: each thread pools four consecutive
// positions per round (2048 per round, one barrier each), reading their
// windows as aligned float4s from the zero-padded stage (vote of slice
// position i at stage[i + K/2]; the stage has 16 floats of slack past its end).
// Sums and maxima run in increasing position order, as in pool_fixed. Average
// pooling is ranked by the window sum itself: the average is the sum divided
// by the fixed width k > 0, the same order, and skipping the division keeps
// sums that differ from rounding to equal averages. Keys go to keys[i] =
// stage[i] after the round's barrier, counted into `hist` by their top 11 bits.
template <int K, bool kMaxPool>
__device__ void key_pass4(float* stage, int n, uint32_t* hist, int* status) {
  constexpr int kW = (K + 3 + 3) / 4;  // float4s covering positions i0 .. i0+3's windows
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t* keys = reinterpret_cast<uint32_t*>(stage);
  for (int c0 = 0; c0 < n; c0 += 4 * kSelThreads) {  // uniform trips
    const int i0 = c0 + 4 * tid;
    float w[4 * kW];
#pragma unroll
    for (int q = 0; q < kW; ++q) {
      const float4 f = i0 < n ? *reinterpret_cast<const float4*>(stage + i0 + 4 * q)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
      w[4 * q] = f.x;
      w[4 * q + 1] = f.y;
      w[4 * q + 2] = f.z;
      w[4 * q + 3] = f.w;
    }
    uint32_t key[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float v;
      if constexpr (!kMaxPool) {
        v = 0.f;
#pragma unroll
        for (int d = 0; d < K; ++d) v += w[u + d];
      } else {
        v = w[u];
#pragma unroll
        for (int d = 1; d < K; ++d) v = fmaxf(v, w[u + d]);
      }
      key[u] = i0 + u < n ? score_key(v, status) : 0u;
      add_bin(hist, i0 + u < n ? key[u] >> 21 : kNoBin, lane);
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i0 + u < n) keys[i0 + u] = key[u];
  }
}

// Ascending sort of the k kept composite keys buf[0..k) (~key << 32 |
// position: larger score first, then smaller position) through buckets of the
// high word w. The kept keys of one head sit in a band [lo, hi] of w (hi is
// the threshold's), denser towards the threshold, so the bucket of w follows
// the distance d = hi - w in a floating-point-like code: d itself below 2^mb,
// above that the position of d's leading bit and the mb bits after it, mb the
// most that keep the codes of [0, hi - lo] within kBins; bucket = kBins - 1 -
// code, which rises with w. Counts per bucket, an exclusive scan, a scatter
// into tmp by bucket, then every key is placed at its bucket's start plus the
// number of smaller keys in its bucket. Returns false, with buf unchanged,
// when a bucket holds more than kRankMax keys (many equal or clustered
// scores): the caller sorts another way. Every thread of the block calls it;
// `cnt` has kBins words; tmp holds k keys.
constexpr uint32_t kRankMax = 256;

__device__ __forceinline__ uint32_t dist_code(uint32_t d, int mb) {
  if (d < (1u << mb)) return d;
  const int e = (32 - __clz((int)d)) - mb;           // >= 1
  return ((uint32_t)e << mb) + ((d >> (e - 1)) - (1u << mb));
}

__device__ bool bucket_sort(unsigned long long* buf, unsigned long long* tmp, int k,
                            uint32_t* cnt, SelShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int i = tid; i < k; i += kSelThreads) {
    const uint32_t w = (uint32_t)(buf[i] >> 32);
    lo = min(lo, w);
    hi = max(hi, w);
  }
  for (int i = tid; i < kBins; i += kSelThreads) cnt[i] = 0u;
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) {
    sh.warp_cnt[warp][0] = lo;
    sh.warp_cnt[warp][1] = hi;
  }
  __syncthreads();
  lo = 0xFFFFFFFFu;
  hi = 0u;
  for (int w = 0; w < kSelWarps; ++w) {
    lo = min(lo, sh.warp_cnt[w][0]);
    hi = max(hi, sh.warp_cnt[w][1]);
  }
  // largest mb whose codes of [0, span] stay below kBins: (B - mb + 1) 2^mb
  // <= kBins for a span of B bits (B <= 11: every distance its own bucket)
  const uint32_t span = hi - lo;
  const int B = 32 - __clz((int)span);
  int mb = 10;
  while (mb > 0 && (B - mb + 1) * (1 << mb) > kBins) --mb;
  auto bucket = [&](unsigned long long v) {
    return (uint32_t)(kBins - 1) - dist_code(hi - (uint32_t)(v >> 32), mb);
  };
  for (int i = tid; i < k; i += kSelThreads) atomicAdd(&cnt[bucket(buf[i])], 1u);
  __syncthreads();
  // exclusive scan (thread t owns buckets 4t .. 4t+3) and the largest bucket
  constexpr int kPer = kBins / kSelThreads;
  uint32_t c[kPer], tot = 0, mx = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    c[q] = cnt[tid * kPer + q];
    tot += c[q];
    mx = max(mx, c[q]);
  }
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 31) sh.warp_cnt[warp][0] = incl;
  if (lane == 0) sh.warp_cnt[warp][1] = mx;
  __syncthreads();
  uint32_t run = incl - tot, biggest = 0;
  for (int w = 0; w < kSelWarps; ++w) {
    if (w < warp) run += sh.warp_cnt[w][0];
    biggest = max(biggest, sh.warp_cnt[w][1]);
  }
  if (biggest > kRankMax) return false;   // the same on every thread
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    cnt[tid * kPer + q] = run;
    run += c[q];
  }
  __syncthreads();
  for (int i = tid; i < k; i += kSelThreads) {
    const unsigned long long v = buf[i];
    tmp[atomicAdd(&cnt[bucket(v)], 1u)] = v;
  }
  __syncthreads();
  // cnt[b] is now the end of bucket b (and the start of b + 1)
  for (int i = tid; i < k; i += kSelThreads) {
    const unsigned long long v = tmp[i];
    const uint32_t b = bucket(v);
    const int b0 = b ? (int)cnt[b - 1] : 0, b1 = (int)cnt[b];
    int rank = 0;
    for (int j = b0; j < b1; ++j) rank += tmp[j] < v;
    buf[b0 + rank] = v;
  }
  __syncthreads();
  return true;
}

// Cluster CTA `rank` of `cs` copies output slots [rank * per, ...) of the
// instance's C: reads their positions from the leader's sorted keys (`sort_r`,
// its shared window) into `idx` and writes them to out_idx (`out`, stride H),
// waits at a cluster barrier (after which the leader's shared memory may go),
// then copies the rows.
template <int kU>
__device__ void select_copy_share(const SelectArgs& a, uint32_t k, int P, int cs, uint32_t rank,
                                  uint32_t sort_r, int32_t* idx, int32_t* out, int64_t src_tok0,
                                  int64_t out_row0, int h) {
  const int per = (a.C + cs - 1) / cs;
  const int s0 = min(a.C, (int)rank * per), s1 = min(a.C, s0 + per);
  for (int s = s0 + (int)threadIdx.x; s < s1; s += kSelThreads) {
    int32_t v;
    if (s < (int)k) {
      uint32_t lo;
      asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(lo) : "r"(sort_r + 8u * s) : "memory");
      v = (int32_t)lo;  // the position: low word of (~key << 32 | position)
    } else {
      v = P + (s - (int)k);
    }
    idx[s - s0] = v;
    out[(int64_t)s * a.H] = v;
  }
  __syncthreads();
  cluster_sync();
  gather_any<kU>(a, s1 - s0, src_tok0, out_row0 + s0, h, GatherBounds{P + a.W, out_row0 + a.C},
                 [&](int s) { return (int)idx[s]; });
}

// stage[c] = score of position jb + c (summed over `groups` planes T floats
// apart, in plane order) for c < count, 0 where that position is outside
// [0, P). Reads whole float4s aligned in memory (the planes share that
// alignment: T is a multiple of 4 when groups > 1), eight per thread in flight.
__device__ __forceinline__ void stage_scores_vec(const float* src, int64_t T, int groups,
                                                 int jb, int count, int P, float* stage) {
  constexpr int kU = 8;
  const int mis = (int)(((reinterpret_cast<uintptr_t>(src) >> 2) + (uintptr_t)(intptr_t)jb) & 3u);
  const int ja = jb - mis;                           // aligned group start (position)
  const int ng = (count + mis + 3) >> 2;
  for (int g0 = threadIdx.x; g0 < ng; g0 += kSelThreads * kU) {
    float4 r[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int g = g0 + u * kSelThreads;
      const int j = ja + 4 * g;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g < ng) {
        if (j >= 0 && j + 3 < P) {
          f = __ldcs(reinterpret_cast<const float4*>(src + j));
          for (int p = 1; p < groups; ++p) {
            const float4 e = __ldcs(reinterpret_cast<const float4*>(src + p * T + j));
            f.x += e.x;
            f.y += e.y;
            f.z += e.z;
            f.w += e.w;
          }
        } else {
          float t[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            t[e] = 0.f;
            if (j + e >= 0 && j + e < P)
              for (int p = 0; p < groups; ++p) t[e] += src[p * T + j + e];
          }
          f = make_float4(t[0], t[1], t[2], t[3]);
        }
      }
      r[u] = f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int g = g0 + u * kSelThreads;
      const int c = ja + 4 * g - jb;
      const float t[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (g < ng && c + e >= 0 && c + e < count) stage[c + e] = t[e];
    }
  }
}

template <bool CS1>
__device__ __forceinline__ void sel_sync() {
  if constexpr (CS1) __syncthreads();
  else cluster_sync();
}

__device__ __forceinline__ void flag_release(int* f) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(1) : "memory");
}

__device__ __forceinline__ int flag_acquire(const int* f) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
  return v;
}

// `selected` (may be null): set by thread 0 once the instance's indices are
// known, before its rows are copied.
template <int R, bool CS1>
__device__ void select_instance(const SelectArgs& a, int inst, uint32_t rank,
                                unsigned char* smem, SelShared& sh, bool gather_here,
                                int* selected) {
  const int pad = a.pool_inline ? (a.pool_k >> 1) : 0;
  float* stage = reinterpret_cast<float*>(smem);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  unsigned long long* sortbuf = reinterpret_cast<unsigned long long*>(smem + a.stage_bytes);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = inst % a.H;                    // inst = ((layer * S) + b) * H + h
  const int lb = inst / a.H;
  const int b = lb % a.n_seqs;
  const int layer = lb / a.n_seqs;
  const SeqDesc sd = a.seqs[b];
  const int L = sd.len;
  const int64_t out_row0 = (int64_t)layer * a.T_out + sd.out_off;
  int32_t* out = a.out_idx + out_row0 * a.H + h;
  const int64_t src_tok0 = (int64_t)layer * a.T + sd.tok_off;

  const int cs = CS1 ? 1 : a.cluster;
  if (L < a.C) {  // bypass: keep everything in order, each CTA a share of the rows
    if (selected && tid == 0) flag_release(selected);
    const int per = (L + cs - 1) / cs, s0 = min(L, (int)rank * per), s1 = min(L, s0 + per);
    for (int s = s0 + tid; s < s1; s += kSelThreads) out[(int64_t)s * a.H] = s;
    if (gather_here)
      gather_any<kGatherU<R>>(a, s1 - s0, src_tok0, out_row0 + s0, h,
                              GatherBounds{L, out_row0 + L}, [&](int s) { return s0 + s; });
    return;
  }
  const int P = L - a.W;
  const uint32_t k = (uint32_t)(a.C - a.W);
  const int j0 = (int)rank * a.slice;                  // slice start
  const int j1 = min(P, j0 + a.slice);                 // slice end (may be <= j0)
  const int n = max(0, j1 - j0);
  // the instance's score planes (several when the selection is shared by a
  // group of heads: their scores are summed in head order)
  const int64_t plane = ((int64_t)layer * a.H + h) * a.vote_group * a.T + sd.tok_off;
  const float* src = a.scores + plane;
  // the cluster's histogram, result and counts live in the leader
  // the leader's cluster histogram lives in its sort buffer, unused until
  // the kept keys are emitted (the launcher gives it at least kBins words)
  uint32_t* ghist = CS1 ? sh.hist : reinterpret_cast<uint32_t*>(sortbuf);
  const uint32_t ghist_r = CS1 ? 0u : dsmem_addr(ghist, 0);
  const uint32_t res_r = CS1 ? 0u : dsmem_addr(sh.res, 0);
  const uint32_t cnt_r = CS1 ? 0u : dsmem_addr(sh.cnt, 0);
  const uint32_t sort_r = CS1 ? 0u : dsmem_addr(sortbuf, 0);

  // ---- stage the scores with the zero halo; clear the first pass's histograms
  if (a.vote_group == 1 || (a.T & 3) == 0) {
    stage_scores_vec(src, a.T, a.vote_group, j0 - pad, n + 2 * pad, P, stage);
  } else {
    for (int c = tid; c < n + 2 * pad; c += kSelThreads) {
      const int j = j0 - pad + c;
      float v = 0.f;
      if (j >= 0 && j < P) {
        v = src[j];
        for (int g = 1; g < a.vote_group; ++g) v += src[(int64_t)g * a.T + j];
      }
      stage[c] = v;
    }
  }
  for (int i = tid; i < kBins; i += kSelThreads) {
    sh.hist[i] = 0;
    if (!CS1 && rank == 0) ghist[i] = 0;
  }
  __syncthreads();
  // ---- keys, counted into the first pass's histogram (top 11 bits) and
  // written at stage index j - j0, over votes no later window needs
  if (a.pool_inline && a.pool_k <= 9) {
    const bool mx = a.pool_kind != KVSEL_POOL_AVG;
    switch (a.pool_k) {
      case 1: key_pass4<1, false>(stage, n, sh.hist, a.status); break;
      case 3:
        if (mx) key_pass4<3, true>(stage, n, sh.hist, a.status);
        else key_pass4<3, false>(stage, n, sh.hist, a.status);
        break;
      case 5:
        if (mx) key_pass4<5, true>(stage, n, sh.hist, a.status);
        else key_pass4<5, false>(stage, n, sh.hist, a.status);
        break;
      case 7:
        if (mx) key_pass4<7, true>(stage, n, sh.hist, a.status);
        else key_pass4<7, false>(stage, n, sh.hist, a.status);
        break;
      default:
        if (mx) key_pass4<9, true>(stage, n, sh.hist, a.status);
        else key_pass4<9, false>(stage, n, sh.hist, a.status);
        break;
    }
  } else {
    // one position per thread and chunk (any width, or no pooling)
    for (int c0 = 0; c0 < n; c0 += kSelThreads) {  // uniform trips
      const int i = c0 + tid;
      uint32_t key = 0u, bin = kNoBin;
      if (i < n) {
        const float v = a.pool_inline ? pool_any(stage, i + pad, a.pool_kind, a.pool_k) : stage[i];
        key = score_key(v, a.status);
        bin = key >> 21;
      }
      add_bin(sh.hist, bin, lane);
      __syncthreads();
      if (i < n) keys[i] = key;
    }
  }
  if constexpr (!CS1) {
    for (int i = tid; i < kBins; i += kSelThreads)
      if (sh.hist[i]) dsmem_add_u32(ghist_r + 4u * i, sh.hist[i]);
  }
  sel_sync<CS1>();

  // ---- three radix passes over (11, 11, 10) bits, summed in the leader
  uint32_t krem = k, prefix = 0;
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : pass == 1 ? 10 : 0;
    const int nb = pass == 2 ? 1024 : kBins;
    const int hi_shift = pass == 0 ? 32 : pass == 1 ? 21 : 10;
    if (pass > 0) {
      for (int i = tid; i < nb; i += kSelThreads) sh.hist[i] = 0;
      __syncthreads();
      // four keys per thread from one 16-byte read (the stage has slack past
      // n); the keys left after the first pass spread over the bins, so
      // plain atomics
      for (int i4 = 4 * tid; i4 < n; i4 += 4 * kSelThreads) {
        const uint4 q = *reinterpret_cast<const uint4*>(keys + i4);
        const uint32_t kq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (i4 + e < n && (kq[e] >> hi_shift) == prefix)
            atomicAdd(&sh.hist[(kq[e] >> shift) & (uint32_t)(nb - 1)], 1u);
      }
      __syncthreads();
      if constexpr (!CS1) {
        for (int i = tid; i < nb; i += kSelThreads)
          if (sh.hist[i]) dsmem_add_u32(ghist_r + 4u * i, sh.hist[i]);
        cluster_sync();
      }
    }
    if (CS1 || rank == 0) {
      find_bin_block(ghist, nb, krem, sh.res, sh.wsum);
      if constexpr (!CS1)
        for (int i = tid; i < nb; i += kSelThreads) ghist[i] = 0;
    }
    sel_sync<CS1>();
    const uint32_t d = CS1 ? sh.res[0] : dsmem_ld_u32(res_r);
    const uint32_t above = CS1 ? sh.res[1] : dsmem_ld_u32(res_r + 4);
    prefix = (prefix << (pass == 2 ? 10 : 11)) | d;
    krem -= above;
  }
  const uint32_t thr = prefix;      // the key of the (C - W)-th largest score
  const uint32_t need_eq = krem;    // how many keys equal to thr are kept

  // ---- counts of this slice, exchanged through the leader
  uint32_t slice_gt = 0, slice_eq = 0, sel_base = 0, take_eq = 0;
  if constexpr (CS1) {
    // one slice: the keys above thr are the k - need_eq kept ones, and the
    // last pass counted the keys equal to thr in the bin of its low bits
    slice_gt = k - need_eq;
    slice_eq = sh.hist[thr & 1023u];
    take_eq = min(slice_eq, need_eq);
  } else {
    uint32_t my_gt = 0, my_eq = 0;
    for (int i = tid; i < n; i += kSelThreads) {
      const uint32_t key = keys[i];
      my_gt += key > thr;
      my_eq += key == thr;
    }
    my_gt = __reduce_add_sync(0xffffffffu, my_gt);
    my_eq = __reduce_add_sync(0xffffffffu, my_eq);
    if (lane == 0) {
      sh.warp_cnt[warp][0] = my_gt;
      sh.warp_cnt[warp][1] = my_eq;
    }
    __syncthreads();
    for (int w = 0; w < kSelWarps; ++w) {
      slice_gt += sh.warp_cnt[w][0];
      slice_eq += sh.warp_cnt[w][1];
    }
    if (tid == 0) {
      dsmem_st_u32(cnt_r + 8u * rank, slice_gt);
      dsmem_st_u32(cnt_r + 8u * rank + 4u, slice_eq);
    }
    cluster_sync();
    uint32_t eq_base = 0;
    for (int r = 0; r <= (int)rank; ++r) {
      const uint32_t g = dsmem_ld_u32(cnt_r + 8u * r), q = dsmem_ld_u32(cnt_r + 8u * r + 4u);
      const uint32_t take = need_eq > eq_base ? min(q, need_eq - eq_base) : 0u;
      if (r == (int)rank) {
        take_eq = take;
      } else {
        sel_base += g + take;
        eq_base += q;
      }
    }
  }
  // equal keys of this slice to keep: the first take_eq in position order
  const bool all_eq = take_eq == slice_eq;
  __syncthreads();  // warp_cnt is reused below

  // ---- emit kept keys (composite ~key << 32 | position) into the leader.
  // Phase 1 marks kept keys (bit m of `mask` for slice index tid + m*NT) and
  // counts them per warp; phase 2 writes them at consecutive places.
  uint32_t mask = 0;
  if (all_eq || take_eq == 0) {
    for (int m = 0, i = tid; m < kMaxE && i < n; ++m, i += kSelThreads) {
      const uint32_t key = keys[i];
      if (key > thr || (all_eq && key == thr)) mask |= 1u << m;
    }
  } else {
    // the straddling slice: rank the equal keys in position order (row m,
    // then warp, then lane): the equal keys of every (row, warp) counted by
    // ballots, one block-wide exclusive scan over those counts in that
    // order (at most kMaxE * kSelWarps = kSelThreads of them, one per
    // thread, in the histogram's words, free here), then each key's rank
    const int rows = min(kMaxE, (n + kSelThreads - 1) / kSelThreads);
    uint32_t* eqc = sh.hist;
    for (int m = 0; m < rows; ++m) {
      const int i = tid + m * kSelThreads;
      const uint32_t bal = __ballot_sync(0xffffffffu, i < n && keys[i] == thr);
      if (lane == 0) eqc[m * kSelWarps + warp] = __popc(bal);
    }
    __syncthreads();
    const uint32_t c = tid < rows * kSelWarps ? eqc[tid] : 0u;
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) sh.wsum[warp] = incl;
    __syncthreads();
    uint32_t before = incl - c;
    for (int w = 0; w < warp; ++w) before += sh.wsum[w];
    if (tid < rows * kSelWarps) eqc[tid] = before;
    __syncthreads();
    for (int m = 0; m < rows; ++m) {
      const int i = tid + m * kSelThreads;
      const uint32_t key = i < n ? keys[i] : 0u;
      const bool eq = i < n && key == thr;
      const uint32_t bal = __ballot_sync(0xffffffffu, eq);
      const uint32_t rank = eqc[m * kSelWarps + warp] + __popc(bal & ((1u << lane) - 1u));
      if ((i < n && key > thr) || (eq && rank < take_eq)) mask |= 1u << m;
    }
  }
  const uint32_t mine = __popc(mask);
  const uint32_t warp_total = __reduce_add_sync(0xffffffffu, mine);
  if (lane == 0) sh.warp_cnt[warp][0] = warp_total;
  __syncthreads();
  uint32_t pos = sel_base;
  for (int w = 0; w < warp; ++w) pos += sh.warp_cnt[w][0];
  uint32_t incl = mine;  // inclusive prefix of `mine` over the warp's lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  pos += incl - mine;
  for (int i = tid; mask; i += kSelThreads) {
    if (mask & 1u) {
      const unsigned long long ck = ((unsigned long long)(~keys[i]) << 32) | (uint32_t)(j0 + i);
      if constexpr (CS1) sortbuf[pos] = ck;
      else dsmem_st_u64(sort_r + 8u * pos, ck);
      ++pos;
    }
    mask >>= 1;
  }
  sel_sync<CS1>();
  if (!CS1 && gather_here && rank != 0) {
    // the leader sorts; then every CTA copies a share of the kept rows, its
    // positions read from the leader's sorted keys
    cluster_sync();
    select_copy_share<kGatherU<R>>(a, k, P, cs, rank, sort_r, reinterpret_cast<int32_t*>(smem), out,
                      src_tok0, out_row0, h);
    return;
  }
  if (rank != 0) return;

  // ---- leader: sort (larger score first, then smaller position), write the
  // slots, then (fused path) copy the kept K/V rows
  const int n2 = kSelThreads * R;
  // the staged keys are no longer needed: the stage (sized by the launcher)
  // is the scratch of the sorts
  unsigned long long* scratch = reinterpret_cast<unsigned long long*>(smem);
  if (R > 16 || !bucket_sort(sortbuf, scratch, (int)k, sh.hist, sh)) {
    for (int i = (int)k + tid; i < n2; i += kSelThreads) sortbuf[i] = ~0ull;
    __syncthreads();
    if constexpr (R <= 16) sort_runs_merge<R>(sortbuf, scratch);
    else bitonic_sort_blocked<R>(sortbuf, kSelThreads);
  }
  // out_idx: here, unless the cluster's CTAs write it with their copy shares
  if (CS1 || !gather_here) {
    for (int s = tid; s < (int)k; s += kSelThreads)
      out[(int64_t)s * a.H] = (int32_t)(sortbuf[s] & 0xFFFFFFFFull);
    for (int w = tid; w < a.W; w += kSelThreads) out[(int64_t)(k + w) * a.H] = P + w;
  }
  if (selected && tid == 0) flag_release(selected);
  if (!gather_here) return;
  if (CS1) {
    const int kk = (int)k;
    gather_any<kGatherU<R>>(a, a.C, src_tok0, out_row0, h, GatherBounds{L, out_row0 + a.C},
                            [&](int s) {
      return s < kk ? (int)(sortbuf[s] & 0xFFFFFFFFull) : P + (s - kk);
    });
  } else {
    __syncthreads();
    cluster_sync();
    select_copy_share<kGatherU<R>>(a, k, P, cs, rank, sort_r, reinterpret_cast<int32_t*>(smem), out,
                      src_tok0, out_row0, h);
  }
}

// Stagger (one-CTA instances with the gather): the two CTAs that start
// together on an SM would select (on-chip work) and then copy rows (HBM work)
// in step, and so would every SM, leaving HBM idle while all select. The
// second CTA to start on an SM therefore waits until the first has selected
// its instance; from then on one CTA of the pair tends to select while the
// other copies. The wait is on a CTA that is already running and is bounded
// (running out of time only costs speed).
template <int R, bool CS1, bool PACK = false>
__global__ void __launch_bounds__(kSelThreads, kSelCtasPerSm<R>) select_kernel(const __grid_constant__ SelectArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ SelShared sh;
  // a programmatic dependent launch may start before the scoring grid is
  // done: wait for it (and its memory) before reading any score (returns at
  // once when the launch has no such dependency)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int* selected = nullptr;
  if (CS1 && a.sched && a.gather) {
    __shared__ int s_slot;
    uint32_t sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    sm %= kSchedSms;
    int* flag = a.sched + 1 + kSchedSms + sm;
    if (threadIdx.x == 0) {
      s_slot = atomicAdd(a.sched + 1 + sm, 1);
      if (s_slot == 1) {
        const unsigned long long t0 = global_ns();
        while (!flag_acquire(flag) && global_ns() - t0 < a.stagger_limit_ns) __nanosleep(500);
      }
    }
    __syncthreads();
    if (s_slot == 0) selected = flag;
  }
  if constexpr (PACK) {
    // packed launch (a separate instantiation, so that the plain cluster
    // kernel keeps its registers): a whole-cluster instance, or one
    // single-CTA instance per CTA (block barriers only: no CTA touches
    // another's shared memory)
    const uint32_t rank = cluster_rank();
    const int32_t* e = a.pack + (int64_t)(blockIdx.x / a.cluster) * kSelMaxCluster;
    if (e[1] == kPackWhole) {
      select_instance<R, false>(a, e[0], rank, smem, sh, a.gather != 0, nullptr);
    } else if (e[rank] >= 0) {
      select_instance<R, true>(a, e[rank], 0u, smem, sh, a.gather != 0, nullptr);
    }
  } else {
    select_instance<R, CS1>(a, blockIdx.x / a.cluster, CS1 ? 0u : cluster_rank(), smem, sh,
                            a.gather != 0, selected);
  }
}

}  // namespace

cudaError_t launch_pool(const PoolArgs& a) {
  const int64_t blocks = (int64_t)a.layers * a.H * a.n_seqs;
  if (blocks == 0) return cudaSuccess;
  pool_kernel<<<(unsigned)blocks, 256, 0, a.stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_select(const SelectArgs& a0) {
  const int64_t blocks = (int64_t)a0.layers * a0.n_seqs * a0.H;
  if (blocks == 0) return cudaSuccess;
  SelectArgs a = a0;
  // one CTA per instance up to kSelThreads * kMaxE prefix positions, else a
  // cluster of CTAs with equal slices
  static_assert(kSelThreads * kMaxE == kSelSliceCap, "selection slice capacity");
  int cs = 1, slice = 1;
  select_geometry(a.max_prefix, &cs, &slice);
  if (cs > kSelMaxCluster) return cudaErrorInvalidValue;
  if (a.pack && cs == 1) return cudaErrorInvalidValue;
  a.cluster = cs;
  a.slice = slice;
  int n2 = kSelThreads;
  while (n2 < a.C - a.W) n2 <<= 1;
  const int pad = a.pool_inline ? a.pool_k / 2 : 0;
  // (16 floats of slack: the four-wide key pass reads whole float4s)
  size_t stage = ((((size_t)a.slice + 2 * pad + 16) * 4) + 15) & ~size_t(15);
  // the merge sort (R <= 16) skews its two buffers by 1/16
  const size_t merge_bytes = (size_t)n2 * 17 / 16 * 8;
  const bool merge = n2 <= kSelThreads * 16;
  if (merge) stage = std::max(stage, merge_bytes);
  stage = std::max(stage, (size_t)((a.C + cs - 1) / cs) * 4);           // a CTA's copy share
  a.stage_bytes = (int)stage;
  const size_t sortbuf = std::max(merge ? merge_bytes : (size_t)n2 * 8, (size_t)kBins * 4);
  const size_t smem = stage + sortbuf;
  void (*kern)(const SelectArgs) = nullptr;
#define KVSEL_SEL_CASE(RR)                                                           \
  case RR:                                                                           \
    kern = cs == 1 ? select_kernel<RR, true>                                         \
                   : (a.pack ? select_kernel<RR, false, true> : select_kernel<RR, false>); \
    break;
  switch (n2 / kSelThreads) {
    KVSEL_SEL_CASE(1)
    KVSEL_SEL_CASE(2)
    KVSEL_SEL_CASE(4)
    KVSEL_SEL_CASE(8)
    KVSEL_SEL_CASE(16)
    KVSEL_SEL_CASE(32)
    default: return cudaErrorInvalidValue;
  }
#undef KVSEL_SEL_CASE
  if (a.gather) {
    auto ok = [&](int vw) {
      if (a.row_bytes % vw) return false;
      for (const void* p : {a.k, a.v, (const void*)a.out_k, (const void*)a.out_v})
        if (reinterpret_cast<uintptr_t>(p) % vw) return false;
      return true;
    };
    a.vec_bytes = ok(16) ? 16 : ok(8) ? 8 : ok(4) ? 4 : 2;
  }
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((a.pack ? (int64_t)a.n_clusters : blocks) * cs));
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace kvsel
