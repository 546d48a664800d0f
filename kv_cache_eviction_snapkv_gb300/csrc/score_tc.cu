// Tensor-core scoring path for sm_103a: window logits on tcgen05, causal
// softmax row statistics and votes without a second read of K.
//
// Method: page "SnapKV: choosing the KV cache of a long prompt with an
// observation window", section "Votes must come from the full-prompt causal
// softmax" (投票必须来自完整提示词的因果 softmax): logits of the W window
// queries against every key scaled by 1/sqrt(D), causal mask (window row r =
// query P + r sees keys j <= P + r), softmax denominator over every visible
// key, vote of prefix key j = sum over rows of its probability. The section
// "A selection costs work before the cache gets smaller" (少读缓存以前，还要
// 支付一次选择成本) sizes that work at about B*H*W*L scores and B*H*W*L*D
// multiply-adds.
//
// Design (one CTA per SM, persistent, cooperative launch):
//   * work item = (layer, sequence, head, chunk of 128 * 512/Wp tokens), Wp =
//     W padded to 16/32/64; items go round-robin to CTAs;
//   * warp 0 streams K tiles (128 tokens x D, bf16) and the head's window
//     queries with TMA (128-byte swizzle) into a shared-memory ring;
//   * warp 1 issues tcgen05.mma (M = 128 tokens, N = Wp, K = D) so that each
//     tile's logits land in their own TMEM columns: the whole chunk's W x
//     tokens fp32 logits stay on chip (512 columns x 128 lanes);
//   * warps 2..9 (two per TMEM lane quarter, alternating tiles) read each
//     tile from TMEM as it completes and keep per-row running (max, sum of
//     2^(x - max)) with transposed butterfly reductions over the 32 tokens of
//     a warp;
//   * the chunk's row statistics go to global memory; the last chunk of an
//     instance to arrive merges them (fixed order) into M_r + log2 Z_r and
//     raises a flag; the others wait for it (bounded);
//   * the votes 2^(x - M_r - log2 Z_r) summed over rows are computed from the
//     logits still held in TMEM and written once (4 bytes per token).
// Every instance's chunks are resident at the same time (the host checks
// chunks <= CTAs), so the waits always end in a correct program; each wait
// is bounded anyway and reports KVSEL_ERR_TIMEOUT instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "kvsel_device.cuh"

namespace kvsel {
namespace {

constexpr int kGroupThreads = 256;   // one epilogue group: 8 warps, 2 per TMEM lane quarter
constexpr int kTileM = 128;           // tokens per MMA tile
constexpr int kMaxStages = 8;
constexpr int kTmemCols = 512;
constexpr int kSmemLimit = 232448;    // 227 KiB opt-in per CTA

struct TcParams {
  CUtensorMap tmk;  // K   viewed as (D, H, layers*T) bf16
  CUtensorMap tmq;  // q   viewed as (D, H, layers*S*W) bf16
  ScoreArgs a;
  int stages;
  int n_items;
};

// Epilogue groups for a padded window NW: two groups ping-pong over the two
// halves of TMEM when their per-thread state fits the register budget of
// 64 + 2 * 256 threads, else one group owns all of TMEM.
__host__ __device__ constexpr int groups_for(int nw) { return nw <= 32 ? 2 : 1; }
__host__ __device__ constexpr int threads_for(int nw) { return 64 + groups_for(nw) * kGroupThreads; }
__host__ __device__ constexpr int tiles_per_item(int nw) { return kTmemCols / groups_for(nw) / nw; }
// Registers per thread such that the CTA fits the register file of each SM
// sub-partition (16K registers; warps are spread round-robin over the four,
// so the busiest one holds ceil(warps / 4) warps): 18 warps -> 96, 10 -> 168.
__host__ __device__ constexpr int regs_for(int nw) {
  return (16384 / (((threads_for(nw) / 32) + 3) / 4 * 32)) / 8 * 8;
}

struct GroupState {
  unsigned long long tile_ready[32];    // MMA -> epilogue, one per TMEM tile
  unsigned long long tmem_empty;        // epilogue -> MMA, the group's TMEM half is free
  int snap;                             // abort flag as seen by one thread of the group
  int timed_out;
  float wm[4][64], wz[4][64];           // per lane quarter row statistics
  float fin[64];                        // M_r + log2 Z_r (+inf for padded rows)
  float2 cst[64];                       // this chunk's (reference, sum) per row
};

struct Misc {
  unsigned long long full[kMaxStages], empty[kMaxStages];
  unsigned long long qfull[2], qempty[2];
  unsigned long long mma_done;
  uint32_t tmem_base;
  int abort_flag;
  GroupState g[2];
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with `parity`; gives up when the limit passes or
// (if `abort_flag` is non-null) when another role has given up.
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                            unsigned long long limit_ns,
                                            const volatile int* abort_flag) {
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 31) == 0) {
      if (abort_flag && *abort_flag) return false;
      if (global_ns() - t0 > limit_ns) return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns,
                                          const volatile int* abort_flag) {
  return mbar_try(bar, parity) || mbar_wait_slow(bar, parity, limit_ns, abort_flag);
}

// Row statistics slots of the cross-chunk exchange: one 8-byte (reference,
// sum) pair per (work item, row), pre-filled with an all-ones pattern (a NaN
// reference, which a published pair never has). A relaxed 8-byte store is
// single-copy atomic, so a reader that sees a value other than the pattern
// sees the whole pair.
constexpr unsigned long long kEmptySlot = ~0ull;

__device__ __forceinline__ void slot_publish(unsigned long long* slot, float m, float z) {
  const unsigned long long v =
      ((unsigned long long)__float_as_uint(z) << 32) | __float_as_uint(m);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(slot), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long slot_read(const unsigned long long* slot) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(slot) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (SBO); version field 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;             // LBO (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;   // SBO
  d |= (uint64_t)1 << 46;             // descriptor version
  d |= (uint64_t)2 << 61;             // 128-byte swizzle
  return d;
}

// Instruction descriptor: D fp32, A and B bf16, both K-major, N and M.
__host__ __device__ constexpr uint32_t instr_desc(int n, int m) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

#define KVSEL_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                    "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : KVSEL_R8(0), KVSEL_R8(8)
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : KVSEL_R8(0), KVSEL_R8(8), KVSEL_R8(16), KVSEL_R8(24)
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// After tcgen05.wait::ld: ties each loaded value to an empty volatile asm that
// follows the wait, so no use of the value can be scheduled before the wait.
template <int N>
__device__ __forceinline__ void after_wait(float (&v)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+f"(v[i]));
}

template <int NW>
__device__ __forceinline__ void tmem_load_row(uint32_t taddr, float (&v)[NW]) {
  if constexpr (NW == 16) {
    tmem_ld16(taddr, v);
  } else {
#pragma unroll
    for (int c = 0; c < NW; c += 32) tmem_ld32(taddr + c, v + c);
  }
  tmem_wait_ld();
  after_wait(v);
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : KVSEL_R8(0)
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// One column, no wait (tcgen05.wait::ld and after_wait must follow).
__device__ __forceinline__ float tmem_ld1_nowait(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
  return __uint_as_float(r);
}

__device__ __forceinline__ float tmem_ld1(uint32_t taddr) {
  float v[1] = {tmem_ld1_nowait(taddr)};
  tmem_wait_ld();
  after_wait(v);
  return v[0];
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, float v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr),
               "r"(__float_as_uint(v))
               : "memory");
}

#define KVSEL_W8(i) "r"(__float_as_uint(v[i])), "r"(__float_as_uint(v[i + 1])), \
                    "r"(__float_as_uint(v[i + 2])), "r"(__float_as_uint(v[i + 3])), \
                    "r"(__float_as_uint(v[i + 4])), "r"(__float_as_uint(v[i + 5])), \
                    "r"(__float_as_uint(v[i + 6])), "r"(__float_as_uint(v[i + 7]))

// Stores N consecutive TMEM columns of this thread's lane (N = 8, 16 or 32).
template <int N>
__device__ __forceinline__ void tmem_store_cols(uint32_t taddr, const float (&v)[N]) {
  if constexpr (N == 8) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"r"(taddr), KVSEL_W8(0) : "memory");
  } else if constexpr (N == 16) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), KVSEL_W8(0), KVSEL_W8(8) : "memory");
  } else {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 ::"r"(taddr), KVSEL_W8(0), KVSEL_W8(8), KVSEL_W8(16), KVSEL_W8(24)
                 : "memory");
  }
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// N consecutive TMEM columns of this thread's lane (N = 8, 16 or 32).
template <int N>
__device__ __forceinline__ void tmem_load_cols_nowait(uint32_t taddr, float* v) {
  if constexpr (N == 8) tmem_ld8(taddr, v);
  else if constexpr (N == 16) tmem_ld16(taddr, v);
  else tmem_ld32(taddr, v);
}

template <int N>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float (&v)[N]) {
  tmem_load_cols_nowait<N>(taddr, v);
  tmem_wait_ld();
  after_wait(v);
}

// All threads of epilogue group g (named barriers 1, 2).
__device__ __forceinline__ void epi_bar(int g) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "n"(kGroupThreads) : "memory");
}

// The two warps of group g on TMEM lane quarter q (named barriers 3..10).
__device__ __forceinline__ void pair_bar(int g, int q) {
  asm volatile("bar.sync %0, 64;" ::"r"(3 + 4 * g + q) : "memory");
}

// (m1, z1) merged with (m2, z2), sums relative to the merged max.
__device__ __forceinline__ void merge_stats(float& m1, float& z1, float m2, float z2) {
  const float m = fmaxf(m1, m2);
  if (m == -INFINITY) return;
  const float a = m1 == -INFINITY ? 0.f : z1 * ex2(m1 - m);
  const float b = m2 == -INFINITY ? 0.f : z2 * ex2(m2 - m);
  m1 = m;
  z1 = a + b;
}

// Transposed butterfly over the 32 lanes for N (reference, sum) pairs per
// lane: afterwards lane l holds the merged pair of row l / (32 / N) (N <= 32).
template <int N>
__device__ __forceinline__ void reduce_stats(float (&m)[N], float (&z)[N], int lane) {
  int count = N;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (count >= 2) {
      const int half = count >> 1;
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < half) {
          const float sm = upper ? m[i] : m[i + half], sz = upper ? z[i] : z[i + half];
          float km = upper ? m[i + half] : m[i], kz = upper ? z[i + half] : z[i];
          const float rm = __shfl_xor_sync(0xffffffffu, sm, off);
          const float rz = __shfl_xor_sync(0xffffffffu, sz, off);
          merge_stats(km, kz, rm, rz);
          m[i] = km;
          z[i] = kz;
        }
      }
      count = half;
    } else {
      const float rm = __shfl_xor_sync(0xffffffffu, m[0], off);
      const float rz = __shfl_xor_sync(0xffffffffu, z[0], off);
      merge_stats(m[0], z[0], rm, rz);
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

template <int NW, int KD, bool LOGITS>
__global__ void __maxnreg__(regs_for(NW)) tc_score_kernel(const __grid_constant__ TcParams P) {
  constexpr int kHalves = KD / 64;
  constexpr int kStageBytes = kTileM * KD * 2;
  constexpr int kQBytes = NW * KD * 2;
  constexpr int kG = groups_for(NW);
  constexpr int kBufCols = kTmemCols / kG;     // TMEM columns of one group
  constexpr int kTiles = kBufCols / NW;        // tiles per work item
  constexpr uint32_t kIdesc = instr_desc(NW, kTileM);
  const ScoreArgs& a = P.a;
  const int stages = P.stages;
  const int W = a.W;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sk = smem;
  unsigned char* sq = sk + (size_t)stages * kStageBytes;
  Misc* ms = reinterpret_cast<Misc*>(sq + 2 * kQBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long limit = a.wait_limit_ns;
  volatile int* abort_flag = &ms->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&ms->full[s]), 1);
      mbar_init(smem_u32(&ms->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ms->qfull[b]), 1);
      mbar_init(smem_u32(&ms->qempty[b]), 1);
    }
    for (int g = 0; g < kG; ++g) {
      for (int t = 0; t < kTiles; ++t) mbar_init(smem_u32(&ms->g[g].tile_ready[t]), 1);
      mbar_init(smem_u32(&ms->g[g].tmem_empty), 8);
    }
    mbar_init(smem_u32(&ms->mma_done), 1);
    ms->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ms->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ms->tmem_base;

  uint32_t prod_armed = 0, prod_par = 0;  // producer lane: stages armed, last parity
  bool mma_issued = false;                // MMA lane: issued at least one MMA
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmk))
                   : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmq))
                   : "memory");
      const uint64_t pol_k = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, last_par = 0;
      bool ok = true;
      for (int it = 0, item = blockIdx.x; ok && item < P.n_items; ++it, item += gridDim.x) {
        const ItemPos ip = decode_item(a, item);
        const SeqDesc sd = a.seqs[ip.s];
        const int tok0 = ip.c * a.chunk_tokens;
        const int ntok = min(a.chunk_tokens, sd.len - tok0);
        const int ntiles = (ntok + kTileM - 1) / kTileM;
        const int qb = it & 1;
        if (!mbar_wait(smem_u32(&ms->qempty[qb]), ((it >> 1) & 1) ^ 1, limit, abort_flag)) {
          ok = false;
          break;
        }
        mbar_expect_tx(smem_u32(&ms->qfull[qb]), kQBytes);
        const int qrow = (int)(ip.layer * a.q_rows + (int64_t)sd.index * W);
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf)
          tma_load_3d(smem_u32(sq + qb * kQBytes + hf * NW * 128), &P.tmq,
                      smem_u32(&ms->qfull[qb]), hf * 64, ip.h, qrow, pol_q);
        const int krow0 = (int)(ip.layer * a.T + sd.tok_off + tok0);
        for (int t = 0; t < ntiles; ++t) {
          if (!mbar_wait(smem_u32(&ms->empty[stage]), phase ^ 1, limit, abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(smem_u32(&ms->full[stage]), kStageBytes);
#pragma unroll
          for (int hf = 0; hf < kHalves; ++hf)
            tma_load_3d(smem_u32(sk + stage * kStageBytes + hf * kTileM * 128), &P.tmk,
                        smem_u32(&ms->full[stage]), hf * 64, ip.h, krow0 + t * kTileM, pol_k);
          armed |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == stages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(a.status, KVSEL_ERR_TIMEOUT);
      }
      prod_armed = armed;
      prod_par = last_par;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sk_addr = smem_u32(sk), sq_addr = smem_u32(sq);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true, issued = false;
      for (int it = 0, item = blockIdx.x; ok && item < P.n_items; ++it, item += gridDim.x) {
        const ItemPos ip = decode_item(a, item);
        const SeqDesc sd = a.seqs[ip.s];
        const int tok0 = ip.c * a.chunk_tokens;
        const int ntok = min(a.chunk_tokens, sd.len - tok0);
        const int ntiles = (ntok + kTileM - 1) / kTileM;
        const int qb = it & 1;
        const int g = it % kG;
        GroupState& gs = ms->g[g];
        if (!mbar_wait(smem_u32(&gs.tmem_empty), ((it / kG) & 1) ^ 1, limit, abort_flag) ||
            !mbar_wait(smem_u32(&ms->qfull[qb]), (it >> 1) & 1, limit, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int t = 0; t < ntiles; ++t) {
          if (!mbar_wait(smem_u32(&ms->full[stage]), phase, limit, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(g * kBufCols + t * NW);
#pragma unroll
          for (int kk = 0; kk < KD / 16; ++kk) {
            const uint32_t a_addr =
                sk_addr + stage * kStageBytes + (kk >> 2) * (kTileM * 128) + (kk & 3) * 32;
            const uint32_t b_addr = sq_addr + qb * kQBytes + (kk >> 2) * (NW * 128) + (kk & 3) * 32;
            tc_mma(d_tmem, smem_desc(a_addr), smem_desc(b_addr), kIdesc, kk > 0 ? 1u : 0u);
          }
          issued = true;
          tc_commit(smem_u32(&ms->empty[stage]));
          tc_commit(smem_u32(&gs.tile_ready[t]));
          if (++stage == stages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) tc_commit(smem_u32(&ms->qempty[qb]));
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(a.status, KVSEL_ERR_TIMEOUT);
      }
      mma_issued = issued;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int g = (warp - 2) >> 3;          // group: the CTA's items it = g, g + kG, ...
    GroupState& gs = ms->g[g];
    const int e = (warp - 2) & 7;
    const int quarter = warp & 3;           // TMEM lanes 32*quarter .. +31
    const int sub = e >> 2;                 // row half (votes) / tile parity (logits)
    const int et = threadIdx.x - 64 - g * kGroupThreads;   // 0..255 within the group
    const uint32_t lane_addr =
        tmem_base + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(g * kBufCols);
    uint32_t tph = 0;                       // per tile barrier: parity of the next phase
    for (int it = g, item = blockIdx.x + g * gridDim.x; item < P.n_items;
         it += kG, item += kG * gridDim.x) {
      const ItemPos ip = decode_item(a, item);
      const SeqDesc sd = a.seqs[ip.s];
      const int tok0 = ip.c * a.chunk_tokens;
      const int ntok = min(a.chunk_tokens, sd.len - tok0);
      const int ntiles = (ntok + kTileM - 1) / kTileM;
      const int prefix = sd.len - W;
      const int64_t plane = ((int64_t)ip.layer * a.H + ip.h) * a.T + sd.tok_off;
      bool ok = true;

      if constexpr (LOGITS) {
        for (int t = sub; t < ntiles; t += 2) {
          if (ok)
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&gs.tile_ready[t]), (tph >> t) & 1,
                                                   limit, abort_flag));
          tph ^= 1u << t;
          if (!ok) continue;
          tc_fence_after();
          float v[NW];
          tmem_load_row<NW>(lane_addr + (uint32_t)(t * NW), v);
          const int tok = tok0 + t * kTileM + 32 * quarter + lane;
          if (tok < sd.len) {
            const int64_t base = ((int64_t)ip.layer * a.H + ip.h) * W;
#pragma unroll
            for (int r = 0; r < NW; ++r)
              if (r < W) a.logits[(base + r) * a.T + sd.tok_off + tok] = v[r] * a.scale;
          }
        }
        if (!ok) {
          *abort_flag = 1;
          record_status(a.status, KVSEL_ERR_TIMEOUT);
        }
      } else {
        // ---- pass A: per-row softmax statistics of this warp's tokens. The two
        // warps of a lane quarter split the rows (half `sub` = rows sub*NH ..
        // sub*NH + NH - 1) and see every tile. Each thread keeps, per row, a
        // reference value and the sum of 2^(x - reference) over its own
        // tokens; the reference moves only when a logit exceeds it by more
        // than 32 (so no term exceeds 2^32), which after the first visible
        // token is rare. The exponentials replace the logits in TMEM.
        constexpr int NH = NW / 2;
        float mref[NH], zsum[NH];
#pragma unroll
        for (int i = 0; i < NH; ++i) {
          mref[i] = -INFINITY;
          zsum[i] = 0.f;
        }
        bool bad = false;
        const int row0 = sub * NH;
        for (int t = 0; t < ntiles; ++t) {
          // warp-uniform: the TMEM loads and stores below are .sync.aligned
          if (ok)
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&gs.tile_ready[t]), (tph >> t) & 1,
                                                   limit, abort_flag));
          tph ^= 1u << t;
          if (!ok) continue;
          tc_fence_after();
          float x[NH];
          tmem_load_cols<NH>(lane_addr + (uint32_t)(t * NW + row0), x);
          const int tok = tok0 + t * kTileM + 32 * quarter + lane;
          // rows visible to this token: row0 + i < W, and tok <= P + row0 + i
          const int lo = max(0, tok - prefix - row0);
          const int hi = tok < sd.len ? min(NH, W - row0) : 0;
          bool need = false, fixany = false;
#pragma unroll
          for (int i = 0; i < NH; ++i) {
            x[i] *= a.scale_log2;
            const bool in = i < hi;
            if (in && !finite_f(x[i])) bad = true;
            const bool up = in && i >= lo && x[i] > mref[i] + 32.f;
            need |= up;
            fixany |= up && mref[i] != -INFINITY;
          }
          if (__any_sync(0xffffffffu, fixany)) {
            // A logit more than 2^32 above a finite reference (rare): rescale
            // the exponentials already stored for that row before moving it.
#pragma unroll
            for (int i = 0; i < NH; ++i) {
              const bool fix = i < hi && i >= lo && x[i] > mref[i] + 32.f &&
                               mref[i] != -INFINITY;
              const float f = fix ? ex2(mref[i] - x[i]) : 1.f;
              if (__any_sync(0xffffffffu, fix)) {
                for (int tp = 0; tp < t; ++tp) {
                  const uint32_t ca = lane_addr + (uint32_t)(tp * NW + row0 + i);
                  tmem_st1(ca, tmem_ld1(ca) * f);
                }
                tmem_wait_st();
              }
            }
          }
          if (need) {  // first visible token of a row, or the rare jump above
#pragma unroll
            for (int i = 0; i < NH; ++i) {
              if (i < hi && i >= lo && x[i] > mref[i] + 32.f) {
                zsum[i] = mref[i] == -INFINITY ? 0.f : zsum[i] * ex2(mref[i] - x[i]);
                mref[i] = x[i];
              }
            }
          }
#pragma unroll
          for (int i = 0; i < NH; ++i) {
            x[i] = (i < hi && i >= lo) ? ex2(x[i] - mref[i]) : 0.f;
            zsum[i] += x[i];
          }
          tmem_store_cols<NH>(lane_addr + (uint32_t)(t * NW + row0), x);
        }
        tmem_wait_st();
        float mkeep[NH];
#pragma unroll
        for (int i = 0; i < NH; ++i) mkeep[i] = mref[i];
        if (bad) record_status(a.status, KVSEL_ERR_NONFINITE);
        if (!ok) *abort_flag = 1;
        reduce_stats<NH>(mref, zsum, lane);
        constexpr int kLanesPerRow = 32 / NH;
        if (lane % kLanesPerRow == 0) {
          gs.wm[quarter][row0 + lane / kLanesPerRow] = mref[0];
          gs.wz[quarter][row0 + lane / kLanesPerRow] = zsum[0];
        }
        // Control flow around the named barriers must be uniform across the
        // group, so decisions use values one thread published between
        // barriers, never a direct read of the abort flag.
        epi_bar(g);
        if (et == 0) {
          gs.snap = *abort_flag;
          gs.timed_out = gs.snap;
        }
        epi_bar(g);
        const bool aborted = gs.snap != 0;
        // ---- chunk statistics: each row's (reference, sum) goes to this
        // item's slot; then every chunk of the instance polls all the slots of
        // the instance and merges them in the same fixed order
        unsigned long long* slots = reinterpret_cast<unsigned long long*>(a.part);
        if (!aborted && et < W) {
          float m = gs.wm[0][et], z = gs.wz[0][et];
#pragma unroll
          for (int w = 1; w < 4; ++w) merge_stats(m, z, gs.wm[w][et], gs.wz[w][et]);
          if (m != m) m = INFINITY;  // keep the empty pattern unique (NONFINITE is recorded)
          if (!(a.inject == 1 && item == 0))
            slot_publish(slots + (int64_t)item * a.wpad + et, m, z);
        }
        const int nc = sd.n_chunks;
        {
          constexpr int tpr = kGroupThreads / NW;   // threads per row: 16, 8 or 4
          constexpr int kPoll = 8;                  // slots read per batch
          const int r = et / tpr, sb = et % tpr;
          const unsigned long long* p0 =
              slots + ((int64_t)ip.layer * a.items_per_layer + sd.item_base +
                       (int64_t)ip.h * nc) * a.wpad + r;
          float m = -INFINITY, z = 0.f;
          bool late = false;
          if (!aborted && r < W) {
            const unsigned long long t0 = global_ns();
            for (int cb = sb; cb < nc && !late; cb += kPoll * tpr) {
              unsigned long long v[kPoll];
              uint32_t pending = 0;
#pragma unroll
              for (int k = 0; k < kPoll; ++k) {
                v[k] = kEmptySlot;
                if (cb + k * tpr < nc) pending |= 1u << k;
              }
              for (;;) {
#pragma unroll
                for (int k = 0; k < kPoll; ++k) {
                  if (pending & (1u << k)) {
                    v[k] = slot_read(p0 + (int64_t)(cb + k * tpr) * a.wpad);
                    if (v[k] != kEmptySlot) pending &= ~(1u << k);
                  }
                }
                if (!pending) break;
                if (global_ns() - t0 > limit) {
                  late = true;
                  break;
                }
                __nanosleep(64);
              }
#pragma unroll
              for (int k = 0; k < kPoll; ++k)
                if (!late && cb + k * tpr < nc)
                  merge_stats(m, z, __uint_as_float((uint32_t)v[k]),
                              __uint_as_float((uint32_t)(v[k] >> 32)));
            }
          }
          if (late) {
            gs.timed_out = 1;
            record_status(a.status, KVSEL_ERR_TIMEOUT);
          }
#pragma unroll
          for (int off = tpr / 2; off >= 1; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const float z2 = __shfl_xor_sync(0xffffffffu, z, off);
            merge_stats(m, z, m2, z2);
          }
          if (sb == 0) gs.fin[r] = r < W ? m + log2f(z) : INFINITY;
        }
        epi_bar(g);
        // ---- pass C: vote of a prefix token = sum over rows of its stored
        // exponential times c_r = 2^(reference_r - M_r - log2 Z_r). Each warp
        // sums its half of the rows for every tile and leaves the partial in
        // TMEM (in the first column of its half, already consumed); after a
        // barrier of the warp pair, each warp adds the two partials of
        // alternate tiles (half 0 first, a fixed order) and writes the votes.
        if (!gs.timed_out) {
          float c[NH];
#pragma unroll
          for (int i = 0; i < NH; ++i) c[i] = ex2(mkeep[i] - gs.fin[row0 + i]);
          constexpr int kB = NH <= 8 ? 2 : 1;  // tiles per batch of TMEM loads
          for (int t0b = 0; t0b < ntiles; t0b += kB) {
            float ev[kB * NH];
#pragma unroll
            for (int b = 0; b < kB; ++b)
              if (t0b + b < ntiles)
                tmem_load_cols_nowait<NH>(lane_addr + (uint32_t)((t0b + b) * NW + row0),
                                          ev + b * NH);
            tmem_wait_ld();
            after_wait(ev);
#pragma unroll
            for (int b = 0; b < kB; ++b) {
              if (t0b + b < ntiles) {
                float p = 0.f;
#pragma unroll
                for (int i = 0; i < NH; ++i) p = fmaf(ev[b * NH + i], c[i], p);
                tmem_st1(lane_addr + (uint32_t)((t0b + b) * NW + row0), p);
              }
            }
          }
          tmem_wait_st();
          tc_fence_before();
          pair_bar(g, quarter);
          tc_fence_after();
          constexpr int kHalfTiles = kTiles / 2;  // tiles finished by each warp of the pair
          float pv[2 * kHalfTiles];
#pragma unroll
          for (int k = 0; k < kHalfTiles; ++k) {
            const int t = sub + 2 * k;
            if (t < ntiles) {
              pv[2 * k] = tmem_ld1_nowait(lane_addr + (uint32_t)(t * NW));
              pv[2 * k + 1] = tmem_ld1_nowait(lane_addr + (uint32_t)(t * NW + NH));
            }
          }
          tmem_wait_ld();
          after_wait(pv);
#pragma unroll
          for (int k = 0; k < kHalfTiles; ++k) {
            const int t = sub + 2 * k;
            const int tok = tok0 + t * kTileM + 32 * quarter + lane;
            if (t < ntiles && tok < sd.len)
              a.votes[plane + tok] = tok < prefix ? pv[2 * k] + pv[2 * k + 1] : 0.f;
          }
        }
        if (et == 0 && gs.timed_out) *abort_flag = 1;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&gs.tmem_empty));
      if constexpr (!LOGITS) {
        if (et == 0) gs.snap = *abort_flag;
        epi_bar(g);  // every thread of the group has read timed_out / fin
        if (gs.snap) break;
      } else {
        if (!ok) break;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // Every role has left its loop, so the abort flag is final. After an abort,
  // drain what is still in flight before the shared memory and TMEM go away:
  // the producer waits for the last copy it started into each stage, the MMA
  // issuer for its last instruction (both bounded, ignoring the abort flag).
  if (ms->abort_flag) {
    if (warp == 0 && lane == 0) {
      for (int s = 0; s < stages; ++s)
        if (prod_armed & (1u << s))
          mbar_wait(smem_u32(&ms->full[s]), (prod_par >> s) & 1, limit, nullptr);
    }
    if (warp == 1 && lane == 0 && mma_issued) {
      tc_commit(smem_u32(&ms->mma_done));
      mbar_wait(smem_u32(&ms->mma_done), 0, limit, nullptr);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, int D, int H, int64_t rows, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int NW, int KD, bool LOGITS>
cudaError_t launch_t(const ScoreArgs& a, int grid) {
  constexpr int kStageBytes = kTileM * KD * 2;
  constexpr int kQBytes = NW * KD * 2;
  const size_t fixed = 1024 + 2 * kQBytes + sizeof(Misc);
  int stages = (int)((kSmemLimit - fixed) / kStageBytes);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + (size_t)stages * kStageBytes;
  TcParams p;
  std::memset(&p, 0, sizeof(p));
  if (!make_map(&p.tmk, a.k, a.D, a.H, (int64_t)a.layers * a.T, kTileM) ||
      !make_map(&p.tmq, a.q, a.D, a.H, (int64_t)a.layers * a.q_rows, NW))
    return cudaErrorInvalidValue;
  p.a = a;
  p.stages = stages;
  p.n_items = a.layers * a.items_per_layer;
  auto kern = tc_score_kernel<NW, KD, LOGITS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(threads_for(NW));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool LOGITS>
cudaError_t launch_mode(const ScoreArgs& a, int grid) {
  const int nw = tc_window_pad(a.W);
  if (a.D == 128) {
    if (nw == 16) return launch_t<16, 128, LOGITS>(a, grid);
    if (nw == 32) return launch_t<32, 128, LOGITS>(a, grid);
    if (nw == 64) return launch_t<64, 128, LOGITS>(a, grid);
  } else if (a.D == 64) {
    if (nw == 16) return launch_t<16, 64, LOGITS>(a, grid);
    if (nw == 32) return launch_t<32, 64, LOGITS>(a, grid);
    if (nw == 64) return launch_t<64, 64, LOGITS>(a, grid);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int tc_window_pad(int W) {
  if (W < 1) return 0;
  if (W <= 16) return 16;
  if (W <= 32) return 32;
  if (W <= 64) return 64;
  return 0;
}

int tc_chunk_tokens(int W) {
  const int nw = tc_window_pad(W);
  return nw ? kTileM * tiles_per_item(nw) : 0;
}

int tc_max_grid(int sm_count) { return sm_count; }

int tc_max_chunks(int W, int sm_count) {
  const int nw = tc_window_pad(W);
  return nw ? groups_for(nw) * tc_max_grid(sm_count) : 0;
}

bool tc_eligible(int dtype, int D, int W, const void* q, const void* k) {
  if (dtype != KVSEL_BF16 || (D != 64 && D != 128) || tc_window_pad(W) == 0) return false;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k)) & 15) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_tc_score(const ScoreArgs& a, bool logits_mode, int grid) {
  if ((int64_t)a.layers * a.T >= 0x7fffffffLL || (int64_t)a.layers * a.q_rows >= 0x7fffffffLL)
    return cudaErrorInvalidValue;
  return logits_mode ? launch_mode<true>(a, grid) : launch_mode<false>(a, grid);
}

}  // namespace kvsel
