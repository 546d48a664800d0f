// Jacap scoring: leverage of each prefix token's value direction under the
// capacity matrix, for a selection that keeps the highest scores.
//
// Method: pages "Jacap reading notes" / "Jacap technical review", section 6
// (practical approximation) and section 7 (Algorithm 1, one eviction event):
// z_i = k_i . mu_Q / (tau sqrt(d)), alpha = softmax(z) over the pool, kappa_i =
// k_i^T Lambda_Q k_i, w_i = [alpha_i (1 - alpha_i)]^2 kappa_i / d, u_i = v_i,
// A = I + sum_i w_i u_i u_i^T, one Cholesky factor of A, r_i = w_i u_i^T A^{-1}
// u_i; section 11 (Algorithm 2): mu_Q and the diagonal Lambda_Q are the
// running mean and second moment of the queries, here over the W window
// queries (our reading for a prompt-time selection), started from the first.
//
// Four kernels per call, bf16 and d = 128 (the tensor-core operands):
//   stats    one CTA per 512 prefix rows: the window statistics (recomputed by
//            every CTA, W x d work), then z (base-2 units) and kappa per row
//            (eight lanes per row, coalesced), and the chunk's max and sum of
//            2^z. HBM-bound on K.
//   gram     one CTA per range of 128-token tiles of an instance: merges the
//            instance's softmax partials, computes w, scales each V tile by
//            sqrt(w) and transposes it into a K-major, 128-byte-swizzled
//            buffer (dimensions as rows, tokens as K), on which one tcgen05.mma
//            with A = B = that buffer accumulates sum_t w_t v_t v_t^T (128 x 128,
//            fp32, in TMEM); the partial is written out. HBM-bound on V.
//   factor   one CTA per instance: A = I + the partials in a fixed order, the
//            Cholesky factor and L^{-1} in fp32 shared memory, written as two
//            bf16 matrices hi + lo (hi = bf16(L^{-1}), lo = bf16(L^{-1} - hi)).
//   leverage one CTA per 8 tiles: y_t = L^{-1} v_t for 128 tokens at a time by
//            tcgen05.mma (A = the V tile as loaded, B = L^{-1} hi, then lo,
//            accumulated), r_t = w_t |y_t|^2 in the epilogue. HBM-bound on V.
// Every wait is bounded (KVSEL_ERR_TIMEOUT, then the roles drain and return).
#include <cmath>
#include <cstring>

#include "kvsel_device.cuh"
#include "tc_common.cuh"

namespace kvsel {
namespace {

constexpr int kJD = 128;                      // head dimension of the tensor path
constexpr int kJTile = 128;                   // tokens per MMA tile
constexpr int kJTileBytes = kJTile * kJD * 2; // one V tile, bf16: 32 KiB
constexpr int kAtom = kJTile * 128;           // one 64-column swizzle atom of a tile: 16 KiB

template <typename F>
__device__ __forceinline__ int find_jseq(const JacapArgs& a, int rem, F base_of) {
  return upper_find(a.n_scored, rem, base_of);
}

// ---------------------------------------------------------------------------
// stats
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(256) jacap_stats_kernel(const __grid_constant__ JacapArgs a) {
  __shared__ float mu_s[kJD], lam_s[kJD];
  __shared__ float wm[8], wl[8];
  __shared__ __align__(16) __nv_bfloat16 qs[32][kJD];   // 32 window queries at a time
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int item = blockIdx.x;
  const int layer = item / a.chunks_per_layer;
  const int rem = item - layer * a.chunks_per_layer;
  const JSeq& sq = a.seqs[find_jseq(a, rem, [&](int i) { return a.seqs[i].chunk_base; })];
  const int local = rem - sq.chunk_base;
  const int h = local / sq.n_chunks, c = local - h * sq.n_chunks;
  const int P = sq.len - a.W;
  const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(a.q);
  {
    // the window statistics: rows staged 32 at a time with every thread
    // loading (16 bytes each), the recursion run by one thread per dimension
    const int64_t row0 = (int64_t)layer * a.S * a.W + (int64_t)sq.index * a.W;
    float mu = 0.f, m2 = 0.f;
    for (int r0 = 0; r0 < a.W; r0 += 32) {
      const int nr = min(32, a.W - r0);
      for (int e = tid; e < nr * (kJD / 8); e += blockDim.x) {
        const int r = e / (kJD / 8), c = e - r * (kJD / 8);
        *reinterpret_cast<uint4*>(&qs[r][c * 8]) = *reinterpret_cast<const uint4*>(
            qb + ((row0 + r0 + r) * a.H + h) * kJD + c * 8);
      }
      __syncthreads();
      if (tid < kJD) {
        for (int r = 0; r < nr; ++r) {
          const float q = __bfloat162float(qs[r][tid]);
          if (r0 + r == 0) {
            mu = q;
            m2 = q * q;
          } else {
            mu = a.beta * mu + (1.f - a.beta) * q;
            m2 = a.beta * m2 + (1.f - a.beta) * (q * q);
          }
        }
      }
      __syncthreads();
    }
    if (tid < kJD) {
      mu_s[tid] = mu * (1.4426950408889634f / (a.tau * sqrtf((float)kJD)));
      lam_s[tid] = fmaxf(m2 - mu * mu, a.eps);
    }
  }
  __syncthreads();
  const int grp = lane >> 3, sub = lane & 7;
  float mu[16], lam[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    mu[e] = mu_s[sub * 16 + e];
    lam[e] = lam_s[sub * 16 + e];
  }
  const int r_begin = c * kJChunk, r_end = min(P, r_begin + kJChunk);
  const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(a.k);
  const int64_t plane = ((int64_t)layer * a.H + h) * a.T + sq.tok_off;
  float m = -INFINITY, l = 0.f;
  for (int wb = r_begin + warp * 4; wb < r_end; wb += 32) {   // warp-uniform trips
    const int row = wb + grp;
    const int j = min(row, r_end - 1);
    const uint4* src = reinterpret_cast<const uint4*>(
        kb + (((int64_t)layer * a.T + sq.tok_off + j) * a.H + h) * kJD + sub * 16);
    const uint4 k0 = __ldcs(src), k1 = __ldcs(src + 1);
    const uint32_t w[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
    float z = 0.f, kap = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float kv = __uint_as_float((e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16));
      z = fmaf(mu[e], kv, z);
      kap = fmaf(lam[e] * kv, kv, kap);
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      z += __shfl_xor_sync(0xffffffffu, z, off);
      kap += __shfl_xor_sync(0xffffffffu, kap, off);
    }
    if (row < r_end) {
      if (sub == 0) a.zk[plane + row] = make_float2(z, kap);
      const float mx = fmaxf(m, z);
      l = (m == -INFINITY ? 0.f : l * ex2(m - mx)) + ex2(z - mx);
      m = mx;
    }
  }
#pragma unroll
  for (int off = 8; off <= 16; off <<= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float lo = __shfl_xor_sync(0xffffffffu, l, off);
    const float mx = fmaxf(m, mo);
    l = (m == -INFINITY ? 0.f : l * ex2(m - mx)) + (mo == -INFINITY ? 0.f : lo * ex2(mo - mx));
    m = mx;
  }
  if (lane == 0) {
    wm[warp] = m;
    wl[warp] = l;
  }
  __syncthreads();
  if (tid == 0) {
    float mx = -INFINITY, sum = 0.f;
    for (int w = 0; w < 8; ++w) mx = fmaxf(mx, wm[w]);
    for (int w = 0; w < 8; ++w)
      if (wm[w] != -INFINITY) sum = fmaf(wl[w], ex2(wm[w] - mx), sum);
    a.part[2 * (int64_t)item] = mx;
    a.part[2 * (int64_t)item + 1] = sum;
    if (!finite_f(mx) || !finite_f(sum)) record_status(a.status, KVSEL_ERR_NONFINITE);
  }
}

// ---------------------------------------------------------------------------
// gram
// ---------------------------------------------------------------------------

constexpr int kGStages = 3;                    // V tile ring
constexpr int kGThreads = 320;                 // warp 0 TMA, warp 1 MMA, warps 2..9 transpose
constexpr int kGWork = 256;                    // transposing threads

struct GramSmem {
  unsigned long long full[kGStages], empty[kGStages];
  unsigned long long tfull[2], tempty[2];
  unsigned long long done;
  unsigned long long drain;                    // abort path: the MMA issuer's last commit
  uint32_t tmem_base;
  int abort_flag;
  float norm_m, norm_s;                        // the instance's base-2 softmax max and sum
  float sw[2][kJTile];                         // sqrt(w) of a tile's tokens (double buffer)
};

struct GramParams {
  CUtensorMap tmv;                             // V as (D, H, layers * T)
  JacapArgs a;
};

__device__ __forceinline__ void work_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGWork) : "memory");
}

// Barrier of the transposing threads that also returns, in every one of them,
// whether any passed `v` true.
__device__ __forceinline__ bool work_bar_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kGWork)
      : "memory");
  return r != 0;
}

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row` in a 64-column
// swizzle atom (128-byte rows, 8-row swizzle period).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(kGThreads, 1)
jacap_gram_kernel(const __grid_constant__ GramParams G) {
  const JacapArgs& a = G.a;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sv = smem;                                   // kGStages x 32 KiB
  unsigned char* st = sv + kGStages * kJTileBytes;            // 2 x 32 KiB, transposed
  GramSmem* ms = reinterpret_cast<GramSmem*>(st + 2 * kJTileBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long limit = a.wait_limit_ns;
  volatile int* abort_flag = &ms->abort_flag;

  const int item = blockIdx.x;
  const int layer = item / a.splits_per_layer;
  const int rem = item - layer * a.splits_per_layer;
  const JSeq& sq = a.seqs[find_jseq(a, rem, [&](int i) { return a.seqs[i].split_base; })];
  const int local = rem - sq.split_base;
  const int h = local / sq.n_split, s = local - h * sq.n_split;
  const int P = sq.len - a.W;
  const int n_tiles = (P + kJTile - 1) / kJTile;
  const int per = (n_tiles + sq.n_split - 1) / sq.n_split;
  const int t_begin = s * per, t_end = min(n_tiles, t_begin + per);
  const int n_my = max(0, t_end - t_begin);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGStages; ++i) {
      mbar_init(smem_u32(&ms->full[i]), 1);
      mbar_init(smem_u32(&ms->empty[i]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ms->tfull[b]), 1);
      mbar_init(smem_u32(&ms->tempty[b]), 1);
    }
    mbar_init(smem_u32(&ms->done), 1);
    mbar_init(smem_u32(&ms->drain), 1);
    ms->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ms->tmem_base)),
                 "r"(kJD)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ms->tmem_base;
  uint32_t armed = 0, armed_par = 0;
  bool mma_issued = false;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      for (int i = 0; i < n_my; ++i) {
        if (!mbar_wait(smem_u32(&ms->empty[stage]), phase ^ 1, limit, abort_flag)) {
          *abort_flag = 1;
          record_status(a.status, KVSEL_ERR_TIMEOUT);
          break;
        }
        const uint32_t bar = smem_u32(&ms->full[stage]);
        mbar_expect_tx(bar, kJTileBytes);
        const int row = (int)((int64_t)layer * a.T + sq.tok_off + (t_begin + i) * kJTile);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(smem_u32(sv + stage * kJTileBytes + hf * kAtom), &G.tmv, bar, hf * 64, h,
                      row, pol);
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        if (++stage == kGStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdesc = instr_desc(kJD, kJD);
      const uint32_t st_addr = smem_u32(st);
      bool ok = true;
      for (int i = 0; ok && i < n_my; ++i) {
        const int b = i & 1;
        if (!mbar_wait(smem_u32(&ms->tfull[b]), (uint32_t)(i >> 1) & 1, limit, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kJTile / 16; ++kk) {
          const uint32_t addr = st_addr + b * kJTileBytes + (kk >> 2) * kAtom + (kk & 3) * 32;
          tc_mma(tmem_base, smem_desc(addr), smem_desc(addr), kIdesc, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_issued = true;
        tc_commit(smem_u32(&ms->tempty[b]));
      }
      if (ok) {
        tc_commit(smem_u32(&ms->done));
      } else {
        *abort_flag = 1;
        record_status(a.status, KVSEL_ERR_TIMEOUT);
      }
    }
  } else {
    // ---- transposers (warps 2..9): softmax normaliser, w, sqrt(w) V^T tiles
    const int tid = threadIdx.x - 64;
    if (warp == 2) {
      // merge the instance's statistics partials in a fixed order
      const float* pr = a.part + 2 * ((int64_t)layer * a.chunks_per_layer + sq.chunk_base +
                                      (int64_t)h * sq.n_chunks);
      float mx = -INFINITY;
      for (int c = lane; c < sq.n_chunks; c += 32) mx = fmaxf(mx, pr[2 * c]);
      for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      float sum = 0.f;
      for (int c = lane; c < sq.n_chunks; c += 32) sum = fmaf(pr[2 * c + 1], ex2(pr[2 * c] - mx), sum);
      for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (lane == 0) {
        ms->norm_m = mx;
        ms->norm_s = sum;
      }
    }
    work_bar();
    const float nm = ms->norm_m, inv_s = 1.f / ms->norm_s;
    const int64_t plane = ((int64_t)layer * a.H + h) * a.T + sq.tok_off;
    // sqrt(w) of a tile's tokens into sw[buf] (threads 0..127, one token each)
    auto weights_of = [&](int tile, int buf) {
      if (tid < kJTile) {
        const int t = tile * kJTile + tid;
        float w = 0.f;
        if (t < P) {
          const float2 zk = a.zk[plane + t];
          const float al = ex2(zk.x - nm) * inv_s;
          const float g = al * (1.f - al);
          w = g * g * zk.y * (1.f / kJD);
          a.wts[plane + t] = w;
        }
        ms->sw[buf][tid] = sqrtf(w);
      }
    };
    if (n_my > 0) weights_of(t_begin, 0);
    work_bar();
    // transposition by 8 x 8 blocks: warp wq takes dimension blocks 2wq, 2wq+1
    // and, per step, token blocks 2p, 2p+1 (four blocks: one ldmatrix.x4.trans
    // from the V tile, one stmatrix.x4 into the transposed buffer; each 8-row
    // phase of either touches eight distinct chunks of a swizzle period)
    const int wq = tid >> 5, lid = tid & 31;
    const int m_of = lid >> 3, r_of = lid & 7;          // the matrix and row this lane addresses
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int i = 0; i < n_my; ++i) {
      const int b = i & 1;
      if (i + 1 < n_my) weights_of(t_begin + i + 1, (i + 1) & 1);
      bool mine = mbar_wait(smem_u32(&ms->full[stage]), phase, limit, abort_flag);
      if (mine && i >= 2)
        mine = mbar_wait(smem_u32(&ms->tempty[b]), (uint32_t)((i - 2) >> 1) & 1, limit, abort_flag);
      if (mine) {
        const uint32_t vt = smem_u32(sv + stage * kJTileBytes);
        const uint32_t tt = smem_u32(st + b * kJTileBytes);
        const float* sw = ms->sw[i & 1];
#pragma unroll 2
        for (int pstep = 0; pstep < 8; ++pstep) {
          // this lane's address: matrix m_of = (token block 2p + m/2, dimension block 2wq + m%2)
          const int tbl = 2 * pstep + (m_of >> 1), dbl = 2 * wq + (m_of & 1);
          const uint32_t src = vt + (dbl >> 3) * kAtom + swz(tbl * 8 + r_of, dbl & 7);
          uint32_t rg[4];
          asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                       : "=r"(rg[0]), "=r"(rg[1]), "=r"(rg[2]), "=r"(rg[3])
                       : "r"(src)
                       : "memory");
          // register m holds, for dimension dbl*8 + lid/4, tokens (lid%4)*2 and +1 of
          // token block 2p + m/2: scale each by its sqrt(w)
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int t0 = (2 * pstep + (m >> 1)) * 8 + (lid & 3) * 2;
            const float f0 = sw[t0], f1 = sw[t0 + 1];
            const float x0 = __uint_as_float(rg[m] << 16), x1 = __uint_as_float(rg[m] & 0xFFFF0000u);
            const __nv_bfloat162 p2 = __floats2bfloat162_rn(f0 != 0.f ? f0 * x0 : 0.f,
                                                            f1 != 0.f ? f1 * x1 : 0.f);
            rg[m] = *reinterpret_cast<const uint32_t*>(&p2);
          }
          // stored matrix m_of: rows = dimensions dbl*8 .., 8 tokens of block tbl
          const uint32_t dst = tt + (tbl >> 3) * kAtom + swz(dbl * 8 + r_of, tbl & 7);
          asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(dst),
                       "r"(rg[0]), "r"(rg[1]), "r"(rg[2]), "r"(rg[3])
                       : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      // the tile written by all, or a wait given up somewhere (same answer everywhere)
      if (work_bar_any(!mine)) {
        ok = false;
        break;
      }
      if (tid == 0) {
        mbar_arrive(smem_u32(&ms->tfull[b]));
        mbar_arrive(smem_u32(&ms->empty[stage]));
      }
      if (++stage == kGStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (!ok) {
      *abort_flag = 1;
      record_status(a.status, KVSEL_ERR_TIMEOUT);
    } else if (n_my > 0 &&
               mbar_wait(smem_u32(&ms->done), 0, limit, abort_flag)) {
      // epilogue: TMEM lanes are dimensions d1, columns d2; warp w reads lane
      // quarter w % 4 and column half (w - 2) / 4
      tc_fence_after();
      const int quarter = warp & 3, half = (warp - 2) >> 2;
      const int d1 = quarter * 32 + lane;
      float* out = a.gram + ((int64_t)item * kJD + d1) * kJD + half * 64;
#pragma unroll
      for (int cblk = 0; cblk < 64; cblk += 32) {
        float v[32];
        tmem_load_cols<32>(tmem_base + ((uint32_t)(quarter * 32) << 16) + half * 64 + cblk, v);
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(out + cblk + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
    } else if (n_my > 0) {
      *abort_flag = 1;
      record_status(a.status, KVSEL_ERR_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (ms->abort_flag) {
    if (warp == 0 && lane == 0) {
      for (int i = 0; i < kGStages; ++i)
        if (armed & (1u << i))
          mbar_wait(smem_u32(&ms->full[i]), (armed_par >> i) & 1, limit, nullptr);
    }
    if (warp == 1 && lane == 0 && mma_issued) {
      tc_commit(smem_u32(&ms->drain));
      mbar_wait(smem_u32(&ms->drain), 0, limit, nullptr);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kJD)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// factor: A = I + sum of the partial Grams, Cholesky, L^{-1} as bf16 hi + lo
// ---------------------------------------------------------------------------

constexpr int kFLd = kJD + 1;                  // padded row of the fp32 matrices

__global__ void __launch_bounds__(256) jacap_factor_kernel(const __grid_constant__ JacapArgs a) {
  extern __shared__ float fs[];
  float* A = fs;                               // [kJD][kFLd]: A, then L in the lower triangle
  float* X = fs + kJD * kFLd;                  // L^{-1} (lower triangle)
  __shared__ int bad;
  const int tid = threadIdx.x;
  const int inst = blockIdx.x;
  const int layer = inst / a.inst_per_layer;
  const int rem = inst - layer * a.inst_per_layer;
  const JSeq& sq = a.seqs[find_jseq(a, rem, [&](int i) { return a.seqs[i].inst_base; })];
  const int h = rem - sq.inst_base;
  const int64_t g0 = (int64_t)layer * a.splits_per_layer + sq.split_base + (int64_t)h * sq.n_split;
  if (tid == 0) bad = 0;
  // A = I + the partial Grams (fixed order), lower triangle
  {
    const float* __restrict__ gp = a.gram + g0 * kJD * kJD;
    constexpr int kPer = kJD * kJD / 256;       // elements per thread (every 256th)
    float acc[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int e = tid + q * 256;
      acc[q] = (e >> 7) == (e & (kJD - 1)) ? 1.f : 0.f;
    }
    const int nsp = sq.n_split;
    for (int sp = 0; sp < nsp; ++sp) {         // every load of a partial in flight at once
#pragma unroll
      for (int q = 0; q < kPer; ++q) acc[q] += __ldg(gp + (int64_t)sp * kJD * kJD + tid + q * 256);
    }
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int e = tid + q * 256, i = e >> 7, j = e & (kJD - 1);
      if (j <= i) A[i * kFLd + j] = acc[q];
    }
  }
  __syncthreads();
  // two threads per row (or column) of each step, each taking every other k
  // of the dot product with four accumulators; the halves are added by a
  // shuffle
  const int pair = tid >> 1, half = tid & 1;
  auto dot = [&](const float* x, int xs, const float* y, int ys, int k0, int k1) {
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    int k = k0 + half;
    for (; k + 6 < k1; k += 8) {
      s0 = fmaf(x[k * xs], y[k * ys], s0);
      s1 = fmaf(x[(k + 2) * xs], y[(k + 2) * ys], s1);
      s2 = fmaf(x[(k + 4) * xs], y[(k + 4) * ys], s2);
      s3 = fmaf(x[(k + 6) * xs], y[(k + 6) * ys], s3);
    }
    for (; k < k1; k += 2) s0 = fmaf(x[k * xs], y[k * ys], s0);
    float acc = (s0 + s1) + (s2 + s3);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    return acc;
  };
  // Cholesky, left-looking, one column at a time: L[j][j] = sqrt(A[j][j] -
  // sum_k L[j][k]^2), then L[i][j] = (A[i][j] - sum_{k<j} L[i][k] L[j][k]) /
  // L[j][j] for the rows below
  for (int j = 0; j < kJD; ++j) {
    if (tid < 32) {                            // the diagonal: one warp, a strided dot product
      float acc = 0.f;
      for (int k = tid; k < j; k += 32) acc = fmaf(A[j * kFLd + k], A[j * kFLd + k], acc);
      for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (tid == 0) {
        const float p = A[j * kFLd + j] - acc;
        if (!(p > 0.f) || !finite_f(p)) bad = 1;
        A[j * kFLd + j] = sqrtf(fmaxf(p, 1e-30f));
      }
    }
    __syncthreads();
    const float inv = 1.f / A[j * kFLd + j];
    const int i = j + 1 + pair;                // rows j+1 .. 127 (pairs of threads)
    const float acc = dot(A + (i < kJD ? i : j) * kFLd, 1, A + j * kFLd, 1, 0, j);
    if (i < kJD && half == 0) A[i * kFLd + j] = (A[i * kFLd + j] - acc) * inv;
    __syncthreads();
  }
  // X = L^{-1}, one row at a time: X[i][i] = 1 / L[i][i] and, for c < i,
  // X[i][c] = -(sum_{k=c}^{i-1} L[i][k] X[k][c]) / L[i][i], a column per pair
  for (int i = 0; i < kJD; ++i) {
    const float inv = 1.f / A[i * kFLd + i];
    const int c = pair;                        // columns 0 .. 127
    const float acc = dot(A + i * kFLd, 1, X + c, kFLd, c, c <= i ? i : c);
    if (c <= i && half == 0) X[i * kFLd + c] = c == i ? inv : -acc * inv;
    __syncthreads();
  }
  __nv_bfloat16* hi = reinterpret_cast<__nv_bfloat16*>(a.linv) + (int64_t)inst * 2 * kJD * kJD;
  __nv_bfloat16* lo = hi + kJD * kJD;
  for (int e = tid; e < kJD * kJD; e += blockDim.x) {
    const int r = e >> 7, c = e & (kJD - 1);
    const float x = c <= r ? X[r * kFLd + c] : 0.f;
    const __nv_bfloat16 xh = __float2bfloat16_rn(x);
    hi[e] = xh;
    lo[e] = __float2bfloat16_rn(x - __bfloat162float(xh));
  }
  if (tid == 0 && bad) record_status(a.status, KVSEL_ERR_NONFINITE);
}

// ---------------------------------------------------------------------------
// leverage: r_t = w_t |L^{-1} v_t|^2
// ---------------------------------------------------------------------------

constexpr int kLStages = 4;
constexpr int kLThreads = 192;                 // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kLBufs = 4;                      // TMEM accumulators of 128 columns

struct LevSmem {
  unsigned long long full[kLStages], empty[kLStages];
  unsigned long long lfull;
  unsigned long long ready[kLBufs], tfree[kLBufs];
  unsigned long long drain;                    // abort path: the MMA issuer's last commit
  uint32_t tmem_base;
  int abort_flag;
};

struct LevParams {
  CUtensorMap tmv;                             // V as (D, H, layers * T)
  CUtensorMap tml;                             // L^{-1} as (D, D, 2 * instances)
  JacapArgs a;
};

__global__ void __launch_bounds__(kLThreads, 1)
jacap_leverage_kernel(const __grid_constant__ LevParams Lp) {
  const JacapArgs& a = Lp.a;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sl = smem;                                   // hi, lo: 2 x 32 KiB
  unsigned char* sv = sl + 2 * kJTileBytes;                   // kLStages x 32 KiB
  LevSmem* ms = reinterpret_cast<LevSmem*>(sv + kLStages * kJTileBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long limit = a.wait_limit_ns;
  volatile int* abort_flag = &ms->abort_flag;

  const int item = blockIdx.x;
  const int layer = item / a.lev_per_layer;
  const int rem = item - layer * a.lev_per_layer;
  const JSeq& sq = a.seqs[find_jseq(a, rem, [&](int i) { return a.seqs[i].lev_base; })];
  const int local = rem - sq.lev_base;
  const int h = local / sq.n_lev, g = local - h * sq.n_lev;
  const int P = sq.len - a.W;
  const int n_tiles = (P + kJTile - 1) / kJTile;
  const int t_begin = g * kJLevTiles, t_end = min(n_tiles, t_begin + kJLevTiles);
  const int n_my = max(0, t_end - t_begin);
  const int inst = layer * a.inst_per_layer + sq.inst_base + h;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kLStages; ++i) {
      mbar_init(smem_u32(&ms->full[i]), 1);
      mbar_init(smem_u32(&ms->empty[i]), 1);
    }
    mbar_init(smem_u32(&ms->lfull), 1);
    for (int b = 0; b < kLBufs; ++b) {
      mbar_init(smem_u32(&ms->ready[b]), 1);
      mbar_init(smem_u32(&ms->tfree[b]), 4);
    }
    mbar_init(smem_u32(&ms->drain), 1);
    ms->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ms->tmem_base)),
                 "r"(kLBufs * kJD)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ms->tmem_base;
  uint32_t armed = 0, armed_par = 0;
  bool l_armed = false, mma_issued = false;

  if (warp == 0) {
    if (lane == 0 && n_my > 0) {
      const uint64_t pol_v = policy_evict_first(), pol_l = policy_evict_last();
      const uint32_t lbar = smem_u32(&ms->lfull);
      mbar_expect_tx(lbar, 2 * kJTileBytes);
#pragma unroll
      for (int which = 0; which < 2; ++which)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(smem_u32(sl + which * kJTileBytes + hf * kAtom), &Lp.tml, lbar, hf * 64, 0,
                      inst * 2 + which, pol_l);
      l_armed = true;
      int stage = 0;
      uint32_t phase = 0;
      for (int i = 0; i < n_my; ++i) {
        if (!mbar_wait(smem_u32(&ms->empty[stage]), phase ^ 1, limit, abort_flag)) {
          *abort_flag = 1;
          record_status(a.status, KVSEL_ERR_TIMEOUT);
          break;
        }
        const uint32_t bar = smem_u32(&ms->full[stage]);
        mbar_expect_tx(bar, kJTileBytes);
        const int row = (int)((int64_t)layer * a.T + sq.tok_off + (t_begin + i) * kJTile);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(smem_u32(sv + stage * kJTileBytes + hf * kAtom), &Lp.tmv, bar, hf * 64, h,
                      row, pol_v);
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        if (++stage == kLStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && n_my > 0) {
      constexpr uint32_t kIdesc = instr_desc(kJD, kJTile);
      const uint32_t sv_addr = smem_u32(sv), sl_addr = smem_u32(sl);
      bool ok = mbar_wait(smem_u32(&ms->lfull), 0, limit, abort_flag);
      int stage = 0;
      uint32_t phase = 0;
      for (int i = 0; ok && i < n_my; ++i) {
        const int b = i % kLBufs;
        if (!mbar_wait(smem_u32(&ms->tfree[b]), ((uint32_t)(i / kLBufs) & 1) ^ 1, limit,
                       abort_flag) ||
            !mbar_wait(smem_u32(&ms->full[stage]), phase, limit, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(b * kJD);
#pragma unroll
        for (int which = 0; which < 2; ++which)
#pragma unroll
          for (int kk = 0; kk < kJD / 16; ++kk) {
            const uint32_t a_addr = sv_addr + stage * kJTileBytes + (kk >> 2) * kAtom + (kk & 3) * 32;
            const uint32_t b_addr = sl_addr + which * kJTileBytes + (kk >> 2) * kAtom + (kk & 3) * 32;
            tc_mma(d_tmem, smem_desc(a_addr), smem_desc(b_addr), kIdesc,
                   (which > 0 || kk > 0) ? 1u : 0u);
          }
        mma_issued = true;
        tc_commit(smem_u32(&ms->empty[stage]));
        tc_commit(smem_u32(&ms->ready[b]));
        if (++stage == kLStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(a.status, KVSEL_ERR_TIMEOUT);
      }
    }
  } else {
    // ---- epilogue (warps 2..5): lane quarter warp % 4, one token per lane
    const int quarter = warp & 3;
    const int64_t plane = ((int64_t)layer * a.H + h) * a.T + sq.tok_off;
    bool ok = true;
    for (int i = 0; ok && i < n_my; ++i) {
      const int b = i % kLBufs;
      const int t = (t_begin + i) * kJTile + quarter * 32 + lane;
      const float w = t < P ? a.wts[plane + t] : 0.f;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ms->ready[b]), (uint32_t)(i / kLBufs) & 1,
                                               limit, abort_flag));
      if (!ok) break;
      tc_fence_after();
      float ss = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < kJD; c0 += 32) {
        float y[32];
        tmem_load_cols<32>(tmem_base + ((uint32_t)(quarter * 32) << 16) + b * kJD + c0, y);
#pragma unroll
        for (int e = 0; e < 32; ++e) ss = fmaf(y[e], y[e], ss);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ms->tfree[b]));
      if (t < P) a.scores[plane + t] = w * ss;
    }
    if (!ok) {
      *abort_flag = 1;
      record_status(a.status, KVSEL_ERR_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (ms->abort_flag) {
    if (warp == 0 && lane == 0) {
      if (l_armed) mbar_wait(smem_u32(&ms->lfull), 0, limit, nullptr);
      for (int i = 0; i < kLStages; ++i)
        if (armed & (1u << i))
          mbar_wait(smem_u32(&ms->full[i]), (armed_par >> i) & 1, limit, nullptr);
    }
    if (warp == 1 && lane == 0 && mma_issued) {
      tc_commit(smem_u32(&ms->drain));
      mbar_wait(smem_u32(&ms->drain), 0, limit, nullptr);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kLBufs * kJD)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// Host
// ---------------------------------------------------------------------------

bool make_rows_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint32_t box1, uint32_t box2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {64, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t gram_smem() {
  return 1024 + (kGStages + 2) * (size_t)kJTileBytes + sizeof(GramSmem);
}

constexpr size_t lev_smem() {
  return 1024 + (2 + kLStages) * (size_t)kJTileBytes + sizeof(LevSmem);
}

}  // namespace

bool jacap_eligible(int dtype, int D, const void* q, const void* k, const void* v) {
  if (dtype != KVSEL_BF16 || D != kJD) return false;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v)) & 15)
    return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_jacap(const JacapArgs& a) {
  const int64_t rows = (int64_t)a.layers * a.T;
  if (rows >= 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaError_t e;
  if (a.layers * a.chunks_per_layer > 0)
    jacap_stats_kernel<<<(unsigned)(a.layers * a.chunks_per_layer), 256, 0, a.stream>>>(a);
  if ((e = cudaGetLastError())) return e;
  {
    GramParams gp;
    std::memset(&gp, 0, sizeof(gp));
    if (!make_rows_map(&gp.tmv, a.v, kJD, a.H, rows, 1, kJTile)) return cudaErrorInvalidValue;
    gp.a = a;
    const size_t smem = gram_smem();
    if ((e = cudaFuncSetAttribute(jacap_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)))
      return e;
    if (a.layers * a.splits_per_layer > 0)
      jacap_gram_kernel<<<(unsigned)(a.layers * a.splits_per_layer), kGThreads, smem, a.stream>>>(gp);
    if ((e = cudaGetLastError())) return e;
  }
  {
    const size_t smem = 2 * (size_t)kJD * kFLd * sizeof(float);
    if ((e = cudaFuncSetAttribute(jacap_factor_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
      return e;
    if (a.layers * a.inst_per_layer > 0)
      jacap_factor_kernel<<<(unsigned)(a.layers * a.inst_per_layer), 256, smem, a.stream>>>(a);
    if ((e = cudaGetLastError())) return e;
  }
  {
    LevParams lp;
    std::memset(&lp, 0, sizeof(lp));
    const int64_t insts = (int64_t)a.layers * a.inst_per_layer;
    if (!make_rows_map(&lp.tmv, a.v, kJD, a.H, rows, 1, kJTile) ||
        !make_rows_map(&lp.tml, a.linv, kJD, kJD, 2 * insts, kJD, 1))
      return cudaErrorInvalidValue;
    lp.a = a;
    const size_t smem = lev_smem();
    if ((e = cudaFuncSetAttribute(jacap_leverage_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
      return e;
    if (a.layers * a.lev_per_layer > 0)
      jacap_leverage_kernel<<<(unsigned)(a.layers * a.lev_per_layer), kLThreads, smem, a.stream>>>(lp);
    if ((e = cudaGetLastError())) return e;
  }
  return cudaSuccess;
}

}  // namespace kvsel
