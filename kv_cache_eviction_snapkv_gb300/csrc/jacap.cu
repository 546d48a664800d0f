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
//            (eight lanes per row, four rows per lane group in flight), and
//            the chunk's max and sum of 2^z. HBM-bound on K.
//   gram     persistent, at most one CTA per SM: the instances' 128-token tiles
//            in instance order, cut into equal ranges, one per CTA; a range
//            splits into pieces at instance boundaries. Per piece: merge the
//            instance's softmax partials; per tile: w, then the V tile as TMA
//            wrote it (128-byte swizzle, tokens as rows) scaled in place by
//            sqrt(w) per token, on which tcgen05.mma with A = B = that tile read
//            MN-major (dimensions as M and N, tokens as K) accumulates
//            sum_t w_t v_t v_t^T (128 x 128, fp32, in TMEM, two accumulators
//            taking pieces in turn); each piece's partial is written out.
//            HBM-bound on V.
//   factor   one CTA per instance: A = I + its pieces' partials in order, the
//            Cholesky factor and L^{-1} in fp32 (8 x 8 register blocks, one
//            column or row per step through shared memory), written as two
//            bf16 matrices hi + lo (hi = bf16(L^{-1}), lo = bf16(L^{-1} - hi)).
//   leverage persistent over the same pieces: L^{-1} (hi, lo) per piece, then
//            y_t = L^{-1} v_t for 128 tokens at a time by tcgen05.mma (A = the
//            V tile as loaded, B = hi, then lo, accumulated), r_t = w_t |y_t|^2
//            in the epilogue. HBM-bound on V.
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

constexpr int kWork = 512;                     // compute threads of the stats and Gram kernels
static_assert(kWork % 128 == 0 && kWork <= 1024 - 64, "whole lane quarters, one CTA");
static_assert(kJTile % (kWork / 8) == 0 && (kJTileBytes / 16) % kWork == 0, "whole steps per tile");

// The instance of a Gram piece: layer, sequence, head.
struct JInst {
  int layer, h;
  const JSeq* sq;
};

__device__ __forceinline__ JInst jinst(const JacapArgs& a, int inst) {
  JInst r;
  r.layer = inst / a.inst_per_layer;
  const int rem = inst - r.layer * a.inst_per_layer;
  r.sq = &a.seqs[upper_find(a.n_scored, rem, [&](int i) { return a.seqs[i].inst_base; })];
  r.h = rem - r.sq->inst_base;
  return r;
}

__device__ __forceinline__ void work_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kWork) : "memory");
}

// Barrier of the scaling threads that also returns, in every one of them,
// whether any passed `v` true.
__device__ __forceinline__ bool work_bar_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kWork)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------------------
// stats
// ---------------------------------------------------------------------------

constexpr int kSStages = 6;                    // K tile ring
constexpr int kSThreads = 32 + kWork;          // warp 0 TMA, warps 1.. compute

struct StatsSmem {
  unsigned long long full[kSStages], empty[kSStages];
  int abort_flag;
  float mu[kJD], lam[kJD];                     // mu scaled to base-2 logits; diag Lambda
  float wm[kWork / 32], wl[kWork / 32];
  __align__(16) __nv_bfloat16 qs[32][kJD];     // 32 window queries at a time
};

struct StatsParams {
  CUtensorMap tmk;                             // K as (D, H, layers * T)
  JacapArgs a;
};

// Persistent over the pieces (the Gram kernel's CTA ranges): per piece the
// window statistics of its instance (the W x d recursion, queries staged 32
// rows at a time), then per K tile (TMA, 128-byte swizzle) z (base-2 units)
// and kappa per token, eight lanes per token (lane s takes 16-byte chunk s of
// both 64-dimension halves: a quarter-warp reads one 128-byte row, no bank
// conflicts), and the piece's max and sum of 2^z. HBM-bound on K.
__global__ void __launch_bounds__(kSThreads, 1)
jacap_stats_kernel(const __grid_constant__ StatsParams S) {
  const JacapArgs& a = S.a;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sk = smem;                                   // kSStages x 32 KiB
  StatsSmem* ms = reinterpret_cast<StatsSmem*>(sk + kSStages * kJTileBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long limit = a.wait_limit_ns;
  volatile int* abort_flag = &ms->abort_flag;
  const int s_begin = a.cta_seg[blockIdx.x], s_end = a.cta_seg[blockIdx.x + 1];

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSStages; ++i) {
      mbar_init(smem_u32(&ms->full[i]), 1);
      mbar_init(smem_u32(&ms->empty[i]), kWork / 32);
    }
    ms->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  uint32_t armed = 0, armed_par = 0;

  if (warp == 0) {
    // ---- TMA producer: the K tiles of every piece, in order
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int sg = s_begin; ok && sg < s_end; ++sg) {
        const JSeg pc = a.segs[sg];
        const JInst in = jinst(a, pc.inst);
        const int64_t row0 = (int64_t)in.layer * a.T + in.sq->tok_off;
        for (int t = pc.t_begin; t < pc.t_end; ++t) {
          if (!mbar_wait(smem_u32(&ms->empty[stage]), phase ^ 1, limit, abort_flag)) {
            *abort_flag = 1;
            record_status(a.status, KVSEL_ERR_TIMEOUT);
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&ms->full[stage]);
          mbar_expect_tx(bar, kJTileBytes);
          const int row = (int)(row0 + (int64_t)t * kJTile);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            tma_load_3d(smem_u32(sk + stage * kJTileBytes + hf * kAtom), &S.tmk, bar, hf * 64, in.h,
                        row, pol);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kSStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else {
    // ---- compute warps (1 ..)
    const int tid = threadIdx.x - 32, cw = tid >> 5;
    const int grp = lane >> 3, sub = lane & 7;
    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(a.q);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int sg = s_begin; sg < s_end; ++sg) {
      const JSeg pc = a.segs[sg];
      const JInst in = jinst(a, pc.inst);
      const int P = in.sq->len - a.W;
      const int64_t plane = ((int64_t)in.layer * a.H + in.h) * a.T + in.sq->tok_off;
      {
        // the window statistics: mu <- beta mu + (1 - beta) q and m <- beta m +
        // (1 - beta) q^2 over the W window queries from the first, one thread
        // per dimension
        const int64_t qrow0 = (int64_t)in.layer * a.S * a.W + (int64_t)in.sq->index * a.W;
        float mu = 0.f, m2 = 0.f;
        for (int r0 = 0; r0 < a.W; r0 += 32) {
          const int nr = min(32, a.W - r0);
          for (int e = tid; e < nr * (kJD / 8); e += kWork) {
            const int r = e / (kJD / 8), c = e - r * (kJD / 8);
            *reinterpret_cast<uint4*>(&ms->qs[r][c * 8]) = *reinterpret_cast<const uint4*>(
                qb + ((qrow0 + r0 + r) * a.H + in.h) * kJD + c * 8);
          }
          work_bar();
          if (tid < kJD) {
            for (int r = 0; r < nr; ++r) {
              const float q = __bfloat162float(ms->qs[r][tid]);
              if (r0 + r == 0) {
                mu = q;
                m2 = q * q;
              } else {
                mu = a.beta * mu + (1.f - a.beta) * q;
                m2 = a.beta * m2 + (1.f - a.beta) * (q * q);
              }
            }
          }
          work_bar();
        }
        if (tid < kJD) {
          ms->mu[tid] = mu * (1.4426950408889634f / (a.tau * sqrtf((float)kJD)));
          ms->lam[tid] = fmaxf(m2 - mu * mu, a.eps);
        }
        work_bar();
      }
      // lane sub: dimensions 8 sub .. 8 sub + 7 and 64 + 8 sub .. 64 + 8 sub + 7
      float mu[16], lam[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int d = (e >> 3) * 64 + sub * 8 + (e & 7);
        mu[e] = ms->mu[d];
        lam[e] = ms->lam[d];
      }
      float m = -INFINITY, l = 0.f;
      for (int t = pc.t_begin; t < pc.t_end; ++t) {
        if (ok) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ms->full[stage]), phase, limit, abort_flag));
          if (ok) {
            const unsigned char* kt = sk + stage * kJTileBytes;
#pragma unroll
            for (int step = 0; step < kJTile / (kWork / 8); ++step) {
              const int row = step * (kWork / 8) + cw * 4 + grp;
              const uint32_t off = (uint32_t)(row * 128 + ((sub ^ (row & 7)) << 4));
              const uint4 k0 = *reinterpret_cast<const uint4*>(kt + off);
              const uint4 k1 = *reinterpret_cast<const uint4*>(kt + kAtom + off);
              const uint32_t w[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
              float z = 0.f, kap = 0.f;
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float kv = __uint_as_float((e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16));
                z = fmaf(mu[e], kv, z);
                kap = fmaf(lam[e] * kv, kv, kap);
              }
#pragma unroll
              for (int off2 = 1; off2 < 8; off2 <<= 1) {
                z += __shfl_xor_sync(0xffffffffu, z, off2);
                kap += __shfl_xor_sync(0xffffffffu, kap, off2);
              }
              const int tok = t * kJTile + row;
              if (tok < P) {
                if (sub == 0) a.zk[plane + tok] = make_float2(z, kap);
                const float mx = fmaxf(m, z);
                l = (m == -INFINITY ? 0.f : l * ex2(m - mx)) + ex2(z - mx);
                m = mx;
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ms->empty[stage]));
          }
        }
        if (++stage == kSStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      // the piece's max and sum: lane groups, then warps; a wait given up
      // anywhere ends every compute warp here
      if (work_bar_any(!ok)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int off2 = 8; off2 <= 16; off2 <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, off2);
        const float lo = __shfl_xor_sync(0xffffffffu, l, off2);
        const float mx = fmaxf(m, mo);
        l = (m == -INFINITY ? 0.f : l * ex2(m - mx)) + (mo == -INFINITY ? 0.f : lo * ex2(mo - mx));
        m = mx;
      }
      if (lane == 0) {
        ms->wm[cw] = m;
        ms->wl[cw] = l;
      }
      work_bar();
      if (tid == 0) {
        float mx = -INFINITY, sum = 0.f;
        for (int w = 0; w < kWork / 32; ++w) mx = fmaxf(mx, ms->wm[w]);
        for (int w = 0; w < kWork / 32; ++w)
          if (ms->wm[w] != -INFINITY) sum = fmaf(ms->wl[w], ex2(ms->wm[w] - mx), sum);
        a.part[2 * (int64_t)sg] = mx;
        a.part[2 * (int64_t)sg + 1] = sum;
        if (!finite_f(mx) || !finite_f(sum)) record_status(a.status, KVSEL_ERR_NONFINITE);
      }
      // wm, wl, mu, lam and qs are rewritten by the next piece only after this
      work_bar();
    }
    if (!ok) {
      *abort_flag = 1;
      record_status(a.status, KVSEL_ERR_TIMEOUT);
    }
  }

  __syncthreads();
  if (ms->abort_flag && warp == 0 && lane == 0) {
    for (int i = 0; i < kSStages; ++i)
      if (armed & (1u << i))
        mbar_wait(smem_u32(&ms->full[i]), (armed_par >> i) & 1, limit, nullptr);
  }
}

// ---------------------------------------------------------------------------
// gram
// ---------------------------------------------------------------------------

constexpr int kGStages = 6;                    // V tile ring
constexpr int kGThreads = 64 + kWork;          // warp 0 TMA, warp 1 MMA, warps 2.. scale

struct GramSmem {
  unsigned long long full[kGStages], empty[kGStages];   // V ring: loaded, free
  unsigned long long scaled[kGStages];                  // V ring: scaled by sqrt(w)
  unsigned long long done[2], tfree[2];                 // TMEM accumulators (one per piece)
  unsigned long long drain;                    // abort path: the MMA issuer's last commit
  uint32_t tmem_base;
  int abort_flag;
  float norm_m, norm_s;                        // the piece's instance: base-2 softmax max and sum
  float sw[2][kJTile];                         // sqrt(w) of a tile's tokens (double buffer)
};

struct GramParams {
  CUtensorMap tmv;                             // V as (D, H, layers * T)
  JacapArgs a;
};


__global__ void __launch_bounds__(kGThreads, 1)
jacap_gram_kernel(const __grid_constant__ GramParams G) {
  const JacapArgs& a = G.a;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sv = smem;                                   // kGStages x 32 KiB
  GramSmem* ms = reinterpret_cast<GramSmem*>(sv + kGStages * kJTileBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long limit = a.wait_limit_ns;
  volatile int* abort_flag = &ms->abort_flag;
  const int s_begin = a.cta_seg[blockIdx.x], s_end = a.cta_seg[blockIdx.x + 1];

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGStages; ++i) {
      mbar_init(smem_u32(&ms->full[i]), 1);
      mbar_init(smem_u32(&ms->empty[i]), 1);
      mbar_init(smem_u32(&ms->scaled[i]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ms->done[b]), 1);
      mbar_init(smem_u32(&ms->tfree[b]), 1);
    }
    mbar_init(smem_u32(&ms->drain), 1);
    ms->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ms->tmem_base)),
                 "r"(2 * kJD)
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
    // ---- TMA producer: the V tiles of every piece, in order
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int sg = s_begin; ok && sg < s_end; ++sg) {
        const JSeg pc = a.segs[sg];
        const JInst in = jinst(a, pc.inst);
        const int64_t row0 = (int64_t)in.layer * a.T + in.sq->tok_off;
        for (int t = pc.t_begin; t < pc.t_end; ++t) {
          if (!mbar_wait(smem_u32(&ms->empty[stage]), phase ^ 1, limit, abort_flag)) {
            *abort_flag = 1;
            record_status(a.status, KVSEL_ERR_TIMEOUT);
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&ms->full[stage]);
          mbar_expect_tx(bar, kJTileBytes);
          const int row = (int)(row0 + (int64_t)t * kJTile);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            tma_load_3d(smem_u32(sv + stage * kJTileBytes + hf * kAtom), &G.tmv, bar, hf * 64, in.h,
                        row, pol);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kGStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: piece k accumulates into TMEM columns (k % 2) * 128 ..
    if (lane == 0) {
      constexpr uint32_t kIdesc = instr_desc(kJD, kJD) | (1u << 15) | (1u << 16);  // A, B MN-major
      const uint32_t sv_addr = smem_u32(sv);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int k = 0; ok && k < s_end - s_begin; ++k) {
        const JSeg pc = a.segs[s_begin + k];
        const int ab = k & 1;
        if (!mbar_wait(smem_u32(&ms->tfree[ab]), ((uint32_t)(k >> 1) & 1) ^ 1, limit, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(ab * kJD);
        for (int t = pc.t_begin; t < pc.t_end; ++t) {
          if (!mbar_wait(smem_u32(&ms->scaled[stage]), phase, limit, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kJTile / 16; ++kk) {          // 16 tokens (2 KiB of rows) each
            const uint32_t addr = sv_addr + stage * kJTileBytes + kk * 2048;
            tc_mma(d_tmem, smem_desc_mn(addr), smem_desc_mn(addr), kIdesc,
                   (t > pc.t_begin || kk > 0) ? 1u : 0u);
          }
          mma_issued = true;
          tc_commit(smem_u32(&ms->empty[stage]));
          if (++stage == kGStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) tc_commit(smem_u32(&ms->done[ab]));
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(a.status, KVSEL_ERR_TIMEOUT);
      }
    }
  } else {
    // ---- scaling warps (2 ..): per piece the instance's softmax normaliser,
    // then per tile w and the tile scaled by sqrt(w); at the end of the piece
    // its partial Gram out of TMEM
    const int tid = threadIdx.x - 64;
    const int wq = tid >> 5, lid = tid & 31;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int i = 0;                                          // tiles so far
    for (int k = 0; ok && k < s_end - s_begin; ++k) {
      const int sg = s_begin + k;
      const JSeg pc = a.segs[sg];
      const JInst in = jinst(a, pc.inst);
      const JSeq& sq = *in.sq;
      const int P = sq.len - a.W;
      const int64_t plane = ((int64_t)in.layer * a.H + in.h) * a.T + sq.tok_off;
      if (wq == 0) {
        // merge the instance's statistics partials (one per piece) in order
        const int p0 = a.inst_seg[pc.inst], np = a.inst_seg[pc.inst + 1] - p0;
        const float* pr = a.part + 2 * (int64_t)p0;
        float mx = -INFINITY;
        for (int c = lid; c < np; c += 32) mx = fmaxf(mx, pr[2 * c]);
        for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float sum = 0.f;
        for (int c = lid; c < np; c += 32) sum = fmaf(pr[2 * c + 1], ex2(pr[2 * c] - mx), sum);
        for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lid == 0) {
          ms->norm_m = mx;
          ms->norm_s = sum;
        }
      }
      work_bar();
      const float nm = ms->norm_m, inv_s = 1.f / ms->norm_s;
      // (z, kappa) of token tid of a tile (threads 0..127), loaded two tiles
      // ahead of its use; then w and sqrt(w) into sw[buf]
      auto fetch = [&](int tile) {
        const int t = tile * kJTile + tid;
        return (tid < kJTile && tile < pc.t_end && t < P) ? a.zk[plane + t] : make_float2(0.f, -1.f);
      };
      auto weigh = [&](int tile, int buf, float2 zk) {
        if (tid < kJTile) {
          float w = 0.f;
          if (zk.y >= 0.f) {                  // a prefix token (kappa >= 0)
            const float al = ex2(zk.x - nm) * inv_s;
            const float g = al * (1.f - al);
            w = g * g * zk.y * (1.f / kJD);
            a.wts[plane + tile * kJTile + tid] = w;
          }
          ms->sw[buf][tid] = sqrtf(w);
        }
      };
      // zo, ze: (z, kappa) of the piece's odd and even tiles (tile - t_begin),
      // each loaded two tiles before its use; the parity branch keeps both in
      // place (no register copy waits on a load in flight)
      float2 zo = fetch(pc.t_begin + 1), ze = fetch(pc.t_begin + 2);
      weigh(pc.t_begin, i & 1, fetch(pc.t_begin));
      work_bar();
      // scaling in place: thread tid takes the 16-byte chunks tid + 256 j of
      // the tile (row (chunk / 8) % 128 of atom chunk / 1024; the swizzle only
      // permutes chunks within a row)
      for (int t = pc.t_begin; t < pc.t_end; ++t, ++i) {
        if (((t - pc.t_begin) & 1) == 0) {
          if (t + 1 < pc.t_end) weigh(t + 1, (i + 1) & 1, zo);
          zo = fetch(t + 3);
        } else {
          if (t + 1 < pc.t_end) weigh(t + 1, (i + 1) & 1, ze);
          ze = fetch(t + 3);
        }
        const bool mine = mbar_wait(smem_u32(&ms->full[stage]), phase, limit, abort_flag);
        if (mine) {
          unsigned char* vt = sv + stage * kJTileBytes;
          const float* sw = ms->sw[i & 1];
#pragma unroll
          for (int j = 0; j < kJTileBytes / 16 / kWork; ++j) {
            const int e = tid + kWork * j;
            const float f = sw[(e >> 3) & (kJTile - 1)];
            uint4* p = reinterpret_cast<uint4*>(vt + e * 16);
            uint4 x = *p;
            uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float x0 = __uint_as_float(w[q] << 16), x1 = __uint_as_float(w[q] & 0xFFFF0000u);
              const __nv_bfloat162 p2 = __floats2bfloat162_rn(f * x0, f * x1);
              w[q] = f != 0.f ? *reinterpret_cast<const uint32_t*>(&p2) : 0u;
            }
            *p = x;
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        // the tile scaled by all, or a wait given up somewhere (same answer everywhere)
        if (work_bar_any(!mine)) {
          ok = false;
          break;
        }
        if (tid == 0) mbar_arrive(smem_u32(&ms->scaled[stage]));
        if (++stage == kGStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      // the piece's partial: TMEM lanes are dimensions d1, columns d2; warp
      // w reads lane quarter w % 4 and the 128 / (kWork / 128) columns of
      // group (w - 2) / 4
      const int ab = k & 1;
      const bool mine = mbar_wait(smem_u32(&ms->done[ab]), (uint32_t)(k >> 1) & 1, limit, abort_flag);
      if (work_bar_any(!mine)) {
        ok = false;
        break;
      }
      tc_fence_after();
      constexpr int kCols = kJD / (kWork / 128);
      const int quarter = warp & 3, cg = (warp - 2) >> 2;
      const int d1 = quarter * 32 + lane;
      float* out = a.gram + ((int64_t)sg * kJD + d1) * kJD + cg * kCols;
#pragma unroll
      for (int cblk = 0; cblk < kCols; cblk += 32) {
        float v[32];
        tmem_load_cols<32>(tmem_base + ((uint32_t)(quarter * 32) << 16) + ab * kJD + cg * kCols + cblk,
                           v);
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(out + cblk + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
      tc_fence_before();
      work_bar();
      if (tid == 0) mbar_arrive(smem_u32(&ms->tfree[ab]));
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
                 "r"(2 * kJD)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// factor: A = I + sum of the partial Grams, Cholesky, L^{-1} as bf16 hi + lo
// ---------------------------------------------------------------------------

constexpr int kFB = kJD / 8;                   // 8 x 8 blocks per side

// One CTA per instance, 160 threads: thread tid < 136 holds the lower block
// (bi, bk), bk <= bi, numbered row by row (tid = bi (bi + 1) / 2 + bk), in
// registers; three CTAs fit an SM (registers and shared memory). Both
// phases take two columns (rows) per step, one barrier per step. Both phases are right-looking, one column (row) per step and
// one barrier per step:
//   Cholesky  step (j, j+1), j even: the owners of the two columns (bk = j / 8)
//             store their current values to shared memory; every thread takes
//             the 2 x 2 pivot block (L00 = sqrt(a_jj), L10 = a_j+1,j / L00,
//             L11 = sqrt(a_j+1,j+1 - L10^2)), the columns of L for its rows
//             and columns (l_i0 = a_ij / L00, l_i1 = (a_i,j+1 - l_i0 L10) / L11)
//             and updates its entries right of j + 1 by -(l_i0 l_k0 + l_i1 l_k1).
//             The stored columns (before scaling) and (1 / L00, L10, 1 / L11)
//             are kept for the inverse.
//   inverse   L X = I by rows: B = I; step (j, j+1): X_j = B_j / L00 and
//             X_j+1 = (B_j+1 - L10 X_j) / L11 (the owners of the two rows,
//             bi = j / 8, store them to a double-buffered pair of rows), then
//             every row i > j + 1 takes B_i -= L_ij X_j + L_i,j+1 X_j+1.
// Entries above the diagonal of a diagonal block collect values that are
// never read; the output writes zeros there.
constexpr int kFThreads = 160;
constexpr int kFBlocks = kFB * (kFB + 1) / 2;   // 136 lower blocks

__global__ void __launch_bounds__(kFThreads, 3) jacap_factor_kernel(const __grid_constant__ JacapArgs a) {
  extern __shared__ float4 fs4[];
  float* Lc = reinterpret_cast<float*>(fs4);    // [kJD][kJD]: column j of the updated matrix at its step
  __shared__ float3 piv[kJD / 2];               // (1 / L00, L10, 1 / L11) of each column pair
  __shared__ __align__(16) float xrow[2][2][kJD];  // X rows j, j+1 of the current inverse step
  __shared__ int bad;
  const int tid = threadIdx.x;
  const bool act = tid < kFBlocks;
  int bi = 0;
  while (bi < kFB - 1 && (bi + 1) * (bi + 2) / 2 <= tid) ++bi;
  int bk = tid - bi * (bi + 1) / 2;
  if (!act) bi = -1, bk = kFB;                  // idle: matches no owner or update test
  const int inst = blockIdx.x;
  const int s_lo = a.inst_seg[inst], n_part = a.inst_seg[inst + 1] - s_lo;
  if (tid == 0) bad = 0;

  float R[8][8];
  auto set_identity = [&]() {
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int c = 0; c < 8; ++c) R[r][c] = (bi == bk && r == c) ? 1.f : 0.f;
  };
  // A = I + the partial Grams, in a fixed order
  set_identity();
  if (act) {
    const float* __restrict__ gp = a.gram + (int64_t)s_lo * kJD * kJD + (bi * 8) * kJD + bk * 8;
    for (int sp = 0; sp < n_part; ++sp) {
      const float4* src = reinterpret_cast<const float4*>(gp + (int64_t)sp * kJD * kJD);
      float4 x[16];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        x[2 * r] = __ldg(src + r * (kJD / 4));
        x[2 * r + 1] = __ldg(src + r * (kJD / 4) + 1);
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        R[r][0] += x[2 * r].x, R[r][1] += x[2 * r].y, R[r][2] += x[2 * r].z, R[r][3] += x[2 * r].w;
        R[r][4] += x[2 * r + 1].x, R[r][5] += x[2 * r + 1].y, R[r][6] += x[2 * r + 1].z;
        R[r][7] += x[2 * r + 1].w;
      }
    }
  }
  auto load8 = [](const float* p, float* v, float s) {
    const float4 u0 = reinterpret_cast<const float4*>(p)[0], u1 = reinterpret_cast<const float4*>(p)[1];
    v[0] = u0.x * s, v[1] = u0.y * s, v[2] = u0.z * s, v[3] = u0.w * s;
    v[4] = u1.x * s, v[5] = u1.y * s, v[6] = u1.z * s, v[7] = u1.w * s;
  };

  // the pivot block of a column pair and the two columns of L at 8 rows
  auto pivot = [&](int j, float& inv0, float& l10, float& inv1) {
    const float pa = Lc[j * kJD + j], pb = Lc[j * kJD + j + 1], pc = Lc[(j + 1) * kJD + j + 1];
    const float l00 = sqrtf(fmaxf(pa, 1e-30f));
    inv0 = 1.f / l00;
    l10 = pb * inv0;
    const float pd = pc - l10 * l10;
    inv1 = 1.f / sqrtf(fmaxf(pd, 1e-30f));
    return (pa > 0.f) && finite_f(pa) && (pd > 0.f) && finite_f(pd);
  };
  auto lcols = [&](int j, int row0, float inv0, float l10, float inv1, float* v0, float* v1) {
    load8(Lc + j * kJD + row0, v0, inv0);
    float w[8];
    load8(Lc + (j + 1) * kJD + row0, w, 1.f);
#pragma unroll
    for (int e = 0; e < 8; ++e) v1[e] = (w[e] - v0[e] * l10) * inv1;
  };

  // ---- Cholesky, two columns per step
  for (int jb = 0; jb < kFB; ++jb) {
#pragma unroll
    for (int jp = 0; jp < 4; ++jp) {
      const int jj = 2 * jp, j = jb * 8 + jj;
      if (bk == jb && bi >= jb) {
        float4* d0 = reinterpret_cast<float4*>(Lc + j * kJD + bi * 8);
        float4* d1 = reinterpret_cast<float4*>(Lc + (j + 1) * kJD + bi * 8);
        d0[0] = make_float4(R[0][jj], R[1][jj], R[2][jj], R[3][jj]);
        d0[1] = make_float4(R[4][jj], R[5][jj], R[6][jj], R[7][jj]);
        d1[0] = make_float4(R[0][jj + 1], R[1][jj + 1], R[2][jj + 1], R[3][jj + 1]);
        d1[1] = make_float4(R[4][jj + 1], R[5][jj + 1], R[6][jj + 1], R[7][jj + 1]);
      }
      __syncthreads();
      float inv0, l10, inv1;
      const bool good = pivot(j, inv0, l10, inv1);
      if (tid == 0) {
        piv[j >> 1] = make_float3(inv0, l10, inv1);
        if (!good) bad = 1;
      }
      if (act && bk >= jb) {
        float r0[8], r1[8], c0[8], c1[8];
        lcols(j, bi * 8, inv0, l10, inv1, r0, r1);
        lcols(j, bk * 8, inv0, l10, inv1, c0, c1);
        if (bk == jb) {
#pragma unroll
          for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = jj + 2; c < 8; ++c)
              R[r][c] = fmaf(-r1[r], c1[c], fmaf(-r0[r], c0[c], R[r][c]));
        } else {
#pragma unroll
          for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              R[r][c] = fmaf(-r1[r], c1[c], fmaf(-r0[r], c0[c], R[r][c]));
        }
      }
    }
  }

  // ---- X = L^{-1}, two rows per step
  set_identity();
  for (int jb = 0; jb < kFB; ++jb) {
#pragma unroll
    for (int jp = 0; jp < 4; ++jp) {
      const int jj = 2 * jp, j = jb * 8 + jj;
      float (*xr)[kJD] = xrow[jp & 1];
      const float3 pv = piv[j >> 1];
      if (bi == jb && bk <= jb) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          R[jj][c] *= pv.x;
          R[jj + 1][c] = (R[jj + 1][c] - pv.y * R[jj][c]) * pv.z;
        }
        float4* d0 = reinterpret_cast<float4*>(xr[0] + bk * 8);
        float4* d1 = reinterpret_cast<float4*>(xr[1] + bk * 8);
        d0[0] = make_float4(R[jj][0], R[jj][1], R[jj][2], R[jj][3]);
        d0[1] = make_float4(R[jj][4], R[jj][5], R[jj][6], R[jj][7]);
        d1[0] = make_float4(R[jj + 1][0], R[jj + 1][1], R[jj + 1][2], R[jj + 1][3]);
        d1[1] = make_float4(R[jj + 1][4], R[jj + 1][5], R[jj + 1][6], R[jj + 1][7]);
      }
      __syncthreads();
      if (bi >= jb && bk <= jb) {
        float l0[8], l1[8], x0[8], x1[8];
        lcols(j, bi * 8, pv.x, pv.y, pv.z, l0, l1);
        load8(xr[0] + bk * 8, x0, 1.f);
        load8(xr[1] + bk * 8, x1, 1.f);
        if (bi == jb) {
#pragma unroll
          for (int r = jj + 2; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              R[r][c] = fmaf(-l1[r], x1[c], fmaf(-l0[r], x0[c], R[r][c]));
        } else {
#pragma unroll
          for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              R[r][c] = fmaf(-l1[r], x1[c], fmaf(-l0[r], x0[c], R[r][c]));
        }
      }
    }
  }

  // ---- output: rows bi*8 .. of L^{-1}, columns bk*8 .., as bf16 hi and lo;
  // the blocks above the diagonal are zero
  __nv_bfloat16* hi = reinterpret_cast<__nv_bfloat16*>(a.linv) + (int64_t)inst * 2 * kJD * kJD;
  __nv_bfloat16* lo = hi + kJD * kJD;
  for (int e = tid; e < kFB * kFB * 8; e += kFThreads) {
    const int blk = e >> 3, r = e & 7, ui = blk / kFB, uk = blk - ui * kFB;
    if (uk > ui) {
      const int64_t off = (int64_t)(ui * 8 + r) * kJD + uk * 8;
      *reinterpret_cast<uint4*>(hi + off) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(lo + off) = make_uint4(0, 0, 0, 0);
    }
  }
  if (act) {
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int c = 0; c < 8; c += 2) {
      const float x0 = (bk < bi || (bk == bi && c <= r)) ? R[r][c] : 0.f;
      const float x1 = (bk < bi || (bk == bi && c + 1 <= r)) ? R[r][c + 1] : 0.f;
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
      const __nv_bfloat162 l2 = __floats2bfloat162_rn(x0 - __low2float(h2), x1 - __high2float(h2));
      ph[c >> 1] = *reinterpret_cast<const uint32_t*>(&h2);
      pl[c >> 1] = *reinterpret_cast<const uint32_t*>(&l2);
    }
    const int64_t off = (int64_t)(bi * 8 + r) * kJD + bk * 8;
    *reinterpret_cast<uint4*>(hi + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
  }
  }
  __syncthreads();
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
  unsigned long long lfull, lfree;             // L^{-1} of the current piece; its last MMA done
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

// Persistent over the Gram kernel's pieces (the same CTA ranges): per piece,
// L^{-1} (hi, lo) is loaded once the previous piece's MMAs are done, then
// its V tiles stream through the ring; the tile count, the ring and the four
// TMEM accumulators run on across pieces.
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
  const int s_begin = a.cta_seg[blockIdx.x], s_end = a.cta_seg[blockIdx.x + 1];

  if (threadIdx.x == 0) {
    for (int i = 0; i < kLStages; ++i) {
      mbar_init(smem_u32(&ms->full[i]), 1);
      mbar_init(smem_u32(&ms->empty[i]), 1);
    }
    mbar_init(smem_u32(&ms->lfull), 1);
    mbar_init(smem_u32(&ms->lfree), 1);
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
  int l_loads = 0;                             // L^{-1} loads issued (lfull phases armed)
  bool mma_issued = false;

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      const uint64_t pol_v = policy_evict_first(), pol_l = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int k = 0; ok && k < s_end - s_begin; ++k) {
        const JSeg pc = a.segs[s_begin + k];
        const JInst in = jinst(a, pc.inst);
        // L^{-1} of this piece's instance, once the last piece's MMAs read theirs
        if (!mbar_wait(smem_u32(&ms->lfree), ((uint32_t)k & 1) ^ 1, limit, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t lbar = smem_u32(&ms->lfull);
        mbar_expect_tx(lbar, 2 * kJTileBytes);
#pragma unroll
        for (int which = 0; which < 2; ++which)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            tma_load_3d(smem_u32(sl + which * kJTileBytes + hf * kAtom), &Lp.tml, lbar, hf * 64, 0,
                        pc.inst * 2 + which, pol_l);
        ++l_loads;
        const int64_t row0 = (int64_t)in.layer * a.T + in.sq->tok_off;
        for (int t = pc.t_begin; t < pc.t_end; ++t) {
          if (!mbar_wait(smem_u32(&ms->empty[stage]), phase ^ 1, limit, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&ms->full[stage]);
          mbar_expect_tx(bar, kJTileBytes);
          const int row = (int)(row0 + (int64_t)t * kJTile);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            tma_load_3d(smem_u32(sv + stage * kJTileBytes + hf * kAtom), &Lp.tmv, bar, hf * 64,
                        in.h, row, pol_v);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kLStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(a.status, KVSEL_ERR_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: y = L^{-1} v for 128 tokens, hi then lo, into TMEM buffer i % 4
    if (lane == 0) {
      constexpr uint32_t kIdesc = instr_desc(kJD, kJTile);
      const uint32_t sv_addr = smem_u32(sv), sl_addr = smem_u32(sl);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int i = 0;
      for (int k = 0; ok && k < s_end - s_begin; ++k) {
        const JSeg pc = a.segs[s_begin + k];
        if (!mbar_wait(smem_u32(&ms->lfull), (uint32_t)k & 1, limit, abort_flag)) {
          ok = false;
          break;
        }
        for (int t = pc.t_begin; t < pc.t_end; ++t, ++i) {
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
        if (ok) tc_commit(smem_u32(&ms->lfree));
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(a.status, KVSEL_ERR_TIMEOUT);
      }
    }
  } else {
    // ---- epilogue (warps 2..5): lane quarter warp % 4, one token per lane
    const int quarter = warp & 3;
    bool ok = true;
    int i = 0;
    for (int k = 0; ok && k < s_end - s_begin; ++k) {
      const JSeg pc = a.segs[s_begin + k];
      const JInst in = jinst(a, pc.inst);
      const int P = in.sq->len - a.W;
      const int64_t plane = ((int64_t)in.layer * a.H + in.h) * a.T + in.sq->tok_off;
      for (int tl = pc.t_begin; tl < pc.t_end; ++tl, ++i) {
        const int b = i % kLBufs;
        const int t = tl * kJTile + quarter * 32 + lane;
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
        if (t < P && KVSEL_IN_BOUNDS(plane + t < (int64_t)a.layers * a.H * a.T, a.status))
          a.scores[plane + t] = w * ss;
      }
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
      if (l_loads > 0) mbar_wait(smem_u32(&ms->lfull), (uint32_t)(l_loads - 1) & 1, limit, nullptr);
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


constexpr size_t stats_smem() {
  return 1024 + kSStages * (size_t)kJTileBytes + sizeof(StatsSmem);
}

constexpr size_t gram_smem() {
  return 1024 + kGStages * (size_t)kJTileBytes + sizeof(GramSmem);
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
  {
    StatsParams sp;
    std::memset(&sp, 0, sizeof(sp));
    if (!make_rows_map(&sp.tmk, a.k, kJD, a.H, rows, 1, kJTile)) return cudaErrorInvalidValue;
    sp.a = a;
    const size_t smem = stats_smem();
    if ((e = cudaFuncSetAttribute(jacap_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)))
      return e;
    if (a.n_gram > 0) jacap_stats_kernel<<<(unsigned)a.n_gram, kSThreads, smem, a.stream>>>(sp);
    if ((e = cudaGetLastError())) return e;
  }
  {
    GramParams gp;
    std::memset(&gp, 0, sizeof(gp));
    if (!make_rows_map(&gp.tmv, a.v, kJD, a.H, rows, 1, kJTile)) return cudaErrorInvalidValue;
    gp.a = a;
    const size_t smem = gram_smem();
    if ((e = cudaFuncSetAttribute(jacap_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)))
      return e;
    if (a.n_gram > 0) jacap_gram_kernel<<<(unsigned)a.n_gram, kGThreads, smem, a.stream>>>(gp);
    if ((e = cudaGetLastError())) return e;
  }
  {
    const size_t smem = (size_t)kJD * kJD * sizeof(float);
    if ((e = cudaFuncSetAttribute(jacap_factor_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
      return e;
    if (a.layers * a.inst_per_layer > 0)
      jacap_factor_kernel<<<(unsigned)(a.layers * a.inst_per_layer), kFThreads, smem, a.stream>>>(a);
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
    if (a.n_gram > 0)
      jacap_leverage_kernel<<<(unsigned)a.n_gram, kLThreads, smem, a.stream>>>(lp);
    if ((e = cudaGetLastError())) return e;
  }
  return cudaSuccess;
}

}  // namespace kvsel
