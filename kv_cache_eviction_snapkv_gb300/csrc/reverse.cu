// Reverse-mask attention of the counter-causal scorer: every cached row of a
// sequence attends only to the rows at later original positions.
//
// Method: page "来自未来的信号：用反因果惊奇度做 KV Cache 淘汰" (signals from the
// future: KV-cache eviction by counter-causal surprise), section 3.2, steps 1
// (a strictly upper-triangular mask over the original order and position
// ids), 3 (the cached K and V reused, queries at the original positions) and
// 5 (the last position has no future context: out = 0, lse = -inf); section
// 4, Algorithm 3 (a refresh reorders the memory by surprise, so the mask
// follows the rows' positions when they are given).
//
// Work item: 128 query rows of one (layer, sequence, query head); bf16,
// D = 128. A persistent CTA per SM takes its items in turn; 320 threads: warp
// 0 TMA, warp 1 MMA, warps 2..9 softmax (query row = TMEM lane: lane quarter
// warp % 4; the two warps of a quarter take one half of the 128 columns each,
// and merge their row statistics after pass 1).
//   pass 1  S = Q K^T per 128-key tile (tcgen05, M = 128 queries, N = 128
//           keys, K = D; two TMEM S buffers so the next tile's MMAs overlap
//           this tile's softmax), then per row the maximum of S over the
//           allowed keys, m = max S log2(e) / sqrt(D);
//   pass 2  S again; P = 2^(x - m), x = S log2(e) / sqrt(D), in fp32 for the
//           allowed keys (0 elsewhere; P <= 1), summed into l and split into
//           bf16 hi = bf16(P) and lo = bf16(P - hi), stored into TMEM (the
//           A operand of the next products, so P never touches shared
//           memory); O += P_hi V + P_lo V (tcgen05, A from TMEM, V read
//           MN-major as TMA wrote it), O in TMEM; at the end O / l and
//           lse = (m + log2 l) ln 2 are written.
// TMEM: S0 columns 0..127, S1 128..255, O 256..383, P hi 384..447, lo 448..511.
// The producer loads in the order the MMA issuer consumes: pass 1 K tiles,
// then K(0), and per tile t: K(t + 1), V(t) (S(t + 1) is issued before
// P(t) V(t)). With positions in row order, key tiles before the query tile
// hold no allowed key and are skipped; with explicit positions every key tile
// of the sequence is visited.
// Every wait is bounded (KVSEL_ERR_TIMEOUT, then the roles drain and return).
#include <cmath>
#include <cstring>

#include "kvsel_device.cuh"
#include "tc_common.cuh"

namespace kvsel {
namespace {

constexpr int kRD = 128;                          // head dimension
constexpr int kRTile = 128;                       // query rows and keys per tile
constexpr int kRTileBytes = kRTile * kRD * 2;     // one bf16 tile: 32 KiB
constexpr int kRAtom = kRTile * 128;              // one 64-column swizzle atom: 16 KiB
constexpr int kRStages = 4;                       // K / V ring
constexpr int kRPCol = 384;                       // TMEM columns of P: hi 384..447, lo 448..511
constexpr int kRThreads = 320;
constexpr int kRSoft = 256;                       // softmax threads (8 warps)

struct RevSmem {
  unsigned long long qfull, qfree;                // Q tile of the current item
  unsigned long long full[kRStages], empty[kRStages];
  unsigned long long s_full[2], s_free[2];        // TMEM S buffers
  unsigned long long p_full, p_free;              // P (hi, lo) in TMEM
  unsigned long long o_done, o_free;              // TMEM O of the current item
  unsigned long long drain;                       // abort path: the MMA issuer's last commit
  uint32_t tmem_base;
  int abort_flag;
  float half_m[2][kRTile], half_l[2][kRTile];    // pass-1 row statistics of each column half
};

struct RevParams {
  CUtensorMap tmq;                                // Q as (D, H, layers * T)
  CUtensorMap tmk;                                // K as (D, H_kv, layers * T)
  CUtensorMap tmv;                                // V likewise
  RevArgs a;
};

// One work item: 128 query rows (tile qt) of one (layer, sequence, query head).
struct RevItem {
  int layer, h, hk, n, i0, kt0, nk, qt;
  int64_t row0;                                   // first row of the sequence in the layer
  int64_t tok_off;
};

template <bool kPos>
__device__ __forceinline__ RevItem rev_item(const RevArgs& a, int item) {
  RevItem it;
  it.layer = item / a.items_per_layer;
  const int rem = item - it.layer * a.items_per_layer;
  const RevSeq& sq = a.seqs[upper_find(a.S, rem, [&](int i) { return a.seqs[i].item_base; })];
  const int local = rem - sq.item_base;
  it.qt = local / a.H;
  it.h = local - it.qt * a.H;
  it.hk = it.h / (a.H / a.Hkv);
  it.n = sq.len;
  it.i0 = it.qt * kRTile;
  const int n_kt = (it.n + kRTile - 1) / kRTile;
  it.kt0 = kPos ? 0 : it.qt;                      // first key tile with an allowed key
  it.nk = n_kt - it.kt0;
  it.tok_off = sq.tok_off;
  it.row0 = (int64_t)it.layer * a.T + sq.tok_off;
  return it;
}

// Persistent: one CTA per SM; its j-th work item is j * G + c in even rounds
// and j * G + G - 1 - c in odd ones (c = blockIdx.x, G = gridDim.x). Items go
// in ascending query tiles, i.e. from the most key tiles to the fewest, so
// the serpentine order gives every CTA about the same number of tiles. The
// next item's Q and K tiles and its first-pass products overlap the current
// item's last products and its output.
__device__ __forceinline__ int rev_nth_item(int j) {
  const int G = gridDim.x, c = blockIdx.x;
  return j * G + ((j & 1) ? G - 1 - c : c);
}

// The maximum of one row's 64 logits of a tile (kMask: only where ok(e)), in
// eight independent chains: the maximum does not depend on the order.
template <bool kMask, class Ok>
__device__ __forceinline__ float rev_tile_max(const float (&x)[64], Ok ok) {
  float mx[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) mx[q] = -INFINITY;
#pragma unroll
  for (int e = 0; e < 64; ++e) mx[e & 7] = fmaxf(mx[e & 7], !kMask || ok(e) ? x[e] : -INFINITY);
  return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
}

// P = 2^(x c2 - m) of one row's 64 keys of a tile (kMask: 0 where !ok(e)) as
// 32 bf16 pairs hi = bf16(P) and lo = bf16(P - hi); returns the tile's sum of
// P, taken in four interleaved partial sums added in a fixed order.
template <bool kMask, class Ok>
__device__ __forceinline__ float rev_tile_p(const float (&x)[64], float c2, float m, Ok ok,
                                            uint32_t (&hw)[32], uint32_t (&lw)[32]) {
  float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    float p0 = ex2(fmaf(x[e], c2, -m)), p1 = ex2(fmaf(x[e + 1], c2, -m));
    if (kMask) {
      p0 = ok(e) ? p0 : 0.f;
      p1 = ok(e + 1) ? p1 : 0.f;
    }
    ls[(e >> 1) & 3] += p0 + p1;
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
    const __nv_bfloat162 l2 = __floats2bfloat162_rn(p0 - __low2float(h2), p1 - __high2float(h2));
    hw[e >> 1] = *reinterpret_cast<const uint32_t*>(&h2);
    lw[e >> 1] = *reinterpret_cast<const uint32_t*>(&l2);
  }
  return (ls[0] + ls[1]) + (ls[2] + ls[3]);
}

// kPos: the rows carry explicit positions (every key tile is visited and the
// mask compares positions); otherwise the row order is the position order.
template <bool kPos>
__global__ void __launch_bounds__(kRThreads, 1)
reverse_kernel(const __grid_constant__ RevParams R) {
  const RevArgs& a = R.a;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* s_q = smem;                                  // Q tile
  unsigned char* s_r = s_q + kRTileBytes;                     // kRStages x 32 KiB
  RevSmem* ms = reinterpret_cast<RevSmem*>(s_r + kRStages * kRTileBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long limit = a.wait_limit_ns;
  volatile int* abort_flag = &ms->abort_flag;
  const int n_items = a.layers * a.items_per_layer;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ms->qfull), 1);
    mbar_init(smem_u32(&ms->qfree), 1);
    for (int i = 0; i < kRStages; ++i) {
      mbar_init(smem_u32(&ms->full[i]), 1);
      mbar_init(smem_u32(&ms->empty[i]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ms->s_full[b]), 1);
      mbar_init(smem_u32(&ms->s_free[b]), kRSoft / 32);
    }
    mbar_init(smem_u32(&ms->p_full), kRSoft / 32);
    mbar_init(smem_u32(&ms->p_free), 1);
    mbar_init(smem_u32(&ms->o_done), 1);
    mbar_init(smem_u32(&ms->o_free), kRSoft / 32);
    mbar_init(smem_u32(&ms->drain), 1);
    ms->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ms->tmem_base)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ms->tmem_base;      // S0: columns 0..127, S1: 128..255, O: 256..383
  uint32_t armed = 0, armed_par = 0, q_par = 0;
  bool q_armed = false, mma_issued = false;

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first(), pol_kv = policy_evict_last();
      const uint32_t qbar = smem_u32(&ms->qfull);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int j = 0, item = rev_nth_item(0); ok && item < n_items; item = rev_nth_item(++j)) {
        const RevItem it = rev_item<kPos>(a, item);
        auto load = [&](const CUtensorMap* map, int kt) {
          if (!mbar_wait(smem_u32(&ms->empty[stage]), phase ^ 1, limit, abort_flag)) return false;
          const uint32_t bar = smem_u32(&ms->full[stage]);
          mbar_expect_tx(bar, kRTileBytes);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            tma_load_3d(smem_u32(s_r + stage * kRTileBytes + hf * kRAtom), map, bar, hf * 64,
                        it.hk, (int)(it.row0 + (int64_t)kt * kRTile), pol_kv);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kRStages) {
            stage = 0;
            phase ^= 1;
          }
          return true;
        };
        // the previous item's last product that reads Q is done
        if (j > 0 && !mbar_wait(smem_u32(&ms->qfree), (uint32_t)(j - 1) & 1, limit, abort_flag)) {
          ok = false;
          break;
        }
        mbar_expect_tx(qbar, kRTileBytes);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(smem_u32(s_q + hf * kRAtom), &R.tmq, qbar, hf * 64, it.h,
                      (int)(it.row0 + it.i0), pol_q);
        q_armed = true;
        q_par = (uint32_t)j & 1;
        for (int t = 0; ok && t < it.nk; ++t) ok = load(&R.tmk, it.kt0 + t);   // pass 1
        if (ok) ok = load(&R.tmk, it.kt0);                                     // pass 2
        for (int t = 0; ok && t < it.nk; ++t) {
          if (t + 1 < it.nk) ok = load(&R.tmk, it.kt0 + t + 1);
          if (ok) ok = load(&R.tmv, it.kt0 + t);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(a.status, KVSEL_ERR_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = instr_desc(kRTile, kRTile);                 // S: K-major A, B
      constexpr uint32_t kIdPV = instr_desc(kRD, kRTile) | (1u << 16);      // O: B (V) MN-major
      const uint32_t q_addr = smem_u32(s_q), r_addr = smem_u32(s_r);
      int stage = 0, u = 0, pc = 0;        // ring stage, S products, P tiles (all items)
      uint32_t phase = 0;
      bool ok = true;
      auto next_stage = [&]() {
        if (++stage == kRStages) {
          stage = 0;
          phase ^= 1;
        }
      };
      auto issue_s = [&]() {                     // S number u from the K tile in the ring
        const int b = u & 1;
        if (!mbar_wait(smem_u32(&ms->s_free[b]), ((uint32_t)(u >> 1) & 1) ^ 1, limit, abort_flag) ||
            !mbar_wait(smem_u32(&ms->full[stage]), phase, limit, abort_flag))
          return false;
        tc_fence_after();
        const uint32_t kb = r_addr + stage * kRTileBytes;
#pragma unroll
        for (int kk = 0; kk < kRD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kRAtom + (kk & 3) * 32;
          tc_mma(tmem_base + (uint32_t)(b * kRTile), smem_desc(q_addr + off), smem_desc(kb + off),
                 kIdS, kk > 0 ? 1u : 0u);
        }
        mma_issued = true;
        tc_commit(smem_u32(&ms->empty[stage]));
        tc_commit(smem_u32(&ms->s_full[b]));
        next_stage();
        ++u;
        return true;
      };
      for (int j = 0, item = rev_nth_item(0); ok && item < n_items; item = rev_nth_item(++j)) {
        const RevItem it = rev_item<kPos>(a, item);
        const int nk = it.nk;
        if (!mbar_wait(smem_u32(&ms->qfull), (uint32_t)j & 1, limit, abort_flag)) {
          ok = false;
          break;
        }
        for (int t = 0; ok && t < nk; ++t) ok = issue_s();                   // pass 1
        if (ok) ok = issue_s();                                               // pass 2: S(0)
        if (ok && nk == 1) tc_commit(smem_u32(&ms->qfree));                  // Q read for the last time
        for (int t = 0; ok && t < nk; ++t) {
          if (t + 1 < nk) {                                                   // S(t + 1)
            if (!(ok = issue_s())) break;
            if (t + 2 == nk) tc_commit(smem_u32(&ms->qfree));
          }
          // O += P(t) V(t), hi then lo; the first product of an item overwrites
          // O, so the previous item's O must have been read
          if ((t == 0 && j > 0 &&
               !mbar_wait(smem_u32(&ms->o_free), (uint32_t)(j - 1) & 1, limit, abort_flag)) ||
              !mbar_wait(smem_u32(&ms->p_full), (uint32_t)pc & 1, limit, abort_flag) ||
              !mbar_wait(smem_u32(&ms->full[stage]), phase, limit, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t vb = r_addr + stage * kRTileBytes;
#pragma unroll
          for (int which = 0; which < 2; ++which)
#pragma unroll
            for (int kk = 0; kk < kRTile / 16; ++kk)   // A = P (hi, then lo) from TMEM, 16 keys
              tc_mma_ts(tmem_base + 2 * kRTile, tmem_base + (uint32_t)(kRPCol + which * 64 + kk * 8),
                        smem_desc_mn(vb + kk * 2048), kIdPV, (t > 0 || which > 0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(&ms->empty[stage]));
          tc_commit(smem_u32(&ms->p_free));
          next_stage();
          ++pc;
        }
        if (ok) tc_commit(smem_u32(&ms->o_done));
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(a.status, KVSEL_ERR_TIMEOUT);
      }
    }
  } else {
    // ---- softmax warps: row r = lane quarter * 32 + lane; columns cb .. cb + 63
    // of every tile (and of O)
    const int quarter = warp & 3, half = (warp - 2) >> 2, cb = half * 64;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const float c2 = 1.4426950408889634f / sqrtf((float)kRD);
    auto bar_soft = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(kRSoft) : "memory"); };
    int u = 0, pc = 0;                   // S products and P tiles read so far (all items)
    bool ok = true;
    // After a failed wait a warp still walks the remaining items, doing no work
    // but taking the two barriers of each, so that every softmax warp reaches
    // every barrier whatever its own waits returned.
    for (int j = 0, item = rev_nth_item(0); item < n_items; item = rev_nth_item(++j)) {
      const RevItem it = rev_item<kPos>(a, item);
      const int n = it.n, i = it.i0 + r, nk = it.nk;
      // debug builds also check the row against the layer's rows
      const bool row_ok = i < n && KVSEL_IN_BOUNDS(it.tok_off + i < a.T, a.status);
      const int pos_i = kPos ? __ldg(a.pos + it.tok_off + min(i, n - 1)) : i;
      auto allowed = [&](int jj) -> bool {   // branch-free: jj in the sequence and later than i
        if (kPos)
          return row_ok & (jj < n) & (__ldg(a.pos + it.tok_off + min(jj, n - 1)) > pos_i);
        return row_ok & (jj < n) & (jj > i);
      };
      // a tile whose keys all lie after every query row of the tile and inside
      // the sequence needs no mask (the same answer in every thread)
      auto tile_full = [&](int jt) {
        return !kPos && jt > it.i0 + kRTile - 1 && jt + kRTile <= n;
      };
      float m = -INFINITY, l = 0.f;
      auto wait_s = [&]() {
        const bool w = mbar_wait(smem_u32(&ms->s_full[u & 1]), (uint32_t)(u >> 1) & 1, limit,
                                 abort_flag);
        return __all_sync(0xffffffffu, w);
      };
      // pass 1: this half's row maximum of the raw logits q . k over the allowed keys
      float smax = -INFINITY;
      for (int t = 0; ok && t < nk; ++t) {
        if (!(ok = wait_s())) break;
        tc_fence_after();
        const int jt = (it.kt0 + t) * kRTile, j0 = jt + cb;
        float x[64];
        tmem_load_cols_nowait<32>(lane_base + (uint32_t)((u & 1) * kRTile + cb), x);
        tmem_load_cols_nowait<32>(lane_base + (uint32_t)((u & 1) * kRTile + cb + 32), x + 32);
        tmem_wait_ld();   // both loads in flight together
        after_wait(x);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ms->s_free[u & 1]));
        ++u;
        auto ok_e = [&](int e) { return allowed(j0 + e); };
        smax = fmaxf(smax, tile_full(jt) ? rev_tile_max<false>(x, ok_e)
                                         : rev_tile_max<true>(x, ok_e));
      }
      // the row maximum in base-2 units, from both halves
      if (ok) ms->half_m[half][r] = smax * c2;
      else *abort_flag = 1;
      bar_soft();
      if (ok) m = fmaxf(ms->half_m[0][r], ms->half_m[1][r]);
      // pass 2: P (hi, lo) of this half in registers, then into TMEM once the
      // previous P V has read it
      for (int t = 0; ok && t < nk; ++t) {
        if (!(ok = wait_s())) break;
        tc_fence_after();
        const int jt = (it.kt0 + t) * kRTile, j0 = jt + cb;
        const bool full = tile_full(jt);
        uint32_t hw[32], lw[32];
        {
          float x[64];
          tmem_load_cols_nowait<32>(lane_base + (uint32_t)((u & 1) * kRTile + cb), x);
          tmem_load_cols_nowait<32>(lane_base + (uint32_t)((u & 1) * kRTile + cb + 32), x + 32);
          tmem_wait_ld();
          after_wait(x);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ms->s_free[u & 1]));
          auto ok_e = [&](int e) { return allowed(j0 + e); };
          l += full ? rev_tile_p<false>(x, c2, m, ok_e, hw, lw)
                    : rev_tile_p<true>(x, c2, m, ok_e, hw, lw);
        }
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ms->p_free), ((uint32_t)pc & 1) ^ 1,
                                               limit, abort_flag));
        if (!ok) break;
        // this half's 64 keys of the row as 32 bf16 pairs (lower half first):
        // columns kRPCol + half * 32 .. (hi) and kRPCol + 64 + half * 32 .. (lo)
        tmem_store32_u(lane_base + (uint32_t)(kRPCol + half * 32), hw);
        tmem_store32_u(lane_base + (uint32_t)(kRPCol + 64 + half * 32), lw);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ms->p_full));
        ++u;
        ++pc;
      }
      // the row sum from both halves (half order), then O / l
      if (ok) ms->half_l[half][r] = l;
      else *abort_flag = 1;
      bar_soft();
      if (ok) {
        l = ms->half_l[0][r] + ms->half_l[1][r];
        if (half == 0 && (!finite_f(l) || (m != -INFINITY && !finite_f(m))))
          record_status(a.status, KVSEL_ERR_NONFINITE);
      }
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      if (ok)
        ok = __all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&ms->o_done), (uint32_t)j & 1, limit, abort_flag));
      if (!ok) {
        *abort_flag = 1;
        continue;
      }
      tc_fence_after();
      float* out = a.out + ((it.row0 + i) * a.H + it.h) * kRD + cb;
#pragma unroll 1
      for (int c0 = 0; c0 < 64; c0 += 32) {
        float o[32];
        tmem_load_cols<32>(lane_base + (uint32_t)(2 * kRTile + cb + c0), o);
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(out + c0 + e) =
                make_float4(o[e] * inv_l, o[e + 1] * inv_l, o[e + 2] * inv_l, o[e + 3] * inv_l);
        }
      }
      // O is read: the next item's first product may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ms->o_free));
      if (row_ok && half == 0 && a.lse)
        a.lse[((int64_t)it.layer * a.H + it.h) * a.T + it.tok_off + i] =
            l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
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
      if (q_armed) mbar_wait(smem_u32(&ms->qfull), q_par, limit, nullptr);
      for (int s = 0; s < kRStages; ++s)
        if (armed & (1u << s))
          mbar_wait(smem_u32(&ms->full[s]), (armed_par >> s) & 1, limit, nullptr);
    }
    if (warp == 1 && lane == 0 && mma_issued) {
      tc_commit(smem_u32(&ms->drain));
      mbar_wait(smem_u32(&ms->drain), 0, limit, nullptr);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512)
                 : "memory");
  }
}

constexpr size_t reverse_smem() {
  return 1024 + (1 + kRStages) * (size_t)kRTileBytes + sizeof(RevSmem);
}
static_assert(reverse_smem() <= 227 * 1024, "the Q tile and the K/V ring exceed a CTA's shared memory");

}  // namespace

bool reverse_eligible(int dtype, int D, const void* q, const void* k, const void* v) {
  if (dtype != KVSEL_BF16 || D != kRD) return false;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v)) & 15)
    return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_reverse(const RevArgs& a) {
  const int64_t rows = (int64_t)a.layers * a.T;
  if (rows >= 0x7fffffffLL) return cudaErrorInvalidValue;
  if (a.layers * a.items_per_layer == 0) return cudaSuccess;
  RevParams rp;
  std::memset(&rp, 0, sizeof(rp));
  if (!make_rows_map(&rp.tmq, a.q, kRD, a.H, rows, 1, kRTile) ||
      !make_rows_map(&rp.tmk, a.k, kRD, a.Hkv, rows, 1, kRTile) ||
      !make_rows_map(&rp.tmv, a.v, kRD, a.Hkv, rows, 1, kRTile))
    return cudaErrorInvalidValue;
  rp.a = a;
  const size_t smem = reverse_smem();
  const auto kern = a.pos ? reverse_kernel<true> : reverse_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)))
    return e;
  const int64_t n_items = (int64_t)a.layers * a.items_per_layer;
  const int grid = (int)(n_items < sms ? n_items : sms);   // persistent: one CTA per SM
  kern<<<(unsigned)grid, kRThreads, smem, a.stream>>>(rp);
  return cudaGetLastError();
}

}  // namespace kvsel
