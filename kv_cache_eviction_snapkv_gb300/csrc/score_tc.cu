// Tensor-core scoring path for sm_103a: window logits on tcgen05, causal
// softmax row statistics and votes, with K read once.
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
//   * work item = (layer, sequence, head, chunk of 128 * 256/Wp tokens), Wp =
//     W padded to 16/32/64; items go round-robin to CTAs, so the chunks of one
//     instance are on neighbouring CTAs at about the same time;
//   * warp 0 streams K tiles (128 tokens x D, bf16) and the head's window
//     queries with TMA (128-byte swizzle) into a shared-memory ring;
//   * warp 1 issues tcgen05.mma (M = 128 tokens, N = Wp, K = D) so that each
//     tile's logits land in their own TMEM columns; TMEM holds two items
//     (256 columns each);
//   * warps 2..9 run two passes per item, interleaved A(0), A(1), C(0), A(2),
//     C(1), ...: pass A reads the item's logits, keeps per-row softmax
//     statistics (a warp-wide reference per row and per-lane sums of
//     2^(x - reference)) and writes the exponentials back in place; the
//     chunk's (reference, sum) pairs are then published, one relaxed 8-byte
//     store per row; pass C, one item later, turns the stored exponentials
//     into votes with the instance's merged statistics: vote = sum over rows
//     of 2^(x - reference_r) * 2^(reference_r - M_r - log2 Z_r);
//   * warp 10 gathers each instance's statistics while pass A of the next
//     item runs: a bulk copy of all its chunks' pairs into shared memory
//     (repeated until every pair is in) merged row by row in chunk order, or,
//     for instances too large for that, through owners (row r is merged by
//     chunk r mod n_chunks, which publishes the instance's final pair).
// The host keeps n_chunks <= 2 x CTAs, which makes every wait end in a
// correct program (the chunks of an instance need passes A of at most two
// rounds beyond their own); each wait is bounded anyway and reports
// KVSEL_ERR_TIMEOUT instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "kvsel_device.cuh"
#include "tc_common.cuh"

namespace kvsel {
namespace {

constexpr int kTileM = 128;           // tokens per MMA tile
constexpr int kThreads = 352;         // 11 warps
constexpr int kMmaWarp = 1;
constexpr int kEpiWarp0 = 2;          // warps 2..9: epilogue
constexpr int kEpiWarps = 8;
constexpr int kStatsWarp = 10;
constexpr int kMaxStages = 8;
constexpr int kTmemCols = 512;
constexpr int kBufCols = kTmemCols / 2;   // TMEM columns of one item
constexpr int kSmemLimit = 232448;    // 227 KiB opt-in per CTA
constexpr int kMaxChunks = 256;       // chunks per instance an owner merges (kPerLane x 32)
constexpr int kPerLane = 8;           // owner loads per lane and turn
// 11 warps, at most 3 on an SM sub-partition: 16384 / (3 * 32) rounded down
// to a multiple of 8.
constexpr int kRegs = 168;
// Shared-memory staging of the exchange pairs of two instances (n_chunks x
// Wp x 8 bytes each, half of this); instances larger than that, and every
// instance at Wp = 64, merge through owners instead.
__host__ __device__ constexpr int slot_stage_for(int nw) { return nw >= 64 ? 0 : 8192; }
__host__ __device__ constexpr int tiles_per_item(int nw) { return kBufCols / nw; }

struct TcParams {
  CUtensorMap tmk;  // K       viewed as (D, H, layers*T) bf16
  CUtensorMap tmq;  // q_win   viewed as (D, H, W, layers*S) bf16, rows >= W read as 0
  ScoreArgs a;
  int stages;
  int n_items;
};

struct Misc {
  unsigned long long full[kMaxStages], empty[kMaxStages];
  unsigned long long qfull[2], qempty[2];
  unsigned long long tile_ready[2][16];                     // per TMEM buffer and tile
  unsigned long long tmem_empty[2];
  unsigned long long ffull[2], fempty[2];                   // statistics warp -> pass C
  unsigned long long slot_bar[2];                           // bulk copies of exchange pairs
  unsigned long long mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int pub_items;                      // items whose chunk statistics are published
  float wm[2][4][64], wz[2][4][64];   // per lane quarter row statistics of one chunk
  alignas(16) float fin[2][64];       // M_r + log2 Z_r (+inf for padded rows)
  alignas(16) float cf[kEpiWarps][64];   // pass C factors of each epilogue warp
};

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


// Eight (two) relaxed loads issued back to back, so that their round trips
// overlap.
__device__ __forceinline__ void slot_read8(const unsigned long long* const (&p)[8],
                                           unsigned long long (&v)[8]) {
  asm volatile(
      "ld.relaxed.gpu.global.b64 %0, [%8];\n\t"
      "ld.relaxed.gpu.global.b64 %1, [%9];\n\t"
      "ld.relaxed.gpu.global.b64 %2, [%10];\n\t"
      "ld.relaxed.gpu.global.b64 %3, [%11];\n\t"
      "ld.relaxed.gpu.global.b64 %4, [%12];\n\t"
      "ld.relaxed.gpu.global.b64 %5, [%13];\n\t"
      "ld.relaxed.gpu.global.b64 %6, [%14];\n\t"
      "ld.relaxed.gpu.global.b64 %7, [%15];"
      : "=l"(v[0]), "=l"(v[1]), "=l"(v[2]), "=l"(v[3]), "=l"(v[4]), "=l"(v[5]), "=l"(v[6]),
        "=l"(v[7])
      : "l"(p[0]), "l"(p[1]), "l"(p[2]), "l"(p[3]), "l"(p[4]), "l"(p[5]), "l"(p[6]), "l"(p[7]));
}

__device__ __forceinline__ void slot_read2(const unsigned long long* p0,
                                           const unsigned long long* p1,
                                           unsigned long long (&v)[2]) {
  asm volatile(
      "ld.relaxed.gpu.global.b64 %0, [%2];\n\t"
      "ld.relaxed.gpu.global.b64 %1, [%3];"
      : "=l"(v[0]), "=l"(v[1])
      : "l"(p0), "l"(p1));
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


// Transposed butterfly sum over the 32 lanes of N values per lane: afterwards
// lane l holds the sum over all lanes of value l / (32 / N) (N <= 32).
template <int N>
__device__ __forceinline__ void reduce_sum(float (&v)[N], int lane) {
  int count = N;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (count >= 2) {
      const int half = count >> 1;
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      count = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    }
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// Lanes that share one row when an owner merges the pairs of nc chunks.
__device__ __forceinline__ int lanes_per_row(int nc) {
  return nc > 16 ? 32 : nc > 8 ? 16 : nc > 4 ? 8 : nc > 2 ? 4 : nc;
}

// The eight epilogue warps (named barrier 1).
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
}

// Multiplies the stored exponentials of one row (TMEM column `col` of every
// tile before `t` of the item at `base`) by f: a row's reference moved.
template <int NW>
__device__ __forceinline__ void rescale_row(uint32_t base, int col, int t, float f) {
  for (int tp = 0; tp < t; ++tp) {
    const uint32_t ca = base + (uint32_t)(tp * NW + col);
    tmem_st1(ca, tmem_ld1(ca) * f);
  }
  tmem_wait_st();
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

// The statistics warp of the scoring kernels: collects, for each of this
// CTA's items in order, M_r + log2 Z_r of every row of its instance for the
// vote pass. Where the pairs of all chunks of the instance fit the staging
// buffer, one bulk copy brings them into shared memory (repeated until every
// pair is published) and the warp merges each row over the chunks in chunk
// order. Larger instances go through owners: row r is merged by chunk r mod nc
// (same order), which publishes the instance's final pair of that row; every
// chunk then reads the W final pairs. The owner step runs at most
// `owner_ahead` items ahead of the collection step (the vote pass lags the
// statistics pass by that much less two); each turn of the loop issues its
// loads together.
template <int NW>
__device__ __forceinline__ void stats_warp_loop(const ScoreArgs& a, Misc* ms, int n_my, int G,
                                                int lane, unsigned long long limit,
                                                volatile int* abort_flag, int owner_ahead) {
  const int W = a.W * a.qg;   // window rows of an instance (qg query heads of W rows)
  constexpr int kStageSlots = slot_stage_for(NW) / 16;   // per staging buffer
  const unsigned long long* part = reinterpret_cast<const unsigned long long*>(a.part);
  unsigned long long* fslots = reinterpret_cast<unsigned long long*>(a.final_stats);
  const unsigned long long* stage = reinterpret_cast<const unsigned long long*>(
      reinterpret_cast<const unsigned char*>(ms) + sizeof(Misc));
  int na = 0, nf = 0;
  int agg_j = 0;                 // owned rows of item na already merged
  int dec_a = -1, dec_f = -1;    // items whose positions are decoded below
  ItemPos ipa{}, ipf{};
  SeqDesc sda{};
  // staging buffer b holds the pairs of item nf or nf + 1 (the one with
  // parity b): its item, whether it is collected directly, a copy in
  // flight, all pairs in, the copy barrier's parity, source and chunks
  int cp_item[2] = {-1, -1}, cp_nc[2] = {0, 0};
  bool cp_direct[2] = {false, false}, cp_out[2] = {false, false}, cp_ready[2] = {false, false};
  uint32_t cp_par[2] = {0, 0};
  float cp_m[2] = {0.f, 0.f}, cp_z[2] = {0.f, 0.f};   // this lane's row, merged
  const unsigned long long* cp_src[2] = {nullptr, nullptr};
  const volatile int* pub_items = &ms->pub_items;
  bool ok = true;
  unsigned long long t_last = global_ns();
  while (nf < n_my) {
    bool prog = false;
    // ---- owner step for item na
    if (na < n_my && na <= nf + owner_ahead) {
      if (dec_a != na) {
        ipa = decode_item(a, blockIdx.x + na * G);
        sda = a.seqs[ipa.s];
        dec_a = na;
      }
      const int nc = sda.n_chunks, c = ipa.c;
      const int n_own = (nc * a.wpad <= kStageSlots || c >= W) ? 0 : (W - 1 - c) / nc + 1;
      if (agg_j >= n_own) {
        ++na;
        agg_j = 0;
        prog = true;
      } else {
        const int g = lanes_per_row(nc);
        const int j = agg_j + lane / g, sl = lane % g;
        const int r = c + j * nc;
        const bool act = j < n_own;
        const unsigned long long* p0 =
            part + ((int64_t)ipa.layer * a.items_per_layer + sda.item_base +
                    (int64_t)ipa.h * nc) * a.wpad + (act ? r : 0);
        const unsigned long long* pp[kPerLane];
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
          const int ch = sl + k * g;
          pp[k] = p0 + (int64_t)((act && ch < nc) ? ch : 0) * a.wpad;
        }
        unsigned long long v[kPerLane];
        slot_read8(pp, v);
        bool have = true;
#pragma unroll
        for (int k = 0; k < kPerLane; ++k)
          if (act && sl + k * g < nc) have &= v[k] != kEmptySlot;
        if (__all_sync(0xffffffffu, have)) {
          float m = -INFINITY, z = 0.f;
#pragma unroll
          for (int k = 0; k < kPerLane; ++k)
            if (act && sl + k * g < nc)
              merge_stats(m, z, __uint_as_float((uint32_t)v[k]),
                          __uint_as_float((uint32_t)(v[k] >> 32)));
          for (int off = g >> 1; off >= 1; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const float z2 = __shfl_xor_sync(0xffffffffu, z, off);
            merge_stats(m, z, m2, z2);
          }
          if (act && sl == 0) {
            if (m != m) m = INFINITY;
            slot_publish(fslots + (int64_t)ipa.inst * a.wpad + r, m, z);
          }
          agg_j += 32 / g;
          if (agg_j >= n_own) {
            ++na;
            agg_j = 0;
          }
          prog = true;
        }
      }
    }
    // ---- bulk copies for items nf and nf + 1, each issued once this
    // CTA's own chunk of the item is published, repeated until every
    // pair of the instance is in
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int x = (nf & 1) == b ? nf : nf + 1;
      if (x >= n_my) continue;
      if (cp_item[b] != x) {  // the buffer's previous item is collected
        const ItemPos ipx = decode_item(a, blockIdx.x + x * G);
        const SeqDesc sdx = a.seqs[ipx.s];
        cp_item[b] = x;
        cp_nc[b] = sdx.n_chunks;
        cp_direct[b] = sdx.n_chunks * a.wpad <= kStageSlots;
        cp_ready[b] = false;
        cp_src[b] = part + ((int64_t)ipx.layer * a.items_per_layer + sdx.item_base +
                            (int64_t)ipx.h * sdx.n_chunks) * a.wpad;
      }
      if (!cp_direct[b] || cp_ready[b]) continue;
      const unsigned long long* buf_b = stage + b * kStageSlots;
      if (!cp_out[b]) {
        if (__shfl_sync(0xffffffffu, *pub_items > x ? 1 : 0, 0)) {
          __syncwarp();  // every lane is done with the staging buffer
          if (lane == 0) {
            const uint32_t bytes = (uint32_t)(cp_nc[b] * a.wpad * 8);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_expect_tx(smem_u32(&ms->slot_bar[b]), bytes);
            bulk_load(smem_u32(buf_b), cp_src[b], bytes, smem_u32(&ms->slot_bar[b]));
          }
          cp_out[b] = true;
        }
      } else if (__shfl_sync(0xffffffffu,
                             mbar_try(smem_u32(&ms->slot_bar[b]), cp_par[b]) ? 1 : 0, 0)) {
        mbar_wait(smem_u32(&ms->slot_bar[b]), cp_par[b], limit, nullptr);  // done: acquire
        cp_par[b] ^= 1;
        cp_out[b] = false;
        // merge each row over the chunks in two passes (max, then the
        // rescaled sum), checking that every pair is in; lane = row, and
        // for W <= 16 a power of two, lane group q takes chunks q, q + ng,
        // ... (the groups merged last)
        const int ng = (W <= 16 && (W & (W - 1)) == 0) ? 32 / W : 1;
        const int rpg = 32 / ng, r = lane % rpg, q = lane / rpg;
        const int nc = cp_nc[b];
        bool have = true;
        float M = -INFINITY, Z = 0.f;
        if (r < W) {
          // four independent chains in each pass (a fixed order)
          const unsigned long long* col = buf_b + r;
          const int st = ng * a.wpad;
          float mk[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          int ch = q;
          for (; ch + 3 * ng < nc; ch += 4 * ng) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const unsigned long long sv = col[(ch * a.wpad) + k * st];
              have &= sv != kEmptySlot;
              mk[k] = fmaxf(mk[k], __uint_as_float((uint32_t)sv));
            }
          }
          for (; ch < nc; ch += ng) {
            const unsigned long long sv = col[ch * a.wpad];
            have &= sv != kEmptySlot;
            mk[0] = fmaxf(mk[0], __uint_as_float((uint32_t)sv));
          }
          M = fmaxf(fmaxf(mk[0], mk[1]), fmaxf(mk[2], mk[3]));
          if (M != -INFINITY) {
            float zk[4] = {0.f, 0.f, 0.f, 0.f};
            ch = q;
            for (; ch + 3 * ng < nc; ch += 4 * ng) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const unsigned long long sv = col[(ch * a.wpad) + k * st];
                zk[k] = fmaf(__uint_as_float((uint32_t)(sv >> 32)),
                             ex2(__uint_as_float((uint32_t)sv) - M), zk[k]);
              }
            }
            for (; ch < nc; ch += ng) {
              const unsigned long long sv = col[ch * a.wpad];
              zk[0] = fmaf(__uint_as_float((uint32_t)(sv >> 32)),
                           ex2(__uint_as_float((uint32_t)sv) - M), zk[0]);
            }
            Z = (zk[0] + zk[1]) + (zk[2] + zk[3]);
          }
        }
        for (int off = 16; off >= rpg; off >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, M, off);
          const float z2 = __shfl_xor_sync(0xffffffffu, Z, off);
          merge_stats(M, Z, m2, z2);
        }
        cp_m[b] = M;
        cp_z[b] = Z;
        cp_ready[b] = __all_sync(0xffffffffu, have);
        prog = true;
      }
    }
    // ---- collection step for item nf
    if (nf < na) {
      const int fbuf = nf & 1;
      const uint32_t fpar = (uint32_t)(nf >> 1) & 1;
      const bool direct = fbuf ? cp_direct[1] : cp_direct[0];
      const bool ready = fbuf ? cp_ready[1] : cp_ready[0];
      float* fin = ms->fin[fbuf];
      bool done = false;
      if (direct) {
        if (ready && __shfl_sync(0xffffffffu,
                                 mbar_try(smem_u32(&ms->fempty[fbuf]), fpar ^ 1) ? 1 : 0, 0)) {
          mbar_wait(smem_u32(&ms->fempty[fbuf]), fpar ^ 1, limit, nullptr);
          const int ng = (W <= 16 && (W & (W - 1)) == 0) ? 32 / W : 1;
          const int r = lane % (32 / ng);
          const float M = fbuf ? cp_m[1] : cp_m[0], Z = fbuf ? cp_z[1] : cp_z[0];
          if (lane < 32 / ng && r < W) fin[r] = M + log2f(Z);
          if (fbuf) cp_ready[1] = false; else cp_ready[0] = false;
          done = true;
        }
      } else if (__shfl_sync(0xffffffffu,
                             mbar_try(smem_u32(&ms->fempty[fbuf]), fpar ^ 1) ? 1 : 0, 0)) {
        if (dec_f != nf) {
          ipf = decode_item(a, blockIdx.x + nf * G);
          dec_f = nf;
        }
        const unsigned long long* f0 = fslots + (int64_t)ipf.inst * a.wpad;
        unsigned long long f[2];
        slot_read2(f0 + min(lane, W - 1), f0 + min(lane + 32, W - 1), f);
        bool have = true;
#pragma unroll
        for (int k = 0; k < 2; ++k)
          if (lane + 32 * k < W) have &= f[k] != kEmptySlot;
        if (__all_sync(0xffffffffu, have)) {
          mbar_wait(smem_u32(&ms->fempty[fbuf]), fpar ^ 1, limit, nullptr);
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int r = lane + 32 * k;
            if (r < W)
              fin[r] = __uint_as_float((uint32_t)f[k]) +
                       log2f(__uint_as_float((uint32_t)(f[k] >> 32)));
          }
          done = true;
        }
      }
      if (done) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int r = lane + 32 * k;
          if (r >= W && r < NW) fin[r] = INFINITY;
        }
        mbar_arrive(smem_u32(&ms->ffull[fbuf]));
        ++nf;
        prog = true;
      }
    }
    const unsigned long long now = global_ns();
    if (prog) {
      t_last = now;
    } else if (__any_sync(0xffffffffu, *abort_flag != 0 || now - t_last > limit)) {
      ok = false;
      break;
    }
  }
  if (!ok && lane == 0) {
    *abort_flag = 1;
    record_status(a.status, KVSEL_ERR_TIMEOUT);
  }
  // a bulk copy still in flight must land before the CTA exits
#pragma unroll
  for (int b = 0; b < 2; ++b)
    if (cp_out[b] && lane == 0) mbar_wait(smem_u32(&ms->slot_bar[b]), cp_par[b], limit, nullptr);
}

template <int NW, int KD, bool LOGITS>
__global__ void __maxnreg__(kRegs) tc_score_kernel(const __grid_constant__ TcParams P) {
  constexpr int kHalves = KD / 64;
  constexpr int kStageBytes = kTileM * KD * 2;
  constexpr int kQBytes = NW * KD * 2;
  constexpr int kTiles = tiles_per_item(NW);   // tiles per item
  constexpr int NH = NW / 2;                   // pass-A rows per epilogue warp
  constexpr uint32_t kIdesc = instr_desc(NW, kTileM);
  const ScoreArgs& a = P.a;
  const int stages = P.stages;
  const int W = a.W;
  // qg query heads share the instance's K: window row r of the tile is query
  // offset r / qg of head r % qg; R rows are valid
  const int qg = a.qg;
  const int R = W * qg;
  const int G = gridDim.x;
  // this CTA's items: blockIdx.x + it * G, it = 0 .. n_my - 1
  const int n_my = P.n_items > (int)blockIdx.x ? (P.n_items - 1 - (int)blockIdx.x) / G + 1 : 0;

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
      for (int t = 0; t < kTiles; ++t) mbar_init(smem_u32(&ms->tile_ready[b][t]), 1);
      mbar_init(smem_u32(&ms->tmem_empty[b]), kEpiWarps);
      mbar_init(smem_u32(&ms->ffull[b]), 32);
      mbar_init(smem_u32(&ms->fempty[b]), kEpiWarps * 32);
      mbar_init(smem_u32(&ms->slot_bar[b]), 1);
    }
    mbar_init(smem_u32(&ms->mma_done), 1);
    ms->abort_flag = 0;
    ms->pub_items = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == kMmaWarp) {
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

  // producer lane: stages (and query buffers) with a copy started, and the
  // parity of the last phase each was armed for; MMA lane: issued anything
  uint32_t armed = 0, armed_par = 0, q_armed = 0, q_par = 0;
  bool mma_issued = false;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmk))
                   : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmq))
                   : "memory");
      const uint64_t pol_k = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      const int seqs_per_layer = (int)(a.q_rows / a.q_W);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; ok && it < n_my; ++it) {
        const int item = blockIdx.x + it * G;
        const ItemPos ip = decode_item(a, item);
        const SeqDesc sd = a.seqs[ip.s];
        const int tok0 = ip.c * a.chunk_tokens;
        const int ntiles = (min(a.chunk_tokens, sd.len - tok0) + kTileM - 1) / kTileM;
        const int qb = it & 1;
        const uint32_t qp = (uint32_t)(it >> 1) & 1;
        if (!mbar_wait(smem_u32(&ms->qempty[qb]), qp ^ 1, limit, abort_flag)) {
          ok = false;
          break;
        }
        mbar_expect_tx(smem_u32(&ms->qfull[qb]), kQBytes);
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf)
          tma_load_4d(smem_u32(sq + qb * kQBytes + hf * NW * 128), &P.tmq,
                      smem_u32(&ms->qfull[qb]), hf * 64, ip.h * qg, 0,
                      ip.layer * seqs_per_layer + sd.index, pol_q);
        q_armed |= 1u << qb;
        q_par = (q_par & ~(1u << qb)) | (qp << qb);
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
                        smem_u32(&ms->full[stage]), hf * 64, ip.h / a.kv_group,
                        krow0 + t * kTileM, pol_k);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
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
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sk_addr = smem_u32(sk), sq_addr = smem_u32(sq);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; ok && it < n_my; ++it) {
        const int item = blockIdx.x + it * G;
        const ItemPos ip = decode_item(a, item);
        const SeqDesc sd = a.seqs[ip.s];
        const int tok0 = ip.c * a.chunk_tokens;
        const int ntiles = (min(a.chunk_tokens, sd.len - tok0) + kTileM - 1) / kTileM;
        const int b = it & 1, qb = it & 1;
        const uint32_t use = (uint32_t)(it >> 1) & 1;
        if (!mbar_wait(smem_u32(&ms->tmem_empty[b]), use ^ 1, limit, abort_flag) ||
            !mbar_wait(smem_u32(&ms->qfull[qb]), use, limit, abort_flag)) {
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
          const uint32_t d_tmem = tmem_base + (uint32_t)(b * kBufCols + t * NW);
#pragma unroll
          for (int kk = 0; kk < KD / 16; ++kk) {
            const uint32_t a_addr =
                sk_addr + stage * kStageBytes + (kk >> 2) * (kTileM * 128) + (kk & 3) * 32;
            const uint32_t b_addr = sq_addr + qb * kQBytes + (kk >> 2) * (NW * 128) + (kk & 3) * 32;
            tc_mma(d_tmem, smem_desc(a_addr), smem_desc(b_addr), kIdesc, kk > 0 ? 1u : 0u);
          }
          mma_issued = true;
          tc_commit(smem_u32(&ms->empty[stage]));
          tc_commit(smem_u32(&ms->tile_ready[b][t]));
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
    }
  } else if (warp == kStatsWarp) {
    if constexpr (!LOGITS) stats_warp_loop<NW>(a, ms, n_my, G, lane, limit, abort_flag, 2);
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - kEpiWarp0;         // 0..7
    const int quarter = warp & 3;           // TMEM lanes 32*quarter .. +31
    const int sub = e >> 2;                 // pass A: row half; pass C: tile parity
    const int row0 = sub * NH;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(32 * quarter) << 16);
    const float s2 = a.scale_log2;
    bool ok = true;
    // parity of the next phase of tile_ready[b][t] is bit 16 * b + t (items
    // may have fewer tiles than a buffer, so each tile counts its own uses)
    uint32_t tph = 0;
    const int n_steps = LOGITS ? n_my : n_my + (n_my > 0 ? 1 : 0);
    for (int step = 0; step < n_steps; ++step) {
      for (int pass = 0; pass < 2; ++pass) {
        const int it = pass == 0 ? step : step - 1;
        if (it < 0 || it >= n_my || (LOGITS && pass == 1)) continue;
        const int item = blockIdx.x + it * G;
        const ItemPos ip = decode_item(a, item);
        const SeqDesc sd = a.seqs[ip.s];
        const int tok0 = ip.c * a.chunk_tokens;
        const int ntiles = (min(a.chunk_tokens, sd.len - tok0) + kTileM - 1) / kTileM;
        const int prefix = sd.len - W;
        const int b = it & 1;
        const uint32_t use = (uint32_t)(it >> 1) & 1;
        const uint32_t item_addr = lane_addr + (uint32_t)(b * kBufCols);
        if (pass == 0) {
          // ---- pass A: per-row softmax statistics of this warp's tokens.
          // The two warps of a TMEM lane quarter split the rows (half `sub`).
          // Per row the warp keeps one reference (the same in every lane: a
          // logit of the chunk) and each lane the sum of 2^(x - reference);
          // the reference moves to the warp's largest logit only when one
          // exceeds it by more than 32 (so no term exceeds 2^32), which after
          // the first tile is rare, and then the row's stored exponentials
          // are rescaled.
          float mref[NH], zsum[NH];
#pragma unroll
          for (int i = 0; i < NH; ++i) {
            mref[i] = -INFINITY;
            zsum[i] = 0.f;
          }
          float ymin = INFINITY;
          bool bad = false, fresh = true;
          for (int t = 0; t < ntiles; ++t) {
            // warp-uniform: the TMEM loads and stores below are .sync.aligned
            const uint32_t tbit = 1u << (16 * b + t);
            if (ok)
              ok = __all_sync(0xffffffffu,
                              mbar_wait(smem_u32(&ms->tile_ready[b][t]), (tph & tbit) ? 1u : 0u,
                                        limit, abort_flag));
            tph ^= tbit;
            if (!ok) continue;
            tc_fence_after();
            const uint32_t taddr = item_addr + (uint32_t)(t * NW + row0);
            const int tbase = tok0 + t * kTileM + 32 * quarter;
            const int tok = tbase + lane;
            if constexpr (LOGITS) {
              float x[NH];
              tmem_load_cols<NH>(taddr, x);
              if (tok < sd.len) {
                const int64_t base = ((int64_t)ip.layer * a.H + ip.h) * W;
#pragma unroll
                for (int i = 0; i < NH; ++i)
                  if (row0 + i < W)
                    a.logits[(base + row0 + i) * a.T + sd.tok_off + tok] = x[i] * a.scale;
              }
            } else if (tbase + 31 < prefix) {
              // every row sees every token of this warp
              float y[NH];
              tmem_load_cols<NH>(taddr, y);
              if (fresh) {  // first tile: lane 0's logits are the references
#pragma unroll
                for (int i = 0; i < NH; ++i) mref[i] = __shfl_sync(0xffffffffu, y[i] * s2, 0);
                fresh = false;
              }
              bool need = false;
#pragma unroll
              for (int i = 0; i < NH; ++i) {
                y[i] = fmaf(y[i], s2, -mref[i]);
                need |= y[i] > 32.f;
              }
              if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int i = 0; i < NH; ++i) {
                  if (__any_sync(0xffffffffu, y[i] > 32.f)) {
                    const float xs = y[i] + mref[i];   // the logit in base-2 units
                    if (!finite_f(xs)) bad = true;
                    const float mx = warp_max(xs);
                    const float f = ex2(mref[i] - mx);
                    rescale_row<NW>(item_addr, row0 + i, t, f);
                    zsum[i] *= f;
                    mref[i] = mx;
                    y[i] = xs - mx;
                  }
                }
              }
#pragma unroll
              for (int i = 0; i < NH; ++i) {
                ymin = fminf(ymin, y[i]);   // a -inf logit shows here
                y[i] = ex2(y[i]);
                zsum[i] += y[i];            // a NaN shows in the sum
              }
              tmem_store_cols<NH>(taddr, y);
            } else {
              // window tokens and the ragged tail, eight rows at a time: rows
              // visible to this token are row0 + i < R with tok <= P + (row0 + i) / qg
              const int lo = max(0, (tok - prefix) * qg - row0);
              const int hi = tok < sd.len ? min(NH, R - row0) : 0;
#pragma unroll
              for (int cb = 0; cb < NH; cb += 8) {
                float xb[8];
                tmem_load_cols<8>(taddr + cb, xb);
                bool need = false;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  const int i = cb + u;
                  xb[u] *= s2;
                  if (i < hi && !finite_f(xb[u])) bad = true;
                  need |= i < hi && i >= lo && xb[u] > mref[i] + 32.f;
                }
                if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                  for (int u = 0; u < 8; ++u) {
                    const int i = cb + u;
                    const bool vis = i < hi && i >= lo;
                    if (__any_sync(0xffffffffu, vis && xb[u] > mref[i] + 32.f)) {
                      const float mx = warp_max(vis ? xb[u] : -INFINITY);
                      if (mref[i] != -INFINITY) {
                        const float f = ex2(mref[i] - mx);
                        rescale_row<NW>(item_addr, row0 + i, t, f);
                        zsum[i] *= f;
                      }
                      mref[i] = mx;
                    }
                  }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  const int i = cb + u;
                  xb[u] = (i < hi && i >= lo) ? ex2(xb[u] - mref[i]) : 0.f;
                  zsum[i] += xb[u];
                }
                tmem_store_cols<8>(taddr + cb, xb);
              }
            }
          }
          if constexpr (LOGITS) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ms->tmem_empty[b]));
          } else {
            // ---- hand the chunk's statistics over: the lanes' sums added by
            // a transposed butterfly; one pair per row and lane quarter; then
            // (all epilogue warps, uniformly) one warp merges the quarters in
            // a fixed order and publishes one pair per row
            tmem_wait_st();
#pragma unroll
            for (int i = 0; i < NH; ++i)
              if (row0 + i < R && zsum[i] != zsum[i]) bad = true;
            if (ymin == -INFINITY) bad = true;
            if (bad) record_status(a.status, KVSEL_ERR_NONFINITE);
            reduce_sum<NH>(zsum, lane);
            constexpr int kLanesPerRow = 32 / NH;
            if (lane == 0) {
#pragma unroll
              for (int i = 0; i < NH; ++i) ms->wm[b][quarter][row0 + i] = mref[i];
            }
            if (lane % kLanesPerRow == 0) ms->wz[b][quarter][row0 + lane / kLanesPerRow] = zsum[0];
            tc_fence_before();
            epi_bar();
            tc_fence_after();
            if (warp == kEpiWarp0) {
              for (int r = lane; r < R; r += 32) {
                float m = ms->wm[b][0][r], z = ms->wz[b][0][r];
#pragma unroll
                for (int q = 1; q < 4; ++q) merge_stats(m, z, ms->wm[b][q][r], ms->wz[b][q][r]);
                if (m != m) m = INFINITY;  // keep the empty pattern unique (NONFINITE is recorded)
                if (!(a.inject == 1 && item == 0))
                  slot_publish(reinterpret_cast<unsigned long long*>(a.part) +
                                   (int64_t)item * a.wpad + r, m, z);
              }
              if (lane == 0) *reinterpret_cast<volatile int*>(&ms->pub_items) = it + 1;
            }
          }
        } else {
          // ---- pass C: the vote of a prefix token is the sum over rows of
          // its stored exponential times cf_r = 2^(reference_r - M_r -
          // log2 Z_r) (the reference of this lane quarter; 0 for padded
          // rows). This warp takes the tiles of parity `sub`, all rows.
          const int64_t plane = ((int64_t)ip.layer * a.H + ip.h) * a.T + sd.tok_off;
          if (ok)
            ok = __all_sync(0xffffffffu,
                            mbar_wait(smem_u32(&ms->ffull[b]), use, limit, abort_flag));
          float* cf = ms->cf[e];
          for (int r = lane; r < NW; r += 32)
            cf[r] = r < R ? ex2(ms->wm[b][quarter][r] - ms->fin[b][r]) : 0.f;
          __syncwarp();
          mbar_arrive(smem_u32(&ms->fempty[b]));
          for (int t = sub; t < ntiles; t += 2) {
            if (!ok) break;
            float ev[NW];
            tmem_load_row<NW>(item_addr + (uint32_t)(t * NW), ev);
            float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < NW; i += 4) {
              const float4 c4 = *reinterpret_cast<const float4*>(cf + i);
              p[0] = fmaf(ev[i], c4.x, p[0]);
              p[1] = fmaf(ev[i + 1], c4.y, p[1]);
              p[2] = fmaf(ev[i + 2], c4.z, p[2]);
              p[3] = fmaf(ev[i + 3], c4.w, p[3]);
            }
            const int tok = tok0 + t * kTileM + 32 * quarter + lane;
            if (tok < sd.len)
              a.votes[plane + tok] =
                  tok < prefix ? (p[0] + p[1]) + (p[2] + p[3]) : 0.f;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ms->tmem_empty[b]));
        }
        if (!ok) *abort_flag = 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // Every role has left its loop, so the abort flag is final. After an abort,
  // drain what is still in flight before the shared memory and TMEM go away:
  // the producer waits for the last copy it started into each stage and
  // query buffer, the MMA issuer for its last instruction (all bounded,
  // ignoring the abort flag).
  if (ms->abort_flag) {
    if (warp == 0 && lane == 0) {
      for (int s = 0; s < kMaxStages; ++s)
        if (armed & (1u << s))
          mbar_wait(smem_u32(&ms->full[s]), (armed_par >> s) & 1, limit, nullptr);
      for (int b = 0; b < 2; ++b)
        if (q_armed & (1u << b))
          mbar_wait(smem_u32(&ms->qfull[b]), (q_par >> b) & 1, limit, nullptr);
    }
    if (warp == kMmaWarp && lane == 0 && mma_issued) {
      tc_commit(smem_u32(&ms->mma_done));
      mbar_wait(smem_u32(&ms->mma_done), 0, limit, nullptr);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// Two-pass variant for long instances
// ---------------------------------------------------------------------------

// An instance whose chunks fill much of the GPU's tensor memory cannot keep
// its exponentials on chip until its statistics are merged without stalling
// the stream of K. Here the chunks' exponentials are not kept: pass 1 of an
// item computes its row statistics from the logits and frees its tensor
// memory at once; pass 2 of the same item runs `lag` items later in the
// same CTA, when the instance's statistics are merged, recomputes the
// logits from the same K tiles (read a second time, now from L2: the lag is
// a few items, tens of MiB over the GPU) and turns them into votes:
//   vote_j = sum over rows of 2^(x_rj * log2(e)/sqrt(D) - M_r - log2 Z_r).
// Per step the producer, the MMA issuer and the epilogue take pass 1 of item
// `step` (TMEM buffer 0, query buffer 0) and then pass 2 of item
// `step - lag` (buffer 1, query buffer 1). Pass 2 of an item waits only for
// passes 1 of chunks that come at most two rounds later (n_chunks <= 2 x
// CTAs), whose steps come no later than its own (lag >= 2), and each of
// those waits for earlier steps only, so every wait ends in a correct
// program; each wait is bounded anyway.
template <int NW, int KD>
__global__ void __maxnreg__(kRegs) tc_score_rc_kernel(const __grid_constant__ TcParams P) {
  constexpr int kHalves = KD / 64;
  constexpr int kStageBytes = kTileM * KD * 2;
  constexpr int kQBytes = NW * KD * 2;
  constexpr int kTiles = tiles_per_item(NW);
  constexpr int NH = NW / 2;                   // pass-1 rows per epilogue warp
  constexpr uint32_t kIdesc = instr_desc(NW, kTileM);
  const ScoreArgs& a = P.a;
  const int stages = P.stages;
  const int W = a.W;
  const int G = gridDim.x;
  const int lag = a.two_pass;
  const int n_my = P.n_items > (int)blockIdx.x ? (P.n_items - 1 - (int)blockIdx.x) / G + 1 : 0;
  const int n_steps = n_my > 0 ? n_my + lag : 0;

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
      for (int t = 0; t < kTiles; ++t) mbar_init(smem_u32(&ms->tile_ready[b][t]), 1);
      mbar_init(smem_u32(&ms->tmem_empty[b]), kEpiWarps);
      mbar_init(smem_u32(&ms->ffull[b]), 32);
      mbar_init(smem_u32(&ms->fempty[b]), kEpiWarps * 32);
      mbar_init(smem_u32(&ms->slot_bar[b]), 1);
    }
    mbar_init(smem_u32(&ms->mma_done), 1);
    ms->abort_flag = 0;
    ms->pub_items = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == kMmaWarp) {
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

  uint32_t armed = 0, armed_par = 0, q_armed = 0, q_par = 0;
  bool mma_issued = false;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmk))
                   : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmq))
                   : "memory");
      // pass 1 leaves its K tiles in L2 for pass 2, which reads them last
      const uint64_t pol_k1 = policy_evict_last();
      const uint64_t pol_k2 = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      const int seqs_per_layer = (int)(a.q_rows / a.q_W);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int step = 0; ok && step < n_steps; ++step) {
        for (int pass = 0; ok && pass < 2; ++pass) {
          const int it = pass == 0 ? step : step - lag;
          if (it < 0 || it >= n_my) continue;
          const ItemPos ip = decode_item(a, blockIdx.x + it * G);
          const SeqDesc sd = a.seqs[ip.s];
          const int tok0 = ip.c * a.chunk_tokens;
          const int ntiles = (min(a.chunk_tokens, sd.len - tok0) + kTileM - 1) / kTileM;
          const uint32_t qp = (uint32_t)it & 1;   // each query buffer serves one pass
          if (!mbar_wait(smem_u32(&ms->qempty[pass]), qp ^ 1, limit, abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(smem_u32(&ms->qfull[pass]), kQBytes);
#pragma unroll
          for (int hf = 0; hf < kHalves; ++hf)
            tma_load_4d(smem_u32(sq + pass * kQBytes + hf * NW * 128), &P.tmq,
                        smem_u32(&ms->qfull[pass]), hf * 64, ip.h, 0,
                        ip.layer * seqs_per_layer + sd.index, pol_q);
          q_armed |= 1u << pass;
          q_par = (q_par & ~(1u << pass)) | (qp << pass);
          const int krow0 = (int)(ip.layer * a.T + sd.tok_off + tok0);
          const uint64_t pol_k = pass == 0 ? pol_k1 : pol_k2;
          for (int t = 0; t < ntiles; ++t) {
            if (!mbar_wait(smem_u32(&ms->empty[stage]), phase ^ 1, limit, abort_flag)) {
              ok = false;
              break;
            }
            mbar_expect_tx(smem_u32(&ms->full[stage]), kStageBytes);
#pragma unroll
            for (int hf = 0; hf < kHalves; ++hf)
              tma_load_3d(smem_u32(sk + stage * kStageBytes + hf * kTileM * 128), &P.tmk,
                          smem_u32(&ms->full[stage]), hf * 64, ip.h / a.kv_group,
                          krow0 + t * kTileM, pol_k);
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
            if (++stage == stages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(a.status, KVSEL_ERR_TIMEOUT);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sk_addr = smem_u32(sk), sq_addr = smem_u32(sq);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int step = 0; ok && step < n_steps; ++step) {
        for (int pass = 0; ok && pass < 2; ++pass) {
          const int it = pass == 0 ? step : step - lag;
          if (it < 0 || it >= n_my) continue;
          const ItemPos ip = decode_item(a, blockIdx.x + it * G);
          const SeqDesc sd = a.seqs[ip.s];
          const int tok0 = ip.c * a.chunk_tokens;
          const int ntiles = (min(a.chunk_tokens, sd.len - tok0) + kTileM - 1) / kTileM;
          const uint32_t use = (uint32_t)it & 1;  // buffer `pass` serves one pass
          if (!mbar_wait(smem_u32(&ms->tmem_empty[pass]), use ^ 1, limit, abort_flag) ||
              !mbar_wait(smem_u32(&ms->qfull[pass]), use, limit, abort_flag)) {
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
            const uint32_t d_tmem = tmem_base + (uint32_t)(pass * kBufCols + t * NW);
#pragma unroll
            for (int kk = 0; kk < KD / 16; ++kk) {
              const uint32_t a_addr =
                  sk_addr + stage * kStageBytes + (kk >> 2) * (kTileM * 128) + (kk & 3) * 32;
              const uint32_t b_addr =
                  sq_addr + pass * kQBytes + (kk >> 2) * (NW * 128) + (kk & 3) * 32;
              tc_mma(d_tmem, smem_desc(a_addr), smem_desc(b_addr), kIdesc, kk > 0 ? 1u : 0u);
            }
            mma_issued = true;
            tc_commit(smem_u32(&ms->empty[stage]));
            tc_commit(smem_u32(&ms->tile_ready[pass][t]));
            if (++stage == stages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (ok) tc_commit(smem_u32(&ms->qempty[pass]));
        }
      }
      if (!ok) {
        *abort_flag = 1;
        record_status(a.status, KVSEL_ERR_TIMEOUT);
      }
    }
  } else if (warp == kStatsWarp) {
    // the owners keep up with pass 1, which runs `lag` items ahead of the
    // collection for pass 2
    stats_warp_loop<NW>(a, ms, n_my, G, lane, limit, abort_flag, 2 + lag);
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - kEpiWarp0;         // 0..7
    const int quarter = warp & 3;           // TMEM lanes 32*quarter .. +31
    const int sub = e >> 2;                 // pass 1: row half; pass 2: tile parity
    const int row0 = sub * NH;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(32 * quarter) << 16);
    const float s2 = a.scale_log2;
    bool ok = true;
    // parity of the next phase of tile_ready[b][t] is bit 16 * b + t (a
    // pass-2 warp waits only on the tiles of its parity, each use of them)
    uint32_t tph = 0;
    for (int step = 0; step < n_steps; ++step) {
      for (int pass = 0; pass < 2; ++pass) {
        const int it = pass == 0 ? step : step - lag;
        if (it < 0 || it >= n_my) continue;
        const int item = blockIdx.x + it * G;
        const ItemPos ip = decode_item(a, item);
        const SeqDesc sd = a.seqs[ip.s];
        const int tok0 = ip.c * a.chunk_tokens;
        const int ntiles = (min(a.chunk_tokens, sd.len - tok0) + kTileM - 1) / kTileM;
        const int prefix = sd.len - W;
        const int pb = it & 1;                     // statistics buffers of this item
        const uint32_t buf_addr = lane_addr + (uint32_t)(pass * kBufCols);
        if (pass == 0) {
          // ---- pass 1: per-row softmax statistics of this warp's tokens, as
          // in the one-pass kernel (a warp-wide reference per row that moves
          // only when a logit exceeds it by more than 32), nothing stored.
          float mref[NH], zsum[NH];
#pragma unroll
          for (int i = 0; i < NH; ++i) {
            mref[i] = -INFINITY;
            zsum[i] = 0.f;
          }
          float ymin = INFINITY;
          bool bad = false, fresh = true;
          for (int t = 0; t < ntiles; ++t) {
            const uint32_t tbit = 1u << t;
            if (ok)
              ok = __all_sync(0xffffffffu,
                              mbar_wait(smem_u32(&ms->tile_ready[0][t]), (tph & tbit) ? 1u : 0u,
                                        limit, abort_flag));
            tph ^= tbit;
            if (!ok) continue;
            tc_fence_after();
            const uint32_t taddr = buf_addr + (uint32_t)(t * NW + row0);
            const int tbase = tok0 + t * kTileM + 32 * quarter;
            const int tok = tbase + lane;
            if (tbase + 31 < prefix) {
              float y[NH];
              tmem_load_cols<NH>(taddr, y);
              if (fresh) {
#pragma unroll
                for (int i = 0; i < NH; ++i) mref[i] = __shfl_sync(0xffffffffu, y[i] * s2, 0);
                fresh = false;
              }
              bool need = false;
#pragma unroll
              for (int i = 0; i < NH; ++i) {
                y[i] = fmaf(y[i], s2, -mref[i]);
                need |= y[i] > 32.f;
              }
              if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int i = 0; i < NH; ++i) {
                  if (__any_sync(0xffffffffu, y[i] > 32.f)) {
                    const float xs = y[i] + mref[i];
                    if (!finite_f(xs)) bad = true;
                    const float mx = warp_max(xs);
                    zsum[i] *= ex2(mref[i] - mx);
                    mref[i] = mx;
                    y[i] = xs - mx;
                  }
                }
              }
#pragma unroll
              for (int i = 0; i < NH; ++i) {
                ymin = fminf(ymin, y[i]);
                zsum[i] += ex2(y[i]);
              }
            } else {
              const int lo = max(0, tok - prefix - row0);
              const int hi = tok < sd.len ? min(NH, W - row0) : 0;
#pragma unroll
              for (int cb = 0; cb < NH; cb += 8) {
                float xb[8];
                tmem_load_cols<8>(taddr + cb, xb);
                bool need = false;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  const int i = cb + u;
                  xb[u] *= s2;
                  if (i < hi && !finite_f(xb[u])) bad = true;
                  need |= i < hi && i >= lo && xb[u] > mref[i] + 32.f;
                }
                if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                  for (int u = 0; u < 8; ++u) {
                    const int i = cb + u;
                    const bool vis = i < hi && i >= lo;
                    if (__any_sync(0xffffffffu, vis && xb[u] > mref[i] + 32.f)) {
                      const float mx = warp_max(vis ? xb[u] : -INFINITY);
                      if (mref[i] != -INFINITY) zsum[i] *= ex2(mref[i] - mx);
                      mref[i] = mx;
                    }
                  }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  const int i = cb + u;
                  zsum[i] += (i < hi && i >= lo) ? ex2(xb[u] - mref[i]) : 0.f;
                }
              }
            }
          }
          // the logits are read: the buffer goes back to the MMA issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ms->tmem_empty[0]));
          // hand the chunk's statistics over (as in the one-pass kernel)
#pragma unroll
          for (int i = 0; i < NH; ++i)
            if (row0 + i < W && zsum[i] != zsum[i]) bad = true;
          if (ymin == -INFINITY) bad = true;
          if (bad) record_status(a.status, KVSEL_ERR_NONFINITE);
          reduce_sum<NH>(zsum, lane);
          constexpr int kLanesPerRow = 32 / NH;
          if (lane == 0) {
#pragma unroll
            for (int i = 0; i < NH; ++i) ms->wm[pb][quarter][row0 + i] = mref[i];
          }
          if (lane % kLanesPerRow == 0) ms->wz[pb][quarter][row0 + lane / kLanesPerRow] = zsum[0];
          epi_bar();
          if (warp == kEpiWarp0) {
            for (int r = lane; r < W; r += 32) {
              float m = ms->wm[pb][0][r], z = ms->wz[pb][0][r];
#pragma unroll
              for (int q = 1; q < 4; ++q) merge_stats(m, z, ms->wm[pb][q][r], ms->wz[pb][q][r]);
              if (m != m) m = INFINITY;
              if (!(a.inject == 1 && item == 0))
                slot_publish(reinterpret_cast<unsigned long long*>(a.part) +
                                 (int64_t)item * a.wpad + r, m, z);
            }
            if (lane == 0) *reinterpret_cast<volatile int*>(&ms->pub_items) = it + 1;
          }
        } else {
          // ---- pass 2: votes from the recomputed logits and the instance's
          // merged statistics F_r = M_r + log2 Z_r (+inf for padded rows, so
          // their terms vanish). This warp takes the tiles of parity `sub`,
          // all rows.
          const int64_t plane = ((int64_t)ip.layer * a.H + ip.h) * a.T + sd.tok_off;
          if (ok)
            ok = __all_sync(0xffffffffu,
                            mbar_wait(smem_u32(&ms->ffull[pb]), (uint32_t)(it >> 1) & 1, limit,
                                      abort_flag));
          const float* F = ms->fin[pb];
          for (int t = sub; t < ntiles; t += 2) {
            const uint32_t tbit = 1u << (16 + t);
            if (ok)
              ok = __all_sync(0xffffffffu,
                              mbar_wait(smem_u32(&ms->tile_ready[1][t]), (tph & tbit) ? 1u : 0u,
                                        limit, abort_flag));
            tph ^= tbit;
            if (!ok) continue;
            tc_fence_after();
            const int tok = tok0 + t * kTileM + 32 * quarter + lane;
            float x[NW];
            tmem_load_row<NW>(buf_addr + (uint32_t)(t * NW), x);
            float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < NW; i += 4) {
              const float4 f4 = *reinterpret_cast<const float4*>(F + i);
              p[0] += ex2(fmaf(x[i], s2, -f4.x));
              p[1] += ex2(fmaf(x[i + 1], s2, -f4.y));
              p[2] += ex2(fmaf(x[i + 2], s2, -f4.z));
              p[3] += ex2(fmaf(x[i + 3], s2, -f4.w));
            }
            if (tok < sd.len)
              a.votes[plane + tok] = tok < prefix ? (p[0] + p[1]) + (p[2] + p[3]) : 0.f;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ms->tmem_empty[1]));
          mbar_arrive(smem_u32(&ms->fempty[pb]));
        }
        if (!ok) *abort_flag = 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (ms->abort_flag) {
    if (warp == 0 && lane == 0) {
      for (int s = 0; s < kMaxStages; ++s)
        if (armed & (1u << s))
          mbar_wait(smem_u32(&ms->full[s]), (armed_par >> s) & 1, limit, nullptr);
      for (int b = 0; b < 2; ++b)
        if (q_armed & (1u << b))
          mbar_wait(smem_u32(&ms->qfull[b]), (q_par >> b) & 1, limit, nullptr);
    }
    if (warp == kMmaWarp && lane == 0 && mma_issued) {
      tc_commit(smem_u32(&ms->mma_done));
      mbar_wait(smem_u32(&ms->mma_done), 0, limit, nullptr);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// K as (D, H, rows): box of 64 elements x 1 head x 128 tokens.
bool make_kmap(CUtensorMap* m, const void* base, int D, int H, int64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kTileM};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// q_win as (D, H, W, layers * S): a box of qg heads x NW / qg window rows
// (row w * qg + g of the tile is row w of head g) reads rows W .. NW/qg - 1 as
// zeros (outside the tensor), so padded rows never see another sequence's
// queries.
bool make_qmap(CUtensorMap* m, const void* base, int D, int H, int W, int64_t seqs, int nw,
               int qg) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)W, (cuuint64_t)seqs};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)W * H * D * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)qg, (cuuint32_t)(nw / qg), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int NW, int KD, bool LOGITS, bool RC = false>
cudaError_t launch_t(const ScoreArgs& a, int grid) {
  constexpr int kStageBytes = kTileM * KD * 2;
  constexpr int kQBytes = NW * KD * 2;
  const size_t fixed = 1024 + 2 * kQBytes + sizeof(Misc) + slot_stage_for(NW);
  int stages = (int)((kSmemLimit - fixed) / kStageBytes);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + (size_t)stages * kStageBytes;
  TcParams p;
  std::memset(&p, 0, sizeof(p));
  if (!make_kmap(&p.tmk, a.k, a.D, a.H / a.kv_group, (int64_t)a.layers * a.T) ||
      !make_qmap(&p.tmq, a.q, a.D, a.H * a.qg, a.q_W, (int64_t)a.layers * (a.q_rows / a.q_W), NW,
                 a.qg))
    return cudaErrorInvalidValue;
  p.a = a;
  p.stages = stages;
  p.n_items = a.layers * a.items_per_layer;
  void (*kern)(const TcParams) = RC ? tc_score_rc_kernel<NW, KD> : tc_score_kernel<NW, KD, LOGITS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
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
  const int nw = tc_window_pad(a.W * a.qg);
  if (a.qg > 1 && (a.two_pass || LOGITS || nw % a.qg)) return cudaErrorInvalidValue;
  if (a.two_pass) {  // long instances: statistics and votes in two passes, never logits
    if (LOGITS || a.two_pass < 2) return cudaErrorInvalidValue;
    if (a.D == 128) {
      if (nw == 16) return launch_t<16, 128, false, true>(a, grid);
      if (nw == 32) return launch_t<32, 128, false, true>(a, grid);
      if (nw == 64) return launch_t<64, 128, false, true>(a, grid);
    } else if (a.D == 64) {
      if (nw == 16) return launch_t<16, 64, false, true>(a, grid);
      if (nw == 32) return launch_t<32, 64, false, true>(a, grid);
      if (nw == 64) return launch_t<64, 64, false, true>(a, grid);
    }
    return cudaErrorInvalidValue;
  }
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
  return tc_window_pad(W) ? std::min(2 * tc_max_grid(sm_count), kMaxChunks) : 0;
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
