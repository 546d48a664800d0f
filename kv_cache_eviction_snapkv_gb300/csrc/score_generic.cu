// CUDA-core scoring path: window logits, causal-softmax row statistics and
// votes for any dtype / head dim / window the tensor-core kernel does not take
// (fp32 inputs, head dims other than 64 and 128, W > 64).
//
// Method: page "SnapKV: choosing the KV cache of a long prompt with an
// observation window", section "Votes must come from the full-prompt causal
// softmax" (投票必须来自完整提示词的因果 softmax): row r of a sequence is window
// query t = P + r; it sees keys j <= t; its softmax denominator runs over every
// visible key; a prefix key's vote is the sum of its probabilities over rows.
//
// Three launches (K is read twice; this path is not the bandwidth-critical
// one): per 256-token chunk, each row's (max, sum of 2^(x - max)) in base-2
// units; per instance, the merge max M and M + log2(sum); per chunk, the votes
// sum_r 2^(x_r - M_r - log2 Z_r). A fourth mode writes raw logits.
#include "kvsel_device.cuh"

#include <cfloat>

namespace kvsel {
namespace {

constexpr int kThreads = kGenericChunk;
constexpr int kWarps = kThreads / 32;

enum Mode { kStats = 0, kVotes = 1, kLogits = 2 };

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) generic_score_kernel(ScoreArgs a) {
  extern __shared__ float qs[];          // [W][D] window queries as fp32
  __shared__ float red[kWarps];
  __shared__ float bcast;

  const ItemPos ip = decode_item(a, blockIdx.x);
  const SeqDesc sd = a.seqs[ip.s];
  const int W = a.W, D = a.D, H = a.H;
  const int prefix = sd.len - W;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Stage this (layer, sequence, head)'s W window queries.
  const int64_t q_row0 = (int64_t)ip.layer * a.q_rows + (int64_t)sd.index * a.q_W;
  for (int e = tid; e < W * D; e += kThreads) {
    int r = e / D, d = e - r * D;
    qs[e] = load_elem(a.q, ((q_row0 + r) * H + ip.h) * D + d, a.dtype);
  }
  __syncthreads();

  const int tok = ip.c * a.chunk_tokens + tid;         // position within the sequence
  const bool valid = tok < sd.len;
  const int64_t krow =
      (((int64_t)ip.layer * a.T + sd.tok_off + tok) * (H / a.kv_group) + ip.h / a.kv_group) *
      (int64_t)D;
  const int64_t head_plane = (int64_t)ip.layer * H + ip.h;

  float vote = 0.f;
  bool bad = false;
  for (int r = 0; r < W; ++r) {
    float dot = 0.f;
    if (valid) {
      const float* qr = qs + r * D;
      for (int d = 0; d < D; ++d) dot = fmaf(qr[d], load_elem(a.k, krow + d, a.dtype), dot);
    }
    if (MODE == kLogits) {
      if (valid)
        a.logits[(head_plane * W + r) * a.T + sd.tok_off + tok] = dot * a.scale;
      continue;
    }
    const float x = dot * a.scale_log2;
    const bool vis = valid && tok <= prefix + r;
    if (MODE == kStats) {
      if (valid && !finite_f(x)) bad = true;
      // chunk max of the visible logits
      float m = warp_max(vis ? x : -INFINITY);
      if (lane == 0) red[warp] = m;
      __syncthreads();
      if (tid < 32) {
        float v = lane < kWarps ? red[lane] : -INFINITY;
        v = warp_max(v);
        if (lane == 0) bcast = v;
      }
      __syncthreads();
      m = bcast;
      float e = vis ? ex2(x - m) : 0.f;
      e = warp_sum(e);
      __syncthreads();
      if (lane == 0) red[warp] = e;
      __syncthreads();
      if (tid < 32) {
        float v = lane < kWarps ? red[lane] : 0.f;
        v = warp_sum(v);
        if (lane == 0) {
          float* pp = a.part + ((int64_t)blockIdx.x * a.wpad + r) * 2;
          pp[0] = m;
          pp[1] = v;
        }
      }
      __syncthreads();
    } else {  // kVotes
      if (vis && tok < prefix)
        vote += ex2(x - a.final_stats[(int64_t)ip.inst * a.wpad + r]);
    }
  }
  if (MODE == kStats && bad) record_status(a.status, KVSEL_ERR_NONFINITE);
  if (MODE == kVotes && valid)
    a.votes[head_plane * a.T + sd.tok_off + tok] = tok < prefix ? vote : 0.f;
}

// One block per instance: merge the chunk statistics of each window row.
__global__ void __launch_bounds__(128) generic_merge_kernel(ScoreArgs a) {
  const int inst = blockIdx.x;
  const int layer = inst / a.inst_per_layer;
  const int local = inst - layer * a.inst_per_layer;
  const SeqDesc* sq = a.seqs;
  const int s = upper_find(a.n_scored, local, [&](int i) { return sq[i].inst_base; });
  const int h = local - sq[s].inst_base;
  const int nc = sq[s].n_chunks;
  const int64_t item0 = (int64_t)layer * a.items_per_layer + sq[s].item_base + (int64_t)h * nc;
  for (int r = threadIdx.x; r < a.W; r += blockDim.x) {
    float M = -INFINITY;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, a.part[((item0 + c) * a.wpad + r) * 2]);
    float Z = 0.f;
    for (int c = 0; c < nc; ++c) {
      const float* pp = a.part + ((item0 + c) * a.wpad + r) * 2;
      Z += pp[1] * ex2(pp[0] - M);
    }
    a.final_stats[(int64_t)inst * a.wpad + r] = M + log2f(Z);
  }
}

}  // namespace

cudaError_t launch_generic_score(const ScoreArgs& a, bool logits_mode) {
  const int items = a.layers * a.items_per_layer;
  if (items == 0) return cudaSuccess;
  const size_t smem = (size_t)a.W * a.D * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(generic_score_kernel<kStats>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
      return e;
    if ((e = cudaFuncSetAttribute(generic_score_kernel<kVotes>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
      return e;
    if ((e = cudaFuncSetAttribute(generic_score_kernel<kLogits>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
      return e;
  }
  if (logits_mode) {
    generic_score_kernel<kLogits><<<items, kThreads, smem, a.stream>>>(a);
    return cudaGetLastError();
  }
  generic_score_kernel<kStats><<<items, kThreads, smem, a.stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e) return e;
  generic_merge_kernel<<<a.layers * a.inst_per_layer, 128, 0, a.stream>>>(a);
  if ((e = cudaGetLastError())) return e;
  generic_score_kernel<kVotes><<<items, kThreads, smem, a.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvsel
