// Host-side plumbing shared by the libkvsel translation units: the per-call
// descriptors handed to each kernel's launch wrapper. No device code here.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kvsel.h"

namespace kvsel {

// One sequence as the kernels see it (copied to device memory per call).
struct SeqDesc {
  int64_t tok_off;    // first token of the sequence within a layer
  int32_t len;        // L_b
  int32_t out_off;    // first output row within a layer: sum_{b'<b} min(L_b', C)
  int32_t n_chunks;   // scoring work items per head (0: not scored)
  int32_t item_base;  // first scoring work item of this sequence within a layer
  int32_t inst_base;  // instance id of (this sequence, head 0) within a layer
  int32_t index;      // position of the sequence in the call (row block of q_win)
};
static_assert(sizeof(SeqDesc) == 32, "SeqDesc layout");

// Scoring: window logits -> causal softmax row statistics -> votes.
// Work item = (layer, scored sequence, head, chunk of chunk_tokens tokens);
// instance = (layer, scored sequence, head).
struct ScoreArgs {
  const void* q;           // q_win
  const void* k;           // K
  int layers, H, D, dtype, W;
  int kv_group;            // query heads per K head: K head of query head h is h / kv_group
  int qg;                  // query heads scored together against one K head (tensor-core
                           // one-pass kernel, group-shared selection): instance head h
                           // takes query heads h * qg .. h * qg + qg - 1 as qg * W window
                           // rows (row w * qg + g); 1 otherwise
  int64_t T;               // tokens per layer
  int64_t q_rows;          // rows of q_win per layer (num_seqs * q_W)
  int q_W;                 // window rows per sequence in q_win (= W)
  int two_pass;            // > 0: the two-pass kernel for long instances (statistics,
                           // then votes from recomputed logits this many items later)
  int n_scored;            // number of scored sequences
  const SeqDesc* seqs;     // device: the scored sequences, in order
  int items_per_layer, inst_per_layer;
  int chunk_tokens;
  int wpad;                // row stride of part / final_stats (>= W)
  float scale_log2;        // log2(e) / sqrt(D): logits in base-2 units
  float scale;             // 1 / sqrt(D): logits as the page defines them
  float* part;             // [items][Wp][2] chunk (max, sum) in base-2 units
  float* final_stats;      // [instances][Wp] max + log2(sum) per window row (CUDA-core
                           // path); [instances][Wp][2] final (max, sum) slots (tensor cores)
  float* votes;            // [layers][H][T]
  float* logits;           // [layers][H][W][T] (logits mode only)
  int* status;             // device status word
  unsigned long long wait_limit_ns;
  int inject;              // test hook (see kvsel_debug_inject)
  int sm_count;
  cudaStream_t stream;
};

struct PoolArgs {
  const float* votes;      // [layers][H][T]
  float* pooled;           // [layers][H][T]
  int layers, H, W, pool_kind, pool_k;
  int64_t T;
  int n_seqs;
  const SeqDesc* seqs;     // every sequence (pooled is computed where L >= W)
  cudaStream_t stream;
};

struct SelectArgs {
  const float* scores;     // pooled, or votes when pool_inline
  int pool_inline, pool_kind, pool_k;
  int layers, H, W, C;
  int64_t T, T_out;
  int n_seqs;
  const SeqDesc* seqs;     // every sequence
  int32_t* out_idx;
  int* status;
  int sm_count;
  int64_t max_prefix;      // largest L - W over the selected sequences
  int cluster;             // CTAs per instance (set by the launcher)
  int slice;               // prefix positions per CTA (set by the launcher)
  int stage_bytes;         // shared bytes before the sort buffer (set by the launcher)
  int gather;              // 1: also copy the kept K/V rows (fused path)
  int vote_group;          // score planes summed per instance: head h takes planes
                           // h * vote_group .. + vote_group - 1 of H * vote_group
  int kv_H, kv_div;        // gather: K/V have kv_H heads; instance head h reads h / kv_div
  const void* k;           // gather: K, V and the compacted outputs
  const void* v;
  void* out_k;
  void* out_v;
  int64_t row_bytes;       // gather: D * element bytes
  int vec_bytes;           // gather: copy width (set by the launcher)
  const int32_t* pack;     // null: one instance per cluster in instance order; else the
                           // packing above, n_clusters clusters
  int n_clusters;
  int pdl;                 // 1: launched as a programmatic dependent of the preceding
                           // kernel on the stream (its CTAs wait for that grid's memory)
  int* sched;              // one-CTA instances with the gather: kSchedWords ints zeroed
                           // before the launch (null: no stagger)
  unsigned long long stagger_limit_ns;  // longest hold-back of an SM's second CTA
  cudaStream_t stream;
};

// Selection stagger words: a spare word, then per SM (%smid modulo kSchedSms)
// the number of CTAs that have started there and a "first selection done" flag.
constexpr int kSchedSms = 1024;
constexpr int kSchedWords = 1 + 2 * kSchedSms;

struct CompactArgs {
  const void* k;
  const void* v;
  const int32_t* idx;
  void* out_k;
  void* out_v;
  int layers, H, S, C;
  int64_t T, T_out;
  int64_t row_bytes;
  const SeqDesc* seqs;     // every sequence
  int64_t max_rows;        // max over sequences of min(L, C) * H
  int kv_H, kv_div;        // K/V have kv_H heads; output head h reads h / kv_div
  int* status;
  int sm_count;
  cudaStream_t stream;
};

// Decode-side attention: one query per (layer, sequence, query head) over the
// sequence's cache rows, then its g appended rows. Work item = (layer,
// sequence, query head, chunk of chunk_rows rows).
struct DecSeq {
  int64_t row_off;         // first cache row of the sequence within a layer
  int32_t n_rows;          // cache rows (the appended ones come after)
  int32_t n_chunks;        // chunks per query head
  int32_t item_base;       // first work item of (this sequence, head 0) within a layer
  int32_t index;           // sequence number (q row block, appended row block)
};

struct DecodeArgs {
  const void* q;           // [layers][S][H][D]
  const void* k;           // cache [layers][T][Hkv][D]
  const void* v;
  const void* k_new;       // appended [layers][S * g][Hkv][D] (g > 0)
  const void* v_new;
  int layers, S, H, Hkv, D, dtype, g;
  int64_t T;               // cache rows per layer
  const DecSeq* seqs;      // device: every sequence, in order
  int items_per_layer;
  int chunk_rows;
  float scale_log2;        // log2(e) / sqrt(D)
  float* part;             // [items][2 + D]: base-2 max, sum, weighted values
  float* out;              // [layers][S][H][D]
  float* lse;              // [layers][S][H] natural log, or null
  int* status;
  cudaStream_t stream;
};

struct QualityArgs {
  int64_t n;               // instances
  int D;
  const float* lse_keep;
  const float* lse_full;
  const float* out_keep;
  const float* out_full;
  float* mass;             // exp(lse_keep - lse_full)
  float* err;              // ||out_full - out_keep||_2
  cudaStream_t stream;
};

// Jacap scoring (leverage of the value directions under the capacity matrix).
// Instance = (layer, scored sequence, head); its pool is the prefix 0 .. P-1.
struct JSeq {
  int64_t tok_off;         // first token of the sequence within a layer
  int32_t len;             // L
  int32_t index;           // sequence number in the call (q_win row block)
  int32_t inst_base;       // instance id of (sequence, head 0) within a layer
  int32_t pad;
};

// One piece of Gram work: tiles [t_begin, t_end) (kJTile tokens each) of one
// instance. The Gram CTAs split the instances' tiles, in instance order, into
// equal contiguous ranges; a range cut at instance boundaries gives the
// pieces, numbered in that order, and piece s writes partial matrix s.
struct JSeg {
  int32_t inst;            // layer * inst_per_layer + instance id within the layer
  int32_t t_begin, t_end;
  int32_t pad;
};

struct JacapArgs {
  const void* q;           // q_win [layers][S * W][H][D] bf16
  const void* k;           // [layers][T][H][D] bf16
  const void* v;
  int layers, H, D, W, S;  // S: sequences in the call (q_win blocks)
  int64_t T;
  int n_scored;
  const JSeq* seqs;        // device: the scored sequences
  int inst_per_layer;
  int n_gram;              // Gram CTAs
  const JSeg* segs;        // device: the pieces
  const int32_t* cta_seg;  // device, n_gram + 1: CTA c takes pieces cta_seg[c] .. cta_seg[c+1]-1
  const int32_t* inst_seg; // device, instances + 1: instance i's pieces (its partials, in order)
  float tau, beta, eps;
  float2* zk;              // [layers][H][T]: (z in base-2 units, kappa) per prefix token
  float* part;             // [pieces][2]: base-2 max and sum of 2^z over the piece's tokens
  float* gram;             // [pieces][D][D] partial sums of w v v^T
  float* wts;              // [layers][H][T]: w per prefix token
  void* linv;              // [instances][2][D][D] bf16: L^{-1} split into hi + lo
  float* scores;           // [layers][H][T]: r per prefix token
  int* status;
  unsigned long long wait_limit_ns;
  cudaStream_t stream;
};

constexpr int kJGramMinTiles = 8;    // fewest tiles per Gram CTA (below that, fewer CTAs)

constexpr int kMaxSelect = 16384;    // largest C - W the select kernel sorts on chip
constexpr int64_t kMaxPrefix = 262144;  // longest prefix L - W the select kernel takes
constexpr int kSelSliceCap = 16384;  // prefix positions one selection CTA holds
constexpr int kSelMaxCluster = 8;    // selection CTAs per cluster (portable size)

// Selection geometry: CTAs per cluster and prefix positions per CTA for the
// longest selected prefix.
inline void select_geometry(int64_t max_prefix, int* cs, int* slice) {
  int c = (int)((max_prefix + kSelSliceCap - 1) / kSelSliceCap);
  if (c < 1) c = 1;
  int sl = (int)((max_prefix + c - 1) / c);
  *cs = c;
  *slice = sl < 1 ? 1 : sl;
}

// Selection packing of ragged batches (launches of clusters of cs > 1 CTAs):
// an instance whose prefix fits one CTA's slice (or that keeps everything)
// runs on a single CTA, so cs of them share a cluster; longer instances take
// a whole cluster. pack[c * kSelMaxCluster + r] for cluster c: either the
// instance at r = 0 and kPackWhole at r = 1, or the instance of CTA rank r
// (-1: that CTA has none).
constexpr int kPackWhole = -2;
constexpr int kGenericChunk = 256;   // tokens per CUDA-core scoring block
constexpr int kGenericMaxQ = 16384;  // W * D floats staged in shared memory

// Launch wrappers (each defined beside its kernels).
cudaError_t launch_generic_score(const ScoreArgs& a, bool logits_mode);
cudaError_t launch_pool(const PoolArgs& a);
cudaError_t launch_select(const SelectArgs& a);
cudaError_t launch_compact(const CompactArgs& a);
cudaError_t launch_decode(const DecodeArgs& a);
cudaError_t launch_jacap(const JacapArgs& a);
bool jacap_eligible(int dtype, int D, const void* q, const void* k, const void* v);

// Reverse-mask attention (counter-causal scorer): every cached row attends to
// the rows of its sequence at later original positions only. One work item =
// 128 query rows of one (layer, sequence, query head).
struct RevSeq {
  int64_t tok_off;         // first row of the sequence within a layer
  int32_t len;             // rows n
  int32_t n_qt;            // query tiles ceil(n / 128)
  int32_t item_base;       // first item of the sequence within a layer (items qt * H + h)
  int32_t pad;
};

struct RevArgs {
  const void* q;           // [layers][T][H][D] bf16
  const void* k;           // [layers][T][H_kv][D] bf16
  const void* v;
  const int32_t* pos;      // [T] sequence-relative original positions, or null (= row order)
  float* out;              // [layers][T][H][D]
  float* lse;              // [layers][H][T] natural log, or null
  int layers, H, Hkv, S;
  int64_t T;
  const RevSeq* seqs;      // device
  int items_per_layer;
  int* status;
  unsigned long long wait_limit_ns;
  cudaStream_t stream;
};

cudaError_t launch_reverse(const RevArgs& a);
bool reverse_eligible(int dtype, int D, const void* q, const void* k, const void* v);
cudaError_t launch_decode_quality(const QualityArgs& a);
int decode_chunk_rows();
bool decode_supported(int dtype, int D);

// Tensor-core path.
int tc_window_pad(int W);                       // padded MMA N for W, 0 if unsupported
int tc_chunk_tokens(int W);                     // tokens per CTA work item
bool tc_eligible(int dtype, int D, int W, const void* q, const void* k);
cudaError_t launch_tc_score(const ScoreArgs& a, bool logits_mode, int grid);
int tc_max_grid(int sm_count);                  // co-resident CTAs (one per SM)
int tc_max_chunks(int W, int sm_count);         // most chunks one instance may have

}  // namespace kvsel
