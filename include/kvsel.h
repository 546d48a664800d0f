/*
 * kvsel.h — C ABI of libkvsel, GB300 (sm_103a) SnapKV observation-window
 * KV-cache selection.
 *
 * Method: page "SnapKV: choosing the KV cache of a long prompt with an
 * observation window" (SnapKV：用观察窗口为长提示词选择 KV Cache,
 * charlestar.github.io, 2026-10-20). For every (layer, sequence, head):
 *   - partition ("要缩小的是提示词缓存" section): prompt length L, window = the
 *     last W tokens, prefix P = L - W, budget C keeps the whole window plus
 *     C - W prefix positions;
 *   - votes ("投票必须来自完整提示词的因果 softmax" section): the W window
 *     queries attend to all L keys with scale 1/sqrt(D) under a causal mask,
 *     the softmax denominator runs over every visible position, and each
 *     prefix position's vote is the sum of its probabilities over the W rows;
 *   - pooling and top-k ("池化把一个峰值扩展成邻域偏好" section): 1-D pooling
 *     of the prefix votes (odd width, stride 1, zero padding; the average
 *     divides by the full width at the edges; or max), then the C - W prefix
 *     positions with the highest pooled score, ties to the smaller position;
 *   - gather ("从 Q 和 K 开始算一次完整选择" section): the kept positions of
 *     K and V with one index list; L < C keeps everything (bypass).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Data layout (row-major, no padding, "layers" outermost):
 *   q_win   [num_layers][num_seqs * W][H][D]  window queries; rows b*W .. b*W+W-1
 *                                             are sequence b's positions P_b .. L_b-1
 *   K, V    [num_layers][T][H][D]             packed prompts (RoPE already applied);
 *                                             sequence b owns tokens
 *                                             seq_offsets[b] .. seq_offsets[b+1]-1
 *   votes, pooled [num_layers][H][T] fp32     entry j of sequence b's token range holds
 *                                             prefix position j's score (j < P_b); window
 *                                             positions hold 0
 *   out_idx [num_layers][T_out][H] int32      positions within the sequence
 *   out_K, out_V [num_layers][T_out][H][D]    same dtype as K and V
 * with T = seq_offsets[num_seqs] and T_out = kvsel_out_tokens(shape, C)
 * = sum_b min(L_b, C); sequence b's output rows start at sum_{b'<b} min(L_b', C).
 * Within a sequence's C output rows: the C - W kept prefix positions in the
 * order (highest pooled score first, equal scores by smaller position), then
 * the window positions P..L-1 ascending. A sequence with L < C (bypass) keeps
 * positions 0..L-1 in order.
 *
 * Memory: every data pointer is device memory allocated by the caller, except
 * shape->seq_offsets, which is HOST memory (it decides launch shapes and which
 * sequences bypass). The library never frees caller memory.
 *
 * Streams and synchronisation: `stream` is a cudaStream_t (NULL = legacy
 * default stream). Calls enqueue work and return without waiting for it.
 * kvsel_score, kvsel_window_logits and kvsel_snapkv use an internal per-device
 * workspace that the library allocates with cudaMalloc and grows on demand
 * (growing synchronises the device); kvsel_release() frees it. Calls that use
 * the workspace on one device must be ordered with one another (one stream,
 * or events between streams): overlapping calls race on it.
 *
 * Errors: arguments are checked on the host before any launch; a rejected
 * call launches nothing. Conditions only the GPU can see (a non-finite window
 * logit, a gather index out of range, a bounded wait that ran out) are
 * recorded in a per-device status word; kvsel_device_status() reads it.
 * Every launch failure returns KVSEL_ERR_CUDA.
 */
#ifndef KVSEL_H_
#define KVSEL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t kvsel_status;
enum {
  KVSEL_OK = 0,
  KVSEL_ERR_INVALID_ARG = 1,  /* an argument rule failed (see each call) */
  KVSEL_ERR_UNSUPPORTED = 2,  /* valid, but beyond a documented limit */
  KVSEL_ERR_NONFINITE = 3,    /* device: a window logit was NaN or +-Inf */
  KVSEL_ERR_TIMEOUT = 4,      /* device: a bounded wait ran out */
  KVSEL_ERR_CUDA = 5,         /* a CUDA runtime call failed */
  KVSEL_ERR_BAD_INDEX = 6     /* device: a gather index was outside [0, L_b) */
};

enum { KVSEL_POOL_AVG = 0, KVSEL_POOL_MAX = 1 };
enum { KVSEL_BF16 = 0, KVSEL_F32 = 1 };

/* Shape of one call. num_layers >= 1 and num_heads >= 1 and head_dim >= 1;
 * num_seqs >= 0 (0 = nothing to do); dtype is KVSEL_BF16 or KVSEL_F32 (for
 * q_win, K, V and the gathered outputs). seq_offsets: HOST array of
 * num_seqs + 1 entries, seq_offsets[0] == 0, nondecreasing.
 * Grouped-query attention (page section "GQA 下的缓存节省不能只算 C 除以 L"):
 * num_heads counts the query heads H (q_win and every per-head output) and
 * num_kv_heads the heads H_kv of K and V: 0 (= num_heads) or a divisor of
 * num_heads (else INVALID_ARG). Query head h then reads K/V head
 * h / (H / H_kv), the expanded (repeat_kv) reading the page describes; the
 * group-shared selection is kvsel_snapkv_grouped. */
typedef struct kvsel_shape {
  int32_t num_layers;
  int32_t num_seqs;
  int32_t num_heads;
  int32_t head_dim;
  int32_t dtype;
  int32_t num_kv_heads; /* 0 = num_heads */
  const int64_t* seq_offsets;
} kvsel_shape;

/* Library version string (static storage). */
const char* kvsel_version(void);

/* Human-readable name of a status code (static storage). */
const char* kvsel_status_string(kvsel_status status);

/* T_out = sum_b min(L_b, C), the number of output rows per layer and head.
 * Returns -1 if the shape or C (< 1) is invalid. Host only, no GPU work. */
int64_t kvsel_out_tokens(const kvsel_shape* shape, int32_t C);

/* Which window-logit kernel a call with this shape takes: 1 = the tensor-core
 * kernel (TMA + tcgen05, bf16, D in {64,128}, W <= 64), 3 = the tensor-core
 * two-pass kernel (the same shapes, on sequences longer than 64 of the
 * kernel's work items: row statistics first, then the votes from logits
 * recomputed from K, which the second pass reads from L2), 0 = the CUDA-core
 * kernel (any other supported shape), -1 = the call would be rejected.
 * C = 0 means "score every sequence" (kvsel_score); otherwise sequences with
 * L < C are not scored. Host only; queries the current device. */
int32_t kvsel_score_path(const kvsel_shape* shape, int32_t W, int32_t C);

/* Window logits z[r][j] = q_{P_b + r} . k_j / sqrt(D) for every sequence b,
 * window row r < W and token j of b (no mask applied), written to
 * logits[num_layers][H][W][T] (fp32, row r of column j belongs to j's
 * sequence). Rules: W >= 1, W <= L_b for every b, non-null pointers when
 * T > 0. Same kernels as kvsel_score, stopped before the softmax; for tests
 * and diagnostics. */
kvsel_status kvsel_window_logits(const kvsel_shape* shape, const void* q_win, const void* K,
                                 int32_t W, float* logits, void* stream);

/* Votes and pooled scores of every sequence ("votes" and "pooling" sections).
 * votes (may be NULL) and pooled: [num_layers][H][T] fp32, prefix positions
 * filled, window positions 0. Rules: W >= 1, W <= L_b for every b, pool_kind
 * in {AVG, MAX}, pool_k odd and >= 1, non-null q_win/K/pooled when T > 0.
 * Device status: NONFINITE if a window logit (any window row, any token of
 * the sequence) is not finite. */
kvsel_status kvsel_score(const kvsel_shape* shape, const void* q_win, const void* K, int32_t W,
                         int32_t pool_kind, int32_t pool_k, float* votes, float* pooled,
                         void* stream);

/* kvsel_score without any device allocation, for callers that cannot call
 * cudaMalloc (an allocator they must not bypass, or a context where
 * allocating is not permitted). The paper has no counterpart; it is a
 * deployment variant of kvsel_score with the same arguments, rules and
 * results, except that votes must be non-NULL (the caller provides it).
 * Scratch: a fixed 8 MiB array in device memory, part of the library image
 * (every GPU that loads the library holds it until the process exits). The
 * first call on a device looks up that array's device address (once per
 * device, with the device current); make that first call before any stream
 * capture. Calls whose scratch need exceeds 8 MiB return
 * KVSEL_ERR_UNSUPPORTED and launch nothing; kvsel_score_static_bytes gives
 * the exact need of a call. All calls on a device share the array and each
 * call resets what must start out empty, so calls that overlap on the GPU
 * (different streams without ordering) race. */
kvsel_status kvsel_score_static(const kvsel_shape* shape, const void* q_win, const void* K,
                                int32_t W, int32_t pool_kind, int32_t pool_k, float* votes,
                                float* pooled, void* stream);

/* Scratch bytes kvsel_score_static needs for this shape, window and the
 * current device (the sequence tables, the cross-chunk statistics slots and
 * the merged statistics of the scoring kernel it would launch; q_win and K
 * are assumed 16-byte aligned), or -1 if the arguments break a rule of
 * kvsel_score. At most 8 MiB is accepted. Host only. */
int64_t kvsel_score_static_bytes(const kvsel_shape* shape, int32_t W);

/* Top-(C - W) selection from given pooled scores ([num_layers][H][T] fp32,
 * only prefix entries are read) into out_idx ([num_layers][T_out][H] int32);
 * bypass sequences (L < C) get 0..L-1. Ordering of scores: IEEE order with
 * -0 == +0; NaN ranks below every number and sets NONFINITE. Rules: W >= 1,
 * C > W, W <= L_b for every b. Limit: C - W <= 16384 (else UNSUPPORTED). */
kvsel_status kvsel_select(const kvsel_shape* shape, const float* pooled, int32_t W, int32_t C,
                          int32_t* out_idx, void* stream);

/* Gather: out_K[row] = K[idx], out_V[row] = V[idx] for every output row, the
 * same idx for K and V, with out_idx as produced by kvsel_select. Rules: C >= 1,
 * non-null pointers when T_out > 0. Device status: BAD_INDEX if an index is
 * outside [0, L_b) (that row is left unwritten). Bit-exact copy. */
kvsel_status kvsel_compact(const kvsel_shape* shape, const void* K, const void* V,
                           const int32_t* out_idx, int32_t C, void* out_K, void* out_V,
                           void* stream);

/* The whole path: score -> pool -> select -> gather, with no host
 * synchronisation in between. Rules: those of kvsel_score and kvsel_select
 * (W >= 1, C > W, W <= L_b for every b, odd pool_k >= 1, pool_kind valid,
 * C - W <= 16384). Sequences with L < C are copied unscored. */
kvsel_status kvsel_snapkv(const kvsel_shape* shape, const void* q_win, const void* K,
                          const void* V, int32_t W, int32_t C, int32_t pool_kind,
                          int32_t pool_k, int32_t* out_idx, void* out_K, void* out_V,
                          void* stream);

/* Group-shared selection under grouped-query attention: one selection per
 * (layer, sequence, K/V head), shared by the G = H / H_kv query heads of the
 * group, so the kept cache has H_kv heads (the page leaves this design open;
 * our reading): each query head computes its own causal-softmax votes against
 * the group's keys, the group's vote of a prefix position is the sum of its
 * G heads' votes, and pooling, the top-(C - W) selection and the gather then
 * run once per group. On the tensor cores with G a power of two and G * W <=
 * 64 the G heads are scored together (K read once per group; the sum is then
 * taken over all G * W rows at once, equal to the head-ordered sum within
 * fp32 rounding). Layouts: q_win [num_layers][S * W][H][D],
 * K and V [num_layers][T][H_kv][D]; out_idx [num_layers][T_out][H_kv] int32,
 * out_K and out_V [num_layers][T_out][H_kv][D]. Rules and limits those of
 * kvsel_snapkv. With H_kv == H it is kvsel_snapkv. */
kvsel_status kvsel_snapkv_grouped(const kvsel_shape* shape, const void* q_win, const void* K,
                                  const void* V, int32_t W, int32_t C, int32_t pool_kind,
                                  int32_t pool_k, int32_t* out_idx, void* out_K, void* out_V,
                                  void* stream);

/* kvsel_snapkv with the cache in host memory: q_win, K, V, out_idx, out_K and
 * out_V are HOST pointers with kvsel_snapkv's layouts. q_win and K are copied
 * to the device one layer at a time on an internal copy stream (two device
 * slots held by the library, so a layer's copy overlaps the previous layer's
 * kernels); V and the three outputs must be page-locked host memory
 * (cudaHostAlloc or cudaHostRegister): the gather reads the kept V rows and
 * writes the outputs in place, so of V only the kept rows cross the link.
 * Pinned q_win and K copy fastest. Asynchronous and ordered on `stream`: it
 * starts after the work already queued there, and the outputs are complete
 * when `stream` reaches the point after the call; the host buffers must stay
 * valid until then. Rules and limits those of kvsel_snapkv; INVALID_ARG also
 * when V or an output is not page-locked host memory. */
kvsel_status kvsel_snapkv_host(const kvsel_shape* shape, const void* q_win, const void* K,
                               const void* V, int32_t W, int32_t C, int32_t pool_kind,
                               int32_t pool_k, int32_t* out_idx, void* out_K, void* out_V,
                               void* stream);

/* ---------------------------------------------------------------------------
 * Jacap scorer (pages "Jacap reading notes" / "Jacap technical review",
 * section 6 (practical approximation) and section 7 (Algorithm 1): per (layer,
 * sequence, head), over the prefix pool 0 .. P-1 with P = L - W:
 * z_i = k_i . mu_Q / (tau sqrt(D)), alpha = softmax(z) over the pool,
 * kappa_i = k_i^T Lambda_Q k_i, w_i = [alpha_i (1 - alpha_i)]^2 kappa_i / D,
 * A = I + sum_i w_i v_i v_i^T, r_i = w_i v_i^T A^{-1} v_i (the value as the
 * output proxy); mu_Q and the diagonal Lambda_Q from the W window queries by
 * the running mean and second moment of section 11 (Algorithm 2) with rate
 * beta and floor eps, started from the first window query (our reading for a
 * prompt-time selection). Tensor-core path only: bf16, D = 128, num_kv_heads
 * equal to num_heads (UNSUPPORTED otherwise). Argument rules of kvsel_score /
 * kvsel_snapkv plus tau > 0 finite, 0 <= beta < 1, eps >= 0 finite
 * (INVALID_ARG). Device status: NONFINITE if a statistic or the capacity
 * matrix is not finite or not positive definite.
 * ------------------------------------------------------------------------- */

/* Scores r [num_layers][H][T] fp32 (caller owned): r at the prefix positions
 * of every sequence with L > W, 0 elsewhere. Layouts as kvsel_score. */
kvsel_status kvsel_jacap_score(const kvsel_shape* shape, const void* q_win, const void* K,
                               const void* V, int32_t W, float tau, float beta, float eps,
                               float* scores, void* stream);

/* The whole Jacap path: scores, the top C - W prefix positions by (-r, j) (the
 * selection of kvsel_select, no pooling), then the window, and the gather of
 * the kept K and V rows; sequences with L < C are copied unscored. Outputs as
 * kvsel_snapkv. */
kvsel_status kvsel_jacap(const kvsel_shape* shape, const void* q_win, const void* K,
                         const void* V, int32_t W, int32_t C, float tau, float beta, float eps,
                         int32_t* out_idx, void* out_K, void* out_V, void* stream);

/* ---------------------------------------------------------------------------
 * Decode-side consumer of a cache (page section "Why deleting positions
 * changes the output" (删除位置为什么会改变输出): one future query, its softmax
 * over the cache rows, the value sum, and the probability mass the full cache
 * gives the kept rows; section "The current prefill still reads the full K/V"
 * (当前 prefill 仍读完整 K/V，压缩缓存服务后续 decode): after g generated
 * tokens the cache holds min(L, C) + g rows; section "Cache slots cannot
 * stand in for the original RoPE positions" (缓存槽位不能代替 RoPE 的原始位置):
 * the next token's logical position is L + g, its physical slot min(L, C) + g).
 * ------------------------------------------------------------------------- */

/* One query per (layer, sequence, query head) attends, unmasked, to every row
 * of its sequence's cache followed by its g appended rows, with the scale
 * 1/sqrt(D). `shape` describes the cache: seq_offsets are cache row offsets
 * (for a compacted cache from kvsel_snapkv the running sum of min(L_b, C);
 * for the full cache the prompt offsets), num_heads the query heads H,
 * num_kv_heads (0 = H) the cache heads; query head h reads cache head
 * h / (H / H_kv). Layouts (dtype of the shape, rows of D elements, 16-byte
 * aligned): q [num_layers][num_seqs][H][D]; K, V [num_layers][T][H_kv][D];
 * K_new, V_new [num_layers][num_seqs * g][H_kv][D] (sequence b's appended rows
 * at b*g .. b*g + g - 1; may be NULL when g == 0). Outputs (fp32, caller
 * owned, device memory): out [num_layers][num_seqs][H][D] the attention
 * output; lse [num_layers][num_seqs][H] the natural log of the sum of
 * exp(q . k / sqrt(D)) over the attended rows, or NULL. Permuting a
 * sequence's cache rows (K and V together) does not change the result, so
 * kvsel_snapkv's score-ordered rows can be read as they are. Rules:
 * INVALID_ARG for g < 0, a sequence with no rows at all (cache + g == 0),
 * NULL or misaligned pointers; UNSUPPORTED for D not in {64, 128}. Device
 * status: NONFINITE if a sum or an output is not finite. Asynchronous. */
kvsel_status kvsel_decode_attention(const kvsel_shape* shape, const void* q, const void* K,
                                    const void* V, int32_t g, const void* K_new,
                                    const void* V_new, float* out, float* lse, void* stream);

/* ---------------------------------------------------------------------------
 * Reverse-mask attention of the counter-causal scorer (page "来自未来的信号：
 * 用反因果惊奇度做 KV Cache 淘汰" (signals from the future: KV-cache eviction by
 * counter-causal surprise), section 3.2, steps 1, 3 and 5; section 4,
 * Algorithm 3). The part that needs no model weights: every cached row i of
 * a sequence attends, with the scale 1/sqrt(D), to the cached rows j of the
 * same sequence whose original position is larger than its own (a strictly
 * upper-triangular mask in position order), reusing the cached K and V with
 * queries recomputed at the original positions.
 * ------------------------------------------------------------------------- */

/* out_i = sum_{j: pos_j > pos_i} softmax_j(q_i . k_j / sqrt(D)) v_j and lse_i
 * = ln sum_j exp(q_i . k_j / sqrt(D)) over the same j; a row with no such j
 * (the last position) gets out = 0 and lse = -inf (the page gives it the
 * largest surprise). `shape`: seq_offsets are the cache rows of each sequence,
 * num_heads the query heads H, num_kv_heads (0 = H) the cache heads; query head
 * h reads cache head h / (H / H_kv). Layouts (bf16, D = 128, rows 16-byte
 * aligned): Q [num_layers][T][H][D]; K, V [num_layers][T][H_kv][D];
 * positions [T] int32, the sequence-relative original position of each row
 * (NULL: the row order; a refresh that reorders the memory passes them; equal
 * positions do not attend to each other). Outputs (fp32, caller-owned device
 * memory): out [num_layers][T][H][D] (16-byte aligned); lse
 * [num_layers][H][T] natural log, or NULL. Rules: INVALID_ARG for NULL or
 * misaligned pointers; UNSUPPORTED for a dtype other than bf16, D != 128,
 * misaligned Q/K/V, or num_layers * T >= 2^31. Device status: NONFINITE if a
 * row's max or sum is not finite; TIMEOUT if a bounded wait ran out.
 * Asynchronous on `stream`. */
kvsel_status kvsel_reverse_attention(const kvsel_shape* shape, const void* Q, const void* K,
                                     const void* V, const int32_t* positions, float* out,
                                     float* lse, void* stream);

/* Per instance (n of them, e.g. layers * seqs * heads): the retained mass
 * mass[i] = exp(lse_keep[i] - lse_full[i]) (the full-cache probability of the
 * rows that the compacted cache kept, when lse_keep comes from the compacted
 * cache and lse_full from the full one, both with the same appended rows) and
 * err[i] = || out_full[i] - out_keep[i] ||_2 over the D values. All device
 * pointers, fp32. INVALID_ARG for n < 0, D < 1 or NULL pointers (n > 0). */
kvsel_status kvsel_decode_quality(int64_t n, int32_t D, const float* lse_keep,
                                  const float* lse_full, const float* out_keep,
                                  const float* out_full, float* mass, float* err, void* stream);

/* Host bookkeeping for a prompt shape (seq_offsets = prompt offsets), budget
 * C and g appended tokens per sequence: physical_length[b] = min(L_b, C) + g
 * (also the slot the next token is written to) and next_logical[b] = L_b + g
 * (its position for RoPE). Host arrays of num_seqs entries. INVALID_ARG for
 * C < 1, g < 0 or NULL arrays (num_seqs > 0). */
kvsel_status kvsel_cache_lengths(const kvsel_shape* shape, int32_t C, int32_t g,
                                 int64_t* physical_length, int64_t* next_logical);

/* Synchronises `stream`, then returns and clears the current device's status
 * word: the first device-side error recorded since the last call, or
 * KVSEL_OK. Returns KVSEL_ERR_CUDA if the synchronisation itself failed. */
kvsel_status kvsel_device_status(void* stream);

/* Upper bound, in nanoseconds, on every spin-wait inside the kernels (default
 * 2e9). A wait that runs out records KVSEL_ERR_TIMEOUT and the kernel skips
 * the dependent work and exits normally. Must be >= 1000. */
kvsel_status kvsel_set_wait_limit_ns(uint64_t ns);

/* Test hook for the bounded waits. what = 1: the next tensor-core scoring
 * launch withholds the row statistics of its first work item, so the other
 * work items of that (layer, sequence, head) wait until the limit and report
 * KVSEL_ERR_TIMEOUT. what = 0 clears it. */
kvsel_status kvsel_debug_inject(int32_t what);

/* Stage timing of kvsel_snapkv with CUDA events recorded on the caller's
 * stream around each stage: [0] scoring kernel(s), [1] selection with the
 * fused K/V gather, [2] unused (0; the gather runs inside stage [1]). kvsel_profile_begin(n) arms it for the next n calls on
 * the current device (n in 1..100000; creates the events); each call records
 * its events without synchronising. kvsel_profile_end() synchronises, writes
 * the summed milliseconds per stage to stage_ms[0..2] and the number of
 * recorded calls to *calls, and disarms. */
kvsel_status kvsel_profile_begin(int32_t max_calls);
kvsel_status kvsel_profile_end(double* stage_ms, int32_t* calls);

/* Frees the internal workspace of every device this process used. Calls
 * still running on the GPU must have finished (the call synchronises each
 * device first). */
void kvsel_release(void);

/* Bytes of the internal workspace (the cudaMalloc'd scratch of every entry
 * point but kvsel_score_static) currently held on the current device; 0
 * before the first call that needs one and after kvsel_release. Host only. */
int64_t kvsel_workspace_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* KVSEL_H_ */
