// libkvsel C ABI: argument rules, per-call planning, the per-device workspace
// and status word, and the launch sequence of each entry point.
//
// Argument rules follow the page "SnapKV: choosing the KV cache of a long
// prompt with an observation window", section "Computing one full selection
// from Q and K" (从 Q 和 K 开始算一次完整选择): positive integer window,
// capacity and kernel, W <= L, C > W, odd kernel, avg or max pooling; a
// prompt shorter than the budget bypasses selection (L == C runs the normal
// path).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "kvsel_internal.h"

namespace kvsel {

__device__ int g_status_word;  // first device-side error of the current device

namespace {

constexpr int kMaxDevices = 64;

struct DevState {
  bool ready = false;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  int* status = nullptr;        // device address of g_status_word
  char* ws = nullptr;           // workspace
  size_t ws_bytes = 0;
  // host-buffer path (kvsel_snapkv_host): two device slots for one layer's
  // q_win and K each, a copy stream and its events
  char* stage = nullptr;
  size_t stage_bytes = 0;
  cudaStream_t copy = nullptr;
  cudaEvent_t ev_entry = nullptr, ev_loaded[2] = {nullptr, nullptr}, ev_freed[2] = {nullptr, nullptr};
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];
unsigned long long g_wait_limit_ns = 2000000000ull;
int g_inject = 0;

// Stage-timing events for kvsel_snapkv (see kvsel_profile_begin).
struct Profile {
  bool armed = false;
  int device = -1;
  int capacity = 0, used = 0;
  std::vector<cudaEvent_t> ev;  // 4 per call
};
Profile g_prof;

// Event slot for the next fused call, or nullptr when profiling is off.
cudaEvent_t* profile_slot() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_prof.armed || g_prof.used >= g_prof.capacity) return nullptr;
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != g_prof.device) return nullptr;
  return &g_prof.ev[4 * (size_t)g_prof.used++];
}

kvsel_status cuda_fail(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return KVSEL_OK;
  std::fprintf(stderr, "libkvsel: %s failed: %s\n", what, cudaGetErrorString(e));
  return KVSEL_ERR_CUDA;
}

kvsel_status device_state(DevState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return KVSEL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState& d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)))
      return cuda_fail(e, "cudaDeviceGetAttribute");
    cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_status_word)))
      return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    d.status = static_cast<int*>(p);
    if ((e = cudaMemset(d.status, 0, sizeof(int)))) return cuda_fail(e, "cudaMemset(status)");
    d.ready = true;
  }
  *out = &d;
  return KVSEL_OK;
}

// Grows the device workspace to at least `bytes` (synchronising the device
// before freeing the old one, which queued work may still use).
kvsel_status workspace(DevState* d, size_t bytes, char** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (bytes > d->ws_bytes) {
    cudaError_t e;
    if (d->ws) {
      if ((e = cudaDeviceSynchronize())) return cuda_fail(e, "cudaDeviceSynchronize");
      cudaFree(d->ws);
      d->ws = nullptr;
      d->ws_bytes = 0;
    }
    size_t want = (bytes + (1u << 20) - 1) & ~size_t((1u << 20) - 1);
    if ((e = cudaMalloc(reinterpret_cast<void**>(&d->ws), want)))
      return cuda_fail(e, "cudaMalloc(workspace)");
    d->ws_bytes = want;
  }
  *out = d->ws;
  return KVSEL_OK;
}

// Bump allocator over the workspace (256-byte aligned pieces).
struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    size_t at = off;
    off += (bytes + 255) & ~size_t(255);
    return at;
  }
};

// The selection's stagger words, zeroed on the stream before the launch.
kvsel_status stagger_words(char* ws, Carve& cv, cudaStream_t s, SelectArgs* sa) {
  int* w = reinterpret_cast<int*>(ws + cv.take(kSchedWords * sizeof(int)));
  cudaError_t e = cudaMemsetAsync(w, 0, kSchedWords * sizeof(int), s);
  if (e) return cuda_fail(e, "cudaMemsetAsync(selection stagger words)");
  sa->sched = w;
  sa->stagger_limit_ns = 500000ull;
  return KVSEL_OK;
}

// ---------------------------------------------------------------------------
// Argument rules and the per-call plan
// ---------------------------------------------------------------------------

struct Plan {
  int layers = 0, S = 0, H = 0, D = 0, dtype = 0;
  int Hkv = 0, G = 1;             // K/V heads, query heads per K/V head
  int64_t T = 0, T_out = 0;
  int elem_bytes = 0;
  std::vector<SeqDesc> all;      // every sequence
  int min_len = 0;
};

kvsel_status plan_shape(const kvsel_shape* sh, int C, Plan* p) {
  if (!sh) return KVSEL_ERR_INVALID_ARG;
  if (sh->num_layers < 1 || sh->num_seqs < 0 || sh->num_heads < 1 || sh->head_dim < 1)
    return KVSEL_ERR_INVALID_ARG;
  const int hkv = sh->num_kv_heads == 0 ? sh->num_heads : sh->num_kv_heads;
  if (hkv < 1 || sh->num_heads % hkv != 0) return KVSEL_ERR_INVALID_ARG;
  if (sh->dtype != KVSEL_BF16 && sh->dtype != KVSEL_F32) return KVSEL_ERR_INVALID_ARG;
  if (sh->num_seqs > 0 && !sh->seq_offsets) return KVSEL_ERR_INVALID_ARG;
  p->layers = sh->num_layers;
  p->S = sh->num_seqs;
  p->H = sh->num_heads;
  p->Hkv = hkv;
  p->G = sh->num_heads / hkv;
  p->D = sh->head_dim;
  p->dtype = sh->dtype;
  p->elem_bytes = sh->dtype == KVSEL_BF16 ? 2 : 4;
  p->all.clear();
  p->min_len = 0x7fffffff;
  if (p->S == 0) {
    p->min_len = 0;
    return KVSEL_OK;
  }
  if (sh->seq_offsets[0] != 0) return KVSEL_ERR_INVALID_ARG;
  int64_t out = 0;
  for (int b = 0; b < p->S; ++b) {
    const int64_t a0 = sh->seq_offsets[b], a1 = sh->seq_offsets[b + 1];
    if (a1 < a0) return KVSEL_ERR_INVALID_ARG;
    if (a1 - a0 > 0x7fffffffLL) return KVSEL_ERR_UNSUPPORTED;
    SeqDesc s{};
    s.tok_off = a0;
    s.len = (int32_t)(a1 - a0);
    s.out_off = (int32_t)out;
    s.index = b;
    if (C > 0) out += s.len < C ? s.len : C;
    if (out > 0x7fffffffLL) return KVSEL_ERR_UNSUPPORTED;
    p->all.push_back(s);
    if (s.len < p->min_len) p->min_len = s.len;
  }
  p->T = sh->seq_offsets[p->S];
  p->T_out = out;
  const double elems = (double)p->layers * (double)p->T * p->H * p->D;
  if (elems > 4.0e18 || p->T > 0x7fffffffLL) return KVSEL_ERR_UNSUPPORTED;
  return KVSEL_OK;
}

kvsel_status check_window(const Plan& p, int W) {
  if (W < 1) return KVSEL_ERR_INVALID_ARG;
  for (const SeqDesc& s : p.all)
    if (W > s.len) return KVSEL_ERR_INVALID_ARG;
  return KVSEL_OK;
}

kvsel_status check_pool(int kind, int k) {
  if (kind != KVSEL_POOL_AVG && kind != KVSEL_POOL_MAX) return KVSEL_ERR_INVALID_ARG;
  if (k < 1 || (k % 2) != 1) return KVSEL_ERR_INVALID_ARG;
  return KVSEL_OK;
}

kvsel_status check_budget(int W, int C) {
  if (C <= W) return KVSEL_ERR_INVALID_ARG;
  if (C - W > kMaxSelect) return KVSEL_ERR_UNSUPPORTED;
  return KVSEL_OK;
}

// Longest prefix among the sequences that are selected (L >= C).
int64_t max_prefix(const Plan& p, int W, int C) {
  int64_t m = 0;
  for (const SeqDesc& s : p.all)
    if (s.len >= C && s.len - W > m) m = s.len - W;
  return m;
}

bool gen_supported(int W, int D) { return (int64_t)W * D <= kGenericMaxQ; }

// One scoring pass: the scored sequences (all when C == 0, else L >= C) with
// their work-item and instance numbering for the chosen kernel, and which of
// the window rows it takes.
struct ScorePass {
  std::vector<SeqDesc> scored;
  int items_per_layer = 0, inst_per_layer = 0, max_chunks = 0;
  int chunk = 0, wpad = 0;
  int W = 0;           // window rows (the causal mask and statistics)
  int two_pass = 0;    // > 0: the two-pass kernel with this lag (long instances)
  int qg = 1;          // query heads scored together per K/V head (group-shared
                       // selection on the tensor cores); instances are then K/V heads
};

struct ScorePlan {
  bool tc = false;
  std::vector<ScorePass> passes;
};

// Long instances (more than kTwoPassChunks work items) take the two-pass
// kernel: pass 1 of an item computes its row statistics and frees its tensor
// memory, pass 2 recomputes the logits kTwoPassLag items later (K from L2)
// and writes the votes, so K is read from HBM once at any window.
#ifndef KVSEL_TWO_PASS_CHUNKS
#define KVSEL_TWO_PASS_CHUNKS 64
#endif
#ifndef KVSEL_TWO_PASS_LAG
#define KVSEL_TWO_PASS_LAG 3
#endif
constexpr int kTwoPassChunks = KVSEL_TWO_PASS_CHUNKS;
constexpr int kTwoPassLag = KVSEL_TWO_PASS_LAG;

// `group` > 1 (the group-shared selection): where the one-pass tensor-core
// kernel can take the group's G * W window rows at once (G a power of two,
// G * W <= 64), each K/V head is scored once against its G query heads and
// the votes come out summed per K/V head (sp->passes[0].qg = G); otherwise
// every query head is scored on its own.
kvsel_status plan_score(const Plan& p, int W, int C, const void* q, const void* k,
                        const DevState* d, ScorePlan* sp, bool allow_two_pass = true,
                        int group = 1) {
  const bool tc_ok = d->cc_major == 10 && tc_eligible(p.dtype, p.D, W, q, k);
  auto build = [&](ScorePass& ps, int chunk, int wpad, int heads) {
    ps.scored.clear();
    ps.items_per_layer = ps.inst_per_layer = ps.max_chunks = 0;
    ps.chunk = chunk;
    ps.wpad = wpad;
    for (const SeqDesc& s0 : p.all) {
      if (C > 0 && s0.len < C) continue;
      SeqDesc s = s0;
      s.n_chunks = (s.len + chunk - 1) / chunk;
      if (s.n_chunks == 0) continue;  // empty sequence (W <= 0 already rejected)
      s.item_base = ps.items_per_layer;
      s.inst_base = ps.inst_per_layer;
      ps.items_per_layer += heads * s.n_chunks;
      ps.inst_per_layer += heads;
      if (s.n_chunks > ps.max_chunks) ps.max_chunks = s.n_chunks;
      ps.scored.push_back(s);
    }
  };
  sp->passes.clear();
  if (tc_ok && group > 1 && (group & (group - 1)) == 0 && group * W <= 64 &&
      tc_eligible(p.dtype, p.D, group * W, q, k)) {
    ScorePass gp;
    gp.W = W;
    gp.qg = group;
    build(gp, tc_chunk_tokens(group * W), tc_window_pad(group * W), p.H / group);
    if (gp.max_chunks <= std::min(tc_max_chunks(group * W, d->sm_count), kTwoPassChunks)) {
      sp->tc = true;
      sp->passes.push_back(std::move(gp));
      return KVSEL_OK;
    }
  }
  if (tc_ok) {
    ScorePass one;
    one.W = W;
    build(one, tc_chunk_tokens(W), tc_window_pad(W), p.H);
    // the waits between the chunks of one instance end only if its chunks
    // span at most three rounds of items (chunks <= 2 x CTAs)
    if (one.max_chunks <= tc_max_chunks(W, d->sm_count)) {
      sp->tc = true;
      // (logits mode keeps the one-pass kernel: it stores logits, not votes)
      if (allow_two_pass && one.max_chunks > kTwoPassChunks) one.two_pass = kTwoPassLag;
      sp->passes.push_back(std::move(one));
      return KVSEL_OK;
    }
  }
  if (!gen_supported(W, p.D)) return KVSEL_ERR_UNSUPPORTED;
  sp->tc = false;
  ScorePass g;
  g.W = W;
  build(g, kGenericChunk, W, p.H);
  sp->passes.push_back(std::move(g));
  return KVSEL_OK;
}

// Uploads the sequence tables and runs the scoring kernels (votes or logits)
// of every pass of the plan, in order.
// `ev` (may be null): recorded just before the first pass's kernel and after
// the last one's.
kvsel_status run_pass(const Plan& p, const ScorePlan& sp, const ScorePass& ps, DevState* d,
                      const void* q, const void* k, int W, float* votes, float* logits,
                      char* ws, Carve& cv, cudaStream_t stream, cudaEvent_t ev_before);

kvsel_status run_score(const Plan& p, const ScorePlan& sp, DevState* d, const void* q,
                       const void* k, int W, float* votes, float* logits, char* ws,
                       Carve& cv, cudaStream_t stream, cudaEvent_t* ev = nullptr) {
  for (size_t i = 0; i < sp.passes.size(); ++i) {
    const kvsel_status st = run_pass(p, sp, sp.passes[i], d, q, k, W, votes, logits, ws, cv,
                                     stream, ev && i == 0 ? ev[0] : nullptr);
    if (st) return st;
  }
  if (ev) cudaEventRecord(ev[1], stream);
  return KVSEL_OK;
}

kvsel_status run_pass(const Plan& p, const ScorePlan& sp, const ScorePass& ps, DevState* d,
                      const void* q, const void* k, int W, float* votes, float* logits,
                      char* ws, Carve& cv, cudaStream_t stream, cudaEvent_t ev_before) {
  const int64_t items = (int64_t)p.layers * ps.items_per_layer;
  const int64_t insts = (int64_t)p.layers * ps.inst_per_layer;
  if (items == 0) return KVSEL_OK;
  if (items > 0x7fffffffLL) return KVSEL_ERR_UNSUPPORTED;
  const size_t o_seq = cv.take(ps.scored.size() * sizeof(SeqDesc));
  const size_t o_part = cv.take((size_t)items * ps.wpad * 2 * sizeof(float));
  const size_t o_fin = cv.take((size_t)insts * ps.wpad * 2 * sizeof(float));
  cudaError_t e = cudaMemcpyAsync(ws + o_seq, ps.scored.data(),
                                  ps.scored.size() * sizeof(SeqDesc),
                                  cudaMemcpyHostToDevice, stream);
  if (e) return cuda_fail(e, "cudaMemcpyAsync(sequence table)");
  ScoreArgs a{};
  a.q = q;
  a.k = k;
  a.layers = p.layers;
  a.H = p.H / ps.qg;            // instance heads
  a.kv_group = ps.qg > 1 ? 1 : p.G;
  a.qg = ps.qg;
  a.D = p.D;
  a.dtype = p.dtype;
  a.W = ps.W;
  a.T = p.T;
  a.q_rows = (int64_t)p.S * W;
  a.q_W = W;
  a.two_pass = ps.two_pass;
  a.n_scored = (int)ps.scored.size();
  a.seqs = reinterpret_cast<const SeqDesc*>(ws + o_seq);
  a.items_per_layer = ps.items_per_layer;
  a.inst_per_layer = ps.inst_per_layer;
  a.chunk_tokens = ps.chunk;
  a.wpad = ps.wpad;
  a.scale = (float)(1.0 / std::sqrt((double)p.D));
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p.D));
  a.part = reinterpret_cast<float*>(ws + o_part);
  a.final_stats = reinterpret_cast<float*>(ws + o_fin);
  a.votes = votes;
  a.logits = logits;
  a.status = d->status;
  a.sm_count = d->sm_count;
  a.stream = stream;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    a.wait_limit_ns = g_wait_limit_ns;
    a.inject = g_inject;
    if (sp.tc && logits == nullptr) g_inject = 0;  // one-shot
  }
  if (sp.tc) {
    // the tensor-core kernel's exchange slots start out as all-ones (empty)
    if ((e = cudaMemsetAsync(a.part, 0xFF, (size_t)items * ps.wpad * 2 * sizeof(float), stream)))
      return cuda_fail(e, "cudaMemsetAsync(exchange slots)");
    if ((e = cudaMemsetAsync(a.final_stats, 0xFF, (size_t)insts * ps.wpad * 2 * sizeof(float),
                             stream)))
      return cuda_fail(e, "cudaMemsetAsync(final slots)");
    int grid = tc_max_grid(d->sm_count);
    if (items < grid) grid = (int)items;
    if (ev_before) cudaEventRecord(ev_before, stream);
    e = launch_tc_score(a, logits != nullptr, grid);
    return cuda_fail(e, "tensor-core scoring launch");
  }
  if (ev_before) cudaEventRecord(ev_before, stream);
  e = launch_generic_score(a, logits != nullptr);
  return cuda_fail(e, "CUDA-core scoring launch");
}

kvsel_status upload_all(const Plan& p, char* ws, Carve& cv, cudaStream_t stream,
                        const SeqDesc** out) {
  const size_t o = cv.take(p.all.size() * sizeof(SeqDesc) + 1);
  cudaError_t e = cudaMemcpyAsync(ws + o, p.all.data(), p.all.size() * sizeof(SeqDesc),
                                  cudaMemcpyHostToDevice, stream);
  if (e) return cuda_fail(e, "cudaMemcpyAsync(sequence table)");
  *out = reinterpret_cast<const SeqDesc*>(ws + o);
  return KVSEL_OK;
}

// Packs the selection's instances (kPackWhole in kvsel_internal.h) when its
// clusters hold more than one CTA and some instances fit one CTA's slice:
// whole-cluster instances first (the longest work starts in the first wave),
// then the others cs to a cluster. Uploads the table; leaves sa->pack null
// when nothing packs. Instances are numbered ((layer * S) + b) * Hsel + h.
size_t select_pack_bytes(const Plan& p) {
  return (size_t)p.layers * p.S * p.H * kSelMaxCluster * sizeof(int32_t) + 256;
}

kvsel_status select_pack(const Plan& p, int W, int C, int Hsel, char* ws, Carve& cv,
                         cudaStream_t stream, SelectArgs* sa) {
  sa->pack = nullptr;
  sa->n_clusters = 0;
  int cs = 1, slice = 1;
  select_geometry(sa->max_prefix, &cs, &slice);
  if (cs <= 1 || cs > kSelMaxCluster) return KVSEL_OK;
  std::vector<int32_t> whole, single;
  for (int layer = 0; layer < p.layers; ++layer)
    for (int b = 0; b < p.S; ++b) {
      const SeqDesc& sd = p.all[b];
      const bool one = sd.len < C || (int64_t)sd.len - W <= slice;
      for (int h = 0; h < Hsel; ++h)
        (one ? single : whole).push_back((int32_t)(((int64_t)layer * p.S + b) * Hsel + h));
    }
  if (single.empty()) return KVSEL_OK;
  const size_t nc = whole.size() + (single.size() + cs - 1) / cs;
  std::vector<int32_t> tab(nc * kSelMaxCluster, -1);
  size_t c = 0;
  for (int32_t i : whole) {
    tab[c * kSelMaxCluster] = i;
    tab[c * kSelMaxCluster + 1] = kPackWhole;
    ++c;
  }
  for (size_t k = 0; k < single.size(); k += cs, ++c)
    for (int r = 0; r < cs && k + r < single.size(); ++r) tab[c * kSelMaxCluster + r] = single[k + r];
  const size_t o = cv.take(tab.size() * sizeof(int32_t));
  cudaError_t e = cudaMemcpyAsync(ws + o, tab.data(), tab.size() * sizeof(int32_t),
                                  cudaMemcpyHostToDevice, stream);
  if (e) return cuda_fail(e, "cudaMemcpyAsync(selection packing)");
  sa->pack = reinterpret_cast<const int32_t*>(ws + o);
  sa->n_clusters = (int)nc;
  return KVSEL_OK;
}

size_t score_ws_bytes(const Plan& p, const ScorePlan& sp) {
  size_t total = 4096;
  for (const ScorePass& ps : sp.passes) {
    const int64_t items = (int64_t)p.layers * ps.items_per_layer;
    const int64_t insts = (int64_t)p.layers * ps.inst_per_layer;
    total += ps.scored.size() * sizeof(SeqDesc) + (size_t)items * ps.wpad * 8 +
             (size_t)insts * ps.wpad * 8 + 3 * 256;
  }
  return total;
}

}  // namespace
}  // namespace kvsel

// ---------------------------------------------------------------------------
// kvsel_score_static: kvsel_score for callers that cannot allocate device
// memory, for instance code that runs under an allocator it must not bypass
// or in a context where cudaMalloc is not permitted. Its scratch (sequence
// tables, the cross-chunk exchange slots, merged row statistics) lives in a
// file-scope device array instead of the cudaMalloc'd workspace. Every GPU
// that loads the library holds this array until the process exits.
// ---------------------------------------------------------------------------

namespace kvsel {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;   // 8 MiB per device
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

char* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device; looked up once
// per device (the host-side name is only a stand-in for the device symbol).
kvsel_status static_scratch(char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return KVSEL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_static_scratch)))
      return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_static_ptr[dev] = static_cast<char*>(p);
  }
  *out = g_static_ptr[dev];
  return KVSEL_OK;
}

// Scratch bytes kvsel_score_static carves, in the order it carves them.
size_t static_score_bytes(const Plan& p, const ScorePlan& sp) {
  Carve c;
  c.take(p.all.size() * sizeof(SeqDesc) + 1);                 // every sequence
  for (const ScorePass& ps : sp.passes) {
    const int64_t items = (int64_t)p.layers * ps.items_per_layer;
    const int64_t insts = (int64_t)p.layers * ps.inst_per_layer;
    c.take(ps.scored.size() * sizeof(SeqDesc));               // scored sequences
    c.take((size_t)items * ps.wpad * 2 * sizeof(float));      // exchange slots / partials
    c.take((size_t)insts * ps.wpad * 2 * sizeof(float));      // merged statistics / slots
  }
  return c.off;
}

}  // namespace

}  // namespace kvsel

extern "C" int64_t kvsel_score_static_bytes(const kvsel_shape* shape, int32_t W) {
  using namespace kvsel;
  Plan p;
  if (plan_shape(shape, 0, &p) != KVSEL_OK || check_window(p, W) != KVSEL_OK) return -1;
  DevState* d = nullptr;
  if (device_state(&d) != KVSEL_OK) return -1;
  ScorePlan sp;
  // alignment is unknown here: assume 256-byte aligned tensors
  static const char probe[512] = {0};
  const void* aligned = reinterpret_cast<const void*>(
      (reinterpret_cast<uintptr_t>(probe) + 255) & ~uintptr_t(255));
  if (plan_score(p, W, 0, aligned, aligned, d, &sp) != KVSEL_OK) return -1;
  return (int64_t)static_score_bytes(p, sp);
}

extern "C" kvsel_status kvsel_score_static(const kvsel_shape* shape, const void* q_win,
                                           const void* K, int32_t W, int32_t pool_kind,
                                           int32_t pool_k, float* votes, float* pooled,
                                           void* stream) {
  using namespace kvsel;
  Plan p;
  kvsel_status st;
  if ((st = plan_shape(shape, 0, &p))) return st;
  if ((st = check_window(p, W))) return st;
  if ((st = check_pool(pool_kind, pool_k))) return st;
  if (p.T == 0) return KVSEL_OK;
  if (!q_win || !K || !votes || !pooled) return KVSEL_ERR_INVALID_ARG;
  DevState* d;
  if ((st = device_state(&d))) return st;
  ScorePlan sp;
  if ((st = plan_score(p, W, 0, q_win, K, d, &sp))) return st;
  const size_t need = static_score_bytes(p, sp);
  if (need > kStaticScratchBytes) {
    std::fprintf(stderr,
                 "libkvsel: kvsel_score_static needs %zu scratch bytes, more than its "
                 "fixed %zu; use kvsel_score\n",
                 need, kStaticScratchBytes);
    return KVSEL_ERR_UNSUPPORTED;
  }
  char* ws;
  if ((st = static_scratch(&ws))) return st;
  Carve cv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const SeqDesc* all_dev;
  if ((st = upload_all(p, ws, cv, s, &all_dev))) return st;
  if ((st = run_score(p, sp, d, q_win, K, W, votes, nullptr, ws, cv, s))) return st;
  PoolArgs pa{};
  pa.votes = votes;
  pa.pooled = pooled;
  pa.layers = p.layers;
  pa.H = p.H;
  pa.W = W;
  pa.pool_kind = pool_kind;
  pa.pool_k = pool_k;
  pa.T = p.T;
  pa.n_seqs = p.S;
  pa.seqs = all_dev;
  pa.stream = s;
  return cuda_fail(launch_pool(pa), "pooling launch");
}

using namespace kvsel;

extern "C" {

const char* kvsel_version(void) { return "kvsel 0.1.0 (sm_103a)"; }

const char* kvsel_status_string(kvsel_status s) {
  switch (s) {
    case KVSEL_OK: return "ok";
    case KVSEL_ERR_INVALID_ARG: return "invalid argument";
    case KVSEL_ERR_UNSUPPORTED: return "unsupported (beyond a documented limit)";
    case KVSEL_ERR_NONFINITE: return "non-finite window logit or score";
    case KVSEL_ERR_TIMEOUT: return "a bounded device wait ran out";
    case KVSEL_ERR_CUDA: return "CUDA runtime error";
    case KVSEL_ERR_BAD_INDEX: return "gather index out of range";
    default: return "unknown status";
  }
}

int64_t kvsel_out_tokens(const kvsel_shape* shape, int32_t C) {
  if (C < 1) return -1;
  Plan p;
  if (plan_shape(shape, C, &p) != KVSEL_OK) return -1;
  return p.T_out;
}

int32_t kvsel_score_path(const kvsel_shape* shape, int32_t W, int32_t C) {
  Plan p;
  if (C < 0 || plan_shape(shape, C, &p) != KVSEL_OK) return -1;
  if (check_window(p, W) != KVSEL_OK) return -1;
  if (C > 0 && check_budget(W, C) != KVSEL_OK) return -1;
  DevState* d = nullptr;
  if (device_state(&d) != KVSEL_OK) return -1;
  ScorePlan sp;
  // alignment is unknown here: assume 256-byte aligned tensors
  static const char probe[512] = {0};
  const void* aligned = reinterpret_cast<const void*>(
      (reinterpret_cast<uintptr_t>(probe) + 255) & ~uintptr_t(255));
  if (plan_score(p, W, C, aligned, aligned, d, &sp) != KVSEL_OK) return -1;
  if (!sp.tc) return 0;
  return sp.passes[0].two_pass ? 3 : 1;
}

kvsel_status kvsel_window_logits(const kvsel_shape* shape, const void* q_win, const void* K,
                                 int32_t W, float* logits, void* stream) {
  Plan p;
  kvsel_status st;
  if ((st = plan_shape(shape, 0, &p))) return st;
  if ((st = check_window(p, W))) return st;
  if (p.T == 0) return KVSEL_OK;
  if (!q_win || !K || !logits) return KVSEL_ERR_INVALID_ARG;
  DevState* d;
  if ((st = device_state(&d))) return st;
  ScorePlan sp;
  if ((st = plan_score(p, W, 0, q_win, K, d, &sp, false))) return st;
  char* ws;
  if ((st = workspace(d, score_ws_bytes(p, sp), &ws))) return st;
  Carve cv;
  return run_score(p, sp, d, q_win, K, W, nullptr, logits, ws, cv,
                   static_cast<cudaStream_t>(stream));
}

kvsel_status kvsel_score(const kvsel_shape* shape, const void* q_win, const void* K, int32_t W,
                         int32_t pool_kind, int32_t pool_k, float* votes, float* pooled,
                         void* stream) {
  Plan p;
  kvsel_status st;
  if ((st = plan_shape(shape, 0, &p))) return st;
  if ((st = check_window(p, W))) return st;
  if ((st = check_pool(pool_kind, pool_k))) return st;
  if (p.T == 0) return KVSEL_OK;
  if (!q_win || !K || !pooled) return KVSEL_ERR_INVALID_ARG;
  DevState* d;
  if ((st = device_state(&d))) return st;
  ScorePlan sp;
  if ((st = plan_score(p, W, 0, q_win, K, d, &sp))) return st;
  const size_t votes_bytes = votes ? 0 : (size_t)p.layers * p.H * p.T * sizeof(float);
  char* ws;
  if ((st = workspace(d, score_ws_bytes(p, sp) + votes_bytes +
                             p.all.size() * sizeof(SeqDesc) + 1024, &ws)))
    return st;
  Carve cv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const SeqDesc* all_dev;
  if ((st = upload_all(p, ws, cv, s, &all_dev))) return st;
  float* v = votes;
  if (!v) v = reinterpret_cast<float*>(ws + cv.take(votes_bytes));
  if ((st = run_score(p, sp, d, q_win, K, W, v, nullptr, ws, cv, s))) return st;
  PoolArgs pa{};
  pa.votes = v;
  pa.pooled = pooled;
  pa.layers = p.layers;
  pa.H = p.H;
  pa.W = W;
  pa.pool_kind = pool_kind;
  pa.pool_k = pool_k;
  pa.T = p.T;
  pa.n_seqs = p.S;
  pa.seqs = all_dev;
  pa.stream = s;
  return cuda_fail(launch_pool(pa), "pooling launch");
}

kvsel_status kvsel_select(const kvsel_shape* shape, const float* pooled, int32_t W, int32_t C,
                          int32_t* out_idx, void* stream) {
  Plan p;
  kvsel_status st;
  if (C < 1) return KVSEL_ERR_INVALID_ARG;
  if ((st = plan_shape(shape, C, &p))) return st;
  if ((st = check_window(p, W))) return st;
  if ((st = check_budget(W, C))) return st;
  if (max_prefix(p, W, C) > kMaxPrefix) return KVSEL_ERR_UNSUPPORTED;
  if (p.T_out == 0) return KVSEL_OK;
  if (!pooled || !out_idx) return KVSEL_ERR_INVALID_ARG;
  DevState* d;
  if ((st = device_state(&d))) return st;
  char* ws;
  if ((st = workspace(d, p.all.size() * sizeof(SeqDesc) + select_pack_bytes(p) + 1024, &ws)))
    return st;
  Carve cv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const SeqDesc* all_dev;
  if ((st = upload_all(p, ws, cv, s, &all_dev))) return st;
  SelectArgs sa{};
  sa.scores = pooled;
  sa.pool_inline = 0;
  sa.layers = p.layers;
  sa.H = p.H;
  sa.W = W;
  sa.C = C;
  sa.T = p.T;
  sa.T_out = p.T_out;
  sa.n_seqs = p.S;
  sa.seqs = all_dev;
  sa.out_idx = out_idx;
  sa.status = d->status;
  sa.sm_count = d->sm_count;
  sa.max_prefix = max_prefix(p, W, C);
  sa.vote_group = 1;
  sa.kv_H = p.H;
  sa.kv_div = 1;
  sa.stream = s;
  if ((st = select_pack(p, W, C, sa.H, ws, cv, s, &sa))) return st;
  return cuda_fail(launch_select(sa), "selection launch");
}

kvsel_status kvsel_compact(const kvsel_shape* shape, const void* K, const void* V,
                           const int32_t* out_idx, int32_t C, void* out_K, void* out_V,
                           void* stream) {
  Plan p;
  kvsel_status st;
  if (C < 1) return KVSEL_ERR_INVALID_ARG;
  if ((st = plan_shape(shape, C, &p))) return st;
  if (p.T_out == 0) return KVSEL_OK;
  if (!K || !V || !out_idx || !out_K || !out_V) return KVSEL_ERR_INVALID_ARG;
  DevState* d;
  if ((st = device_state(&d))) return st;
  char* ws;
  if ((st = workspace(d, p.all.size() * sizeof(SeqDesc) + 1024, &ws))) return st;
  Carve cv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const SeqDesc* all_dev;
  if ((st = upload_all(p, ws, cv, s, &all_dev))) return st;
  CompactArgs ca{};
  ca.k = K;
  ca.v = V;
  ca.idx = out_idx;
  ca.out_k = out_K;
  ca.out_v = out_V;
  ca.layers = p.layers;
  ca.H = p.H;
  ca.S = p.S;
  ca.C = C;
  ca.T = p.T;
  ca.T_out = p.T_out;
  ca.row_bytes = (int64_t)p.D * p.elem_bytes;
  ca.seqs = all_dev;
  int64_t mr = 0;
  for (const SeqDesc& q : p.all) {
    const int64_t n = (int64_t)(q.len < C ? q.len : C) * p.H;
    if (n > mr) mr = n;
  }
  ca.max_rows = mr;
  if ((double)mr * (double)(ca.row_bytes / 2) > 4.0e9) return KVSEL_ERR_UNSUPPORTED;
  ca.status = d->status;
  ca.sm_count = d->sm_count;
  ca.kv_H = p.Hkv;
  ca.kv_div = p.G;
  ca.stream = s;
  return cuda_fail(launch_compact(ca), "gather launch");
}

}  // extern "C"

namespace kvsel {
namespace {

// Jacap work plan: the scored sequences (L >= max(C, W + 1)) with their
// statistics, Gram and leverage item numbering (per layer).
struct JacapPlan {
  std::vector<JSeq> seqs;
  int insts = 0;
  // Gram work: pieces, the pieces of each CTA and of each instance
  std::vector<JSeg> segs;
  std::vector<int32_t> cta_seg, inst_seg;
};

JacapPlan plan_jacap(const Plan& p, int W, int C, int sm_count) {
  JacapPlan jp;
  std::vector<int> tiles_of;                   // per scored sequence
  for (const SeqDesc& sd : p.all) {
    if (sd.len < C || sd.len <= W) continue;
    JSeq j{};
    const int P = sd.len - W;
    const int n_tiles = (P + 127) / 128;
    j.tok_off = sd.tok_off;
    j.len = sd.len;
    j.index = sd.index;
    j.inst_base = jp.insts;
    jp.insts += p.H;
    jp.seqs.push_back(j);
    tiles_of.push_back(n_tiles);
  }
  if (jp.seqs.empty()) return jp;
  // Gram: every instance's tiles in instance order (layer, sequence, head),
  // cut into n_gram equal contiguous ranges, each range into pieces at the
  // instance boundaries
  const int64_t n_inst = (int64_t)p.layers * jp.insts;
  std::vector<int64_t> start(n_inst + 1, 0);
  {
    int64_t i = 0;
    for (int layer = 0; layer < p.layers; ++layer)
      for (size_t q = 0; q < jp.seqs.size(); ++q)
        for (int h = 0; h < p.H; ++h, ++i) start[i + 1] = start[i] + tiles_of[q];
  }
  const int64_t total = start[n_inst];
  const int64_t n_gram = std::max<int64_t>(
      1, std::min<int64_t>(sm_count, total / kJGramMinTiles));
  jp.cta_seg.assign(n_gram + 1, 0);
  jp.inst_seg.assign(n_inst + 1, 0);
  int64_t inst = 0;
  for (int64_t c = 0; c < n_gram; ++c) {
    int64_t lo = c * total / n_gram;
    const int64_t hi = (c + 1) * total / n_gram;
    while (lo < hi) {
      while (start[inst + 1] <= lo) ++inst;
      const int64_t end = std::min(hi, start[inst + 1]);
      if (lo == start[inst]) jp.inst_seg[inst] = (int32_t)jp.segs.size();
      jp.segs.push_back(JSeg{(int32_t)inst, (int32_t)(lo - start[inst]),
                             (int32_t)(end - start[inst]), 0});
      lo = end;
    }
    jp.cta_seg[c + 1] = (int32_t)jp.segs.size();
  }
  jp.inst_seg[n_inst] = (int32_t)jp.segs.size();
  return jp;
}

// The tables the kernels read, packed for one host-to-device copy: sequences,
// pieces, the CTAs' and the instances' piece ranges.
size_t jacap_table_bytes(const JacapPlan& jp) {
  auto up16 = [](size_t x) { return (x + 15) & ~size_t(15); };
  return up16(jp.seqs.size() * sizeof(JSeq)) + up16(jp.segs.size() * sizeof(JSeg)) +
         up16(jp.cta_seg.size() * sizeof(int32_t)) + up16(jp.inst_seg.size() * sizeof(int32_t));
}

size_t jacap_ws_bytes(const Plan& p, const JacapPlan& jp) {
  const size_t plane = (size_t)p.layers * p.H * p.T;
  return 8 * 256 + plane * (sizeof(float2) + sizeof(float)) +
         jp.segs.size() * 2 * sizeof(float) + jacap_table_bytes(jp) +
         jp.segs.size() * 128 * 128 * sizeof(float) +
         (size_t)p.layers * jp.insts * 2 * 128 * 128 * 2;
}

// Jacap scores into `scores` ([layers][H][T], zeroed first; prefix positions
// of the planned sequences get r, the rest 0).
kvsel_status run_jacap(const Plan& p, const JacapPlan& jp, DevState* d, const void* q_win,
                       const void* K, const void* V, int W, float tau, float beta, float eps,
                       float* scores, char* ws, Carve& cv, cudaStream_t s,
                       cudaEvent_t* ev = nullptr) {
  const std::vector<JSeq>& seqs = jp.seqs;
  const int insts = jp.insts;
  const size_t plane = (size_t)p.layers * p.H * p.T;
  cudaError_t e = cudaMemsetAsync(scores, 0, plane * sizeof(float), s);
  if (e) return cuda_fail(e, "cudaMemsetAsync(scores)");
  if (seqs.empty()) return KVSEL_OK;
  if ((int64_t)p.layers * insts > 0x7fffffffLL)
    return KVSEL_ERR_UNSUPPORTED;
  const size_t o_tab = cv.take(jacap_table_bytes(jp));
  const size_t o_zk = cv.take(plane * sizeof(float2));
  const size_t o_w = cv.take(plane * sizeof(float));
  const size_t o_part = cv.take(jp.segs.size() * 2 * sizeof(float));
  const size_t o_gram = cv.take(jp.segs.size() * 128 * 128 * sizeof(float));
  const size_t o_linv = cv.take((size_t)p.layers * insts * 2 * 128 * 128 * 2);
  // the tables, packed as jacap_table_bytes lays them out
  std::vector<char> tab(jacap_table_bytes(jp), 0);
  size_t o_segs = 0, o_cta = 0, o_inst = 0;
  {
    size_t at = 0;
    auto put = [&](const void* src, size_t bytes) {
      const size_t here = at;
      if (bytes) std::memcpy(tab.data() + at, src, bytes);
      at += (bytes + 15) & ~size_t(15);
      return here;
    };
    put(seqs.data(), seqs.size() * sizeof(JSeq));
    o_segs = put(jp.segs.data(), jp.segs.size() * sizeof(JSeg));
    o_cta = put(jp.cta_seg.data(), jp.cta_seg.size() * sizeof(int32_t));
    o_inst = put(jp.inst_seg.data(), jp.inst_seg.size() * sizeof(int32_t));
  }
  if ((e = cudaMemcpyAsync(ws + o_tab, tab.data(), tab.size(), cudaMemcpyHostToDevice, s)))
    return cuda_fail(e, "cudaMemcpyAsync(jacap tables)");
  JacapArgs a{};
  a.q = q_win;
  a.k = K;
  a.v = V;
  a.layers = p.layers;
  a.H = p.H;
  a.D = p.D;
  a.W = W;
  a.S = p.S;
  a.T = p.T;
  a.n_scored = (int)seqs.size();
  a.seqs = reinterpret_cast<const JSeq*>(ws + o_tab);
  a.segs = reinterpret_cast<const JSeg*>(ws + o_tab + o_segs);
  a.cta_seg = reinterpret_cast<const int32_t*>(ws + o_tab + o_cta);
  a.inst_seg = reinterpret_cast<const int32_t*>(ws + o_tab + o_inst);
  a.n_gram = (int)(jp.cta_seg.size() - 1);
  a.inst_per_layer = insts;
  a.tau = tau;
  a.beta = beta;
  a.eps = eps;
  a.zk = reinterpret_cast<float2*>(ws + o_zk);
  a.part = reinterpret_cast<float*>(ws + o_part);
  a.gram = reinterpret_cast<float*>(ws + o_gram);
  a.wts = reinterpret_cast<float*>(ws + o_w);
  a.linv = ws + o_linv;
  a.scores = scores;
  a.status = d->status;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    a.wait_limit_ns = g_wait_limit_ns;
  }
  a.stream = s;
  if (ev) cudaEventRecord(ev[0], s);
  e = launch_jacap(a);
  if (ev) cudaEventRecord(ev[1], s);
  return cuda_fail(e, "jacap launch");
}

kvsel_status check_jacap(const Plan& p, const void* q, const void* K, const void* V, float tau,
                         float beta, float eps) {
  if (!(tau > 0.f) || !(beta >= 0.f && beta < 1.f) || !(eps >= 0.f) || !std::isfinite(tau) ||
      !std::isfinite(eps))
    return KVSEL_ERR_INVALID_ARG;
  if (p.Hkv != p.H || !jacap_eligible(p.dtype, p.D, q, K, V)) return KVSEL_ERR_UNSUPPORTED;
  return KVSEL_OK;
}

// The fused path. grouped = 0: one selection per query head (outputs over H
// heads; query head h gathers K/V head h / G); grouped = 1: one selection per
// K/V head on the summed votes of its G query heads (outputs over H_kv heads).
kvsel_status snapkv_impl(const kvsel_shape* shape, const void* q_win, const void* K,
                         const void* V, int32_t W, int32_t C, int32_t pool_kind,
                         int32_t pool_k, int32_t* out_idx, void* out_K, void* out_V,
                         void* stream, bool grouped) {
  Plan p;
  kvsel_status st;
  if (C < 1) return KVSEL_ERR_INVALID_ARG;
  if ((st = plan_shape(shape, C, &p))) return st;
  if ((st = check_window(p, W))) return st;
  if ((st = check_budget(W, C))) return st;
  if ((st = check_pool(pool_kind, pool_k))) return st;
  if (max_prefix(p, W, C) > kMaxPrefix) return KVSEL_ERR_UNSUPPORTED;
  if (p.T_out == 0) return KVSEL_OK;
  if (!q_win || !K || !V || !out_idx || !out_K || !out_V) return KVSEL_ERR_INVALID_ARG;
  DevState* d;
  if ((st = device_state(&d))) return st;
  ScorePlan sp;
  if ((st = plan_score(p, W, C, q_win, K, d, &sp, true, grouped ? p.G : 1))) return st;
  // group-shared scoring writes one vote plane per K/V head, already summed
  const bool group_scored = !sp.passes.empty() && sp.passes[0].qg > 1;
  const size_t plane_bytes = (size_t)p.layers * p.H * p.T * sizeof(float);
  char* ws;
  if ((st = workspace(d, score_ws_bytes(p, sp) + plane_bytes + 2 * 256 +
                             kSchedWords * sizeof(int) + p.all.size() * sizeof(SeqDesc) +
                             select_pack_bytes(p) + 1024,
                      &ws)))
    return st;
  Carve cv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const SeqDesc* all_dev;
  if ((st = upload_all(p, ws, cv, s, &all_dev))) return st;
  float* votes = reinterpret_cast<float*>(ws + cv.take(plane_bytes));
  cudaEvent_t* ev = profile_slot();
  // the selection's stagger words and packing go out before the scoring, so
  // the selection kernel directly follows the scoring kernel on the stream
  // (a programmatic dependent launch: its CTAs may start as the scoring CTAs
  // leave and wait for the scoring grid's memory before reading the votes)
  SelectArgs sa{};
  if ((st = stagger_words(ws, cv, s, &sa))) return st;
  sa.scores = votes;
  sa.pool_inline = 1;
  sa.pool_kind = pool_kind;
  sa.pool_k = pool_k;
  sa.layers = p.layers;
  sa.H = grouped ? p.Hkv : p.H;
  sa.vote_group = grouped && !group_scored ? p.G : 1;
  sa.kv_H = p.Hkv;
  sa.kv_div = grouped ? 1 : p.G;
  sa.W = W;
  sa.C = C;
  sa.T = p.T;
  sa.T_out = p.T_out;
  sa.n_seqs = p.S;
  sa.seqs = all_dev;
  sa.out_idx = out_idx;
  sa.status = d->status;
  sa.sm_count = d->sm_count;
  sa.max_prefix = max_prefix(p, W, C);
  sa.gather = 1;
  sa.k = K;
  sa.v = V;
  sa.out_k = out_K;
  sa.out_v = out_V;
  sa.row_bytes = (int64_t)p.D * p.elem_bytes;
  sa.stream = s;
  sa.pdl = 1;
  if ((st = select_pack(p, W, C, sa.H, ws, cv, s, &sa))) return st;
  if ((st = run_score(p, sp, d, q_win, K, W, votes, nullptr, ws, cv, s, ev))) return st;
  if ((st = cuda_fail(launch_select(sa), "selection and gather launch"))) return st;
  if (ev) {
    cudaEventRecord(ev[2], s);
    cudaEventRecord(ev[3], s);
  }
  return KVSEL_OK;
}

}  // namespace
}  // namespace kvsel

extern "C" {

kvsel_status kvsel_jacap_score(const kvsel_shape* shape, const void* q_win, const void* K,
                               const void* V, int32_t W, float tau, float beta, float eps,
                               float* scores, void* stream) {
  using namespace kvsel;
  Plan p;
  kvsel_status st;
  if ((st = plan_shape(shape, 0, &p))) return st;
  if ((st = check_window(p, W))) return st;
  if (p.T == 0) return KVSEL_OK;
  if (!q_win || !K || !V || !scores) return KVSEL_ERR_INVALID_ARG;
  if ((st = check_jacap(p, q_win, K, V, tau, beta, eps))) return st;
  DevState* d;
  if ((st = device_state(&d))) return st;
  const JacapPlan jp = plan_jacap(p, W, 0, d->sm_count);
  char* ws;
  if ((st = workspace(d, jacap_ws_bytes(p, jp), &ws))) return st;
  Carve cv;
  return run_jacap(p, jp, d, q_win, K, V, W, tau, beta, eps, scores, ws, cv,
                   static_cast<cudaStream_t>(stream));
}

kvsel_status kvsel_jacap(const kvsel_shape* shape, const void* q_win, const void* K,
                         const void* V, int32_t W, int32_t C, float tau, float beta, float eps,
                         int32_t* out_idx, void* out_K, void* out_V, void* stream) {
  using namespace kvsel;
  Plan p;
  kvsel_status st;
  if (C < 1) return KVSEL_ERR_INVALID_ARG;
  if ((st = plan_shape(shape, C, &p))) return st;
  if ((st = check_window(p, W))) return st;
  if ((st = check_budget(W, C))) return st;
  if (max_prefix(p, W, C) > kMaxPrefix) return KVSEL_ERR_UNSUPPORTED;
  if (p.T_out == 0) return KVSEL_OK;
  if (!q_win || !K || !V || !out_idx || !out_K || !out_V) return KVSEL_ERR_INVALID_ARG;
  if ((st = check_jacap(p, q_win, K, V, tau, beta, eps))) return st;
  DevState* d;
  if ((st = device_state(&d))) return st;
  const size_t plane_bytes = (size_t)p.layers * p.H * p.T * sizeof(float);
  const JacapPlan jp = plan_jacap(p, W, C, d->sm_count);
  char* ws;
  if ((st = workspace(d, jacap_ws_bytes(p, jp) + plane_bytes + 2 * 256 +
                             kSchedWords * sizeof(int) + p.all.size() * sizeof(SeqDesc) +
                             select_pack_bytes(p) + 1024,
                      &ws)))
    return st;
  Carve cv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const SeqDesc* all_dev;
  if ((st = upload_all(p, ws, cv, s, &all_dev))) return st;
  float* scores = reinterpret_cast<float*>(ws + cv.take(plane_bytes));
  cudaEvent_t* ev = profile_slot();
  // selection set-up first, so the selection kernel directly follows the
  // scoring kernels (programmatic dependent launch, as in the SnapKV path)
  SelectArgs sa{};
  if ((st = stagger_words(ws, cv, s, &sa))) return st;
  sa.scores = scores;
  sa.pool_inline = 0;
  sa.layers = p.layers;
  sa.H = p.H;
  sa.vote_group = 1;
  sa.kv_H = p.H;
  sa.kv_div = 1;
  sa.W = W;
  sa.C = C;
  sa.T = p.T;
  sa.T_out = p.T_out;
  sa.n_seqs = p.S;
  sa.seqs = all_dev;
  sa.out_idx = out_idx;
  sa.status = d->status;
  sa.sm_count = d->sm_count;
  sa.max_prefix = max_prefix(p, W, C);
  sa.gather = 1;
  sa.k = K;
  sa.v = V;
  sa.out_k = out_K;
  sa.out_v = out_V;
  sa.row_bytes = (int64_t)p.D * p.elem_bytes;
  sa.stream = s;
  sa.pdl = 1;
  if ((st = select_pack(p, W, C, sa.H, ws, cv, s, &sa))) return st;
  if ((st = run_jacap(p, jp, d, q_win, K, V, W, tau, beta, eps, scores, ws, cv, s, ev)))
    return st;
  if ((st = cuda_fail(launch_select(sa), "selection and gather launch"))) return st;
  if (ev) {
    cudaEventRecord(ev[2], s);
    cudaEventRecord(ev[3], s);
  }
  return KVSEL_OK;
}

kvsel_status kvsel_decode_attention(const kvsel_shape* shape, const void* q, const void* K,
                                    const void* V, int32_t g, const void* K_new,
                                    const void* V_new, float* out, float* lse, void* stream) {
  using namespace kvsel;
  Plan p;
  kvsel_status st;
  if (g < 0) return KVSEL_ERR_INVALID_ARG;
  if ((st = plan_shape(shape, 0, &p))) return st;
  if (!decode_supported(p.dtype, p.D)) return KVSEL_ERR_UNSUPPORTED;
  if (p.S == 0) return KVSEL_OK;
  if (!q || !out || (p.T > 0 && (!K || !V)) || (g > 0 && (!K_new || !V_new)))
    return KVSEL_ERR_INVALID_ARG;
  for (const void* ptr : {q, K, V, K_new, V_new})
    if (reinterpret_cast<uintptr_t>(ptr) & 15) return KVSEL_ERR_INVALID_ARG;
  const int chunk = decode_chunk_rows();
  std::vector<DecSeq> seqs(p.S);
  int64_t items = 0;
  for (int b = 0; b < p.S; ++b) {
    const SeqDesc& sd = p.all[b];
    const int64_t n = (int64_t)sd.len + g;
    if (n == 0) return KVSEL_ERR_INVALID_ARG;
    if (n > 0x7fffffffLL) return KVSEL_ERR_UNSUPPORTED;
    DecSeq& d = seqs[b];
    d.row_off = sd.tok_off;
    d.n_rows = sd.len;
    d.n_chunks = (int32_t)((n + chunk - 1) / chunk);
    d.item_base = (int32_t)items;
    d.index = b;
    items += (int64_t)p.H * d.n_chunks;
    if (items > 0x7fffffffLL) return KVSEL_ERR_UNSUPPORTED;
  }
  if ((int64_t)p.layers * items > 0x7fffffffLL) return KVSEL_ERR_UNSUPPORTED;
  DevState* d;
  if ((st = device_state(&d))) return st;
  const size_t part_bytes = (size_t)p.layers * items * (2 + p.D) * sizeof(float);
  char* ws;
  if ((st = workspace(d, seqs.size() * sizeof(DecSeq) + part_bytes + 2 * 256, &ws))) return st;
  Carve cv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t o_seq = cv.take(seqs.size() * sizeof(DecSeq));
  const size_t o_part = cv.take(part_bytes);
  cudaError_t e = cudaMemcpyAsync(ws + o_seq, seqs.data(), seqs.size() * sizeof(DecSeq),
                                  cudaMemcpyHostToDevice, s);
  if (e) return cuda_fail(e, "cudaMemcpyAsync(decode sequence table)");
  DecodeArgs a{};
  a.q = q;
  a.k = K;
  a.v = V;
  a.k_new = K_new;
  a.v_new = V_new;
  a.layers = p.layers;
  a.S = p.S;
  a.H = p.H;
  a.Hkv = p.Hkv;
  a.D = p.D;
  a.dtype = p.dtype;
  a.g = g;
  a.T = p.T;
  a.seqs = reinterpret_cast<const DecSeq*>(ws + o_seq);
  a.items_per_layer = (int)items;
  a.chunk_rows = chunk;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p.D));
  a.part = reinterpret_cast<float*>(ws + o_part);
  a.out = out;
  a.lse = lse;
  a.status = d->status;
  a.stream = s;
  cudaEvent_t* ev = profile_slot();
  if (ev) cudaEventRecord(ev[0], s);
  e = launch_decode(a);
  if (ev) {
    cudaEventRecord(ev[1], s);
    cudaEventRecord(ev[2], s);
    cudaEventRecord(ev[3], s);
  }
  return cuda_fail(e, "decode attention launch");
}

kvsel_status kvsel_reverse_attention(const kvsel_shape* shape, const void* Q, const void* K,
                                     const void* V, const int32_t* positions, float* out,
                                     float* lse, void* stream) {
  using namespace kvsel;
  Plan p;
  kvsel_status st;
  if ((st = plan_shape(shape, 0, &p))) return st;
  if (p.T == 0) return KVSEL_OK;
  if (!Q || !K || !V || !out) return KVSEL_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(out) & 15) return KVSEL_ERR_INVALID_ARG;
  if (!reverse_eligible(p.dtype, p.D, Q, K, V)) return KVSEL_ERR_UNSUPPORTED;
  std::vector<RevSeq> seqs;
  int64_t items = 0;
  for (const SeqDesc& sd : p.all) {
    if (sd.len == 0) continue;
    RevSeq r{};
    r.tok_off = sd.tok_off;
    r.len = sd.len;
    r.n_qt = (sd.len + 127) / 128;
    r.item_base = (int32_t)items;
    items += (int64_t)p.H * r.n_qt;
    if (items > 0x7fffffffLL) return KVSEL_ERR_UNSUPPORTED;
    seqs.push_back(r);
  }
  if ((int64_t)p.layers * items > 0x7fffffffLL || (int64_t)p.layers * p.T >= 0x7fffffffLL)
    return KVSEL_ERR_UNSUPPORTED;
  DevState* d;
  if ((st = device_state(&d))) return st;
  char* ws;
  if ((st = workspace(d, seqs.size() * sizeof(RevSeq) + 256, &ws))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(ws, seqs.data(), seqs.size() * sizeof(RevSeq),
                                  cudaMemcpyHostToDevice, s);
  if (e) return cuda_fail(e, "cudaMemcpyAsync(reverse sequence table)");
  RevArgs a{};
  a.q = Q;
  a.k = K;
  a.v = V;
  a.pos = positions;
  a.out = out;
  a.lse = lse;
  a.layers = p.layers;
  a.H = p.H;
  a.Hkv = p.Hkv;
  a.S = (int)seqs.size();
  a.T = p.T;
  a.seqs = reinterpret_cast<const RevSeq*>(ws);
  a.items_per_layer = (int)items;
  a.status = d->status;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    a.wait_limit_ns = g_wait_limit_ns;
  }
  a.stream = s;
  cudaEvent_t* ev = profile_slot();
  if (ev) cudaEventRecord(ev[0], s);
  e = launch_reverse(a);
  if (ev) {
    cudaEventRecord(ev[1], s);
    cudaEventRecord(ev[2], s);
    cudaEventRecord(ev[3], s);
  }
  return cuda_fail(e, "reverse attention launch");
}

kvsel_status kvsel_decode_quality(int64_t n, int32_t D, const float* lse_keep,
                                  const float* lse_full, const float* out_keep,
                                  const float* out_full, float* mass, float* err, void* stream) {
  using namespace kvsel;
  if (n < 0 || D < 1) return KVSEL_ERR_INVALID_ARG;
  if (n == 0) return KVSEL_OK;
  if (!lse_keep || !lse_full || !out_keep || !out_full || !mass || !err)
    return KVSEL_ERR_INVALID_ARG;
  if (n > 0x7fffffffLL * 8) return KVSEL_ERR_UNSUPPORTED;
  DevState* d;
  kvsel_status st;
  if ((st = device_state(&d))) return st;
  QualityArgs a{};
  a.n = n;
  a.D = D;
  a.lse_keep = lse_keep;
  a.lse_full = lse_full;
  a.out_keep = out_keep;
  a.out_full = out_full;
  a.mass = mass;
  a.err = err;
  a.stream = static_cast<cudaStream_t>(stream);
  return cuda_fail(launch_decode_quality(a), "decode quality launch");
}

kvsel_status kvsel_cache_lengths(const kvsel_shape* shape, int32_t C, int32_t g,
                                 int64_t* physical_length, int64_t* next_logical) {
  using namespace kvsel;
  Plan p;
  kvsel_status st;
  if (C < 1 || g < 0) return KVSEL_ERR_INVALID_ARG;
  if ((st = plan_shape(shape, C, &p))) return st;
  if (p.S > 0 && (!physical_length || !next_logical)) return KVSEL_ERR_INVALID_ARG;
  for (int b = 0; b < p.S; ++b) {
    const int64_t L = p.all[b].len;
    physical_length[b] = std::min<int64_t>(L, C) + g;
    next_logical[b] = L + g;
  }
  return KVSEL_OK;
}

kvsel_status kvsel_snapkv(const kvsel_shape* shape, const void* q_win, const void* K,
                          const void* V, int32_t W, int32_t C, int32_t pool_kind,
                          int32_t pool_k, int32_t* out_idx, void* out_K, void* out_V,
                          void* stream) {
  return kvsel::snapkv_impl(shape, q_win, K, V, W, C, pool_kind, pool_k, out_idx, out_K, out_V,
                            stream, false);
}

kvsel_status kvsel_snapkv_grouped(const kvsel_shape* shape, const void* q_win, const void* K,
                                  const void* V, int32_t W, int32_t C, int32_t pool_kind,
                                  int32_t pool_k, int32_t* out_idx, void* out_K, void* out_V,
                                  void* stream) {
  return kvsel::snapkv_impl(shape, q_win, K, V, W, C, pool_kind, pool_k, out_idx, out_K, out_V,
                            stream, true);
}

// Host-buffer path: q_win and K are copied to the device one layer at a time
// on a copy stream (two slots, so the next layer's copy overlaps this layer's
// kernels); V and the outputs stay in pinned host memory, read and written in
// place by the gather (only the kept V rows cross the link).
kvsel_status kvsel_snapkv_host(const kvsel_shape* shape, const void* q_win, const void* K,
                               const void* V, int32_t W, int32_t C, int32_t pool_kind,
                               int32_t pool_k, int32_t* out_idx, void* out_K, void* out_V,
                               void* stream) {
  using namespace kvsel;
  Plan p;
  kvsel_status st;
  if (C < 1) return KVSEL_ERR_INVALID_ARG;
  if ((st = plan_shape(shape, C, &p))) return st;
  if ((st = check_window(p, W))) return st;
  if ((st = check_budget(W, C))) return st;
  if ((st = check_pool(pool_kind, pool_k))) return st;
  if (max_prefix(p, W, C) > kMaxPrefix) return KVSEL_ERR_UNSUPPORTED;
  if (p.T_out == 0) return KVSEL_OK;
  if (!q_win || !K || !V || !out_idx || !out_K || !out_V) return KVSEL_ERR_INVALID_ARG;
  // V and the outputs are read and written by the kernels in place: they
  // must be page-locked host memory (cudaHostAlloc / cudaHostRegister)
  void* dev_ptr[4];
  const void* host_ptr[4] = {V, out_idx, out_K, out_V};
  for (int i = 0; i < 4; ++i) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, host_ptr[i]) != cudaSuccess || at.type != cudaMemoryTypeHost ||
        cudaHostGetDevicePointer(&dev_ptr[i], const_cast<void*>(host_ptr[i]), 0) != cudaSuccess) {
      cudaGetLastError();
      return KVSEL_ERR_INVALID_ARG;
    }
  }
  DevState* d;
  if ((st = device_state(&d))) return st;
  const size_t eb = (size_t)p.elem_bytes;
  const size_t q_layer = (size_t)p.S * W * p.H * p.D * eb;
  const size_t k_layer = (size_t)p.T * p.Hkv * p.D * eb;
  const size_t slot = ((q_layer + 255) & ~size_t(255)) + ((k_layer + 255) & ~size_t(255));
  {
    std::lock_guard<std::mutex> lock(g_mu);
    cudaError_t e;
    if (d->stage_bytes < 2 * slot) {
      if (d->stage) {
        cudaDeviceSynchronize();
        cudaFree(d->stage);
        d->stage = nullptr;
        d->stage_bytes = 0;
      }
      if ((e = cudaMalloc(reinterpret_cast<void**>(&d->stage), 2 * slot)))
        return cuda_fail(e, "cudaMalloc(host-path staging)");
      d->stage_bytes = 2 * slot;
    }
    if (!d->copy) {
      if ((e = cudaStreamCreateWithFlags(&d->copy, cudaStreamNonBlocking)))
        return cuda_fail(e, "cudaStreamCreate(copy)");
      for (cudaEvent_t* ev : {&d->ev_entry, &d->ev_loaded[0], &d->ev_loaded[1], &d->ev_freed[0],
                              &d->ev_freed[1]})
        if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)))
          return cuda_fail(e, "cudaEventCreate");
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  // the copies start after the work already queued on the caller's stream
  if ((e = cudaEventRecord(d->ev_entry, s)) || (e = cudaStreamWaitEvent(d->copy, d->ev_entry, 0)))
    return cuda_fail(e, "stream ordering");
  kvsel_shape one = *shape;
  one.num_layers = 1;
  const int Hout = p.H;
  const size_t oi_layer = (size_t)p.T_out * Hout * sizeof(int32_t);
  const size_t o_layer = (size_t)p.T_out * Hout * p.D * eb;
  for (int l = 0; l < p.layers; ++l) {
    const int b = l & 1;
    char* qd = d->stage + b * slot;
    char* kd = qd + ((q_layer + 255) & ~size_t(255));
    if (l >= 2 && (e = cudaStreamWaitEvent(d->copy, d->ev_freed[b], 0)))
      return cuda_fail(e, "stream ordering");
    if ((e = cudaMemcpyAsync(qd, static_cast<const char*>(q_win) + l * q_layer, q_layer,
                             cudaMemcpyHostToDevice, d->copy)) ||
        (e = cudaMemcpyAsync(kd, static_cast<const char*>(K) + l * k_layer, k_layer,
                             cudaMemcpyHostToDevice, d->copy)) ||
        (e = cudaEventRecord(d->ev_loaded[b], d->copy)) ||
        (e = cudaStreamWaitEvent(s, d->ev_loaded[b], 0)))
      return cuda_fail(e, "host-path copy");
    st = snapkv_impl(&one, qd, kd, static_cast<const char*>(dev_ptr[0]) + l * k_layer, W, C,
                     pool_kind, pool_k,
                     reinterpret_cast<int32_t*>(static_cast<char*>(dev_ptr[1]) + l * oi_layer),
                     static_cast<char*>(dev_ptr[2]) + l * o_layer,
                     static_cast<char*>(dev_ptr[3]) + l * o_layer, stream, false);
    if (st) return st;
    if ((e = cudaEventRecord(d->ev_freed[b], s))) return cuda_fail(e, "stream ordering");
  }
  return KVSEL_OK;
}

kvsel_status kvsel_device_status(void* stream) {
  DevState* d;
  kvsel_status st;
  if ((st = device_state(&d))) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  if ((e = cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost)))
    return cuda_fail(e, "cudaMemcpy(status)");
  if ((e = cudaMemset(d->status, 0, sizeof(int)))) return cuda_fail(e, "cudaMemset(status)");
  return v;
}

kvsel_status kvsel_set_wait_limit_ns(uint64_t ns) {
  if (ns < 1000) return KVSEL_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  g_wait_limit_ns = ns;
  return KVSEL_OK;
}

kvsel_status kvsel_debug_inject(int32_t what) {
  if (what != 0 && what != 1) return KVSEL_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  g_inject = what;
  return KVSEL_OK;
}

kvsel_status kvsel_profile_begin(int32_t max_calls) {
  if (max_calls < 1 || max_calls > 100000) return KVSEL_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  for (cudaEvent_t e : g_prof.ev) cudaEventDestroy(e);
  g_prof = Profile();
  cudaError_t e = cudaGetDevice(&g_prof.device);
  if (e) return cuda_fail(e, "cudaGetDevice");
  g_prof.ev.resize(4 * (size_t)max_calls);
  for (auto& ev : g_prof.ev)
    if ((e = cudaEventCreate(&ev))) return cuda_fail(e, "cudaEventCreate");
  g_prof.capacity = max_calls;
  g_prof.armed = true;
  return KVSEL_OK;
}

kvsel_status kvsel_profile_end(double* stage_ms, int32_t* calls) {
  if (!stage_ms || !calls) return KVSEL_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  stage_ms[0] = stage_ms[1] = stage_ms[2] = 0.0;
  *calls = g_prof.used;
  kvsel_status st = KVSEL_OK;
  for (int c = 0; c < g_prof.used && st == KVSEL_OK; ++c) {
    cudaEvent_t* ev = &g_prof.ev[4 * (size_t)c];
    cudaError_t e = cudaEventSynchronize(ev[3]);
    for (int i = 0; i < 3 && !e; ++i) {
      float ms = 0.f;
      e = cudaEventElapsedTime(&ms, ev[i], ev[i + 1]);
      stage_ms[i] += ms;
    }
    if (e) st = cuda_fail(e, "cudaEventElapsedTime");
  }
  for (cudaEvent_t e : g_prof.ev) cudaEventDestroy(e);
  g_prof = Profile();
  return st;
}

void kvsel_release(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (int i = 0; i < kMaxDevices; ++i) {
    if (g_dev[i].ws || g_dev[i].stage) {
      cudaSetDevice(i);
      cudaDeviceSynchronize();
      cudaFree(g_dev[i].ws);
      cudaFree(g_dev[i].stage);
      g_dev[i].ws = g_dev[i].stage = nullptr;
      g_dev[i].ws_bytes = g_dev[i].stage_bytes = 0;
    }
  }
  cudaSetDevice(cur);
}

int64_t kvsel_workspace_bytes(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  return (int64_t)(g_dev[dev].ws_bytes + g_dev[dev].stage_bytes);
}

}  // extern "C"
