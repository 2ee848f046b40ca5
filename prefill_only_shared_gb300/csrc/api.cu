// C-ABI entry points that touch the GPU: descriptor upload, the three
// attention calls (prefix, branch, whole tree), the label readout and
// softmax, the question-type and option decisions, the whole-pass calls
// (device or host buffers), the bounded flag wait and the device error word.
// Every argument is validated on the host before anything is launched.
#include <climits>
#include <cstring>
#include <mutex>

#include "../../include/sp.h"
#include "common.cuh"
#include "launch.h"
#include "plan_internal.h"

namespace {

// Sticky device error word (bits sp::kErrTimeout, sp::kErrBounds).
__device__ unsigned g_sp_error_word;

constexpr int kMaxDevices = 64;
thread_local int32_t t_last_launches = 0;

unsigned* error_word_ptr() {
  static unsigned* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sp_error_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned*>(p);
  }
  return ptrs[dev];
}

int sm_count() {
  static int counts[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
  if (!counts[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    counts[dev] = n;
  }
  return counts[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The host checks of sp_label_logprobs' arguments; the whole-pass calls make
// them before their first launch.
sp_status readout_args(const void* h, const void* W, int32_t N, int32_t H, int32_t V,
                       const int32_t* label_off, const int32_t* label_ids, int32_t n_labels,
                       const float* logprobs, const float* lse) {
  if (!h || !W || !label_off || !logprobs || !lse) return SP_ERR_ARG;
  if (N < 1 || N > 4096 || H < 8 || H % 8 || V < 2 || n_labels < 0) return SP_ERR_ARG;
  if (n_labels > 0 && !label_ids) return SP_ERR_ARG;
  if (!aligned16(h) || !aligned16(W)) return SP_ERR_ARG;
  return SP_OK;
}

sp_status attn_call(const sp_plan* P, const void* dev_desc, int32_t round, int kind, const void* q,
                    const void* k, const void* v, void* kv_pool, void* out, float* lse,
                    void* workspace, size_t ws_bytes, void* stream) {
  t_last_launches = 0;
  if (!P || !dev_desc || !q || !k || !v || !kv_pool || !out || !lse) return SP_ERR_ARG;
  if (round < -1 || round >= P->stats.n_rounds) return SP_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(kv_pool) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(dev_desc) & 255u))
    return SP_ERR_ARG;
  const int32_t r = round < 0 ? (int32_t)P->stats.n_rounds : round;
  const sp_plan::Call& c = P->calls[(size_t)sp_plan::kCallKinds * r + kind];
  const size_t need = (size_t)c.n_parts * P->shape.n_kv_heads * sp::kRowsPerTile *
                      (P->shape.head_dim + 1) * sizeof(float);
  if (need > 0 && (!workspace || ws_bytes < need || !aligned16(workspace)))
    return SP_ERR_WORKSPACE;
  sp::AttnLaunch L;
  L.hdr = &P->hdr;
  L.dev_desc = dev_desc;
  L.tile_off = c.tile_off;
  L.n_tiles = c.n_tiles;
  L.merge_off = c.merge_off;
  L.n_merges = c.n_merges;
  L.n_parts = c.n_parts;
  L.round = round;
  L.kind = kind;
  L.q = q;
  L.k = k;
  L.v = v;
  L.pool = kv_pool;
  L.out = out;
  L.lse = lse;
  L.workspace = workspace;
  L.Hq = P->shape.n_q_heads;
  L.Hkv = P->shape.n_kv_heads;
  L.head_dim = P->shape.head_dim;
  L.node_tokens = P->stats.node_tokens;
  L.pool_pages = P->pool_pages;
  L.err = error_word_ptr();
  if (!L.err) return SP_ERR_CUDA;
  L.stream = stream;
  int launches = 0;
  L.launches = &launches;
  cudaError_t e = sp::attn_run_call(L);
  t_last_launches = launches;
  return e == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

}  // namespace

namespace sp {
EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A tensor map is a host-side encoding of (base, shape, strides, box,
// swizzle): calls that pass the same buffers reuse the encoded map from a
// small per-thread table instead of encoding it again.
namespace {
struct MapKey {
  const void* base;
  uint32_t rank, dtype, swz, l2, fill;
  cuuint64_t dims[5];
  cuuint64_t strides[4];
  cuuint32_t box[5];
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool valid;
};
constexpr int kMapCache = 32;
}  // namespace

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                  CUtensorMapSwizzle swz, CUtensorMapL2promotion l2,
                  CUtensorMapFloatOOBfill fill) {
  if (rank < 1 || rank > 5) return false;
  MapKey k;
  std::memset(&k, 0, sizeof(k));
  k.base = base;
  k.rank = rank;
  k.dtype = (uint32_t)dtype;
  k.swz = (uint32_t)swz;
  k.l2 = (uint32_t)l2;
  k.fill = (uint32_t)fill;
  for (uint32_t i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  thread_local MapEntry cache[kMapCache];
  thread_local int next = 0;
  for (int i = 0; i < kMapCache; ++i)
    if (cache[i].valid && std::memcmp(&cache[i].key, &k, sizeof(k)) == 0) {
      *map = cache[i].map;
      return true;
    }
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  if (enc(map, dtype, rank, const_cast<void*>(base), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, l2, fill) != CUDA_SUCCESS)
    return false;
  MapEntry& e = cache[next];
  next = (next + 1) % kMapCache;
  e.key = k;
  e.map = *map;
  e.valid = true;
  return true;
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per kernel and device.
cudaError_t ensure_dynamic_smem(const void* func, int bytes) {
  struct Done {
    const void* func;
    int dev;
    int bytes;
  };
  static std::mutex mu;
  static Done done[64];
  static int n_done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done[i].func == func && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (n_done < 64) done[n_done++] = Done{func, dev, bytes};
  return cudaSuccess;
}
}  // namespace sp

extern "C" sp_status sp_plan_upload(const sp_plan* plan, void* dev_desc, size_t bytes,
                                    void* stream) {
  if (!plan || !dev_desc) return SP_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(dev_desc) & 255u) return SP_ERR_ARG;
  if (bytes < plan->blob.size()) return SP_ERR_WORKSPACE;
  cudaError_t e = cudaMemcpyAsync(dev_desc, plan->blob.data(), plan->blob.size(),
                                  cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

extern "C" sp_status sp_prefix_attn(const sp_plan* plan, const void* dev_desc, int32_t round,
                                    const void* q, const void* k, const void* v, void* kv_pool,
                                    void* out, float* lse, void* workspace, size_t ws_bytes,
                                    void* stream) {
  return attn_call(plan, dev_desc, round, 0, q, k, v, kv_pool, out, lse, workspace, ws_bytes,
                   stream);
}

extern "C" sp_status sp_branch_attn(const sp_plan* plan, const void* dev_desc, int32_t round,
                                    const void* q, const void* k, const void* v, void* kv_pool,
                                    void* out, float* lse, void* workspace, size_t ws_bytes,
                                    void* stream) {
  return attn_call(plan, dev_desc, round, 1, q, k, v, kv_pool, out, lse, workspace, ws_bytes,
                   stream);
}

extern "C" sp_status sp_tree_attn(const sp_plan* plan, const void* dev_desc, int32_t round,
                                    const void* q, const void* k, const void* v, void* kv_pool,
                                    void* out, float* lse, void* workspace, size_t ws_bytes,
                                    void* stream) {
  return attn_call(plan, dev_desc, round, 2, q, k, v, kv_pool, out, lse, workspace, ws_bytes,
                   stream);
}

extern "C" size_t sp_label_workspace_bytes(int32_t n_branches, int32_t vocab, int32_t n_sms) {
  if (n_branches <= 0 || vocab < 2) return 0;
  return sp::lmhead_workspace_bytes(n_branches, vocab, n_sms > 0 ? n_sms : sm_count());
}

extern "C" sp_status sp_label_logprobs(const void* h, const void* W, int32_t N, int32_t H,
                                       int32_t V, const int32_t* label_off,
                                       const int32_t* label_ids, int32_t n_labels, float* logprobs,
                                       float* lse, void* workspace, size_t ws_bytes,
                                       void* stream) {
  t_last_launches = 0;
  const sp_status arg = readout_args(h, W, N, H, V, label_off, label_ids, n_labels, logprobs, lse);
  if (arg != SP_OK) return arg;
  const int n_sms = sm_count();
  const size_t need = sp::lmhead_workspace_bytes(N, V, n_sms);
  if (!workspace || ws_bytes < need || !aligned16(workspace)) return SP_ERR_WORKSPACE;
  sp::LmheadLaunch L;
  L.h = h;
  L.W = W;
  L.N = N;
  L.H = H;
  L.V = V;
  L.label_off = label_off;
  L.label_ids = label_ids;
  L.n_labels = n_labels;
  L.logprobs = logprobs;
  L.lse = lse;
  L.workspace = workspace;
  L.ws_bytes = ws_bytes;
  L.err = error_word_ptr();
  L.n_sms = n_sms;
  L.stream = stream;
  int launches = 0;
  L.launches = &launches;
  if (!L.err) return SP_ERR_CUDA;
  cudaError_t e = sp::lmhead_run(L);
  t_last_launches = launches;
  return e == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

extern "C" sp_status sp_label_logprobs_noalloc(const void* h, const void* W, int32_t N, int32_t H,
                                               int32_t V, const int32_t* label_off,
                                               const int32_t* label_ids, int32_t n_labels,
                                               float* logprobs, float* lse, void* stream) {
  t_last_launches = 0;
  const sp_status arg = readout_args(h, W, N, H, V, label_off, label_ids, n_labels, logprobs, lse);
  if (arg != SP_OK) return arg;
  const int n_sms = sm_count();
  // the one size error of this entry point: the static scratch is too small
  if (!sp::lmhead_noalloc_fits(N, V, n_sms)) return SP_ERR_WORKSPACE;
  sp::LmheadLaunch L;
  L.h = h;
  L.W = W;
  L.N = N;
  L.H = H;
  L.V = V;
  L.label_off = label_off;
  L.label_ids = label_ids;
  L.n_labels = n_labels;
  L.logprobs = logprobs;
  L.lse = lse;
  L.workspace = nullptr;
  L.ws_bytes = 0;
  L.err = error_word_ptr();
  L.n_sms = n_sms;
  L.stream = stream;
  int launches = 0;
  L.launches = &launches;
  if (!L.err) return SP_ERR_CUDA;
  cudaError_t e = sp::lmhead_run_noalloc(L);
  t_last_launches = launches;
  return e == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

extern "C" sp_status sp_label_softmax(const float* logprobs, const int32_t* label_off, int32_t N,
                                      float* probs, int32_t* argmax, void* stream) {
  t_last_launches = 0;
  if (!logprobs || !label_off || !probs || !argmax || N < 1) return SP_ERR_ARG;
  unsigned* err = error_word_ptr();
  if (!err) return SP_ERR_CUDA;
  cudaError_t e = sp::label_softmax_run(logprobs, label_off, N, probs, argmax, err, stream);
  t_last_launches = 1;
  return e == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

extern "C" sp_status sp_label_decide(const float* logprobs, const int32_t* label_off,
                                     const int32_t* qtype, int32_t N, float* probs,
                                     int32_t* argmax, float* value, float* confidence,
                                     void* stream) {
  t_last_launches = 0;
  if (!logprobs || !label_off || !qtype || !probs || !argmax || !value || !confidence || N < 1)
    return SP_ERR_ARG;
  unsigned* err = error_word_ptr();
  if (!err) return SP_ERR_CUDA;
  cudaError_t e = sp::label_decide_run(logprobs, label_off, qtype, N, probs, argmax, value,
                                       confidence, err, stream);
  t_last_launches = 1;
  return e == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

extern "C" sp_status sp_candidate_decide(const float* probs, const int32_t* label_off,
                                         int32_t n_branches, const int32_t* cand_off,
                                         const int32_t* qtype, int32_t n_questions, float* dist,
                                         int32_t* argmax, float* value, float* confidence,
                                         void* stream) {
  t_last_launches = 0;
  if (!probs || !label_off || !cand_off || !qtype || !dist || !argmax || !value || !confidence ||
      n_branches < 1 || n_questions < 1)
    return SP_ERR_ARG;
  unsigned* err = error_word_ptr();
  if (!err) return SP_ERR_CUDA;
  cudaError_t e = sp::candidate_decide_run(probs, label_off, n_branches, cand_off, qtype,
                                           n_questions, dist, argmax, value, confidence, err,
                                           stream);
  t_last_launches = 1;
  return e == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

extern "C" sp_status sp_option_softmax(const float* row_logprobs, int32_t n_rows,
                                       const int32_t* opt_off, int32_t n_opts,
                                       const int32_t* q_off, int32_t n_questions,
                                       const float* prior, float* scores, float* probs,
                                       int32_t* argmax, void* stream) {
  t_last_launches = 0;
  if (!row_logprobs || !opt_off || !q_off || !scores || !probs || !argmax || n_rows < 1 ||
      n_opts < 2 || n_questions < 1)
    return SP_ERR_ARG;
  unsigned* err = error_word_ptr();
  if (!err) return SP_ERR_CUDA;
  cudaError_t e = sp::option_softmax_run(row_logprobs, n_rows, opt_off, n_opts, q_off,
                                         n_questions, prior, scores, probs, argmax, err, stream);
  t_last_launches = 1;
  return e == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

namespace {

// Plans a whole pass (without a page limit, so that a pool that is too small
// still reports the pages needed) and checks every capacity of sp_run_pass.
// On SP_OK *plan is the caller's to free; otherwise it is freed here.
sp_status plan_pass(const sp_shape* shape, int32_t n_branches, const int32_t* req_of_branch,
                    const int64_t* tok_offsets, const int32_t* tokens, int64_t node_rows,
                    int32_t pool_pages, size_t desc_bytes, size_t attn_ws_bytes,
                    size_t lm_ws_bytes, sp_plan** plan, sp_plan_stats* stats) {
  sp_status st = sp_plan_build(shape, n_branches, req_of_branch, tok_offsets, tokens, INT32_MAX,
                               sm_count(), plan);
  if (st != SP_OK) return st;
  sp_plan_stats ps;
  sp_plan_get_stats(*plan, &ps);
  if (stats) *stats = ps;
  const size_t lm_need = sp::lmhead_workspace_bytes(n_branches, shape->vocab, sm_count());
  if (ps.node_tokens != node_rows) st = SP_ERR_ARG;
  else if (ps.pages_used > pool_pages) st = SP_ERR_POOL_FULL;
  else if ((size_t)ps.desc_bytes > desc_bytes || (size_t)ps.attn_workspace_bytes > attn_ws_bytes ||
           lm_ws_bytes < lm_need)
    st = SP_ERR_WORKSPACE;
  if (st != SP_OK) {
    sp_plan_free(*plan);
    *plan = nullptr;
  }
  return st;
}

// The launches of a pass whose descriptor is already enqueued for upload:
// one tree attention call, the readout and the label softmax.
sp_status launch_pass(const sp_plan* plan, const sp_shape* shape, int32_t n_branches,
                      const void* desc, const void* q, const void* k, const void* v,
                      void* kv_pool, void* out, float* lse, void* attn_ws, size_t attn_ws_bytes,
                      const void* h, const void* W, const int32_t* label_off,
                      const int32_t* label_ids, int32_t n_labels, float* logprobs,
                      float* lse_vocab, void* lm_ws, size_t lm_ws_bytes, float* probs,
                      int32_t* argmax, void* stream) {
  int32_t launches = 0;
  sp_status st = sp_tree_attn(plan, desc, SP_ALL_ROUNDS, q, k, v, kv_pool, out, lse, attn_ws,
                              attn_ws_bytes, stream);
  launches += t_last_launches;
  if (st == SP_OK) {
    st = sp_label_logprobs(h, W, n_branches, shape->hidden, shape->vocab, label_off, label_ids,
                           n_labels, logprobs, lse_vocab, lm_ws, lm_ws_bytes, stream);
    launches += t_last_launches;
  }
  if (st == SP_OK) {
    st = sp_label_softmax(logprobs, label_off, n_branches, probs, argmax, stream);
    launches += t_last_launches;
  }
  t_last_launches = launches;
  return st;
}

}  // namespace

extern "C" sp_status sp_run_pass(const sp_shape* shape, int32_t n_branches,
                                   const int32_t* req_of_branch, const int64_t* tok_offsets,
                                   const int32_t* tokens, int64_t node_rows, const void* q,
                                   const void* k, const void* v, void* kv_pool, int32_t pool_pages,
                                   void* out, float* lse, void* desc, size_t desc_bytes,
                                   void* attn_ws, size_t attn_ws_bytes, const void* h,
                                   const void* W, const int32_t* label_off,
                                   const int32_t* label_ids, int32_t n_labels, float* logprobs,
                                   float* lse_vocab, void* lm_ws, size_t lm_ws_bytes,
                                   float* probs, int32_t* argmax, void* stream,
                                   sp_plan_stats* stats) {
  t_last_launches = 0;
  if (!shape || !probs || !argmax) return SP_ERR_ARG;
  sp_status st = readout_args(h, W, n_branches, shape->hidden, shape->vocab, label_off, label_ids,
                              n_labels, logprobs, lse_vocab);
  if (st != SP_OK) return st;
  sp_plan* plan = nullptr;
  st = plan_pass(shape, n_branches, req_of_branch, tok_offsets, tokens, node_rows,
                           pool_pages, desc_bytes, attn_ws_bytes, lm_ws_bytes, &plan, stats);
  if (st != SP_OK) return st;
  st = sp_plan_upload(plan, desc, desc_bytes, stream);
  if (st == SP_OK)
    st = launch_pass(plan, shape, n_branches, desc, q, k, v, kv_pool, out, lse, attn_ws,
                     attn_ws_bytes, h, W, label_off, label_ids, n_labels, logprobs, lse_vocab,
                     lm_ws, lm_ws_bytes, probs, argmax, stream);
  // the upload staged the descriptor out of the plan's (pageable) memory
  // before returning, so the plan can go
  sp_plan_free(plan);
  return st;
}

// One library-owned event per (device, descriptor buffer) that
// sp_run_pass_host has uploaded into: recorded after each pass that reads the
// buffer, waited for by the copy stream before the next upload into it.
// Events are created on first use (no device memory); the table keeps the
// most recent buffers and hands out a slot of the least recently used one
// when full (its event was recorded passes ago, so waiting on it costs
// nothing).
static cudaEvent_t desc_release_event(const void* desc) {
  struct Slot {
    const void* desc;
    int device;
    cudaEvent_t ev;
    uint64_t used;
  };
  constexpr int kSlots = 32;
  static Slot slots[kSlots] = {};
  static uint64_t clock = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  Slot* lru = &slots[0];
  for (Slot& x : slots) {
    if (x.ev && x.desc == desc && x.device == dev) {
      x.used = ++clock;
      return x.ev;
    }
    if (!x.ev || x.used < lru->used) lru = &x;
  }
  if (lru->ev && lru->device != dev) {
    cudaEventDestroy(lru->ev);  // an event belongs to its device
    lru->ev = nullptr;
  }
  if (!lru->ev && cudaEventCreateWithFlags(&lru->ev, cudaEventDisableTiming) != cudaSuccess) {
    lru->ev = nullptr;
    return nullptr;
  }
  lru->desc = desc;
  lru->device = dev;
  lru->used = ++clock;
  return lru->ev;
}

extern "C" sp_status sp_run_pass_host(
    const sp_shape* shape, int32_t n_branches, const int32_t* req_of_branch,
    const int64_t* tok_offsets, const int32_t* tokens, int64_t node_rows, const void* q_host,
    const void* k_host, const void* v_host, const void* h_host, const int32_t* label_off_host,
    const int32_t* label_ids_host, int32_t n_labels, const sp_input_set* set, void* kv_pool,
    int32_t pool_pages, void* out, float* lse, void* desc, size_t desc_bytes, void* attn_ws,
    size_t attn_ws_bytes, const void* W, float* logprobs, float* lse_vocab, void* lm_ws,
    size_t lm_ws_bytes, float* probs, int32_t* argmax, float* probs_host, int32_t* argmax_host,
    void* stream, void* copy_stream, sp_plan_stats* stats) {
  t_last_launches = 0;
  if (!shape || !set || !q_host || !k_host || !v_host || !h_host || !label_off_host ||
      !label_ids_host || !probs || !argmax || !probs_host || !argmax_host || !set->q || !set->k ||
      !set->v || !set->h || !set->label_off || !set->label_ids || !set->desc_host ||
      !set->done_event || !set->copied_event || !desc || n_branches < 1 || n_labels < 1)
    return SP_ERR_ARG;
  if (label_off_host[0] != 0 || label_off_host[n_branches] != n_labels) return SP_ERR_ARG;
  sp_status st = sp_check_labels(label_off_host, label_ids_host, n_branches, shape->vocab);
  if (st == SP_OK)
    st = readout_args(set->h, W, n_branches, shape->hidden, shape->vocab, set->label_off,
                      set->label_ids, n_labels, logprobs, lse_vocab);
  if (st != SP_OK) return st;
  sp_plan* plan = nullptr;
  st = plan_pass(shape, n_branches, req_of_branch, tok_offsets, tokens, node_rows, pool_pages,
                 desc_bytes, attn_ws_bytes, lm_ws_bytes, &plan, stats);
  if (st != SP_OK) return st;
  const size_t blob = plan->blob.size();
  if (node_rows > set->q_rows || n_branches > set->h_rows || n_labels > set->labels_cap ||
      blob > set->desc_host_bytes) {
    sp_plan_free(plan);
    return SP_ERR_WORKSPACE;
  }
  if (reinterpret_cast<uintptr_t>(desc) & 255u) {
    sp_plan_free(plan);
    return SP_ERR_ARG;
  }
  const auto done = static_cast<cudaEvent_t>(set->done_event);
  const auto copied = static_cast<cudaEvent_t>(set->copied_event);
  const auto cs = static_cast<cudaStream_t>(copy_stream);
  const auto ms = static_cast<cudaStream_t>(stream);
  // the last pass that used this set has read its inputs and its staged
  // descriptor (an event that was never recorded counts as done)
  if (cudaEventSynchronize(done) != cudaSuccess) {
    sp_plan_free(plan);
    return SP_ERR_CUDA;
  }
  std::memcpy(set->desc_host, plan->blob.data(), blob);
  const size_t e = 2;  // bf16
  const size_t q_bytes = (size_t)node_rows * shape->n_q_heads * shape->head_dim * e;
  const size_t kv_bytes = (size_t)node_rows * shape->n_kv_heads * shape->head_dim * e;
  const size_t h_bytes = (size_t)n_branches * shape->hidden * e;
  cudaError_t ce = cudaSuccess;
  const void* src[6] = {q_host, k_host, v_host, h_host, label_off_host, label_ids_host};
  void* dst[6] = {set->q, set->k, set->v, set->h, set->label_off, set->label_ids};
  const size_t bytes[6] = {q_bytes, kv_bytes, kv_bytes, h_bytes,
                           ((size_t)n_branches + 1) * sizeof(int32_t),
                           (size_t)n_labels * sizeof(int32_t)};
  for (int i = 0; i < 6 && ce == cudaSuccess; ++i)
    ce = cudaMemcpyAsync(dst[i], src[i], bytes[i], cudaMemcpyHostToDevice, cs);
  // The descriptor goes up on the copy stream too, right behind this pass's
  // inputs: on `stream` it would queue on the copy engine behind the next
  // call's input copies (enqueued meanwhile on the copy stream), and the pass
  // could not start before they end.  A pass that still reads the same
  // descriptor buffer (an earlier call's, when callers share one) finishes
  // first.
  cudaEvent_t desc_free = ce == cudaSuccess ? desc_release_event(desc) : nullptr;
  if (ce == cudaSuccess && !desc_free) ce = cudaErrorUnknown;
  if (ce == cudaSuccess) ce = cudaStreamWaitEvent(cs, desc_free, 0);
  if (ce == cudaSuccess)
    ce = cudaMemcpyAsync(desc, set->desc_host, blob, cudaMemcpyHostToDevice, cs);
  // however many copies were enqueued, they finish before anything `stream`
  // runs from here on, done_event included
  cudaError_t cw = cudaEventRecord(copied, cs);
  if (cw == cudaSuccess) cw = cudaStreamWaitEvent(ms, copied, 0);
  if (cw != cudaSuccess) cudaStreamSynchronize(cs);
  st = ce == cudaSuccess && cw == cudaSuccess ? SP_OK : SP_ERR_CUDA;
  if (st == SP_OK)
    st = launch_pass(plan, shape, n_branches, desc, set->q, set->k, set->v, kv_pool, out, lse,
                     attn_ws, attn_ws_bytes, set->h, W, set->label_off, set->label_ids, n_labels,
                     logprobs, lse_vocab, lm_ws, lm_ws_bytes, probs, argmax, stream);
  // the next upload into this descriptor buffer waits for this pass
  if (desc_free && cudaEventRecord(desc_free, ms) != cudaSuccess && st == SP_OK) st = SP_ERR_CUDA;
  sp_plan_free(plan);
  if (st == SP_OK &&
      (cudaMemcpyAsync(probs_host, probs, (size_t)n_labels * sizeof(float),
                       cudaMemcpyDeviceToHost, ms) != cudaSuccess ||
       cudaMemcpyAsync(argmax_host, argmax, (size_t)n_branches * sizeof(int32_t),
                       cudaMemcpyDeviceToHost, ms) != cudaSuccess))
    st = SP_ERR_CUDA;
  if (cudaEventRecord(done, ms) != cudaSuccess && st == SP_OK) st = SP_ERR_CUDA;
  return st;
}

extern "C" sp_status sp_wait_flag(const uint32_t* flag, uint32_t expect, int64_t limit_ns,
                                  void* stream) {
  t_last_launches = 0;
  if (!flag || (reinterpret_cast<uintptr_t>(flag) & 3u) || limit_ns < 0) return SP_ERR_ARG;
  unsigned* err = error_word_ptr();
  if (!err) return SP_ERR_CUDA;
  cudaError_t e = sp::wait_flag_run(flag, expect, static_cast<unsigned long long>(limit_ns), err,
                                    stream);
  t_last_launches = 1;
  return e == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

extern "C" sp_status sp_check_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SP_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_sp_error_word, sizeof(word)) != cudaSuccess)
    return SP_ERR_CUDA;
  if (word) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_sp_error_word, &zero, sizeof(zero)) != cudaSuccess)
      return SP_ERR_CUDA;
  }
  if (word & sp::kErrTimeout) return SP_ERR_DEVICE_TIMEOUT;
  if (word & sp::kErrBounds) return SP_ERR_DEVICE_BOUNDS;
  return SP_OK;
}

extern "C" int32_t sp_last_launch_count(void) { return t_last_launches; }
