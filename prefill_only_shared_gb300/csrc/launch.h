// Internal launcher interfaces between the ABI layer (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "desc.h"

namespace sp {

struct AttnLaunch {
  const DescHeader* hdr;
  const void* dev_desc;
  int64_t tile_off, n_tiles, merge_off, n_merges;
  int32_t n_parts;
  int32_t round;  // the call's round, -1 for all rounds
  int32_t kind;   // 0 prefix, 1 branch
  const void* q;
  const void* k;
  const void* v;
  void* pool;
  void* out;
  float* lse;
  void* workspace;
  int Hq, Hkv, head_dim;
  int64_t node_tokens;  // rows of q/out (bounds the Q tensor map)
  int64_t pool_pages;   // pages the plan uses (bounds the pool tensor maps)
  unsigned* err;
  void* stream;
  int* launches;
};

cudaError_t attn_run_call(const AttnLaunch& L);

struct LmheadLaunch {
  const void* h;
  const void* W;
  int N, H, V;
  const int32_t* label_off;
  const int32_t* label_ids;
  int32_t n_labels;
  float* logprobs;
  float* lse;
  void* workspace;
  size_t ws_bytes;
  unsigned* err;
  int n_sms;
  void* stream;
  int* launches;
};

// Workspace layout of the readout: partial (max, sum) per CTA and branch.
size_t lmhead_workspace_bytes(int N, int V, int n_sms);
cudaError_t lmhead_run(const LmheadLaunch& L);

// The readout with its scratch in the library's static device array (no
// allocation): up to kNoallocMaxCtas x kNoallocMaxBranches partial pairs, then
// the two counters.  The caller checks lmhead_noalloc_fits first.
constexpr int kNoallocMaxBranches = 1024;
constexpr int kNoallocMaxCtas = 256;
constexpr size_t kNoallocScratchBytes =
    (size_t)kNoallocMaxCtas * kNoallocMaxBranches * 8 /* float2 */ + 256;
bool lmhead_noalloc_fits(int N, int V, int n_sms);
cudaError_t lmhead_run_noalloc(LmheadLaunch L);

cudaError_t label_softmax_run(const float* logprobs, const int32_t* label_off, int N, float* probs,
                              int32_t* argmax, unsigned* err, void* stream);
cudaError_t label_decide_run(const float* logprobs, const int32_t* label_off, const int32_t* qtype,
                             int N, float* probs, int32_t* argmax, float* value, float* conf,
                             unsigned* err, void* stream);
cudaError_t candidate_decide_run(const float* probs, const int32_t* label_off, int n_branches,
                                 const int32_t* cand_off, const int32_t* qtype, int Q, float* dist,
                                 int32_t* argmax, float* value, float* conf, unsigned* err,
                                 void* stream);

cudaError_t option_softmax_run(const float* row_lp, int n_rows, const int32_t* opt_off,
                               int n_opts, const int32_t* q_off, int Q, const float* prior,
                               float* scores, float* probs, int32_t* argmax, unsigned* err,
                               void* stream);

// One thread polls *flag until it equals `expect` or limit_ns (clamped to
// 1 us .. kWaitLimitNs) passes; on timeout the device error word gets
// kErrTimeout.
cudaError_t wait_flag_run(const unsigned* flag, unsigned expect, unsigned long long limit_ns,
                          unsigned* err, void* stream);

// cuTensorMapEncodeTiled, fetched from the driver through the runtime.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();

// cuTensorMapEncodeTiled with element strides 1 and no interleave, through a
// per-thread cache of recent encodings.  `fill`: what a load reads outside
// the tensor (zeros by default; NaN for maps whose out-of-range reads can
// only come from a bad descriptor, so such reads poison the results).
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                  CUtensorMapSwizzle swz, CUtensorMapL2promotion l2,
                  CUtensorMapFloatOOBfill fill = CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);

// Raise a kernel's dynamic shared memory limit, once per kernel and device.
cudaError_t ensure_dynamic_smem(const void* func, int bytes);

}  // namespace sp
