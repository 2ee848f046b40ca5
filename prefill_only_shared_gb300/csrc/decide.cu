// Label softmax and the question-type decision.
//
// Sources:
// * openjev-sglang article (jdon.com): request flow step 5 and the worked
//   yes/no example (stable softmax over the label log-probabilities); the
//   section on the three question types (noul -> P(yes), choice -> argmax and
//   distribution, score -> sum_i i * P_i with i from 0); the confidence
//   section (1 - H(P) / ln K, H the entropy in nats).
// * LLM2Jev page, on why the same material is computed many times and on the
//   outputs: every choice option and score level is its own yes/no input and
//   the final answers are read after normalisation.
//
// * openjev-multimodal "performance" page, section on next steps: multi-token
//   option scoring and label-prior calibration (read as the chain-rule sum of
//   the option tokens' log-probabilities, minus an optional prior, then the
//   stable softmax over the question's options).
//
// One warp per branch (or per question), at most 64 options: two per lane.
#include "../../include/sp.h"
#include "common.cuh"
#include "launch.h"

namespace sp {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fc00000); }

// Lowest-index argmax over the two values each lane holds (index lane and
// lane + 32); every lane returns the warp's winner.
__device__ __forceinline__ void warp_argmax(float x0, float x1, int lane, float& bv, int& bi) {
  bv = x0;
  bi = lane;
  if (x1 > bv) {
    bv = x1;
    bi = lane + 32;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(kFull, bv, o);
    const int oi = __shfl_xor_sync(kFull, bi, o);
    if (ov > bv || (ov == bv && oi < bi)) {
      bv = ov;
      bi = oi;
    }
  }
}

// Entropy term -p ln p with 0 ln 0 = 0.
__device__ __forceinline__ float plogp_neg(float p) { return p > 0.f ? -p * logf(p) : 0.f; }

// Label softmax (and, with kDecide, the question-type value and confidence),
// one warp per branch.
template <bool kDecide>
__global__ void __launch_bounds__(128) label_softmax_kernel(const float* lp, const int32_t* off,
                                                            const int32_t* qtype, int N,
                                                            float* probs, int32_t* argmax,
                                                            float* value, float* conf,
                                                            unsigned* err) {
  const int n = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (n >= N) return;
  const int a0 = off[n], k = off[n + 1] - a0;
  if (k < 2 || k > 64) {
    for (int j = lane; j < (k > 0 ? k : 0); j += 32) probs[a0 + j] = qnan();
    if (lane == 0) {
      argmax[n] = -1;
      if (kDecide) {
        value[n] = qnan();
        conf[n] = qnan();
      }
      raise_error(err, kErrBounds);
    }
    return;
  }
  const float x0 = lane < k ? lp[a0 + lane] : -INFINITY;
  const float x1 = lane + 32 < k ? lp[a0 + lane + 32] : -INFINITY;
  float m;
  int bi;
  warp_argmax(x0, x1, lane, m, bi);
  const float e0 = lane < k ? __expf(x0 - m) : 0.f;
  const float e1 = lane + 32 < k ? __expf(x1 - m) : 0.f;
  const float s = warp_sum(e0 + e1);
  const float inv = 1.f / s;
  const float p0 = e0 * inv, p1 = e1 * inv;
  if (lane < k) probs[a0 + lane] = p0;
  if (lane + 32 < k) probs[a0 + lane + 32] = p1;
  if (lane == 0) argmax[n] = bi;
  if constexpr (kDecide) {
    // ln p_i = (x_i - m) - ln s, so H = ln s - sum_i p_i (x_i - m); a label
    // whose exponential underflowed to 0 contributes 0.
    const float t = (e0 > 0.f ? p0 * (x0 - m) : 0.f) + (e1 > 0.f ? p1 * (x1 - m) : 0.f);
    const float ent = logf(s) - warp_sum(t);
    const float c = 1.f - ent / logf(static_cast<float>(k));
    const int qt = qtype[n];
    const float p_first = __shfl_sync(kFull, p0, 0);
    const float p_best = __shfl_sync(kFull, bi < 32 ? p0 : p1, bi & 31);
    const float sc = warp_sum(static_cast<float>(lane) * p0 + static_cast<float>(lane + 32) * p1);
    if (lane == 0) {
      float v;
      if (qt == SP_QTYPE_NOUL) {
        v = p_first;
      } else if (qt == SP_QTYPE_CHOICE) {
        v = p_best;
      } else if (qt == SP_QTYPE_SCORE) {
        v = sc;
      } else {
        v = qnan();
        raise_error(err, kErrBounds);
      }
      value[n] = v;
      conf[n] = c;
    }
  }
}

// One warp per question over its candidate branches' P(yes).
__global__ void __launch_bounds__(128) candidate_decide_kernel(
    const float* probs, const int32_t* label_off, int n_branches, const int32_t* cand_off,
    const int32_t* qtype, int Q, float* dist, int32_t* argmax, float* value, float* conf,
    unsigned* err) {
  const int q = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (q >= Q) return;
  const int a = cand_off[q], b = cand_off[q + 1], total = cand_off[Q];
  const int K = b - a;
  const int qt = qtype[q];
  // The question's own range lies inside [0, total) and total <= n_branches:
  // then every dist / label_off index below is in bounds.
  const bool range_ok = a >= 0 && K >= 0 && b <= total && total <= n_branches;
  const bool count_ok = qt == SP_QTYPE_NOUL ? K == 1
                        : (qt == SP_QTYPE_CHOICE || qt == SP_QTYPE_SCORE) ? (K >= 2 && K <= 64)
                                                                            : false;
  if (!range_ok || !count_ok) {
    if (range_ok)
      for (int j = lane; j < K; j += 32) dist[a + j] = qnan();
    if (lane == 0) {
      argmax[q] = -1;
      value[q] = qnan();
      conf[q] = qnan();
      raise_error(err, kErrBounds);
    }
    return;
  }
  if (qt == SP_QTYPE_NOUL) {
    if (lane == 0) {
      const float y = probs[label_off[a]];
      dist[a] = y;
      argmax[q] = 0;
      value[q] = y;
      conf[q] = 1.f - (plogp_neg(y) + plogp_neg(1.f - y)) / logf(2.f);
    }
    return;
  }
  const bool h0 = lane < K, h1 = lane + 32 < K;
  const float y0 = h0 ? probs[label_off[a + lane]] : 0.f;
  const float y1 = h1 ? probs[label_off[a + lane + 32]] : 0.f;
  float ym;
  int bi;
  warp_argmax(h0 ? y0 : -INFINITY, h1 ? y1 : -INFINITY, lane, ym, bi);
  const float inv = 1.f / warp_sum(y0 + y1);
  const float d0 = y0 * inv, d1 = y1 * inv;
  if (h0) dist[a + lane] = d0;
  if (h1) dist[a + lane + 32] = d1;
  const float ent = warp_sum(plogp_neg(d0) + plogp_neg(d1));
  const float c = 1.f - ent / logf(static_cast<float>(K));
  const float d_best = __shfl_sync(kFull, bi < 32 ? d0 : d1, bi & 31);
  const float sc = warp_sum(static_cast<float>(lane) * d0 + static_cast<float>(lane + 32) * d1);
  if (lane == 0) {
    argmax[q] = bi;
    value[q] = qt == SP_QTYPE_CHOICE ? d_best : sc;
    conf[q] = c;
  }
}

// Option scores and their calibrated softmax, one warp per question.  Lane l
// sums the rows of options l and l + 32 of the question (their token
// log-probabilities, in token order), subtracts the option's prior, and the
// warp takes the stable softmax and the lowest-index argmax.
__global__ void __launch_bounds__(128) option_softmax_kernel(
    const float* row_lp, int n_rows, const int32_t* opt_off, int n_opts, const int32_t* q_off,
    int Q, const float* prior, float* scores, float* probs, int32_t* argmax, unsigned* err) {
  const int q = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (q >= Q) return;
  const int a = q_off[q], b = q_off[q + 1], total = q_off[Q];
  const int K = b - a;
  // The question's options lie inside [0, total) and total <= n_opts: every
  // opt_off / prior / scores / probs index below is then in bounds.
  const bool range_ok = a >= 0 && K >= 0 && b <= total && total <= n_opts;
  bool bad = !range_ok || K < 2 || K > 64;
  float sc[2] = {0.f, 0.f}, x[2] = {-INFINITY, -INFINITY};
  if (!bad) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int j = lane + 32 * i;
      if (j >= K) continue;
      const int o = a + j;
      const int r0 = opt_off[o], r1 = opt_off[o + 1];
      if (r0 < 0 || r1 <= r0 || r1 > n_rows) {  // an empty option or rows out of range
        bad = true;
        continue;
      }
      float t = 0.f;
      for (int r = r0; r < r1; ++r) t += row_lp[r];
      sc[i] = t;
      x[i] = prior ? t - prior[o] : t;
    }
  }
  if (__any_sync(kFull, bad)) {
    if (range_ok)
      for (int j = lane; j < K; j += 32) {
        scores[a + j] = qnan();
        probs[a + j] = qnan();
      }
    if (lane == 0) {
      argmax[q] = -1;
      raise_error(err, kErrBounds);
    }
    return;
  }
  float m;
  int bi;
  warp_argmax(x[0], x[1], lane, m, bi);
  const float e0 = lane < K ? __expf(x[0] - m) : 0.f;
  const float e1 = lane + 32 < K ? __expf(x[1] - m) : 0.f;
  const float inv = 1.f / warp_sum(e0 + e1);
  if (lane < K) {
    scores[a + lane] = sc[0];
    probs[a + lane] = e0 * inv;
  }
  if (lane + 32 < K) {
    scores[a + lane + 32] = sc[1];
    probs[a + lane + 32] = e1 * inv;
  }
  if (lane == 0) argmax[q] = bi;
}

}  // namespace

cudaError_t option_softmax_run(const float* row_lp, int n_rows, const int32_t* opt_off,
                               int n_opts, const int32_t* q_off, int Q, const float* prior,
                               float* scores, float* probs, int32_t* argmax, unsigned* err,
                               void* stream) {
  option_softmax_kernel<<<(Q + 3) / 4, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      row_lp, n_rows, opt_off, n_opts, q_off, Q, prior, scores, probs, argmax, err);
  return cudaGetLastError();
}

cudaError_t label_softmax_run(const float* logprobs, const int32_t* label_off, int N, float* probs,
                              int32_t* argmax, unsigned* err, void* stream) {
  label_softmax_kernel<false><<<(N + 3) / 4, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      logprobs, label_off, nullptr, N, probs, argmax, nullptr, nullptr, err);
  return cudaGetLastError();
}

cudaError_t label_decide_run(const float* logprobs, const int32_t* label_off, const int32_t* qtype,
                             int N, float* probs, int32_t* argmax, float* value, float* conf,
                             unsigned* err, void* stream) {
  label_softmax_kernel<true><<<(N + 3) / 4, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      logprobs, label_off, qtype, N, probs, argmax, value, conf, err);
  return cudaGetLastError();
}

cudaError_t candidate_decide_run(const float* probs, const int32_t* label_off, int n_branches,
                                 const int32_t* cand_off, const int32_t* qtype, int Q, float* dist,
                                 int32_t* argmax, float* value, float* conf, unsigned* err,
                                 void* stream) {
  candidate_decide_kernel<<<(Q + 3) / 4, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      probs, label_off, n_branches, cand_off, qtype, Q, dist, argmax, value, conf, err);
  return cudaGetLastError();
}

}  // namespace sp
