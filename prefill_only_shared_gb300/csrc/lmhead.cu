// Fused final-position LM-head readout: full-vocabulary log-sum-exp and the
// logits of the requested label ids, without writing logits to memory.
//
// Source: openjev-sglang article (jdon.com), section on what prefill-only
// means: the label log-probabilities at the last prompt position are the
// log-softmax over the whole vocabulary, read at the label ids.
//
// Data path (one persistent CTA per SM):
//   warp 0      TMA producer: W tile [128 vocab x 64 k] and h tile [nc x 64 k]
//               per pipeline stage (128-byte swizzle), W streamed evict-first;
//   warp 1      tcgen05.mma issuer: D[128 x nc] (fp32, TMEM) += W_tile . h_tile^T
//               over H / 64 stages; two accumulator buffers in TMEM;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one vocab row per
//               thread), per-column max / sum-of-exp over the 128 rows, merged
//               into a running (max, sum) per branch; label logits picked out
//               of TMEM when a label id falls in the tile.
// Work: vocab tiles x branch chunks ("units").  Each CTA first takes a fixed
// run of units, all CTAs together all but about two per CTA; the rest are
// taken one at a time from a global counter, so CTAs on SMs that stream
// faster take more of them.  The producer publishes each unit's index in a
// small shared-memory ring for the issuer and the epilogue.
// After a grid barrier (cooperative launch, one CTA per SM), every warp of
// the grid merges the per-CTA (max, sum) pairs of some branches into lse and
// turns their label logits into log-probabilities.
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "sp.h"

namespace sp {
namespace {

constexpr int kVT = 128;         // vocab rows per tile (MMA M)
constexpr int kKT = 64;          // hidden elements per stage (128 bytes of bf16)
constexpr int kWBytes = kVT * kKT * 2;
constexpr int kThreads = 192;
constexpr int kMaxStages = 16;
constexpr int kLabelCache = 4096;  // label bookkeeping entries kept in shared memory
constexpr size_t kSmemCap = 227 * 1024;

struct LmArgs {
  int N, H, V;
  int nc;       // branch columns per chunk (multiple of 16, <= 256)
  int n_ch;     // chunks
  int n_units;  // vocab tiles x chunks
  int stages;
  uint32_t tmem_cols;
  int n_labels;
  int lab_cap;  // entries of the shared-memory label branch map and local list
  const int32_t* label_off;
  const int32_t* label_ids;
  float* logits_out;  // raw label logits, [n_labels]; log-probabilities on exit
  float* lse;         // [N]
  float2* partials;   // [gridDim.x][N]
  unsigned* grid_arrivals;  // zero at launch
  unsigned* unit_counter;   // zero at launch: units taken from the shared tail
  int n_static;             // units of each CTA's fixed run
  unsigned* err;
};

constexpr int kUnitRing = 4;  // unit indices published ahead of the consumers

// A load with acquire semantics at GPU scope (a polling read of a flag that
// other CTAs update with atomics).
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__global__ void __launch_bounds__(kThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                  LmArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stage_bytes = kWBytes + a.nc * kKT * 2;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)a.stages * stage_bytes);
  uint64_t* empty = full + a.stages;
  uint64_t* acc_full = empty + a.stages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* unit_full = drain + 1;             // [kUnitRing]: a unit index is published
  uint64_t* unit_empty = unit_full + kUnitRing;  // [kUnitRing]: read by the issuer and 4 epilogue warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(unit_empty + kUnitRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* unit_ring = reinterpret_cast<int*>(tmem_slot + 2);  // [kUnitRing], -1 ends the sequence
  int* dyn_count = unit_ring + kUnitRing;                  // labels of the shared tail's rows
  float2* state = reinterpret_cast<float2*>(tmem_slot + 8);  // [4][N]
  // labels whose id falls in this CTA's vocab rows (indices into label_ids),
  // with their ids (so a tile's scan stays in shared memory), the branch of
  // every label j < lab_cap, and the list length
  int32_t* lab_list = reinterpret_cast<int32_t*>(state + 4 * a.N);     // [lab_cap]
  int32_t* lab_id = lab_list + a.lab_cap;                               // [lab_cap]
  uint16_t* lab_br = reinterpret_cast<uint16_t*>(lab_id + a.lab_cap);   // [lab_cap]
  int* lab_count = reinterpret_cast<int*>(lab_br + ((a.lab_cap + 1) & ~1));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's fixed run of units, then the shared tail [tail_lo, n_units)
  const int u_begin = blockIdx.x * a.n_static;
  const int u_end = u_begin + a.n_static;
  const int tail_lo = (int)gridDim.x * a.n_static;
  const int nk = (a.H + kKT - 1) / kKT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
    mbar_init(drain, 1);
    for (int r = 0; r < kUnitRing; ++r) {
      mbar_init(&unit_full[r], 1);
      mbar_init(&unit_empty[r], 5);
    }
    *abort_flag = 0;
    *lab_count = 0;
    *dyn_count = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmH);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, a.tmem_cols);
    tmem_relinquish();
  }
  if (warp >= 2) {
    const int q = warp & 3;
    for (int n = lane; n < a.N; n += 32) state[q * a.N + n] = make_float2(-INFINITY, 0.f);
    // branch of each label j < lab_cap: every thread walks its branches' labels
    for (int n = threadIdx.x - 64; n < a.N; n += 128) {
      const int j1 = min(a.label_off[n + 1], a.lab_cap);
      for (int j = max(a.label_off[n], 0); j < j1; ++j) lab_br[j] = (uint16_t)n;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    // W is streamed once: evict-first, except that a vocab tile read again
    // by the next branch chunk (its units are consecutive) stays in L2 until
    // its last chunk reads it
    const uint64_t pol_first = l2_policy_evict_first();
    const uint64_t pol_keep = l2_policy_evict_last();
    const uint64_t pol_h = l2_policy_evict_last();
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[kMaxStages];
    for (int i = 0; i < kMaxStages; ++i) issued_phase[i] = -1;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      // the unit: the fixed run first, then the shared tail
      int u = u_begin + i;
      if (i >= a.n_static) {
        u = tail_lo + (int)atomicAdd(a.unit_counter, 1u);
        if (u >= a.n_units) u = -1;
      }
      const int r = i % kUnitRing;
      const uint32_t ruse = (uint32_t)(i / kUnitRing);
      if (ruse > 0 && !mbar_wait(&unit_empty[r], (ruse - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      unit_ring[r] = u;
      mbar_arrive(&unit_full[r]);  // releases the write above
      if (u < 0) break;
      const int t = u / a.n_ch, c = u % a.n_ch;
      const uint64_t pol_w = c == a.n_ch - 1 ? pol_first : pol_keep;
      for (int k = 0; k < nk; ++k) {
        if (!mbar_wait(&empty[s], ph ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        mbar_expect_tx(&full[s], (uint32_t)stage_bytes);
        unsigned char* sw = smem + (size_t)s * stage_bytes;
        tma_load_2d(sw, &tmW, &full[s], k * kKT, t * kVT, pol_w);
        tma_load_2d(sw + kWBytes, &tmH, &full[s], k * kKT, c * a.nc, pol_h);
        issued_phase[s] = (int)ph;
        if (++s == a.stages) {
          s = 0;
          ph ^= 1;
        }
      }
    }
    if (!ok) {
      if (!*abort_flag) raise_error(a.err, kErrTimeout);
      *abort_flag = 1;
    }
    // let the copies already issued land before the CTA exits: after an
    // abort the issuer may not have read them all (on the normal path it
    // has, and these waits end at once)
    for (int i = 0; i < a.stages; ++i)
      if (issued_phase[i] >= 0) mbar_wait(&full[i], (uint32_t)issued_phase[i], nullptr);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = umma_idesc_bf16_f32(kVT, a.nc);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int r = i % kUnitRing;
      if (!mbar_wait(&unit_full[r], (uint32_t)(i / kUnitRing) & 1, abort_flag)) {
        ok = false;
        break;
      }
      const int u = unit_ring[r];
      mbar_arrive(&unit_empty[r]);
      if (u < 0) break;
      const int b = i & 1;
      const uint32_t use = (uint32_t)(i >> 1);
      if (!mbar_wait(&acc_empty[b], (use & 1) ^ 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(b * a.nc);
      for (int k = 0; k < nk; ++k) {
        if (!mbar_wait(&full[s], ph, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
        const uint64_t da = umma_desc_k_sw128(sa);
        const uint64_t db = umma_desc_k_sw128(sa + kWBytes);
#pragma unroll
        for (int kk = 0; kk < kKT / 16; ++kk)
          umma_bf16(d_tmem, da + 2 * kk, db + 2 * kk, idesc, (k | kk) != 0);
        umma_commit(&empty[s]);
        if (++s == a.stages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (ok) umma_commit(&acc_full[b]);
    }
    if (!ok) {
      if (!*abort_flag) raise_error(a.err, kErrTimeout);
      *abort_flag = 1;
    }
    // wait for every MMA issued by this thread before TMEM is released
    umma_commit(drain);
    mbar_wait(drain, 0, nullptr);
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    float2* st = state + q * a.N;
    // The labels whose id lies in this CTA's fixed run of vocab rows, and
    // those in the shared tail's rows, once (the stream is already filling
    // the pipeline): the first list from the front of lab_list, the second
    // from its back; each tile then checks only its list.
    {
      const int v_lo = (u_begin / a.n_ch) * kVT;
      const int v_hi = u_end > u_begin ? ((u_end - 1) / a.n_ch + 1) * kVT : v_lo;
      const int t_lo = (tail_lo / a.n_ch) * kVT;
      // one shared-memory atomic per warp and list (ballot, then each lane
      // takes its rank among the warp's matches)
      const unsigned below = (1u << lane) - 1u;
      for (int j0 = (warp - 2) * 32; j0 < a.n_labels; j0 += 128) {
        const int j = j0 + lane;
        const int id = j < a.n_labels ? a.label_ids[j] : -1;
        const bool in_run = id >= v_lo && id < v_hi;
        const bool in_tail = id >= t_lo && tail_lo < a.n_units;
        const unsigned m_run = __ballot_sync(0xffffffffu, in_run);
        const unsigned m_tail = __ballot_sync(0xffffffffu, in_tail);
        int b_run = 0, b_tail = 0;
        if (lane == 0) {
          if (m_run) b_run = atomicAdd(lab_count, __popc(m_run));
          if (m_tail) b_tail = atomicAdd(dyn_count, __popc(m_tail));
        }
        b_run = __shfl_sync(0xffffffffu, b_run, 0);
        b_tail = __shfl_sync(0xffffffffu, b_tail, 0);
        if (in_run) {
          const int k = b_run + __popc(m_run & below);
          if (k < a.lab_cap) {
            lab_list[k] = j;
            lab_id[k] = id;
          }
        }
        if (in_tail) {
          const int k = b_tail + __popc(m_tail & below);
          if (k < a.lab_cap) {
            lab_list[a.lab_cap - 1 - k] = j;
            lab_id[a.lab_cap - 1 - k] = id;
          }
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
    }
    const int n_fixed = *lab_count, n_tail = *dyn_count;
    const bool use_list = n_fixed + n_tail <= a.lab_cap;
    for (int i = 0;; ++i) {
      const int r = i % kUnitRing;
      if (!__all_sync(0xffffffffu, mbar_wait(&unit_full[r], (uint32_t)(i / kUnitRing) & 1, abort_flag))) {
        if (!*abort_flag) raise_error(a.err, kErrTimeout);
        *abort_flag = 1;
        break;
      }
      const int u = unit_ring[r];
      __syncwarp();
      if (lane == 0) mbar_arrive(&unit_empty[r]);  // after every lane's read
      if (u < 0) break;
      const bool in_tail = u >= tail_lo;
      const int n_local = in_tail ? n_tail : n_fixed;
      const int b = i & 1;
      const uint32_t use = (uint32_t)(i >> 1);
      if (!mbar_wait(&acc_full[b], use & 1, abort_flag)) {
        if (!*abort_flag) raise_error(a.err, kErrTimeout);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int t = u / a.n_ch, c = u % a.n_ch;
      const int v_base = t * kVT + 32 * q;
      const bool row_ok = v_base + lane < a.V;
      const uint32_t trow = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * a.nc);
      for (int g = 0; g < a.nc / 16; ++g) {
        const int col0 = c * a.nc + g * 16;
        if (col0 >= a.N) break;
        float x[16];
        tmem_ld16(trow + (uint32_t)(g * 16), x);
        float my_m = -INFINITY, my_s = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float xv = row_ok ? x[j] : -INFINITY;
          const float m = warp_max(xv);
          const float e = xv == -INFINITY ? 0.f : __expf(xv - m);
          const float sm = warp_sum(e);
          if (lane == j) {
            my_m = m;
            my_s = sm;
          }
        }
        if (lane < 16 && col0 + lane < a.N) {
          float2 cur = st[col0 + lane];
          lse_merge(cur.x, cur.y, my_m, my_s);
          st[col0 + lane] = cur;
        }
      }
      // label logits that fall in this warp's 32 vocab rows (from the local
      // list, or, when it overflowed, from the chunk's whole label range)
      const int n_lo = c * a.nc;
      const int n_hi = min(a.N, n_lo + a.nc);
      const int j_lo = use_list ? 0 : a.label_off[n_lo];
      const int j_hi = use_list ? n_local : a.label_off[n_hi];
      for (int jb = j_lo; jb < j_hi; jb += 32) {
        const int e = jb + lane;
        const int slot = in_tail ? a.lab_cap - 1 - e : e;
        const int j = e < j_hi ? (use_list ? lab_list[slot] : e) : -1;
        const int id = j < 0 ? -1 : use_list ? lab_id[slot] : a.label_ids[j];
        bool match = id >= v_base && id < v_base + 32 && id < a.V;
        int br = -1;
        if (match) {
          // branch of label j: the shared map, else the last n with
          // label_off[n] <= j (the chunk's range suffices outside list mode)
          if (j < a.lab_cap) {
            br = lab_br[j];
          } else {
            int lo = use_list ? 0 : n_lo, hi = use_list ? a.N - 1 : n_hi - 1;
            while (lo < hi) {
              const int mid = (lo + hi + 1) >> 1;
              if (a.label_off[mid] <= j) lo = mid; else hi = mid - 1;
            }
            br = lo;
          }
          match = br >= n_lo && br < n_hi;
        }
        unsigned bal = __ballot_sync(0xffffffffu, match);
        while (bal) {
          const int src = __ffs(bal) - 1;
          bal &= bal - 1;
          const int jj = __shfl_sync(0xffffffffu, j, src);
          const int idd = __shfl_sync(0xffffffffu, id, src);
          const int bb = __shfl_sync(0xffffffffu, br, src);
          const float y = tmem_ld1(trow + (uint32_t)(bb - n_lo));
          if (lane == idd - v_base) a.logits_out[jj] = y;
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[b]);
    }
    // merge the four lane quarters and publish this CTA's partials
    asm volatile("bar.sync 1, 128;" ::: "memory");
    for (int n = threadIdx.x - 64; n < a.N; n += 128) {
      float m = -INFINITY, s = 0.f;
      for (int qq = 0; qq < 4; ++qq) {
        const float2 v = state[qq * a.N + n];
        lse_merge(m, s, v.x, v.y);
      }
      a.partials[(size_t)blockIdx.x * a.N + n] = make_float2(m, s);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, a.tmem_cols);
  }

  // ---- grid barrier (the launch is cooperative: every CTA is resident) ----
  volatile int* go = abort_flag;  // reused as the barrier verdict
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(a.grid_arrivals, 1u);
    const unsigned long long t0 = globaltimer();
    int ok = 1;
    while (ld_acquire_gpu(a.grid_arrivals) < gridDim.x) {
      if (globaltimer() - t0 > kWaitLimitNs) {
        raise_error(a.err, kErrTimeout);
        ok = 0;
        break;
      }
    }
    __threadfence();
    *go = ok && !*abort_flag;
  }
  __syncthreads();
  if (!*go) return;

  // ---- finalize, one warp per branch across the grid: merge the per-CTA
  // (max, sum) pairs into lse and turn the label logits into log-probs ----
  const int n_warps = kThreads / 32;
  for (int n = blockIdx.x * n_warps + warp; n < a.N; n += gridDim.x * n_warps) {
    float m = -INFINITY, sum = 0.f;
    for (int p = lane; p < (int)gridDim.x; p += 32) {
      const float2 v = __ldcg(&a.partials[(size_t)p * a.N + n]);
      lse_merge(m, sum, v.x, v.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, sum, o);
      lse_merge(m, sum, m2, s2);
    }
    const float L = m + __logf(sum);
    if (lane == 0) a.lse[n] = L;
    for (int j = a.label_off[n] + lane; j < a.label_off[n + 1]; j += 32) {
      const int id = a.label_ids[j];
      if (id < 0 || id >= a.V) {
        a.logits_out[j] = __int_as_float(0x7fc00000);
        raise_error(a.err, kErrBounds);
      } else {
        a.logits_out[j] = __ldcg(&a.logits_out[j]) - L;
      }
    }
  }
}

struct Geometry {
  int nc, n_ch, n_units, grid, stages, lab_cap;
  size_t smem;
  uint32_t tmem_cols;
};

Geometry geometry(int N, int V, int n_sms, int n_labels = 0) {
  Geometry g{};
  g.n_ch = (N + 255) / 256;
  const int per = (N + g.n_ch - 1) / g.n_ch;
  g.nc = ((per + 15) / 16) * 16;
  const int n_vt = (V + kVT - 1) / kVT;
  g.n_units = n_vt * g.n_ch;
  g.grid = n_sms < g.n_units ? n_sms : g.n_units;
  const size_t stage = (size_t)kWBytes + (size_t)g.nc * kKT * 2;
  const size_t base = 1024 /*align slack*/ + (2 * kMaxStages + 5 + 2 * kUnitRing) * 8 + 32 +
                      (size_t)4 * N * 8;
  // the label cache takes only what is left after min(4, stages that fit
  // without it) pipeline stages
  const int st_free = base < kSmemCap ? (int)((kSmemCap - base) / stage) : 0;
  const int st_keep = st_free < 4 ? st_free : 4;
  const size_t room = base + (size_t)st_keep * stage < kSmemCap
                          ? kSmemCap - base - (size_t)st_keep * stage
                          : 0;
  int lab = n_labels < kLabelCache ? n_labels : kLabelCache;
  if ((size_t)lab * 10 + 32 > room) lab = room > 32 ? (int)((room - 32) / 10) : 0;
  g.lab_cap = lab;
  const size_t fixed = base + (size_t)g.lab_cap * 10 + 32;
  int st = (int)((kSmemCap - fixed) / stage);
  if (st > kMaxStages) st = kMaxStages;
  g.stages = st;
  g.smem = fixed + (size_t)st * stage;
  uint32_t cols = 32;
  while (cols < (uint32_t)(2 * g.nc)) cols <<= 1;
  g.tmem_cols = cols;
  return g;
}

bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_in,
               uint32_t box_out) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_in, box_out};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

}  // namespace

// Workspace: per-CTA partials [grid][N] float2, then the grid-barrier counter
// and the shared-tail unit counter (both zeroed by each call).
size_t lmhead_workspace_bytes(int N, int V, int n_sms) {
  Geometry g = geometry(N, V, n_sms > 0 ? n_sms : 152);
  return ((size_t)g.grid * N * sizeof(float2) + 16 + 255) & ~size_t(255);
}

cudaError_t lmhead_run(const LmheadLaunch& L) {
  Geometry g = geometry(L.N, L.V, L.n_sms, L.n_labels);
  if (g.stages < 2) return cudaErrorInvalidValue;
  CUtensorMap tmW, tmH;
  if (!encode_2d(&tmW, L.W, (uint64_t)L.H, (uint64_t)L.V, kKT, kVT)) return cudaErrorInvalidValue;
  if (!encode_2d(&tmH, L.h, (uint64_t)L.H, (uint64_t)L.N, kKT, (uint32_t)g.nc))
    return cudaErrorInvalidValue;
  LmArgs a;
  a.N = L.N;
  a.H = L.H;
  a.V = L.V;
  a.nc = g.nc;
  a.n_labels = L.n_labels;
  a.lab_cap = g.lab_cap;
  a.n_ch = g.n_ch;
  a.n_units = g.n_units;
  a.stages = g.stages;
  a.tmem_cols = g.tmem_cols;
  a.label_off = L.label_off;
  a.label_ids = L.label_ids;
  a.logits_out = L.logprobs;
  a.partials = static_cast<float2*>(L.workspace);
  a.grid_arrivals = reinterpret_cast<unsigned*>(a.partials + (size_t)g.grid * L.N);
  a.unit_counter = a.grid_arrivals + 1;
  // a fixed run per CTA; the last units (about two per CTA) are shared
  a.n_static = g.n_units / g.grid > 1 ? g.n_units / g.grid - 1 : 0;
  a.lse = L.lse;
  a.err = L.err;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(lmhead_kernel), (int)g.smem);
  if (e != cudaSuccess) return e;
  cudaStream_t st = static_cast<cudaStream_t>(L.stream);
  e = cudaMemsetAsync(a.grid_arrivals, 0, 2 * sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  void* args[] = {&tmW, &tmH, &a};
  e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(lmhead_kernel), dim3(g.grid),
                                  dim3(kThreads), args, g.smem, st);
  if (e != cudaSuccess) return e;
  *L.launches = 1;
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// No-allocation readout: the per-CTA partials and the two counters live in
// this file-scope device array (2 MiB + 256 bytes: up to 256 CTAs x 1024
// branches x one float2, then the counters), which every GPU
// that loads the library holds until exit.  Host code cannot use the array's
// name as a device address, so its address is looked up once per device (with
// that device current) and passed to the kernel like any workspace.  Calls
// share the array; each call writes every partial it reads, so nothing needs
// clearing, and overlapping calls would race.
static_assert(SP_NOALLOC_SCRATCH_BYTES == kNoallocScratchBytes,
              "the header's scratch size must be the array's");
static_assert(SP_NOALLOC_MAX_BRANCHES == kNoallocMaxBranches,
              "the header's branch limit must be the library's");
static_assert(sizeof(float2) == 8, "one partial pair is 8 bytes");
namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

cudaError_t noalloc_scratch_address(void** out) {
  constexpr int kMaxDevices = 64;
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}
}  // namespace

bool lmhead_noalloc_fits(int N, int V, int n_sms) {
  if (N < 1 || N > kNoallocMaxBranches) return false;
  if (n_sms > kNoallocMaxCtas) n_sms = kNoallocMaxCtas;
  return lmhead_workspace_bytes(N, V, n_sms) <= kNoallocScratchBytes;
}

cudaError_t lmhead_run_noalloc(LmheadLaunch L) {
  // the grid is capped so the partials fit the array (checked by the caller
  // through lmhead_noalloc_fits with the same cap)
  if (L.n_sms > kNoallocMaxCtas) L.n_sms = kNoallocMaxCtas;
  void* scratch = nullptr;
  cudaError_t e = noalloc_scratch_address(&scratch);
  if (e != cudaSuccess) return e;
  L.workspace = scratch;
  L.ws_bytes = kNoallocScratchBytes;
  return lmhead_run(L);
}

}  // namespace sp
