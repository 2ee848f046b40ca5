// Shared-prefix (cascade) attention over the paged KV pool, on tcgen05.
//
// Sources: openjev-sglang article (jdon.com), sections on the radix cache and
// on the N+1 prefills (the shared prefix is computed once; every branch
// prefill reuses the prefix KV and computes only its own suffix), and the
// LLM2Jev "shared prefix" page (branches continue from the cached prefix).
//
// Work unit (one CTA): 128 query rows = (128 / G) consecutive tokens of one
// segment x the G query heads of one KV head (grouped-query packing: every KV
// tile loaded into shared memory serves all G heads).  The CTA walks the KV of
// the segment's ancestors (all keys visible) and then its own keys up to the
// causal bound, 128 keys (eight 16-token pages) per step.  Long contexts are
// split over several CTAs whose partial (O, lse) are merged by a log-sum-exp
// combine in a separate, fully parallel kernel (one warp per row).
//
// Roles (192 threads, one CTA per SM):
//   warps 0..3  softmax: one query row per thread (= TMEM lane); read S from
//               TMEM, mask, online max with lazy rescaling (the running max is
//               only moved when it grows by more than 2^8), P = exp2(S - m) in
//               bf16 into 128B-swizzled shared memory, rescale O in TMEM when
//               the max moved, final normalisation and store;
//   warp 4      TMA producer: Q tile once (3-D box: 64 dims x G heads x
//               128/G tokens), then per step eight K pages (128B swizzle) and
//               eight transposed V pages (32B swizzle) into a 2-stage ring,
//               lane p issuing page p, page ids fetched one step ahead;
//   warp 5      MMA issuer: S = Q K^T (M 128, N 128, K d) into one of two TMEM
//               buffers, then O += P V (M 128, N d, K 16 per page) into TMEM.
// The QK product of step j+1 runs on the tensor pipe while the softmax of
// step j runs.
#include "common.cuh"
#include "desc.h"
#include "launch.h"

namespace sp {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kThreads = 224;  // 4 softmax warps, K producer, MMA issuer, V producer
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kPages = kKeysPerUnit / kPageSize;  // pages per unit
constexpr float kRescaleLog2 = 8.f;  // move the running max only when it grows by > 2^8

// The PV product runs with N = D + 16: each transposed V page carries 16
// extra rows, the first all ones, so column D of O accumulates the row sum
// of the same bf16 P that weights V (the softmax denominator).
template <int D>
struct Cfg {
  static constexpr int kVRows = D + 16;                  // rows of a transposed V page block
  static constexpr int kQ = kRowsPerTile * D * 2;        // Q tile, slabs of 64 dims
  static constexpr int kK = kKeysPerUnit * D * 2;        // K tile
  static constexpr int kVPage = kVRows * 32;             // one transposed V page (16 keys)
  static constexpr int kV = kPages * kVPage;             // V^T tile
  static constexpr int kP = kRowsPerTile * kKeysPerUnit * 2;  // P tile, 2 slabs of 64 keys
  static constexpr int kSlab = kRowsPerTile * 128;       // one 64-wide bf16 slab of 128 rows
  static constexpr size_t kSmem =
      1024 + kQ + kP + (size_t)kKStages * kK + (size_t)kVStages * kV + 256;
  static constexpr uint32_t kColO = 2 * kKeysPerUnit;    // TMEM: S0 | S1 | O (D + 16 columns)
  static constexpr uint32_t kColSum = kColO + D;         // row sum of P
};

struct AttnArgs {
  const SegDesc* segs;
  const int32_t* page_ids;
  const int32_t* chain;
  const TileDesc* tiles;
  bf16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  unsigned* err;
  int Hq, Hkv, G;
  float scale_log2;  // log2(e) / sqrt(d)
};

// K-major operand, 32-byte swizzle: rows of 32 bytes (16 bf16 of K), 8-row
// groups 256 bytes apart, swizzle mode 6 = 32B.
__device__ __forceinline__ uint64_t umma_desc_k_sw32(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(256u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)6 << 61;
  return d;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_nohint(void* dst, const CUtensorMap* map, uint64_t* bar,
                                                   int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// 32 lanes x 32 columns, load and wait in one statement so no register is
// read before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// 2^x on the special-function unit (ex2.approx, flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float tmem_ld1_sync(uint32_t taddr) {
  uint32_t r;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r)
      : "r"(taddr)
      : "memory");
  return __uint_as_float(r);
}

__device__ __forceinline__ void tmem_st1_sync(uint32_t taddr, float v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(v))
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Walks the KV units of a tile: ancestor levels (root first), then the own
// segment up to the tile's causal bound.
struct Cursor {
  int level;     // 0..chain_len (chain_len = own segment)
  int j;         // unit within the level
  int n_units;   // units in this level
  int len;       // visible keys in this level (own: t0 + nt)
  int n_pages;   // pages the level's segment owns (page-table bound)
  int page_off;  // first page-table entry of the level's segment
  bool own;
};

__device__ __forceinline__ void cursor_level(Cursor& c, const AttnArgs& a, const SegDesc& sd,
                                             const TileDesc& td) {
  if (c.level < sd.chain_len) {
    const SegDesc an = a.segs[a.chain[sd.chain_off + c.level]];
    c.len = an.len;
    c.n_pages = (an.len + kPageSize - 1) / kPageSize;
    c.page_off = an.page_off;
    c.own = false;
  } else {
    c.len = td.t0 + td.nt;
    c.n_pages = (sd.len + kPageSize - 1) / kPageSize;
    c.page_off = sd.page_off;
    c.own = true;
  }
  c.n_units = (c.len + kKeysPerUnit - 1) / kKeysPerUnit;
}

__device__ __forceinline__ void cursor_next(Cursor& c, const AttnArgs& a, const SegDesc& sd,
                                            const TileDesc& td) {
  if (++c.j >= c.n_units && c.level < sd.chain_len) {
    c.level += 1;
    c.j = 0;
    cursor_level(c, a, sd, td);
  }
}

__device__ __forceinline__ Cursor cursor_at(const AttnArgs& a, const SegDesc& sd,
                                            const TileDesc& td) {
  Cursor c;
  c.level = 0;
  c.j = 0;
  cursor_level(c, a, sd, td);
  for (int u = 0; u < td.u_lo; ++u) cursor_next(c, a, sd, td);
  return c;
}

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                          ~uintptr_t(1023));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, AttnArgs a) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  unsigned char* sQ = smem;
  unsigned char* sP = sQ + C::kQ;
  unsigned char* sK = sP + C::kP;
  unsigned char* sV = sK + kKStages * C::kK;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + kVStages * C::kV);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + kKStages;
  uint64_t* v_full = k_empty + kKStages;
  uint64_t* v_empty = v_full + kVStages;
  uint64_t* s_full = v_empty + kVStages;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* drain = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const TileDesc td = a.tiles[blockIdx.x];
  const int hkv = blockIdx.y;
  const SegDesc sd = a.segs[td.seg];
  const int n_units = td.u_hi - td.u_lo;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // constant rows of every V page block: row D all ones, rows D+1.. zero
  for (int i = threadIdx.x; i < kVStages * kPages * 16 * 2; i += blockDim.x) {
    const int half = i & 1, row = (i >> 1) & 15, blk = i >> 5;
    const uint32_t one = row == 0 ? 0x3F803F80u : 0u;  // bf16 1.0 pairs
    *reinterpret_cast<uint4*>(sV + blk * C::kVPage + (D + row) * 32 + half * 16) =
        make_uint4(one, one, one, one);
  }
  fence_proxy_async_smem();
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4 || warp == 6) {
    if (n_units > 0) {
      // -------- TMA producers: warp 4 loads Q and K, warp 6 loads V --------
      // lane p < 8 issues page p of a unit; page ids are fetched one unit ahead
      const bool is_k = warp == 4;
      if (is_k && lane == 0) {
        prefetch_tensormap(&tmQ);
        prefetch_tensormap(&tmK);
        mbar_expect_tx(q_full, (uint32_t)C::kQ);
        for (int slab = 0; slab < D / 64; ++slab)
          tma_load_3d(sQ + slab * C::kSlab, &tmQ, q_full, slab * 64, hkv * a.G,
                      (int32_t)(sd.node_start + td.t0));
      }
      if (!is_k && lane == 0) prefetch_tensormap(&tmV);
      const int n_st = is_k ? kKStages : kVStages;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      const uint32_t bytes = is_k ? (uint32_t)C::kK : (uint32_t)(kPages * D * 32);
      Cursor cur = cursor_at(a, sd, td);
      auto page_of = [&](const Cursor& c) -> int {
        int pi = c.j * kPages + lane;
        if (pi >= c.n_pages) pi = c.n_pages - 1;  // finite filler; its keys are masked
        return a.page_ids[c.page_off + pi];
      };
      int page = lane < kPages ? page_of(cur) : 0;
      int s = 0;
      uint32_t ph = 0;
      int issued[kKStages > kVStages ? kKStages : kVStages];
      for (int i = 0; i < n_st; ++i) issued[i] = -1;
      bool ok = true;
      for (int it = 0; it < n_units; ++it) {
        int got = 1;
        if (lane == 0) got = mbar_wait(&empty[s], ph ^ 1, abort_flag) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_expect_tx(&full[s], bytes);
        __syncwarp();
        if (lane < kPages) {
          if (is_k) {
            unsigned char* dK = sK + s * C::kK;
            const int kb = (page * 2 + 0) * a.Hkv + hkv;
            for (int slab = 0; slab < D / 64; ++slab)
              tma_load_2d_nohint(dK + slab * C::kSlab + lane * (kPageSize * 128), &tmK, &full[s],
                                 slab * 64, kb * kPageSize);
          } else {
            const int vb = (page * 2 + 1) * a.Hkv + hkv;
            tma_load_2d_nohint(sV + s * C::kV + lane * C::kVPage, &tmV, &full[s], 0, vb * D);
          }
        }
        issued[s] = (int)ph;
        cursor_next(cur, a, sd, td);
        if (it + 1 < n_units && lane < kPages) page = page_of(cur);
        if (++s == n_st) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok && lane == 0) {
        if (!*abort_flag) raise_error(a.err, kErrTimeout);
        *abort_flag = 1;
        if (is_k) mbar_wait(q_full, 0, nullptr);
        for (int i = 0; i < n_st; ++i)
          if (issued[i] >= 0) mbar_wait(&full[i], (uint32_t)issued[i], nullptr);
      }
    }
  } else if (warp == 5) {
    if (lane == 0 && n_units > 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idesc_qk = umma_idesc_bf16_f32(kRowsPerTile, kKeysPerUnit);
      const uint32_t idesc_pv = umma_idesc_bf16_f32(kRowsPerTile, C::kVRows);
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t p_addr = smem_u32(sP);
      bool ok = mbar_wait(q_full, 0, abort_flag);
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;
      auto issue_pv = [&](int j) -> bool {
        if (!mbar_wait(p_full, (uint32_t)(j & 1), abort_flag)) return false;
        if (!mbar_wait(&v_full[vs], vph, abort_flag)) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(sV + vs * C::kV);
#pragma unroll
        for (int p = 0; p < kPages; ++p) {
          const uint64_t da = umma_desc_k_sw128(p_addr + (p >> 2) * C::kSlab + (p & 3) * 32);
          const uint64_t db = umma_desc_k_sw32(v_addr + p * C::kVPage);
          umma_bf16(tmem + C::kColO, da, db, idesc_pv, (j > 0 || p > 0) ? 1u : 0u);
        }
        umma_commit(&v_empty[vs]);
        umma_commit(pv_done);
        if (++vs == kVStages) {
          vs = 0;
          vph ^= 1;
        }
        return true;
      };
      for (int it = 0; it < n_units && ok; ++it) {
        const int sb = it & 1;
        if (!mbar_wait(&k_full[ks], kph, abort_flag) ||
            !mbar_wait(&s_empty[sb], (uint32_t)(((it >> 1) & 1) ^ 1), abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_addr = smem_u32(sK + ks * C::kK);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kSlab + (kk & 3) * 32;
          umma_bf16(tmem + (uint32_t)(sb * kKeysPerUnit), umma_desc_k_sw128(q_addr + off),
                    umma_desc_k_sw128(k_addr + off), idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(&k_empty[ks]);
        umma_commit(&s_full[sb]);
        if (++ks == kKStages) {
          ks = 0;
          kph ^= 1;
        }
        if (it > 0 && !issue_pv(it - 1)) {
          ok = false;
          break;
        }
      }
      if (ok) ok = issue_pv(n_units - 1);
      if (!ok) {
        if (!*abort_flag) raise_error(a.err, kErrTimeout);
        *abort_flag = 1;
      }
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else if (warp < 4 && n_units > 0) {
    // ---------------- softmax / epilogue (warps 0..3) ----------------
    const int r = threadIdx.x;  // query row = TMEM lane
    const int G = a.G;
    const int tok = r / G;
    const int token = td.t0 + tok;  // position within the own segment
    const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
    const float scale = a.scale_log2;
    float m_used = -INFINITY;  // running max, in scaled log2 units
    Cursor cur = cursor_at(a, sd, td);
    bool ok = true;
    for (int it = 0; it < n_units; ++it) {
      const int sb = it & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (uint32_t)((it >> 1) & 1), abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[kKeysPerUnit];
#pragma unroll
      for (int c = 0; c < kKeysPerUnit / 32; ++c) {
        float t[32];
        tmem_ld32(trow + (uint32_t)(sb * kKeysPerUnit + 32 * c), t);
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[32 * c + i] = t[i];
      }
      tc_fence_before();
      mbar_arrive(&s_empty[sb]);
      // visible keys of this row in this unit: c < lim
      const int key0 = cur.j * kKeysPerUnit;
      int lim = cur.len - key0;
      if (cur.own) lim = min(lim, token - key0 + 1);
      if (__any_sync(0xffffffffu, lim < kKeysPerUnit)) {
#pragma unroll
        for (int c = 0; c < kKeysPerUnit; ++c) sv[c] = c < lim ? sv[c] : -INFINITY;
      }
      float mt = sv[0];
#pragma unroll
      for (int c = 1; c < kKeysPerUnit; ++c) mt = fmaxf(mt, sv[c]);
      const float m_new = fmaxf(m_used, mt * scale);
      float alpha = 1.f;
      if (m_new > m_used + kRescaleLog2) {  // also true for the first finite max
        alpha = m_used == -INFINITY ? 0.f : ex2(m_used - m_new);
        m_used = m_new;
      }
      const float nbase = m_used == -INFINITY ? 0.f : -m_used;
#pragma unroll
      for (int c = 0; c < kKeysPerUnit; ++c) sv[c] = ex2(fmaf(sv[c], scale, nbase));
      if (it > 0 &&
          !__all_sync(0xffffffffu, mbar_wait(pv_done, (uint32_t)((it - 1) & 1), abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(trow + C::kColO + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(trow + C::kColO + 32 * c, o);
        }
        tmem_st1_sync(trow + C::kColSum, tmem_ld1_sync(trow + C::kColSum) * alpha);
      }
      // P row -> shared memory, bf16, 128B swizzle (2 slabs of 64 keys)
      unsigned char* prow = sP + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (int ch = 0; ch < kKeysPerUnit / 8; ++ch) {
        uint4 w;
        w.x = pack_bf16(sv[8 * ch + 0], sv[8 * ch + 1]);
        w.y = pack_bf16(sv[8 * ch + 2], sv[8 * ch + 3]);
        w.z = pack_bf16(sv[8 * ch + 4], sv[8 * ch + 5]);
        w.w = pack_bf16(sv[8 * ch + 6], sv[8 * ch + 7]);
        const int slab = ch >> 3, cc = ch & 7;
        *reinterpret_cast<uint4*>(prow + slab * C::kSlab + ((cc ^ (r & 7)) << 4)) = w;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
      cursor_next(cur, a, sd, td);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (uint32_t)((n_units - 1) & 1), abort_flag));
    if (!ok) {
      if (!*abort_flag) raise_error(a.err, kErrTimeout);
      *abort_flag = 1;
    } else {
      tc_fence_after();
      const float l = tmem_ld1_sync(trow + C::kColSum);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      const bool row_ok = tok < td.nt;
      const int head = hkv * G + (r % G);
      const size_t orow = (size_t)(sd.node_start + token) * a.Hq + head;
      const size_t prow_i = ((size_t)td.part * a.Hkv + hkv) * kRowsPerTile + r;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(trow + C::kColO + 32 * c, o);
        if (!row_ok) continue;
        if (td.part < 0) {
          uint4* dst = reinterpret_cast<uint4*>(a.out + orow * D + 32 * c);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv);
            w.y = pack_bf16(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv);
            w.z = pack_bf16(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv);
            w.w = pack_bf16(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv);
            dst[q4] = w;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(a.part_o + prow_i * D + 32 * c);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            dst[q4] = make_float4(o[4 * q4] * inv, o[4 * q4 + 1] * inv, o[4 * q4 + 2] * inv,
                                  o[4 * q4 + 3] * inv);
        }
      }
      if (row_ok) {
        if (td.part < 0)
          a.lse[orow] = lse;
        else
          a.part_lse[prow_i] = lse;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Combine the partial (O, lse) of split tiles: O = sum_i e^(lse_i - L) O_i,
// L = ln sum_i e^(lse_i).  One warp per query row (grid.x = merges x 16
// blocks of 8 rows, grid.y = KV head), lanes across head_dim; the loads of
// every part are in flight together.
template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const SegDesc* segs, const MergeDesc* merges,
                                                         const float* part_o, const float* part_lse,
                                                         bf16* out, float* lse_out, int Hq, int Hkv,
                                                         int G) {
  constexpr int PER = D / 32;
  constexpr int kBatch = 8;
  const MergeDesc md = merges[blockIdx.x >> 4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = (blockIdx.x & 15) * 8 + warp;
  const int hkv = blockIdx.y;
  if (row / G >= md.nt) return;
  const size_t step = (size_t)Hkv * kRowsPerTile;
  const size_t base = ((size_t)md.part0 * Hkv + hkv) * kRowsPerTile + row;
  float M = -INFINITY;
  for (int i = lane; i < md.nparts; i += 32) M = fmaxf(M, part_lse[base + i * step]);
  M = warp_max(M);
  float S = 0.f;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int i0 = 0; i0 < md.nparts; i0 += kBatch) {
    float li[kBatch];
    float x[kBatch][PER];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = i0 + j;
      li[j] = -INFINITY;
      if (i < md.nparts) {
        li[j] = part_lse[base + i * step];
        const float* src = part_o + (base + i * step) * D + lane * PER;
        if constexpr (PER == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          x[j][0] = v.x; x[j][1] = v.y; x[j][2] = v.z; x[j][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          x[j][0] = v.x; x[j][1] = v.y;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (li[j] == -INFINITY) continue;
      const float w = __expf(li[j] - M);
      S += w;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] += w * x[j][e];
    }
  }
  const float inv = S > 0.f ? 1.f / S : 0.f;
  const SegDesc sd = segs[md.seg];
  const size_t orow = (size_t)(sd.node_start + md.t0 + row / G) * Hq + hkv * G + (row % G);
#pragma unroll
  for (int e = 0; e < PER; e += 2)
    *reinterpret_cast<uint32_t*>(out + orow * D + lane * PER + e) =
        pack_bf16(acc[e] * inv, acc[e + 1] * inv);
  if (lane == 0) lse_out[orow] = S > 0.f ? M + __logf(S) : -INFINITY;
}

// Copy the K/V of one 16-token page of a segment, for one KV head (grid.y),
// into its pool page.  Pool page layout: K as [Hkv][16][D], V transposed as
// [Hkv][D][16]; slots past the segment end are zero-filled.
template <int D>
__global__ void __launch_bounds__(256) kv_append_kernel(const SegDesc* segs, const int32_t* page_ids,
                                                        const AppendDesc* app, const bf16* k,
                                                        const bf16* v, bf16* pool, int Hkv) {
  constexpr int CPR = D / 8;
  __shared__ __align__(16) bf16 sv[kPageSize][D + 8];
  const AppendDesc ad = app[blockIdx.x];
  const int h = blockIdx.y;
  const SegDesc sd = segs[ad.seg];
  const int tok0 = ad.page_in_seg * kPageSize;
  const int ntok = min(kPageSize, sd.len - tok0);
  const int page = page_ids[sd.page_off + ad.page_in_seg];
  const size_t kbase = (((size_t)page * 2) * Hkv + h) * kPageSize * D;
  const size_t vbase = (((size_t)page * 2 + 1) * Hkv + h) * (size_t)D * kPageSize;
  for (int i = threadIdx.x; i < kPageSize * CPR; i += blockDim.x) {
    const int ch = i % CPR, slot = i / CPR;
    uint4 kk = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
    if (slot < ntok) {
      const size_t src = ((size_t)(sd.node_start + tok0 + slot) * Hkv + h) * D + ch * 8;
      kk = *reinterpret_cast<const uint4*>(k + src);
      vv = *reinterpret_cast<const uint4*>(v + src);
    }
    *reinterpret_cast<uint4*>(pool + kbase + (size_t)slot * D + ch * 8) = kk;
    *reinterpret_cast<uint4*>(&sv[slot][ch * 8]) = vv;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < D * 2; i += blockDim.x) {
    const int dd = i >> 1, half = i & 1;
    uint4 w;
    bf16* e = reinterpret_cast<bf16*>(&w);
#pragma unroll
    for (int t = 0; t < 8; ++t) e[t] = sv[half * 8 + t][dd];
    *reinterpret_cast<uint4*>(pool + vbase + (size_t)dd * kPageSize + half * 8) = w;
  }
}

bool encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t run_call(const AttnLaunch& L) {
  const DescHeader& h = *L.hdr;
  const unsigned char* base = static_cast<const unsigned char*>(L.dev_desc);
  const SegDesc* segs = reinterpret_cast<const SegDesc*>(base + h.off_segs);
  const int32_t* pages = reinterpret_cast<const int32_t*>(base + h.off_pages);
  const int32_t* chain = reinterpret_cast<const int32_t*>(base + h.off_chain);
  const AppendDesc* app =
      reinterpret_cast<const AppendDesc*>(base + h.off_append) + L.append_off;
  const TileDesc* tiles = reinterpret_cast<const TileDesc*>(base + h.off_tiles) + L.tile_off;
  const MergeDesc* merges = reinterpret_cast<const MergeDesc*>(base + h.off_merges) + L.merge_off;
  cudaStream_t st = static_cast<cudaStream_t>(L.stream);
  bf16* pool = static_cast<bf16*>(L.pool);
  const int G = L.Hq / L.Hkv;
  int launches = 0;
  if (L.n_append > 0) {
    kv_append_kernel<D><<<dim3((unsigned)L.n_append, (unsigned)L.Hkv), 256, 0, st>>>(
        segs, pages, app, static_cast<const bf16*>(L.k), static_cast<const bf16*>(L.v), pool, L.Hkv);
    ++launches;
  }
  float* part_o = static_cast<float*>(L.workspace);
  float* part_lse = part_o + (size_t)L.n_parts * L.Hkv * kRowsPerTile * D;
  if (L.n_tiles > 0) {
    CUtensorMap tmQ, tmK, tmV;
    {
      cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L.Hq, (cuuint64_t)L.node_tokens};
      cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L.Hq * D * 2};
      cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(kRowsPerTile / G)};
      if (!encode(&tmQ, L.q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    const cuuint64_t blocks = (cuuint64_t)L.pool_pages * 2 * L.Hkv;
    {
      cuuint64_t dims[2] = {(cuuint64_t)D, blocks * kPageSize};
      cuuint64_t strides[1] = {(cuuint64_t)D * 2};
      cuuint32_t box[2] = {64, (cuuint32_t)kPageSize};
      if (!encode(&tmK, pool, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    {
      cuuint64_t dims[2] = {(cuuint64_t)kPageSize, blocks * D};
      cuuint64_t strides[1] = {(cuuint64_t)kPageSize * 2};
      cuuint32_t box[2] = {(cuuint32_t)kPageSize, (cuuint32_t)D};
      if (!encode(&tmV, pool, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_32B))
        return cudaErrorInvalidValue;
    }
    AttnArgs a;
    a.segs = segs;
    a.page_ids = pages;
    a.chain = chain;
    a.tiles = tiles;
    a.out = static_cast<bf16*>(L.out);
    a.lse = L.lse;
    a.part_o = part_o;
    a.part_lse = part_lse;
    a.err = L.err;
    a.Hq = L.Hq;
    a.Hkv = L.Hkv;
    a.G = G;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    const size_t smem = Cfg<D>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)L.n_tiles, (unsigned)L.Hkv);
    attn_tc_kernel<D><<<grid, kThreads, smem, st>>>(tmQ, tmK, tmV, a);
    ++launches;
  }
  if (L.n_merges > 0) {
    dim3 grid((unsigned)L.n_merges * 16, (unsigned)L.Hkv);
    attn_merge_kernel<D><<<grid, 256, 0, st>>>(segs, merges, part_o, part_lse,
                                               static_cast<bf16*>(L.out), L.lse, L.Hq, L.Hkv, G);
    ++launches;
  }
  *L.launches = launches;
  return cudaGetLastError();
}

}  // namespace

cudaError_t attn_run_call(const AttnLaunch& L) {
  if (L.head_dim == 64) return run_call<64>(L);
  return run_call<128>(L);
}

}  // namespace sp
