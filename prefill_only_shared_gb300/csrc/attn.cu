// Shared-prefix (cascade) attention over the paged KV pool.
//
// Sources: openjev-sglang article (jdon.com), sections on the radix cache and
// on the N+1 prefills (the shared prefix is computed once; every branch
// prefill reuses the prefix KV and computes only its own suffix), and the
// LLM2Jev "shared prefix" page (branches continue from the cached prefix).
//
// Work unit (one CTA): 128 query rows = (128 / G) consecutive tokens of one
// segment x the G query heads of one KV head (grouped-query packing: every KV
// tile loaded into shared memory serves all G heads).  The CTA walks the KV
// of the segment's ancestors (all keys visible) and then its own keys up to
// the causal bound, 64 keys (four 16-token pages) per step, with an online
// (max, sum) softmax in registers.  Long contexts are split over several CTAs
// whose partial (O, lse) are merged by a log-sum-exp combine.
#include "common.cuh"
#include "desc.h"
#include "launch.h"

namespace sp {
namespace {

using bf16 = __nv_bfloat16;

struct AttnArgs {
  const SegDesc* segs;
  const int32_t* page_ids;
  const int32_t* chain;
  const TileDesc* tiles;
  const bf16* q;
  const bf16* pool;
  bf16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  int Hq, Hkv, G;
  float scale_log2;  // log2(e) / sqrt(d)
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Element offset of 16-byte chunk c of row r in a [rows][D] bf16 tile whose
// chunks are XOR-swizzled by (r & 7), so ldmatrix rows hit distinct banks.
template <int D>
__device__ __forceinline__ int swz(int r, int c) {
  return r * D + ((c ^ (r & 7)) << 3);
}

struct Cursor {
  int level;     // 0..chain_len (chain_len = own segment)
  int j;         // unit within level
  int n_units;   // units in this level
  int len;       // keys in this level (own: causal bound of the tile)
  int page_off;  // first page-table entry of the level's segment
  bool own;
};

__device__ __forceinline__ void cursor_level(Cursor& c, const AttnArgs& a, const SegDesc& sd,
                                             const TileDesc& td) {
  if (c.level < sd.chain_len) {
    const SegDesc an = a.segs[a.chain[sd.chain_off + c.level]];
    c.len = an.len;
    c.page_off = an.page_off;
    c.own = false;
  } else {
    c.len = td.t0 + td.nt;
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

template <int D>
__device__ __forceinline__ void load_kv(const AttnArgs& a, const Cursor& c, int hkv, bf16* sK,
                                        bf16* sV) {
  constexpr int CPR = D / 8;
  const size_t kv_stride = (size_t)a.Hkv * kPageSize * D;
  for (int i = threadIdx.x; i < kKeysPerUnit * CPR; i += blockDim.x) {
    const int key = i / CPR, ch = i % CPR;
    const int pos = c.j * kKeysPerUnit + key;
    const bool valid = pos < c.len;
    const bf16* src = a.pool;
    if (valid) {
      const int page = a.page_ids[c.page_off + pos / kPageSize];
      src = a.pool + (((size_t)page * 2) * a.Hkv + hkv) * kPageSize * D +
            (size_t)(pos % kPageSize) * D + ch * 8;
    }
    cp_async16(sK + swz<D>(key, ch), src, valid);
    cp_async16(sV + swz<D>(key, ch), valid ? src + kv_stride : a.pool, valid);
  }
}

template <int D>
__global__ void __launch_bounds__(256, D == 64 ? 2 : 1) attn_mma_kernel(AttnArgs a) {
  constexpr int CPR = D / 8;
  constexpr int KS = D / 16;  // k-steps over head_dim
  constexpr int ON = D / 8;   // n-tiles over head_dim
  extern __shared__ __align__(128) unsigned char smem_raw[];
  bf16* sQ = reinterpret_cast<bf16*>(smem_raw);
  bf16* sK = sQ + kRowsPerTile * D;
  bf16* sV = sK + 2 * kKeysPerUnit * D;

  const TileDesc td = a.tiles[blockIdx.x];
  const int hkv = blockIdx.y;
  const SegDesc sd = a.segs[td.seg];
  const int G = a.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Q tile (gathered rows) -> shared memory
  for (int i = tid; i < kRowsPerTile * CPR; i += blockDim.x) {
    const int r = i / CPR, ch = i % CPR;
    const int tok = r / G;
    const bool valid = tok < td.nt;
    const bf16* src = a.q;
    if (valid)
      src = a.q + ((size_t)(sd.node_start + td.t0 + tok) * a.Hq + hkv * G + (r % G)) * D + ch * 8;
    cp_async16(sQ + swz<D>(r, ch), src, valid);
  }
  cp_async_commit();

  // position the cursor on unit u_lo
  Cursor cur;
  cur.level = 0;
  cur.j = 0;
  cursor_level(cur, a, sd, td);
  while (cur.level < sd.chain_len && cur.n_units == 0) {
    cur.level++;
    cursor_level(cur, a, sd, td);
  }
  for (int u = 0; u < td.u_lo; ++u) cursor_next(cur, a, sd, td);

  const int n_units = td.u_hi - td.u_lo;
  if (n_units > 0) load_kv<D>(a, cur, hkv, sK, sV);
  cp_async_commit();

  uint32_t qf[KS][4];
  float o[ON][4];
#pragma unroll
  for (int i = 0; i < ON; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  const int row0 = warp * 16 + (lane >> 2);
  const int tok_r[2] = {row0 / G, (row0 + 8) / G};

  for (int it = 0; it < n_units; ++it) {
    const int buf = it & 1;
    Cursor nxt = cur;
    const bool more = it + 1 < n_units;
    if (more) {
      cursor_next(nxt, a, sd, td);
      load_kv<D>(a, nxt, hkv, sK + (buf ^ 1) * kKeysPerUnit * D, sV + (buf ^ 1) * kKeysPerUnit * D);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (it == 0) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
        ldsm_x4(qf[ks], sQ + swz<D>(warp * 16 + (lane & 15), 2 * ks + (lane >> 4)));
    }
    const bf16* bK = sK + buf * kKeysPerUnit * D;
    const bf16* bV = sV + buf * kKeysPerUnit * D;

    // S = Q K^T (16 rows x 64 keys per warp)
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b[4];
        ldsm_x4(b, bK + swz<D>(16 * np + (lane & 7) + ((lane >> 4) << 3), 2 * ks + ((lane >> 3) & 1)));
        mma16816(s[2 * np], qf[ks], b[0], b[1]);
        mma16816(s[2 * np + 1], qf[ks], b[2], b[3]);
      }
    }
    // mask, scale, online softmax
    const int key0 = cur.j * kKeysPerUnit + 2 * (lane & 3);
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = key0 + nt * 8 + (e & 1);
        const int ri = e >> 1;
        bool ok = key < cur.len;
        if (cur.own) ok = ok && key <= td.t0 + tok_r[ri];
        const float v = ok ? s[nt][e] * a.scale_log2 : -INFINITY;
        s[nt][e] = v;
        mx[ri] = fmaxf(mx[ri], v);
      }
    }
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 1));
      mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 2));
    }
    float alpha[2], mu[2];
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      const float mn = fmaxf(m_run[ri], mx[ri]);
      mu[ri] = mn == -INFINITY ? 0.f : mn;
      alpha[ri] = exp2f(m_run[ri] - mu[ri]);
      m_run[ri] = mn;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ri = e >> 1;
        const float p = exp2f(s[nt][e] - mu[ri]);
        s[nt][e] = p;
        rs[ri] += p;
      }
    }
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) l_run[ri] = l_run[ri] * alpha[ri] + rs[ri];
#pragma unroll
    for (int nt = 0; nt < ON; ++nt) {
      o[nt][0] *= alpha[0];
      o[nt][1] *= alpha[0];
      o[nt][2] *= alpha[1];
      o[nt][3] *= alpha[1];
    }
    // O += P V
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * j][0], s[2 * j][1]);
      pa[1] = pack_bf16(s[2 * j][2], s[2 * j][3]);
      pa[2] = pack_bf16(s[2 * j + 1][0], s[2 * j + 1][1]);
      pa[3] = pack_bf16(s[2 * j + 1][2], s[2 * j + 1][3]);
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        uint32_t b[4];
        ldsm_x4_t(b, bV + swz<D>(16 * j + (lane & 7) + (((lane >> 3) & 1) << 3), 2 * dn + (lane >> 4)));
        mma16816(o[2 * dn], pa, b[0], b[1]);
        mma16816(o[2 * dn + 1], pa, b[2], b[3]);
      }
    }
    __syncthreads();  // buffer `buf` is refilled two iterations later
    cur = nxt;
  }
  cp_async_wait<0>();

  // finalize rows
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    float l = l_run[ri];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int row = row0 + 8 * ri;
    const int tok = tok_r[ri];
    if (tok >= td.nt) continue;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse = l > 0.f ? (m_run[ri] + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    const int head = hkv * G + (row % G);
    const size_t orow = (size_t)(sd.node_start + td.t0 + tok) * a.Hq + head;
    if (td.part < 0) {
#pragma unroll
      for (int nt = 0; nt < ON; ++nt) {
        const int d = nt * 8 + 2 * (lane & 3);
        *reinterpret_cast<uint32_t*>(a.out + orow * D + d) =
            pack_bf16(o[nt][2 * ri] * inv, o[nt][2 * ri + 1] * inv);
      }
      if ((lane & 3) == 0) a.lse[orow] = lse;
    } else {
      const size_t prow = ((size_t)td.part * a.Hkv + hkv) * kRowsPerTile + row;
#pragma unroll
      for (int nt = 0; nt < ON; ++nt) {
        const int d = nt * 8 + 2 * (lane & 3);
        *reinterpret_cast<float2*>(a.part_o + prow * D + d) =
            make_float2(o[nt][2 * ri] * inv, o[nt][2 * ri + 1] * inv);
      }
      if ((lane & 3) == 0) a.part_lse[prow] = lse;
    }
  }
}

// Combine the partial (O, lse) of split tiles: O = sum_i e^(lse_i - L) O_i,
// L = ln sum_i e^(lse_i).
template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const SegDesc* segs, const MergeDesc* merges,
                                                         const float* part_o, const float* part_lse,
                                                         bf16* out, float* lse_out, int Hq, int Hkv,
                                                         int G) {
  const MergeDesc md = merges[blockIdx.x];
  const int hkv = blockIdx.y;
  const SegDesc sd = segs[md.seg];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int PER = D / 32;
  for (int row = warp; row < kRowsPerTile; row += 8) {
    const int tok = row / G;
    if (tok >= md.nt) break;
    float M = -INFINITY;
    for (int i = 0; i < md.nparts; ++i)
      M = fmaxf(M, part_lse[((size_t)(md.part0 + i) * Hkv + hkv) * kRowsPerTile + row]);
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float S = 0.f;
    for (int i = 0; i < md.nparts; ++i) {
      const size_t prow = ((size_t)(md.part0 + i) * Hkv + hkv) * kRowsPerTile + row;
      const float li = part_lse[prow];
      if (li == -INFINITY) continue;
      const float w = __expf(li - M);
      S += w;
      const float* src = part_o + prow * D + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] += w * src[e];
    }
    const float inv = S > 0.f ? 1.f / S : 0.f;
    const size_t orow = (size_t)(sd.node_start + md.t0 + tok) * Hq + hkv * G + (row % G);
#pragma unroll
    for (int e = 0; e < PER; e += 2)
      *reinterpret_cast<uint32_t*>(out + orow * D + lane * PER + e) =
          pack_bf16(acc[e] * inv, acc[e + 1] * inv);
    if (lane == 0) lse_out[orow] = S > 0.f ? M + __logf(S) : -INFINITY;
  }
}

// Copy the K/V of one 16-token page of a segment into its pool page
// ([page][K|V][Hkv][16][D]); slots past the segment end are zero-filled.
template <int D>
__global__ void __launch_bounds__(256) kv_append_kernel(const SegDesc* segs, const int32_t* page_ids,
                                                        const AppendDesc* app, const bf16* k,
                                                        const bf16* v, bf16* pool, int Hkv) {
  constexpr int CPR = D / 8;
  const AppendDesc ad = app[blockIdx.x];
  const SegDesc sd = segs[ad.seg];
  const int tok0 = ad.page_in_seg * kPageSize;
  const int ntok = min(kPageSize, sd.len - tok0);
  const int page = page_ids[sd.page_off + ad.page_in_seg];
  const size_t kv_stride = (size_t)Hkv * kPageSize * D;
  const int total = Hkv * kPageSize * CPR;
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int ch = i % CPR;
    const int slot = (i / CPR) % kPageSize;
    const int h = i / (CPR * kPageSize);
    const size_t dst = (((size_t)page * 2) * Hkv + h) * kPageSize * D + (size_t)slot * D + ch * 8;
    uint4 kk = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
    if (slot < ntok) {
      const size_t src = ((size_t)(sd.node_start + tok0 + slot) * Hkv + h) * D + ch * 8;
      kk = *reinterpret_cast<const uint4*>(k + src);
      vv = *reinterpret_cast<const uint4*>(v + src);
    }
    *reinterpret_cast<uint4*>(pool + dst) = kk;
    *reinterpret_cast<uint4*>(pool + dst + kv_stride) = vv;
  }
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
  const bf16* k = static_cast<const bf16*>(L.k);
  const bf16* v = static_cast<const bf16*>(L.v);
  bf16* pool = static_cast<bf16*>(L.pool);
  int launches = 0;
  if (L.n_append > 0) {
    kv_append_kernel<D><<<(unsigned)L.n_append, 256, 0, st>>>(segs, pages, app, k, v, pool, L.Hkv);
    ++launches;
  }
  float* part_o = static_cast<float*>(L.workspace);
  float* part_lse = part_o + (size_t)L.n_parts * L.Hkv * kRowsPerTile * D;
  if (L.n_tiles > 0) {
    AttnArgs a;
    a.segs = segs;
    a.page_ids = pages;
    a.chain = chain;
    a.tiles = tiles;
    a.q = static_cast<const bf16*>(L.q);
    a.pool = pool;
    a.out = static_cast<bf16*>(L.out);
    a.lse = L.lse;
    a.part_o = part_o;
    a.part_lse = part_lse;
    a.Hq = L.Hq;
    a.Hkv = L.Hkv;
    a.G = L.Hq / L.Hkv;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    const size_t smem = (size_t)(kRowsPerTile + 4 * kKeysPerUnit) * D * sizeof(bf16);
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)L.n_tiles, (unsigned)L.Hkv);
    attn_mma_kernel<D><<<grid, 256, smem, st>>>(a);
    ++launches;
  }
  if (L.n_merges > 0) {
    dim3 grid((unsigned)L.n_merges, (unsigned)L.Hkv);
    attn_merge_kernel<D><<<grid, 256, 0, st>>>(segs, merges, part_o, part_lse,
                                               static_cast<bf16*>(L.out), L.lse, L.Hq, L.Hkv,
                                               L.Hq / L.Hkv);
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
