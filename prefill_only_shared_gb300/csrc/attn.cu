// Shared-prefix (cascade) attention over the paged KV pool, on tcgen05.
//
// Sources: openjev-sglang article (jdon.com), sections on the radix cache and
// on the N+1 prefills (the shared prefix is computed once; every branch
// prefill reuses the prefix KV and computes only its own suffix), and the
// LLM2Jev "shared prefix" page (branches continue from the cached prefix).
//
// Work unit (one CTA): 256 query rows = (256 / G) consecutive tokens of one
// segment x the G query heads of one KV head, as two 128-row halves A and B
// (grouped-query packing: every KV tile in shared memory serves 2 x 128 rows,
// which halves the L2 bytes per flop against one 128-row tile).  The CTA walks
// the KV of the segment's ancestors (all keys visible) and then its own keys
// up to the causal bound, 128 keys (eight 16-token pages) per step, starting at
// a rotated step so CTAs sharing a prefix spread their reads.  Long contexts
// are split over several CTAs whose partial (O, lse) are merged by a
// log-sum-exp combine in a separate, fully parallel kernel.
//
// Roles (384 threads, one CTA per SM):
//   warps 0..3 / 4..7  softmax of half A / half B: one query row per thread
//               (= TMEM lane); S from TMEM, mask, online max with lazy
//               rescaling (the running max only moves when it grows by more
//               than 2^8), row sums in fp32, P = exp2(S - m) written back as
//               bf16 pairs over the first 64 columns of S in TMEM, rescale of
//               O in TMEM when the max moved, final normalisation and store;
//   warp 8      TMA producer of Q (3-D boxes: 64 dims x G heads x 128/G
//               tokens per half) and of the K pages (128B swizzle, 3 stages);
//   warp 10     TMA producer of the V pages (128B swizzle, 2 stages); a unit
//               whose eight page ids are consecutive comes in one 4-D box per
//               64-dim slab, otherwise one box per page and slab;
//   warps 9 / 11  MMA issuers of half A / half B, per unit j: PV_h(j-1),
//               then QK_h(j), with S_h = Q_h K^T (M 128, N 128, K d, operands
//               in shared memory) and O_h += P_h V (M 128, N d, K 16 per page,
//               P_h read from TMEM, V an MN-major operand).  A K / V stage is
//               released when both halves' products that read it are done.
// The halves take turns on the tensor pipe (A0 B0 A1 B1 ...), so one half's
// softmax runs while the other half's products do.  Each half has its own
// issuing thread, which does its barrier waits while the other half's group
// runs: the pipe holds about one product ahead, so a wait between two issues
// would leave it idle.
#include "common.cuh"
#include "desc.h"
#include "launch.h"

namespace sp {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kThreads = 384;
constexpr int kHalf = 128;                        // rows per half tile (MMA M)
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kPages = kKeysPerUnit / kPageSize;  // pages per unit
constexpr float kRescaleLog2 = 8.f;  // move the running max only when it grows by > 2^8

template <int D>
struct Cfg {
  static constexpr int kQSlab = kHalf * 128;             // [128 rows x 64 dims] bf16
  static constexpr int kQHalf = (D / 64) * kQSlab;       // one half's Q tile
  static constexpr int kKSlab = kKeysPerUnit * 128;      // [128 keys x 64 dims] bf16
  static constexpr int kK = (D / 64) * kKSlab;           // K tile of one unit
  static constexpr int kV = (D / 64) * kKSlab;           // V tile of one unit (like K)
  static constexpr size_t kSmem =
      1024 + 2 * kQHalf + (size_t)kKStages * kK + (size_t)kVStages * kV + 512;
  // TMEM columns: S_A | S_B (128 each; P_h overwrites the first 64 columns of
  // S_h as packed bf16 pairs) | O_A | O_B (D each)
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColO = 2 * kKeysPerUnit;
};

struct AttnArgs {
  const SegDesc* segs;
  const int32_t* page_ids;
  const int32_t* chain;
  const TileDesc* tiles;
  const bf16* k_in;  // k / v inputs [node_tokens][Hkv][D]
  const bf16* v_in;
  bf16* pool;        // [page][K: Hkv x 16 x D | V: Hkv x 16 x D]
  int call_round;    // round of this call, -1 for all rounds
  int call_kind;     // 0 prefix (shared segments), 1 branch (leaves), 2 both
  bf16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  unsigned* err;
  int Hq, Hkv, G;
  float scale_log2;  // log2(e) / sqrt(d)
  // bounds of the descriptor's indices, checked on the device: rows of the
  // q / k / v / out inputs, pages of the pool, page-table entries, partial slots
  int64_t node_tokens;
  int64_t pool_pages;
  int64_t n_page_entries;
  int32_t n_parts;
};

// MN-major operand, 128-byte swizzle (V as the B operand of P.V: rows are
// keys = K, 128-byte rows hold 64 consecutive head dims = N): 8-row K groups
// 1024 bytes apart (stride byte offset), 64-column N slabs `slab_bytes` apart
// (leading byte offset), swizzle mode 2 = 128B.
__device__ __forceinline__ uint64_t umma_desc_mn_sw128(uint32_t smem_addr, uint32_t slab_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((slab_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
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

// TMA store of a 3-D box from shared memory, tracked as a bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int32_t x,
                                             int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_and_wait_read() {
  asm volatile(
      "cp.async.bulk.commit_group;\n\t"
      "cp.async.bulk.wait_group.read 0;" ::
          : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z, int32_t w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
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

// 32 lanes x 128 columns in one load, one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 64 columns stored in one instruction, then wait.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&w)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]), "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]), "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31]), "r"(w[32]), "r"(w[33]), "r"(w[34]), "r"(w[35]), "r"(w[36]), "r"(w[37]), "r"(w[38]), "r"(w[39]), "r"(w[40]), "r"(w[41]), "r"(w[42]), "r"(w[43]), "r"(w[44]), "r"(w[45]), "r"(w[46]), "r"(w[47]), "r"(w[48]), "r"(w[49]), "r"(w[50]), "r"(w[51]), "r"(w[52]), "r"(w[53]), "r"(w[54]), "r"(w[55]), "r"(w[56]), "r"(w[57]), "r"(w[58]), "r"(w[59]), "r"(w[60]), "r"(w[61]), "r"(w[62]), "r"(w[63])
      : "memory");
}

// D (TMEM) += A (TMEM: lane = row, 32-bit column c = bf16 pair of K elements
// 2c, 2c+1) x B (shared-memory descriptor).
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
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

// Packed fp32 pairs (Blackwell f32x2 arithmetic) and a three-input maximum.
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void uf2(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Walks the KV units of a tile: ancestor levels (root first), then the own
// segment up to the tile's causal bound.
// A segment computed by this call has its K/V in the k / v inputs only (the
// call writes shared segments into the pool for later calls); every other
// segment was computed by an earlier call and is read from the pool.
__device__ __forceinline__ bool computed_here(const AttnArgs& a, const SegDesc& x) {
  if (x.shared == 2) return false;  // a level of the prefix cache: pool only
  const bool kind_ok = a.call_kind == 2 || (x.shared != 0) == (a.call_kind == 0);
  return kind_ok && (a.call_round < 0 || x.round == a.call_round);
}

struct Cursor {
  int level;      // 0..chain_len (chain_len = own segment)
  int j;          // unit within the level
  int n_units;    // units in this level
  int len;        // visible keys in this level (own: t0 + nt)
  int n_pages;    // pages the level's segment owns (page-table bound)
  int page_off;   // first page-table entry of the level's segment
  int64_t row0;   // the level's first row in the k / v inputs
  bool own;
  bool local;     // read from the k / v inputs, not from the pool
};

__device__ __forceinline__ void cursor_level(Cursor& c, const AttnArgs& a, const SegDesc& sd,
                                             const TileDesc& td) {
  if (c.level < sd.chain_len) {
    const SegDesc an = a.segs[a.chain[sd.chain_off + c.level]];
    c.len = an.len;
    c.n_pages = (an.len + kPageSize - 1) / kPageSize;
    c.page_off = an.page_off;
    c.row0 = an.node_start;
    c.own = false;
    c.local = computed_here(a, an);
  } else if (c.level == sd.chain_len) {
    c.len = td.t0 + td.nt;
    c.n_pages = (sd.len + kPageSize - 1) / kPageSize;
    c.page_off = sd.page_off;
    c.row0 = sd.node_start;
    c.own = true;
    c.local = computed_here(a, sd);
  } else {  // a paired tile's second own level: the sibling leaf of half B
    const SegDesc s2 = a.segs[td.seg2];
    c.len = td.t0b + td.ntb;
    c.n_pages = (s2.len + kPageSize - 1) / kPageSize;
    c.page_off = s2.page_off;
    c.row0 = s2.node_start;
    c.own = true;
    c.local = computed_here(a, s2);
  }
  c.n_units = (c.len + kKeysPerUnit - 1) / kKeysPerUnit;
}

__device__ __forceinline__ void cursor_next(Cursor& c, const AttnArgs& a, const SegDesc& sd,
                                            const TileDesc& td) {
  const int last = sd.chain_len + (td.seg2 >= 0 ? 1 : 0);
  if (++c.j >= c.n_units && c.level < last) {
    c.level += 1;
    c.j = 0;
    cursor_level(c, a, sd, td);
  }
}

__device__ __forceinline__ Cursor cursor_at(const AttnArgs& a, const SegDesc& sd,
                                            const TileDesc& td, int unit) {
  Cursor c;
  c.level = 0;
  c.j = 0;
  cursor_level(c, a, sd, td);
  for (int u = 0; u < unit; ++u) cursor_next(c, a, sd, td);
  return c;
}

// A CTA walks its units [u_lo, u_hi) starting at a rotated position and
// wrapping around, so the CTAs that share a prefix do not all request the
// same KV lines at the same moment.  The online softmax does not depend on
// the order of the units.
struct UnitWalk {
  Cursor cur;
  int u;
  __device__ __forceinline__ void start(const AttnArgs& a, const SegDesc& sd, const TileDesc& td) {
    const int n = td.u_hi - td.u_lo;
    const unsigned tile = blockIdx.x / (unsigned)a.Hkv, hkv = blockIdx.x % (unsigned)a.Hkv;
    u = td.u_lo + (int)((tile * 5u + hkv * 3u) % (unsigned)(n > 0 ? n : 1));
    cur = cursor_at(a, sd, td, u);
  }
  __device__ __forceinline__ void next(const AttnArgs& a, const SegDesc& sd, const TileDesc& td) {
    if (++u == td.u_hi) {
      u = td.u_lo;
      cur = cursor_at(a, sd, td, u);
    } else {
      cursor_next(cur, a, sd, td);
    }
  }
};

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                          ~uintptr_t(1023));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKr,
                   const __grid_constant__ CUtensorMap tmK1, const __grid_constant__ CUtensorMap tmVr,
                   const __grid_constant__ CUtensorMap tmV1, const __grid_constant__ CUtensorMap tmKi,
                   const __grid_constant__ CUtensorMap tmVi, const __grid_constant__ CUtensorMap tmO,
                   AttnArgs a) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  unsigned char* sQ = smem;                        // [2 halves][D/64 slabs][128 x 128 B]
  unsigned char* sK = sQ + 2 * C::kQHalf;          // [stages][D/64 slabs][128 x 128 B]
  unsigned char* sV = sK + kKStages * C::kK;       // [stages][8 pages][D x 32 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + kVStages * C::kV);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + kKStages;
  uint64_t* v_full = k_empty + kKStages;
  uint64_t* v_empty = v_full + kVStages;
  uint64_t* s_full = v_empty + kVStages;  // [2]: S_h of the current unit is in TMEM
  uint64_t* p_full = s_full + 2;          // [2]: P_h of the current unit is in TMEM
  uint64_t* o_full = p_full + 2;          // [2]: all products of half h done, O_h complete
  uint64_t* drain = o_full + 2;           // [2]: the products half h issued before it gave up
  uint64_t* first_turn = drain + 2;       // half A issued its first group
  uint64_t* stage_full = first_turn + 1;  // [2]: half h's output rows are staged in smem
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stage_full + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // one CTA per (tile, KV head), KV head innermost: blocks start in tile
  // order, and the planner lists tiles longest first
  const TileDesc td = a.tiles[blockIdx.x / a.Hkv];
  const int hkv = (int)(blockIdx.x % a.Hkv);
  const SegDesc sd = a.segs[td.seg];
  const int n_units = td.u_hi - td.u_lo;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.G;
  // half B continues half A's tokens, or (a paired tile) holds the tail of
  // a sibling leaf
  const bool has_b = td.seg2 >= 0 || td.nt > kHalf / G;  // half B holds at least one token

  const int n_halves = has_b ? 2 : 1;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    // a K / V stage is free once every half's products that read it are done
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], (uint32_t)n_halves);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], (uint32_t)n_halves);
    }
    // p_full[h] phase m: the 4 warps of half h have written P_h(m) to TMEM and, with two
    // halves, the other half's issuer has issued the group before half h's
    // next one (its turn on the tensor pipe)
    for (int h = 0; h < 2; ++h) {
      mbar_init(&s_full[h], 1);
      mbar_init(&p_full[h], 4u + (n_halves == 2 ? 1u : 0u));
      mbar_init(&o_full[h], 1);
      mbar_init(&drain[h], 1);
    }
    mbar_init(first_turn, 1);
    mbar_init(&stage_full[0], 4);
    mbar_init(&stage_full[1], 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8 || warp == 10) {
    if (n_units > 0) {
      // -------- TMA producers: warp 8 loads Q and K, warp 10 loads V --------
      const bool is_k = warp == 8;
      if (is_k && lane == 0) {
        prefetch_tensormap(&tmQ);
        prefetch_tensormap(&tmKr);
        prefetch_tensormap(&tmK1);
        prefetch_tensormap(&tmKi);
        mbar_expect_tx(q_full, (uint32_t)(2 * C::kQHalf));
        for (int h = 0; h < 2; ++h)
          for (int slab = 0; slab < D / 64; ++slab)
            tma_load_3d(sQ + h * C::kQHalf + slab * C::kQSlab, &tmQ, q_full, slab * 64, hkv * G,
                        (int32_t)(h == 0 ? sd.node_start + td.t0
                                  : td.seg2 >= 0 ? a.segs[td.seg2].node_start + td.t0b
                                                 : sd.node_start + td.t0 + kHalf / G));
      }
      if (!is_k && lane == 0) {
        prefetch_tensormap(&tmVr);
        prefetch_tensormap(&tmV1);
        prefetch_tensormap(&tmVi);
      }
      const int n_st = is_k ? kKStages : kVStages;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      const uint32_t bytes = is_k ? (uint32_t)C::kK : (uint32_t)C::kV;
      UnitWalk walk;
      walk.start(a, sd, td);
      int page = 0;
      bool in_seg = false;
      // A level read from the pool names its pages through the page table.  A
      // page-table index or a page id out of range (a stale or mismatched
      // descriptor) sets the bounds bit of the error word; the fetch then
      // reads outside the pool tensor, which the pool maps fill with NaN, so
      // the rows that use it come out NaN and nothing outside the pool is read.
      auto fetch_page = [&](const Cursor& c) {
        int pi = c.j * kPages + lane;
        in_seg = pi < c.n_pages;
        if (!in_seg) pi = c.n_pages - 1;  // finite filler; its keys are masked
        const int64_t e = (int64_t)c.page_off + pi;
        page = e >= 0 && e < a.n_page_entries ? a.page_ids[e] : -1;
        if (!c.local && (page < 0 || (int64_t)page >= a.pool_pages)) {
          raise_error(a.err, kErrBounds);
          page = -1;
        }
      };
      if (lane < kPages) fetch_page(walk.cur);
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
        const int p0 = __shfl_sync(0xffffffffu, page, 0);
        const bool run = __all_sync(0xffffffffu, lane >= kPages || (in_seg && page == p0 + lane));
        if (lane == 0) mbar_expect_tx(&full[s], bytes);
        __syncwarp();
        unsigned char* dst = is_k ? sK + s * C::kK : sV + s * C::kV;
        if (walk.cur.local) {
          // 128 consecutive rows of the inputs: one box per 64-dim slab (rows
          // past the level's end are masked by the softmax)
          if (lane == 0)
            for (int slab = 0; slab < D / 64; ++slab)
              tma_load_3d(dst + slab * C::kKSlab, is_k ? &tmKi : &tmVi, &full[s], slab * 64, hkv,
                          (int32_t)(walk.cur.row0 + (int64_t)walk.cur.j * kKeysPerUnit));
        } else if (run) {
          if (lane == 0)
            for (int slab = 0; slab < D / 64; ++slab)
              tma_load_4d(dst + slab * C::kKSlab, is_k ? &tmKr : &tmVr, &full[s], slab * 64, 0, hkv, p0);
        } else if (lane < kPages) {
          for (int slab = 0; slab < D / 64; ++slab)
            tma_load_4d(dst + slab * C::kKSlab + lane * (kPageSize * 128), is_k ? &tmK1 : &tmV1,
                        &full[s], slab * 64, 0, hkv, page);
        }
        issued[s] = (int)ph;
        walk.next(a, sd, td);
        if (it + 1 < n_units && lane < kPages) fetch_page(walk.cur);
        if (++s == n_st) {
          s = 0;
          ph ^= 1;
        }
      }
      if (lane == 0) {
        if (!ok) {
          if (!*abort_flag) raise_error(a.err, kErrTimeout);
          *abort_flag = 1;
        }
        // every load issued has landed before the CTA exits: after an abort
        // the issuers may not have read them all (on the normal path they
        // have, and these waits end at once)
        if (is_k) mbar_wait(q_full, 0, nullptr);
        for (int i = 0; i < n_st; ++i)
          if (issued[i] >= 0) mbar_wait(&full[i], (uint32_t)issued[i], nullptr);
      }
      // A shared segment computed here goes into the pool for later calls:
      // the first part of each tile copies the tile's tokens for its KV head
      // (warp 8 the K rows, warp 10 the V rows), and the tile holding the
      // segment's last token zero-fills the rest of that page.  No tile of
      // this call reads these pages.
      if (ok && td.u_lo == 0 && sd.shared == 1 && computed_here(a, sd)) {
        // a page id or a source row out of range skips its store and sets the
        // bounds bit of the error word
        constexpr int kChunks = D / 8;  // 16-byte chunks per row
        const bf16* src = is_k ? a.k_in : a.v_in;
        const size_t page_elems = (size_t)2 * a.Hkv * kPageSize * D;
        const size_t kv_off = ((size_t)(is_k ? 0 : a.Hkv) + hkv) * kPageSize * D;
        const int t_end = td.t0 + td.nt;
        const int t_fill = t_end == sd.len ? ((sd.len + kPageSize - 1) / kPageSize) * kPageSize : t_end;
        const int n_items = (t_fill - td.t0) * kChunks;
        constexpr int kBatch = 8;  // loads in flight per lane before the stores
        for (int i0 = 0; i0 < n_items; i0 += 32 * kBatch) {
          uint4 val[kBatch];
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int i = i0 + b * 32 + lane;
            const int t = td.t0 + i / kChunks, ch = i % kChunks;
            val[b] = make_uint4(0, 0, 0, 0);
            if (i < n_items && t < t_end) {
              const int64_t row = sd.node_start + t;
              if (row >= 0 && row < a.node_tokens)
                val[b] = *reinterpret_cast<const uint4*>(src + ((size_t)row * a.Hkv + hkv) * D + ch * 8);
              else
                raise_error(a.err, kErrBounds);
            }
          }
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int i = i0 + b * 32 + lane;
            if (i >= n_items) break;
            const int t = td.t0 + i / kChunks, ch = i % kChunks;
            const int64_t e = (int64_t)sd.page_off + t / kPageSize;
            const int page = e >= 0 && e < a.n_page_entries ? a.page_ids[e] : -1;
            if (page < 0 || (int64_t)page >= a.pool_pages) {
              raise_error(a.err, kErrBounds);
              continue;
            }
            *reinterpret_cast<uint4*>(a.pool + (size_t)page * page_elems + kv_off +
                                      (size_t)(t % kPageSize) * D + ch * 8) = val[b];
          }
        }
      }
    }
  } else if (warp == 9 || warp == 11) {
    const int h = warp == 9 ? 0 : 1;
    if (lane == 0 && n_units > 0 && h < n_halves) {
      // ---------------- MMA issuer of half h ----------------
      // Group g of half h = PV_h(g-1) (g > 0) then QK_h(g) (g < n_units).
      // The halves take turns on the tensor pipe, A0 B0 A1 B1 ..., so one
      // half's softmax always overlaps the other half's products.  An issuer
      // does its data waits (P, V, K) while the other half's group runs and
      // then waits only for its turn: the pipe holds about one product at a
      // time, so every wait between two issues would leave it idle.  QK_h(g)
      // overwrites S_h, where P_h(g-1) lives, only after PV_h(g-1) (same
      // thread, in order); the commit after QK_h(g) covers PV_h(g-1) too, so
      // it also tells the softmax that O_h is stable and may be rescaled.
      const uint32_t idesc_qk = umma_idesc_bf16_f32(kHalf, kKeysPerUnit);
      const uint32_t idesc_pv = umma_idesc_bf16_f32(kHalf, D) | (1u << 16);  // B (V) MN-major
      const uint32_t q_addr = smem_u32(sQ) + (uint32_t)(h * C::kQHalf);
      const uint32_t s_col = tmem + C::kColS + (uint32_t)(h * kKeysPerUnit);
      const uint32_t o_col = tmem + C::kColO + (uint32_t)(h * D);
      const bool paired = n_halves == 2;
      bool ok = mbar_wait(q_full, 0, abort_flag);
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;
      for (int g = 0; g <= n_units && ok; ++g) {
        const bool do_pv = g > 0, do_qk = g < n_units;
        // K and V are usually in place already; P_h(g-1) together with the
        // turn (A's group g after B's group g-1, B's group g after A's group
        // g) is one barrier phase, the only wait that is usually not over
        if (do_qk) ok = mbar_wait(&k_full[ks], kph, abort_flag);
        if (ok && do_pv) ok = mbar_wait(&v_full[vs], vph, abort_flag);
        if (ok && do_pv) ok = mbar_wait_poll(&p_full[h], (uint32_t)((g - 1) & 1), abort_flag);
        if (ok && paired && h == 1 && g == 0) ok = mbar_wait_poll(first_turn, 0, abort_flag);
        if (!ok) break;
        tc_fence_after();
        if (do_pv) {
          const uint32_t v_addr = smem_u32(sV + vs * C::kV);
#pragma unroll
          for (int p = 0; p < kPages; ++p) {
            umma_bf16_tmem_a(o_col, s_col + 8 * p,
                             umma_desc_mn_sw128(v_addr + p * (kPageSize * 128), C::kKSlab), idesc_pv,
                             (g > 1 || p > 0) ? 1u : 0u);
          }
        }
        if (do_qk) {
          const uint32_t k_addr = smem_u32(sK + ks * C::kK);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t qo = (kk >> 2) * C::kQSlab + (kk & 3) * 32;
            const uint32_t ko = (kk >> 2) * C::kKSlab + (kk & 3) * 32;
            umma_bf16(s_col, umma_desc_k_sw128(q_addr + qo), umma_desc_k_sw128(k_addr + ko),
                      idesc_qk, kk > 0 ? 1u : 0u);
          }
        }
        if (paired) mbar_arrive(h == 1 ? &p_full[0] : (g == 0 ? first_turn : &p_full[1]));
        if (do_pv) {
          umma_commit(&v_empty[vs]);
          if (++vs == kVStages) {
            vs = 0;
            vph ^= 1;
          }
        }
        if (do_qk) {
          umma_commit(&s_full[h]);
          umma_commit(&k_empty[ks]);
          if (++ks == kKStages) {
            ks = 0;
            kph ^= 1;
          }
        }
      }
      if (ok) {
        umma_commit(&o_full[h]);  // every product of this half: O_h is complete
        mbar_wait(&o_full[h], 0, nullptr);
      } else {
        // gave up: o_full stays incomplete (the softmax sees the abort flag
        // instead), and the products issued so far finish before the exit
        if (!*abort_flag) raise_error(a.err, kErrTimeout);
        *abort_flag = 1;
        umma_commit(&drain[h]);
        mbar_wait(&drain[h], 0, nullptr);
      }
    }
  } else if (warp < 8 && n_units > 0 && (warp < 4 || has_b)) {
    // ---------------- softmax / epilogue of one half ----------------
    const int h = warp >> 2;
    const int r = threadIdx.x & 127;  // row within the half = TMEM lane
    const int tok = r / G;  // token within the half
    // the row's position within its half's segment
    const int token = (h == 0 ? td.t0 : td.seg2 >= 0 ? td.t0b : td.t0 + kHalf / G) + tok;
    const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t s_col = C::kColS + (uint32_t)(h * kKeysPerUnit);
    const uint32_t o_col = C::kColO + (uint32_t)(h * D);
    const float scale = a.scale_log2;
    float m_used = -INFINITY;  // running max, in scaled log2 units
    float l = 0.f;             // running sum of exp2(s * scale - m_used)
    UnitWalk walk;
    walk.start(a, sd, td);
    bool ok = true;
    for (int it = 0; it < n_units; ++it) {
      if (!__all_sync(0xffffffffu, mbar_wait_poll(&s_full[h], (uint32_t)(it & 1), abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // visible keys of this row in this unit: c < lim
      const int key0 = walk.cur.j * kKeysPerUnit;
      int lim = walk.cur.len - key0;
      if (walk.cur.own) {
        // a paired tile's own levels: half A's segment, then half B's; each
        // half sees only its own (causally)
        const bool other = td.seg2 >= 0 && ((walk.cur.level > sd.chain_len) != (h == 1));
        lim = other ? 0 : min(lim, token - key0 + 1);
      }
      // The running maximum only keeps 2^(s * scale - m) finite: P, the row
      // sum and O are exact in relative terms for any reference m, which
      // cancels in O / l.  A row takes it on its first unit with a finite
      // score, and again only when a unit's sum shows a score more than 64
      // above the reference (P > 2^64) or a value that is not finite; that
      // second pass reloads S (P goes over it only after the loop).
      const float m_prev = m_used;
      const bool masked = __any_sync(0xffffffffu, lim < kKeysPerUnit);
      const uint64_t sc2 = f2(scale, scale);
      uint32_t pw[kKeysPerUnit / 2];
      float ls = 0.f;
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        float sv[kKeysPerUnit];
        tmem_ld128(trow + s_col, sv);
        if (masked) {
#pragma unroll
          for (int c = 0; c < kKeysPerUnit; ++c) sv[c] = c < lim ? sv[c] : -INFINITY;
        }
        if (pass == 1 || __any_sync(0xffffffffu, m_used == -INFINITY)) {
          // tree maximum: eight independent chains of three-input maxima
          float mx8[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) mx8[c] = fmaxf(sv[2 * c], sv[2 * c + 1]);
#pragma unroll
          for (int c = 16; c < kKeysPerUnit; c += 2)
            mx8[(c >> 1) & 7] = max3(mx8[(c >> 1) & 7], sv[c], sv[c + 1]);
          const float mt = fmaxf(max3(mx8[0], mx8[1], mx8[2]),
                                 fmaxf(max3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
          const float m_new = fmaxf(m_used, mt * scale);
          // a first maximum, or an overflow; otherwise only a rise by > 2^8
          if (pass == 1 || m_used == -INFINITY || m_new > m_used + kRescaleLog2) m_used = m_new;
        }
        const float nbase = m_used == -INFINITY ? 0.f : -m_used;
        const uint64_t nb2 = f2(nbase, nbase);
        uint64_t sum4[4] = {0, 0, 0, 0};
#pragma unroll
        for (int c = 0; c < kKeysPerUnit; c += 2) {
          float x0, x1;
          uf2(fma_f2(f2(sv[c], sv[c + 1]), sc2, nb2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          sum4[(c >> 1) & 3] = add_f2(sum4[(c >> 1) & 3], f2(p0, p1));
          pw[c >> 1] = pack_bf16(p0, p1);
        }
        float s0, s1, s2, s3, s4, s5, s6, s7;
        uf2(sum4[0], s0, s1);
        uf2(sum4[1], s2, s3);
        uf2(sum4[2], s4, s5);
        uf2(sum4[3], s6, s7);
        ls = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
        if (!__any_sync(0xffffffffu, !(ls <= 0x1p64f))) break;
      }
      const float alpha = m_used == m_prev ? 1.f : m_prev == -INFINITY ? 0.f : ex2(m_prev - m_used);
      l = l * alpha + ls;
      // O_h is stable: PV_h of the previous unit completed before S_h arrived
      if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(trow + o_col + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(trow + o_col + 32 * c, o);
        }
      }
      // P_h (bf16 pairs) over the first 64 columns of S_h
      tmem_st64(trow + s_col, pw);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[h]);  // one arrival per warp
      walk.next(a, sd, td);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_full[h], 0, abort_flag));
    if (!ok) {
      if (!*abort_flag) raise_error(a.err, kErrTimeout);
      *abort_flag = 1;
    } else {
      tc_fence_after();
      // (a NaN sum, from a NaN key or value, stays NaN in both)
      const float inv = l == 0.f ? 0.f : 1.f / l;
      const float lse = l == 0.f ? -INFINITY : (m_used + __log2f(l)) * 0.69314718055994531f;
      // half h's rows: tokens of its segment from seg_row0 on, nt_h of them
      const bool pair_b = h == 1 && td.seg2 >= 0;
      const int nt_h = h == 0 ? min(td.nt, kHalf / G) : pair_b ? td.ntb : td.nt - kHalf / G;
      const int64_t seg_row0 = pair_b ? a.segs[td.seg2].node_start : sd.node_start;
      // a row or a partial slot out of range (a bad descriptor) is not
      // written and sets the bounds bit of the error word
      const bool in_range = td.part < 0 ? seg_row0 + token >= 0 && seg_row0 + token < a.node_tokens
                                        : td.part < a.n_parts;
      if (tok < nt_h && !in_range) raise_error(a.err, kErrBounds);
      const bool row_ok = tok < nt_h && in_range;
      const int head = hkv * G + (r % G);
      const size_t orow = (size_t)(seg_row0 + token) * a.Hq + head;
      const size_t prow_i = ((size_t)td.part * a.Hkv + hkv) * kRowsPerTile + h * kHalf + r;
      // A final half whose rows are all tokens of the tile goes out through
      // the Q_h buffer (its products are done) and TMA stores: rows laid out
      // like the Q box (token x head), 128-byte swizzled.
      // (TMA stores start only inside the output: a store must not start at
      // a negative row, so a half whose rows fall outside goes the checked way)
      const int64_t half_row0 = seg_row0 + (token - tok);
      const bool staged = td.part < 0 && nt_h >= kHalf / G && half_row0 >= 0 &&
                          half_row0 + kHalf / G <= a.node_tokens;
      unsigned char* stage = sQ + h * C::kQHalf;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(trow + o_col + 32 * c, o);
        if (staged) {
          unsigned char* rowp = stage + (c >> 1) * C::kQSlab + r * 128;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv);
            w.y = pack_bf16(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv);
            w.z = pack_bf16(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv);
            w.w = pack_bf16(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv);
            const int chunk = (c & 1) * 4 + q4;
            *reinterpret_cast<uint4*>(rowp + ((chunk ^ (r & 7)) << 4)) = w;
          }
          continue;
        }
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
      if (staged) {
        fence_proxy_async_smem();  // the TMA (async proxy) reads what this thread wrote
        __syncwarp();
        if (lane == 0) mbar_arrive(&stage_full[h]);
        if ((warp & 3) == 0 && lane == 0) {
          if (mbar_wait(&stage_full[h], 0, abort_flag)) {
            for (int slab = 0; slab < D / 64; ++slab)
              tma_store_3d(&tmO, stage + slab * C::kQSlab, slab * 64, hkv * G, (int32_t)half_row0);
            bulk_commit_and_wait_read();  // the smem stays valid until the stores read it
          } else {
            if (!*abort_flag) raise_error(a.err, kErrTimeout);
            *abort_flag = 1;
          }
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
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Combine the partial (O, lse) of split tiles: O = sum_i e^(lse_i - L) O_i,
// L = ln sum_i e^(lse_i).  One warp per query row (grid.x = merges x 32
// blocks of 8 rows, grid.y = KV head), lanes across head_dim; the loads of
// every part are in flight together.
template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const SegDesc* segs, const MergeDesc* merges,
                                                         const float* part_o, const float* part_lse,
                                                         bf16* out, float* lse_out, int Hq, int Hkv,
                                                         int G, int64_t node_tokens, int n_parts,
                                                         unsigned* err) {
  constexpr int PER = D / 32;
  constexpr int kBatch = 8;
  const MergeDesc md = merges[blockIdx.x >> 5];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = (blockIdx.x & 31) * 8 + warp;
  const int hkv = blockIdx.y;
  if (row / G >= md.nt) return;
  // partial slots and the output row inside their buffers, else the bounds
  // bit of the error word and nothing read or written
  const int64_t out_row = segs[md.seg].node_start + md.t0 + row / G;
  if (md.part0 < 0 || md.nparts < 0 || (int64_t)md.part0 + md.nparts > n_parts || out_row < 0 ||
      out_row >= node_tokens) {
    if (lane == 0) raise_error(err, kErrBounds);
    return;
  }
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
  const size_t orow = (size_t)out_row * Hq + hkv * G + (row % G);
#pragma unroll
  for (int e = 0; e < PER; e += 2)
    *reinterpret_cast<uint32_t*>(out + orow * D + lane * PER + e) =
        pack_bf16(acc[e] * inv, acc[e + 1] * inv);
  if (lane == 0) lse_out[orow] = S > 0.f ? M + __logf(S) : -INFINITY;
}

bool encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz,
            CUtensorMapFloatOOBfill fill = CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) {
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (uint32_t)rank, base, dims, strides,
                      box, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, fill);
}

template <int D>
cudaError_t run_call(const AttnLaunch& L) {
  const DescHeader& h = *L.hdr;
  const unsigned char* base = static_cast<const unsigned char*>(L.dev_desc);
  const SegDesc* segs = reinterpret_cast<const SegDesc*>(base + h.off_segs);
  const int32_t* pages = reinterpret_cast<const int32_t*>(base + h.off_pages);
  const int32_t* chain = reinterpret_cast<const int32_t*>(base + h.off_chain);
  const TileDesc* tiles = reinterpret_cast<const TileDesc*>(base + h.off_tiles) + L.tile_off;
  const MergeDesc* merges = reinterpret_cast<const MergeDesc*>(base + h.off_merges) + L.merge_off;
  cudaStream_t st = static_cast<cudaStream_t>(L.stream);
  bf16* pool = static_cast<bf16*>(L.pool);
  const int G = L.Hq / L.Hkv;
  int launches = 0;
  float* part_o = static_cast<float*>(L.workspace);
  float* part_lse = part_o + (size_t)L.n_parts * L.Hkv * kRowsPerTile * D;
  if (L.n_tiles > 0) {
    CUtensorMap tmQ, tmKr, tmK1, tmVr, tmV1, tmKi, tmVi, tmO;
    {
      // k / v inputs [node_tokens][Hkv][D]: 128 rows of one KV head per box
      cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L.Hkv, (cuuint64_t)L.node_tokens};
      cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L.Hkv * D * 2};
      cuuint32_t box[3] = {64, 1, (cuuint32_t)kKeysPerUnit};
      if (!encode(&tmKi, L.k, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !encode(&tmVi, L.v, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    {
      cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L.Hq, (cuuint64_t)L.node_tokens};
      cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L.Hq * D * 2};
      cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(kHalf / G)};
      if (!encode(&tmQ, L.q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !encode(&tmO, L.out, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    }
    // pool page: [K: Hkv][16][D] then [V: Hkv][16][D]; dims (inner first)
    constexpr CUtensorMapFloatOOBfill kNanFill = CU_TENSOR_MAP_FLOAT_OOB_FILL_NAN_REQUEST_ZERO_FMA;
    const cuuint64_t page_bytes = (cuuint64_t)2 * L.Hkv * kPageSize * D * 2;
    {
      cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)kPageSize, (cuuint64_t)L.Hkv,
                            (cuuint64_t)L.pool_pages};
      cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)kPageSize * D * 2, page_bytes};
      cuuint32_t boxr[4] = {64, (cuuint32_t)kPageSize, 1, (cuuint32_t)kPages};
      cuuint32_t box1[4] = {64, (cuuint32_t)kPageSize, 1, 1};
      // a valid descriptor never reads outside the plan's pages: NaN there
      if (!encode(&tmKr, pool, 4, dims, strides, boxr, CU_TENSOR_MAP_SWIZZLE_128B, kNanFill) ||
          !encode(&tmK1, pool, 4, dims, strides, box1, CU_TENSOR_MAP_SWIZZLE_128B, kNanFill))
        return cudaErrorInvalidValue;
    }
    {
      const bf16* vbase = pool + (size_t)L.Hkv * kPageSize * D;
      cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)kPageSize, (cuuint64_t)L.Hkv,
                            (cuuint64_t)L.pool_pages};
      cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)kPageSize * D * 2, page_bytes};
      cuuint32_t boxr[4] = {64, (cuuint32_t)kPageSize, 1, (cuuint32_t)kPages};
      cuuint32_t box1[4] = {64, (cuuint32_t)kPageSize, 1, 1};
      if (!encode(&tmVr, vbase, 4, dims, strides, boxr, CU_TENSOR_MAP_SWIZZLE_128B, kNanFill) ||
          !encode(&tmV1, vbase, 4, dims, strides, box1, CU_TENSOR_MAP_SWIZZLE_128B, kNanFill))
        return cudaErrorInvalidValue;
    }
    AttnArgs a;
    a.segs = segs;
    a.page_ids = pages;
    a.chain = chain;
    a.tiles = tiles;
    a.k_in = static_cast<const bf16*>(L.k);
    a.v_in = static_cast<const bf16*>(L.v);
    a.pool = pool;
    a.call_round = L.round;
    a.call_kind = L.kind;
    a.out = static_cast<bf16*>(L.out);
    a.lse = L.lse;
    a.part_o = part_o;
    a.part_lse = part_lse;
    a.err = L.err;
    a.Hq = L.Hq;
    a.Hkv = L.Hkv;
    a.G = G;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    a.node_tokens = L.node_tokens;
    a.pool_pages = L.pool_pages;
    a.n_page_entries = h.n_pages;
    a.n_parts = L.n_parts;
    const size_t smem = Cfg<D>::kSmem;
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(attn_tc_kernel<D>), (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)L.n_tiles * (unsigned)L.Hkv);
    attn_tc_kernel<D><<<grid, kThreads, smem, st>>>(tmQ, tmKr, tmK1, tmVr, tmV1, tmKi, tmVi, tmO,
                                                    a);
    ++launches;
  }
  if (L.n_merges > 0) {
    dim3 grid((unsigned)L.n_merges * 32, (unsigned)L.Hkv);
    attn_merge_kernel<D><<<grid, 256, 0, st>>>(segs, merges, part_o, part_lse,
                                               static_cast<bf16*>(L.out), L.lse, L.Hq, L.Hkv, G,
                                               L.node_tokens, L.n_parts, L.err);
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
