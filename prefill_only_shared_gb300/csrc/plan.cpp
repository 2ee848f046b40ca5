// Host planner: token trie -> segments -> staged rounds -> KV pages ->
// per-round launch lists, plus the host-only ABI helpers.
//
// Sources: LLM2Jev "shared prefix" page (sharing follows the tokenised prefix;
// staged submission builds each shared prefix with one real candidate, then
// the candidates that reuse it; independent branches share a round; the
// final scoring position is always computed) and the openjev-sglang article
// (radix cache over token prefixes; request limits of 32768 tokens per branch
// and 262144 per request).
//
// The trie is a radix tree built by inserting each request's branches in
// index order; a child is created by the first branch that reaches it, so the
// children of a node stay sorted by their smallest member branch, which is
// the order the depth-first node-token layout uses.
#include <algorithm>
#include <cstring>
#include <map>
#include <new>
#include <tuple>
#include <vector>

#include "plan_internal.h"

namespace {

using sp::kMaxBranchTokens;
using sp::kMaxRequestTokens;
constexpr int32_t kMinUnitsPerPart = 4;

struct TNode {
  int64_t src = 0;  // index into tokens[] of the node's first token
  int32_t len = 0;
  int32_t first_branch = 0;
  int32_t parent = -1;
  std::vector<int32_t> children;
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool shape_ok(const sp_shape& s) {
  if (s.n_q_heads <= 0 || s.n_kv_heads <= 0 || s.n_q_heads % s.n_kv_heads) return false;
  int g = s.n_q_heads / s.n_kv_heads;
  if (g > 128 || 128 % g) return false;  // each 128-row half holds whole tokens
  if (s.head_dim != 64 && s.head_dim != 128) return false;
  if (s.page_size != sp::kPageSize) return false;
  if (s.hidden <= 0 || s.hidden % 8) return false;
  if (s.vocab < 2) return false;
  return true;
}

}  // namespace

namespace {

sp_status build(const sp_shape* shape, sp_cache* cache, int32_t n_branches,
                const int32_t* req_of_branch, const int64_t* tok_offsets, const int32_t* tokens,
                int32_t max_pages, int32_t n_sms, sp_plan** out) {
  if (!out) return SP_ERR_ARG;
  *out = nullptr;
  if (!shape || !req_of_branch || !tok_offsets || !tokens || n_branches <= 0 || max_pages < 0)
    return SP_ERR_ARG;
  if (!shape_ok(*shape)) return SP_ERR_ARG;
  const int32_t N = n_branches;
  if (tok_offsets[0] != 0) return SP_ERR_ARG;
  for (int32_t b = 0; b < N; ++b) {
    if (req_of_branch[b] < 0) return SP_ERR_ARG;
    int64_t L = tok_offsets[b + 1] - tok_offsets[b];
    if (L <= 0) return SP_ERR_ARG;
    if (L > kMaxBranchTokens) return SP_ERR_LIMIT;
  }
  // requests in increasing id; branches of each request in index order
  std::map<int32_t, std::vector<int32_t>> by_req;
  for (int32_t b = 0; b < N; ++b) by_req[req_of_branch[b]].push_back(b);
  for (auto& kv : by_req) {
    int64_t tot = 0;
    for (int32_t b : kv.second) tot += tok_offsets[b + 1] - tok_offsets[b];
    if (tot > kMaxRequestTokens) return SP_ERR_LIMIT;
  }

  sp_plan* P = new (std::nothrow) sp_plan();
  if (!P) return SP_ERR_ARG;
  P->shape = *shape;
  P->n_sms = n_sms > 0 ? n_sms : 152;
  P->max_pages = max_pages;
  P->n_branches = N;
  P->n_requests = (int32_t)by_req.size();
  P->cache = cache;

  // ---- prefix cache and match groups -------------------------------------
  // With a cache every branch first reuses its longest cached prefix, capped
  // one short of its length (the last position is always computed); the
  // remainders are planned like a cold request, in groups of the branches of
  // one request whose match ends at the same place (group order: request id,
  // then smallest branch).  Without a cache a group is a request.
  std::vector<int64_t> rem_off(N), rem_len(N);
  std::vector<std::vector<std::pair<int32_t, int32_t>>> bchain(N);
  int64_t hit_tokens = 0;
  for (int32_t b = 0; b < N; ++b) {
    const int64_t off = tok_offsets[b], L = tok_offsets[b + 1] - off;
    int64_t m = 0;
    if (cache) {
      m = sp::cache_match(*cache, tokens + off, L, bchain[b]);
      if (m > L - 1) {
        auto& e = bchain[b].back();
        if (e.second > 1)
          e.second -= 1;
        else
          bchain[b].pop_back();
        m -= 1;
      }
    }
    rem_off[b] = off + m;
    rem_len[b] = L - m;
    hit_tokens += m;
  }
  struct Group {
    int32_t req;
    std::pair<int32_t, int32_t> end;
    std::vector<int32_t> members;
  };
  std::vector<Group> groups;
  {
    std::map<std::tuple<int32_t, int32_t, int32_t>, int32_t> idx;
    for (int32_t b = 0; b < N; ++b) {
      const std::pair<int32_t, int32_t> end =
          bchain[b].empty() ? std::make_pair(0, 0) : bchain[b].back();
      const auto key = std::make_tuple(req_of_branch[b], end.first, end.second);
      auto it = idx.find(key);
      if (it == idx.end()) {
        idx.emplace(key, (int32_t)groups.size());
        groups.push_back({req_of_branch[b], end, {b}});
      } else {
        groups[it->second].members.push_back(b);
      }
    }
    std::stable_sort(groups.begin(), groups.end(), [](const Group& x, const Group& y) {
      return x.req != y.req ? x.req < y.req : x.members[0] < y.members[0];
    });
  }

  // ---- radix trie per request ------------------------------------------
  std::vector<TNode> nodes;
  std::vector<int32_t> roots;  // virtual root per request (len 0)
  std::vector<std::vector<int32_t>> path(N);
  for (auto& grp : groups) {
    int32_t root = (int32_t)nodes.size();
    nodes.emplace_back();
    roots.push_back(root);
    for (int32_t b : grp.members) {
      const int64_t off = rem_off[b];
      const int64_t L = rem_len[b];
      int32_t cur = root;
      int64_t pos = 0;
      while (pos < L) {
        const int32_t tok = tokens[off + pos];
        int32_t c = -1;
        for (int32_t ch : nodes[cur].children)
          if (tokens[nodes[ch].src] == tok) { c = ch; break; }
        if (c < 0) {
          TNode n;
          n.src = off + pos;
          n.len = (int32_t)(L - pos);
          n.first_branch = b;
          n.parent = cur;
          int32_t id = (int32_t)nodes.size();
          nodes.push_back(n);
          nodes[cur].children.push_back(id);
          break;
        }
        int64_t lim = std::min<int64_t>(nodes[c].len, L - pos);
        int64_t m = 0;
        while (m < lim && tokens[nodes[c].src + m] == tokens[off + pos + m]) ++m;
        if (m < nodes[c].len) {  // split edge c at m
          TNode mid;
          mid.src = nodes[c].src;
          mid.len = (int32_t)m;
          mid.first_branch = nodes[c].first_branch;
          mid.parent = cur;
          mid.children.push_back(c);
          int32_t id = (int32_t)nodes.size();
          nodes.push_back(mid);
          nodes[c].src += m;
          nodes[c].len -= (int32_t)m;
          nodes[c].parent = id;
          for (auto& ch : nodes[cur].children)
            if (ch == c) ch = id;
          cur = id;
        } else {
          cur = c;
        }
        pos += m;
      }
    }
    // second pass: every branch's path now ends on a node boundary
    for (int32_t b : grp.members) {
      const int64_t off = rem_off[b];
      const int64_t L = rem_len[b];
      int32_t cur = root;
      int64_t pos = 0;
      while (pos < L) {
        int32_t c = -1;
        for (int32_t ch : nodes[cur].children)
          if (tokens[nodes[ch].src] == tokens[off + pos]) { c = ch; break; }
        path[b].push_back(c);
        pos += nodes[c].len;
        cur = c;
      }
    }
  }

  // ---- node-token layout: depth-first pre-order ------------------------
  std::vector<int32_t> seg_of_node(nodes.size(), -1);
  std::vector<int32_t> order;
  order.reserve(nodes.size());
  {
    std::vector<int32_t> stack;
    for (int32_t root : roots) {
      for (auto it = nodes[root].children.rbegin(); it != nodes[root].children.rend(); ++it)
        stack.push_back(*it);
      while (!stack.empty()) {
        int32_t n = stack.back();
        stack.pop_back();
        seg_of_node[n] = (int32_t)order.size();
        order.push_back(n);
        for (auto it = nodes[n].children.rbegin(); it != nodes[n].children.rend(); ++it)
          stack.push_back(*it);
      }
    }
  }
  const int32_t S = (int32_t)order.size();
  std::vector<int32_t> count(S, 0);
  for (int32_t b = 0; b < N; ++b) {
    for (auto& n : path[b]) {
      n = seg_of_node[n];
      count[n] += 1;
    }
  }
  P->seg_req.resize(S);
  P->seg_parent.resize(S);
  P->seg_len.resize(S);
  P->seg_shared.resize(S);
  P->seg_round.assign(S, -1);
  P->seg_first_page.resize(S);
  P->seg_node_start.resize(S);
  P->seg_group.resize(S);
  P->seg_branch.resize(S);
  P->seg_pos.resize(S);
  std::vector<int64_t> seg_src(S);
  {
    // group of each root's subtree
    std::vector<int32_t> group_of_root_node(nodes.size(), -1);
    for (size_t g = 0; g < groups.size(); ++g) group_of_root_node[roots[g]] = (int32_t)g;
    int64_t row = 0;
    for (int32_t s = 0; s < S; ++s) {
      const TNode& n = nodes[order[s]];
      P->seg_len[s] = n.len;
      P->seg_parent[s] = group_of_root_node[n.parent] >= 0 ? -1 : seg_of_node[n.parent];
      P->seg_shared[s] = count[s] >= 2 ? 1 : 0;
      P->seg_node_start[s] = row;
      seg_src[s] = n.src;
      P->seg_branch[s] = n.first_branch;
      P->seg_pos[s] = (int32_t)(n.src - tok_offsets[n.first_branch]);
      row += n.len;
    }
    for (int32_t s = 0; s < S; ++s) {
      int32_t p = s;
      while (P->seg_parent[p] >= 0) p = P->seg_parent[p];
      P->seg_group[s] = group_of_root_node[nodes[order[p]].parent];
      P->seg_req[s] = groups[P->seg_group[s]].req;
    }
    P->stats.node_tokens = row;
  }

  // ---- KV pages ------------------------------------------------------------
  // Without a cache every segment owns consecutive pages 0, 1, ... in layout
  // order.  With a cache only the new shared segments are written to the
  // pool (leaves are read by no later call): they take pages from the cache,
  // after evicting least recently used cache leaves when the free pages do not
  // cover them; a leaf's page-table entries are placeholders (never read).
  std::vector<int32_t> page_table;
  if (!cache) {
    int64_t page = 0;
    for (int32_t s = 0; s < S; ++s) {
      P->seg_first_page[s] = (int32_t)page;
      page += ceil_div(P->seg_len[s], sp::kPageSize);
    }
    P->stats.pages_used = page;
    if (page > max_pages) {
      delete P;
      return SP_ERR_POOL_FULL;
    }
    page_table.resize((size_t)page);
    for (int64_t i = 0; i < page; ++i) page_table[i] = (int32_t)i;
    P->pool_pages = page;
  } else {
    // pin and mark used every node the plan reads
    for (int32_t b = 0; b < N; ++b)
      for (auto& e : bchain[b]) P->pinned.push_back(e.first);
    std::sort(P->pinned.begin(), P->pinned.end());
    P->pinned.erase(std::unique(P->pinned.begin(), P->pinned.end()), P->pinned.end());
    for (int32_t nd : P->pinned) {
      cache->nodes[nd].pins += 1;
      cache->nodes[nd].last_used = cache->clock;
    }
    cache->clock += 1;
    int64_t need = 0;
    for (int32_t s = 0; s < S; ++s)
      if (P->seg_shared[s]) need += ceil_div(P->seg_len[s], sp::kPageSize);
    while (cache->n_free < need)
      if (!sp::cache_evict_one(*cache)) {
        delete P;  // releases the pins
        return SP_ERR_POOL_FULL;
      }
    P->seg_pages.resize(S);
    P->seg_tokens.resize(S);
    P->seg_cache_node.assign(S, -1);
    for (int32_t s = 0; s < S; ++s) {
      const int32_t np = (int32_t)ceil_div(P->seg_len[s], sp::kPageSize);
      P->seg_first_page[s] = (int32_t)page_table.size();
      if (P->seg_shared[s]) {
        sp::cache_alloc(*cache, np, P->seg_pages[s]);
        page_table.insert(page_table.end(), P->seg_pages[s].begin(), P->seg_pages[s].end());
        P->seg_tokens[s].assign(tokens + seg_src[s], tokens + seg_src[s] + P->seg_len[s]);
      } else {
        page_table.insert(page_table.end(), (size_t)np, 0);
      }
    }
    P->stats.pages_used = need;
    P->pool_pages = (int64_t)cache->page_free.size();
    for (auto& grp : groups) P->group_end.push_back(grp.end);
  }

  // ---- staged rounds per request ---------------------------------------
  P->branch_round.assign(N, -1);
  P->branch_recompute.assign(N, 0);
  P->branch_last_seg.resize(N);
  P->branch_last_row.resize(N);
  int32_t n_rounds = 0;
  {
    std::vector<char> cached(S, 0);
    std::vector<int32_t> claim_stamp(S, -1);
    int32_t stamp = 0;
    for (auto& grp : groups) {
      std::vector<int32_t> unscored = grp.members;
      int32_t rnd = 0;
      while (!unscored.empty()) {
        ++stamp;
        std::vector<int32_t> joined, rest;
        for (int32_t b : unscored) {
          bool ok = true;
          for (int32_t s : path[b])
            if (P->seg_shared[s] && !cached[s] && claim_stamp[s] == stamp) { ok = false; break; }
          if (!ok) { rest.push_back(b); continue; }
          joined.push_back(b);
          for (int32_t s : path[b])
            if (P->seg_shared[s] && !cached[s]) {
              claim_stamp[s] = stamp;
              P->seg_round[s] = rnd;
            }
        }
        for (int32_t b : joined) {
          P->branch_round[b] = rnd;
          int32_t last = path[b].back();
          P->branch_recompute[b] = (P->seg_shared[last] && cached[last]) ? 1 : 0;
          for (int32_t s : path[b]) cached[s] = 1;
        }
        unscored.swap(rest);
        ++rnd;
      }
      n_rounds = std::max(n_rounds, rnd);
    }
  }
  for (int32_t b = 0; b < N; ++b) {
    int32_t last = path[b].back();
    P->branch_last_seg[b] = last;
    P->branch_last_row[b] = P->seg_node_start[last] + P->seg_len[last] - 1;
    if (!P->seg_shared[last]) P->seg_round[last] = P->branch_round[b];
  }
  P->round_off.assign(n_rounds + 1, 0);
  for (int32_t b = 0; b < N; ++b) P->round_off[P->branch_round[b] + 1] += 1;
  for (int32_t r = 0; r < n_rounds; ++r) P->round_off[r + 1] += P->round_off[r];
  P->round_branches.resize(N);
  {
    std::vector<int32_t> fill(P->round_off.begin(), P->round_off.end() - 1);
    for (int32_t b = 0; b < N; ++b) P->round_branches[fill[P->branch_round[b]]++] = b;
  }

  // ---- segment descriptors and ancestor chains -------------------------
  std::vector<sp::SegDesc> segd(S);
  std::vector<int32_t> chain;
  std::vector<int64_t> anc_units(S, 0);
  // cached levels: descriptors S, S + 1, ... (K/V in the pool only), one per
  // (node, visible length) that a group's match passes through
  std::vector<std::vector<int32_t>> group_levels(groups.size());
  std::vector<int32_t> level_len;  // visible length per cached level
  {
    std::map<std::pair<int32_t, int32_t>, int32_t> level_of;
    for (size_t g = 0; g < groups.size(); ++g)
      for (auto& e : bchain[groups[g].members[0]]) {
        auto it = level_of.find(e);
        if (it == level_of.end()) {
          const int32_t id = S + (int32_t)level_len.size();
          level_of.emplace(e, id);
          sp::SegDesc d{};
          d.node_start = 0;
          d.len = e.second;
          d.page_off = (int32_t)page_table.size();
          d.chain_off = 0;
          d.chain_len = 0;
          d.round = -1;
          d.shared = 2;  // cached: read from the pool only
          const std::vector<int32_t>& pg = cache->nodes[e.first].pages;
          page_table.insert(page_table.end(), pg.begin(), pg.end());
          segd.push_back(d);
          level_len.push_back(e.second);
          it = level_of.find(e);
        }
        group_levels[g].push_back(it->second);
      }
  }
  for (int32_t s = 0; s < S; ++s) {
    std::vector<int32_t> anc = group_levels[P->seg_group[s]];
    const size_t n_cached = anc.size();
    for (int32_t p = P->seg_parent[s]; p >= 0; p = P->seg_parent[p]) anc.push_back(p);
    std::reverse(anc.begin() + (long)n_cached, anc.end());
    segd[s].node_start = P->seg_node_start[s];
    segd[s].len = P->seg_len[s];
    segd[s].page_off = P->seg_first_page[s];
    segd[s].chain_off = (int32_t)chain.size();
    segd[s].chain_len = (int32_t)anc.size();
    segd[s].round = P->seg_round[s];
    segd[s].shared = P->seg_shared[s] ? 1 : 0;
    for (int32_t a : anc) {
      chain.push_back(a);
      const int32_t alen = a < S ? P->seg_len[a] : level_len[a - S];
      anc_units[s] += ceil_div(alen, sp::kKeysPerUnit);
    }
  }

  // ---- launch lists per round ------------------------------------------
  const int32_t G = shape->n_q_heads / shape->n_kv_heads;
  const int32_t TPT = sp::kRowsPerTile / G;
  const int32_t Hkv = shape->n_kv_heads;
  // one attention CTA per SM (the kernel holds all 512 TMEM columns)
  const int64_t part_target = std::max<int64_t>(1, ((int64_t)P->n_sms + Hkv - 1) / Hkv);
  std::vector<sp::AppendDesc> appends;
  std::vector<sp::TileDesc> tiles;
  std::vector<sp::MergeDesc> merges;
  int64_t max_parts = 0;
  // calls[kCallKinds r + kind] for rounds r < n_rounds; calls[kCallKinds
  // n_rounds + kind] run the work of every round in one call.  Kind 0 holds
  // the shared segments (prefix call), kind 1 the leaves and the recomputed
  // final rows (branch call), kind 2 both (tree call).  A call reads the levels
  // it computes itself from the k / v inputs and every other level from the
  // pool, which earlier calls have filled, so any grouping of rounds and kinds
  // into calls is valid.
  P->calls.resize((size_t)sp_plan::kCallKinds * ((size_t)n_rounds + 1));
  for (int32_t r = 0; r <= n_rounds; ++r) {
    const bool all = r == n_rounds;
    for (int kind = 0; kind < sp_plan::kCallKinds; ++kind) {
      sp_plan::Call& call = P->calls[(size_t)sp_plan::kCallKinds * r + kind];
      struct Raw {
        int32_t seg, t0, nt;
        int64_t units;
        int32_t seg2, t0b, ntb;  // a paired sibling tail (seg2 >= 0)
      };
      std::vector<Raw> raw;
      call.append_off = (int64_t)appends.size();
      for (int32_t s = 0; s < S; ++s) {
        if (!all && P->seg_round[s] != r) continue;
        if (kind < 2 && (kind == 0) != (P->seg_shared[s] != 0)) continue;
        if (P->seg_shared[s])  // leaves are read by no later call
          for (int32_t pg = 0; pg < ceil_div(P->seg_len[s], sp::kPageSize); ++pg)
            appends.push_back({s, pg});
        for (int32_t t0 = 0; t0 < P->seg_len[s]; t0 += TPT) {
          int32_t nt = std::min(TPT, P->seg_len[s] - t0);
          raw.push_back({s, t0, nt, anc_units[s] + ceil_div(t0 + nt, sp::kKeysPerUnit), -1, 0, 0});
        }
      }
      if (kind >= 1) {
        const int32_t i0 = all ? 0 : P->round_off[r], i1 = all ? N : P->round_off[r + 1];
        for (int32_t i = i0; i < i1; ++i) {
          int32_t b = all ? i : P->round_branches[i];
          if (!P->branch_recompute[b]) continue;
          int32_t s = P->branch_last_seg[b];
          int32_t t0 = P->seg_len[s] - 1;
          raw.push_back({s, t0, 1, anc_units[s] + ceil_div(t0 + 1, sp::kKeysPerUnit), -1, 0, 0});
        }
      }
      call.n_append = (int64_t)appends.size() - call.append_off;
      // When the call has fewer tiles than one wave of CTAs, split the long
      // tiles' KV walks into parts (merged afterwards) so the call fills the
      // GPU, keeping the total within one wave; then order them (below).
      const bool split_mode = (int64_t)raw.size() < part_target;
      // Otherwise pair the last tiles of sibling leaves whose tokens fit one
      // 128-row half each: one CTA walks their common ancestors once, then
      // both own segments (each half masking the other's), where two CTAs
      // would each run one half alone.
      if (!split_mode) {
        const int32_t half = TPT / 2;
        std::map<int32_t, size_t> open;  // parent segment -> an unpaired tail
        std::vector<char> drop(raw.size(), 0);
        for (size_t i = 0; i < raw.size(); ++i) {
          const Raw& x = raw[i];
          const int32_t par = P->seg_parent[x.seg];
          if (P->seg_shared[x.seg] || par < 0 || x.nt > half || x.t0 + x.nt != P->seg_len[x.seg])
            continue;
          auto it = open.find(par);
          if (it == open.end()) {
            open[par] = i;
            continue;
          }
          Raw& y = raw[it->second];
          y.seg2 = x.seg;
          y.t0b = x.t0;
          y.ntb = x.nt;
          y.units += ceil_div(x.t0 + x.nt, sp::kKeysPerUnit);  // x's own units
          drop[i] = 1;
          open.erase(it);
        }
        size_t w = 0;
        for (size_t i = 0; i < raw.size(); ++i)
          if (!drop[i]) raw[w++] = raw[i];
        raw.resize(w);
      }
      int64_t total_units = 0, max_units = 0;
      for (auto& x : raw) {
        total_units += x.units;
        max_units = std::max<int64_t>(max_units, x.units);
      }
      int64_t budget = std::max<int64_t>(max_units, 1);  // no split
      if (split_mode) {
        budget = std::max<int64_t>(kMinUnitsPerPart, ceil_div(std::max<int64_t>(total_units, 1), part_target));
        auto n_ctas = [&](int64_t b) {
          int64_t n = 0;
          for (auto& x : raw) n += ceil_div(x.units, b);
          return n;
        };
        while (budget < max_units && n_ctas(budget) > part_target) ++budget;
      }
      struct Work { sp::TileDesc t; int64_t units; };
      std::vector<Work> work;
      call.merge_off = (int64_t)merges.size();
      int32_t parts = 0;
      for (auto& x : raw) {
        if (x.units <= budget) {
          work.push_back({{x.seg, x.t0, x.nt, 0, (int32_t)x.units, -1, -1, x.seg2, x.t0b, x.ntb, 0, 0},
                          x.units});
          continue;
        }
        int32_t np = (int32_t)ceil_div(x.units, budget);
        const int32_t mi = (int32_t)(merges.size() - call.merge_off);  // index within the call
        merges.push_back({x.seg, x.t0, x.nt, parts, np, 0, 0, 0});
        for (int32_t i = 0; i < np; ++i) {
          int32_t lo = (int32_t)(x.units * i / np), hi = (int32_t)(x.units * (i + 1) / np);
          work.push_back({{x.seg, x.t0, x.nt, lo, hi, parts + i, mi, -1, 0, 0, 0, 0}, (int64_t)(hi - lo)});
        }
        parts += np;
      }
      // Blocks start in list order.  Requests go one after another, so the
      // CTAs running at any moment read the KV of one or two requests, which
      // stays in L2 (taking every request's longest tiles first instead mixes
      // all of a batch's requests at once: a 64-request batch then read its
      // K / V from DRAM about four times over).  Within a request the longest
      // tiles go first, so the last blocks of the call are short ones.
      std::stable_sort(work.begin(), work.end(), [&](const Work& a, const Work& b) {
        const int32_t ra = P->seg_req[a.t.seg], rb = P->seg_req[b.t.seg];
        if (ra != rb) return ra < rb;
        return a.units > b.units;
      });
      call.tile_off = (int64_t)tiles.size();
      for (auto& w : work) tiles.push_back(w.t);
      call.n_tiles = (int64_t)work.size();
      call.n_merges = (int64_t)merges.size() - call.merge_off;
      call.n_parts = parts;
      max_parts = std::max<int64_t>(max_parts, parts);
    }
  }

  // ---- descriptor image --------------------------------------------------
  sp::DescHeader h{};
  size_t off = align256(sizeof(sp::DescHeader));
  h.off_segs = (int64_t)off;    off = align256(off + segd.size() * sizeof(sp::SegDesc));
  h.off_pages = (int64_t)off;   off = align256(off + page_table.size() * sizeof(int32_t));
  h.off_chain = (int64_t)off;   off = align256(off + chain.size() * sizeof(int32_t));
  h.off_append = (int64_t)off;  off = align256(off + appends.size() * sizeof(sp::AppendDesc));
  h.off_tiles = (int64_t)off;   off = align256(off + tiles.size() * sizeof(sp::TileDesc));
  h.off_merges = (int64_t)off;  off = align256(off + merges.size() * sizeof(sp::MergeDesc));
  h.n_segs = (int64_t)segd.size();
  h.n_pages = (int64_t)page_table.size();
  h.n_chain = (int64_t)chain.size();
  h.n_append = (int64_t)appends.size();
  h.n_tiles = (int64_t)tiles.size();
  h.n_merges = (int64_t)merges.size();
  P->blob.assign(off, 0);
  std::memcpy(P->blob.data(), &h, sizeof(h));
  if (!segd.empty()) std::memcpy(P->blob.data() + h.off_segs, segd.data(), segd.size() * sizeof(sp::SegDesc));
  if (!page_table.empty())
    std::memcpy(P->blob.data() + h.off_pages, page_table.data(), page_table.size() * sizeof(int32_t));
  if (!chain.empty()) std::memcpy(P->blob.data() + h.off_chain, chain.data(), chain.size() * sizeof(int32_t));
  if (!appends.empty()) std::memcpy(P->blob.data() + h.off_append, appends.data(), appends.size() * sizeof(sp::AppendDesc));
  if (!tiles.empty()) std::memcpy(P->blob.data() + h.off_tiles, tiles.data(), tiles.size() * sizeof(sp::TileDesc));
  if (!merges.empty()) std::memcpy(P->blob.data() + h.off_merges, merges.data(), merges.size() * sizeof(sp::MergeDesc));
  P->hdr = h;

  // ---- statistics --------------------------------------------------------
  int64_t logical = 0, recomputed = 0;
  for (int32_t b = 0; b < N; ++b) {
    logical += tok_offsets[b + 1] - tok_offsets[b];
    recomputed += P->branch_recompute[b];
  }
  int64_t shared = 0;
  for (int32_t s = 0; s < S; ++s) shared += P->seg_shared[s];
  P->stats.n_requests = P->n_requests;
  P->stats.n_branches = N;
  P->stats.n_segments = S;
  P->stats.n_shared_segments = shared;
  P->stats.n_rounds = n_rounds;
  P->stats.logical_tokens = logical;
  P->stats.computed_tokens = P->stats.node_tokens + recomputed;
  P->stats.reused_tokens = logical - P->stats.computed_tokens;
  P->stats.cache_hit_tokens = hit_tokens;
  P->stats.desc_bytes = (int64_t)P->blob.size();
  // partial O and lse per split part
  P->stats.attn_workspace_bytes = (int64_t)align256(
      (size_t)std::max<int64_t>(max_parts, 1) * Hkv * sp::kRowsPerTile * (shape->head_dim + 1) *
      sizeof(float));
  *out = P;
  return SP_OK;
}

}  // namespace

extern "C" sp_status sp_plan_build(const sp_shape* shape, int32_t n_branches,
                                   const int32_t* req_of_branch, const int64_t* tok_offsets,
                                   const int32_t* tokens, int32_t max_pages, int32_t n_sms,
                                   sp_plan** out) {
  return build(shape, nullptr, n_branches, req_of_branch, tok_offsets, tokens, max_pages, n_sms,
               out);
}

extern "C" sp_status sp_plan_build_cached(const sp_shape* shape, sp_cache* cache,
                                          int32_t n_branches, const int32_t* req_of_branch,
                                          const int64_t* tok_offsets, const int32_t* tokens,
                                          int32_t n_sms, sp_plan** out) {
  if (!cache) {
    if (out) *out = nullptr;
    return SP_ERR_ARG;
  }
  return build(shape, cache, n_branches, req_of_branch, tok_offsets, tokens, 0, n_sms, out);
}

extern "C" void sp_plan_free(sp_plan* plan) { delete plan; }

extern "C" sp_status sp_plan_get_stats(const sp_plan* plan, sp_plan_stats* out) {
  if (!plan || !out) return SP_ERR_ARG;
  *out = plan->stats;
  return SP_OK;
}

extern "C" sp_status sp_plan_rounds(const sp_plan* plan, int32_t* n_rounds,
                                    const int32_t** round_offsets,
                                    const int32_t** round_branches) {
  if (!plan || !n_rounds || !round_offsets || !round_branches) return SP_ERR_ARG;
  *n_rounds = (int32_t)plan->stats.n_rounds;
  *round_offsets = plan->round_off.data();
  *round_branches = plan->round_branches.data();
  return SP_OK;
}

extern "C" sp_status sp_plan_segments(const sp_plan* plan, int32_t* n_segments,
                                      const int32_t** seg_req, const int32_t** seg_parent,
                                      const int64_t** seg_node_start, const int32_t** seg_len,
                                      const int32_t** seg_round, const int32_t** seg_shared,
                                      const int32_t** seg_first_page) {
  if (!plan || !n_segments || !seg_req || !seg_parent || !seg_node_start || !seg_len ||
      !seg_round || !seg_shared || !seg_first_page)
    return SP_ERR_ARG;
  *n_segments = (int32_t)plan->seg_len.size();
  *seg_req = plan->seg_req.data();
  *seg_parent = plan->seg_parent.data();
  *seg_node_start = plan->seg_node_start.data();
  *seg_len = plan->seg_len.data();
  *seg_round = plan->seg_round.data();
  *seg_shared = plan->seg_shared.data();
  *seg_first_page = plan->seg_first_page.data();
  return SP_OK;
}

extern "C" sp_status sp_plan_segment_sources(const sp_plan* plan, const int32_t** seg_branch,
                                             const int32_t** seg_pos) {
  if (!plan || !seg_branch || !seg_pos) return SP_ERR_ARG;
  *seg_branch = plan->seg_branch.data();
  *seg_pos = plan->seg_pos.data();
  return SP_OK;
}

extern "C" sp_status sp_plan_branches(const sp_plan* plan, const int32_t** branch_last_seg,
                                      const int64_t** branch_last_row,
                                      const int32_t** branch_round,
                                      const int32_t** branch_recompute) {
  if (!plan || !branch_last_seg || !branch_last_row || !branch_round || !branch_recompute)
    return SP_ERR_ARG;
  *branch_last_seg = plan->branch_last_seg.data();
  *branch_last_row = plan->branch_last_row.data();
  *branch_round = plan->branch_round.data();
  *branch_recompute = plan->branch_recompute.data();
  return SP_OK;
}

extern "C" sp_status sp_plan_descriptor(const sp_plan* plan, const void** data, size_t* bytes) {
  if (!plan || !data || !bytes) return SP_ERR_ARG;
  *data = plan->blob.data();
  *bytes = plan->blob.size();
  return SP_OK;
}

extern "C" sp_status sp_plan_call_info(const sp_plan* plan, int32_t round, int32_t kind,
                                       int64_t info[7]) {
  if (!plan || !info || round < -1 || round >= plan->stats.n_rounds || kind < 0 ||
      kind >= sp_plan::kCallKinds)
    return SP_ERR_ARG;
  const int32_t r = round < 0 ? (int32_t)plan->stats.n_rounds : round;
  const sp_plan::Call& c = plan->calls[(size_t)sp_plan::kCallKinds * r + kind];
  info[0] = c.append_off;
  info[1] = c.n_append;
  info[2] = c.tile_off;
  info[3] = c.n_tiles;
  info[4] = c.merge_off;
  info[5] = c.n_merges;
  info[6] = c.n_parts;
  return SP_OK;
}

extern "C" sp_status sp_check_labels(const int32_t* label_off, const int32_t* label_ids,
                                     int32_t N, int32_t vocab) {
  if (!label_off || N <= 0 || vocab < 2) return SP_ERR_ARG;
  if (label_off[0] != 0) return SP_ERR_ARG;
  for (int32_t n = 0; n < N; ++n) {
    int32_t k = label_off[n + 1] - label_off[n];
    if (k < 2 || k > 64) return SP_ERR_ARG;
  }
  if (label_off[N] > 0 && !label_ids) return SP_ERR_ARG;
  for (int32_t j = 0; j < label_off[N]; ++j)
    if (label_ids[j] < 0 || label_ids[j] >= vocab) return SP_ERR_ARG;
  return SP_OK;
}

extern "C" sp_status sp_check_options(const int32_t* opt_off, int32_t n_opts, int32_t n_rows,
                                      const int32_t* q_off, int32_t n_questions) {
  if (!opt_off || !q_off || n_opts < 2 || n_rows < 1 || n_questions < 1) return SP_ERR_ARG;
  if (opt_off[0] != 0 || opt_off[n_opts] > n_rows || q_off[0] != 0 || q_off[n_questions] > n_opts)
    return SP_ERR_ARG;
  for (int32_t o = 0; o < n_opts; ++o)
    if (opt_off[o + 1] <= opt_off[o]) return SP_ERR_ARG;
  for (int32_t q = 0; q < n_questions; ++q) {
    const int32_t k = q_off[q + 1] - q_off[q];
    if (k < 2 || k > 64) return SP_ERR_ARG;
  }
  return SP_OK;
}

extern "C" const char* sp_status_str(sp_status s) {
  switch (s) {
    case SP_OK: return "ok";
    case SP_ERR_ARG: return "invalid argument";
    case SP_ERR_LIMIT: return "request limit exceeded";
    case SP_ERR_POOL_FULL: return "KV pool too small for the plan";
    case SP_ERR_CUDA: return "CUDA error";
    case SP_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case SP_ERR_DEVICE_BOUNDS: return "device bounds check failed";
    case SP_ERR_WORKSPACE: return "workspace or descriptor buffer too small";
  }
  return "unknown status";
}
