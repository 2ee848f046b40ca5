// Prefix cache across calls: a radix tree of the shared segments earlier plans
// computed, owning their pool pages, with least-recently-used eviction.
//
// Sources: LLM2Jev "shared prefix" page, section on reusing SGLang's radix
// cache (the engine keeps token prefixes whose KV exists across requests, a
// later input continues from its first uncached position, prefixes are
// evicted when memory is short; a hot request finds its prefix cached) and
// the openjev-sglang article, section on the repeated state (requests that
// repeat a state and change the questions read only their questions).
//
// Rules (the pages leave them open; the oracle states the same ones):
// * a branch reuses its longest cached prefix, whole nodes and possibly the
//   start of one more, capped one short of its length (its last position is
//   always computed);
// * after a plan ran, its new shared segments are inserted under the node
//   where their group's match ended, when it ended on a node boundary and no
//   child of that node starts with the same token;
// * when the free pages do not cover a plan, unpinned cache leaves are
//   evicted, least recently used first (ties: older node first);
// * pages: the lowest run of free consecutive pages, else the lowest free.
#include <algorithm>
#include <new>

#include "plan_internal.h"

namespace sp {

int64_t cache_match(const sp_cache& c, const int32_t* seq, int64_t L,
                    std::vector<std::pair<int32_t, int32_t>>& chain) {
  chain.clear();
  int32_t cur = 0;
  int64_t pos = 0;
  while (pos < L) {
    int32_t nxt = -1;
    for (int32_t ch : c.nodes[cur].children)
      if (c.nodes[ch].tokens[0] == seq[pos]) {
        nxt = ch;
        break;
      }
    if (nxt < 0) break;
    const std::vector<int32_t>& toks = c.nodes[nxt].tokens;
    int64_t m = 0;
    while (m < (int64_t)toks.size() && pos + m < L && toks[m] == seq[pos + m]) ++m;
    chain.push_back({nxt, (int32_t)m});
    pos += m;
    if (m < (int64_t)toks.size()) break;
    cur = nxt;
  }
  return pos;
}

bool cache_evict_one(sp_cache& c) {
  int32_t best = -1;
  for (int32_t i = 1; i < (int32_t)c.nodes.size(); ++i) {
    const sp_cache::Node& n = c.nodes[i];
    if (!n.alive || n.pins > 0) continue;
    bool leaf = true;
    for (int32_t ch : n.children)
      if (c.nodes[ch].alive) {
        leaf = false;
        break;
      }
    if (!leaf) continue;
    if (best < 0 || n.last_used < c.nodes[best].last_used) best = i;
  }
  if (best < 0) return false;
  sp_cache::Node& n = c.nodes[best];
  n.alive = false;
  for (int32_t p : n.pages) {
    c.page_free[p] = 1;
    ++c.n_free;
  }
  std::vector<int32_t>& sib = c.nodes[n.parent].children;
  sib.erase(std::find(sib.begin(), sib.end(), best));
  ++c.evictions;
  return true;
}

void cache_alloc(sp_cache& c, int32_t n, std::vector<int32_t>& out) {
  out.clear();
  const int32_t P = (int32_t)c.page_free.size();
  int32_t run = 0;
  for (int32_t p = 0; p < P; ++p) {
    run = c.page_free[p] ? run + 1 : 0;
    if (run == n) {
      for (int32_t q = p - n + 1; q <= p; ++q) out.push_back(q);
      break;
    }
  }
  if ((int32_t)out.size() < n) {
    out.clear();
    for (int32_t p = 0; p < P && (int32_t)out.size() < n; ++p)
      if (c.page_free[p]) out.push_back(p);
  }
  for (int32_t p : out) c.page_free[p] = 0;
  c.n_free -= (int64_t)out.size();
}

}  // namespace sp

sp_plan::~sp_plan() {
  if (!cache) return;
  for (int32_t nd : pinned) cache->nodes[nd].pins -= 1;
  for (auto& pg : seg_pages)
    for (int32_t p : pg) {
      cache->page_free[p] = 1;
      ++cache->n_free;
    }
}

extern "C" sp_status sp_cache_create(int32_t n_pages, sp_cache** out) {
  if (!out) return SP_ERR_ARG;
  *out = nullptr;
  if (n_pages < 1) return SP_ERR_ARG;
  sp_cache* c = new (std::nothrow) sp_cache();
  if (!c) return SP_ERR_ARG;
  c->nodes.emplace_back();  // root
  c->page_free.assign((size_t)n_pages, 1);
  c->n_free = n_pages;
  *out = c;
  return SP_OK;
}

extern "C" void sp_cache_free(sp_cache* cache) { delete cache; }

extern "C" sp_status sp_cache_get_stats(const sp_cache* c, int64_t out[5]) {
  if (!c || !out) return SP_ERR_ARG;
  int64_t nodes = 0, tokens = 0;
  for (size_t i = 1; i < c->nodes.size(); ++i)
    if (c->nodes[i].alive) {
      ++nodes;
      tokens += (int64_t)c->nodes[i].tokens.size();
    }
  out[0] = nodes;
  out[1] = tokens;
  out[2] = (int64_t)c->page_free.size() - c->n_free;
  out[3] = c->n_free;
  out[4] = c->evictions;
  return SP_OK;
}

extern "C" sp_status sp_cache_commit(sp_cache* c, sp_plan* P) {
  if (!c || !P || P->cache != c) return SP_ERR_ARG;
  if (P->committed) return SP_OK;
  P->committed = true;
  const int64_t stamp = c->clock++;
  const int32_t S = (int32_t)P->seg_len.size();
  for (int32_t s = 0; s < S; ++s) {
    if (!P->seg_shared[s]) continue;
    int32_t parent;
    if (P->seg_parent[s] >= 0) {
      parent = P->seg_cache_node[P->seg_parent[s]];
      if (parent < 0) continue;
    } else {
      const auto& end = P->group_end[P->seg_group[s]];
      if (end.first > 0 && end.second < (int32_t)c->nodes[end.first].tokens.size())
        continue;  // the match ended inside a node
      parent = end.first;
    }
    const std::vector<int32_t>& toks = P->seg_tokens[s];
    bool taken = false;
    for (int32_t ch : c->nodes[parent].children)
      if (c->nodes[ch].tokens[0] == toks[0]) {
        taken = true;
        break;
      }
    if (taken) continue;
    sp_cache::Node n;
    n.tokens = toks;
    n.pages.swap(P->seg_pages[s]);  // the cache owns them now
    n.parent = parent;
    n.last_used = stamp;
    const int32_t id = (int32_t)c->nodes.size();
    c->nodes.push_back(std::move(n));
    c->nodes[parent].children.push_back(id);
    P->seg_cache_node[s] = id;
  }
  return SP_OK;
}
