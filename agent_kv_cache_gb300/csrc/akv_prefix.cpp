// History-keyed prefix index: radix tree of published snapshots' context
// records, exact / retrigger matching, drop-aware eviction order.
//
// "Cache Engineering for Agents" paper review, Appendix A.1.2 (Reposition
// Scheme): a token record T(x, p) has the token id and the position of the
// key as stored now; an exact match needs equal ids, positions and operation
// records; the projection phi drops the positions, and a phi-equal prefix
// can be reused after rotating its keys.  The longest valid exact prefix is
// the start, a compatible prefix wins only when strictly longer, and the
// search stops at the first differing token or operation.  4.2.2 / "[Repo
// Review] AKV" 5.6: dropped caches are evicted before finished ones, via
// two heaps, and only the DELTA records on an entry's own extending path
// prove its KV unneeded.
//
// Positions are not stored in the tree: with the records equal up to n,
// positions follow from the records (Eq. 6), so the tree compares phi
// records, and exactness is decided per entry from its stored positions.
#include "akv_prefix.h"

#include <algorithm>
#include <cstring>
#include <queue>
#include <string>

namespace akv {

PrefixIndex::PrefixIndex(int32_t page_size) : S_(page_size) {
  nodes_.emplace_back();   // root
}

int PrefixIndex::expand(const akv_op* ops, int32_t n_ops, const int32_t* token_ids,
                        int32_t n_tokens, PProgram* out, const char** why) {
  out->recs.clear();
  out->rec_op.clear();
  out->rec_tok.clear();
  out->op_count.assign(n_ops > 0 ? (size_t)n_ops : 0, 0);
  if (n_ops < 0 || (n_ops > 0 && !ops) || n_tokens < 0 || (n_tokens > 0 && !token_ids)) {
    *why = "bad program arguments";
    return AKV_EINVAL;
  }
  int64_t t = 0;
  for (int32_t i = 0; i < n_ops; ++i) {
    const akv_op& op = ops[i];
    if (op.kind == AKV_OP_APPEND) {
      if (op.count < 0 || t + op.count > n_tokens) {
        *why = "program appends more tokens than token ids given";
        return AKV_EINVAL;
      }
      out->op_count[i] = op.count;
      for (int32_t k = 0; k < op.count; ++k) {
        out->recs.push_back({kRecT, token_ids[t++]});
        out->rec_op.push_back(i);
        out->rec_tok.push_back(k);
      }
    } else if (op.kind == AKV_OP_DROP) {
      if (op.count < 0 || (op.count > 0 && !op.ranges)) {
        *why = "bad drop op";
        return AKV_EINVAL;
      }
      std::vector<std::pair<int64_t, int64_t>> rs;
      for (int32_t r = 0; r < op.count; ++r) {
        const int64_t b = op.ranges[2 * r], e = op.ranges[2 * r + 1];
        if (b < 0 || e < b || e > t) {
          *why = "drop range outside the appended tokens";
          return AKV_ERANGE;
        }
        if (e > b) rs.push_back({b, e});
      }
      std::sort(rs.begin(), rs.end());
      std::vector<std::pair<int64_t, int64_t>> m;
      for (const auto& r : rs) {
        if (!m.empty() && r.first <= m.back().second)
          m.back().second = std::max(m.back().second, r.second);
        else
          m.push_back(r);
      }
      if (m.empty()) continue;             // an empty drop is no operation
      auto it = delta_ids_.find(m);
      int32_t id;
      if (it == delta_ids_.end()) {
        id = (int32_t)deltas_.size();
        deltas_.push_back(m);
        delta_ids_.emplace(m, id);
      } else {
        id = it->second;
      }
      out->recs.push_back({kRecD, id});
      out->rec_op.push_back(i);
      out->rec_tok.push_back(0);
    } else if (op.kind == AKV_OP_REPOS) {
      out->recs.push_back({kRecR, 0});
      out->rec_op.push_back(i);
      out->rec_tok.push_back(0);
    } else {
      *why = "unknown op kind";
      return AKV_EINVAL;
    }
  }
  if (t != n_tokens) {
    *why = "program appends fewer tokens than token ids given";
    return AKV_EINVAL;
  }
  out->n_tokens = (int32_t)t;
  return AKV_OK;
}

PrefixIndex::State PrefixIndex::replay(const std::vector<PRec>& recs, size_t n) const {
  State s;
  for (size_t i = 0; i < n; ++i) {
    const PRec& r = recs[i];
    if (r.kind == kRecT) {
      s.active.push_back(1);
      s.held.push_back(1);
      s.pos.push_back(s.next_pos++);
    } else if (r.kind == kRecD) {
      for (const auto& iv : deltas_[r.v])
        for (int64_t t = iv.first; t < iv.second && t < (int64_t)s.active.size(); ++t) s.active[t] = 0;
    } else {
      int32_t j = 0;
      for (size_t t = 0; t < s.active.size(); ++t) {
        s.held[t] = s.active[t];
        if (s.active[t]) s.pos[t] = j++;
      }
      s.next_pos = j;
    }
  }
  return s;
}

int PrefixIndex::insert(int64_t id, const PProgram& p, int64_t use_time) {
  if (id < 0 || entries_.count(id)) return AKV_EINVAL;
  PEntry e;
  e.id = id;
  e.recs = p.recs;
  e.last_use = use_time >= 0 ? use_time : tick();
  // stored keys: slot held and its page holding an active token
  const State st = replay(e.recs, e.recs.size());
  const size_t n = st.active.size();
  std::vector<char> live_page((size_t)st.next_pos / S_ + 1, 0);
  for (size_t t = 0; t < n; ++t)
    if (st.active[t]) live_page[st.pos[t] / S_] = 1;
  e.stored.assign(n, -1);
  e.active.assign(st.active.begin(), st.active.end());
  for (size_t t = 0; t < n; ++t)
    if (st.held[t] && live_page[st.pos[t] / S_]) e.stored[t] = st.pos[t];
  // walk / split the radix tree
  int x = 0;
  size_t i = 0;
  const std::vector<PRec>& r = e.recs;
  while (i < r.size()) {
    auto it = nodes_[x].kids.find(key(r[i]));
    if (it == nodes_[x].kids.end()) {
      PNode leaf;
      leaf.parent = x;
      leaf.label.assign(r.begin() + i, r.end());
      leaf.depth = (int32_t)r.size();
      const int id_leaf = (int)nodes_.size();
      nodes_.push_back(std::move(leaf));
      nodes_[x].kids[key(r[i])] = id_leaf;
      x = id_leaf;
      i = r.size();
      break;
    }
    const int c = it->second;
    const std::vector<PRec>& L = nodes_[c].label;
    size_t k = 0;
    while (k < L.size() && i + k < r.size() && L[k] == r[i + k]) ++k;
    if (k == L.size()) {
      x = c;
      i += k;
      continue;
    }
    // split c after k records
    PNode mid;
    mid.parent = x;
    mid.label.assign(L.begin(), L.begin() + k);
    mid.depth = nodes_[x].depth + (int32_t)k;
    const int m = (int)nodes_.size();
    nodes_.push_back(std::move(mid));
    std::vector<PRec> rest(nodes_[c].label.begin() + k, nodes_[c].label.end());
    nodes_[c].label = std::move(rest);
    nodes_[c].parent = m;
    nodes_[m].kids[key(nodes_[c].label[0])] = c;
    nodes_[x].kids[key(r[i])] = m;
    x = m;
    i += k;
  }
  nodes_[x].ends.push_back(id);
  e.node = x;
  entries_.emplace(id, std::move(e));
  return AKV_OK;
}

int PrefixIndex::remove(int64_t id) {
  auto it = entries_.find(id);
  if (it == entries_.end()) return AKV_ENOSEQ;
  int x = it->second.node;
  auto& ends = nodes_[x].ends;
  ends.erase(std::find(ends.begin(), ends.end(), id));
  entries_.erase(it);
  // prune leaves left without entries
  while (x != 0 && nodes_[x].ends.empty() && nodes_[x].kids.empty()) {
    const int p = nodes_[x].parent;
    nodes_[p].kids.erase(key(nodes_[x].label[0]));
    nodes_[x].live = false;
    nodes_[x].label.clear();
    x = p;
  }
  return AKV_OK;
}

const PEntry* PrefixIndex::entry(int64_t id) const {
  auto it = entries_.find(id);
  return it == entries_.end() ? nullptr : &it->second;
}

void PrefixIndex::touch(int64_t id, int64_t use_time) {
  auto it = entries_.find(id);
  if (it != entries_.end()) it->second.last_use = use_time >= 0 ? use_time : tick();
}

int64_t PrefixIndex::find_equal(const PProgram& p) const {
  int x = 0;
  size_t i = 0;
  while (i < p.recs.size()) {
    auto it = nodes_[x].kids.find(key(p.recs[i]));
    if (it == nodes_[x].kids.end()) return -1;
    const std::vector<PRec>& L = nodes_[it->second].label;
    if (i + L.size() > p.recs.size()) return -1;
    for (size_t k = 0; k < L.size(); ++k)
      if (L[k] != p.recs[i + k]) return -1;
    i += L.size();
    x = it->second;
  }
  const auto& ends = nodes_[x].ends;
  return ends.empty() ? -1 : *std::min_element(ends.begin(), ends.end());
}

// Request state over req[0..m) against entry e's stored keys; records the
// longest prefix that is exact and the longest that is valid (with its
// rotated count).
void PrefixIndex::scan(const PEntry& e, const std::vector<PRec>& req, int32_t m,
                       int32_t* best_exact, int32_t* best_valid, int32_t* valid_rot) const {
  std::vector<char> act;
  std::vector<int32_t> pos;
  act.reserve(e.stored.size());
  pos.reserve(e.stored.size());
  int32_t next = 0;
  int64_t missing = 0, rotated = 0;
  *best_exact = 0;
  *best_valid = 0;
  *valid_rot = 0;
  auto count = [&](int64_t t, int sign) {
    const int32_t s = t < (int64_t)e.stored.size() ? e.stored[t] : -1;
    if (s < 0) missing += sign;
    else if (s != pos[t]) rotated += sign;
  };
  for (int32_t i = 0; i < m; ++i) {
    const PRec& r = req[i];
    if (r.kind == kRecT) {
      act.push_back(1);
      pos.push_back(next++);
      count((int64_t)act.size() - 1, +1);
    } else if (r.kind == kRecD) {
      for (const auto& iv : deltas_[r.v])
        for (int64_t t = iv.first; t < iv.second && t < (int64_t)act.size(); ++t)
          if (act[t]) { count(t, -1); act[t] = 0; }
    } else {
      int32_t j = 0;
      rotated = 0;
      for (size_t t = 0; t < act.size(); ++t) {
        if (!act[t]) continue;
        pos[t] = j++;
        const int32_t s = t < e.stored.size() ? e.stored[t] : -1;
        if (s >= 0 && s != pos[t]) ++rotated;
      }
      next = j;
    }
    if (missing == 0) {
      *best_valid = i + 1;
      *valid_rot = (int32_t)rotated;
      if (rotated == 0) *best_exact = i + 1;
    }
  }
}

PMatch PrefixIndex::match(const PProgram& req) const {
  PMatch out;
  const std::vector<PRec>& r = req.recs;
  // walk the request's records down the tree; path[k] = (node, matched depth)
  std::vector<std::pair<int, int32_t>> path;
  int x = 0;
  size_t i = 0;
  while (i < r.size()) {
    auto it = nodes_[x].kids.find(key(r[i]));
    if (it == nodes_[x].kids.end()) break;
    const int c = it->second;
    const std::vector<PRec>& L = nodes_[c].label;
    size_t k = 0;
    while (k < L.size() && i + k < r.size() && L[k] == r[i + k]) ++k;
    path.push_back({c, (int32_t)(i + k)});
    if (k < L.size()) break;
    x = c;
    i += k;
  }
  // common length of every entry below the path: deepest path node first
  std::vector<std::pair<int32_t, int64_t>> cand;   // (common length, id)
  std::vector<char> seen(nodes_.size(), 0);
  for (size_t k = path.size(); k-- > 0;) {
    const int top = path[k].first;
    const int32_t m = path[k].second;
    std::vector<int> stack{top};
    while (!stack.empty()) {
      const int y = stack.back();
      stack.pop_back();
      if (seen[y]) continue;
      seen[y] = 1;
      for (int64_t id : nodes_[y].ends) cand.push_back({m, id});
      for (const auto& kv : nodes_[y].kids) stack.push_back(kv.second);
    }
  }
  std::sort(cand.begin(), cand.end(), [](const auto& a, const auto& b) {
    return a.first != b.first ? a.first > b.first : a.second < b.second;
  });
  int32_t bx_n = 0, bv_n = 0, bv_rot = 0;
  int64_t bx_id = -1, bv_id = -1;
  for (const auto& c : cand) {
    if (c.first == 0 || c.first < bv_n) break;     // cannot reach the best any more
    const PEntry& e = entries_.at(c.second);
    int32_t ex, va, rot;
    scan(e, r, c.first, &ex, &va, &rot);
    if (ex > bx_n || (ex == bx_n && ex > 0 && c.second < bx_id)) { bx_n = ex; bx_id = c.second; }
    if (va > bv_n || (va == bv_n && va > 0 && (rot < bv_rot || (rot == bv_rot && c.second < bv_id)))) {
      bv_n = va;
      bv_rot = rot;
      bv_id = c.second;
    }
  }
  if (bv_n == 0) return out;
  int32_t n;
  if (bx_n >= bv_n) {
    out.kind = AKV_MATCH_EXACT;
    out.entry = bx_id;
    n = bx_n;
  } else {
    out.kind = AKV_MATCH_RETRIGGER;
    out.entry = bv_id;
    out.n_rotated = bv_rot;
    n = bv_n;
  }
  out.n_records = n;
  int32_t nt = 0;
  for (int32_t k = 0; k < n; ++k) nt += r[k].kind == kRecT;
  out.n_tokens = nt;
  const int32_t last = n - 1;
  if (r[last].kind == kRecT && req.rec_tok[last] + 1 < req.op_count[req.rec_op[last]]) {
    out.op_index = req.rec_op[last];
    out.op_tokens = req.rec_tok[last] + 1;
  } else {
    out.op_index = req.rec_op[last] + 1;
    out.op_tokens = 0;
  }
  return out;
}

std::vector<int64_t> PrefixIndex::evict_order() const {
  struct Item { int klass; int64_t use, id; };
  std::vector<Item> items;
  items.reserve(entries_.size());
  for (const auto& kv : entries_) {
    const PEntry& a = kv.second;
    // entries that extend a: everything below a's end node, except the ones
    // ending at it (equal records)
    std::vector<int64_t> ext;
    std::vector<int> stack;
    for (const auto& k : nodes_[a.node].kids) stack.push_back(k.second);
    while (!stack.empty()) {
      const int y = stack.back();
      stack.pop_back();
      for (int64_t id : nodes_[y].ends) ext.push_back(id);
      for (const auto& k : nodes_[y].kids) stack.push_back(k.second);
    }
    int klass = 1;
    if (!ext.empty()) {
      klass = 2;
      const size_t la = a.recs.size();
      for (int64_t b : ext) {
        const PEntry& eb = entries_.at(b);
        for (size_t i = la; i < eb.recs.size() && klass == 2; ++i) {
          if (eb.recs[i].kind != kRecD) continue;
          for (const auto& iv : deltas_[eb.recs[i].v]) {
            for (int64_t t = iv.first; t < iv.second && t < (int64_t)a.active.size(); ++t)
              if (a.active[t]) { klass = 0; break; }
            if (klass == 0) break;
          }
        }
        if (klass == 0) break;
      }
    }
    items.push_back({klass, a.last_use, a.id});
  }
  std::sort(items.begin(), items.end(), [](const Item& x, const Item& y) {
    if (x.klass != y.klass) return x.klass < y.klass;
    if (x.use != y.use) return x.use < y.use;
    return x.id < y.id;
  });
  std::vector<int64_t> out;
  out.reserve(items.size());
  for (const Item& it : items) out.push_back(it.id);
  return out;
}

}  // namespace akv

// ---- C ABI of the host-only index --------------------------------------------


namespace {
int pfail(akv_prefix_index* x, int code, const char* why) {
  if (x) x->err = why;
  return code;
}
}  // namespace

extern "C" {

int akv_prefix_index_create(int32_t page_size, akv_prefix_index** out) {
  if (!out || page_size < 1 || page_size > 64 || (page_size & (page_size - 1))) return AKV_EINVAL;
  *out = new akv_prefix_index{akv::PrefixIndex(page_size), std::string()};
  return AKV_OK;
}

int akv_prefix_index_destroy(akv_prefix_index* index) {
  delete index;
  return AKV_OK;
}

const char* akv_prefix_last_error(akv_prefix_index* index) {
  return index ? index->err.c_str() : "null index";
}

int akv_prefix_insert(akv_prefix_index* x, int64_t entry, const akv_op* ops, int32_t n_ops,
                      const int32_t* token_ids, int32_t n_tokens, int64_t use_time) {
  if (!x) return AKV_EINVAL;
  akv::PProgram p;
  const char* why = "";
  int rc = x->idx.expand(ops, n_ops, token_ids, n_tokens, &p, &why);
  if (rc) return pfail(x, rc, why);
  rc = x->idx.insert(entry, p, use_time);
  return rc ? pfail(x, rc, "entry id negative or already present") : AKV_OK;
}

int akv_prefix_remove(akv_prefix_index* x, int64_t entry) {
  if (!x) return AKV_EINVAL;
  const int rc = x->idx.remove(entry);
  return rc ? pfail(x, rc, "unknown entry") : AKV_OK;
}

int akv_prefix_touch(akv_prefix_index* x, int64_t entry, int64_t use_time) {
  if (!x) return AKV_EINVAL;
  if (!x->idx.has(entry)) return pfail(x, AKV_ENOSEQ, "unknown entry");
  x->idx.touch(entry, use_time);
  return AKV_OK;
}

int akv_prefix_match(akv_prefix_index* x, const akv_op* ops, int32_t n_ops,
                     const int32_t* token_ids, int32_t n_tokens, akv_prefix_match_t* out) {
  if (!x || !out) return AKV_EINVAL;
  akv::PProgram p;
  const char* why = "";
  const int rc = x->idx.expand(ops, n_ops, token_ids, n_tokens, &p, &why);
  if (rc) return pfail(x, rc, why);
  const akv::PMatch m = x->idx.match(p);
  out->kind = m.kind;
  out->n_records = m.n_records;
  out->entry = m.entry;
  out->n_tokens = m.n_tokens;
  out->n_rotated = m.n_rotated;
  out->op_index = m.op_index;
  out->op_tokens = m.op_tokens;
  return AKV_OK;
}

int akv_prefix_evict_order(akv_prefix_index* x, int64_t* entries, int32_t capacity, int32_t* n) {
  if (!x || !n || capacity < 0 || (capacity > 0 && !entries)) return AKV_EINVAL;
  const std::vector<int64_t> order = x->idx.evict_order();
  *n = (int32_t)order.size();
  if ((int32_t)order.size() > capacity) return pfail(x, AKV_ECAPACITY, "output array too small");
  std::copy(order.begin(), order.end(), entries);
  return AKV_OK;
}

}  // extern "C"
