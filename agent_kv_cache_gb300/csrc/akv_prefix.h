// History-keyed prefix index ("Cache Engineering for Agents" paper review,
// 4.2.2 Drop-aware Cache Management, 4.2.3 Reposition-aware Cache
// Management, Appendix A.1.2 Reposition Scheme; "[Repo Review] AKV", 5.4
// and 5.6).  Host only: a radix tree over context records of published
// snapshots, exact / retrigger matching of a request's records, and the
// drop-aware eviction order.
#pragma once

#include <cstdint>
#include <map>
#include <memory>
#include <string>
#include <unordered_map>
#include <vector>

#include "akv.h"

namespace akv {

// One context record: TOKEN(id), DELTA(interned merged ranges), REPOSITION.
struct PRec {
  int32_t kind;   // AKV_REC_*
  int32_t v;      // token id, or delta id
  bool operator==(const PRec& o) const { return kind == o.kind && v == o.v; }
  bool operator!=(const PRec& o) const { return !(*this == o); }
};
constexpr int32_t kRecT = 0, kRecD = 1, kRecR = 2;

// A request or entry program expanded into records, with the program
// coordinates of every record (for reporting a match as ops + tokens).
struct PProgram {
  std::vector<PRec> recs;
  std::vector<int32_t> rec_op;     // op index of each record
  std::vector<int32_t> rec_tok;    // for TOKEN records: index of the token within its op
  std::vector<int32_t> op_count;   // tokens appended by each op (0 for drop / repos)
  int32_t n_tokens = 0;
};

struct PEntry {
  int64_t id = -1;
  std::vector<PRec> recs;
  std::vector<int32_t> stored;     // per logical token: position of its stored key, -1 none
  std::vector<char> active;        // per logical token: active at the entry's end
  int64_t last_use = 0;
  int node = -1;                   // tree node the entry ends at
};

struct PNode {
  int parent = -1;
  int32_t depth = 0;               // records from the root through this node's label
  std::vector<PRec> label;         // edge label into this node
  std::map<uint64_t, int> kids;    // first record of the child's label -> child
  std::vector<int64_t> ends;       // entries ending here
  bool live = true;
};

struct PMatch {
  int32_t kind = AKV_MATCH_NONE;
  int64_t entry = -1;
  int32_t n_records = 0, n_tokens = 0, n_rotated = 0, op_index = 0, op_tokens = 0;
};

class PrefixIndex {
 public:
  explicit PrefixIndex(int32_t page_size);
  // Expands ops into records; interns DELTA contents.  Returns AKV_OK or an
  // error code with a message in *why.
  int expand(const akv_op* ops, int32_t n_ops, const int32_t* token_ids, int32_t n_tokens,
             PProgram* out, const char** why);
  int insert(int64_t id, const PProgram& p, int64_t use_time);
  int remove(int64_t id);
  bool has(int64_t id) const { return entries_.count(id) != 0; }
  const PEntry* entry(int64_t id) const;
  void touch(int64_t id, int64_t use_time);
  int64_t tick() { return ++clock_; }
  // first entry whose records equal p's, or -1
  int64_t find_equal(const PProgram& p) const;
  PMatch match(const PProgram& req) const;
  std::vector<int64_t> evict_order() const;
  int32_t page_size() const { return S_; }
  const std::vector<std::pair<int64_t, int64_t>>& delta(int32_t id) const { return deltas_[id]; }
  size_t size() const { return entries_.size(); }
  // state of a record prefix: per logical token active flag and position
  struct State {
    std::vector<char> active, held;
    std::vector<int32_t> pos;
    int32_t next_pos = 0;
  };
  State replay(const std::vector<PRec>& recs, size_t n) const;

 private:
  static uint64_t key(const PRec& r) { return ((uint64_t)(uint32_t)r.kind << 32) | (uint32_t)r.v; }
  void scan(const PEntry& e, const std::vector<PRec>& req, int32_t m, int32_t* best_exact,
            int32_t* best_valid, int32_t* valid_rot) const;
  int32_t S_;
  int64_t clock_ = 0;
  std::vector<PNode> nodes_;
  std::unordered_map<int64_t, PEntry> entries_;
  std::map<std::vector<std::pair<int64_t, int64_t>>, int32_t> delta_ids_;
  std::vector<std::vector<std::pair<int64_t, int64_t>>> deltas_;
};

}  // namespace akv

// The C ABI's opaque index handle.
struct akv_prefix_index {
  akv::PrefixIndex idx;
  std::string err;
};
