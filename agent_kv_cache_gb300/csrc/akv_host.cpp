// Host side of the active-KV cache library: the C ABI of include/akv.h.
//
// The host owns page allocation (free list + reference counts), the
// per-sequence bookkeeping (held slots, active slot intervals, the
// slot -> logical-index runs, history key) and the launch plans.  Each call
// (1) checks and plans without changing anything, (2) packs one descriptor
// blob and copies it to the device through a pinned staging ring, (3)
// commits the host state and (4) enqueues its kernels.  Nothing on the
// append / drop / reposition / decode path waits for the GPU.
//
// Sources: "Cache Engineering for Agents" paper review, 3.3 (Eqs. 3-5), 3.4
// (Eq. 6), 4.2.3 (position versions: a reposition by one request makes new
// K/V, other requests keep the old version); "[Repo Review] AKV", 5.4
// (OccurrenceState: reuse, borrow, or allocate-and-copy per occurrence;
// copy-on-write when ownership passes to another branch) and 5.6 (dropping
// is a visibility change; memory is reclaimed only when no one refers to it).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <queue>
#include <string>
#include <unordered_map>
#include <vector>

#include "akv.h"
#include "akv_internal.h"
#include "akv_prefix.h"

using namespace akv;

namespace {

struct Interval { int64_t a, b; };        // half-open
struct Run { int64_t slot0, log0, len; }; // slots [slot0, slot0+len) hold logical [log0, ...)

constexpr int kStages = 32;
constexpr int kMaxItems = 4096;            // decode work items (and partial slots) per call
constexpr int kMaxMembers = 16384;         // members of shared decode items per call
constexpr int kMinSharedPages = 4;         // shorter runs of common pages are read per row
constexpr int kShareRows = 128;            // query rows of a shared-prefix (tensor-core) item
constexpr int kShareMaxMembers = 128;
constexpr int kSharePagesMin = 32;         // pages per shared-prefix item (the kernel takes <= 256)
constexpr int kSharePagesMax = 256;
constexpr int kBlockStartPages = 6;       // a decode block's start-up, in pages of work

// 128-bit key of an operation history: two independent 64-bit chains, each
// step finished with the MurmurHash3 64-bit finaliser (Appleby).
inline uint64_t fmix64(uint64_t k) {
  k ^= k >> 33; k *= 0xff51afd7ed558ccdULL;
  k ^= k >> 33; k *= 0xc4ceb9fe1a85ec53ULL;
  k ^= k >> 33;
  return k;
}
struct HKey {
  uint64_t a = 0x6a09e667f3bcc908ULL, b = 0xbb67ae8584caa73bULL;
  void absorb(uint64_t w) {
    a = fmix64(a ^ (w + 0x9e3779b97f4a7c15ULL));
    b = fmix64(b + w * 0xc2b2ae3d27d4eb4fULL + 0x165667b19e3779f9ULL) ^ (a >> 7);
  }
};
constexpr uint64_t kRecAppend = 1, kRecDrop = 2, kRecRepos = 3;
constexpr uint64_t kNoToken = 1ULL << 40;

struct HostSeq {
  int32_t dslot = -1;
  int64_t n_logical = 0, n_slots = 0, n_alive = 0;
  int32_t n_active_pages = 0;
  std::vector<int32_t> pages;      // per slot page, -1 once released
  std::vector<Interval> alive;     // active slots, sorted, disjoint, merged
  std::vector<Run> runs;
  int64_t gather_n = 0;
  bool gather_identity = true;     // last reposition moved nothing
  HKey key;
  bool frozen = false;             // snapshot of a published prefix entry
  int64_t family = 0;              // pages are shared only within a family: a created
                                   // sequence starts one, forks inherit it
  // changes whenever a held page below the tail or a held slot changes
  // (drop, reposition, a new sequence); an append does not change it
  uint64_t layout = 0;
};

// A range of one row's active list that the decode reads for one or more
// rows of a call: `rows` are the members (rows[0] is the row whose active
// list [a0, a1) the kernel walks); member k holds the same pool pages at the
// same slot pages with the same keep bits over the first lens[k] pages of it,
// at its own active indices starts[k]...
struct Segment {
  int32_t a0, a1;
  std::vector<int32_t> rows, lens, starts;
  int32_t ns = 1;
};

// A staging block: pinned host memory (hd: its device view) and a device copy.
struct Stage {
  char* h = nullptr;
  char* hd = nullptr;
  char* d = nullptr;
  cudaEvent_t ev = nullptr;
  bool used = false;
};

struct Blob {
  std::vector<char> b;
  template <class T> size_t put(const T* p, size_t n) {
    const size_t off = (b.size() + 15) & ~size_t(15);
    b.resize(off + n * sizeof(T));
    if (n) std::memcpy(b.data() + off, p, n * sizeof(T));
    return off;
  }
};

// ---- interval sets --------------------------------------------------------

void iv_subtract(std::vector<Interval>& v, int64_t a, int64_t b, std::vector<Interval>* removed) {
  if (a >= b) return;
  std::vector<Interval> out;
  out.reserve(v.size() + 1);
  for (const Interval& iv : v) {
    if (iv.b <= a || iv.a >= b) { out.push_back(iv); continue; }
    if (iv.a < a) out.push_back({iv.a, a});
    if (removed) removed->push_back({std::max(iv.a, a), std::min(iv.b, b)});
    if (iv.b > b) out.push_back({b, iv.b});
  }
  v.swap(out);
}

bool iv_any(const std::vector<Interval>& v, int64_t a, int64_t b) {
  auto it = std::upper_bound(v.begin(), v.end(), a,
                             [](int64_t x, const Interval& iv) { return x < iv.b; });
  return it != v.end() && it->a < b;
}

int32_t iv_count_pages(const std::vector<Interval>& v, int S) {
  int64_t last = -1, count = 0;
  for (const Interval& iv : v) {
    int64_t k0 = iv.a / S;
    const int64_t k1 = (iv.b - 1) / S;
    if (k0 <= last) k0 = last + 1;
    if (k0 <= k1) count += k1 - k0 + 1;
    last = std::max(last, k1);
  }
  return (int32_t)count;
}

// Pages with index < k that hold an active slot.
int32_t iv_count_pages_below(const std::vector<Interval>& v, int S, int64_t k) {
  std::vector<Interval> clip;
  for (const Interval& iv : v) {
    if (iv.a >= k * S) break;
    clip.push_back({iv.a, std::min(iv.b, k * S)});
  }
  return iv_count_pages(clip, S);
}

void logical_to_slots(const std::vector<Run>& runs, int64_t lb, int64_t le,
                      std::vector<Interval>& out) {
  auto it = std::upper_bound(runs.begin(), runs.end(), lb,
                             [](int64_t x, const Run& r) { return x < r.log0 + r.len; });
  for (; it != runs.end() && it->log0 < le; ++it) {
    const int64_t a = std::max(lb, it->log0), b = std::min(le, it->log0 + it->len);
    if (a < b) out.push_back({it->slot0 + (a - it->log0), it->slot0 + (b - it->log0)});
  }
}

std::vector<Interval> merge(std::vector<Interval> v) {
  std::sort(v.begin(), v.end(), [](const Interval& x, const Interval& y) { return x.a < y.a; });
  std::vector<Interval> out;
  for (const Interval& iv : v) {
    if (iv.b <= iv.a) continue;
    if (!out.empty() && iv.a <= out.back().b) out.back().b = std::max(out.back().b, iv.b);
    else out.push_back(iv);
  }
  return out;
}

}  // namespace

struct akv_cache {
  akv_config cfg{};
  Geom g{};
  SeqArrays sa{};
  cudaStream_t stream = nullptr;
  float2* d_cs = nullptr;
  float2* d_cs_lo = nullptr;
  float* d_part_acc = nullptr;
  float2* d_part_ml = nullptr;
  uint32_t* d_err = nullptr;
  Stage stages[kStages];
  size_t stage_bytes = 0;
  int stage_next = 0;
  // decode plans (device copies kept while the metadata epoch is unchanged),
  // one per (sequence list, window) most recently used
  struct Plan {
    char* d = nullptr;
    uint64_t epoch = ~0ULL;
    std::vector<int64_t> seqs;
    int32_t window = -1;
    int items = 0;
    bool combine = false;
    bool shared = false;      // has items whose pages several rows read
    int shared_items = 0;
    int members = 0;
    int sitems = 0;           // tensor-core shared-prefix items
    size_t o_sitems = 0;
    int items_w = 0;          // the same call split for a whole wave (0: none)
    size_t o_items_w = 0;
    size_t o_members = 0;
    uint64_t used = 0;
  };
  static constexpr int kPlans = 4;
  Plan plans[kPlans];
  uint64_t plan_clock = 0;
  size_t plan_cap = 0;
  std::vector<int32_t> windows;     // per logical layer, 0 = full attention
  // host state
  std::vector<int32_t> refcnt, free_pages;
  std::unordered_map<int64_t, HostSeq> seqs;
  std::vector<int32_t> free_dslots;
  int64_t next_id = 1;
  uint64_t epoch = 0;
  std::string err;
  uint32_t wait_limit = 1u << 22;
  int sm_count = 148;
  uint64_t launches = 0;
  uint64_t decode_tail = ~0ULL;     // launches right after the last decode call
  CUtensorMap tm_k{}, tm_v{}, tm_k4{}, tm_v4{};
  bool use_mma = false;
  int mma_blocks_per_sm = 0;
  int32_t decode_waves = 1;
  int32_t decode_share = 1;        // rows holding the same pages read them once (0 off,
                                   // 1 automatic, else the most rows per item)
  int32_t last_items = 0, last_shared = 0, last_members = 0;   // plan of the last decode call
  std::vector<int32_t> share_head;  // decode planner scratch: first group of each pool page (-1)
  uint64_t layout_clock = 0;
  // the shared segments of the last call planned with them: valid while the
  // call has the same rows, each with the same layout version
  struct ShareCache {
    std::vector<int64_t> seqs;
    std::vector<uint64_t> layout;
    int cap = 0;
    bool full_only = false;
    std::vector<Segment> shared;
  } share_cache;
  int32_t* d_counters = nullptr;   // fused split merge: finished splits per (row, kv head)
  // device plan choice of the one-row decode kernel: per-call words
  uint32_t* d_mode = nullptr;          // [kDecodeModeWords]
  uint32_t* d_exits = nullptr;         // [kDecodeExitWords]
  uint32_t* d_done = nullptr;
  uint32_t decode_call = 0;            // id of the last one-row decode call
  void* d_restore = nullptr;       // temporary key/value versions of restore attention
  size_t restore_cap = 0;
  void* d_fork = nullptr;          // descriptor of a prefix fork
  size_t fork_cap = 0;
  bool restore_generic = false;    // CUDA-core restore kernel for every shape
  bool restore_pairs = true;       // tensor-core restore: two query tiles per CTA
};

namespace {

int fail(akv_cache* c, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (c) c->err = buf;
  return code;
}

#define CK(call)                                                               \
  do {                                                                         \
    cudaError_t e_ = (call);                                                   \
    if (e_ != cudaSuccess)                                                     \
      return fail(c, AKV_ECUDA, "%s: %s", #call, cudaGetErrorString(e_));      \
  } while (0)

int check_config(const akv_config* cfg) {
  if (!cfg) return AKV_EINVAL;
  const int S = cfg->page_size;
  const int G = cfg->hkv > 0 ? cfg->hq / cfg->hkv : 0;
  if (cfg->layers < 1 || cfg->phys_layers < 0 || cfg->phys_layers > cfg->layers) return AKV_EINVAL;
  if (cfg->hkv < 1 || cfg->hq < cfg->hkv || cfg->hq % cfg->hkv) return AKV_EINVAL;
  if (!(G == 1 || G == 2 || G == 4 || G == 8 || G == 16)) return AKV_EINVAL;
  if (cfg->head_dim != 64 && cfg->head_dim != 128) return AKV_EINVAL;
  if (!(S == 1 || S == 2 || S == 4 || S == 8 || S == 16 || S == 32 || S == 64)) return AKV_EINVAL;
  if (cfg->dtype != AKV_DTYPE_BF16 && cfg->dtype != AKV_DTYPE_FP32) return AKV_EINVAL;
  if (cfg->max_pages < 1 || cfg->max_seqs < 1) return AKV_EINVAL;
  if (cfg->max_slots < 1 || cfg->max_slots > (1 << 30)) return AKV_EINVAL;
  if (!(cfg->rope_theta > 1.0)) return AKV_EINVAL;
  if (cfg->rope_dim != 0 &&
      (cfg->rope_dim < 16 || cfg->rope_dim > cfg->head_dim || cfg->rope_dim % 16))
    return AKV_EINVAL;
  return AKV_OK;
}

HostSeq* find(akv_cache* c, int64_t id) {
  auto it = c->seqs.find(id);
  return it == c->seqs.end() ? nullptr : &it->second;
}

void decref(akv_cache* c, int32_t p) {
  if (p < 0) return;
  if (--c->refcnt[p] == 0) c->free_pages.push_back(p);
}

// The next n page ids the allocator will hand out (without taking them).
std::vector<int32_t> peek_pages(akv_cache* c, size_t n) {
  std::vector<int32_t> out(n);
  for (size_t i = 0; i < n; ++i) out[i] = c->free_pages[c->free_pages.size() - 1 - i];
  return out;
}
void take_pages(akv_cache* c, size_t n) {
  for (size_t i = 0; i < n; ++i) {
    const int32_t p = c->free_pages.back();
    c->free_pages.pop_back();
    c->refcnt[p] = 1;
  }
}

// Device-to-device bytes on the cache's stream, by a kernel (no copy-engine
// work on the caller's stream); n may be 0.
cudaError_t copy_rows(akv_cache* c, void* dst, const void* src, size_t n) {
  if (n == 0) return cudaSuccess;
  ++c->launches;
  return launch_copy_bytes(dst, src, n, c->stream);
}

int upload(akv_cache* c, const Blob& blob, char* dst, char** dptr) {
  if (blob.b.size() > c->stage_bytes)
    return fail(c, AKV_ECAPACITY, "descriptor of %zu bytes exceeds the staging block (%zu)",
                blob.b.size(), c->stage_bytes);
  Stage& s = c->stages[c->stage_next];
  c->stage_next = (c->stage_next + 1) % kStages;
  if (s.used) CK(cudaEventSynchronize(s.ev));
  if (!blob.b.empty()) {
    std::memcpy(s.h, blob.b.data(), blob.b.size());
    CK(launch_copy_bytes(dst ? dst : s.d, s.hd, blob.b.size(), c->stream));
    ++c->launches;
  }
  CK(cudaEventRecord(s.ev, c->stream));
  s.used = true;
  *dptr = dst ? dst : s.d;
  return AKV_OK;
}

// A descriptor of any size copied to device memory at dst through the
// staging ring, one staging block per copy.
int upload_large(akv_cache* c, const Blob& blob, char* dst) {
  for (size_t off = 0; off < blob.b.size(); off += c->stage_bytes) {
    const size_t m = std::min(c->stage_bytes, blob.b.size() - off);
    Stage& s = c->stages[c->stage_next];
    c->stage_next = (c->stage_next + 1) % kStages;
    if (s.used) CK(cudaEventSynchronize(s.ev));
    std::memcpy(s.h, blob.b.data() + off, m);
    CK(launch_copy_bytes(dst + off, s.hd, m, c->stream));
    ++c->launches;
    CK(cudaEventRecord(s.ev, c->stream));
    s.used = true;
  }
  return AKV_OK;
}

void destroy(akv_cache* c) {
  if (!c) return;
  cudaStreamSynchronize(c->stream);
  cudaFree(c->sa.keep);
  cudaFree(c->sa.pages);
  cudaFree(c->sa.active);
  cudaFree(c->sa.gather);
  cudaFree(c->sa.old_pages);
  cudaFree(c->d_cs);
  cudaFree(c->d_cs_lo);
  cudaFree(c->d_part_acc);
  cudaFree(c->d_part_ml);
  cudaFree(c->d_err);
  for (auto& pl : c->plans) cudaFree(pl.d);
  cudaFree(c->d_counters);
  cudaFree(c->d_mode);
  cudaFree(c->d_exits);
  cudaFree(c->d_done);
  cudaFree(c->d_restore);
  cudaFree(c->d_fork);
  for (Stage& s : c->stages) {
    if (s.h) cudaFreeHost(s.h);
    if (s.d) cudaFree(s.d);
    if (s.ev) cudaEventDestroy(s.ev);
  }
  delete c;
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================

extern "C" {

size_t akv_pool_bytes(const akv_config* cfg) {
  if (check_config(cfg) != AKV_OK) return 0;
  const int64_t phys = cfg->phys_layers ? cfg->phys_layers : cfg->layers;
  const int64_t elem = cfg->dtype == AKV_DTYPE_BF16 ? 2 : 4;
  return (size_t)(phys * cfg->max_pages * (int64_t)cfg->hkv * cfg->page_size * cfg->head_dim * elem);
}

int akv_cache_create(const akv_config* cfg, void* k_pool, void* v_pool, size_t pool_bytes,
                     void* stream, akv_cache** out) {
  if (!out) return AKV_EINVAL;
  *out = nullptr;
  if (check_config(cfg) != AKV_OK) return AKV_EINVAL;
  const size_t need = akv_pool_bytes(cfg);
  if (!k_pool || !v_pool || pool_bytes < need) return AKV_EINVAL;
  if ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) & 255) return AKV_EINVAL;

  akv_cache* c = new akv_cache();
  c->cfg = *cfg;
  if (!c->cfg.phys_layers) c->cfg.phys_layers = c->cfg.layers;
  c->stream = static_cast<cudaStream_t>(stream);
  const akv_config& f = c->cfg;
  Geom& g = c->g;
  g.k = k_pool;
  g.v = v_pool;
  g.layers = f.layers;
  g.phys_layers = f.phys_layers;
  g.hq = f.hq;
  g.hkv = f.hkv;
  g.d = f.head_dim;
  g.s = f.page_size;
  g.dtype = f.dtype;
  g.max_pages = f.max_pages;
  g.rope = f.rope_dim ? f.rope_dim : f.head_dim;
  c->cfg.rope_dim = g.rope;
  c->windows.assign(f.layers, 0);
  g.head_stride = (int64_t)f.page_size * f.head_dim;
  g.page_stride = g.head_stride * f.hkv;
  g.layer_stride = g.page_stride * f.max_pages;

  SeqArrays& sa = c->sa;
  sa.max_slots = f.max_slots;
  sa.keep_words = (f.max_slots + 31) / 32;
  sa.seq_pages = (f.max_slots + f.page_size - 1) / f.page_size;
  const size_t ns = (size_t)f.max_seqs;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, dev);
#define CKC(call)                                                              \
  do {                                                                         \
    cudaError_t e_ = (call);                                                   \
    if (e_ != cudaSuccess) { destroy(c); return AKV_ECUDA; }                   \
  } while (0)
  CKC(e);
  CKC(cudaMalloc(&sa.keep, ns * sa.keep_words * sizeof(uint32_t)));
  CKC(cudaMemset(sa.keep, 0, ns * sa.keep_words * sizeof(uint32_t)));
  CKC(cudaMalloc(&sa.pages, ns * sa.seq_pages * sizeof(int32_t)));
  CKC(cudaMemset(sa.pages, 0xff, ns * sa.seq_pages * sizeof(int32_t)));
  CKC(cudaMalloc(&sa.active, ns * sa.seq_pages * sizeof(int32_t)));
  CKC(cudaMalloc(&sa.old_pages, ns * sa.seq_pages * sizeof(int32_t)));
  CKC(cudaMalloc(&sa.gather, ns * (size_t)sa.max_slots * sizeof(int32_t)));

  // RoPE table cos/sin(m f_i), m < max_slots, f_i = theta^(-2i/R): fp64,
  // rounded once to fp32; and the low parts left by that rounding (fp32),
  // which the stored-key kernels add back for rotations that nearly cancel.
  {
    const int H = g.rope / 2;
    std::vector<float2> cs((size_t)f.max_slots * H), lo((size_t)f.max_slots * H);
    std::vector<double> fr(H);
    for (int i = 0; i < H; ++i) fr[i] = std::pow(f.rope_theta, -2.0 * i / g.rope);
    for (int64_t m = 0; m < f.max_slots; ++m)
      for (int i = 0; i < H; ++i) {
        const double ang = (double)m * fr[i];
        const double co = std::cos(ang), si = std::sin(ang);
        const float ch = (float)co, sh = (float)si;
        cs[m * H + i] = make_float2(ch, sh);
        lo[m * H + i] = make_float2((float)(co - (double)ch), (float)(si - (double)sh));
      }
    CKC(cudaMalloc(&c->d_cs, cs.size() * sizeof(float2)));
    CKC(cudaMemcpy(c->d_cs, cs.data(), cs.size() * sizeof(float2), cudaMemcpyHostToDevice));
    CKC(cudaMalloc(&c->d_cs_lo, lo.size() * sizeof(float2)));
    CKC(cudaMemcpy(c->d_cs_lo, lo.data(), lo.size() * sizeof(float2), cudaMemcpyHostToDevice));
    g.cs_lo = c->d_cs_lo;
  }
  CKC(cudaMalloc(&c->d_part_acc, (size_t)kMaxItems * f.hq * f.head_dim * sizeof(float)));
  CKC(cudaMalloc(&c->d_part_ml, (size_t)kMaxItems * f.hq * sizeof(float2)));
  CKC(cudaMalloc(&c->d_err, sizeof(uint32_t)));
  CKC(cudaMemset(c->d_err, 0, sizeof(uint32_t)));
  c->plan_cap = 2 * kMaxItems * sizeof(DecodeItem) + 2 * ns * sizeof(int32_t) +
                kMaxMembers * sizeof(DecodeMember) + kMaxItems * sizeof(ShareItem) + 96;
  for (auto& pl : c->plans) CKC(cudaMalloc(&pl.d, c->plan_cap));
  c->stage_bytes = std::max<size_t>(1 << 20, 8 * (size_t)f.max_pages + 96 * ns +
                                                 kMaxItems * sizeof(DecodeItem) + 65536);
  c->stage_bytes = (c->stage_bytes + 4095) & ~size_t(4095);
  for (Stage& s : c->stages) {
    CKC(cudaMallocHost(&s.h, c->stage_bytes));
    CKC(cudaHostGetDevicePointer(reinterpret_cast<void**>(&s.hd), s.h, 0));
    CKC(cudaMalloc(&s.d, c->stage_bytes));
    CKC(cudaEventCreateWithFlags(&s.ev, cudaEventDisableTiming));
  }
  CKC(cudaMalloc(&c->d_counters, (size_t)kMaxItems * f.hkv * sizeof(int32_t)));
  CKC(cudaMemset(c->d_counters, 0, (size_t)kMaxItems * f.hkv * sizeof(int32_t)));
  CKC(cudaMalloc(&c->d_mode, kDecodeModeWords * sizeof(uint32_t)));
  CKC(cudaMemset(c->d_mode, 0, kDecodeModeWords * sizeof(uint32_t)));
  CKC(cudaMalloc(&c->d_exits, kDecodeExitWords * sizeof(uint32_t)));
  CKC(cudaMemset(c->d_exits, 0, kDecodeExitWords * sizeof(uint32_t)));
  CKC(cudaMalloc(&c->d_done, sizeof(uint32_t)));
  CKC(cudaMemset(c->d_done, 0, sizeof(uint32_t)));
  c->use_mma = make_pool_tensor_maps(g, &c->tm_k, &c->tm_v) &&
               make_pool_tensor_maps4(g, &c->tm_k4, &c->tm_v4);
  if (c->use_mma) {
    c->mma_blocks_per_sm = decode_mma_blocks_per_sm(f.head_dim);
    if (c->mma_blocks_per_sm < 1) c->use_mma = false;
  }
  CKC(cudaDeviceSynchronize());
#undef CKC

  c->refcnt.assign(f.max_pages, 0);
  c->free_pages.resize(f.max_pages);
  for (int32_t i = 0; i < f.max_pages; ++i) c->free_pages[i] = f.max_pages - 1 - i;
  c->free_dslots.resize(f.max_seqs);
  for (int32_t i = 0; i < f.max_seqs; ++i) c->free_dslots[i] = f.max_seqs - 1 - i;
  *out = c;
  return AKV_OK;
}

int akv_cache_destroy(akv_cache* c) {
  if (!c) return AKV_EINVAL;
  destroy(c);
  return AKV_OK;
}

int akv_set_stream(akv_cache* c, void* stream) {
  if (!c) return AKV_EINVAL;
  c->stream = static_cast<cudaStream_t>(stream);
  return AKV_OK;
}

int akv_seq_create(akv_cache* c, int64_t* seq) {
  if (!c || !seq) return AKV_EINVAL;
  if (c->free_dslots.empty()) return fail(c, AKV_ECAPACITY, "max_seqs (%d) sequences alive", c->cfg.max_seqs);
  HostSeq s;
  s.dslot = c->free_dslots.back();
  c->free_dslots.pop_back();
  const int64_t id = c->next_id++;
  s.family = id;
  s.layout = ++c->layout_clock;
  c->seqs.emplace(id, std::move(s));
  ++c->epoch;
  *seq = id;
  return AKV_OK;
}

int akv_seq_fork(akv_cache* c, int64_t parent, int64_t* child) {
  if (!c || !child) return AKV_EINVAL;
  HostSeq* p = find(c, parent);
  if (!p) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)parent);
  if (c->free_dslots.empty()) return fail(c, AKV_ECAPACITY, "max_seqs (%d) sequences alive", c->cfg.max_seqs);
  HostSeq s = *p;
  s.frozen = false;
  s.dslot = c->free_dslots.back();
  const SeqArrays& sa = c->sa;
  const int64_t ps = p->dslot, cs = s.dslot;
  const size_t nw = (size_t)((p->n_slots + 31) / 32);
  const size_t np = p->pages.size();
  CK(copy_rows(c, sa.keep + cs * sa.keep_words, sa.keep + ps * sa.keep_words,
               nw * sizeof(uint32_t)));
  CK(copy_rows(c, sa.pages + cs * sa.seq_pages, sa.pages + ps * sa.seq_pages,
               np * sizeof(int32_t)));
  CK(copy_rows(c, sa.active + cs * sa.seq_pages, sa.active + ps * sa.seq_pages,
               (size_t)p->n_active_pages * sizeof(int32_t)));
  if (!p->gather_identity && p->gather_n)
    CK(copy_rows(c, sa.gather + cs * sa.max_slots, sa.gather + ps * sa.max_slots,
                 (size_t)p->gather_n * sizeof(int32_t)));
  c->free_dslots.pop_back();
  for (int32_t pg : s.pages)
    if (pg >= 0) ++c->refcnt[pg];
  const int64_t id = c->next_id++;
  s.layout = ++c->layout_clock;
  c->seqs.emplace(id, std::move(s));
  ++c->epoch;
  *child = id;
  return AKV_OK;
}

int akv_seq_free(akv_cache* c, int64_t seq) {
  if (!c) return AKV_EINVAL;
  HostSeq* s = find(c, seq);
  if (!s) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seq);
  // a free device row keeps all keep bits clear (append only sets bits)
  CK(launch_fill_u32(c->sa.keep + (int64_t)s->dslot * c->sa.keep_words, 0,
                     (size_t)c->sa.keep_words, c->stream));
  ++c->launches;
  for (int32_t pg : s->pages) decref(c, pg);
  c->free_dslots.push_back(s->dslot);
  c->seqs.erase(seq);
  ++c->epoch;
  return AKV_OK;
}

// ---- Eq. (3) ---------------------------------------------------------------

int akv_append(akv_cache* c, const int64_t* seqs, const int32_t* n_tokens, int32_t n_seqs,
               const void* k_raw, const void* v, const int32_t* token_ids) {
  if (!c || n_seqs < 0 || (n_seqs > 0 && (!seqs || !n_tokens))) return AKV_EINVAL;
  const int S = c->cfg.page_size;
  std::vector<HostSeq*> hs(n_seqs);
  int64_t total = 0;
  size_t need_pages = 0;
  for (int i = 0; i < n_seqs; ++i) {
    hs[i] = find(c, seqs[i]);
    if (!hs[i]) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seqs[i]);
    if (hs[i]->frozen) return fail(c, AKV_EINVAL, "sequence %lld is a published snapshot", (long long)seqs[i]);
    for (int j = 0; j < i; ++j)
      if (hs[j] == hs[i]) return fail(c, AKV_EINVAL, "sequence %lld repeated", (long long)seqs[i]);
    const int64_t n = n_tokens[i];
    if (n < 0) return fail(c, AKV_EINVAL, "negative token count");
    if (hs[i]->n_slots + n > c->cfg.max_slots)
      return fail(c, AKV_ECAPACITY, "sequence %lld would hold %lld > max_slots %d tokens",
                  (long long)seqs[i], (long long)(hs[i]->n_slots + n), c->cfg.max_slots);
    if (n == 0) continue;
    const int64_t old = hs[i]->n_slots;
    need_pages += (size_t)((old + n + S - 1) / S - (old + S - 1) / S);
    if (old % S && c->refcnt[hs[i]->pages[old / S]] > 1) ++need_pages;   // copy-on-write
    total += n;
  }
  if (total == 0) return AKV_OK;
  if (!k_raw || !v) return AKV_EINVAL;
  if (total > INT32_MAX) return fail(c, AKV_ECAPACITY, "too many tokens in one call");
  if (need_pages > c->free_pages.size())
    return fail(c, AKV_ENOPAGES, "append needs %zu pages, %zu free", need_pages, c->free_pages.size());

  // plan
  std::vector<int32_t> fresh = peek_pages(c, need_pages);
  size_t fi = 0;
  std::vector<AppendItem> items;
  std::vector<AppendBlock> blocks;
  std::vector<int32_t> ids, act;
  std::vector<PagePair> cow;
  struct Commit { HostSeq* s; int64_t n; std::vector<std::pair<int64_t, int32_t>> set; int32_t n_act_new; };
  std::vector<Commit> commits;
  int64_t tok = 0;
  for (int i = 0; i < n_seqs; ++i) {
    const int64_t n = n_tokens[i];
    if (n == 0) continue;
    HostSeq* s = hs[i];
    const int64_t old = s->n_slots;
    AppendItem it{};
    it.dslot = s->dslot;
    it.slot0 = (int32_t)old;
    it.n = (int32_t)n;
    it.tok0 = (int32_t)tok;
    it.k0 = (int32_t)(old / S);
    const int64_t k1 = (old + n - 1) / S;
    it.nk = (int32_t)(k1 - it.k0 + 1);
    it.ids_off = (int32_t)ids.size();
    it.act0 = s->n_active_pages;
    it.act_off = (int32_t)act.size();
    Commit cm{s, n, {}, 0};
    for (int64_t k = it.k0; k <= k1; ++k) {
      int32_t pid;
      if (k < (int64_t)s->pages.size()) {          // partly filled tail page
        pid = s->pages[k];
        if (c->refcnt[pid] > 1) {
          const int32_t np = fresh[fi++];
          cow.push_back({pid, np});
          cm.set.push_back({k, np});
          pid = np;
        }
        if (!iv_any(s->alive, k * S, (k + 1) * S)) act.push_back((int32_t)k);
      } else {
        pid = fresh[fi++];
        cm.set.push_back({k, pid});
        act.push_back((int32_t)k);
      }
      ids.push_back(pid);
    }
    it.n_act = (int32_t)(act.size() - it.act_off);
    cm.n_act_new = it.n_act;
    for (int64_t t0 = 0; t0 < n; t0 += kAppendTokens) blocks.push_back({(int32_t)items.size(), (int32_t)t0});
    items.push_back(it);
    commits.push_back(std::move(cm));
    tok += n;
  }
  Blob blob;
  const size_t o_items = blob.put(items.data(), items.size());
  const size_t o_blocks = blob.put(blocks.data(), blocks.size());
  const size_t o_ids = blob.put(ids.data(), ids.size());
  const size_t o_act = blob.put(act.data(), act.size());
  const size_t o_cow = blob.put(cow.data(), cow.size());
  char* d = nullptr;
  int rc = upload(c, blob, nullptr, &d);
  if (rc) return rc;

  // commit
  take_pages(c, need_pages);
  size_t ti = 0;
  for (Commit& cm : commits) {
    HostSeq* s = cm.s;
    const int64_t old = s->n_slots;
    for (auto& kp : cm.set) {
      if (kp.first < (int64_t)s->pages.size()) {
        decref(c, s->pages[kp.first]);
        s->pages[kp.first] = kp.second;
      } else {
        s->pages.push_back(kp.second);
      }
    }
    if (!s->alive.empty() && s->alive.back().b == old) s->alive.back().b = old + cm.n;
    else s->alive.push_back({old, old + cm.n});
    if (!s->runs.empty() && s->runs.back().slot0 + s->runs.back().len == old &&
        s->runs.back().log0 + s->runs.back().len == s->n_logical)
      s->runs.back().len += cm.n;
    else
      s->runs.push_back({old, s->n_logical, cm.n});
    for (int64_t t = 0; t < cm.n; ++t) {
      s->key.absorb(kRecAppend);
      s->key.absorb(token_ids ? (uint64_t)(uint32_t)token_ids[ti + t] : kNoToken);
    }
    ti += cm.n;
    s->n_slots += cm.n;
    s->n_logical += cm.n;
    s->n_alive += cm.n;
    s->n_active_pages += cm.n_act_new;
  }
  ++c->epoch;

  if (!cow.empty()) {
    CK(launch_copy_pages(c->g, reinterpret_cast<const PagePair*>(d + o_cow), (int)cow.size(),
                         c->d_err, c->stream));
    ++c->launches;
  }
  ++c->launches;
  CK(launch_append(c->g, c->sa, reinterpret_cast<const AppendItem*>(d + o_items),
                   reinterpret_cast<const AppendBlock*>(d + o_blocks), (int)blocks.size(),
                   reinterpret_cast<const int32_t*>(d + o_ids),
                   reinterpret_cast<const int32_t*>(d + o_act), k_raw, v, total, c->d_cs,
                   c->d_err,
                   AppendLimits{(int32_t)items.size(), (int32_t)ids.size(), (int32_t)act.size(),
                                c->cfg.max_seqs},
                   c->stream));
  return AKV_OK;
}

// ---- Eq. (4) ---------------------------------------------------------------

int akv_drop(akv_cache* c, int64_t seq, const int64_t* ranges, int32_t n_ranges) {
  if (!c || n_ranges < 0 || (n_ranges > 0 && !ranges)) return AKV_EINVAL;
  HostSeq* s = find(c, seq);
  if (!s) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seq);
  if (s->frozen) return fail(c, AKV_EINVAL, "sequence %lld is a published snapshot", (long long)seq);
  std::vector<Interval> logical;
  for (int i = 0; i < n_ranges; ++i) {
    const int64_t b = ranges[2 * i], e = ranges[2 * i + 1];
    if (b < 0 || e < b || e > s->n_logical)
      return fail(c, AKV_ERANGE, "range [%lld, %lld) outside [0, %lld)", (long long)b,
                  (long long)e, (long long)s->n_logical);
    logical.push_back({b, e});
  }
  logical = merge(logical);
  if (logical.empty()) return AKV_OK;     // dropping the empty set is no operation

  const int S = c->cfg.page_size;
  std::vector<Interval> slots;
  for (const Interval& iv : logical) logical_to_slots(s->runs, iv.a, iv.b, slots);
  slots = merge(slots);
  std::vector<Interval> alive = s->alive, removed;
  for (const Interval& iv : slots) iv_subtract(alive, iv.a, iv.b, &removed);
  int64_t n_removed = 0;
  std::vector<int64_t> dead_pages;
  for (const Interval& iv : removed) {
    n_removed += iv.b - iv.a;
    for (int64_t k = iv.a / S; k <= (iv.b - 1) / S; ++k) {
      if ((k + 1) * S > s->n_slots || s->pages[k] < 0) continue;
      if (!dead_pages.empty() && dead_pages.back() == k) continue;
      if (!iv_any(alive, k * S, (k + 1) * S)) dead_pages.push_back(k);
    }
  }
  const int32_t n_active = iv_count_pages(alive, S);

  std::vector<int32_t> r32;
  for (const Interval& iv : slots) { r32.push_back((int32_t)iv.a); r32.push_back((int32_t)iv.b); }
  DropItem it{};
  it.dslot = s->dslot;
  it.n_slots = (int32_t)s->n_slots;
  it.n_pages = (int32_t)s->pages.size();
  it.range_off = 0;
  it.n_ranges = (int32_t)slots.size();
  it.expect_active = n_active;
  Blob blob;
  const size_t o_item = blob.put(&it, 1);
  const size_t o_r = blob.put(r32.data(), r32.size());
  char* d = nullptr;
  int rc = upload(c, blob, nullptr, &d);
  if (rc) return rc;

  // commit
  s->alive.swap(alive);
  s->layout = ++c->layout_clock;
  s->n_alive -= n_removed;
  s->n_active_pages = n_active;
  for (int64_t k : dead_pages) { decref(c, s->pages[k]); s->pages[k] = -1; }
  s->key.absorb(kRecDrop);
  s->key.absorb(logical.size());
  for (const Interval& iv : logical) { s->key.absorb((uint64_t)iv.a); s->key.absorb((uint64_t)iv.b); }
  ++c->epoch;
  CK(launch_drop(c->g, c->sa, reinterpret_cast<const DropItem*>(d + o_item), 1,
                 reinterpret_cast<const int32_t*>(d + o_r), c->d_err, c->stream));
  ++c->launches;
  return AKV_OK;
}

// ---- Eq. (5) ---------------------------------------------------------------

int akv_reposition(akv_cache* c, const int64_t* seqs, int32_t n_seqs) {
  if (!c || n_seqs < 0 || (n_seqs > 0 && !seqs)) return AKV_EINVAL;
  const int S = c->cfg.page_size;
  std::vector<HostSeq*> hs(n_seqs);
  size_t need = 0;
  std::vector<ReposItem> items;
  std::vector<int32_t> ids;
  std::vector<char> dense(n_seqs, 0);
  for (int i = 0; i < n_seqs; ++i) {
    hs[i] = find(c, seqs[i]);
    if (!hs[i]) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seqs[i]);
    if (hs[i]->frozen) return fail(c, AKV_EINVAL, "sequence %lld is a published snapshot", (long long)seqs[i]);
    for (int j = 0; j < i; ++j)
      if (hs[j] == hs[i]) return fail(c, AKV_EINVAL, "sequence %lld repeated", (long long)seqs[i]);
    const HostSeq* s = hs[i];
    const bool is_dense = s->alive.empty() ? s->n_slots == 0
                                           : (s->alive.size() == 1 && s->alive[0].a == 0 &&
                                              s->alive[0].b == s->n_slots);
    dense[i] = is_dense;
    if (is_dense) continue;
    const int64_t r = s->n_alive;
    const int64_t u = (!s->alive.empty() && s->alive[0].a == 0) ? s->alive[0].b : 0;
    const int64_t n_kept = u / S;
    const int64_t new_pages = (r + S - 1) / S;
    need += (size_t)(new_pages - n_kept);
  }
  if (need > c->free_pages.size())
    return fail(c, AKV_ENOPAGES, "reposition needs %zu pages, %zu free", need, c->free_pages.size());
  std::vector<int32_t> fresh = peek_pages(c, need);
  size_t fi = 0;
  int32_t blocks = 0;
  for (int i = 0; i < n_seqs; ++i) {
    if (dense[i]) continue;
    const HostSeq* s = hs[i];
    const int64_t r = s->n_alive;
    const int64_t u = (!s->alive.empty() && s->alive[0].a == 0) ? s->alive[0].b : 0;
    ReposItem it{};
    it.dslot = s->dslot;
    it.old_slots = (int32_t)s->n_slots;
    it.old_pages = (int32_t)s->pages.size();
    it.r = (int32_t)r;
    it.n_kept = (int32_t)(u / S);
    it.new_pages = (int32_t)((r + S - 1) / S);
    it.fresh_off = (int32_t)ids.size();
    it.block0 = blocks;
    for (int32_t k = it.n_kept; k < it.new_pages; ++k) ids.push_back(fresh[fi++]);
    blocks += it.new_pages - it.n_kept;
    items.push_back(it);
  }
  char* d = nullptr;
  size_t o_items = 0, o_ids = 0;
  if (!items.empty()) {
    Blob blob;
    o_items = blob.put(items.data(), items.size());
    o_ids = blob.put(ids.data(), ids.size());
    int rc = upload(c, blob, nullptr, &d);
    if (rc) return rc;
  }

  // commit
  take_pages(c, need);
  size_t ii = 0;
  for (int i = 0; i < n_seqs; ++i) {
    HostSeq* s = hs[i];
    s->key.absorb(kRecRepos);
    if (dense[i]) {
      s->gather_identity = true;
      s->gather_n = s->n_slots;
      continue;
    }
    const ReposItem& it = items[ii++];
    // slot -> logical runs of the survivors, now dense
    std::vector<Run> nr;
    size_t ri = 0;
    int64_t j = 0;
    for (const Interval& iv : s->alive) {
      while (ri < s->runs.size() && s->runs[ri].slot0 + s->runs[ri].len <= iv.a) ++ri;
      for (size_t rk = ri; rk < s->runs.size() && s->runs[rk].slot0 < iv.b; ++rk) {
        const Run& r0 = s->runs[rk];
        const int64_t a = std::max(iv.a, r0.slot0), b = std::min(iv.b, r0.slot0 + r0.len);
        if (a >= b) continue;
        const int64_t lg = r0.log0 + (a - r0.slot0);
        if (!nr.empty() && nr.back().log0 + nr.back().len == lg) nr.back().len += b - a;
        else nr.push_back({j, lg, b - a});
        j += b - a;
      }
    }
    for (int64_t k = it.n_kept; k < (int64_t)s->pages.size(); ++k) decref(c, s->pages[k]);
    s->pages.resize(it.n_kept);
    for (int32_t k = 0; k < it.new_pages - it.n_kept; ++k) s->pages.push_back(ids[it.fresh_off + k]);
    s->runs.swap(nr);
    s->alive.clear();
    if (it.r > 0) s->alive.push_back({0, it.r});
    s->layout = ++c->layout_clock;
    s->n_slots = it.r;
    s->n_alive = it.r;
    s->n_active_pages = it.new_pages;
    s->gather_identity = false;
    s->gather_n = it.r;
  }
  ++c->epoch;
  if (!items.empty()) {
    CK(launch_compact(c->g, c->sa, reinterpret_cast<const ReposItem*>(d + o_items),
                      (int)items.size(), reinterpret_cast<const int32_t*>(d + o_ids), c->d_err,
                      c->stream));
    CK(launch_gather(c->g, c->sa, reinterpret_cast<const ReposItem*>(d + o_items),
                     (int)items.size(), blocks, c->d_cs, c->d_err, c->wait_limit, c->stream));
    c->launches += blocks > 0 ? 2 : 1;
  }
  return AKV_OK;
}

// ---- decode ------------------------------------------------------------------

namespace {

struct ActivePage { int32_t kidx, page; uint64_t mask; };

// A sequence's active slot pages in ascending order (the device's active
// list), each with its pool page and the keep bits of its slots.
void active_pages(const HostSeq& sq, int S, std::vector<ActivePage>* out) {
  out->clear();
  for (const Interval& iv : sq.alive)
    for (int64_t k = iv.a / S; k * S < iv.b; ++k) {
      const int64_t lo = std::max(iv.a, k * S) - k * S, hi = std::min(iv.b, (k + 1) * S) - k * S;
      const uint64_t bits = (hi - lo >= 64 ? ~0ULL : ((1ULL << (hi - lo)) - 1)) << lo;
      if (!out->empty() && out->back().kidx == k) out->back().mask |= bits;
      else out->push_back({(int32_t)k, sq.pages[k], bits});
    }
}

// Shared segments: walking the rows in order, an active page that other rows
// hold identically (same pool page, slot page and keep bits) and that none
// of them has read yet starts a segment.  Each such row joins for as long as
// its next active pages stay identical (at consecutive places of both
// lists); rows that stay fewer than kMinSharedPages pages read privately.
// The members are then taken longest first in chunks of at most `cap`, each
// chunk a segment walked along its longest member's list.  Every page not
// covered this way is read per row.  full_only: share only pages whose every
// slot has been written (below the row's held slots), so that no unwritten
// pool memory is read for another row.
void find_shared(akv_cache* c, const std::vector<const HostSeq*>& hs, int cap, bool full_only,
                 std::vector<Segment>* segs) {
  const int n = (int)hs.size(), S = c->cfg.page_size;
  std::vector<std::vector<ActivePage>> ap(n);
  std::vector<std::vector<int32_t>> gid(n);        // entry -> group of >= 2 rows, or -1
  std::vector<std::vector<char>> covered(n);
  // groups of identical entries: a reused page-indexed head, chained when a
  // page appears under another slot page or other keep bits; members laid
  // out flat by group (rows ascending)
  struct Group { int32_t kidx; uint64_t mask; int32_t next, count, start; };
  std::vector<Group> gk;
  std::vector<int32_t> touched;
  if ((int)c->share_head.size() < c->cfg.max_pages) c->share_head.assign(c->cfg.max_pages, -1);
  std::vector<int32_t>& head = c->share_head;
  for (int i = 0; i < n; ++i) {
    active_pages(*hs[i], S, &ap[i]);
    gid[i].assign(ap[i].size(), -1);
    covered[i].assign(ap[i].size(), 0);
    if ((int64_t)ap[i].size() != hs[i]->n_active_pages) continue;   // never share then
    for (int32_t a = 0; a < (int32_t)ap[i].size(); ++a) {
      const ActivePage& e = ap[i][a];
      if (e.page < 0 || e.page >= c->cfg.max_pages || c->refcnt[e.page] < 2) continue;
      if (full_only && (int64_t)(e.kidx + 1) * S > hs[i]->n_slots) continue;
      int32_t g = head[e.page];
      while (g >= 0 && !(gk[g].kidx == e.kidx && gk[g].mask == e.mask)) g = gk[g].next;
      if (g < 0) {
        g = (int32_t)gk.size();
        if (head[e.page] < 0) touched.push_back(e.page);
        gk.push_back({e.kidx, e.mask, head[e.page], 0, 0});
        head[e.page] = g;
      }
      gid[i][a] = g;
      ++gk[g].count;
    }
  }
  for (int32_t p : touched) head[p] = -1;
  bool any = false;
  int32_t total = 0;
  for (Group& gr : gk) {
    gr.start = total;
    total += gr.count;
    any |= gr.count > 1;
    gr.count = 0;
  }
  std::vector<std::pair<int32_t, int32_t>> flat(total);   // (row, active index) by group
  for (int i = 0; i < n; ++i)
    for (int32_t a = 0; a < (int32_t)gid[i].size(); ++a)
      if (gid[i][a] >= 0) {
        Group& gr = gk[gid[i][a]];
        flat[gr.start + gr.count++] = {i, a};
      }
  // the members of group g: flat[gk[g].start .. + gk[g].count)
  if (any) {
    struct Cand { int32_t row, start, len; };
    std::vector<Cand> cand;
    for (int i = 0; i < n; ++i)
      for (int32_t a = 0; a < (int32_t)ap[i].size();) {
        const int32_t g0 = gid[i][a];
        if (g0 < 0 || covered[i][a] || gk[g0].count < 2) { ++a; continue; }
        // how long each other row that holds this page stays identical
        cand.clear();
        int32_t longest = 0;
        for (int32_t f = gk[g0].start; f < gk[g0].start + gk[g0].count; ++f) {
          const auto& m = flat[f];
          if (m.first == i || covered[m.first][m.second]) continue;
          const int j = m.first;
          int32_t len = 0;
          while (a + len < (int32_t)ap[i].size() && m.second + len < (int32_t)ap[j].size() &&
                 gid[i][a + len] >= 0 && gid[i][a + len] == gid[j][m.second + len] &&
                 !covered[i][a + len] && !covered[j][m.second + len])
            ++len;
          if (len >= kMinSharedPages) {
            cand.push_back({j, m.second, len});
            longest = std::max(longest, len);
          }
        }
        if (cand.empty()) { ++a; continue; }
        cand.push_back({i, a, longest});
        std::stable_sort(cand.begin(), cand.end(),
                         [](const Cand& x, const Cand& y) { return x.len > y.len; });
        const int nm = (int)cand.size(), nch = (nm + cap - 1) / cap;
        for (int ch = 0, k0 = 0; ch < nch; ++ch) {
          const int k1 = k0 + (nm - k0 + (nch - ch) - 1) / (nch - ch);
          Segment sg;
          sg.a0 = cand[k0].start;
          sg.a1 = sg.a0 + cand[k0].len;
          for (int k = k0; k < k1; ++k) {
            sg.rows.push_back(cand[k].row);
            sg.lens.push_back(cand[k].len);
            sg.starts.push_back(cand[k].start);
            for (int32_t t = 0; t < cand[k].len; ++t) covered[cand[k].row][cand[k].start + t] = 1;
          }
          segs->push_back(std::move(sg));
          k0 = k1;
        }
        a += longest;
      }
  }
}

// Every active page of a row not covered by the shared segments, as per-row
// segments (maximal uncovered ranges; a row with no active page still gets
// one empty segment for its output).
void complete_segments(const std::vector<const HostSeq*>& hs, const std::vector<Segment>& shared,
                       std::vector<Segment>* segs) {
  const int n = (int)hs.size();
  std::vector<std::vector<std::pair<int32_t, int32_t>>> cov(n);   // covered [start, end) per row
  for (const Segment& sg : shared)
    for (size_t k = 0; k < sg.rows.size(); ++k)
      cov[sg.rows[k]].push_back({sg.starts[k], sg.starts[k] + sg.lens[k]});
  for (int i = 0; i < n; ++i) {
    std::sort(cov[i].begin(), cov[i].end());
    const int32_t na = hs[i]->n_active_pages;
    bool any_seg = !cov[i].empty();
    int32_t a = 0;
    auto gap = [&](int32_t b) {
      if (b > a) {
        Segment sg;
        sg.a0 = a;
        sg.a1 = b;
        sg.rows = {i};
        sg.lens = {b - a};
        sg.starts = {a};
        segs->push_back(std::move(sg));
        any_seg = true;
      }
    };
    for (const auto& iv : cov[i]) {
      gap(std::min(iv.first, na));
      a = std::max(a, iv.second);
    }
    gap(na);
    if (!any_seg) {
      Segment sg;
      sg.a0 = sg.a1 = 0;
      sg.rows = {i};
      sg.lens = {0};
      sg.starts = {0};
      segs->push_back(std::move(sg));
    }
  }
}

}  // namespace

int akv_decode_attention(akv_cache* c, int32_t layer, const void* q, const int64_t* seqs,
                         int32_t n_seqs, float* out) {
  if (!c || n_seqs < 0 || (n_seqs > 0 && (!seqs || !q || !out))) return AKV_EINVAL;
  if (layer < 0 || layer >= c->cfg.layers) return fail(c, AKV_EINVAL, "layer %d out of range", layer);
  if (n_seqs == 0) return AKV_OK;
  const int32_t window = c->windows[layer];
  akv_cache::Plan* plan = nullptr;
  for (auto& pl : c->plans)
    if (pl.epoch == c->epoch && pl.window == window && (int)pl.seqs.size() == n_seqs &&
        std::equal(pl.seqs.begin(), pl.seqs.end(), seqs))
      plan = &pl;
  if (!plan) {
    std::vector<const HostSeq*> hs(n_seqs);
    std::vector<int32_t> first(n_seqs, 0), win_lo(n_seqs, 0);
    int64_t total = 0;
    for (int i = 0; i < n_seqs; ++i) {
      hs[i] = find(c, seqs[i]);
      if (!hs[i]) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seqs[i]);
      if (window > 0) {
        // the query at position p reads positions (p - window, p]: slots are
        // positions, so the read range starts at the page of slot p - window + 1
        const int64_t lo = std::max<int64_t>(0, hs[i]->n_slots - window);
        win_lo[i] = (int32_t)lo;
        first[i] = iv_count_pages_below(hs[i]->alive, c->cfg.page_size, lo / c->cfg.page_size);
      }
      total += hs[i]->n_active_pages - first[i];
    }
    std::vector<DecodeItem> items, items_w;
    std::vector<DecodeMember> members;
    std::vector<ShareItem> sitems;
    std::vector<int32_t> item0(n_seqs), splits(n_seqs);
    bool combine = false, shared = false;
    auto emit = [&](int i, int32_t ns, bool even) {
      const HostSeq* sq = hs[i];
      const int64_t f0 = first[i], na = sq->n_active_pages - f0;
      item0[i] = (int32_t)items.size();
      splits[i] = ns;
      combine |= ns > 1;
      for (int32_t k = 0; k < ns; ++k) {
        DecodeItem it{};
        it.dslot = sq->dslot;
        it.row = i;
        it.p0 = (int32_t)(f0 + (even ? na * k / ns : std::min<int64_t>(na, k * ((na + ns - 1) / ns))));
        it.p1 = (int32_t)(f0 + (even ? na * (k + 1) / ns
                                     : std::min<int64_t>(na, (k + 1) * ((na + ns - 1) / ns))));
        it.pos_q = (int32_t)(sq->n_slots - 1);
        it.n_splits = ns;
        it.item0 = item0[i];
        it.win_lo = win_lo[i];
        it.part = (int32_t)items.size();
        it.nb = 1;
        items.push_back(it);
      }
    };
    if (c->use_mma) {
      // Tensor-core path: the work is a list of segments (ranges of one
      // row's active pages, read for one row or for several rows that hold
      // them identically); blocks for a quarter of what fits the GPU at once
      // (times decode_waves), the splits of each segment proportional to its
      // pages and equal within it; one split holds at most kDecodeMaxTiles
      // tiles.  Leaving most block slots free lets the next decode call's
      // blocks start while this call runs (programmatic dependent launch):
      // back to back, a quarter wave beat a whole wave by 2-45% depending on
      // the batch.
      const int64_t tpp = c->cfg.page_size / 16;
      const int G = c->cfg.hq / c->cfg.hkv;
      std::vector<Segment> segs, tsegs;   // one-row kernel / tensor-core shared-prefix kernel
      // share: 0 none, 1 tensor-core shared-prefix items, 2 shared items of
      // the one-row kernel (at most `mcap` rows each)
      auto plan_mma = [&](int share, int mcap, int64_t min_waves) -> int {
        segs.clear();
        tsegs.clear();
        sitems.clear();
        if (share) {
          const int cap = share == 1 ? std::min(kShareRows / G, kShareMaxMembers) : mcap;
          const bool full_only = share == 1;
          // the shared segments found for the same rows at the same layout
          // versions are still exact (appends change only pages past them)
          auto& sc = c->share_cache;
          bool hit = full_only && sc.full_only && sc.cap == cap && (int)sc.seqs.size() == n_seqs &&
                     std::equal(sc.seqs.begin(), sc.seqs.end(), seqs);
          for (int i = 0; hit && i < n_seqs; ++i) hit = sc.layout[i] == hs[i]->layout;
          std::vector<Segment> shared;
          if (hit) {
            shared = sc.shared;
          } else {
            find_shared(c, hs, cap, full_only, &shared);
            if (full_only) {
              sc.seqs.assign(seqs, seqs + n_seqs);
              sc.layout.resize(n_seqs);
              for (int i = 0; i < n_seqs; ++i) sc.layout[i] = hs[i]->layout;
              sc.cap = cap;
              sc.full_only = true;
              sc.shared = shared;
            }
          }
          std::vector<Segment> rest;
          complete_segments(hs, shared, &rest);
          for (auto& sg : shared) (share == 1 && sg.rows.size() > 1 ? tsegs : segs).push_back(sg);
          for (auto& sg : rest) segs.push_back(std::move(sg));
        } else {
          for (int i = 0; i < n_seqs; ++i) {
            Segment sg;
            sg.a0 = first[i];
            sg.a1 = hs[i]->n_active_pages;
            sg.rows = {i};
            sg.lens = {sg.a1 - sg.a0};
            sg.starts = {sg.a0};
            segs.push_back(std::move(sg));
          }
        }
        // a row read by shared-prefix items is merged by a one-row item of
        // the one-row kernel (launched after them): give it one if needed
        {
          std::vector<char> has(n_seqs, 0);
          for (auto& sg : segs) has[sg.rows[0]] = 1;
          for (auto& sg : tsegs)
            for (int32_t r : sg.rows)
              if (!has[r]) {
                Segment e;
                e.a0 = e.a1 = 0;
                e.rows = {r};
                e.lens = {0};
                segs.push_back(std::move(e));
                has[r] = 1;
              }
        }
        const int64_t resident = (int64_t)c->sm_count * c->mma_blocks_per_sm;
        const int64_t quarter = std::max<int64_t>(1, resident / 4);
        const int64_t pairs = (int64_t)segs.size() * c->cfg.hkv;
        const int64_t waves = std::max<int64_t>(min_waves, (pairs + quarter - 1) / quarter);
        int64_t target = std::max<int64_t>((int64_t)segs.size(), waves * quarter / c->cfg.hkv);
        // A consumer warp of an item with nb column blocks reads nb/4 of the
        // tiles (one row: a quarter), so the work of a split, the cap of
        // kDecodeMaxTiles tiles for a one-row split and the balancing all
        // count pages * nb.
        auto nb_of = [&](const Segment& sg) -> int64_t {
          const int cols = ((int)sg.rows.size() * G + 7) / 8;
          return sg.rows.size() < 2 || cols <= 1 ? 1 : cols <= 2 ? 2 : 4;
        };
        int64_t sum = 0, parts = 0;
        using Entry = std::pair<int64_t, int>;        // (work per split, segment)
        std::priority_queue<Entry> pq;
        for (int k = 0; k < (int)segs.size(); ++k) {
          const int64_t w = (segs[k].a1 - segs[k].a0) * nb_of(segs[k]);
          segs[k].ns = (int32_t)std::max<int64_t>(1, (w * tpp + kDecodeMaxTiles - 1) / kDecodeMaxTiles);
          segs[k].ns = (int32_t)std::min<int64_t>(segs[k].ns, std::max<int64_t>(1, segs[k].a1 - segs[k].a0));
          sum += segs[k].ns;
          parts += (int64_t)segs[k].ns * segs[k].rows.size();
          pq.push({(w + segs[k].ns - 1) / segs[k].ns, k});
        }
        // shared-prefix items: at least kSharePagesMin pages each, longer
        // until all of them fit one wave of CTAs (two per SM), counting the
        // rounding up of every segment: a CTA's set-up and epilogue weigh
        // like a few tiles, and a second, partial wave costs a whole CTA's
        // time -- and holds back the one-row kernel of the call, which
        // starts only once every CTA of this one has
        if (!tsegs.empty()) {
          int64_t tp = 0;
          for (auto& sg : tsegs) tp += sg.a1 - sg.a0;
          const int64_t wave = std::max<int64_t>(1, 2 * c->sm_count);
          auto ctas = [&](int64_t per) {
            int64_t n = 0;
            for (auto& sg : tsegs) n += (sg.a1 - sg.a0 + per - 1) / per;
            return n * c->cfg.hkv;
          };
          int64_t per = std::min<int64_t>(
              kSharePagesMax,
              std::max<int64_t>(kSharePagesMin, (tp * c->cfg.hkv + wave - 1) / wave));
          while (per < kSharePagesMax && ctas(per) > wave)
            per = std::min<int64_t>(kSharePagesMax, per + std::max<int64_t>(1, per / 16));
          for (auto& sg : tsegs) {
            sg.ns = (int32_t)std::max<int64_t>(1, (sg.a1 - sg.a0 + per - 1) / per);
            parts += (int64_t)sg.ns * sg.rows.size();
          }
        }
        // next to shared-prefix items the one-row items are what is left of
        // each row (its own pages, often long): a full wave of blocks keeps
        // the longest of them off the critical path
        if (!tsegs.empty()) target = std::max<int64_t>(target, resident / c->cfg.hkv);
        target = std::min<int64_t>(std::max(target, sum), kMaxItems);
        // a call with nothing to overlap its end with (a whole-wave split, or
        // one-row items next to shared-prefix items) runs whole waves of
        // blocks: a partial last wave would leave the rest of the GPU idle
        if (min_waves >= 4 || !tsegs.empty()) {
          const int64_t per_wave = std::max<int64_t>(1, resident / c->cfg.hkv);
          if (target > per_wave)
            target = std::min<int64_t>(kMaxItems, (target + per_wave - 1) / per_wave * per_wave);
        }
        // split the segment with the most work per split until there are
        // `tgt` splits (or nothing worth splitting is left)
        auto split_upto = [&](int64_t tgt, std::vector<int32_t>* ns, int64_t* n_sum, int64_t* n_parts) {
          ns->resize(segs.size());
          for (size_t k = 0; k < segs.size(); ++k) (*ns)[k] = segs[k].ns;
          auto q = pq;
          int64_t s = sum, p = parts;
          while (s < tgt && !q.empty()) {
            const Entry e = q.top();
            q.pop();
            const Segment& sg = segs[e.second];
            int32_t& m = (*ns)[e.second];
            const int64_t na = sg.a1 - sg.a0;
            if ((na + m - 1) / m <= 2) break;           // splits of 1-2 pages gain nothing
            if (p + (int64_t)sg.rows.size() > kMaxItems) continue;
            ++m;
            ++s;
            p += sg.rows.size();
            q.push({(na * nb_of(sg) + m - 1) / m, e.second});
          }
          *n_sum = s;
          *n_parts = p;
        };
        std::vector<int32_t> ns_best;
        int64_t sum_best = sum, parts_best = parts;
        if (tsegs.empty()) {
          split_upto(target, &ns_best, &sum_best, &parts_best);
        } else {
          // Next to shared-prefix items the one-row kernel runs on its own
          // (nothing of the next call overlaps its end), so the split count
          // is chosen by the time the block scheduler would take: blocks
          // dispatched in plan order (longest first, an item's KV heads
          // together) onto the resident block slots as they free up, a block
          // costing its pages x column blocks plus a fixed start-up.  The
          // count that evens the slots out best wins; whole waves of
          // similar items can end with some slots holding two long ones.
          const int64_t per_wave = std::max<int64_t>(1, resident / c->cfg.hkv);
          const int64_t step = std::max<int64_t>(1, per_wave / 4);
          double best = -1.0;
          std::vector<int32_t> ns;
          std::vector<int64_t> w;
          for (int64_t tgt = target; tgt <= std::min<int64_t>(kMaxItems, target + 4 * per_wave);
               tgt += step) {
            int64_t s = 0, p = 0;
            split_upto(tgt, &ns, &s, &p);
            w.clear();
            for (size_t k = 0; k < segs.size(); ++k) {
              const int64_t na = segs[k].a1 - segs[k].a0;
              for (int32_t j = 0; j < ns[k]; ++j)
                w.push_back((na * (j + 1) / ns[k] - na * j / ns[k]) * nb_of(segs[k]) + kBlockStartPages);
            }
            std::sort(w.begin(), w.end(), std::greater<int64_t>());
            std::priority_queue<int64_t, std::vector<int64_t>, std::greater<int64_t>> slots;
            for (int64_t i = 0; i < resident; ++i) slots.push(0);
            int64_t end = 0;
            for (int64_t x : w)
              for (int h = 0; h < c->cfg.hkv; ++h) {
                const int64_t t = slots.top() + x;
                slots.pop();
                slots.push(t);
                end = std::max(end, t);
              }
            if (best < 0 || end < best) {
              best = (double)end;
              ns_best = ns;
              sum_best = s;
              parts_best = p;
            }
          }
        }
        for (size_t k = 0; k < segs.size(); ++k) segs[k].ns = ns_best[k];
        sum = sum_best;
        parts = parts_best;
        if (sum > kMaxItems || parts > kMaxItems) return AKV_ECAPACITY;
        // the members of split k of a segment: those whose part reaches
        // into it; a row's partial slots are side by side
        auto split_range = [](const Segment& sg, int32_t k, int64_t* s0, int64_t* s1) {
          const int64_t na = sg.a1 - sg.a0;
          *s0 = na * k / sg.ns;
          *s1 = na * (k + 1) / sg.ns;
        };
        auto n_in = [&](const Segment& sg, int64_t s0) {
          int nm = 0;
          for (size_t m = 0; m < sg.rows.size(); ++m) nm += m == 0 || sg.lens[m] > s0;
          return nm;
        };
        for (auto* list : {&segs, &tsegs})
          for (auto& sg : *list)
            for (int32_t k = 0; k < sg.ns; ++k) {
              int64_t s0, s1;
              split_range(sg, k, &s0, &s1);
              for (size_t m = 0; m < sg.rows.size(); ++m)
                if (m == 0 || sg.lens[m] > s0) ++splits[sg.rows[m]];
            }
        std::vector<int32_t> cursor(n_seqs, 0);
        for (int i = 0, acc = 0; i < n_seqs; ++i) {
          item0[i] = acc;
          acc += splits[i];
        }
        items.clear();
        members.clear();
        shared = false;
        auto add_members = [&](const Segment& sg, int64_t s0, int64_t s1) -> int {
          for (size_t m = 0; m < sg.rows.size(); ++m) {
            if (m > 0 && sg.lens[m] <= s0) continue;
            if (members.size() >= (size_t)kMaxMembers) return AKV_ECAPACITY;
            const int32_t r = sg.rows[m];
            const int64_t pages = std::min<int64_t>(sg.lens[m], s1) - s0;
            members.push_back(DecodeMember{r, (int32_t)(hs[r]->n_slots - 1), item0[r], splits[r],
                                           item0[r] + cursor[r]++, (int32_t)(pages * tpp)});
          }
          return AKV_OK;
        };
        auto one_row = [&](int r0, int64_t p0, int64_t p1) {
          DecodeItem it{};
          it.dslot = hs[r0]->dslot;
          it.row = r0;
          it.p0 = (int32_t)p0;
          it.p1 = (int32_t)p1;
          it.pos_q = (int32_t)(hs[r0]->n_slots - 1);
          it.n_splits = splits[r0];
          it.item0 = item0[r0];
          it.win_lo = win_lo[r0];
          it.part = item0[r0] + cursor[r0];
          it.nb = 1;
          return it;
        };
        for (auto& sg : tsegs) {
          for (int32_t k = 0; k < sg.ns; ++k) {
            int64_t s0, s1;
            split_range(sg, k, &s0, &s1);
            if (n_in(sg, s0) < 2) {                      // only the first row left
              items.push_back(one_row(sg.rows[0], sg.a0 + s0, sg.a0 + s1));
              ++cursor[sg.rows[0]];
              continue;
            }
            ShareItem si{};
            si.dslot = hs[sg.rows[0]]->dslot;
            si.p0 = (int32_t)(sg.a0 + s0);
            si.p1 = (int32_t)(sg.a0 + s1);
            si.mem0 = (int32_t)members.size();
            if (add_members(sg, s0, s1)) return AKV_ECAPACITY;
            si.n_mem = (int32_t)members.size() - si.mem0;
            sitems.push_back(si);
          }
        }
        for (auto& sg : segs) {
          const int r0 = sg.rows[0];
          for (int32_t k = 0; k < sg.ns; ++k) {
            int64_t s0, s1;
            split_range(sg, k, &s0, &s1);
            const int nm = n_in(sg, s0);
            DecodeItem it = one_row(r0, sg.a0 + s0, sg.a0 + s1);
            const int cols = (nm * G + 7) / 8;
            it.nb = cols <= 1 ? 1 : cols <= 2 ? 2 : 4;
            if (nm > 1) {
              it.mem0 = (int32_t)members.size();
              it.n_mem = nm;
              if (add_members(sg, s0, s1)) return AKV_ECAPACITY;
              shared = true;
            } else {
              ++cursor[r0];
            }
            items.push_back(it);
          }
        }
        if ((int64_t)items.size() > kMaxItems || (int64_t)sitems.size() > kMaxItems) return AKV_ECAPACITY;
        // longest first: the kernel's blocks go out in plan order
        std::stable_sort(items.begin(), items.end(), [](const DecodeItem& x, const DecodeItem& y) {
          return (int64_t)(x.p1 - x.p0) * x.nb > (int64_t)(y.p1 - y.p0) * y.nb;
        });
        return AKV_OK;
      };
      // rows can hold the same pages only within a fork family
      bool share = c->decode_share > 0 && window == 0 && n_seqs > 1;
      if (share) {
        std::vector<int64_t> fam(n_seqs);
        for (int i = 0; i < n_seqs; ++i) fam[i] = hs[i]->family;
        std::sort(fam.begin(), fam.end());
        share = std::adjacent_find(fam.begin(), fam.end()) != fam.end();
      }
      const int mode = !share ? 0 : (c->decode_share == 1 && decode_share_supported(c->g)) ? 1 : 2;
      const int mcap = c->decode_share > 1 ? c->decode_share : std::max(1, 16 / G);
      int rc = plan_mma(mode, std::min(mcap, 32 / G), c->decode_waves);
      bool plain = mode == 0;
      if (rc && mode) {
        std::fill(splits.begin(), splits.end(), 0);
        rc = plan_mma(0, 1, c->decode_waves);
        plain = true;
      }
      if (rc) return fail(c, AKV_ECAPACITY, "decode needs more than %d work items", kMaxItems);
      combine = false;                                 // merged inside the kernel
      // Calls without shared items get a second split for a whole wave of
      // blocks; the kernel takes it when the call runs on its own (see
      // DecodeArgs::items_w).  The quarter-wave split above is best when
      // calls come back to back, and a call on its own would leave three
      // quarters of the GPU idle with it.
      // Only where the quarter-wave split keeps too few tile copies in flight
      // to fill HBM on its own (its blocks x the ring's 8 stages of K and V
      // tiles): the 120B-shaped call (120 blocks, D 64: ~4 MB) gains from a
      // whole wave alone, the 8B-shaped one (256 blocks, D 128: 16 MB)
      // loses to the extra splits' merges.
      const int64_t q_blocks = (int64_t)items.size() * c->cfg.hkv;
      const int64_t in_flight = q_blocks * 8 * 2 * 16 * (int64_t)c->cfg.head_dim * 2;
      if (plain && c->decode_waves < 4 && in_flight < ((int64_t)12 << 20)) {
        std::vector<DecodeItem> q_items = std::move(items);
        std::vector<int32_t> q_item0 = item0, q_splits = splits;
        std::fill(splits.begin(), splits.end(), 0);
        if (plan_mma(0, 1, 4) == AKV_OK && items.size() > q_items.size()) items_w = std::move(items);
        items = std::move(q_items);
        item0 = std::move(q_item0);
        splits = std::move(q_splits);
      }
    } else {
      // split so that the (item, kv head) blocks fill the GPU a few times over
      const int64_t tgt = (int64_t)c->sm_count * 8;
      int64_t pps = std::max<int64_t>(4, (total * c->cfg.hkv + tgt - 1) / tgt);
      for (;;) {
        int64_t n_it = 0;
        for (int i = 0; i < n_seqs; ++i)
          n_it += std::max<int64_t>(1, (hs[i]->n_active_pages - first[i] + pps - 1) / pps);
        if (n_it <= kMaxItems) break;
        pps *= 2;
      }
      for (int i = 0; i < n_seqs; ++i)
        emit(i, (int32_t)std::max<int64_t>(1, (hs[i]->n_active_pages - first[i] + pps - 1) / pps),
             false);
    }
    Blob blob;
    blob.put(items.data(), items.size());
    blob.put(item0.data(), item0.size());
    blob.put(splits.data(), splits.size());
    const size_t o_members = blob.put(members.data(), members.size());
    const size_t o_sitems = blob.put(sitems.data(), sitems.size());
    const size_t o_items_w = blob.put(items_w.data(), items_w.size());
    if (blob.b.size() > c->plan_cap) return fail(c, AKV_ECAPACITY, "decode plan too large");
    plan = &c->plans[0];
    for (auto& pl : c->plans)
      if (pl.used < plan->used) plan = &pl;
    int rc = upload_large(c, blob, plan->d);
    if (rc) {
      plan->epoch = ~0ULL;
      return rc;
    }
    plan->epoch = c->epoch;
    plan->window = window;
    plan->seqs.assign(seqs, seqs + n_seqs);
    plan->items = (int)items.size();
    plan->combine = combine;
    plan->shared = shared;
    plan->members = (int)members.size();
    plan->shared_items = (int)sitems.size();
    for (const DecodeItem& it : items) plan->shared_items += it.n_mem > 0;
    plan->o_members = o_members;
    plan->sitems = (int)sitems.size();
    plan->o_sitems = o_sitems;
    plan->items_w = (int)items_w.size();
    plan->o_items_w = o_items_w;
  }
  plan->used = ++c->plan_clock;
  c->last_items = plan->items + plan->sitems;
  c->last_shared = plan->shared_items;
  c->last_members = plan->members;
  const size_t n_items = (size_t)plan->items;
  const size_t o_item0 = (n_items * sizeof(DecodeItem) + 15) & ~size_t(15);
  const size_t o_splits = (o_item0 + n_seqs * sizeof(int32_t) + 15) & ~size_t(15);
  DecodeArgs a{};
  a.tm_k = c->tm_k;
  a.tm_v = c->tm_v;
  a.tm_k4 = c->tm_k4;
  a.tm_v4 = c->tm_v4;
  a.use_mma = c->use_mma;
  a.g = c->g;
  a.sa = c->sa;
  a.items = reinterpret_cast<const DecodeItem*>(plan->d);
  a.n_items = plan->items;
  a.layer = layer;
  a.q = q;
  a.out = out;
  a.part_acc = c->d_part_acc;
  a.part_ml = c->d_part_ml;
  a.cs = c->d_cs;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c->cfg.head_dim));
  a.err = c->d_err;
  a.wait_limit = c->wait_limit;
  a.counters = c->d_counters;
  a.n_rows = n_seqs;
  a.max_seqs = c->cfg.max_seqs;
  a.counter_rows = kMaxItems;
  a.part_cap = kMaxItems;
  a.members = reinterpret_cast<const DecodeMember*>(plan->d + plan->o_members);
  a.n_members = plan->members;
  a.shared = plan->shared;
  a.share_items = reinterpret_cast<const ShareItem*>(plan->d + plan->o_sitems);
  a.n_share_items = plan->sitems;
  a.items_w = reinterpret_cast<const DecodeItem*>(plan->d + plan->o_items_w);
  a.n_items_w = plan->items_w;
  a.mode_words = c->d_mode;
  a.exit_words = c->d_exits;
  a.done_word = c->d_done;
  if (c->use_mma && plan->items > 0) {
    if (++c->decode_call >= (1u << 29)) c->decode_call = 1;   // the words keep 29 bits of it
    a.call_id = c->decode_call;
  }
  // early launch only right behind a decode call of this cache (not behind
  // the copy of a new plan, an append or any other kernel of this cache)
  a.pdl = c->launches == c->decode_tail;
  const uint64_t before = c->launches;
  if (plan->sitems > 0) {
    CK(launch_decode_share(a, c->stream));
    ++c->launches;
    a.pdl = true;                 // behind the shared-prefix kernel, a decode kernel
  }
  CK(launch_decode(a, plan->combine, n_seqs, reinterpret_cast<const int32_t*>(plan->d + o_item0),
                   reinterpret_cast<const int32_t*>(plan->d + o_splits), c->stream));
  if (plan->items > 0) c->launches += plan->combine ? 2 : 1;
  if (c->launches != before) c->decode_tail = c->launches;
  return AKV_OK;
}

// ---- segment-batch restore attention -------------------------------------------

namespace {

// Restore attention of the tokens with want[t] (all of them when `sel` is
// null; else the n_sel increasing tokens of `sel`).
int restore_impl(akv_cache* c, const akv_op* ops, int32_t n_ops, int32_t layer, const void* q,
                 const void* k_raw, const void* v, int32_t n_tokens, const int32_t* sel,
                 int32_t n_sel, float* out) {
  if (!c || n_ops < 0 || (n_ops > 0 && !ops) || n_tokens < 0) return AKV_EINVAL;
  if (layer < 0 || layer >= c->cfg.layers) return fail(c, AKV_EINVAL, "layer %d out of range", layer);
  if (n_tokens > 0 && (!q || !k_raw || !v || !out)) return AKV_EINVAL;
  std::vector<char> want(n_tokens, sel ? 0 : 1);
  if (sel || n_sel) {
    if (n_sel < 0 || (n_sel > 0 && !sel)) return AKV_EINVAL;
    for (int32_t i = 0; i < n_sel; ++i) {
      if (sel[i] < 0 || sel[i] >= n_tokens || (i > 0 && sel[i] <= sel[i - 1]))
        return fail(c, AKV_EINVAL, "selected tokens must increase within [0, %d)", n_tokens);
      want[sel[i]] = 1;
    }
  }
  // plan: times, eras, era slots (page 1 A.1.1: split at every drop/repos)
  constexpr int32_t kNever = INT32_MAX;
  std::vector<int32_t> held, pending;
  std::vector<char> alive(n_tokens, 0);
  std::vector<int32_t> birth(n_tokens, 0), death(n_tokens, kNever);
  std::vector<RestoreKey> keys;
  std::vector<RestoreQuery> queries(n_tokens);
  int32_t next = 0, clock = 0;
  auto close_era = [&]() {
    const int32_t off = (int32_t)keys.size();
    for (size_t slot = 0; slot < held.size(); ++slot) {
      const int32_t t = held[slot];
      keys.push_back({t, (int32_t)slot, birth[t], death[t]});
    }
    for (int32_t t : pending) queries[t].era_off = off;
    pending.clear();
    std::vector<int32_t> keep;
    for (int32_t t : held)
      if (alive[t]) keep.push_back(t);
    held.swap(keep);
  };
  for (int32_t i = 0; i < n_ops; ++i) {
    const akv_op& op = ops[i];
    if (op.kind == AKV_OP_APPEND) {
      if (op.count < 0 || next + (int64_t)op.count > n_tokens)
        return fail(c, AKV_EINVAL, "program appends more than %d tokens", n_tokens);
      for (int32_t k = 0; k < op.count; ++k) {
        const int32_t t = next++;
        birth[t] = clock++;
        alive[t] = 1;
        held.push_back(t);
        if ((int64_t)held.size() > c->cfg.max_slots)
          return fail(c, AKV_ECAPACITY, "restore position reaches max_slots %d", c->cfg.max_slots);
        const int32_t pos = (int32_t)held.size() - 1;
        queries[t] = {t, pos, birth[t], 0, pos + 1};
        pending.push_back(t);
      }
    } else if (op.kind == AKV_OP_DROP) {
      if (op.count < 0 || (op.count > 0 && !op.ranges)) return fail(c, AKV_EINVAL, "bad drop op");
      for (int32_t r = 0; r < op.count; ++r) {
        const int64_t b = op.ranges[2 * r], e = op.ranges[2 * r + 1];
        if (b < 0 || e < b || e > next)
          return fail(c, AKV_ERANGE, "drop range [%lld, %lld) outside [0, %d)", (long long)b,
                      (long long)e, next);
        for (int64_t t = b; t < e; ++t)
          if (alive[t]) { alive[t] = 0; death[t] = clock; }
      }
      ++clock;
    } else if (op.kind == AKV_OP_REPOS) {
      close_era();
      ++clock;
    } else {
      return fail(c, AKV_EINVAL, "unknown op kind %d", op.kind);
    }
  }
  if (next != n_tokens) return fail(c, AKV_EINVAL, "program appends %d tokens, not %d", next, n_tokens);
  close_era();
  if (n_tokens == 0 || (sel && n_sel == 0)) return AKV_OK;
  // the selected queries, in order (the CUDA-core kernel takes one per block)
  std::vector<RestoreQuery> squeries;
  for (int32_t t = 0; t < n_tokens; ++t)
    if (want[t]) squeries.push_back(queries[t]);

  // tensor-core path: tiles of consecutive selected query tokens of one era
  std::vector<RestoreTile> tiles;
  const bool mma = restore_mma_supported(c->g) && !c->restore_generic;
  if (mma) {
    const int tt = restore_tile_tokens(c->g);
    const int32_t W = c->windows[layer];
    for (int32_t t = 0; t < n_tokens;) {
      if (!want[t]) {
        ++t;
        continue;
      }
      int32_t e = t + 1;
      while (e < n_tokens && e - t < tt && want[e] && queries[e].era_off == queries[t].era_off) ++e;
      const int32_t lo = W > 0 ? std::max(0, queries[t].pos - W + 1) : 0;
      tiles.push_back({queries[t].era_off, t, e - t, lo, queries[e - 1].key_end});
      t = e;
    }
  }
  // two-tile form: consecutive tiles of one era share a CTA (the later one's
  // key range extends the earlier one's by its own tokens)
  std::vector<int2> pairs;
  if (mma && c->restore_pairs) {
    for (size_t i = 0; i < tiles.size();) {
      if (i + 1 < tiles.size() && tiles[i + 1].era_off == tiles[i].era_off) {
        pairs.push_back(make_int2((int)i, (int)i + 1));
        i += 2;
      } else {
        pairs.push_back(make_int2((int)i, -1));
        i += 1;
      }
    }
  }
  Blob blob;
  const size_t o_keys = blob.put(keys.data(), keys.size());
  const size_t o_q = blob.put(queries.data(), queries.size());
  const size_t o_sq = blob.put(squeries.data(), squeries.size());
  const size_t o_t = blob.put(tiles.data(), tiles.size());
  const size_t o_p = blob.put(pairs.data(), pairs.size());
  // scratch: [K versions | V versions | descriptor]
  const size_t elem = c->cfg.dtype == AKV_DTYPE_BF16 ? 2 : 4;
  const size_t half = (keys.size() * (size_t)c->cfg.hkv * c->cfg.head_dim * elem + 255) & ~size_t(255);
  const size_t need = 2 * half + blob.b.size();
  if (need > c->restore_cap) {
    CK(cudaStreamSynchronize(c->stream));
    cudaFree(c->d_restore);
    c->d_restore = nullptr;
    c->restore_cap = 0;
    CK(cudaMalloc(&c->d_restore, need));
    c->restore_cap = need;
  }
  char* d = static_cast<char*>(c->d_restore) + 2 * half;
  int rc = upload_large(c, blob, d);
  if (rc) return rc;
  RestoreArgs a{};
  a.tiles = reinterpret_cast<const RestoreTile*>(d + o_t);
  a.n_tiles = (int32_t)tiles.size();
  a.pairs = reinterpret_cast<const int2*>(d + o_p);
  a.n_pairs = (int32_t)pairs.size();
  a.use_mma = mma;
  a.wait_limit = c->wait_limit;
  if (mma && !make_restore_tensor_maps(c->g, c->d_restore, static_cast<char*>(c->d_restore) + half,
                                       (int64_t)keys.size(), &a.tm_k, &a.tm_v))
    a.use_mma = 0;   // no tensor maps: the CUDA-core kernel
  a.g = c->g;
  a.keys = reinterpret_cast<const RestoreKey*>(d + o_keys);
  a.n_keys = (int32_t)keys.size();
  // the tensor-core kernels read queries by token, the CUDA-core one the
  // selected ones in order
  a.queries = reinterpret_cast<const RestoreQuery*>(d + (a.use_mma ? o_q : o_sq));
  a.n_queries = a.use_mma ? n_tokens : (int32_t)squeries.size();
  a.q = q;
  a.k_raw = k_raw;
  a.v = v;
  a.n_tokens = n_tokens;
  a.k_era = c->d_restore;
  a.v_era = static_cast<char*>(c->d_restore) + half;
  a.out = out;
  a.cs = c->d_cs;
  a.max_pos = c->cfg.max_slots;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c->cfg.head_dim));
  a.window = c->windows[layer];
  a.err = c->d_err;
  CK(launch_restore(a, c->stream));
  c->launches += 2;
  return AKV_OK;
}

}  // namespace

int akv_restore_attention(akv_cache* c, const akv_op* ops, int32_t n_ops, int32_t layer,
                          const void* q, const void* k_raw, const void* v, int32_t n_tokens,
                          float* out) {
  return restore_impl(c, ops, n_ops, layer, q, k_raw, v, n_tokens, nullptr, 0, out);
}

int akv_restore_attention_tokens(akv_cache* c, const akv_op* ops, int32_t n_ops, int32_t layer,
                                 const void* q, const void* k_raw, const void* v, int32_t n_tokens,
                                 const int32_t* tokens, int32_t n_sel, float* out) {
  if (n_sel > 0 && !tokens) return AKV_EINVAL;
  static const int32_t kNone = 0;
  return restore_impl(c, ops, n_ops, layer, q, k_raw, v, n_tokens, tokens ? tokens : &kNone,
                      n_sel, out);
}

// Recovery plan (see akv.h).  A token u is in the plan when it is missing and
// either needed or read by a plan token t > u: t's query read u when u was
// still active at t's append (u dropped after t's append, or never).  Over
// the plan tokens after u that holds for the earliest of them if it holds for
// any (the earliest has the earliest append time), so one backward pass over
// the tokens decides every token.
int akv_restore_plan_recovery(const akv_op* ops, int32_t n_ops, int32_t n_tokens,
                              const uint8_t* missing, const uint8_t* need,
                              int32_t* tokens_out, int32_t* n_out) {
  if (n_ops < 0 || (n_ops > 0 && !ops) || n_tokens < 0 || !n_out ||
      (n_tokens > 0 && (!missing || !tokens_out)))
    return AKV_EINVAL;
  constexpr int64_t kNever = INT64_MAX;
  std::vector<int64_t> birth(n_tokens, 0), death(n_tokens, kNever);
  std::vector<char> alive(n_tokens, 0);
  int32_t next = 0;
  int64_t clock = 0;                     // one tick per appended token and per drop
  for (int32_t i = 0; i < n_ops; ++i) {
    const akv_op& op = ops[i];
    if (op.kind == AKV_OP_APPEND) {
      if (op.count < 0 || next + (int64_t)op.count > n_tokens) return AKV_EINVAL;
      for (int32_t k = 0; k < op.count; ++k) {
        birth[next] = clock++;
        alive[next++] = 1;
      }
    } else if (op.kind == AKV_OP_DROP) {
      if (op.count < 0 || (op.count > 0 && !op.ranges)) return AKV_EINVAL;
      for (int32_t r = 0; r < op.count; ++r) {
        const int64_t b = op.ranges[2 * r], e = op.ranges[2 * r + 1];
        if (b < 0 || e < b || e > next) return AKV_ERANGE;
        for (int64_t t = b; t < e; ++t)
          if (alive[t]) {
            alive[t] = 0;
            death[t] = clock;
          }
      }
      ++clock;
    } else if (op.kind != AKV_OP_REPOS) {
      return AKV_EINVAL;
    }
  }
  if (next != n_tokens) return AKV_EINVAL;
  int64_t first_birth = kNever;          // append time of the earliest plan token so far
  int32_t n = 0;
  for (int32_t u = n_tokens - 1; u >= 0; --u) {
    if (!missing[u]) continue;
    const bool needed = need ? need[u] != 0 : alive[u] != 0;
    if (needed || death[u] > first_birth) {
      tokens_out[n++] = u;
      first_birth = birth[u];
    }
  }
  std::reverse(tokens_out, tokens_out + n);
  *n_out = n;
  return AKV_OK;
}

int akv_set_layer_window(akv_cache* c, int32_t layer, int32_t window) {
  if (!c) return AKV_EINVAL;
  if (layer < 0 || layer >= c->cfg.layers || window < 0)
    return fail(c, AKV_EINVAL, "bad layer %d or window %d", layer, window);
  c->windows[layer] = window;
  return AKV_OK;
}


// ---- history-keyed prefix sharing / drop-aware eviction ----------------------
//
// Paper review A.1.2 and 4.2.2-4.2.3; repo review 5.4 (materialisation plan:
// reuse a stored version, or take a new slot and copy, with copy-on-write of
// pages handed to another branch) and 5.6 (eviction candidates).


namespace {

HKey history_key(const PrefixIndex& idx, const std::vector<PRec>& recs, size_t n) {
  HKey k;
  for (size_t i = 0; i < n; ++i) {
    const PRec& r = recs[i];
    if (r.kind == kRecT) {
      k.absorb(kRecAppend);
      k.absorb((uint64_t)(uint32_t)r.v);
    } else if (r.kind == kRecD) {
      const auto& d = idx.delta(r.v);
      k.absorb(kRecDrop);
      k.absorb(d.size());
      for (const auto& iv : d) { k.absorb((uint64_t)iv.first); k.absorb((uint64_t)iv.second); }
    } else {
      k.absorb(kRecRepos);
    }
  }
  return k;
}

int grow_fork_scratch(akv_cache* c, size_t need) {
  if (need <= c->fork_cap) return AKV_OK;
  CK(cudaStreamSynchronize(c->stream));
  cudaFree(c->d_fork);
  c->d_fork = nullptr;
  c->fork_cap = 0;
  CK(cudaMalloc(&c->d_fork, need));
  c->fork_cap = need;
  return AKV_OK;
}

}  // namespace

int akv_prefix_publish(akv_cache* c, akv_prefix_index* x, int64_t seq, const akv_op* ops,
                       int32_t n_ops, const int32_t* token_ids, int32_t n_tokens, int64_t* entry) {
  if (!c || !x || !entry) return AKV_EINVAL;
  if (x->idx.page_size() != c->cfg.page_size)
    return fail(c, AKV_EINVAL, "index page size %d != cache page size %d", x->idx.page_size(),
                c->cfg.page_size);
  HostSeq* s = find(c, seq);
  if (!s) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seq);
  PProgram p;
  const char* why = "";
  int rc = x->idx.expand(ops, n_ops, token_ids, n_tokens, &p, &why);
  if (rc) return fail(c, rc, "%s", why);
  const HKey k = history_key(x->idx, p.recs, p.recs.size());
  if (k.a != s->key.a || k.b != s->key.b)
    return fail(c, AKV_EINVAL, "the program is not the history of sequence %lld", (long long)seq);
  const int64_t same = x->idx.find_equal(p);
  if (same >= 0 && find(c, same)) {
    x->idx.touch(same, -1);
    *entry = same;
    return AKV_OK;
  }
  int64_t snap = -1;
  rc = akv_seq_fork(c, seq, &snap);
  if (rc) return rc;
  find(c, snap)->frozen = true;
  if (x->idx.insert(snap, p, -1) != AKV_OK) {
    akv_seq_free(c, snap);
    return fail(c, AKV_EINVAL, "entry %lld already in the index", (long long)snap);
  }
  *entry = snap;
  return AKV_OK;
}

int akv_prefix_fork(akv_cache* c, akv_prefix_index* x, const akv_op* ops, int32_t n_ops,
                    const int32_t* token_ids, int32_t n_tokens, akv_prefix_match_t* mo,
                    int64_t* child) {
  if (!c || !x || !child) return AKV_EINVAL;
  *child = -1;
  if (x->idx.page_size() != c->cfg.page_size)
    return fail(c, AKV_EINVAL, "index page size %d != cache page size %d", x->idx.page_size(),
                c->cfg.page_size);
  PProgram req;
  const char* why = "";
  int rc = x->idx.expand(ops, n_ops, token_ids, n_tokens, &req, &why);
  if (rc) return fail(c, rc, "%s", why);
  const PMatch m = x->idx.match(req);
  if (mo) {
    mo->kind = m.kind;
    mo->n_records = m.n_records;
    mo->entry = m.entry;
    mo->n_tokens = m.n_tokens;
    mo->n_rotated = m.n_rotated;
    mo->op_index = m.op_index;
    mo->op_tokens = m.op_tokens;
  }
  if (m.kind == AKV_MATCH_NONE) return AKV_OK;
  HostSeq* E = find(c, m.entry);
  const PEntry* pe = x->idx.entry(m.entry);
  if (!E || !pe) return fail(c, AKV_ENOSEQ, "entry %lld has no snapshot in this cache", (long long)m.entry);
  const PrefixIndex::State st = x->idx.replay(req.recs, (size_t)m.n_records);
  const int S = c->cfg.page_size;
  const int64_t n_slots = st.next_pos;
  const int64_t n_pages = (n_slots + S - 1) / S;
  if (n_slots > c->cfg.max_slots) return fail(c, AKV_ECAPACITY, "prefix holds more than max_slots");
  if (c->free_dslots.empty()) return fail(c, AKV_ECAPACITY, "max_seqs (%d) sequences alive", c->cfg.max_seqs);
  // per destination page: 0 no needed token, 1 every needed token keeps its slot, 2 fresh
  std::vector<int8_t> kind((size_t)n_pages, 0);
  const size_t n_tok = st.active.size();
  for (size_t t = 0; t < n_tok; ++t) {
    if (!st.active[t]) continue;
    const int32_t src = pe->stored[t];
    if (src < 0 || src / S >= (int64_t)E->pages.size() || E->pages[src / S] < 0)
      return fail(c, AKV_EINVAL, "entry %lld lost the key of token %zu", (long long)m.entry, t);
    const int64_t k = st.pos[t] / S;
    if (kind[k] == 0) kind[k] = 1;
    if (src != st.pos[t]) kind[k] = 2;
  }
  // a partly filled tail page is always held (the next append writes into
  // it), even when none of its slots is needed: a fresh empty page
  if (n_slots % S && kind[n_pages - 1] == 0) kind[n_pages - 1] = 3;
  size_t n_fresh = 0;
  for (int8_t k : kind) n_fresh += k >= 2;
  if (n_fresh > c->free_pages.size())
    return fail(c, AKV_ENOPAGES, "prefix fork needs %zu pages, %zu free", n_fresh, c->free_pages.size());

  // plan the new sequence
  HostSeq s;
  s.family = E->family;
  s.layout = ++c->layout_clock;
  s.pages.assign((size_t)n_pages, -1);
  std::vector<int32_t> fresh = peek_pages(c, n_fresh);
  size_t fi = 0;
  for (int64_t k = 0; k < n_pages; ++k) {
    if (kind[k] == 1) s.pages[k] = E->pages[k];
    else if (kind[k] >= 2) s.pages[k] = fresh[fi++];
  }
  std::vector<MoveItem> moves;
  std::vector<int32_t> act;
  for (int64_t k = 0; k < n_pages; ++k)
    if (kind[k] == 1 || kind[k] == 2) act.push_back((int32_t)k);
  std::vector<uint32_t> keep((size_t)((n_slots + 31) / 32), 0u);
  int64_t n_alive = 0;
  for (size_t t = 0; t < n_tok; ++t) {
    if (st.held[t]) {
      const int64_t slot = st.pos[t];
      if (!s.runs.empty() && s.runs.back().slot0 + s.runs.back().len == slot &&
          s.runs.back().log0 + s.runs.back().len == (int64_t)t)
        ++s.runs.back().len;
      else
        s.runs.push_back({slot, (int64_t)t, 1});
    }
    if (!st.active[t]) continue;
    const int64_t slot = st.pos[t];
    keep[slot / 32] |= 1u << (slot % 32);
    ++n_alive;
    if (!s.alive.empty() && s.alive.back().b == slot) s.alive.back().b = slot + 1;
    else s.alive.push_back({slot, slot + 1});
    const int32_t src = pe->stored[t];
    if (kind[slot / S] == 2)
      moves.push_back({E->pages[src / S], src % S, s.pages[slot / S], (int32_t)(slot % S),
                       (int32_t)(slot - src)});
  }
  s.n_logical = (int64_t)n_tok;
  s.n_slots = n_slots;
  s.n_alive = n_alive;
  s.n_active_pages = (int32_t)act.size();
  s.gather_identity = true;
  s.gather_n = 0;
  s.key = history_key(x->idx, req.recs, (size_t)m.n_records);

  // moves are in slot order, so each fresh page's moves are contiguous
  std::vector<MoveBlock> mblocks;
  for (size_t m = 0; m < moves.size(); ++m) {
    if (mblocks.empty() || mblocks.back().dst_page != moves[m].dst_page)
      mblocks.push_back({(int32_t)m, 0, moves[m].dst_page});
    ++mblocks.back().count;
  }
  Blob blob;
  const size_t o_keep = blob.put(keep.data(), keep.size());
  const size_t o_pages = blob.put(s.pages.data(), s.pages.size());
  const size_t o_act = blob.put(act.data(), act.size());
  const size_t o_mv = blob.put(moves.data(), moves.size());
  const size_t o_mb = blob.put(mblocks.data(), mblocks.size());
  rc = grow_fork_scratch(c, blob.b.size() + 16);
  if (rc) return rc;
  rc = upload_large(c, blob, static_cast<char*>(c->d_fork));
  if (rc) return rc;

  // commit
  take_pages(c, n_fresh);
  for (int64_t k = 0; k < n_pages; ++k)
    if (kind[k] == 1) ++c->refcnt[s.pages[k]];
  s.dslot = c->free_dslots.back();
  c->free_dslots.pop_back();
  const SeqArrays& sa = c->sa;
  char* d = static_cast<char*>(c->d_fork);
  CK(copy_rows(c, sa.keep + (int64_t)s.dslot * sa.keep_words, d + o_keep,
               keep.size() * sizeof(uint32_t)));
  CK(copy_rows(c, sa.pages + (int64_t)s.dslot * sa.seq_pages, d + o_pages,
               s.pages.size() * sizeof(int32_t)));
  CK(copy_rows(c, sa.active + (int64_t)s.dslot * sa.seq_pages, d + o_act,
               act.size() * sizeof(int32_t)));
  const int64_t id = c->next_id++;
  c->seqs.emplace(id, std::move(s));
  ++c->epoch;
  x->idx.touch(m.entry, -1);
  *child = id;
  if (!moves.empty()) {
    CK(launch_transplant(c->g, reinterpret_cast<const MoveItem*>(d + o_mv), (int)moves.size(),
                         reinterpret_cast<const MoveBlock*>(d + o_mb), (int)mblocks.size(),
                         c->d_cs, c->cfg.max_slots, c->d_err, c->wait_limit, c->stream));
    ++c->launches;
  }
  return AKV_OK;
}

int akv_prefix_evict(akv_cache* c, akv_prefix_index* x, int32_t want_pages, int32_t* freed_pages,
                     int32_t* n_evicted) {
  if (!c || !x || want_pages < 0) return AKV_EINVAL;
  const std::vector<int64_t> order = x->idx.evict_order();
  const size_t before = c->free_pages.size();
  int32_t ev = 0;
  for (int64_t id : order) {
    if ((int64_t)(c->free_pages.size() - before) >= want_pages) break;
    HostSeq* s = find(c, id);
    if (s) {
      s->frozen = false;
      const int rc = akv_seq_free(c, id);
      if (rc) return rc;
    }
    x->idx.remove(id);
    ++ev;
  }
  if (freed_pages) *freed_pages = (int32_t)(c->free_pages.size() - before);
  if (n_evicted) *n_evicted = ev;
  return AKV_OK;
}

// ---- introspection -------------------------------------------------------------

int akv_seq_info(akv_cache* c, int64_t seq, akv_seq_info_t* info) {
  if (!c || !info) return AKV_EINVAL;
  HostSeq* s = find(c, seq);
  if (!s) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seq);
  info->n_logical = s->n_logical;
  info->n_held = s->n_slots;
  info->n_active = s->n_alive;
  info->next_pos = s->n_slots;
  info->n_pages = (int32_t)s->pages.size();
  info->n_active_pages = s->n_active_pages;
  int32_t own = 0, shared = 0;
  for (int32_t p : s->pages) {
    if (p < 0) continue;
    if (c->refcnt[p] > 1) ++shared; else ++own;
  }
  info->n_owned_pages = own;
  info->n_shared_pages = shared;
  return AKV_OK;
}

int akv_seq_positions(akv_cache* c, int64_t seq, int32_t* pos) {
  if (!c || !pos) return AKV_EINVAL;
  HostSeq* s = find(c, seq);
  if (!s) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seq);
  for (int64_t i = 0; i < s->n_slots; ++i) pos[i] = (int32_t)i;   // slot s is position s
  return AKV_OK;
}

int akv_seq_keep_mask(akv_cache* c, int64_t seq, uint8_t* keep) {
  if (!c || !keep) return AKV_EINVAL;
  HostSeq* s = find(c, seq);
  if (!s) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seq);
  const size_t nw = (size_t)((s->n_slots + 31) / 32);
  std::vector<uint32_t> w(nw);
  if (nw) {
    CK(cudaMemcpyAsync(w.data(), c->sa.keep + (int64_t)s->dslot * c->sa.keep_words,
                       nw * sizeof(uint32_t), cudaMemcpyDeviceToHost, c->stream));
    CK(cudaStreamSynchronize(c->stream));
  }
  for (int64_t i = 0; i < s->n_slots; ++i) keep[i] = (w[i / 32] >> (i % 32)) & 1u;
  return AKV_OK;
}

int akv_seq_logical(akv_cache* c, int64_t seq, int64_t* logical) {
  if (!c || !logical) return AKV_EINVAL;
  HostSeq* s = find(c, seq);
  if (!s) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seq);
  for (const Run& r : s->runs)
    for (int64_t t = 0; t < r.len; ++t) logical[r.slot0 + t] = r.log0 + t;
  return AKV_OK;
}

int akv_seq_gather_map(akv_cache* c, int64_t seq, int32_t* map, int64_t* n) {
  if (!c || !n) return AKV_EINVAL;
  HostSeq* s = find(c, seq);
  if (!s) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seq);
  *n = s->gather_n;
  if (!map || !s->gather_n) return AKV_OK;
  if (s->gather_identity) {
    for (int64_t i = 0; i < s->gather_n; ++i) map[i] = (int32_t)i;
    return AKV_OK;
  }
  CK(cudaMemcpyAsync(map, c->sa.gather + (int64_t)s->dslot * c->sa.max_slots,
                     (size_t)s->gather_n * sizeof(int32_t), cudaMemcpyDeviceToHost, c->stream));
  CK(cudaStreamSynchronize(c->stream));
  return AKV_OK;
}

int akv_seq_page_table(akv_cache* c, int64_t seq, int32_t* pages, int32_t* n_pages,
                       int32_t* active, int32_t* n_active) {
  if (!c) return AKV_EINVAL;
  HostSeq* s = find(c, seq);
  if (!s) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seq);
  if (n_pages) *n_pages = (int32_t)s->pages.size();
  if (n_active) *n_active = s->n_active_pages;
  const int64_t row = (int64_t)s->dslot * c->sa.seq_pages;
  if (pages && !s->pages.empty())
    CK(cudaMemcpyAsync(pages, c->sa.pages + row, s->pages.size() * sizeof(int32_t),
                       cudaMemcpyDeviceToHost, c->stream));
  if (active && s->n_active_pages)
    CK(cudaMemcpyAsync(active, c->sa.active + row, (size_t)s->n_active_pages * sizeof(int32_t),
                       cudaMemcpyDeviceToHost, c->stream));
  CK(cudaStreamSynchronize(c->stream));
  return AKV_OK;
}

int akv_seq_host_pages(akv_cache* c, int64_t seq, int32_t* pages, int32_t* n_pages) {
  if (!c || !n_pages) return AKV_EINVAL;
  HostSeq* s = find(c, seq);
  if (!s) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seq);
  *n_pages = (int32_t)s->pages.size();
  if (pages && !s->pages.empty()) std::memcpy(pages, s->pages.data(), s->pages.size() * sizeof(int32_t));
  return AKV_OK;
}

int akv_history_key(akv_cache* c, int64_t seq, uint64_t key[2]) {
  if (!c || !key) return AKV_EINVAL;
  HostSeq* s = find(c, seq);
  if (!s) return fail(c, AKV_ENOSEQ, "unknown sequence %lld", (long long)seq);
  key[0] = s->key.a;
  key[1] = s->key.b;
  return AKV_OK;
}

int akv_page_refcount(akv_cache* c, int32_t page, int32_t* refcount) {
  if (!c || !refcount || page < 0 || page >= c->cfg.max_pages) return AKV_EINVAL;
  *refcount = c->refcnt[page];
  return AKV_OK;
}

int akv_pool_stats(akv_cache* c, int32_t* free_pages, int32_t* used_pages) {
  if (!c) return AKV_EINVAL;
  if (free_pages) *free_pages = (int32_t)c->free_pages.size();
  if (used_pages) *used_pages = c->cfg.max_pages - (int32_t)c->free_pages.size();
  return AKV_OK;
}

const char* akv_last_error(akv_cache* c) { return c ? c->err.c_str() : "null cache"; }

int akv_sync_errors(akv_cache* c, uint32_t* word) {
  if (!c) return AKV_EINVAL;
  uint32_t w = 0;
  CK(cudaStreamSynchronize(c->stream));
  CK(cudaMemcpy(&w, c->d_err, sizeof(w), cudaMemcpyDeviceToHost));
  CK(cudaMemset(c->d_err, 0, sizeof(w)));
  // a kernel that gave up may have left split counters behind
  if (w) CK(cudaMemset(c->d_counters, 0, (size_t)kMaxItems * c->cfg.hkv * sizeof(int32_t)));
  if (word) *word = w;
  return w ? fail(c, AKV_EDEVICE, "device error word 0x%x", w) : AKV_OK;
}

int akv_set_decode_waves(akv_cache* c, int32_t waves) {
  if (!c || waves < 1 || waves > 64) return AKV_EINVAL;
  c->decode_waves = waves;
  for (auto& pl : c->plans) pl.epoch = ~0ULL;   // re-plan on the next call
  return AKV_OK;
}

int akv_set_decode_sharing(akv_cache* c, int32_t mode) {
  if (!c || mode < 0 || mode > kDecodeMaxMembers) return AKV_EINVAL;
  c->decode_share = mode;
  for (auto& pl : c->plans) pl.epoch = ~0ULL;   // re-plan on the next call
  return AKV_OK;
}

int akv_decode_plan_stats(akv_cache* c, int32_t* items, int32_t* shared_items, int32_t* members) {
  if (!c || !items || !shared_items || !members) return AKV_EINVAL;
  *items = c->last_items;
  *shared_items = c->last_shared;
  *members = c->last_members;
  return AKV_OK;
}

int akv_set_restore_tensor_cores(akv_cache* c, int32_t enable) {
  if (!c || enable < 0 || enable > 2) return AKV_EINVAL;
  c->restore_generic = enable == 0;
  c->restore_pairs = enable == 1;
  return AKV_OK;
}

int akv_kernel_launches(akv_cache* c, uint64_t* count) {
  if (!c || !count) return AKV_EINVAL;
  *count = c->launches;
  return AKV_OK;
}

int akv_set_wait_limit(akv_cache* c, uint32_t polls) {
  if (!c || polls == 0) return AKV_EINVAL;
  c->wait_limit = polls;
  return AKV_OK;
}

}  // extern "C"
