// Internal interface between the host planner (akv_host.cpp) and the CUDA
// kernels (akv_kernels.cu, akv_decode.cu).  Not part of the public ABI.
//
// Every operation is planned on the host (which owns page allocation and the
// per-sequence counts), packed into one small descriptor blob, copied to the
// device once, and executed by one to three kernels on the cache's stream.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace akv {

// Pool geometry.  Layout: [phys_layer][page][kv_head][slot_in_page][head_dim].
struct Geom {
  void* k;
  void* v;
  int64_t layer_stride;  // elements between physical layers
  int64_t page_stride;   // elements between pages (hkv * S * D)
  int64_t head_stride;   // elements between heads (S * D)
  int32_t layers, phys_layers, hq, hkv, d, s, dtype, max_pages;
  int32_t rope;          // rotary dims R (first R dims rotate, the rest are copied)
  // low parts of the RoPE table, (cos - RN(cos), sin - RN(sin)) in fp32,
  // [max_slots][R/2]: the stored-key kernels use them for rotations that
  // nearly cancel (exact rounding to bf16)
  const float2* cs_lo;
};

// Per-sequence device arrays, one fixed-size row per device sequence slot
// ("dslot"); row i of `keep` starts at i * keep_words, and so on.
struct SeqArrays {
  uint32_t* keep;       // keep bit per held slot
  int32_t* pages;       // pool page id per slot page (-1 once released)
  int32_t* active;      // slot-page indices holding an active token, ascending
  int32_t* gather;      // last reposition's gather map (new slot -> old slot)
  int32_t* old_pages;   // snapshot of replaced page ids during a reposition
  int32_t keep_words;   // ceil(max_slots / 32)
  int32_t seq_pages;    // ceil(max_slots / S)
  int32_t max_slots;
};

// ---- append (Eq. 3) -------------------------------------------------------
struct AppendItem {
  int32_t dslot;
  int32_t slot0;     // first new slot (== old n_held == position)
  int32_t n;         // tokens appended
  int32_t tok0;      // row of the first token in k_raw / v
  int32_t k0;        // first slot page touched
  int32_t nk;        // slot pages touched (page ids in ids[ids_off..])
  int32_t ids_off;
  int32_t act0;      // first active-list entry written
  int32_t n_act;     // active-list entries written (from act[act_off..])
  int32_t act_off;
};
struct AppendBlock { int32_t item, t0; };   // block -> (item, first token)
constexpr int kAppendTokens = 16;           // tokens per append block

// ---- copy-on-write page copy ----------------------------------------------
struct PagePair { int32_t src, dst; };

// ---- drop (Eq. 4) -----------------------------------------------------------
struct DropItem {
  int32_t dslot;
  int32_t n_slots;      // held slots
  int32_t n_pages;      // slot pages
  int32_t range_off;    // slot ranges (pairs) in ranges[range_off..]
  int32_t n_ranges;
  int32_t expect_active;  // host's count of active pages afterwards
};

// ---- reposition (Eq. 5) -------------------------------------------------------
struct ReposItem {
  int32_t dslot;
  int32_t old_slots;    // held slots before
  int32_t old_pages;    // slot pages before
  int32_t r;            // survivors (host count)
  int32_t n_kept;       // leading pages that keep their id
  int32_t new_pages;    // ceil(r / S)
  int32_t fresh_off;    // fresh page ids in ids[fresh_off..], new_pages - n_kept
  int32_t block0;       // first gather block of this item (prefix sum)
};

// ---- decode ---------------------------------------------------------------------
struct DecodeItem {
  int32_t dslot;
  int32_t row;          // row of q / out
  int32_t p0, p1;       // active-list range [p0, p1) of this split
  int32_t pos_q;        // query position (next_pos - 1), -1 if no token held
  int32_t n_splits;     // splits of this row
  int32_t item0;        // first item of this row
  int32_t win_lo;       // sliding window: slots below are not read (0 = none)
  // tensor-core path: this item's partial slot; the row's partials are
  // [item0, item0 + n_splits)
  int32_t part;
  // pages shared by several rows: members [mem0, mem0 + n_mem) of
  // DecodeArgs::members read the range once (n_mem 0: the item's own row);
  // nb = blocks of 8 head columns (1, 2 or 4)
  int32_t mem0, n_mem, nb;
};
// one row of a shared item: the query's row and position, the row's partial
// slots [item0, item0 + n_splits), this item's slot among them, and the
// item's leading tiles that hold the row's pages (its columns see no others)
struct DecodeMember { int32_t row, pos_q, item0, n_splits, part, n_tiles; };
constexpr int kDecodeMaxMembers = 16;

// shared-prefix decode on the tensor cores (page size 16): one CTA per
// (item, KV head) computes up to 128 query rows (members x GQA heads) over a
// range of the first member's active pages and writes every member's
// partial; members are DecodeArgs::members, n_tiles = the member's pages
struct ShareItem {
  int32_t dslot;        // sequence whose active list is walked
  int32_t p0, p1;       // its active-list range (pages)
  int32_t mem0, n_mem;
};

struct DecodeArgs {
  CUtensorMap tm_k;     // TMA maps over the pools (tensor-core paths): (D, rows, slab),
  CUtensorMap tm_v;     // 64 x 16 boxes
  CUtensorMap tm_k4;    // the same pools as (64, rows, D / 64, slab): both 64-column
  CUtensorMap tm_v4;    // atoms of a 16-row tile in one copy (one-row kernel)
  Geom g;
  SeqArrays sa;
  const DecodeItem* items;
  int32_t n_items;
  int32_t layer;        // logical layer (slab = layer % phys_layers)
  const void* q;
  float* out;
  float* part_acc;      // [item][hkv][group][D]
  float2* part_ml;      // [item][hkv][group] (max, sum) in log2 units
  const float2* cs;     // RoPE table [max_slots][R/2] (cos, sin)
  float scale_log2;     // log2(e) / sqrt(D)
  uint32_t* err;
  uint32_t wait_limit;
  int32_t use_mma;      // tensor-core kernel (bf16 pools, page % 16 == 0, group <= 8)
  int32_t* counters;    // [row][hkv] finished splits (tensor-core path; reset by the last)
  int32_t n_rows;       // rows of q / out in this call
  int32_t max_seqs;     // device rows of the per-sequence arrays
  int32_t counter_rows; // rows of `counters`
  int32_t part_cap;     // partial slots of part_acc / part_ml
  const DecodeMember* members;   // shared items (tensor-core path)
  int32_t n_members;
  int32_t shared;       // the plan has shared items
  const ShareItem* share_items;   // tensor-core shared-prefix items (before the others)
  int32_t n_share_items;
  // Plan choice made on the device (tensor-core one-row kernel): items_w is
  // the same call split for a whole wave of blocks (0: no second plan).  The
  // call's first block takes it iff the previous decode call had finished
  // (nothing of it left to overlap with: a call on its own), else the
  // call keeps `items` (a quarter wave: room for its neighbours' blocks).
  const DecodeItem* items_w;
  int32_t n_items_w;
  uint32_t call_id;             // > 0, one per call of this cache
  uint32_t* mode_words;         // [8] (call_id << 3 | plan) once a call has chosen
  uint32_t* exit_words;         // [1024] blocks of call c exited, at c % 1024
  uint32_t* done_word;          // last call whose blocks have all exited
  bool pdl;                     // host only: launch with programmatic stream serialisation
};
constexpr int kDecodeModeWords = 8;
constexpr int kDecodeExitWords = 1024;
constexpr int kDecodeMaxTiles = 512;   // 16-token tiles in one split of the tensor-core path
// bound of the waits that let a kernel's own copies / MMAs land before it
// exits after a failed wait (independent of the user's wait limit)
constexpr uint32_t kDrainPolls = 1u << 22;

// ---- segment-batch restore attention -------------------------------------------
struct RestoreKey { int32_t tok, pos, birth, death; };      // one era key row
struct RestoreQuery { int32_t tok, pos, time, era_off, key_end; };
// tensor-core path: consecutive query tokens of one era, their key range
struct RestoreTile { int32_t era_off, tok0, n_tok, key_lo, key_hi; };
struct RestoreArgs {
  CUtensorMap tm_k, tm_v;     // tensor-core path: era K / V, (D, hkv, n_keys), 64 x 1 x 64 boxes
  Geom g;
  const RestoreKey* keys;
  int32_t n_keys;
  const RestoreQuery* queries;
  int32_t n_queries;
  const void* q;        // [T][hq][D] pool dtype, pre-RoPE
  const void* k_raw;    // [T][hkv][D] pool dtype, pre-RoPE
  const void* v;        // [T][hkv][D]
  int32_t n_tokens;
  void* k_era;          // [n_keys][hkv][D] temporary key versions
  void* v_era;
  float* out;           // [T][hq][D]
  const float2* cs;
  int32_t max_pos;
  float scale_log2;
  int32_t window;
  uint32_t* err;
  const RestoreTile* tiles;   // tensor-core path only
  int32_t n_tiles;
  // two-tile tensor-core kernel: (tile A, tile B or -1) per CTA, consecutive
  // tiles of one era; 0 pairs: one tile per CTA
  const int2* pairs;
  int32_t n_pairs;
  int32_t use_mma;
  uint32_t wait_limit;        // bounded waits of the tensor-core path
};
cudaError_t launch_restore(const RestoreArgs& a, cudaStream_t st);
bool restore_mma_supported(const Geom& g);
int restore_tile_tokens(const Geom& g);       // query tokens per tensor-core block
// tensor maps over the era buffers of the tensor-core path (false: unavailable)
bool make_restore_tensor_maps(const Geom& g, const void* k_era, const void* v_era, int64_t n_keys,
                              CUtensorMap* tk, CUtensorMap* tv);

// ---- prefix fork: stored keys of a snapshot moved into fresh pages ----------
struct MoveItem { int32_t src_page, src_off, dst_page, dst_off, delta; };
struct MoveBlock { int32_t first, count, dst_page; };   // the moves into one fresh page
cudaError_t launch_transplant(const Geom& g, const MoveItem* moves, int n_moves,
                              const MoveBlock* blocks, int n_blocks, const float2* cs, int max_pos,
                              uint32_t* err, uint32_t wait_limit, cudaStream_t st);

// Launchers (akv_kernels.cu / akv_decode.cu).  All enqueue on `st`.
struct AppendLimits { int32_t n_items, n_ids, n_act, max_seqs; };
cudaError_t launch_append(const Geom& g, const SeqArrays& sa, const AppendItem* items,
                          const AppendBlock* blocks, int n_blocks, const int32_t* ids,
                          const int32_t* act, const void* k_raw, const void* v,
                          int64_t total_tokens, const float2* cs, uint32_t* err,
                          AppendLimits lim, cudaStream_t st);
cudaError_t launch_copy_pages(const Geom& g, const PagePair* pairs, int n_pairs,
                              uint32_t* err, cudaStream_t st);
// n bytes from src to dst by a kernel (src may be pinned host memory, read
// over the host link); any alignment, n may be 0.
cudaError_t launch_copy_bytes(void* dst, const void* src, size_t n, cudaStream_t st);
// dst[0..n) = v by a kernel.
cudaError_t launch_fill_u32(uint32_t* dst, uint32_t v, size_t n, cudaStream_t st);
cudaError_t launch_drop(const Geom& g, const SeqArrays& sa, const DropItem* items,
                        int n_items, const int32_t* ranges, uint32_t* err, cudaStream_t st);
cudaError_t launch_compact(const Geom& g, const SeqArrays& sa, const ReposItem* items,
                           int n_items, const int32_t* ids, uint32_t* err, cudaStream_t st);
cudaError_t launch_gather(const Geom& g, const SeqArrays& sa, const ReposItem* items,
                          int n_items, int n_blocks, const float2* cs, uint32_t* err,
                          uint32_t wait_limit, cudaStream_t st);
cudaError_t launch_decode(const DecodeArgs& a, bool need_combine, int n_rows,
                          const int32_t* row_item0, const int32_t* row_splits,
                          cudaStream_t st);
// Tensor-core decode (akv_decode_mma.cu).
bool decode_mma_supported(const Geom& g);
bool make_pool_tensor_maps(const Geom& g, CUtensorMap* tk, CUtensorMap* tv);
bool make_pool_tensor_maps4(const Geom& g, CUtensorMap* tk, CUtensorMap* tv);
cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t st);
int decode_mma_blocks_per_sm(int head_dim);
// Shared-prefix decode (akv_decode_share.cu): bf16 pools, page size 16,
// head dim 64 / 128, GQA group <= 8.
bool decode_share_supported(const Geom& g);
cudaError_t launch_decode_share(const DecodeArgs& a, cudaStream_t st);

}  // namespace akv
