/*
 * akv.h -- C ABI of the active-KV cache library (GB300, sm_103a).
 *
 * The library keeps, for many sequences, a paged K/V cache in which a set of
 * logical tokens can be dropped from attention, the survivors repositioned
 * to dense positions with their keys re-rotated, and decode attention read
 * only the active tokens.  Sources ("Cache Engineering for Agents" paper
 * review; "[Repo Review] AKV" code review):
 *
 *   append      -- paper review, 3.3 Cache Operations, Eq. (3)
 *   drop        -- paper review, 3.3, Eq. (4); AKV review, 1 (Drop)
 *   reposition  -- paper review, 3.3, Eq. (5); AKV review, 5.5 (kernel)
 *   history     -- paper review, 3.4 Cache Operation Sequence, Eq. (6)
 *   copy-on-write of shared pages -- paper review, 4.2.3 Reposition-aware
 *                  Cache Management; AKV review, 5.4 (OccurrenceState)
 *   decode      -- attention over the active KV only; paper review, A.4.1
 *
 * Conventions (all calls):
 *   - Every function returns AKV_OK (0) or a negative AKV_E* code.  On an
 *     error the cache state is unchanged (each call plans on the host, checks
 *     every limit, then commits).  akv_last_error() gives a message.
 *   - "device" pointers are CUDA device memory; "host" pointers are host
 *     memory read (or written) before the call returns.
 *   - All GPU work of a cache is enqueued on the cache's stream (set at
 *     creation, changeable with akv_set_stream) and is asynchronous: no call
 *     on the append/drop/reposition/decode path waits for the GPU.  Device
 *     buffers passed in must stay valid until that work has run.  Calls on
 *     one cache must not run concurrently from several host threads.
 *   - Positions: a sequence's held tokens (everything since its last
 *     reposition, dropped or not) sit in slots 0..n_held-1; the RoPE position
 *     of slot s is s, and the next append lands at n_held.  Drop does not
 *     move anything, so it never lowers the next position (paper review,
 *     Appendix A.1.1, Figure 10: E lands at 3 after D is dropped).
 *   - RoPE is the half-split form (pairs (i, i+D/2), f_i = theta^(-2i/D)).
 */
#ifndef AKV_H
#define AKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AKV_OK 0
#define AKV_EINVAL (-1)    /* invalid argument or configuration */
#define AKV_ERANGE (-2)    /* token range outside [0, n_logical) */
#define AKV_ENOSEQ (-3)    /* unknown or freed sequence id */
#define AKV_ENOPAGES (-4)  /* the page pool has too few free pages */
#define AKV_ECAPACITY (-5) /* a per-sequence or per-call capacity is exceeded */
#define AKV_ECUDA (-6)     /* a CUDA runtime call failed */
#define AKV_EDEVICE (-7)   /* a kernel reported an inconsistency */

#define AKV_DTYPE_BF16 0
#define AKV_DTYPE_FP32 1

/* Device error word bits (akv_sync_errors). */
#define AKV_DERR_PAGE 0x1u     /* a page id outside the pool was met */
#define AKV_DERR_INDEX 0x2u    /* a slot/index outside its array was met */
#define AKV_DERR_WAIT 0x4u     /* a bounded wait gave up (pipeline stalled) */
#define AKV_DERR_COUNT 0x8u    /* a device count disagreed with the host plan */

typedef struct akv_config {
  int32_t layers;      /* logical transformer layers (>= 1) */
  int32_t phys_layers; /* K/V slabs held in the pool; logical layer l uses
                          slab l % phys_layers.  0 means == layers. */
  int32_t hq;          /* query heads (multiple of hkv; hq/hkv <= 16) */
  int32_t hkv;         /* key/value heads */
  int32_t head_dim;    /* 64 or 128 */
  int32_t page_size;   /* tokens per page: 1, 2, 4, 8, 16, 32 or 64 */
  int32_t dtype;       /* AKV_DTYPE_BF16 or AKV_DTYPE_FP32 (pool and inputs) */
  int32_t max_pages;   /* pages in the pool */
  int32_t max_seqs;    /* sequences alive at the same time */
  int32_t max_slots;   /* held tokens per sequence (positions stay below) */
  double rope_theta;   /* RoPE base */
  int32_t rope_dim;    /* rotary dims R: the first R dims of K and q rotate
                          (half-split pairs (i, i+R/2), f_i = theta^(-2i/R)),
                          dims R.. are not rotated (partial RoPE; "[Repo
                          Review] AKV" 5.5).  0 means R = head_dim; else a
                          multiple of 16 in [16, head_dim]. */
} akv_config;

typedef struct akv_cache akv_cache;

typedef struct akv_seq_info_t {
  int64_t n_logical;      /* tokens ever appended (logical indices 0..n-1) */
  int64_t n_held;         /* tokens held since the last reposition */
  int64_t n_active;       /* held tokens not dropped */
  int64_t next_pos;       /* position of the next append (== n_held) */
  int32_t n_pages;        /* pages spanned by the held slots */
  int32_t n_active_pages; /* pages holding at least one active token */
  int32_t n_owned_pages;  /* pages referenced only by this sequence */
  int32_t n_shared_pages; /* pages also referenced by another sequence */
} akv_seq_info_t;

/* Bytes of ONE pool (the K pool and the V pool have the same size):
 * phys_layers * max_pages * hkv * page_size * head_dim * sizeof(dtype).
 * Pool layout: [phys_layer][page][kv_head][slot_in_page][head_dim],
 * so one (page, head) tile is page_size*head_dim contiguous elements.
 * Returns 0 for an invalid configuration. */
size_t akv_pool_bytes(const akv_config* cfg);

/* Creates a cache over caller-owned K and V pools (device, akv_pool_bytes
 * each, 256-byte aligned; contents need not be initialised).  The library
 * allocates its own metadata, RoPE table and workspace on the device and
 * keeps host state; the pools stay the caller's and must outlive the cache.
 * `stream` is a cudaStream_t (NULL = legacy default stream).  Validates the
 * configuration (AKV_EINVAL) and allocations (AKV_ECUDA). */
int akv_cache_create(const akv_config* cfg, void* k_pool, void* v_pool,
                     size_t pool_bytes, void* stream, akv_cache** out);

/* Waits for the cache's stream, then frees what the library allocated. */
int akv_cache_destroy(akv_cache* cache);

/* Later calls enqueue on `stream`.  The caller orders it after the old one. */
int akv_set_stream(akv_cache* cache, void* stream);

/* A new, empty sequence.  AKV_ECAPACITY when max_seqs are alive. */
int akv_seq_create(akv_cache* cache, int64_t* seq);

/* A branch of `parent`: same tokens, positions, drops and history; every
 * page is shared (reference counted).  Pages are copied only when a branch
 * writes into a shared partly filled page (append) -- reposition always
 * writes fresh pages, so a shared page is never written (paper review,
 * 4.2.3: a reposition by one request makes a new version; others keep the
 * old one). */
int akv_seq_fork(akv_cache* cache, int64_t parent, int64_t* child);

/* Releases the sequence's page references (pages are reused at zero). */
int akv_seq_free(akv_cache* cache, int64_t seq);

/* Eq. (3), append: for each i < n_seqs, appends n_tokens[i] tokens to
 * seqs[i] at positions next_pos.. (K is rotated to its position here).
 *   k_raw, v : device, [layers][T][hkv][head_dim] in the pool dtype, with
 *              T = sum(n_tokens) and the tokens of seqs[0], seqs[1], ... in
 *              order; k_raw is the key BEFORE RoPE.  Logical layer l is
 *              written to slab l % phys_layers (aliased layers: the last
 *              logical layer of a slab wins).
 *   token_ids: host, [T] or NULL; only enters the history key.
 * Keys are computed in fp32 from the table cos/sin(p f_i) (fp64 -> fp32)
 * and stored rounded to nearest even.  A sequence may appear once per call.
 * Errors: AKV_ENOSEQ, AKV_ECAPACITY (max_slots), AKV_ENOPAGES. */
int akv_append(akv_cache* cache, const int64_t* seqs, const int32_t* n_tokens,
               int32_t n_seqs, const void* k_raw, const void* v,
               const int32_t* token_ids);

/* Eq. (4), drop: removes logical indices in the half-open ranges
 * ranges[2i]..ranges[2i+1] (host, n_ranges pairs) from all later attention.
 * Overlapping, repeated or already dropped indices are allowed (P is a
 * set).  Nothing moves: positions and next_pos are unchanged.  A full page
 * left with no active token loses this sequence's reference.
 * Errors: AKV_ERANGE (begin < 0, end < begin or end > n_logical). */
int akv_drop(akv_cache* cache, int64_t seq, const int64_t* ranges,
             int32_t n_ranges);

/* Eq. (5), reposition, batched over n_seqs sequences (host ids): the r
 * active tokens of each move, in logical order, to slots/positions 0..r-1;
 * each key is re-rotated by K' = R(q) R(p)^-1 K = R(q - p) K in fp32 (a key
 * whose position does not change is copied bit for bit) and V is copied;
 * next_pos becomes r.  The gather map is the exclusive prefix sum of the
 * keep mask.  Leading pages whose every slot stays put keep their page id
 * (and stay shared); all other survivors are written to fresh pages, and
 * the old pages lose this sequence's reference.  A sequence with nothing
 * dropped since it was last dense only gets a history record.
 * Errors: AKV_ENOSEQ, AKV_EINVAL (repeated id), AKV_ENOPAGES. */
int akv_reposition(akv_cache* cache, const int64_t* seqs, int32_t n_seqs);

/* Decode attention of one layer over the active tokens only:
 *   q   : device, [n_seqs][hq][head_dim] pool dtype, BEFORE RoPE; it is
 *         rotated to next_pos - 1 (the position of the last appended token).
 *   seqs: host, [n_seqs] sequence ids.
 *   out : device, [n_seqs][hq][head_dim] fp32,
 *         out = softmax(q' K^T / sqrt(D)) V over active tokens; query head h
 *         reads KV head h / (hq/hkv).  A sequence with no active token gets 0.
 * Split-KV over pages with a library-owned partial workspace, then a merge.
 * Errors: AKV_ENOSEQ, AKV_EINVAL (layer), AKV_ECAPACITY (work items). */
int akv_decode_attention(akv_cache* cache, int32_t layer, const void* q,
                         const int64_t* seqs, int32_t n_seqs, float* out);

/* Sliding-window attention for one layer ("[Repo Review] AKV" 5.5): with
 * window W > 0, akv_decode_attention on this layer reads, for a query at
 * position p, only the active tokens whose position lies in (p - W, p] --
 * a window of positions, so position gaps left by a drop hold fewer keys.
 * W = 0 (the default) is full attention.  Errors: AKV_EINVAL. */
int akv_set_layer_window(akv_cache* cache, int32_t layer, int32_t window);

/* ---- segment-batch restore attention ------------------------------------
 * Paper review 4.2.2 / 4.2.3 / Appendix A.1.1: after eviction, a sequence is
 * rebuilt by one forward over its whole operation program, in which each
 * token's query must see exactly the keys it saw originally -- keys dropped
 * later included -- at the positions of that time (temporary rotated
 * versions).  The program is an array of operations applied to an empty
 * sequence: */
#define AKV_OP_APPEND 0   /* append `count` tokens (the next rows of q/k/v) */
#define AKV_OP_DROP 1     /* drop `count` logical ranges ranges[2i]..ranges[2i+1] */
#define AKV_OP_REPOS 2    /* reposition */
typedef struct akv_op {
  int32_t kind;
  int32_t count;
  const int64_t* ranges;  /* host; AKV_OP_DROP only */
} akv_op;

/* Attention outputs of one layer for every appended token of the program,
 * in one batched pass: out[t] = softmax(q_t' K^T / sqrt(D)) V over the keys
 * active when token t was appended (t included), keys and query rotated to
 * the positions of that moment.  Sliding window: the layer's
 * akv_set_layer_window setting.
 *   q    : device [n_tokens][hq][D] pool dtype, before RoPE
 *   k_raw, v : device [n_tokens][hkv][D] pool dtype, K before RoPE
 *   out  : device [n_tokens][hq][D] fp32
 * No sequence is read or changed: rebuild the cache state by replaying the
 * program with akv_append / akv_drop / akv_reposition.  The library keeps a
 * scratch buffer for the temporary key versions and the program's device
 * descriptor and grows it (cudaMalloc, which waits for the device) when a
 * program needs more.  bf16 pools with D 64 or 128 run a tensor-core kernel
 * (see akv_set_restore_tensor_cores).
 * Errors: AKV_EINVAL (program appends a different number of tokens than
 * n_tokens, bad op), AKV_ERANGE (drop range), AKV_ECAPACITY (a position
 * reaches max_slots). */
int akv_restore_attention(akv_cache* cache, const akv_op* ops, int32_t n_ops, int32_t layer,
                          const void* q, const void* k_raw, const void* v,
                          int32_t n_tokens, float* out);

/* The same for selected tokens only: out rows of tokens[0..n_sel) (host
 * int32, increasing, each < n_tokens) are written, every other row is left
 * as it is; q, k_raw and v still cover all n_tokens (every token's key
 * versions are formed, since a selected query may read any earlier key).
 * n_sel == 0 does nothing.  Used with akv_restore_plan_recovery to recompute
 * only what is missing.  Errors: those of akv_restore_attention, and
 * AKV_EINVAL for a token list that is not increasing or out of range. */
int akv_restore_attention_tokens(akv_cache* cache, const akv_op* ops, int32_t n_ops,
                                 int32_t layer, const void* q, const void* k_raw, const void* v,
                                 int32_t n_tokens, const int32_t* tokens, int32_t n_sel,
                                 float* out);

/* Recovery plan of a restore ([Repo Review] AKV, 5.4: the dependencies of
 * KV that later queries read but that is missing are closed backwards into
 * the query ranges to recompute, resident ranges are kept; paper review
 * 4.2.2 / A.1.1: a token's query reads the keys active when it was
 * appended).  For the program ops[0..n_ops) of n_tokens appended tokens,
 * with missing[t] != 0 for tokens whose KV is not resident and need[t] != 0
 * for tokens whose KV the next step reads (need NULL: the tokens active at
 * the end of the program), writes to tokens_out[0..*n_out), increasing, the
 * least set of tokens that holds every needed missing token and, with each
 * token in it, every missing token its query read (the tokens appended
 * before it and not dropped by then).  Resident tokens are never in it.
 *   missing, need : host uint8 [n_tokens]
 *   tokens_out    : host int32, room for n_tokens
 * Host only: no cache, no GPU work.  Errors: AKV_EINVAL (null pointer, bad
 * op, the program appends a different number of tokens), AKV_ERANGE (drop
 * range outside the tokens appended so far). */
int akv_restore_plan_recovery(const akv_op* ops, int32_t n_ops, int32_t n_tokens,
                              const uint8_t* missing, const uint8_t* need,
                              int32_t* tokens_out, int32_t* n_out);

/* ---- decode attention that allocates nothing (no counterpart in the paper) ----
 *
 * For callers that cannot allocate device memory: applications that reserve
 * all of their GPU memory once at start-up and forbid cudaMalloc/cudaFree
 * while serving (those calls synchronise the device, can fail mid-request
 * and fragment memory already planned), for example a plugin running inside
 * another runtime's memory pool.  Such a caller cannot create an akv_cache,
 * so this call takes only its own pointers and computes the same decode
 * attention as akv_decode_attention() over metadata in the same layout:
 *
 *   k_slab, v_slab : device, one layer's slab [max_pages][hkv][page_size][D]
 *   page_table     : device int32 [n_seqs][row_stride], pool page per slot page
 *   active_pages   : device int32 [n_seqs][row_stride], ascending slot-page
 *                    indices that hold an active token (first n_active_pages)
 *   keep_bits      : device uint32 [n_seqs][keep_stride], bit s = slot s active
 *   n_active_pages : host int32 [n_seqs]
 *   n_held         : host int32 [n_seqs]; the query is rotated to n_held - 1
 *   q, out         : device [n_seqs][hq][D] (pool dtype) / fp32
 *
 * The split-KV partial sums live in one file-scope device array of
 * AKV_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU loading this library
 * holds until the process exits; the call calls no cudaMalloc, cudaFree or
 * other allocating routine.  Its first call on each device (with that device
 * current) looks up the array's device address with cudaGetSymbolAddress;
 * make that first call before any stream capture.  All calls share the
 * array and it keeps the last call's contents (nothing in it needs to start
 * at zero: a call writes every partial it reads), so calls that overlap on
 * the GPU -- on different streams, or from several host threads -- race and
 * must be serialised by the caller.  Splits are sized so the partials fit.
 * It covers the plain method: full-width RoPE and full attention (no
 * rope_dim, no window).
 * Errors: AKV_ECAPACITY when n_seqs > AKV_NOALLOC_MAX_SEQS; AKV_EINVAL for
 * a bad shape or pointer, or a sequence with active pages but no held token;
 * AKV_ECUDA when a launch fails. */
#define AKV_NOALLOC_SCRATCH_BYTES (8 << 20)
#define AKV_NOALLOC_MAX_SEQS 256
int akv_decode_attention_noalloc(
    const void* k_slab, const void* v_slab, int32_t max_pages, int32_t hq,
    int32_t hkv, int32_t head_dim, int32_t page_size, int32_t dtype,
    double rope_theta, const int32_t* page_table, const int32_t* active_pages,
    const uint32_t* keep_bits, int32_t row_stride, int32_t keep_stride,
    const int32_t* n_active_pages, const int32_t* n_held, const void* q,
    float* out, int32_t n_seqs, void* stream);

/* ---- introspection (tests, tools): these wait for the cache's stream ---- */

int akv_seq_info(akv_cache* cache, int64_t seq, akv_seq_info_t* info);

/* Host outputs of n_held entries: position of each held slot, whether it is
 * active (device keep mask), and its logical index. */
int akv_seq_positions(akv_cache* cache, int64_t seq, int32_t* pos);
int akv_seq_keep_mask(akv_cache* cache, int64_t seq, uint8_t* keep);
int akv_seq_logical(akv_cache* cache, int64_t seq, int64_t* logical);

/* Gather map of the sequence's last reposition: map[j] = old slot of the
 * token now in slot j (host, n entries; *n is set even if map is NULL). */
int akv_seq_gather_map(akv_cache* cache, int64_t seq, int32_t* map, int64_t* n);

/* Device page table (pool page id per slot page, -1 once released) and the
 * device active page list (slot-page indices, ascending).  Host outputs; a
 * NULL output is skipped; counts are always set. */
int akv_seq_page_table(akv_cache* cache, int64_t seq, int32_t* pages,
                       int32_t* n_pages, int32_t* active, int32_t* n_active);

/* The planner's page table of a sequence: pool page per slot page, -1 once
 * released (host output of n_pages entries; *n_pages is always set).  It is
 * host state and needs no wait: the device table holds the same once the
 * cache's stream reaches the calls made so far. */
int akv_seq_host_pages(akv_cache* cache, int64_t seq, int32_t* pages, int32_t* n_pages);

/* 128-bit key of the sequence's operation history (Eq. 6): equal histories
 * give equal keys; different ones differ (with overwhelming probability).
 * One record per appended token (its id, or none), one per non-empty drop
 * (its sorted, merged ranges), one per reposition. */
int akv_history_key(akv_cache* cache, int64_t seq, uint64_t key[2]);

/* Reference count of a pool page (0 = free) and pool occupancy. */
int akv_page_refcount(akv_cache* cache, int32_t page, int32_t* refcount);
int akv_pool_stats(akv_cache* cache, int32_t* free_pages, int32_t* used_pages);

/* Message of the last error on this cache (static storage of the cache). */
const char* akv_last_error(akv_cache* cache);

/* Waits for the stream and returns (then clears) the device error word
 * (AKV_DERR_* bits).  Returns AKV_EDEVICE when it was non-zero. */
int akv_sync_errors(akv_cache* cache, uint32_t* word);

/* Tuning: the tensor-core decode plans `waves` quarters of the blocks that
 * fit the GPU at once (default 1: a quarter, which leaves room for the next
 * call's blocks to start early; 1..64). */
int akv_set_decode_waves(akv_cache* cache, int32_t waves);

/* Tuning: in a decode call, rows that hold the same pool pages at the same
 * slot pages with the same keep bits (branches forked from one prefix:
 * "Cache Engineering for Agents" paper review, 3.2, copy-on-write branches)
 * may read those pages once for all of them, as one tensor-core work item
 * whose query columns are the rows' GQA groups side by side (runs of at
 * least 4 such pages).  mode 0 = every row reads its own pages; 1 (default)
 * = automatic (up to 32 / (hq/hkv) rows per item); 2..16 = at most that many
 * rows per item.  The split boundaries differ between plans, and the
 * softmax weights are rounded to bf16 against each split's running maximum,
 * so results differ by bf16 roundings of those weights.  Applies to
 * full-attention layers of the tensor-core decode; AKV_EINVAL for other
 * values. */
int akv_set_decode_sharing(akv_cache* cache, int32_t mode);

/* The plan of the most recent decode call: work items, items read for
 * several rows, and the rows of those items (host values; no GPU work). */
int akv_decode_plan_stats(akv_cache* cache, int32_t* items, int32_t* shared_items,
                          int32_t* members);

/* Kernel choice for akv_restore_attention: 1 (default) = tensor-core
 * kernel where it applies (bf16 pool, D 64 or 128) with two query tiles
 * per CTA, 2 = the tensor-core kernel with one query tile per CTA, 0 = the
 * CUDA-core kernel for every shape.  All compute the same attention. */
int akv_set_restore_tensor_cores(akv_cache* cache, int32_t enable);

/* Number of kernels this cache has launched since creation. */
int akv_kernel_launches(akv_cache* cache, uint64_t* count);

/* Iteration limit of every bounded device wait (default 1<<22 polls). */
int akv_set_wait_limit(akv_cache* cache, uint32_t polls);

/* ==== History-keyed prefix sharing and drop-aware eviction ====
 *
 * Paper review, Appendix A.1.2 (Reposition Scheme) and 4.2.2 / 4.2.3;
 * repo review 5.4 (context records TOKEN / DELTA / REPOSITION, plan of
 * occurrence materialisation) and 5.6 (drop-aware eviction candidates).
 *
 * A program (akv_op list plus one token id per appended token) is expanded
 * into context records: TOKEN(id) per appended token, DELTA(ranges) per
 * non-empty drop (sorted, merged), REPOSITION per reposition.  An index
 * holds published entries: snapshots of sequences, each with its records.
 * A request matches an entry on a prefix of n records when the records are
 * equal up to n and every token active after those n records still has its
 * key stored in the entry (its slot held and its page holding an active
 * token).  The match is EXACT when each such key is stored at the position
 * the request gives it, RETRIGGER when some keys have to be rotated.  The
 * longest exact prefix is taken unless a retrigger prefix is strictly
 * longer; ties between entries go to the lowest entry id (for retrigger: the
 * fewest rotated keys first).  The search stops at the first differing
 * record: an operation cannot be skipped to line up final positions
 * (paper review, Figure 11). */
#define AKV_MATCH_NONE 0
#define AKV_MATCH_EXACT 1
#define AKV_MATCH_RETRIGGER 2

typedef struct akv_prefix_index akv_prefix_index;

typedef struct akv_prefix_match_t {
  int32_t kind;        /* AKV_MATCH_* */
  int32_t n_records;   /* records of the request covered */
  int64_t entry;       /* entry id, -1 for none */
  int32_t n_tokens;    /* appended tokens covered */
  int32_t n_rotated;   /* keys whose stored position differs (retrigger) */
  int32_t op_index;    /* the covered prefix is ops[0..op_index) plus ... */
  int32_t op_tokens;   /* ... the first op_tokens tokens of ops[op_index]
                        * (0 when the prefix ends at an op boundary) */
} akv_prefix_match_t;

/* Host-only index (no GPU work); page_size must equal the cache's.  The
 * index and its entries belong to the caller; one index serves one cache. */
int akv_prefix_index_create(int32_t page_size, akv_prefix_index** index);
int akv_prefix_index_destroy(akv_prefix_index* index);
const char* akv_prefix_last_error(akv_prefix_index* index);

/* Inserts a program as entry `entry` (>= 0, unused).  use_time orders
 * eviction (older first); < 0 takes the index's own clock.
 * Errors: AKV_EINVAL (bad program, id taken), AKV_ERANGE (drop range). */
int akv_prefix_insert(akv_prefix_index* index, int64_t entry, const akv_op* ops,
                      int32_t n_ops, const int32_t* token_ids, int32_t n_tokens,
                      int64_t use_time);
int akv_prefix_remove(akv_prefix_index* index, int64_t entry);
int akv_prefix_touch(akv_prefix_index* index, int64_t entry, int64_t use_time);

/* Best match of a request program (host only). */
int akv_prefix_match(akv_prefix_index* index, const akv_op* ops, int32_t n_ops,
                     const int32_t* token_ids, int32_t n_tokens, akv_prefix_match_t* out);

/* Drop-aware eviction order of all entries: first the entries that another
 * entry extends with a DELTA record dropping a token active at the entry's
 * end (their KV is proven unneeded on that path), then leaves, then the
 * remaining ancestors; oldest use first within each class, then lower id.
 * Writes *n ids (AKV_ECAPACITY when capacity < *n). */
int akv_prefix_evict_order(akv_prefix_index* index, int64_t* entries, int32_t capacity,
                           int32_t* n);

/* Publishes sequence `seq` as an entry: the program must be the sequence's
 * own history (checked against its history key, which must have been built
 * with token ids).  The entry is a snapshot (a fork sharing all pages; it
 * counts against max_seqs); its id is returned in *entry.  A program equal
 * to an existing entry's returns that entry (its use time refreshed).
 * Errors: AKV_EINVAL (program is not the history), AKV_ECAPACITY. */
int akv_prefix_publish(akv_cache* cache, akv_prefix_index* index, int64_t seq,
                       const akv_op* ops, int32_t n_ops, const int32_t* token_ids,
                       int32_t n_tokens, int64_t* entry);

/* Matches the request and materialises the covered prefix as a new
 * sequence (*child; -1 with kind NONE): the request's slots, positions,
 * keep mask and history; each needed key comes from the entry's stored key,
 * rotated by R(p_request - p_stored) in fp32 and rounded once (copied when
 * the positions agree), V copied.  A page whose needed slots all keep their
 * slot is shared with the entry (reference count), the others are fresh.
 * The caller continues the program from (op_index, op_tokens).
 * Errors: AKV_ENOSEQ (entry's snapshot gone), AKV_ENOPAGES, AKV_ECAPACITY. */
int akv_prefix_fork(akv_cache* cache, akv_prefix_index* index, const akv_op* ops,
                    int32_t n_ops, const int32_t* token_ids, int32_t n_tokens,
                    akv_prefix_match_t* match, int64_t* child);

/* Frees entries in drop-aware eviction order until at least want_pages
 * pool pages returned to the free list (or no entry is left): each evicted
 * entry's snapshot is freed (pages still used by other sequences or
 * entries stay) and the entry leaves the index. */
int akv_prefix_evict(akv_cache* cache, akv_prefix_index* index, int32_t want_pages,
                     int32_t* freed_pages, int32_t* n_evicted);

#ifdef __cplusplus
}
#endif

#endif /* AKV_H */
