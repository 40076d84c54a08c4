// Decode attention over the active KV on the tensor cores (bf16 pools).
//
// One block per (split of a sequence's active page list, KV head).  A
// producer warp streams the 16-token tiles of the split's pages into a ring
// of shared-memory stages with TMA (cp.async.bulk.tensor, 128-byte swizzle),
// completing one mbarrier per stage; four consumer warps take tiles in turn:
//
//   S^T[16 tok x 8 heads] = K[16 tok x D] . Q^T[D x 8 heads]   (mma m16n8k16)
//   online softmax per head column (keep bits mask dropped slots)
//   O^T[D x 8 heads]     += V^T[D x 16 tok] . P^T[16 tok x 8 heads]
//
// Tokens sit on the MMA's M dimension and the GQA group (padded to 8) on N,
// so one tile is 2*D/16 MMAs for the whole group.  P^T's operand layout is
// the transpose of S^T's accumulator layout; movmatrix transposes it in
// registers.  K fragments come from ldmatrix, V^T fragments from
// ldmatrix.trans, both conflict-free on the swizzled tiles.
//
// Every mbarrier wait is bounded: on expiry the block sets AKV_DERR_WAIT in
// the error word, drains its own copies (again bounded) and returns.
//
// Sources: "Cache Engineering for Agents" paper review, 3.3 and A.4.1
// (attention reads only the active KV); the split-KV online softmax is the
// standard flash-decoding recurrence.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "akv.h"
#include "akv_internal.h"

namespace akv {
namespace {

constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kStages = 8;
// Tile i goes to stage i % kStages and consumer warp i % kConsumers.  With
// kStages a multiple of kConsumers every stage always belongs to the same
// warp, which consumes its fills in order; the parity waits then never look
// at a barrier two phases behind (a parity wait cannot tell phase k-1 from
// phase k+1).
static_assert(kStages % kConsumers == 0, "each stage must have a single consumer warp");
constexpr int kTile = 16;   // tokens per MMA tile
constexpr int kMaxTiles = kDecodeMaxTiles;   // tiles of one split (prefetched)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(a, parity)) return true;
  return false;
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of (row, 16-byte chunk) inside a 16-row tile stored as D/64
// boxes of 16 x 128 bytes with the 128-byte swizzle (chunk ^= row % 8).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)((chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// Which split of the call the blocks use (DecodeArgs::items_w): decided by
// the first block of the call to get here, from whether every block of the
// previous decode call had finished its work by then; the others read that
// decision.  Only this call's blocks write its word (the word of call c is
// reused by call c + 8, which cannot start before every block of call c has
// passed this point and signalled its dependents).  1: the whole-wave split.
__device__ __forceinline__ uint32_t choose_split(const DecodeArgs& a) {
  const uint32_t id = a.call_id & 0x1fffffffu;
  uint32_t* word = a.mode_words + (a.call_id % kDecodeModeWords);
  uint32_t v = *reinterpret_cast<volatile uint32_t*>(word);
  if ((v >> 3) != id) {
    const uint32_t done = *reinterpret_cast<volatile uint32_t*>(a.done_word);
    const uint32_t want = (id << 3) | (done + 1 == a.call_id ? 1u : 0u);
    const uint32_t prev = atomicCAS(word, v, want);
    v = prev == v ? want : prev;                // else another block of this call chose
  }
  return v & 7u;
}

// A block of the call has done its work: count it (one atomic add; a loop
// of compare-and-swap on one word serialises the call's blocks); the last
// one resets the count for the call that reuses the word and publishes the
// call as finished.  Read by the next call's choice only, so a count that
// goes astray (a block that stopped on an error) costs a plan choice,
// never a result.
__device__ __forceinline__ void count_exit(const DecodeArgs& a) {
  uint32_t* cnt = a.exit_words + (a.call_id % kDecodeExitWords);
  if (atomicAdd(cnt, 1u) + 1u == gridDim.x * gridDim.y) {
    atomicExch(cnt, 0u);
    atomicMax(a.done_word, a.call_id);
  }
}

// A member (query row) must name memory this call owns.
__device__ __forceinline__ bool member_ok(const DecodeMember& m, const DecodeArgs& a) {
  return m.row >= 0 && m.row < a.n_rows && m.row < a.counter_rows && m.n_splits >= 1 &&
         m.item0 >= 0 && m.item0 + m.n_splits <= a.part_cap && m.part >= m.item0 &&
         m.part < m.item0 + m.n_splits && m.n_tiles >= 0;
}

// SHARE: the plan has items whose pages several rows hold (same pages, same
// keep bits).  Such an item reads its range once for all of them: its query
// columns are the members' GQA groups side by side, nb blocks of 8 columns,
// and warp w computes column block w % nb on every (4/nb)-th tile.  A member
// holds a leading part of the range (n_tiles tiles); its columns mask the
// tiles after it.  Without SHARE the kernel is the one-row form (nb = 1).
template <int D, bool SHARE>
__global__ void __launch_bounds__(kThreads) k_decode_mma(const __grid_constant__ DecodeArgs a) {
  constexpr int KS = D / 16;                    // k-steps of Q K^T, m-tiles of V^T P^T
  constexpr int TILE_BYTES = kTile * D * 2;     // one K (or V) tile
  constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // The stage ring also holds, before the tile loop, the rotated query
  // [8 nb][D] and, after it, the consumer warps' partials [4][8][D+2].
  float* s_q = reinterpret_cast<float*>(smem);
  float* s_merge = reinterpret_cast<float*>(smem);
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages];
  __shared__ int s_row[kMaxTiles];              // TMA row of each tile, -1 = unusable
  __shared__ uint16_t s_bits[kMaxTiles];        // keep bits of each tile's 16 slots
  __shared__ DecodeMember s_mem[SHARE ? kDecodeMaxMembers : 1];
  __shared__ int s_lastm[SHARE ? kDecodeMaxMembers : 1];

  // the split this call uses (one of two when the planner made a whole-wave
  // split too), chosen before the next call may start
  const DecodeItem* items = a.items;
  int n_items = a.n_items;
  if (a.n_items_w > 0 && a.call_id > 0) {
    __shared__ uint32_t s_split;
    if (threadIdx.x == 0) s_split = choose_split(a);
    __syncthreads();
    if (s_split == 1) {
      items = a.items_w;
      n_items = a.n_items_w;
    }
  }
  // the next decode call may be scheduled now: its blocks start as this
  // grid's blocks retire and wait (griddepcontrol.wait) before writing
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // grid (KV head, item): the blocks of an item go out together, in the
  // plan's order (longest items first)
  if ((int)blockIdx.y >= n_items) {             // the grid is sized for the larger split
    if (threadIdx.x == 0 && a.call_id > 0) count_exit(a);
    return;
  }
  const DecodeItem it = items[blockIdx.y];
  const int kvh = blockIdx.x;
  const Geom& g = a.g;
  const int G = g.hq / g.hkv;
  const int tpp = g.s / kTile;                  // tiles per page
  const int t0 = it.p0 * tpp;
  int n = it.p1 * tpp - t0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // column blocks and members (rows) of this item
  const int nb = SHARE ? it.nb : 1;
  const int n_mem = SHARE && it.n_mem > 0 ? it.n_mem : 1;
  // the work item must describe memory this call owns (uniform per block)
  bool bad = it.dslot < 0 || it.dslot >= a.max_seqs || it.p0 < 0 || it.p1 < it.p0 ||
             it.p1 > a.sa.seq_pages;
  // the one-row form keeps its member in registers (no start-up barrier)
  const DecodeMember me{it.row, it.pos_q, it.item0, it.n_splits, it.part, kMaxTiles};
  auto member = [&](int m) -> const DecodeMember& { return SHARE ? s_mem[m] : me; };
  if constexpr (SHARE) {
    bad |= !(nb == 1 || nb == 2 || nb == 4) || n_mem > kDecodeMaxMembers ||
           n_mem * G > 8 * nb ||
           (it.n_mem > 0 && (it.mem0 < 0 || it.mem0 + it.n_mem > a.n_members));
    if (!bad && tid < n_mem) {
      const DecodeMember m = it.n_mem > 0 ? a.members[it.mem0 + tid] : me;
      bad = !member_ok(m, a);
      s_mem[tid] = m;
    }
    if (__syncthreads_or(bad)) {
      if (tid == 0) atomicOr(a.err, AKV_DERR_INDEX);
      return;
    }
  } else {
    if (bad || !member_ok(me, a)) {
      if (tid == 0) atomicOr(a.err, AKV_DERR_INDEX);
      return;
    }
  }
  if (n > kMaxTiles) {                          // the planner never makes such a split
    if (tid == 0) atomicOr(a.err, AKV_DERR_INDEX);
    n = kMaxTiles;
  }
  const int64_t slab_rows = (int64_t)g.max_pages * g.hkv * g.s;

  if (tid == 0) {
    // a stage is released by the nb warps (one per column block) that read it
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&s_empty[s]), nb);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // tile coordinates and keep bits of the whole split, read once
  {
    const int32_t* active = a.sa.active + (int64_t)it.dslot * a.sa.seq_pages;
    const int32_t* pages = a.sa.pages + (int64_t)it.dslot * a.sa.seq_pages;
    const uint32_t* keep = a.sa.keep + (int64_t)it.dslot * a.sa.keep_words;
    for (int i = tid; i < n; i += kThreads) {
      const int ti = t0 + i, sub = ti % tpp;
      const int kidx = active[ti / tpp];
      const int page = (kidx >= 0 && kidx < a.sa.seq_pages) ? pages[kidx] : -1;
      int row = -1;
      uint32_t bits = 0;
      if (page >= 0 && page < g.max_pages &&
          ((int64_t)page * g.hkv + kvh) * g.s + (sub + 1) * kTile <= slab_rows) {
        row = (page * g.hkv + kvh) * g.s + sub * kTile;
        const int slot0 = (kidx * tpp + sub) * kTile;
        bits = (keep[slot0 >> 5] >> (slot0 & 31)) & 0xffffu;
        // sliding window: slots below win_lo are not read
        if (it.win_lo > slot0) bits &= it.win_lo - slot0 >= kTile ? 0u : (0xffffu << (it.win_lo - slot0));
      } else {
        atomicOr(a.err, AKV_DERR_PAGE);
      }
      s_row[i] = row;
      s_bits[i] = (uint16_t)bits;
    }
  }
  // rotated, scaled queries: column c is head c % G of member c / G
  // (columns past the members stay zero); the first R dims rotate in pairs
  // (d, d + R/2), dims R.. are only scaled
  {
    const int R = g.rope, RH = R / 2;
    for (int i = tid; i < 8 * nb * D; i += kThreads) {
      const int c = i / D, d = i % D, m = c / G, gq = c % G;
      const DecodeMember& mm = member(m < n_mem ? m : 0);
      const bool have_q = m < n_mem && mm.pos_q >= 0 && mm.pos_q < a.sa.max_slots;
      const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) +
                               ((int64_t)mm.row * g.hq + (int64_t)kvh * G + gq) * D;
      if (d < RH) {
        float x = 0.f, y = 0.f;
        if (have_q) {
          const float qx = __bfloat162float(q[d]), qy = __bfloat162float(q[d + RH]);
          const float2 t = a.cs[(int64_t)mm.pos_q * RH + d];
          x = fmaf(qx, t.x, -qy * t.y) * a.scale_log2;
          y = fmaf(qx, t.y, qy * t.x) * a.scale_log2;
        }
        s_q[c * D + d] = x;
        s_q[c * D + d + RH] = y;
      } else if (d >= R) {
        s_q[c * D + d] = have_q ? __bfloat162float(q[d]) * a.scale_log2 : 0.f;
      }
    }
  }
  __syncthreads();
  // Q^T fragments (B operand of the score MMA) of the warp's column block:
  // lane holds column lane/4, dims 2*(lane%4)+{0,1} and +8 of each k-step
  const int nblk = warp % nb, phase = warp / nb, n_phase = kConsumers / nb;
  uint32_t qf[KS][2];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int h = (warp < kConsumers ? nblk * 8 : 0) + (lane >> 2), c = ks * 16 + (lane & 3) * 2;
    qf[ks][0] = pack_bf16(s_q[h * D + c], s_q[h * D + c + 1]);
    qf[ks][1] = pack_bf16(s_q[h * D + c + 8], s_q[h * D + c + 9]);
  }
  // s_q is dead: order these generic-proxy accesses before the TMA writes
  // (async proxy) that reuse the ring
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();

  const int slab = (a.layer >= 0 ? a.layer : 0) % g.phys_layers;
  float o[KS][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // columns 2*(lane%4), +1

  if (warp == kConsumers) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int s = i % kStages;
        if (i >= kStages &&
            !mbar_wait(smem_u32(&s_empty[s]), ((i / kStages) - 1) & 1, a.wait_limit)) {
          atomicOr(a.err, AKV_DERR_WAIT);
          break;
        }
        const uint32_t full = smem_u32(&s_full[s]);
        const int row = s_row[i];
        if (row < 0) {
          mbar_arrive(full);
        } else {
          mbar_expect_tx(full, STAGE_BYTES);
          // one copy per tensor: both 64-column atoms of the 16 rows, laid
          // out [atom][row][64] (the same bytes as one 64 x 16 box per atom)
          const uint32_t dk = smem_u32(smem + s * STAGE_BYTES);
          tma_load_4d(dk, &a.tm_k4, 0, row, 0, slab, full);
          tma_load_4d(dk + TILE_BYTES, &a.tm_v4, 0, row, 0, slab, full);
        }
        ++issued;
      }
      // this block's copies must have landed before the ring is reused or
      // the block exits (immediate unless a consumer gave up early)
      // (a fixed, generous limit: copies in flight land in microseconds, and
      // a small user limit must not let the block exit before they do)
      for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
        if (!mbar_wait(smem_u32(&s_full[i % kStages]), (i / kStages) & 1, kDrainPolls))
          atomicOr(a.err, AKV_DERR_WAIT);
    }
  } else {
    // ---------------- consumers ----------------
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    // ldmatrix row addresses (tile-relative)
    const int k_row = (lane & 7) + ((lane >> 3) & 1) * 8;   // K: (r0-7,c0),(r8-15,c0),(r0-7,c1),(r8-15,c1)
    const int k_cb = lane >> 4;
    const int v_row = (lane & 7) + (lane >> 4) * 8;         // V: (t0-7,d0),(t0-7,d1),(t8-15,d0),(t8-15,d1)
    const int v_cb = (lane >> 3) & 1;
    const int r0 = lane >> 2;
    const int tk = (lane & 3) * 2;

    // tiles of the lane's two columns (shared items: the member's part)
    int end0 = n, end1 = n;
    if (SHARE) {
      const int c0 = nblk * 8 + (lane & 3) * 2;
      if (c0 / G < n_mem) end0 = member(c0 / G).n_tiles;
      if ((c0 + 1) / G < n_mem) end1 = member((c0 + 1) / G).n_tiles;
    }
    for (int i = phase; i < n; i += n_phase) {
      const int s = i % kStages;
      // every lane waits (acquire for its own reads); the outcome is made
      // warp-uniform before the warp-synchronous MMAs
      const bool got = mbar_wait(smem_u32(&s_full[s]), (i / kStages) & 1, a.wait_limit);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) atomicOr(a.err, AKV_DERR_WAIT);
        break;
      }
      if (s_row[i] >= 0) {
        const uint32_t kb = smem_u32(smem + s * STAGE_BYTES);
        const uint32_t vb = kb + TILE_BYTES;
        const uint32_t bits = s_bits[i];
        // S^T = K Q^T
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        if (SHARE) {
          // two accumulation chains (even / odd k-steps) halve the dependent
          // MMA latency of a tile, which bounds items whose warps read every
          // tile; the one-row form waits on memory instead
          float sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ks = 0; ks < KS; ks += 2) {
            uint32_t af[4], ag[4];
            ldsm_x4(kb + swz(k_row, ks * 2 + k_cb), af);
            ldsm_x4(kb + swz(k_row, ks * 2 + 2 + k_cb), ag);
            mma16816(sc, af, qf[ks][0], qf[ks][1]);
            mma16816(sd, ag, qf[ks + 1][0], qf[ks + 1][1]);
          }
          sc[0] += sd[0]; sc[1] += sd[1]; sc[2] += sd[2]; sc[3] += sd[3];
        } else {
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            uint32_t af[4];
            ldsm_x4(kb + swz(k_row, ks * 2 + k_cb), af);
            mma16816(sc, af, qf[ks][0], qf[ks][1]);
          }
        }
        if (!((bits >> r0) & 1u)) sc[0] = sc[1] = -INFINITY;
        if (!((bits >> (r0 + 8)) & 1u)) sc[2] = sc[3] = -INFINITY;
        if (SHARE) {
          if (i >= end0) sc[0] = sc[2] = -INFINITY;
          if (i >= end1) sc[1] = sc[3] = -INFINITY;
        }
        // online softmax over the tile (columns = heads)
        float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float a0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0);
        const float a1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
        const float p0 = n0 == -INFINITY ? 0.f : exp2f(sc[0] - n0);
        const float p1 = n1 == -INFINITY ? 0.f : exp2f(sc[1] - n1);
        const float p2 = n0 == -INFINITY ? 0.f : exp2f(sc[2] - n0);
        const float p3 = n1 == -INFINITY ? 0.f : exp2f(sc[3] - n1);
        m0 = n0;
        m1 = n1;
        l0 = fmaf(l0, a0, p0 + p2);
        l1 = fmaf(l1, a1, p1 + p3);
        if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            o[mt][0] *= a0; o[mt][1] *= a1; o[mt][2] *= a0; o[mt][3] *= a1;
          }
        }
        // P^T as the B operand: transpose the two 8x8 halves of P in registers
        const uint32_t pb0 = movm_t(pack_bf16(p0, p1));
        const uint32_t pb1 = movm_t(pack_bf16(p2, p3));
        // O^T += V^T P^T.  A slot that is not active may hold any bit pattern
        // (never-written pool memory included); its P is 0, but 0 * NaN is
        // NaN, so its V is zeroed too.  Lane holds tokens 2*(lane%4)+{0,1}
        // in fragment registers 0-1 and the same +8 in registers 2-3.
        const bool full_tile = bits == 0xffffu;
        const uint32_t mlo = ((bits >> tk) & 1u ? 0x0000ffffu : 0u) |
                             ((bits >> (tk + 1)) & 1u ? 0xffff0000u : 0u);
        const uint32_t mhi = ((bits >> (tk + 8)) & 1u ? 0x0000ffffu : 0u) |
                             ((bits >> (tk + 9)) & 1u ? 0xffff0000u : 0u);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          uint32_t vf[4];
          ldsm_x4_t(vb + swz(v_row, mt * 2 + v_cb), vf);
          if (!full_tile) {
            vf[0] &= mlo; vf[1] &= mlo; vf[2] &= mhi; vf[3] &= mhi;
          }
          mma16816(o[mt], vf, pb0, pb1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s_empty[s]));
    }
    // row sums: reduce over the 8 lanes that share a head column
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
  }
  __syncthreads();   // every tile consumed and every copy landed: the ring is free
  if (warp < kConsumers) {
    // per-warp partial -> shared: [warp][column][D] then m, l at [D], [D+1]
    float* wm = s_merge + warp * 8 * (D + 2);
    const int h0 = (lane & 3) * 2;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const int d = mt * 16 + (lane >> 2);
      wm[h0 * (D + 2) + d] = o[mt][0];
      wm[(h0 + 1) * (D + 2) + d] = o[mt][1];
      wm[h0 * (D + 2) + d + 8] = o[mt][2];
      wm[(h0 + 1) * (D + 2) + d + 8] = o[mt][3];
    }
    if (lane < 4) {
      wm[h0 * (D + 2) + D] = m0;
      wm[h0 * (D + 2) + D + 1] = l0;
      wm[(h0 + 1) * (D + 2) + D] = m1;
      wm[(h0 + 1) * (D + 2) + D + 1] = l1;
    }
  }
  __syncthreads();

  // The previous decode call (launched before this one may start, see the
  // launcher) writes the same kind of partials, counters and outputs; this
  // block's first global write waits until that grid has finished.  Nothing
  // above reads memory a decode call writes.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // merge the consumer warps of each column (the n_phase warps of its
  // block): the member's output (its only split) or this split's partial
  bool multi = false;
  for (int m = 0; m < n_mem; ++m) multi |= member(m).n_splits > 1;
  for (int i = tid; i < n_mem * G * D; i += kThreads) {
    const int c = i / D, d = i % D, hc = c & 7, cb = c >> 3;
    float M = -INFINITY;
    for (int ph = 0; ph < n_phase; ++ph)
      M = fmaxf(M, s_merge[((ph * nb + cb) * 8 + hc) * (D + 2) + D]);
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
      for (int ph = 0; ph < n_phase; ++ph) {
        const float* wm = s_merge + ((ph * nb + cb) * 8 + hc) * (D + 2);
        const float f = exp2f(wm[D] - M);
        L = fmaf(wm[D + 1], f, L);
        A = fmaf(wm[d], f, A);
      }
    }
    const DecodeMember& mm = member(c / G);
    const int gq = c % G, hq = kvh * G + gq;
    if (mm.n_splits == 1) {
      a.out[((int64_t)mm.row * g.hq + hq) * D + d] = L > 0.f ? A / L : 0.f;
    } else {
      const int64_t pi = ((int64_t)mm.part * g.hkv + kvh) * G + gq;
      a.part_acc[pi * D + d] = A;
      if (d == 0) a.part_ml[pi] = make_float2(M, L);
    }
  }
  if (tid == 0 && a.call_id > 0) count_exit(a);
  if (!multi) return;

  // for each member, the last split of (row, kv head) to finish merges all
  // of that row's splits
  __threadfence();
  __syncthreads();
  if (tid < n_mem) {
    const DecodeMember& mm = member(tid);
    int last = 0;
    if (mm.n_splits > 1)
      last = atomicAdd(&a.counters[mm.row * g.hkv + kvh], 1) == mm.n_splits - 1;
    s_lastm[tid] = last;
  }
  __syncthreads();
  int n_fin = 0;
  for (int m = 0; m < n_mem; ++m) n_fin += s_lastm[m];
  if (n_fin == 0) return;
  __threadfence();
  // k-th member whose merge falls to this block
  auto fin_member = [&](int k) {
    int m = 0;
    for (; m < n_mem; ++m)
      if (s_lastm[m] && k-- == 0) break;
    return m;
  };
  // pass 1, one warp per (row, head): maximum and sum over the row's splits,
  // the splits spread over the lanes (the stage ring is free: (M, L) there)
  float2* s_ml = reinterpret_cast<float2*>(s_merge);
  for (int p = warp; p < n_fin * G; p += kThreads / 32) {
    const DecodeMember& mm = member(fin_member(p / G));
    const int gq = p % G;
    const float2* ml = a.part_ml + ((int64_t)mm.item0 * g.hkv + kvh) * G + gq;
    const int64_t stride = (int64_t)g.hkv * G;
    // lane c holds split c (and c + 32, ... past 32 splits)
    const float2 v0 = lane < mm.n_splits ? __ldcg(ml + lane * stride) : make_float2(-INFINITY, 0.f);
    float M = v0.x;
    for (int c = lane + 32; c < mm.n_splits; c += 32) M = fmaxf(M, __ldcg(ml + c * stride).x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    if (M != -INFINITY) {
      if (lane < mm.n_splits) L = v0.y * exp2f(v0.x - M);
      for (int c = lane + 32; c < mm.n_splits; c += 32) {
        const float2 v = __ldcg(ml + c * stride);
        L = fmaf(v.y, exp2f(v.x - M), L);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane == 0) s_ml[p] = make_float2(M, L);
  }
  if (tid < n_mem && s_lastm[tid])
    a.counters[member(tid).row * g.hkv + kvh] = 0;   // ready for the next call
  __syncthreads();
  // pass 2: the weighted sum of the partials, four dims per output; a thread
  // takes up to kPer outputs at once so that their loads are in flight
  // together
  constexpr int kPer = SHARE ? 8 : 1;
  const int n_out = n_fin * G * (D / 4);
  const bool vec_out = (reinterpret_cast<uintptr_t>(a.out) & 15) == 0;
  for (int e0 = tid; e0 < n_out; e0 += kThreads * kPer) {
    float4 A[kPer];
    int64_t base[kPer];
    int nsp[kPer];
    float Mx[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = e0 + k * kThreads;
      A[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      nsp[k] = 0;
      base[k] = 0;
      Mx[k] = -INFINITY;
      if (e < n_out) {
        const int p = e / (D / 4);
        const DecodeMember& mm = member(fin_member(p / G));
        base[k] = ((int64_t)mm.item0 * g.hkv + kvh) * G + p % G;
        Mx[k] = s_ml[p].x;
        nsp[k] = Mx[k] == -INFINITY ? 0 : mm.n_splits;
      }
    }
    int most = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) most = max(most, nsp[k]);
    const int64_t stride = (int64_t)g.hkv * G;
    for (int c = 0; c < most; ++c) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        if (c < nsp[k]) {
          const int e = e0 + k * kThreads, d = (e % (D / 4)) * 4;
          const int64_t pi = base[k] + c * stride;
          const float f = exp2f(__ldcg(&a.part_ml[pi]).x - Mx[k]);
          const float4 v = __ldcg(reinterpret_cast<const float4*>(a.part_acc + pi * D + d));
          A[k].x = fmaf(v.x, f, A[k].x);
          A[k].y = fmaf(v.y, f, A[k].y);
          A[k].z = fmaf(v.z, f, A[k].z);
          A[k].w = fmaf(v.w, f, A[k].w);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = e0 + k * kThreads;
      if (e >= n_out) continue;
      const int p = e / (D / 4), d = (e % (D / 4)) * 4;
      const DecodeMember& mm = member(fin_member(p / G));
      const int gq = p % G;
      const float L = s_ml[p].y;
      const float4 o = L > 0.f ? make_float4(A[k].x / L, A[k].y / L, A[k].z / L, A[k].w / L)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
      float* dst = a.out + ((int64_t)mm.row * g.hq + kvh * G + gq) * D + d;
      if (vec_out) {
        *reinterpret_cast<float4*>(dst) = o;
      } else {                                  // the caller's output need only be 4-byte aligned
        dst[0] = o.x; dst[1] = o.y; dst[2] = o.z; dst[3] = o.w;
      }
    }
  }
}

template <int D>
constexpr size_t mma_smem() {
  static_assert((size_t)kConsumers * 8 * (D + 2) * 4 <= (size_t)kStages * 2 * kTile * D * 2,
                "the partials must fit in the stage ring");
  static_assert((size_t)4 * 8 * D * 4 <= (size_t)kStages * 2 * kTile * D * 2,
                "the queries of four column blocks must fit in the stage ring");
  return 1024 + (size_t)kStages * 2 * kTile * D * 2;
}

template <int D>
void set_smem_attr() {
  static bool done = false;
  if (!done) {
    cudaFuncSetAttribute(k_decode_mma<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)mma_smem<D>());
    cudaFuncSetAttribute(k_decode_mma<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)mma_smem<D>());
    done = true;
  }
}

}  // namespace

bool decode_mma_supported(const Geom& g) {
  return g.dtype == AKV_DTYPE_BF16 && g.s % kTile == 0 && (g.hq / g.hkv) <= 8 &&
         (g.d == 64 || g.d == 128);
}

// Tensor maps over the K and V pools: 3-D (D, rows of one slab, slab),
// boxes of 64 x 16 elements with the 128-byte swizzle.
bool make_pool_tensor_maps(const Geom& g, CUtensorMap* tk, CUtensorMap* tv) {
  if (!decode_mma_supported(g)) return false;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&encode),
                                       12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !encode)
    return false;
  const uint64_t rows = (uint64_t)g.max_pages * g.hkv * g.s;
  const cuuint64_t dims[3] = {(cuuint64_t)g.d, rows, (cuuint64_t)g.phys_layers};
  const cuuint64_t strides[2] = {(cuuint64_t)g.d * 2, (cuuint64_t)(rows * g.d * 2)};
  const cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  for (int i = 0; i < 2; ++i) {
    CUresult r = encode(i == 0 ? tk : tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        i == 0 ? g.k : g.v, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
  }
  return true;
}

// Launched with programmatic stream serialisation when the previous work on
// the stream is a decode call (a.pdl; such a call signals launch_dependents
// at its start): this grid's blocks may start while that grid's last blocks
// still run, so its start-up (work item, tile list, query) hides behind the
// other's tail.  A decode call reads nothing a decode call writes before its
// griddepcontrol.wait.  After anything else (append, drop, reposition, the
// kernel that copies this call's new plan in) the launch is plain stream
// order.
cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t st) {
  const dim3 grid(a.g.hkv, a.n_items_w > a.n_items ? a.n_items_w : a.n_items);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  if (a.g.d == 64) {
    set_smem_attr<64>();
    cfg.dynamicSmemBytes = mma_smem<64>();
    return a.shared ? cudaLaunchKernelEx(&cfg, k_decode_mma<64, true>, a)
                    : cudaLaunchKernelEx(&cfg, k_decode_mma<64, false>, a);
  }
  set_smem_attr<128>();
  cfg.dynamicSmemBytes = mma_smem<128>();
  return a.shared ? cudaLaunchKernelEx(&cfg, k_decode_mma<128, true>, a)
                  : cudaLaunchKernelEx(&cfg, k_decode_mma<128, false>, a);
}

// The same pools as 4-D maps (64 columns, rows, D / 64 atoms, slab): the atom
// dimension steps 128 bytes inside a row, so one box (64 x 16 x D/64) lands
// a 16-row tile's atoms one after the other, each in the 128-byte swizzled
// layout of a 64 x 16 box.
bool make_pool_tensor_maps4(const Geom& g, CUtensorMap* tk, CUtensorMap* tv) {
  if (!decode_mma_supported(g)) return false;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&encode),
                                       12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !encode)
    return false;
  const uint64_t rows = (uint64_t)g.max_pages * g.hkv * g.s;
  const cuuint64_t dims[4] = {64, rows, (cuuint64_t)(g.d / 64), (cuuint64_t)g.phys_layers};
  const cuuint64_t strides[3] = {(cuuint64_t)g.d * 2, 128, (cuuint64_t)(rows * g.d * 2)};
  const cuuint32_t box[4] = {64, (cuuint32_t)kTile, (cuuint32_t)(g.d / 64), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  for (int i = 0; i < 2; ++i) {
    CUresult r = encode(i == 0 ? tk : tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                        i == 0 ? g.k : g.v, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
  }
  return true;
}

int decode_mma_blocks_per_sm(int d) {
  int n = 0;
  if (d == 64) {
    set_smem_attr<64>();
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_decode_mma<64, false>, kThreads, mma_smem<64>());
  } else {
    set_smem_attr<128>();
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_decode_mma<128, false>, kThreads, mma_smem<128>());
  }
  return n;
}

}  // namespace akv
