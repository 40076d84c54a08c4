// Shared-prefix decode attention on the tensor cores (tcgen05).
//
// Branches forked from one prefix hold the same pool pages ("Cache
// Engineering for Agents" paper review, 3.2: a fork shares its parent's pages
// copy-on-write), so in one decode call their queries can read those pages
// once.  A CTA takes up to 128 query rows -- the GQA heads of up to 128 / G
// rows of the call, its "members" -- and one KV head, and walks a range of
// the first member's active pages in tiles of 64 tokens (4 pages):
//
//   S = Q K^T      M=128, N=64, K=D    -> one of two S buffers in TMEM
//   softmax        per row: the keep bits of the tile's slots and the
//                  member's own run of pages (a member holds a leading part
//                  of the range); online max / sum, P (bf16) over S in TMEM
//   O += P V       M=128, N=D, K=64, A = P from TMEM
//
// The item's page ids and keep bits (at most kMaxItemPages pages) are read
// into shared memory first.  A load warp copies each tile's four pages of K
// and V with TMA (a page past the range is read at an out-of-range row,
// which TMA fills with zeros) and an MMA warp issues the MMAs, each from one
// thread: the SM's TMA unit takes its requests one after another, so copies
// and MMAs issued by one thread would make a tile wait for both; eight
// softmax warps, two per TMEM lane quarter, split the tile's tokens and O's
// columns in halves.  Every wait is bounded.  The epilogue writes each
// member's partial (unnormalised O, reference max, sum) and counts it in the
// row's split counter; the one-row decode kernel of the same call, launched
// after this grid, merges all partials of a row.
//
// Pool memory of a slot that no row sees may hold any bits (a prefix fork's
// empty tail page is held but never written, and appends may later fill the
// rest of it): its score is masked, and its V row is zeroed in shared memory
// before the PV MMA, since P = 0 does not cancel a NaN there.  The planner
// also keeps each sequence's partly filled tail page out of shared items.
#include <cuda.h>
#include <cuda_bf16.h>

#include "akv.h"
#include "akv_internal.h"
#include "akv_tc.cuh"

namespace akv {
namespace {

constexpr int kBM = 128;                    // query rows per CTA
constexpr int kBN = 64;                     // tokens per tile
constexpr int kPageRows = 16;               // the page size this kernel reads
constexpr int kTilePages = kBN / kPageRows;
constexpr int kSoftmaxWarps = 8;
constexpr int kMmaWarp = kSoftmaxWarps;      // issues the MMAs (one thread)
constexpr int kLoadWarp = kSoftmaxWarps + 1; // issues the tile copies (one thread)
constexpr int kThreads = 32 * (kSoftmaxWarps + 2);
constexpr int kHalf = kBN / 2;              // tokens per softmax warp and tile
constexpr int kCols = 256;                  // TMEM: two S buffers (2 x 64) and O (<= 128)
constexpr int kMaxItemPages = 256;          // pages of one item (the planner takes 32..256)
static_assert(2 * kBN + 128 <= kCols, "S buffers and O must fit the TMEM allocation");

// Bounded wait for the phase of `parity` to complete, polling try_wait
// (which suspends the thread in hardware for a while) without a sleep in
// between: an item has few tiles, and each hand-off sits on its critical path.
__device__ __forceinline__ bool wait_phase(uint32_t mbar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 "selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok) : "r"(mbar), "r"(parity) : "memory");
    if (ok) return true;
  }
  return false;
}

template <int D>
constexpr size_t share_smem() {
  return 1024 /* alignment slack */ + (size_t)kBM * D * 2 + 4 * (size_t)kBN * D * 2;
}

__device__ __forceinline__ bool share_member_ok(const DecodeMember& m, const DecodeArgs& a) {
  return m.row >= 0 && m.row < a.n_rows && m.row < a.counter_rows && m.n_splits >= 1 &&
         m.item0 >= 0 && m.item0 + m.n_splits <= a.part_cap && m.part >= m.item0 &&
         m.part < m.item0 + m.n_splits && m.n_tiles >= 0;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
k_decode_share_tc(const __grid_constant__ DecodeArgs a) {
  constexpr uint32_t KV_BYTES = kBN * D * 2;    // one tile of K (or V)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm;                             // kBM x D (K-major)
  uint8_t* sK = sQ + kBM * D * 2;               // [2] kBN x D, 64-element atoms
  uint8_t* sV = sK + 2 * kBN * D * 2;           // [2] same layout, read MN-major
  __shared__ DecodeMember s_mem[kBM];
  // row maxima of the two halves per tile parity, then the two row sums
  __shared__ float s_mx[6 * kBM];
  __shared__ int s_prow[kMaxItemPages];         // TMA row of each page (past the pool: zeros)
  __shared__ uint32_t s_pbits[kMaxItemPages];   // keep bits of each page's 16 slots
  __shared__ int s_abort_v;
  // S[2] O[2] K[2] V[2] P[2], then X[4 quarters][2]: row-max exchange of a pair
  __shared__ __align__(8) uint64_t mbar[18];
  __shared__ uint32_t tslot;
  volatile int* s_abort = &s_abort_v;

  // the next kernel on the stream (this call's one-row decode) may start
  // now; it waits for this grid before its first write
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const ShareItem it = a.share_items[blockIdx.x];
  const int kvh = blockIdx.y;
  const Geom& g = a.g;
  const int G = g.hq / g.hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool control = warp == kMmaWarp, loader = warp == kLoadWarp;
  // the item and its members must describe memory this call owns
  bool bad = it.dslot < 0 || it.dslot >= a.max_seqs || it.p0 < 0 || it.p1 < it.p0 ||
             it.p1 > a.sa.seq_pages || it.p1 - it.p0 > kMaxItemPages || it.n_mem < 1 ||
             it.n_mem * G > kBM || it.mem0 < 0 || it.mem0 + it.n_mem > a.n_members;
  if (!bad && tid < it.n_mem) {
    const DecodeMember m = a.members[it.mem0 + tid];
    bad = !share_member_ok(m, a);
    s_mem[tid] = m;
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicOr(a.err, AKV_DERR_INDEX);
    return;
  }
  const int n_used = it.n_mem * G;              // rows = member * G + head
  const int n_pages = it.p1 - it.p0;
  // the pages' TMA rows and keep bits, read once
  {
    const int oob_row = (int)((int64_t)g.max_pages * g.hkv * kPageRows);
    const int32_t* active = a.sa.active + (int64_t)it.dslot * a.sa.seq_pages;
    const int32_t* pages = a.sa.pages + (int64_t)it.dslot * a.sa.seq_pages;
    const uint32_t* keep = a.sa.keep + (int64_t)it.dslot * a.sa.keep_words;
    for (int i = tid; i < kMaxItemPages; i += kThreads) {
      int row = oob_row;
      uint32_t bits = 0;
      if (i < n_pages) {
        const int kidx = active[it.p0 + i];
        const int page = (kidx >= 0 && kidx < a.sa.seq_pages) ? pages[kidx] : -1;
        if (page >= 0 && page < g.max_pages) {
          row = (page * g.hkv + kvh) * kPageRows;
          const int slot0 = kidx * kPageRows;
          bits = (keep[slot0 >> 5] >> (slot0 & 31)) & 0xffffu;
        } else {
          atomicOr(a.err, AKV_DERR_PAGE);
        }
      }
      s_prow[i] = row;
      s_pbits[i] = bits;
    }
  }

  const uint32_t mbS0 = smem_u32(mbar), mbO0 = smem_u32(mbar + 2), mbK0 = smem_u32(mbar + 4),
                 mbV0 = smem_u32(mbar + 6), mbP0 = smem_u32(mbar + 8), mbX0 = smem_u32(mbar + 10);
  if (control) {
    if (lane == 0) {
      for (int i = 0; i < 18; ++i) {
        // P: one arrival per softmax warp; X: one per warp of the pair
        const uint32_t cnt = (i == 8 || i == 9) ? kSoftmaxWarps : (i >= 10 ? 2 : 1);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(mbar + i)), "r"(cnt) : "memory");
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      *s_abort = 0;
    }
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(&tslot)), "r"(kCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  const int n_kt = (n_pages + kTilePages - 1) / kTilePages;
  const int slab = (a.layer >= 0 ? a.layer : 0) % g.phys_layers;
  int k_pend[2] = {-1, -1}, v_pend[2] = {-1, -1};   // load warp: copies in flight
  // load lane 0: the four pages of tile kt into K (or V) buffer kt & 1
  // K: [atom][64 rows][128 B] (the S MMA spans the tile's four pages), one
  // 64 x 16 box per (atom, page); V: [page][atom][16 rows][128 B] (a PV
  // MMA step is one page), one 64 x 16 x D/64 box per page over the pool
  // seen as (64 columns, rows, atoms, slab)
  auto tma_tile = [&](int kt, bool is_k) {
    const int b = kt & 1;
    const uint32_t bar = (is_k ? mbK0 : mbV0) + 8 * b;
    uint8_t* dst = (is_k ? sK : sV) + b * kBN * D * 2;
    mbar_expect_tx(bar, KV_BYTES);
    if (is_k) {
#pragma unroll
      for (int at = 0; at < D / 64; ++at)
#pragma unroll
        for (int j = 0; j < kTilePages; ++j)
          tma_load_3d(smem_u32(dst + at * kBN * 128 + j * kPageRows * 128), &a.tm_k, at * 64,
                      s_prow[kt * kTilePages + j < kMaxItemPages ? kt * kTilePages + j : 0], slab, bar);
      k_pend[b] = kt;
    } else {
#pragma unroll
      for (int j = 0; j < kTilePages; ++j)
        tma_load_4d(smem_u32(dst + j * kPageRows * D * 2), &a.tm_v4, 0,
                    s_prow[kt * kTilePages + j < kMaxItemPages ? kt * kTilePages + j : 0], 0, slab, bar);
      v_pend[b] = kt;
    }
  };

  // rotated, scaled queries in the swizzled K-major layout; the first R dims
  // rotate in pairs (d, d + R/2), the rest are only scaled.  The raw rows
  // are staged in the V buffers first (free until their first copy), with
  // independent 16-byte loads; the first two K tiles are already on their way
  // (nothing reads the K buffers before them) while the rotation reads the
  // staged rows and issues its table loads kBatch at a time.
  {
    const int R = g.rope, RH = R / 2;
    constexpr int kChunks = D / 8;                // 16-byte chunks of a row
    if ((reinterpret_cast<uintptr_t>(a.q) & 15) == 0) {
      uint4* stage = reinterpret_cast<uint4*>(sV);  // [kBM][kChunks]
      const uint4* qg = static_cast<const uint4*>(a.q);
      // four loads in flight per thread before their stores
      constexpr int kUnroll = 4;
      for (int i0 = tid; i0 < n_used * kChunks; i0 += kThreads * kUnroll) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int i = i0 + u * kThreads;
          if (i < n_used * kChunks) {
            const int row = i / kChunks, ch = i % kChunks;
            const DecodeMember& mm = s_mem[row / G];
            v[u] = qg[((int64_t)mm.row * g.hq + (int64_t)kvh * G + row % G) * kChunks + ch];
          }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (i0 + u * kThreads < n_used * kChunks) stage[i0 + u * kThreads] = v[u];
      }
    } else {                                        // the caller's q need only be 2-byte aligned
      __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(sV);
      const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
      for (int i = tid; i < n_used * D; i += kThreads) {
        const int row = i / D, d = i % D;
        const DecodeMember& mm = s_mem[row / G];
        stage[i] = qg[((int64_t)mm.row * g.hq + (int64_t)kvh * G + row % G) * D + d];
      }
    }
    __syncthreads();   // staged rows, page rows and the barriers' initialisation are visible
    if (loader && lane == 0 && n_kt > 0) {
      tma_tile(0, true);
      if (n_kt > 1) tma_tile(1, true);
    }
    // one (member, pair) per step: one table load, then the member's G
    // heads; kBatch steps' loads are in flight together
    const __nv_bfloat16* sq = reinterpret_cast<const __nv_bfloat16*>(sV);
    constexpr int kBatch = 16;
    auto put = [&](int row, int dx, float x) {
      *(reinterpret_cast<__nv_bfloat16*>(sQ + sw128(row, dx / 8, kBM)) + dx % 8) = __float2bfloat16_rn(x);
    };
    const int n_pairs = it.n_mem * (D / 2);
    for (int i0 = tid; i0 < n_pairs; i0 += kThreads * kBatch) {
      float2 c[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j * kThreads, d = i % (D / 2);
        c[j] = make_float2(1.f, 0.f);
        if (i < n_pairs && d < RH) {
          const int pos = s_mem[i / (D / 2)].pos_q;
          if (pos >= 0 && pos < a.sa.max_slots) c[j] = a.cs[(int64_t)pos * RH + d];
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j * kThreads;
        if (i >= n_pairs) break;
        const int m = i / (D / 2), d = i % (D / 2);
        int dx, dy;
        if (d < RH) { dx = d; dy = d + RH; }
        else { dx = R + 2 * (d - RH); dy = dx + 1; }
        const int pos = s_mem[m].pos_q;
        const bool have = pos >= 0 && pos < a.sa.max_slots;
        for (int h = 0; h < G; ++h) {
          const int row = m * G + h;
          float x = 0.f, y = 0.f;
          if (have) {
            const float qx = __bfloat162float(sq[row * D + dx]), qy = __bfloat162float(sq[row * D + dy]);
            if (d < RH) {
              x = fmaf(qx, c[j].x, -qy * c[j].y) * a.scale_log2;
              y = fmaf(qx, c[j].y, qy * c[j].x) * a.scale_log2;
            } else {
              x = qx * a.scale_log2;
              y = qy * a.scale_log2;
            }
          }
          put(row, dx, x);
          put(row, dy, y);
        }
      }
    }
    // rows past the members: zero queries
    for (int i = n_used * (D / 2) + tid; i < kBM * (D / 2); i += kThreads) {
      const int row = i / (D / 2), d = i % (D / 2);
      int dx, dy;
      if (d < RH) { dx = d; dy = d + RH; }
      else { dx = R + 2 * (d - RH); dy = dx + 1; }
      put(row, dx, 0.f);
      put(row, dy, 0.f);
    }
  }
  proxy_fence();
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tbase = tslot;
  const uint32_t tO = tbase + 2 * kBN;          // S buffers at 0 and kBN
  auto fail = [&]() {
    *s_abort = 1;
    atomicOr(a.err, AKV_DERR_WAIT);
  };

  float m_r = -INFINITY, l_r = 0.f;
  if (loader) {
    // ---- load warp: K(kt + 2) once softmax(kt) has read S(kt), V(kt + 2)
    // once PV(kt) has read V(kt) (lane 0) ----
    if (lane == 0 && n_kt > 0) {
      tma_tile(0, false);                       // K(0), K(1) went out before the rotation
      if (n_kt > 1) tma_tile(1, false);
      bool ok = true;
      for (int kt = 0; kt + 2 < n_kt && ok && !*s_abort; ++kt) {
        const int b = kt & 1;
        ok = wait_phase(mbP0 + 8 * b, (kt >> 1) & 1, a.wait_limit);
        if (ok) tma_tile(kt + 2, true);
        if (ok) ok = wait_phase(mbO0 + 8 * b, (kt >> 1) & 1, a.wait_limit);
        if (ok) tma_tile(kt + 2, false);
        if (!ok) fail();
      }
      if (*s_abort) {
        // this warp's copies land before the CTA's memory goes (bounded by a
        // fixed limit, independent of the user's wait limit)
        for (int b = 0; b < 2; ++b) {
          if (k_pend[b] >= 0) wait_phase(mbK0 + 8 * b, (k_pend[b] >> 1) & 1, kDrainPolls);
          if (v_pend[b] >= 0) wait_phase(mbV0 + 8 * b, (v_pend[b] >> 1) & 1, kDrainPolls);
        }
      }
    }
    __syncwarp();
  } else if (control) {
    // ---- MMA warp: S(kt + 1) while softmax(kt) runs, then PV(kt) (lane 0) ----
    const uint32_t id_s = idesc_bf16(kBM, kBN, 0), id_o = idesc_bf16(kBM, D, 1);
    int s_pend = -1, o_pend[2] = {-1, -1};
    // descriptors built once; a k step or a buffer adds a constant to the
    // start-address field (addresses stay below 256 KB: no carry)
    const uint64_t dq = sdesc(smem_u32(sQ), 16, 1024);
    const uint64_t dk = sdesc(smem_u32(sK), 16, 1024);
    const uint64_t dv = sdesc(smem_u32(sV), kPageRows * 128, 1024);   // atoms 2 KB apart in a page
    auto issue_s = [&](int kt) {
      const int b = kt & 1;
      const uint64_t kb = dk + (uint64_t)((b * kBN * D * 2) >> 4);
      const uint32_t ts = tbase + b * kBN;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        umma(ts, dq + (uint64_t)((((kk >> 2) * kBM * 128) + (kk & 3) * 32) >> 4),
             kb + (uint64_t)((((kk >> 2) * kBN * 128) + (kk & 3) * 32) >> 4), id_s, kk > 0);
      umma_commit(mbS0 + 8 * b);
      s_pend = kt;
    };
    bool ok = true;
    if (n_kt > 0 && lane == 0) {
      ok = wait_phase(mbK0, 0, a.wait_limit);
      if (ok) { tc_after(); issue_s(0); } else fail();
    }
    for (int kt = 0; kt < n_kt; ++kt) {
      const int b = kt & 1;
      ok = __shfl_sync(0xffffffffu, ok, 0) && !*s_abort;
      if (!ok) break;
      if (lane == 0) {
        // S(kt+1) into the other S buffer once PV(kt-1) has read its P
        if (kt + 1 < n_kt) {
          if (kt > 0) {
            ok = wait_phase(mbO0 + 8 * (b ^ 1), ((kt - 1) >> 1) & 1, a.wait_limit);
            if (ok) o_pend[b ^ 1] = -1;
          }
          if (ok) ok = wait_phase(mbK0 + 8 * (b ^ 1), ((kt + 1) >> 1) & 1, a.wait_limit);
          if (ok) {
            tc_after();
            issue_s(kt + 1);
          }
        }
        // softmax of tile kt done (S(kt) consumed, P(kt) written) and V(kt) in
        if (ok) ok = wait_phase(mbP0 + 8 * b, (kt >> 1) & 1, a.wait_limit);
        if (ok) {
          s_pend = s_pend == kt ? -1 : s_pend;
          ok = wait_phase(mbV0 + 8 * b, (kt >> 1) & 1, a.wait_limit);
        }
        if (!ok) fail();
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      {
        // V rows of slots no row sees (keep bit clear: the same for every
        // member) may hold any bits -- a prefix fork's empty tail page, for
        // one, is held but never written -- and 0 * NaN is NaN in the MMA:
        // zero them in shared memory first (rare; pages past the range were
        // filled with zeros by the copy)
        uint64_t dead = 0;
#pragma unroll
        for (int j = 0; j < kTilePages; ++j) {
          const int pg = kt * kTilePages + j;
          if (pg < n_pages) dead |= (uint64_t)(~s_pbits[pg] & 0xffffu) << (16 * j);
        }
        if (dead) {
          // every lane observes the copy's completion before writing over it
          if (!__all_sync(0xffffffffu, wait_phase(mbV0 + 8 * b, (kt >> 1) & 1, kDrainPolls))) {
            if (lane == 0) fail();
            break;
          }
          uint8_t* vt = sV + b * kBN * D * 2;
          for (int u = lane; u < kBN * (D / 64) * 8; u += 32) {
            const int r = u / ((D / 64) * 8), at = (u / 8) % (D / 64), c = u % 8;
            if ((dead >> r) & 1)
              *reinterpret_cast<uint4*>(vt + (r / kPageRows) * kPageRows * D * 2 + at * kPageRows * 128 +
                                        (r % kPageRows) * 128 + c * 16) = make_uint4(0, 0, 0, 0);
          }
          proxy_fence();
          __syncwarp();
        }
      }
      if (lane == 0) {
        // O += P(kt) V(kt)
        tc_after();
        const uint64_t vb = dv + (uint64_t)((b * kBN * D * 2) >> 4);
        const uint32_t tSb = tbase + b * kBN;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_ts(tO, tSb + kk * 8, vb + (uint64_t)((kk * kPageRows * D * 2) >> 4), id_o, kt > 0 || kk > 0);
        umma_commit(mbO0 + 8 * b);
        o_pend[b] = kt;
      }
      __syncwarp();
    }
    if (lane == 0 && *s_abort) {
      // this warp's MMAs finish before the CTA's memory goes (bounded)
      if (s_pend >= 0) wait_phase(mbS0 + 8 * (s_pend & 1), (s_pend >> 1) & 1, kDrainPolls);
      for (int b = 0; b < 2; ++b)
        if (o_pend[b] >= 0) wait_phase(mbO0 + 8 * b, (o_pend[b] >> 1) & 1, kDrainPolls);
    }
  } else {
    // ---- softmax warps: row = TMEM lane, tokens and O columns split in halves ----
    const int quarter = warp & 3, half = warp >> 2;
    const int row = 32 * quarter + lane;
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    // token j of the range is visible to the row iff its keep bit is set
    // and j lies in the member's run of pages; padding rows see nothing
    const int end_r = row < n_used ? s_mem[row / G].n_tiles * kPageRows : 0;
    const int w_end = __reduce_min_sync(0xffffffffu, row < n_used ? end_r : INT32_MAX);
    for (int kt = 0; kt < n_kt; ++kt) {
      const int b = kt & 1;
      const int k0 = kt * kBN + half * kHalf;
      const uint32_t tSb = tbase + b * kBN;
      bool ok = wait_phase(mbS0 + 8 * b, (kt >> 1) & 1, a.wait_limit);
      ok = __all_sync(0xffffffffu, ok) && !*s_abort;
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_after();
      uint32_t sr[kHalf];
      tmem_ld32(tSb + lane_off + half * kHalf, sr);
      tmem_wait_ld();
      // keep bits of this half's two pages (pages past the range: none)
      const int pg = kt * kTilePages + 2 * half;
      const uint32_t kb = (pg < n_pages ? s_pbits[pg] : 0u) |
                          ((pg + 1 < n_pages ? s_pbits[pg + 1] : 0u) << 16);
      const bool full = kb == 0xffffffffu && k0 + kHalf <= w_end;   // warp-uniform
      float sv[kHalf];
      float mx = -INFINITY;
      if (full) {
#pragma unroll
        for (int c = 0; c < kHalf; ++c) sv[c] = __uint_as_float(sr[c]);
#pragma unroll
        for (int c = 0; c < kHalf; c += 2) mx = fmax3(mx, sv[c], sv[c + 1]);
      } else {
#pragma unroll
        for (int c = 0; c < kHalf; ++c) {
          const bool vis = ((kb >> c) & 1u) && k0 + c < end_r;
          sv[c] = vis ? __uint_as_float(sr[c]) : -INFINITY;
          mx = fmaxf(mx, sv[c]);
        }
      }
      // row max over both halves (bounded exchange with the partner warp)
      s_mx[(b * 2 + half) * kBM + row] = mx;
      __syncwarp();
      const uint32_t xb = mbX0 + 8 * (quarter * 2 + b);
      if (lane == 0) mbar_arrive(xb);
      if (!__all_sync(0xffffffffu, wait_phase(xb, (kt >> 1) & 1, a.wait_limit))) {
        if (lane == 0) fail();
        break;
      }
      mx = fmaxf(mx, s_mx[(b * 2 + (half ^ 1)) * kBM + row]);
      // the reference max moves only when the row max grows by more than 2^8
      const float m_new = (mx > m_r + 8.f) ? mx : m_r;
      const float alpha = m_new == -INFINITY ? 1.f : ex2(m_r - m_new);
      const float msub = m_new == -INFINITY ? 0.f : m_new;
      uint64_t ps2 = 0;
      const uint64_t neg_m = pack_f32x2(-msub, -msub);
      uint32_t pk[kHalf / 2];
#pragma unroll
      for (int c = 0; c < kHalf; c += 2) {
        float d0, d1;
        unpack_f32x2(add_f32x2(pack_f32x2(sv[c], sv[c + 1]), neg_m), d0, d1);
        const float p0 = ex2(d0), p1 = ex2(d1);
        ps2 = add_f32x2(ps2, pack_f32x2(p0, p1));
        pk[c / 2] = pack_bf16x2(p0, p1);
      }
      float ps_lo, ps_hi;
      unpack_f32x2(ps2, ps_lo, ps_hi);
      l_r = fmaf(l_r, alpha, ps_lo + ps_hi);     // this half's share of the row sum
      m_r = m_new;
      tmem_st16(tSb + lane_off + half * (kHalf / 2), pk);   // P(kt) over S(kt)
      if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O is stable once PV(kt-1) is done; this half rescales its columns
        const bool okv = __all_sync(0xffffffffu, wait_phase(mbO0 + 8 * ((kt - 1) & 1), ((kt - 1) >> 1) & 1,
                                                             a.wait_limit));
        if (!okv) {
          if (lane == 0) fail();
          break;
        }
        tc_after();
#pragma unroll
        for (int c = 0; c < D / 2; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + lane_off + half * (D / 2) + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + lane_off + half * (D / 2) + c, o);
        }
      }
      tmem_wait_st();
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(mbP0 + 8 * b);
    }
    // the last PV
    if (n_kt > 0 && !*s_abort) {
      const bool okv = __all_sync(0xffffffffu, wait_phase(mbO0 + 8 * ((n_kt - 1) & 1),
                                                           ((n_kt - 1) >> 1) & 1, a.wait_limit));
      if (!okv && lane == 0) fail();
    }
    // this half's row sum, combined in the epilogue
    s_mx[(4 + half) * kBM + row] = l_r;
  }
  tc_before();
  __syncthreads();
  tc_after();

  // The previous decode call (launched before this grid may start, see the
  // launcher) merges partials from the slots this grid writes: the first
  // global write waits until that grid has finished.  Nothing above reads
  // memory a decode call writes.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (warp < kSoftmaxWarps && !*s_abort) {
    // epilogue: this half's columns of the unnormalised O, and (max, sum)
    const int quarter = warp & 3, half = warp >> 2;
    const int row = 32 * quarter + lane;
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const bool real = row < n_used;
    int64_t pi = 0;
    if (real) pi = ((int64_t)s_mem[row / G].part * g.hkv + kvh) * G + row % G;
    float* pa = a.part_acc + pi * D + half * (D / 2);
    const float l = s_mx[4 * kBM + row] + s_mx[5 * kBM + row];
#pragma unroll
    for (int c = 0; c < D / 2; c += 32) {
      uint32_t o[32];
      if (n_kt > 0) {
        tmem_ld32(tO + lane_off + half * (D / 2) + c, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      if (real) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(pa + c + e) =
              make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                          __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
      }
    }
    if (real && half == 0) a.part_ml[pi] = make_float2(l > 0.f ? m_r : -INFINITY, l);
  }
  __threadfence();
  tc_before();
  __syncthreads();
  // each member's partial is in: count it (the row's last split merges)
  if (!*s_abort && tid < it.n_mem) atomicAdd(&a.counters[s_mem[tid].row * g.hkv + kvh], 1);
  if (control)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kCols) : "memory");
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t st) {
  constexpr size_t smem = share_smem<D>();
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(k_decode_share_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attr = true;
  }
  // programmatic stream serialisation (a.pdl: the stream's previous work is
  // a decode call, which signals its dependents at its start): this grid's
  // blocks start early and wait (griddepcontrol.wait) before their first write
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_share_items, a.g.hkv);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr_pdl[1];
  attr_pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr_pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr_pdl;
  cfg.numAttrs = a.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_decode_share_tc<D>, a);
}

}  // namespace

bool decode_share_supported(const Geom& g) {
  const int G = g.hq / g.hkv;
  return g.dtype == AKV_DTYPE_BF16 && g.s == kPageRows && (g.d == 64 || g.d == 128) &&
         (G == 1 || G == 2 || G == 4 || G == 8);
}

cudaError_t launch_decode_share(const DecodeArgs& a, cudaStream_t st) {
  if (a.n_share_items <= 0) return cudaSuccess;
  return a.g.d == 64 ? launch_d<64>(a, st) : launch_d<128>(a, st);
}

}  // namespace akv
