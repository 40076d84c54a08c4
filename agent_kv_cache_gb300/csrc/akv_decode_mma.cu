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
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
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

template <int D>
__global__ void __launch_bounds__(kThreads) k_decode_mma(const __grid_constant__ DecodeArgs a) {
  constexpr int KS = D / 16;                    // k-steps of Q K^T, m-tiles of V^T P^T
  constexpr int TILE_BYTES = kTile * D * 2;     // one K (or V) tile
  constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // The stage ring also holds, before the tile loop, the rotated query
  // [8][D] and, after it, the consumer warps' partials [4][8][D+2].
  float* s_q = reinterpret_cast<float*>(smem);
  float* s_merge = reinterpret_cast<float*>(smem);
  __shared__ __align__(8) uint64_t s_full[kStages], s_empty[kStages];
  __shared__ int s_row[kMaxTiles];              // TMA row of each tile, -1 = unusable
  __shared__ uint16_t s_bits[kMaxTiles];        // keep bits of each tile's 16 slots
  __shared__ int s_last;

  // the next decode call may be scheduled now: its blocks start as this
  // grid's blocks retire and wait (griddepcontrol.wait) before writing
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const DecodeItem it = a.items[blockIdx.x];
  const int kvh = blockIdx.y;
  const Geom& g = a.g;
  const int G = g.hq / g.hkv;
  const int tpp = g.s / kTile;                  // tiles per page
  const int t0 = it.p0 * tpp;
  int n = it.p1 * tpp - t0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the work item must describe memory this call owns (uniform per block)
  const bool bad_item =
      it.dslot < 0 || it.dslot >= a.max_seqs || it.row < 0 || it.row >= a.n_rows ||
      it.p0 < 0 || it.p1 < it.p0 || it.p1 > a.sa.seq_pages || it.n_splits < 1 ||
      it.item0 < 0 || it.item0 + it.n_splits > a.n_items || (int)blockIdx.x < it.item0 ||
      (int)blockIdx.x >= it.item0 + it.n_splits || it.row >= a.counter_rows;
  if (bad_item) {
    if (tid == 0) atomicOr(a.err, AKV_DERR_INDEX);
    return;
  }
  if (n > kMaxTiles) {                          // the planner never makes such a split
    if (tid == 0) atomicOr(a.err, AKV_DERR_INDEX);
    n = kMaxTiles;
  }
  const int64_t slab_rows = (int64_t)g.max_pages * g.hkv * g.s;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&s_empty[s]), 1);
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
  // rotated, scaled query of the group (heads >= G stay zero); the first R
  // dims rotate in pairs (d, d + R/2), dims R.. are only scaled
  {
    const int R = g.rope, RH = R / 2;
    const bool have_q = it.pos_q >= 0 && it.pos_q < a.sa.max_slots;
    for (int i = tid; i < 8 * D; i += kThreads) {
      const int gq = i / D, d = i % D;
      const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) +
                               ((int64_t)it.row * g.hq + (int64_t)kvh * G + gq) * D;
      if (d < RH) {
        float x = 0.f, y = 0.f;
        if (gq < G && have_q) {
          const float qx = __bfloat162float(q[d]), qy = __bfloat162float(q[d + RH]);
          const float2 t = a.cs[(int64_t)it.pos_q * RH + d];
          x = fmaf(qx, t.x, -qy * t.y) * a.scale_log2;
          y = fmaf(qx, t.y, qy * t.x) * a.scale_log2;
        }
        s_q[gq * D + d] = x;
        s_q[gq * D + d + RH] = y;
      } else if (d >= R) {
        s_q[gq * D + d] = (gq < G && have_q) ? __bfloat162float(q[d]) * a.scale_log2 : 0.f;
      }
    }
  }
  __syncthreads();
  // Q^T fragments (B operand of the score MMA): lane holds head lane/4,
  // dims 2*(lane%4)+{0,1} and +8 of each 16-dim k-step
  uint32_t qf[KS][2];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int h = lane >> 2, c = ks * 16 + (lane & 3) * 2;
    qf[ks][0] = pack_bf16(s_q[h * D + c], s_q[h * D + c + 1]);
    qf[ks][1] = pack_bf16(s_q[h * D + c + 8], s_q[h * D + c + 9]);
  }
  // s_q is dead: order these generic-proxy accesses before the TMA writes
  // (async proxy) that reuse the ring
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();

  const int slab = (a.layer >= 0 ? a.layer : 0) % g.phys_layers;
  float o[KS][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // heads 2*(lane%4), +1

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
          const uint32_t dk = smem_u32(smem + s * STAGE_BYTES);
#pragma unroll
          for (int b = 0; b < D / 64; ++b) {
            tma_load_3d(dk + b * 2048, &a.tm_k, b * 64, row, slab, full);
            tma_load_3d(dk + TILE_BYTES + b * 2048, &a.tm_v, b * 64, row, slab, full);
          }
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

    for (int i = warp; i < n; i += kConsumers) {
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
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t af[4];
          ldsm_x4(kb + swz(k_row, ks * 2 + k_cb), af);
          mma16816(sc, af, qf[ks][0], qf[ks][1]);
        }
        if (!((bits >> r0) & 1u)) sc[0] = sc[1] = -INFINITY;
        if (!((bits >> (r0 + 8)) & 1u)) sc[2] = sc[3] = -INFINITY;
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
    // per-warp partial -> shared: [warp][head][D] then m, l at [D], [D+1]
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
  // merge the consumer warps: the output (one split) or this split's partial
  for (int i = tid; i < G * D; i += kThreads) {
    const int gq = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, s_merge[(w * 8 + gq) * (D + 2) + D]);
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float* wm = s_merge + (w * 8 + gq) * (D + 2);
        const float f = exp2f(wm[D] - M);
        L = fmaf(wm[D + 1], f, L);
        A = fmaf(wm[d], f, A);
      }
    }
    const int hq = kvh * G + gq;
    if (it.n_splits == 1) {
      a.out[((int64_t)it.row * g.hq + hq) * D + d] = L > 0.f ? A / L : 0.f;
    } else {
      const int64_t pi = ((int64_t)blockIdx.x * g.hkv + kvh) * G + gq;
      a.part_acc[pi * D + d] = A;
      if (d == 0) a.part_ml[pi] = make_float2(M, L);
    }
  }
  if (it.n_splits == 1) return;

  // the last split of (row, kv head) to finish merges all of them
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int old = atomicAdd(&a.counters[it.row * g.hkv + kvh], 1);
    s_last = old == it.n_splits - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int i = tid; i < G * D; i += kThreads) {
    const int gq = i / D, d = i % D;
    float M = -INFINITY;
    for (int c = 0; c < it.n_splits; ++c)
      M = fmaxf(M, __ldcg(&a.part_ml[((int64_t)(it.item0 + c) * g.hkv + kvh) * G + gq]).x);
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
      for (int c = 0; c < it.n_splits; ++c) {
        const int64_t pi = ((int64_t)(it.item0 + c) * g.hkv + kvh) * G + gq;
        const float2 ml = __ldcg(&a.part_ml[pi]);
        const float f = exp2f(ml.x - M);
        L = fmaf(ml.y, f, L);
        A = fmaf(__ldcg(&a.part_acc[pi * D + d]), f, A);
      }
    }
    a.out[((int64_t)it.row * g.hq + kvh * G + gq) * D + d] = L > 0.f ? A / L : 0.f;
  }
  if (tid == 0) a.counters[it.row * g.hkv + kvh] = 0;   // ready for the next call
}

template <int D>
constexpr size_t mma_smem() {
  static_assert((size_t)kConsumers * 8 * (D + 2) * 4 <= (size_t)kStages * 2 * kTile * D * 2,
                "the partials must fit in the stage ring");
  return 1024 + (size_t)kStages * 2 * kTile * D * 2;
}

template <int D>
void set_smem_attr() {
  static bool done = false;
  if (!done) {
    cudaFuncSetAttribute(k_decode_mma<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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

// Launched with programmatic stream serialisation: when the previous work on
// the stream is a decode call (which signals launch_dependents at its start),
// this grid's blocks may start while that grid's last blocks still run, so
// its start-up (work item, tile list, query) hides behind the other's tail.
// A decode call reads nothing a decode call writes before its
// griddepcontrol.wait; any other predecessor (append, drop, reposition, a
// copy, the caller's kernels) never signals early, so for it the ordering is
// the plain stream order.
cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t st) {
  const dim3 grid(a.n_items, a.g.hkv);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.g.d == 64) {
    set_smem_attr<64>();
    cfg.dynamicSmemBytes = mma_smem<64>();
    return cudaLaunchKernelEx(&cfg, k_decode_mma<64>, a);
  }
  set_smem_attr<128>();
  cfg.dynamicSmemBytes = mma_smem<128>();
  return cudaLaunchKernelEx(&cfg, k_decode_mma<128>, a);
}

int decode_mma_blocks_per_sm(int d) {
  int n = 0;
  if (d == 64) {
    set_smem_attr<64>();
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_decode_mma<64>, kThreads, mma_smem<64>());
  } else {
    set_smem_attr<128>();
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_decode_mma<128>, kThreads, mma_smem<128>());
  }
  return n;
}

}  // namespace akv
