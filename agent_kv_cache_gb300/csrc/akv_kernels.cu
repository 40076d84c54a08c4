// Cache-maintenance kernels: append (Eq. 3), drop (Eq. 4), reposition
// (Eq. 5: compaction + gather/rotate/store), and the copy-on-write page copy.
//
// Sources: "Cache Engineering for Agents" paper review, 3.3 Cache Operations
// (Eqs. 3-5); "[Repo Review] AKV", 5.5 (the reposition kernel un-rotates the
// old position and rotates the new one in FP32, copies V and non-RoPE parts,
// copies raw values when the position is unchanged, and writes to a separate
// destination slot).
//
// Every kernel validates the indices it takes from metadata and, instead of
// touching memory out of bounds, sets a bit in the device error word and
// skips the access.
#include <algorithm>
#include <cmath>
#include <type_traits>

#include <cuda_bf16.h>

#include "akv.h"
#include "akv_internal.h"

namespace akv {
namespace {

// ---------------------------------------------------------------------------
// 16-byte vectors of the pool dtype
// ---------------------------------------------------------------------------

template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
  static constexpr int E = 8;
  __device__ static void unpack(uint4 u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static uint4 pack(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <> struct Vec<float> {
  static constexpr int E = 4;
  __device__ static void unpack(uint4 u, float* f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  __device__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                      __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};

__device__ __forceinline__ uint4 ld16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st16(void* p, uint4 v) {
  *reinterpret_cast<uint4*>(p) = v;
}

// Exact rounding of nearly cancelling pairs.  The fp32 rotation below,
// xo = fma(x, c, -RN(y s)) with c, s the table entries rounded once to fp32,
// is off the exact value by at most 2^-24 (|x c| + |y s|) (table) +
// 2^-24 |y s| (product) + 2^-24 |xo| (fma), i.e. about 2^-23 |(x, y)|: an
// error that scales with the pair, not with the element.  Rounding to bf16
// then lands within one bf16 ulp of the exactly rotated value rounded to
// nearest even whenever that error is below half the bf16 spacing at the
// element, 2^-9 |X|, i.e. whenever |X| >= 2^-14 |(x, y)|.  Elements below
// 2^-13 (|x| + |y|) (rotations that nearly cancel, about 2 pairs in 10^4) are
// recomputed in compensated fp32: the products with the fp32 table entries
// exactly (an fma recovers each rounding error), the table's own rounding
// error from a second fp32 table of low parts (cos - RN(cos), sin - RN(sin)),
// so the result is the exact rotation to ~2^-46 |(x, y)| before its final
// roundings.  Every stored bf16 key is then within one bf16 ulp of Eq. (5)
// evaluated exactly (page 2, 5.5 keeps fp32 arithmetic, which the common
// path still is).  fp32 pools need no fix-up (their bound is on the pair).
//
// The common path only tests; the recomputation is a separate, never-inlined
// function entered by the few threads that need it (inlined, the compiler
// predicates it into every element).
__device__ __forceinline__ bool cancels(float x, float y, float xo, float yo) {
  return fminf(fabsf(xo), fabsf(yo)) < (fabsf(x) + fabsf(y)) * 0x1p-13f;
}

// Recompute the cancelling pairs of one unit (E pairs; table entry of pair
// e at cs[e * cs_stride], its low part at lo[e * lo_stride] with the sine's
// part times lo_sy, or zero when lo is null) and overwrite them in dst_lo /
// dst_hi.  `lo` may point to global memory: this path is rare.
template <int E>
__device__ __noinline__ void refine_cancelling(uint4 u_lo, uint4 u_hi, __nv_bfloat16* dst_lo,
                                               __nv_bfloat16* dst_hi, const float2* cs,
                                               int cs_stride, const float2* lo, int lo_stride,
                                               float lo_sy) {
  float x[E], y[E];
  Vec<__nv_bfloat16>::unpack(u_lo, x);
  Vec<__nv_bfloat16>::unpack(u_hi, y);
  for (int e = 0; e < E; ++e) {
    const float2 t = cs[e * cs_stride];
    const float xo = fmaf(x[e], t.x, -y[e] * t.y);
    const float yo = fmaf(x[e], t.y, y[e] * t.x);
    if (!cancels(x[e], y[e], xo, yo)) continue;
    float2 l = lo ? lo[e * lo_stride] : make_float2(0.f, 0.f);
    l.y *= lo_sy;
    // x (c + cl) - y (s + sl) and x (s + sl) + y (c + cl); each product with
    // the fp32 entry split into its rounded value and its exact error
    const float p1 = x[e] * t.x, e1 = fmaf(x[e], t.x, -p1);
    const float p2 = y[e] * t.y, e2 = fmaf(y[e], t.y, -p2);
    const float p3 = x[e] * t.y, e3 = fmaf(x[e], t.y, -p3);
    const float p4 = y[e] * t.x, e4 = fmaf(y[e], t.x, -p4);
    const float rx = (p1 - p2) + ((e1 - e2) + fmaf(x[e], l.x, -y[e] * l.y));
    const float ry = (p3 + p4) + ((e3 + e4) + fmaf(x[e], l.y, y[e] * l.x));
    dst_lo[e] = __float2bfloat16_rn(rx);
    dst_hi[e] = __float2bfloat16_rn(ry);
  }
}

// One rotation unit, already loaded into registers: E consecutive pairs
// (i, i + D/2) starting at i = c*E, (x, y) -> (x cos - y sin, x sin + y cos)
// in fp32, rounded once to T, with the row's cos/sin stored unit-minor:
// pair c*E + e at cs_t[e * n_units + c], so the lanes rotating one row read
// consecutive words (no bank conflicts); the low parts of the row's entries
// in the table's own row lo_row (pair order, read only for a cancelling
// pair; null: zero), the sine's part times lo_sy.
template <typename T>
__device__ __forceinline__ void rotate_regs(uint4 lo, uint4 hi, T* dst, int c, int half,
                                            const float2* cs_t, int n_units, const float2* lo_row,
                                            float lo_sy) {
  constexpr int E = Vec<T>::E;
  float x[E], y[E], xo[E], yo[E];
  Vec<T>::unpack(lo, x);
  Vec<T>::unpack(hi, y);
  bool any = false;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float2 t = cs_t[e * n_units + c];
    xo[e] = fmaf(x[e], t.x, -y[e] * t.y);
    yo[e] = fmaf(x[e], t.y, y[e] * t.x);
    any |= cancels(x[e], y[e], xo[e], yo[e]);
  }
  st16(dst + c * E, Vec<T>::pack(xo));
  st16(dst + half + c * E, Vec<T>::pack(yo));
  if constexpr (std::is_same<T, __nv_bfloat16>::value)
    if (any) refine_cancelling<E>(lo, hi, dst + c * E, dst + half + c * E, cs_t + c, n_units,
                                  lo_row ? lo_row + c * E : nullptr, 1, lo_sy);
}

template <typename T>
__device__ __forceinline__ void copy_unit(const T* src, T* dst, int c, int half) {
  constexpr int E = Vec<T>::E;
  st16(dst + c * E, ld16(src + c * E));
  st16(dst + half + c * E, ld16(src + half + c * E));
}

__device__ __forceinline__ void flag(uint32_t* err, uint32_t bit) { atomicOr(err, bit); }

// ---------------------------------------------------------------------------
// append: K = R(pos) K_raw, V copied; pages/active/keep metadata updated
// ---------------------------------------------------------------------------

template <typename T>
__global__ void __launch_bounds__(256, 4)
k_append(Geom g, SeqArrays sa, const AppendItem* __restrict__ items,
         const AppendBlock* __restrict__ blocks, const int32_t* __restrict__ ids,
         const int32_t* __restrict__ act, const T* __restrict__ k_raw,
         const T* __restrict__ v_raw, int64_t total_tokens,
         const float2* __restrict__ cs, uint32_t* err, AppendLimits lim) {
  extern __shared__ float2 s_cs[];   // [kAppendTokens][R/2] cos/sin, unit-minor
  __shared__ int s_page[kAppendTokens];
  __shared__ int s_off[kAppendTokens];
  const AppendBlock blk = blocks[blockIdx.x];
  if (blk.item < 0 || blk.item >= lim.n_items) {
    if (threadIdx.x == 0) flag(err, AKV_DERR_INDEX);
    return;
  }
  const AppendItem it = items[blk.item];
  // the item must describe memory this call owns (uniform per block)
  if (it.dslot < 0 || it.dslot >= lim.max_seqs || it.ids_off < 0 || it.nk < 0 ||
      it.ids_off + it.nk > lim.n_ids || it.act_off < 0 || it.n_act < 0 ||
      it.act_off + it.n_act > lim.n_act || it.tok0 < 0 || it.n < 0 || blk.t0 < 0 ||
      blk.t0 >= it.n || (int64_t)it.tok0 + it.n > total_tokens) {
    if (threadIdx.x == 0) flag(err, AKV_DERR_INDEX);
    return;
  }
  const int nt = min(kAppendTokens, it.n - blk.t0);
  const int D = g.d, S = g.s;
  const int tid = threadIdx.x, bs = blockDim.x;
  const int64_t row_base = (int64_t)it.dslot;

  // blockIdx.y picks the physical slab; the block writes the logical layers
  // stored there in order (y, y + phys_layers, ...; with one slab per layer
  // that is one layer), so the last of them is what the slab keeps
  const int l_begin = blockIdx.y, l_step = g.phys_layers;
  const bool meta = blockIdx.y == 0;

  if (blk.t0 == 0 && meta) {
    for (int i = tid; i < it.nk; i += bs) {
      const int k = it.k0 + i;
      if (k >= 0 && k < sa.seq_pages) sa.pages[row_base * sa.seq_pages + k] = ids[it.ids_off + i];
      else flag(err, AKV_DERR_INDEX);
    }
    for (int i = tid; i < it.n_act; i += bs) {
      const int a = it.act0 + i;
      if (a >= 0 && a < sa.seq_pages) sa.active[row_base * sa.seq_pages + a] = act[it.act_off + i];
      else flag(err, AKV_DERR_INDEX);
    }
  }
  for (int t = tid; t < nt; t += bs) {
    const int slot = it.slot0 + blk.t0 + t;
    int pid = -1;
    if (slot >= 0 && slot < sa.max_slots) {
      if (meta) atomicOr(&sa.keep[row_base * sa.keep_words + slot / 32], 1u << (slot % 32));
      const int pk = slot / S - it.k0;
      if (pk >= 0 && pk < it.nk) pid = ids[it.ids_off + pk];
    }
    if (pid < 0 || pid >= g.max_pages) { if (meta) flag(err, AKV_DERR_PAGE); pid = -1; }
    s_page[t] = pid;
    s_off[t] = slot % S;
  }
  // the rows' cos/sin, unit-minor (pair c*E + e of row t at
  // s_cs[t*RH + e*kr + c]: the lanes rotating one row read consecutive words)
  constexpr int E = Vec<T>::E;
  const int R = g.rope, RH = R / 2;
  const int kr = RH / E, kc = (D - R) / E, vu = D / E, per_row = kr + kc + vu;
  for (int i = tid; i < nt * RH; i += bs) {
    const int t = i / RH, jj = i % RH;
    const int slot = it.slot0 + blk.t0 + t;
    const bool in = slot >= 0 && slot < sa.max_slots;
    s_cs[t * RH + (jj % E) * kr + jj / E] = in ? cs[(int64_t)slot * RH + jj] : make_float2(1.f, 0.f);
  }
  __syncthreads();

  // units of a row: rotary (pairs of 16-byte chunks), K dims past the rotary
  // part (copied), V chunks (copied).  A thread's unit goes to several
  // layers: the loads of kLayerBatch of them go out before their stores
  // (they are independent; the stores keep layer order, so a slab shared by
  // several logical layers keeps the last one).
  constexpr int kLayerBatch = 2;
  const int units = g.hkv * nt * per_row;
  const T* __restrict__ kb = k_raw;
  const T* __restrict__ vb = v_raw;
  T* kp = static_cast<T*>(g.k);
  T* vp = static_cast<T*>(g.v);
  for (int u = tid; u < units; u += bs) {
    const int r = u % per_row;
    const int t = (u / per_row) % nt;
    const int h = u / (per_row * nt);
    const int pid = s_page[t];
    if (pid < 0) continue;
    const int64_t tok = it.tok0 + blk.t0 + t;
    const int64_t dst_off = (int64_t)pid * g.page_stride + (int64_t)h * g.head_stride +
                            (int64_t)s_off[t] * D;
    const int slot = it.slot0 + blk.t0 + t;
    const float2* lo_row = (slot >= 0 && slot < sa.max_slots) ? g.cs_lo + (int64_t)slot * RH : nullptr;
    // element offset of this unit in a source row and in a stored row
    const int o_a = r < kr ? r * E : r < kr + kc ? R + (r - kr) * E : (r - kr - kc) * E;
    const T* src = r < kr + kc ? kb : vb;
    T* dst = r < kr + kc ? kp : vp;
    for (int l0 = l_begin; l0 < g.layers; l0 += kLayerBatch * l_step) {
      uint4 a[kLayerBatch], b[kLayerBatch];
#pragma unroll
      for (int q = 0; q < kLayerBatch; ++q) {
        const int l = l0 + q * l_step;
        if (l < g.layers) {
          const int64_t src_off = ((int64_t)l * total_tokens + tok) * g.hkv * D + (int64_t)h * D;
          a[q] = ld16(src + src_off + o_a);
          if (r < kr) b[q] = ld16(src + src_off + RH + o_a);
        }
      }
#pragma unroll
      for (int q = 0; q < kLayerBatch; ++q) {
        const int l = l0 + q * l_step;
        if (l >= g.layers) break;
        T* row = dst + (int64_t)(l % g.phys_layers) * g.layer_stride + dst_off;
        if (r < kr)
          rotate_regs<T>(a[q], b[q], row, r, RH, s_cs + t * RH, kr, lo_row, 1.f);
        else
          st16(row + o_a, a[q]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// copy-on-write: copy whole pages (every physical layer, K and V)
// ---------------------------------------------------------------------------

template <typename T>
__global__ void __launch_bounds__(256)
k_copy_pages(Geom g, const PagePair* __restrict__ pairs, uint32_t* err) {
  const PagePair pp = pairs[blockIdx.x];
  if (pp.src < 0 || pp.src >= g.max_pages || pp.dst < 0 || pp.dst >= g.max_pages) {
    if (threadIdx.x == 0) flag(err, AKV_DERR_PAGE);
    return;
  }
  constexpr int E = Vec<T>::E;
  const int64_t slab = (int64_t)blockIdx.y * g.layer_stride;
  const int n = (int)(g.page_stride / E);
  const T* ks = static_cast<const T*>(g.k) + slab + pp.src * g.page_stride;
  const T* vs = static_cast<const T*>(g.v) + slab + pp.src * g.page_stride;
  T* kd = static_cast<T*>(g.k) + slab + pp.dst * g.page_stride;
  T* vd = static_cast<T*>(g.v) + slab + pp.dst * g.page_stride;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    st16(kd + i * E, ld16(ks + i * E));
    st16(vd + i * E, ld16(vs + i * E));
  }
}

// ---------------------------------------------------------------------------
// block-wide exclusive scan of one int per thread (blockDim.x == 1024)
// ---------------------------------------------------------------------------

__device__ __forceinline__ int block_exclusive_scan(int x, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) s_warp[lane] = wi - w;   // exclusive warp offsets
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const int r = s_warp[warp] + incl - x;
  __syncthreads();   // s_warp is reused by the next call
  return r;
}

// keep bits of slot page k (S slots starting at k*S), S in {1,...,64}
__device__ __forceinline__ int page_popc(const uint32_t* keep, int k, int S) {
  const int64_t first = (int64_t)k * S;
  if (S >= 32) {
    int c = 0;
    for (int w = 0; w < S / 32; ++w) c += __popc(keep[first / 32 + w]);
    return c;
  }
  const uint32_t word = keep[first / 32];
  const uint32_t m = (S == 32) ? 0xffffffffu : ((1u << S) - 1u);
  return __popc((word >> (first % 32)) & m);
}

// ---------------------------------------------------------------------------
// drop: clear keep bits of slot ranges, rebuild the active page list,
// release (mark -1) full pages left with no active token
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(1024)
k_drop(Geom g, SeqArrays sa, const DropItem* __restrict__ items,
       const int32_t* __restrict__ ranges, uint32_t* err) {
  __shared__ int s_warp[32];
  __shared__ int s_total;
  const DropItem it = items[blockIdx.x];
  uint32_t* keep = sa.keep + (int64_t)it.dslot * sa.keep_words;
  int32_t* pages = sa.pages + (int64_t)it.dslot * sa.seq_pages;
  int32_t* active = sa.active + (int64_t)it.dslot * sa.seq_pages;
  const int S = g.s;

  for (int r = 0; r < it.n_ranges; ++r) {
    const int a = ranges[it.range_off + 2 * r];
    const int b = ranges[it.range_off + 2 * r + 1];
    if (a < 0 || b > it.n_slots || a > b) {
      if (threadIdx.x == 0) flag(err, AKV_DERR_INDEX);
      continue;
    }
    if (a == b) continue;
    const int w0 = a / 32, w1 = (b - 1) / 32;
    for (int w = w0 + (int)threadIdx.x; w <= w1; w += blockDim.x) {
      const int lo = max(a - w * 32, 0), hi = min(b - w * 32, 32);
      const uint32_t m = (hi == 32 ? 0xffffffffu : ((1u << hi) - 1u)) & ~((1u << lo) - 1u);
      atomicAnd(&keep[w], ~m);
    }
  }
  __syncthreads();

  // each thread a run of consecutive pages: one block scan of the run counts
  // (not one per blockDim pages), then each run writes its live pages in order
  const int per = (it.n_pages + (int)blockDim.x - 1) / (int)blockDim.x;
  const int k0 = (int)threadIdx.x * per, k1 = min(it.n_pages, k0 + per);
  int live_n = 0;
  for (int k = k0; k < k1; ++k) {
    const bool live = page_popc(keep, k, S) > 0;
    if (!live && (int64_t)(k + 1) * S <= it.n_slots) pages[k] = -1;
    live_n += live;
  }
  int o = block_exclusive_scan(live_n, s_warp, &s_total);
  for (int k = k0; k < k1; ++k)
    if (page_popc(keep, k, S) > 0) active[o++] = k;
  if (threadIdx.x == 0 && s_total != it.expect_active) flag(err, AKV_DERR_COUNT);
}

// ---------------------------------------------------------------------------
// reposition, part 1: compaction.  Exclusive prefix sum of the keep bits
// (each thread owns a run of 32-slot words: popc + one block scan) gives the
// gather map; the new page table, keep bits and active list follow.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(1024)
k_compact(Geom g, SeqArrays sa, const ReposItem* __restrict__ items,
          const int32_t* __restrict__ ids, uint32_t* err) {
  __shared__ int s_warp[32];
  __shared__ int s_total;
  const ReposItem it = items[blockIdx.x];
  uint32_t* keep = sa.keep + (int64_t)it.dslot * sa.keep_words;
  int32_t* pages = sa.pages + (int64_t)it.dslot * sa.seq_pages;
  int32_t* active = sa.active + (int64_t)it.dslot * sa.seq_pages;
  int32_t* oldp = sa.old_pages + (int64_t)it.dslot * sa.seq_pages;
  int32_t* gather = sa.gather + (int64_t)it.dslot * sa.max_slots;

  // snapshot the page ids the gather will read from
  for (int k = it.n_kept + (int)threadIdx.x; k < it.old_pages; k += blockDim.x)
    oldp[k] = pages[k];

  // gather map: new slot j <- old slot of the j-th set keep bit.  Each
  // thread owns a run of consecutive words: one block scan of the runs'
  // counts, then each run writes its entries in order.
  const int nw = (it.old_slots + 31) / 32;
  auto word = [&](int w) {
    uint32_t bits = keep[w];
    const int tail = it.old_slots - w * 32;
    if (tail < 32) bits &= (1u << tail) - 1u;
    return bits;
  };
  const int per = (nw + (int)blockDim.x - 1) / (int)blockDim.x;
  const int w0 = (int)threadIdx.x * per, w1 = min(nw, w0 + per);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(word(w));
  int j = block_exclusive_scan(cnt, s_warp, &s_total);
  for (int w = w0; w < w1; ++w) {
    uint32_t bits = word(w);
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1u;
      if (j < sa.max_slots) gather[j] = w * 32 + b;
      else flag(err, AKV_DERR_INDEX);
      ++j;
    }
  }
  if (threadIdx.x == 0 && s_total != it.r) flag(err, AKV_DERR_COUNT);
  __syncthreads();

  // new page table: kept prefix unchanged, fresh ids after, released tail
  for (int k = it.n_kept + (int)threadIdx.x; k < max(it.new_pages, it.old_pages); k += blockDim.x)
    pages[k] = k < it.new_pages ? ids[it.fresh_off + (k - it.n_kept)] : -1;
  // keep bits: exactly slots [0, r)
  for (int w = threadIdx.x; w < nw; w += blockDim.x) {
    const int n = it.r - w * 32;
    keep[w] = n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
  }
  for (int k = threadIdx.x; k < it.new_pages; k += blockDim.x) active[k] = k;
}

// ---------------------------------------------------------------------------
// reposition, part 2 (staged): one block per fresh destination page; each
// (layer, KV head) tile of the page goes through shared memory: bulk copies
// bring the source rows in (one copy per run of consecutive source slots in
// one source page), the block rotates the keys in place, and one bulk copy
// per tensor writes the page tile out.  A ring of stages keeps several
// tiles' copies in flight per block.  Survivor j moves from old slot src_j
// to j: K' = R(j - src_j) K (bit copy when j == src_j), V copied.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t sm32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               ::"l"(dst), "r"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool gwait(uint32_t bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 "selp.u32 %0, 1, 0, p;\n}\n" : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    if (ok) return true;
  }
  return false;
}

// The staged tile pipeline shared by the reposition gather and the prefix
// fork: for every (layer, KV head) tile of destination page `dpage`, rows
// t of the stage receive source rows (s_src_page[t], s_src_off[t]) through
// one bulk copy per run, keys with s_rot[t] set are rotated in place with the
// row's cos/sin (s_cs, unit-minor; their low parts read from the table's row
// s_lrow[t] of g.cs_lo when a pair nearly cancels, the sine's part times
// s_lsy[t]),
// and rows [0, n_store) go out with one
// bulk copy per tensor.  Rows without a source (dead slots of a prefix fork)
// are written as zeros, so that a stored slot never holds stale bits.  Layers
// l_begin..l_end-1 map to slab l % phys_layers.
template <typename T>
__device__ __forceinline__ void tile_pipeline(
    const Geom& g, int l_begin, int l_end, unsigned char* stage0, const float2* s_cs,
    const int* s_lrow, const float* s_lsy, const int* s_src_page,
    const int* s_src_off, const int* s_rot, const int* s_run_t0, const int* s_run_len, int n_runs,
    uint32_t bytes, int dpage, int n_store, int n_stages, uint64_t* s_full, uint32_t* err,
    uint32_t wait_limit) {
  constexpr int E = Vec<T>::E;
  const int D = g.d, RH = g.rope / 2, kr = RH / E;
  const uint32_t row_bytes = D * sizeof(T);
  const uint32_t tile_bytes = g.s * row_bytes;
  const int tid = threadIdx.x;
  const int n = (l_end - l_begin) * g.hkv;       // tiles: (layer, KV head)
  T* kp = static_cast<T*>(g.k);
  T* vp = static_cast<T*>(g.v);
  const int n_dead = __syncthreads_count(tid < n_store && s_src_page[tid] < 0);   // n_store <= 64
  auto issue = [&](int i) {                      // thread 0: loads of tile i into its stage
    const int st = i % n_stages;
    const int l = l_begin + i / g.hkv, h = i % g.hkv;
    const int64_t slab = (int64_t)(l % g.phys_layers) * g.layer_stride;
    const uint32_t bar = sm32(&s_full[st]);
    const uint32_t kd = sm32(stage0 + (size_t)st * 2 * tile_bytes), vd = kd + tile_bytes;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
    for (int r = 0; r < n_runs; ++r) {
      const int t0 = s_run_t0[r];
      const int64_t off = slab + (int64_t)s_src_page[t0] * g.page_stride + (int64_t)h * g.head_stride +
                          (int64_t)s_src_off[t0] * D;
      const uint32_t len = s_run_len[r] * row_bytes;
      bulk_load(kd + t0 * row_bytes, kp + off, len, bar);
      bulk_load(vd + t0 * row_bytes, vp + off, len, bar);
    }
  };
  int issued = 0, waited = 0;                    // thread 0: tiles issued / complete
  if (tid == 0)
    for (; issued < min(n_stages - 1, n); ++issued) issue(issued);
  bool ok = true;
  for (int i = 0; i < n; ++i) {
    const int st = i % n_stages;
    if (tid == 0 && i + n_stages - 1 < n) {
      // the stage of tile i - 1 is free once its stores have read it
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      issue(i + n_stages - 1);
      issued = i + n_stages;
    }
    ok = __syncthreads_and(gwait(sm32(&s_full[st]), (i / n_stages) & 1, wait_limit));
    if (!ok) break;
    waited = i + 1;
    T* kt = reinterpret_cast<T*>(stage0 + (size_t)st * 2 * tile_bytes);
    for (int u = tid; u < n_store * kr; u += blockDim.x) {
      const int t = u / kr, c = u % kr;
      if (!s_rot[t] || s_src_page[t] < 0) continue;
      T* row = kt + (size_t)t * D;
      const uint4 lo = *reinterpret_cast<const uint4*>(row + c * E);
      const uint4 hi = *reinterpret_cast<const uint4*>(row + RH + c * E);
      rotate_regs<T>(lo, hi, row, c, RH, s_cs + t * RH, kr,
                     s_lrow[t] >= 0 ? g.cs_lo + (int64_t)s_lrow[t] * RH : nullptr, s_lsy[t]);
    }
    if (n_dead > 0) {
      const int ch = (int)(row_bytes / 16);      // 16-byte chunks of a row
      for (int u = tid; u < n_store * ch; u += blockDim.x) {
        const int t = u / ch, c = u % ch;
        if (s_src_page[t] >= 0) continue;
        unsigned char* r = reinterpret_cast<unsigned char*>(kt) + (size_t)t * row_bytes + (size_t)c * 16;
        *reinterpret_cast<uint4*>(r) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(r + tile_bytes) = make_uint4(0, 0, 0, 0);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) {
      const int l = l_begin + i / g.hkv, h = i % g.hkv;
      const int64_t dst = (int64_t)(l % g.phys_layers) * g.layer_stride +
                          (int64_t)dpage * g.page_stride + (int64_t)h * g.head_stride;
      const uint32_t src = sm32(stage0 + (size_t)st * 2 * tile_bytes);
      bulk_store(kp + dst, src, n_store * row_bytes);
      bulk_store(vp + dst, src + tile_bytes, n_store * row_bytes);
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
  }
  if (tid == 0) {
    if (!ok) flag(err, AKV_DERR_WAIT);
    // every store has finished before the block (and its shared memory) goes;
    // loads still in flight after a failed wait land first (bounded)
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    if (!ok)
      for (int i = waited; i < issued; ++i)
        gwait(sm32(&s_full[i % n_stages]), (i / n_stages) & 1, kDrainPolls);
  }
  __syncthreads();
}

// runs of rows whose source slots are consecutive in one source page
__device__ __forceinline__ void find_runs(int n_rows, const int* s_src_page, const int* s_src_off,
                                          uint32_t row_bytes, int* s_run_t0, int* s_run_len,
                                          int* s_n_runs, uint32_t* s_bytes) {
  int nr = 0;
  uint32_t bytes = 0;
  for (int t = 0; t < n_rows; ++t) {
    if (s_src_page[t] < 0) continue;
    if (nr > 0 && s_run_t0[nr - 1] + s_run_len[nr - 1] == t && s_src_page[t] == s_src_page[t - 1] &&
        s_src_off[t] == s_src_off[t - 1] + 1) {
      ++s_run_len[nr - 1];
    } else {
      s_run_t0[nr] = t;
      s_run_len[nr] = 1;
      ++nr;
    }
    bytes += 2 * row_bytes;
  }
  *s_n_runs = nr;
  *s_bytes = bytes;
}

constexpr int kGatherThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kGatherThreads)
k_gather(Geom g, SeqArrays sa, const ReposItem* __restrict__ items, int n_items,
         const float2* __restrict__ cs, uint32_t* err, int n_stages, uint32_t wait_limit) {
  constexpr int E = Vec<T>::E;
  extern __shared__ __align__(128) unsigned char gsm[];
  const int S = g.s, D = g.d, R = g.rope, RH = R / 2;
  const uint32_t row_bytes = D * sizeof(T);
  const uint32_t tile_bytes = S * row_bytes;                 // one (layer, head) tile of one tensor
  unsigned char* stage0 = gsm;                                // [n_stages][K, V][S][D]
  float2* s_cs = reinterpret_cast<float2*>(gsm + (size_t)n_stages * 2 * tile_bytes);   // [S][R/2]
  __shared__ int s_src_page[64], s_src_off[64], s_rot[64], s_lrow[64];
  __shared__ float s_lsy[64];
  __shared__ int s_run_t0[64], s_run_len[64], s_n_runs, s_dst_page;
  __shared__ uint32_t s_bytes;
  __shared__ __align__(8) uint64_t s_full[8];

  int lo = 0, hi = n_items - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (items[mid].block0 <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
  }
  const ReposItem it = items[lo];
  const int k = it.n_kept + ((int)blockIdx.x - it.block0);
  const int j0 = k * S;
  const int nj = min(S, it.r - j0);
  const int32_t* gather = sa.gather + (int64_t)it.dslot * sa.max_slots;
  const int32_t* oldp = sa.old_pages + (int64_t)it.dslot * sa.seq_pages;
  const int tid = threadIdx.x;

  for (int t = tid; t < nj; t += kGatherThreads) {
    const int j = j0 + t;
    const int src = gather[j];
    int sp = -1;
    if (src >= j && src < it.old_slots) sp = oldp[src / S];
    if (sp < 0 || sp >= g.max_pages) { flag(err, AKV_DERR_PAGE); sp = -1; }
    s_src_page[t] = sp;
    s_src_off[t] = src % S;
    s_rot[t] = src != j;
    // the keys move down by delta = src - j: rotation by -delta
    s_lrow[t] = (src - j >= 0 && src - j < sa.max_slots) ? src - j : -1;
    s_lsy[t] = -1.f;
  }
  {
    const int kr = RH / E;
    for (int i = tid; i < nj * RH; i += kGatherThreads) {
      const int t = i / RH, jj = i % RH;
      const int delta = gather[j0 + t] - (j0 + t);
      float2 c = make_float2(1.f, 0.f);
      if (delta >= 0 && delta < sa.max_slots) c = cs[(int64_t)delta * RH + jj];
      s_cs[t * RH + (jj % E) * kr + jj / E] = make_float2(c.x, -c.y);
    }
  }
  if (tid == 0) {
    int p = (k >= 0 && k < sa.seq_pages) ? sa.pages[(int64_t)it.dslot * sa.seq_pages + k] : -1;
    if (p < 0 || p >= g.max_pages) { flag(err, AKV_DERR_PAGE); p = -1; }
    s_dst_page = p;
    for (int s = 0; s < n_stages; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sm32(&s_full[s])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tid == 0) find_runs(nj, s_src_page, s_src_off, row_bytes, s_run_t0, s_run_len, &s_n_runs, &s_bytes);
  __syncthreads();
  const int dpage = s_dst_page;
  if (dpage < 0) return;
  const int lper = (g.layers + gridDim.y - 1) / gridDim.y;    // layers of this block
  tile_pipeline<T>(g, blockIdx.y * lper, min(g.layers, (int)(blockIdx.y + 1) * lper), stage0, s_cs,
                   s_lrow, s_lsy, s_src_page, s_src_off, s_rot, s_run_t0, s_run_len, s_n_runs, s_bytes, dpage, nj,
                   n_stages, s_full, err, wait_limit);
}

// ---------------------------------------------------------------------------
// prefix fork: needed keys of a published snapshot moved into a fresh page
// of a new sequence, each rotated by its own delta = p_request - p_stored
// (bit copy when delta == 0), V copied.  One block per fresh destination
// page and its moves, through the staged tile pipeline (all physical
// layers and KV heads).  Rows of the page that no move fills are dead
// slots of the new sequence.
// ---------------------------------------------------------------------------

template <typename T>
__global__ void __launch_bounds__(kGatherThreads)
k_transplant(Geom g, const MoveItem* __restrict__ moves, int n_moves,
             const MoveBlock* __restrict__ blocks, const float2* __restrict__ cs, int max_pos,
             uint32_t* err, int n_stages, uint32_t wait_limit) {
  constexpr int E = Vec<T>::E;
  extern __shared__ __align__(128) unsigned char gsm[];
  const int S = g.s, D = g.d, RH = g.rope / 2, kr = RH / E;
  const uint32_t row_bytes = D * sizeof(T);
  const uint32_t tile_bytes = S * row_bytes;
  unsigned char* stage0 = gsm;                                // [n_stages][K, V][S][D]
  float2* s_cs = reinterpret_cast<float2*>(gsm + (size_t)n_stages * 2 * tile_bytes);   // [S][R/2]
  __shared__ int s_src_page[64], s_src_off[64], s_rot[64], s_delta[64], s_lrow[64];
  __shared__ float s_lsy[64];
  __shared__ int s_run_t0[64], s_run_len[64], s_n_runs, s_n_store;
  __shared__ uint32_t s_bytes;
  __shared__ __align__(8) uint64_t s_full[8];
  const MoveBlock mb = blocks[blockIdx.x];
  const int tid = threadIdx.x;
  if (mb.dst_page < 0 || mb.dst_page >= g.max_pages || mb.first < 0 || mb.count < 1 ||
      mb.count > S || mb.first + mb.count > n_moves) {
    if (tid == 0) flag(err, AKV_DERR_PAGE);
    return;
  }
  for (int t = tid; t < S; t += kGatherThreads) {
    s_src_page[t] = -1;
    s_src_off[t] = 0;
    s_rot[t] = 0;
    s_delta[t] = 0;
  }
  if (tid == 0) s_n_store = 0;
  __syncthreads();
  for (int m = tid; m < mb.count; m += kGatherThreads) {
    const MoveItem mv = moves[mb.first + m];
    const bool ok = mv.src_page >= 0 && mv.src_page < g.max_pages && mv.dst_page == mb.dst_page &&
                    mv.src_off >= 0 && mv.src_off < S && mv.dst_off >= 0 && mv.dst_off < S &&
                    mv.delta > -max_pos && mv.delta < max_pos;
    if (!ok) {
      flag(err, AKV_DERR_PAGE);
      continue;
    }
    s_src_page[mv.dst_off] = mv.src_page;
    s_src_off[mv.dst_off] = mv.src_off;
    s_rot[mv.dst_off] = mv.delta != 0;
    s_delta[mv.dst_off] = mv.delta;
    atomicMax(&s_n_store, mv.dst_off + 1);
  }
  __syncthreads();
  const int n_store = s_n_store;
  for (int i = tid; i < n_store * RH; i += kGatherThreads) {
    const int t = i / RH, j = i % RH;
    const int delta = s_delta[t];
    const int a = delta < 0 ? -delta : delta;
    const float2 c = a < max_pos ? cs[(int64_t)a * RH + j] : make_float2(1.f, 0.f);
    s_cs[t * RH + (j % E) * kr + j / E] = make_float2(c.x, delta < 0 ? -c.y : c.y);
  }
  for (int t = tid; t < n_store; t += kGatherThreads) {
    const int a = s_delta[t] < 0 ? -s_delta[t] : s_delta[t];
    s_lrow[t] = a < max_pos ? a : -1;
    s_lsy[t] = s_delta[t] < 0 ? -1.f : 1.f;
  }
  if (tid == 0) {
    for (int st = 0; st < n_stages; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sm32(&s_full[st])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    find_runs(n_store, s_src_page, s_src_off, row_bytes, s_run_t0, s_run_len, &s_n_runs, &s_bytes);
  }
  __syncthreads();
  const int lper = (g.phys_layers + gridDim.y - 1) / gridDim.y;   // slabs of this block
  tile_pipeline<T>(g, blockIdx.y * lper, min(g.phys_layers, (int)(blockIdx.y + 1) * lper), stage0,
                   s_cs, s_lrow, s_lsy, s_src_page, s_src_off, s_rot, s_run_t0, s_run_len, s_n_runs, s_bytes,
                   mb.dst_page, n_store, n_stages, s_full, err, wait_limit);
}

}  // namespace

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

// Layer groups per destination page.  At least enough (page, layer group)
// blocks for about 32 per SM, so small calls still fill the GPU evenly; then
// the count (up to four times that, at most one group per layer) whose
// blocks fill their last wave best: every block moves the same tiles, so a
// last wave of a few blocks runs nearly as long as a full one, against a
// block's fixed start-up of about four tiles.  `per_sm`: blocks resident per
// SM; `tiles`: (layer, head) tiles of one page over all its layers.
inline int layer_groups(int n_blocks, int n_layers, int per_sm, int tiles) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  const int g0 = std::max(1, std::min(n_layers, (32 * sms + n_blocks - 1) / n_blocks));
  const double slots = (double)std::max(1, per_sm) * sms;
  int best = g0;
  double best_cost = 0.0;
  for (int gr = g0; gr <= std::min(n_layers, 4 * g0); ++gr) {
    const double waves = (double)n_blocks * gr / slots;
    const double per_block = (double)tiles / gr;             // tiles of one block
    const double cost = std::ceil(waves) * (per_block + 4.0);
    if (gr == g0 || cost < best_cost) {
      best = gr;
      best_cost = cost;
    }
  }
  return best;
}

// Blocks of `kernel` resident per SM with `smem` bytes of dynamic shared
// memory (which it is also allowed here).
template <typename K>
int resident_blocks(K kernel, size_t smem) {
  int n = 0;
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kGatherThreads, smem) != cudaSuccess)
    return 1;
  return std::max(1, n);
}

cudaError_t launch_transplant(const Geom& g, const MoveItem* moves, int n_moves,
                              const MoveBlock* blocks, int n_blocks, const float2* cs, int max_pos,
                              uint32_t* err, uint32_t wait_limit, cudaStream_t st) {
  if (n_blocks <= 0) return cudaSuccess;
  const size_t elem = g.dtype == AKV_DTYPE_BF16 ? 2 : 4;
  const size_t tile = (size_t)g.s * g.d * elem;
  const int n_stages = (int)std::max<size_t>(2, std::min<size_t>(4, (96 << 10) / (2 * tile)));
  const size_t smem = (size_t)n_stages * 2 * tile + (size_t)g.s * (g.rope / 2) * sizeof(float2);
  const int per_sm = g.dtype == AKV_DTYPE_BF16 ? resident_blocks(k_transplant<__nv_bfloat16>, smem)
                                              : resident_blocks(k_transplant<float>, smem);
  const dim3 grid(n_blocks, layer_groups(n_blocks, g.phys_layers, per_sm, g.phys_layers * g.hkv));
  if (g.dtype == AKV_DTYPE_BF16) {
    cudaFuncSetAttribute(k_transplant<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_transplant<__nv_bfloat16><<<grid, kGatherThreads, smem, st>>>(
        g, moves, n_moves, blocks, cs, max_pos, err, n_stages, wait_limit);
  } else {
    cudaFuncSetAttribute(k_transplant<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_transplant<float><<<grid, kGatherThreads, smem, st>>>(
        g, moves, n_moves, blocks, cs, max_pos, err, n_stages, wait_limit);
  }
  return cudaGetLastError();
}

cudaError_t launch_append(const Geom& g, const SeqArrays& sa, const AppendItem* items,
                          const AppendBlock* blocks, int n_blocks, const int32_t* ids,
                          const int32_t* act, const void* k_raw, const void* v,
                          int64_t total_tokens, const float2* cs, uint32_t* err,
                          AppendLimits lim, cudaStream_t st) {
  if (n_blocks <= 0) return cudaSuccess;
  const size_t smem = (size_t)kAppendTokens * (g.rope / 2) * sizeof(float2);
  const dim3 grid(n_blocks, g.phys_layers);
  if (g.dtype == AKV_DTYPE_BF16)
    k_append<__nv_bfloat16><<<grid, 256, smem, st>>>(
        g, sa, items, blocks, ids, act, static_cast<const __nv_bfloat16*>(k_raw),
        static_cast<const __nv_bfloat16*>(v), total_tokens, cs, err, lim);
  else
    k_append<float><<<grid, 256, smem, st>>>(
        g, sa, items, blocks, ids, act, static_cast<const float*>(k_raw),
        static_cast<const float*>(v), total_tokens, cs, err, lim);
  return cudaGetLastError();
}

cudaError_t launch_copy_pages(const Geom& g, const PagePair* pairs, int n_pairs,
                              uint32_t* err, cudaStream_t st) {
  if (n_pairs <= 0) return cudaSuccess;
  dim3 grid(n_pairs, g.phys_layers);
  if (g.dtype == AKV_DTYPE_BF16)
    k_copy_pages<__nv_bfloat16><<<grid, 256, 0, st>>>(g, pairs, err);
  else
    k_copy_pages<float><<<grid, 256, 0, st>>>(g, pairs, err);
  return cudaGetLastError();
}

// Byte copy by the SMs: descriptors staged in pinned host memory (read over
// the host link) and metadata rows moved inside device memory.  The copy
// engines stay out of the caller's stream: a small engine copy queued there
// behind the caller's own bulk host-to-device traffic on another stream can
// wait for milliseconds, and the decode step behind it with it.
__global__ void k_copy_bytes(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                             int64_t n) {
  const int64_t n16 = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15)
                          ? 0 : n / 16;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t i = t0; i < n16; i += stride)
    reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
  for (int64_t i = n16 * 16 + t0; i < n; i += stride) dst[i] = src[i];
}

__global__ void k_fill_u32(uint32_t* __restrict__ dst, uint32_t v, int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) dst[i] = v;
}

namespace {
int copy_grid(int64_t units) {
  const int64_t b = (units + 255) / 256;
  return (int)std::max<int64_t>(1, std::min<int64_t>(b, 1024));
}
}  // namespace

cudaError_t launch_copy_bytes(void* dst, const void* src, size_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  k_copy_bytes<<<copy_grid((int64_t)(n + 15) / 16), 256, 0, st>>>(
      static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), (int64_t)n);
  return cudaGetLastError();
}

cudaError_t launch_fill_u32(uint32_t* dst, uint32_t v, size_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  k_fill_u32<<<copy_grid((int64_t)n), 256, 0, st>>>(dst, v, (int64_t)n);
  return cudaGetLastError();
}

cudaError_t launch_drop(const Geom& g, const SeqArrays& sa, const DropItem* items,
                        int n_items, const int32_t* ranges, uint32_t* err, cudaStream_t st) {
  if (n_items <= 0) return cudaSuccess;
  k_drop<<<n_items, 1024, 0, st>>>(g, sa, items, ranges, err);
  return cudaGetLastError();
}

cudaError_t launch_compact(const Geom& g, const SeqArrays& sa, const ReposItem* items,
                           int n_items, const int32_t* ids, uint32_t* err, cudaStream_t st) {
  if (n_items <= 0) return cudaSuccess;
  k_compact<<<n_items, 1024, 0, st>>>(g, sa, items, ids, err);
  return cudaGetLastError();
}

cudaError_t launch_gather(const Geom& g, const SeqArrays& sa, const ReposItem* items,
                          int n_items, int n_blocks, const float2* cs, uint32_t* err,
                          uint32_t wait_limit, cudaStream_t st) {
  if (n_blocks <= 0) return cudaSuccess;
  const size_t elem = g.dtype == AKV_DTYPE_BF16 ? 2 : 4;
  const size_t tile = (size_t)g.s * g.d * elem;             // one (layer, head) tile, one tensor
  const int n_stages = (int)std::max<size_t>(2, std::min<size_t>(4, (96 << 10) / (2 * tile)));
  const size_t smem = (size_t)n_stages * 2 * tile + (size_t)g.s * (g.rope / 2) * sizeof(float2);
  const int per_sm = g.dtype == AKV_DTYPE_BF16 ? resident_blocks(k_gather<__nv_bfloat16>, smem)
                                              : resident_blocks(k_gather<float>, smem);
  const dim3 grid(n_blocks, layer_groups(n_blocks, g.layers, per_sm, g.layers * g.hkv));
  if (g.dtype == AKV_DTYPE_BF16) {
    cudaFuncSetAttribute(k_gather<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_gather<__nv_bfloat16><<<grid, kGatherThreads, smem, st>>>(g, sa, items, n_items, cs, err,
                                                               n_stages, wait_limit);
  } else {
    cudaFuncSetAttribute(k_gather<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_gather<float><<<grid, kGatherThreads, smem, st>>>(g, sa, items, n_items, cs, err,
                                                       n_stages, wait_limit);
  }
  return cudaGetLastError();
}

}  // namespace akv
