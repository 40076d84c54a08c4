// Segment-batch restore attention ("Cache Engineering for Agents" paper
// review, 4.2.2 Drop-aware Cache Management, 4.2.3 Reposition-aware Cache
// Management, Appendix A.1.1 Restore with Segment-batch Attention).
//
// A restore recomputes all tokens of an operation program in one forward.
// Per layer, every appended token's query must see exactly the keys it saw
// when it was appended -- keys dropped later included -- at the positions of
// that time.  The host splits the program into eras at repositions; inside
// an era the held tokens sit at fixed slots (= positions).  Each era's keys
// are materialised once as a temporary version (K rotated to the era
// position, V copied); a query x at time t(x) reads key k of its era iff
// birth(k) <= t(x) < death(k), which also makes the attention causal.
#include <algorithm>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "akv.h"
#include "akv_internal.h"
#include "akv_tc.cuh"

namespace akv {
namespace {

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ void from_f(float x, __nv_bfloat16* p) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void from_f(float x, float* p) { *p = x; }

// Temporary key versions: row r = token tok at era position pos.
//   K_era[r] = R(pos) k_raw[tok] (fp32, rounded to T), V_era[r] = v[tok].
template <typename T>
__global__ void __launch_bounds__(256)
k_restore_keys(Geom g, const RestoreKey* __restrict__ keys, int n_keys,
               const T* __restrict__ k_raw, const T* __restrict__ v, T* __restrict__ k_era,
               T* __restrict__ v_era, int n_tokens, const float2* __restrict__ cs, int max_pos,
               uint32_t* err) {
  const int D = g.d, R = g.rope, RH = R / 2, H = g.hkv;
  const int64_t per_key = (int64_t)H * D;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)n_keys * H * D;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / per_key);
    const int e = (int)(i % per_key);
    const int d = e % D;
    const RestoreKey kk = keys[r];
    if (kk.tok < 0 || kk.tok >= n_tokens || kk.pos < 0 || kk.pos >= max_pos) {
      if (d == 0) atomicOr(err, AKV_DERR_INDEX);
      continue;
    }
    const T* src = k_raw + (int64_t)kk.tok * per_key + (e - d);
    float val;
    if (d < RH) {
      const float2 t = cs[(int64_t)kk.pos * RH + d];
      val = fmaf(to_f(src[d]), t.x, -to_f(src[d + RH]) * t.y);
    } else if (d < R) {
      const float2 t = cs[(int64_t)kk.pos * RH + d - RH];
      val = fmaf(to_f(src[d - RH]), t.y, to_f(src[d]) * t.x);
    } else {
      val = to_f(src[d]);
    }
    from_f(val, k_era + (int64_t)r * per_key + e);
    v_era[(int64_t)r * per_key + e] = v[(int64_t)kk.tok * per_key + e];
  }
}

constexpr int kWarps = 4;

// Generic attention of one query token (all heads of one KV group) over its
// era's keys, with the interval mask; CUDA cores, any dtype, G <= 16.
template <typename T, int D, int G>
__global__ void __launch_bounds__(kWarps * 32)
k_restore_attn_simple(Geom g, const RestoreQuery* __restrict__ queries,
                      const RestoreKey* __restrict__ keys, const T* __restrict__ q,
                      const T* __restrict__ k_era, const T* __restrict__ v_era, float* __restrict__ out,
                      const float2* __restrict__ cs, int max_pos, float scale_log2, int window,
                      uint32_t* err) {
  constexpr int J = D / 32;
  __shared__ float s_q[G][D];
  __shared__ float s_m[kWarps][G], s_l[kWarps][G];
  __shared__ float s_acc[kWarps][G][D];
  const RestoreQuery qq = queries[blockIdx.x];
  const int kvh = blockIdx.y, H = g.hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = g.rope, RH = R / 2;
  const bool ok = qq.pos >= 0 && qq.pos < max_pos;
  if (!ok && tid == 0) atomicOr(err, AKV_DERR_INDEX);
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int gq = i / D, d = i % D;
    const T* qr = q + ((int64_t)qq.tok * g.hq + (int64_t)kvh * G + gq) * D;
    if (!ok) {
      s_q[gq][d] = 0.f;
    } else if (d < RH) {
      const float2 t = cs[(int64_t)qq.pos * RH + d];
      const float x = to_f(qr[d]), y = to_f(qr[d + RH]);
      s_q[gq][d] = fmaf(x, t.x, -y * t.y) * scale_log2;
      s_q[gq][d + RH] = fmaf(x, t.y, y * t.x) * scale_log2;
    } else if (d >= R) {
      s_q[gq][d] = to_f(qr[d]) * scale_log2;
    }
  }
  __syncthreads();
  float m[G], l[G], acc[G][J];
#pragma unroll
  for (int gq = 0; gq < G; ++gq) {
    m[gq] = -INFINITY; l[gq] = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) acc[gq][j] = 0.f;
  }
  const int lo = window > 0 ? max(0, qq.pos - window + 1) : 0;
  for (int j = lo + warp; j < qq.key_end && ok; j += kWarps) {
    const RestoreKey kk = keys[qq.era_off + j];
    if (!(kk.birth <= qq.time && qq.time < kk.death)) continue;
    const T* kr = k_era + ((int64_t)(qq.era_off + j) * H + kvh) * D;
    const T* vr = v_era + ((int64_t)(qq.era_off + j) * H + kvh) * D;
    float kd[J], vd[J];
#pragma unroll
    for (int jj = 0; jj < J; ++jj) { kd[jj] = to_f(kr[lane + 32 * jj]); vd[jj] = to_f(vr[lane + 32 * jj]); }
#pragma unroll
    for (int gq = 0; gq < G; ++gq) {
      float part = 0.f;
#pragma unroll
      for (int jj = 0; jj < J; ++jj) part = fmaf(s_q[gq][lane + 32 * jj], kd[jj], part);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      const float mn = fmaxf(m[gq], part);
      const float alpha = exp2f(m[gq] - mn);
      const float w = exp2f(part - mn);
      l[gq] = fmaf(l[gq], alpha, w);
#pragma unroll
      for (int jj = 0; jj < J; ++jj) acc[gq][jj] = fmaf(acc[gq][jj], alpha, w * vd[jj]);
      m[gq] = mn;
    }
  }
#pragma unroll
  for (int gq = 0; gq < G; ++gq) {
    if (lane == 0) { s_m[warp][gq] = m[gq]; s_l[warp][gq] = l[gq]; }
#pragma unroll
    for (int jj = 0; jj < J; ++jj) s_acc[warp][gq][lane + 32 * jj] = acc[gq][jj];
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int gq = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][gq]);
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(s_m[w][gq] - M);
        L = fmaf(s_l[w][gq], f, L);
        A = fmaf(s_acc[w][gq][d], f, A);
      }
    }
    out[((int64_t)qq.tok * g.hq + kvh * G + gq) * D + d] = L > 0.f ? A / L : 0.f;
  }
}

template <typename T, int D>
cudaError_t launch_simple_g(const RestoreArgs& a, int G, cudaStream_t st) {
  const dim3 grid(a.n_queries, a.g.hkv);
  const T* q = static_cast<const T*>(a.q);
  const T* ke = static_cast<const T*>(a.k_era);
  const T* ve = static_cast<const T*>(a.v_era);
#define AKV_RESTORE_CASE(GG)                                                                    \
  case GG:                                                                                      \
    k_restore_attn_simple<T, D, GG><<<grid, kWarps * 32, 0, st>>>(                               \
        a.g, a.queries, a.keys, q, ke, ve, a.out, a.cs, a.max_pos, a.scale_log2, a.window, a.err); \
    break;
  switch (G) {
    AKV_RESTORE_CASE(1)
    AKV_RESTORE_CASE(2)
    AKV_RESTORE_CASE(4)
    AKV_RESTORE_CASE(8)
    AKV_RESTORE_CASE(16)
    default: return cudaErrorInvalidValue;
  }
#undef AKV_RESTORE_CASE
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Tensor-core path (bf16, D in {64, 128}): tcgen05 UMMA with accumulators in
// tensor memory.  One CTA = 128 query rows (TT tokens x NH heads of one KV
// group, NH = min(G, 8)); TMEM lane r holds row r.  Per 64-key tile:
//   S = Q K^T      M=128, N=64, K=D    -> one of two S buffers in TMEM
//   softmax        tcgen05.ld of the S row, interval mask, online max/sum,
//                  P (bf16 pairs) written back over S with tcgen05.st, O
//                  rescaled in TMEM when the reference max moves
//   O += P V       M=128, N=D,  K=64, A = P from TMEM -> TMEM after the S
//                  buffers
// Q, K and V live in shared memory in the 128-byte swizzled layout (rows of
// 128 bytes, 16-byte chunk c of row r at c ^ (r % 8), 64-element atoms of
// rows*128 bytes): Q and K K-major, V (the same bytes as K's layout) read
// MN-major.  A load warp issues the TMA copies and loads the keys' death
// times, an MMA warp issues the MMAs (each from one thread, so that neither
// waits behind the other's issue); four softmax warps, one per TMEM lane
// quarter, each thread owning a whole query row (all 64 scores of a tile:
// no exchange between warps for the row maximum).  Hand-offs are bounded
// mbarrier waits.  Two CTAs share an SM (about 100 KB of shared memory and
// 256 TMEM columns each for D = 128).
// ---------------------------------------------------------------------------

constexpr int kBM = 128;   // query rows per CTA
constexpr int kBN = 64;    // keys per tile


// TMEM columns: two S buffers (kBN each) and O (D), rounded to a power of 2
template <int D>
__host__ __device__ constexpr int restore_tc_cols() { return 256; }
static_assert(2 * kBN + 128 <= 256, "S buffers and O must fit the TMEM allocation");
template <int D>
constexpr size_t restore_tc_smem() {
  return 1024 /* alignment slack */ + (size_t)kBM * D * 2 + 4 * (size_t)kBN * D * 2 +
         2 * kBN * sizeof(int) + 4 * sizeof(int) + 12 * sizeof(uint64_t) + 16;
}

// softmax warps: warp w reads TMEM lanes 32 w .. 32 w + 31 (its rows), all
// columns of every S tile and of O.  (Eight warps, two per lane quarter
// splitting the keys and exchanging row maxima through shared memory, ran at
// 865 against 894 TFLOP/s on the 8B-shaped restore workload.)
constexpr int kSoftmaxWarps = 4;
constexpr int kMmaWarp = kSoftmaxWarps;                     // issues the MMAs (one thread)
constexpr int kLoadWarp = kSoftmaxWarps + 1;                // copies, key deaths
constexpr int kRestoreThreads = 32 * (kSoftmaxWarps + 2);

template <int D, int NH>
__global__ void __launch_bounds__(kRestoreThreads, 2)
k_restore_attn_tc(const __grid_constant__ RestoreArgs a) {
  constexpr int NCOL = restore_tc_cols<D>();
  constexpr uint32_t KV_BYTES = kBN * D * 2;     // one tile of K (or V)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm;                           // kBM x D (K-major)
  uint8_t* sK = sQ + kBM * D * 2;             // [2] kBN x D, TMA 64-element atoms
  uint8_t* sV = sK + 2 * kBN * D * 2;         // [2] same layout, read MN-major
  int* s_death = reinterpret_cast<int*>(sV + 2 * kBN * D * 2);   // [2][kBN]
  int* s_dmin = s_death + 2 * kBN;                                // [2]
  volatile int* s_abort = s_dmin + 2;
  // S[2] O[2] K[2] V[2] P[2] D[2]
  uint64_t* mbar = reinterpret_cast<uint64_t*>(s_dmin + 4);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 12);

  const RestoreTile tl = a.tiles[blockIdx.x];
  const int kvh = blockIdx.y;
  const int G = a.g.hq / a.g.hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool control = warp == kMmaWarp, loader = warp == kLoadWarp;
  const int tend = tl.tok0 + tl.n_tok;
  const int R = a.g.rope, RH = R / 2;
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);

  // rotated, scaled Q rows: row = token * NH + head
  for (int i = tid; i < kBM * (D / 2); i += kRestoreThreads) {
    const int row = i / (D / 2), d = i % (D / 2);
    const int t = tl.tok0 + row / NH;
    const int hq = kvh * G + blockIdx.z * NH + row % NH;
    float x = 0.f, y = 0.f;
    int dx, dy;
    if (d < RH) { dx = d; dy = d + RH; }
    else { dx = R + 2 * (d - RH); dy = dx + 1; }
    if (t < tend) {
      const RestoreQuery qq = a.queries[t];
      if (qq.pos >= 0 && qq.pos < a.max_pos) {
        const __nv_bfloat16* qr = qg + ((int64_t)t * a.g.hq + hq) * D;
        if (d < RH) {
          const float2 c = a.cs[(int64_t)qq.pos * RH + d];
          const float qx = __bfloat162float(qr[dx]), qy = __bfloat162float(qr[dy]);
          x = fmaf(qx, c.x, -qy * c.y) * a.scale_log2;
          y = fmaf(qx, c.y, qy * c.x) * a.scale_log2;
        } else {
          x = __bfloat162float(qr[dx]) * a.scale_log2;
          y = __bfloat162float(qr[dy]) * a.scale_log2;
        }
      } else if (d == 0 && row % NH == 0) {
        atomicOr(a.err, AKV_DERR_INDEX);
      }
    }
    *(reinterpret_cast<__nv_bfloat16*>(sQ + sw128(row, dx / 8, kBM)) + dx % 8) = __float2bfloat16_rn(x);
    *(reinterpret_cast<__nv_bfloat16*>(sQ + sw128(row, dy / 8, kBM)) + dy % 8) = __float2bfloat16_rn(y);
  }
  const uint32_t mbS0 = smem_u32(mbar), mbO0 = smem_u32(mbar + 2), mbK0 = smem_u32(mbar + 4),
                 mbV0 = smem_u32(mbar + 6), mbP0 = smem_u32(mbar + 8), mbD0 = smem_u32(mbar + 10);
  if (control) {
    if (lane == 0) {
      for (int i = 0; i < 12; ++i) {
        // P: one arrival per softmax warp
        const uint32_t cnt = (i == 8 || i == 9) ? kSoftmaxWarps : 1;
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(mbar + i)), "r"(cnt) : "memory");
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      *s_abort = 0;
    }
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tslot)), "r"(NCOL) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  proxy_fence();
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tbase = *tslot;
  const uint32_t tO = tbase + 2 * kBN;                          // S buffers at 0 and kBN
  const int n_kt = (tl.key_hi - tl.key_lo + kBN - 1) / kBN;
  auto fail = [&]() {
    *s_abort = 1;
    atomicOr(a.err, AKV_DERR_WAIT);
  };

  float m_r = -INFINITY, l_r = 0.f;
  int t_r = 0;
  if (loader) {
    // ---- load warp: K(kt + 2) and the key deaths of kt + 2 once softmax(kt)
    // is done, V(kt + 2) once PV(kt) is done (lane 0 issues the copies) ----
    int k_pend[2] = {-1, -1}, v_pend[2] = {-1, -1};
    auto tma_k = [&](int kt) {
      const int b = kt & 1;
      mbar_expect_tx(mbK0 + 8 * b, KV_BYTES);
#pragma unroll
      for (int at = 0; at < D / 64; ++at)
        tma_load_3d(smem_u32(sK + b * kBN * D * 2 + at * kBN * 128), &a.tm_k, at * 64, kvh,
                    tl.era_off + tl.key_lo + kt * kBN, mbK0 + 8 * b);
      k_pend[b] = kt;
    };
    auto tma_v = [&](int kt) {
      const int b = kt & 1;
      mbar_expect_tx(mbV0 + 8 * b, KV_BYTES);
#pragma unroll
      for (int at = 0; at < D / 64; ++at)
        tma_load_3d(smem_u32(sV + b * kBN * D * 2 + at * kBN * 128), &a.tm_v, at * 64, kvh,
                    tl.era_off + tl.key_lo + kt * kBN, mbV0 + 8 * b);
      v_pend[b] = kt;
    };
    // whole warp: deaths of tile kt (loaded early into registers, stored
    // once the buffer is free) and their minimum
    auto fetch_deaths = [&](int kt, int* dd) {
#pragma unroll
      for (int h = 0; h < kBN / 32; ++h) {
        const int j = tl.key_lo + kt * kBN + lane + 32 * h;
        dd[h] = (kt < n_kt && j < tl.key_hi) ? a.keys[tl.era_off + j].death : 0;
      }
    };
    auto store_deaths = [&](int kt, const int* dd) {
      const int b = kt & 1;
      int mn = INT32_MAX;
#pragma unroll
      for (int h = 0; h < kBN / 32; ++h) {
        s_death[b * kBN + lane + 32 * h] = dd[h];
        mn = min(mn, dd[h]);
      }
      mn = __reduce_min_sync(0xffffffffu, mn);
      if (lane == 0) s_dmin[b] = mn;
      __syncwarp();
      if (lane == 0) mbar_arrive(mbD0 + 8 * b);
    };
    auto deaths = [&](int kt) {
      int dd[kBN / 32];
      fetch_deaths(kt, dd);
      store_deaths(kt, dd);
    };
    bool ok = true;
    if (n_kt > 0) {
      if (lane == 0) {
        tma_k(0);
        tma_v(0);
        if (n_kt > 1) { tma_k(1); tma_v(1); }
      }
      deaths(0);
      if (n_kt > 1) deaths(1);
    }
    for (int kt = 0; kt + 2 < n_kt; ++kt) {
      const int b = kt & 1;
      ok = __shfl_sync(0xffffffffu, ok, 0) && !*s_abort;
      if (!ok) break;
      int dnext[kBN / 32];
      fetch_deaths(kt + 2, dnext);      // in flight while lane 0 waits
      if (lane == 0) {
        // softmax of tile kt done: S(kt) has read K buffer b, deaths(kt) consumed
        ok = mbar_wait(mbP0 + 8 * b, (kt >> 1) & 1, a.wait_limit);
        if (ok) tma_k(kt + 2);
        else fail();
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      store_deaths(kt + 2, dnext);
      if (lane == 0) {
        // PV(kt) has read V buffer b
        ok = mbar_wait(mbO0 + 8 * b, (kt >> 1) & 1, a.wait_limit);
        if (ok) tma_v(kt + 2);
        else fail();
      }
    }
    if (lane == 0 && *s_abort) {
      // this warp's copies land before the CTA's memory goes (bounded by a
      // fixed limit, independent of the user's wait limit)
      for (int b = 0; b < 2; ++b) {
        if (k_pend[b] >= 0) mbar_wait(mbK0 + 8 * b, (k_pend[b] >> 1) & 1, kDrainPolls);
        if (v_pend[b] >= 0) mbar_wait(mbV0 + 8 * b, (v_pend[b] >> 1) & 1, kDrainPolls);
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
    const uint64_t dv = sdesc(smem_u32(sV), kBN * 128, 1024);
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
      ok = mbar_wait(mbK0, 0, a.wait_limit);
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
            ok = mbar_wait(mbO0 + 8 * (b ^ 1), ((kt - 1) >> 1) & 1, a.wait_limit);
            if (ok) o_pend[b ^ 1] = -1;
          }
          if (ok) ok = mbar_wait(mbK0 + 8 * (b ^ 1), ((kt + 1) >> 1) & 1, a.wait_limit);
          if (ok) {
            tc_after();
            issue_s(kt + 1);
          }
        }
        // O += P(kt) V(kt) once the softmax of kt is done and V(kt) is in
        if (ok) ok = mbar_wait(mbP0 + 8 * b, (kt >> 1) & 1, a.wait_limit);
        if (ok) {
          s_pend = s_pend == kt ? -1 : s_pend;
          ok = mbar_wait(mbV0 + 8 * b, (kt >> 1) & 1, a.wait_limit);
        }
        if (ok) {
          tc_after();
          const uint64_t vb = dv + (uint64_t)((b * kBN * D * 2) >> 4);
          const uint32_t tSb = tbase + b * kBN;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            umma_ts(tO, tSb + kk * 8, vb + (uint64_t)((kk * 16 * 128) >> 4), id_o, kt > 0 || kk > 0);
          umma_commit(mbO0 + 8 * b);
          o_pend[b] = kt;
        } else {
          fail();
        }
      }
    }
    if (lane == 0 && *s_abort) {
      // this warp's MMAs finish before the CTA's memory goes (bounded)
      if (s_pend >= 0) mbar_wait(mbS0 + 8 * (s_pend & 1), (s_pend >> 1) & 1, kDrainPolls);
      for (int b = 0; b < 2; ++b)
        if (o_pend[b] >= 0) mbar_wait(mbO0 + 8 * b, (o_pend[b] >> 1) & 1, kDrainPolls);
    }
    __syncwarp();
  } else {
    // ---- softmax warps: row = TMEM lane, all of its scores and O columns ----
    const int row = 32 * warp + lane;
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    // key j is visible iff lo_r <= j < kend_r and the key is still alive at
    // time_r (keys are born in slot order: "born by time_r" is j < kend_r);
    // padding rows see nothing
    int time_r = -1, lo_r = 0, kend_r = 0;
    t_r = tl.tok0 + row / NH;
    if (t_r < tend) {
      const RestoreQuery qq = a.queries[t_r];
      if (qq.pos >= 0 && qq.pos < a.max_pos) {
        time_r = qq.time;
        kend_r = qq.key_end;
        lo_r = a.window > 0 ? max(0, qq.pos - a.window + 1) : 0;
      }
    }
    const bool real = t_r < tend;
    const int w_kend = __reduce_min_sync(0xffffffffu, real ? kend_r : INT32_MAX);
    const int w_lo = __reduce_max_sync(0xffffffffu, real ? lo_r : INT32_MIN);
    const int w_time = __reduce_max_sync(0xffffffffu, real ? time_r : INT32_MIN);
    for (int kt = 0; kt < n_kt; ++kt) {
      const int b = kt & 1;
      const int k0 = tl.key_lo + kt * kBN;
      const uint32_t tSb = tbase + b * kBN;
      bool ok = mbar_wait(mbD0 + 8 * b, (kt >> 1) & 1, a.wait_limit) &&
                mbar_wait(mbS0 + 8 * b, (kt >> 1) & 1, a.wait_limit);
      ok = __all_sync(0xffffffffu, ok) && !*s_abort;
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_after();
      uint32_t sr[kBN];
#pragma unroll
      for (int u = 0; u < kBN / 32; ++u) tmem_ld32(tSb + lane_off + 32 * u, sr + 32 * u);
      tmem_wait_ld();
      const int* de = s_death + b * kBN;
      const bool full = k0 >= w_lo && k0 + kBN <= w_kend && s_dmin[b] > w_time;   // warp-uniform
      float sv[kBN];
      if (full) {
#pragma unroll
        for (int c = 0; c < kBN; ++c) sv[c] = __uint_as_float(sr[c]);
      } else {
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
          const int j = k0 + c;
          const bool vis = j >= lo_r && j < kend_r && de[c] > time_r;
          sv[c] = vis ? __uint_as_float(sr[c]) : -INFINITY;
        }
      }
      // the row maximum in four independent chains (a short dependence path)
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < kBN; c += 8)
#pragma unroll
        for (int u = 0; u < 4; ++u) m4[u] = fmax3(m4[u], sv[c + 2 * u], sv[c + 2 * u + 1]);
      const float mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
      // the reference max moves only when the row max grows by more than 2^8
      const float m_new = (mx > m_r + 8.f) ? mx : m_r;
      const float alpha = m_new == -INFINITY ? 1.f : ex2(m_r - m_new);
      const float msub = m_new == -INFINITY ? 0.f : m_new;
      // pairs of scores in packed f32x2 arithmetic: s - m, then the sums
      uint64_t ps2[2] = {0, 0};   // two accumulators (a short dependence path)
      const uint64_t neg_m = pack_f32x2(-msub, -msub);
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int c = 0; c < kBN; c += 2) {
        float d0, d1;
        unpack_f32x2(add_f32x2(pack_f32x2(sv[c], sv[c + 1]), neg_m), d0, d1);
        const float p0 = ex2(d0), p1 = ex2(d1);
        ps2[(c / 2) & 1] = add_f32x2(ps2[(c / 2) & 1], pack_f32x2(p0, p1));
        pk[c / 2] = pack_bf16x2(p0, p1);
      }
      float ps_lo, ps_hi;
      unpack_f32x2(add_f32x2(ps2[0], ps2[1]), ps_lo, ps_hi);
      l_r = fmaf(l_r, alpha, ps_lo + ps_hi);
      m_r = m_new;
#pragma unroll
      for (int u = 0; u < kBN / 32; ++u)   // P(kt) over S(kt)
        tmem_st16(tSb + lane_off + 16 * u, pk + 16 * u);
      if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O is stable once PV(kt-1) is done: rescale the row
        const bool okv = __all_sync(0xffffffffu, mbar_wait(mbO0 + 8 * ((kt - 1) & 1), ((kt - 1) >> 1) & 1,
                                                           a.wait_limit));
        if (!okv) {
          if (lane == 0) fail();
          break;
        }
        tc_after();
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + lane_off + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + lane_off + c, o);
        }
      }
      tmem_wait_st();
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(mbP0 + 8 * b);
    }
    // the last PV
    if (n_kt > 0 && !*s_abort) {
      const bool okv = __all_sync(0xffffffffu, mbar_wait(mbO0 + 8 * ((n_kt - 1) & 1),
                                                         ((n_kt - 1) >> 1) & 1, a.wait_limit));
      if (!okv && lane == 0) fail();
    }
  }
  tc_before();
  __syncthreads();
  tc_after();
  if (warp < kSoftmaxWarps && n_kt > 0 && !*s_abort) {
    // epilogue: the row of O / l (l_r: this thread's row sum)
    const int row = 32 * warp + lane;
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const int hq = kvh * G + blockIdx.z * NH + row % NH;
    float* po = a.out + ((int64_t)t_r * a.g.hq + hq) * D;
    const float inv = l_r > 0.f ? 1.f / l_r : 0.f;
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      uint32_t o[32];
      tmem_ld32(tO + lane_off + c, o);
      tmem_wait_ld();
      if (t_r < tend) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(po + c + e) =
              make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                          __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
      }
    }
  }
  tc_before();
  __syncthreads();
  if (control)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(NCOL) : "memory");
}

// ---------------------------------------------------------------------------
// Two query tiles per CTA (one CTA per SM): consecutive 128-row tiles A and B
// of one era walk the union of their key ranges in 128-key tiles, so that
// one tile's softmax runs while the tensor pipe works on the other's
// products.  TMEM (512 columns): S_A, S_B (128 each), O_A, O_B (D each).
// Warps: 0-3 softmax of A, 4-7 softmax of B (warp w reads TMEM lanes
// 32 (w % 4) .. +31: its rows), 8 issues the MMAs (one thread), 9 the copies
// and the keys' death times.  Per key tile j the MMA thread issues
//
//   PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
//
// each after its inputs are ready.  S_X(j+1) overwrites the columns from
// which PV_X(j), issued just before it by the same thread, reads P_X(j):
// tcgen05.mma operations of one thread are performed in issue order, so no
// wait is needed between the two (the parity tests would show a hazard as
// wrong numbers).  K(j+2) goes into K(j)'s buffer once S_A(j) and S_B(j)
// have completed, V(j+2) into V(j)'s once PV_A(j) and PV_B(j) have.  A tile
// with no partner (the last of an era, odd count) runs as A alone.
// ---------------------------------------------------------------------------

constexpr int kBN2 = 128;                 // keys per tile
constexpr int kGroupWarps = 4;            // softmax warps per query tile
constexpr int kMmaWarp2 = 2 * kGroupWarps;
constexpr int kLoadWarp2 = kMmaWarp2 + 1;
constexpr int kRestoreThreads2 = 32 * (kLoadWarp2 + 1);
constexpr int kCols2 = 512;
static_assert(2 * kBN2 + 2 * 128 <= kCols2, "S_A, S_B, O_A, O_B must fit the TMEM allocation");

template <int D>
constexpr size_t restore_tc2_smem() {
  return 1024 /* alignment slack */ + 2 * (size_t)kBM * D * 2 + 4 * (size_t)kBN2 * D * 2 +
         2 * kBN2 * sizeof(int) + 4 * sizeof(int) + 19 * sizeof(uint64_t) + 16;
}

template <int D, int NH>
// 320 threads, one CTA per SM: the register file is split between the SM's
// four sub-partitions, and with ten warps one of them holds three, so a
// thread may have at most 168 registers
__global__ void __launch_bounds__(kRestoreThreads2, 1)
k_restore_attn_tc2(const __grid_constant__ RestoreArgs a) {
  constexpr uint32_t KV_BYTES = kBN2 * D * 2;    // one tile of K (or V)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm;                              // [2 tiles] kBM x D (K-major)
  uint8_t* sK = sQ + 2 * kBM * D * 2;            // [2] kBN2 x D, 64-element atoms of 128 rows
  uint8_t* sV = sK + 2 * kBN2 * D * 2;           // [2] same layout, read MN-major
  int* s_death = reinterpret_cast<int*>(sV + 2 * kBN2 * D * 2);   // [2][kBN2]
  int* s_dmin = s_death + 2 * kBN2;                                // [2]
  volatile int* s_abort = s_dmin + 2;
  // K[2] V[2] D[2] Kf[2] Vf[2] S[A,B] P[A][2] P[B][2] O[A,B], and one for the
  // drain.  P has one barrier per tile and buffer (tiles b, b + 2, ...): a
  // waiter on the phase of tile kt can then never see the barrier two
  // phases further (that would need K(kt + 2), which the waiter itself loads)
  uint64_t* mbar = reinterpret_cast<uint64_t*>(s_dmin + 4);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 19);

  const int2 pr = a.pairs[blockIdx.x];
  const RestoreTile tA = a.tiles[pr.x];
  const bool hasB = pr.y >= 0;
  const RestoreTile tB = hasB ? a.tiles[pr.y] : tA;
  const int kvh = blockIdx.y;
  const int G = a.g.hq / a.g.hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool control = warp == kMmaWarp2, loader = warp == kLoadWarp2;
  const int R = a.g.rope, RH = R / 2;
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
  // the union of the two tiles' key ranges (B follows A in the same era)
  const int key_lo = hasB ? min(tA.key_lo, tB.key_lo) : tA.key_lo;
  const int key_hi = hasB ? max(tA.key_hi, tB.key_hi) : tA.key_hi;
  bool bad = tA.era_off < 0 || (hasB && tB.era_off != tA.era_off) || key_hi < key_lo;
  if (bad) {
    if (tid == 0) atomicOr(a.err, AKV_DERR_INDEX);
    return;
  }

  // rotated, scaled Q rows of both tiles: row = token * NH + head
  for (int i = tid; i < 2 * kBM * (D / 2); i += kRestoreThreads2) {
    const int x = i / (kBM * (D / 2));
    const int row = (i / (D / 2)) % kBM, d = i % (D / 2);
    const RestoreTile& tl = x == 0 ? tA : tB;
    const int t = tl.tok0 + row / NH;
    const int hq = kvh * G + blockIdx.z * NH + row % NH;
    float xv = 0.f, yv = 0.f;
    int dx, dy;
    if (d < RH) { dx = d; dy = d + RH; }
    else { dx = R + 2 * (d - RH); dy = dx + 1; }
    if ((x == 0 || hasB) && t < tl.tok0 + tl.n_tok) {
      const RestoreQuery qq = a.queries[t];
      if (qq.pos >= 0 && qq.pos < a.max_pos) {
        const __nv_bfloat16* qr = qg + ((int64_t)t * a.g.hq + hq) * D;
        if (d < RH) {
          const float2 c = a.cs[(int64_t)qq.pos * RH + d];
          const float qx = __bfloat162float(qr[dx]), qy = __bfloat162float(qr[dy]);
          xv = fmaf(qx, c.x, -qy * c.y) * a.scale_log2;
          yv = fmaf(qx, c.y, qy * c.x) * a.scale_log2;
        } else {
          xv = __bfloat162float(qr[dx]) * a.scale_log2;
          yv = __bfloat162float(qr[dy]) * a.scale_log2;
        }
      } else if (d == 0 && row % NH == 0) {
        atomicOr(a.err, AKV_DERR_INDEX);
      }
    }
    uint8_t* qx = sQ + x * kBM * D * 2;
    *(reinterpret_cast<__nv_bfloat16*>(qx + sw128(row, dx / 8, kBM)) + dx % 8) = __float2bfloat16_rn(xv);
    *(reinterpret_cast<__nv_bfloat16*>(qx + sw128(row, dy / 8, kBM)) + dy % 8) = __float2bfloat16_rn(yv);
  }
  const uint32_t mbK0 = smem_u32(mbar), mbV0 = smem_u32(mbar + 2), mbD0 = smem_u32(mbar + 4),
                 mbKf0 = smem_u32(mbar + 6), mbVf0 = smem_u32(mbar + 8), mbS0 = smem_u32(mbar + 10),
                 mbP0 = smem_u32(mbar + 12), mbO0 = smem_u32(mbar + 16);
  if (control) {
    if (lane == 0) {
      for (int i = 0; i < 19; ++i) {
        // P: one arrival per softmax warp of the tile
        const uint32_t cnt = (i >= 12 && i < 16) ? kGroupWarps : 1;
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(mbar + i)), "r"(cnt) : "memory");
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      *s_abort = 0;
    }
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tslot)), "r"(kCols2) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  proxy_fence();
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tbase = *tslot;
  // TMEM columns: S_A at 0, S_B at kBN2, O_A at 2 kBN2, O_B at 2 kBN2 + 128
  const int n_kt = (key_hi - key_lo + kBN2 - 1) / kBN2;
  auto fail = [&]() {
    *s_abort = 1;
    atomicOr(a.err, AKV_DERR_WAIT);
  };

  float m_r = -INFINITY, l_r = 0.f;
  int t_r = 0;
  if (loader) {
    // ---- load warp (lane 0 issues the copies; the whole warp the deaths) ----
    int k_pend[2] = {-1, -1}, v_pend[2] = {-1, -1};
    auto tma_kv = [&](int kt, bool is_k) {
      const int b = kt & 1;
      const uint32_t bar = (is_k ? mbK0 : mbV0) + 8 * b;
      uint8_t* dst = (is_k ? sK : sV) + b * kBN2 * D * 2;
      mbar_expect_tx(bar, KV_BYTES);
#pragma unroll
      for (int at = 0; at < D / 64; ++at)
#pragma unroll
        for (int hlf = 0; hlf < kBN2 / 64; ++hlf)
          tma_load_3d(smem_u32(dst + at * kBN2 * 128 + hlf * 64 * 128), is_k ? &a.tm_k : &a.tm_v,
                      at * 64, kvh, tA.era_off + key_lo + kt * kBN2 + hlf * 64, bar);
      (is_k ? k_pend : v_pend)[b] = kt;
    };
    auto fetch_deaths = [&](int kt, int* dd) {
#pragma unroll
      for (int h = 0; h < kBN2 / 32; ++h) {
        const int j = key_lo + kt * kBN2 + lane + 32 * h;
        dd[h] = (kt < n_kt && j < key_hi) ? a.keys[tA.era_off + j].death : 0;
      }
    };
    auto store_deaths = [&](int kt, const int* dd) {
      const int b = kt & 1;
      int mn = INT32_MAX;
#pragma unroll
      for (int h = 0; h < kBN2 / 32; ++h) {
        s_death[b * kBN2 + lane + 32 * h] = dd[h];
        mn = min(mn, dd[h]);
      }
      mn = __reduce_min_sync(0xffffffffu, mn);
      if (lane == 0) s_dmin[b] = mn;
      __syncwarp();
      if (lane == 0) mbar_arrive(mbD0 + 8 * b);
    };
    bool ok = true;
    if (n_kt > 0) {
      if (lane == 0) {
        tma_kv(0, true);
        tma_kv(0, false);
        if (n_kt > 1) { tma_kv(1, true); tma_kv(1, false); }
      }
      int dd[kBN2 / 32];
      fetch_deaths(0, dd);
      store_deaths(0, dd);
      if (n_kt > 1) {
        fetch_deaths(1, dd);
        store_deaths(1, dd);
      }
    }
    for (int kt = 0; kt + 2 < n_kt; ++kt) {
      const int b = kt & 1;
      ok = __shfl_sync(0xffffffffu, ok, 0) && !*s_abort;
      if (!ok) break;
      int dnext[kBN2 / 32];
      fetch_deaths(kt + 2, dnext);      // in flight while lane 0 waits
      if (lane == 0) {
        // K(kt) read by S_A(kt) and S_B(kt); the deaths of kt by both softmaxes
        ok = mbar_wait(mbKf0 + 8 * b, (kt >> 1) & 1, a.wait_limit) &&
             mbar_wait(mbP0 + 8 * b, (kt >> 1) & 1, a.wait_limit) &&
             (!hasB || mbar_wait(mbP0 + 8 * (2 + b), (kt >> 1) & 1, a.wait_limit));
        if (ok) tma_kv(kt + 2, true);
        else fail();
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      store_deaths(kt + 2, dnext);
      if (lane == 0) {
        ok = mbar_wait(mbVf0 + 8 * b, (kt >> 1) & 1, a.wait_limit);   // PV_A(kt), PV_B(kt) done
        if (ok) tma_kv(kt + 2, false);
        else fail();
      }
    }
    if (lane == 0 && *s_abort) {
      // this warp's copies land before the CTA's memory goes (bounded)
      for (int b = 0; b < 2; ++b) {
        if (k_pend[b] >= 0) mbar_wait(mbK0 + 8 * b, (k_pend[b] >> 1) & 1, kDrainPolls);
        if (v_pend[b] >= 0) mbar_wait(mbV0 + 8 * b, (v_pend[b] >> 1) & 1, kDrainPolls);
      }
    }
    __syncwarp();
  } else if (control) {
    // ---- MMA warp (lane 0) ----
    const uint32_t id_s = idesc_bf16(kBM, kBN2, 0), id_o = idesc_bf16(kBM, D, 1);
    int pend = 0;                                  // an MMA of this thread may be in flight
    const uint64_t dq = sdesc(smem_u32(sQ), 16, 1024);
    const uint64_t dk = sdesc(smem_u32(sK), 16, 1024);
    const uint64_t dv = sdesc(smem_u32(sV), kBN2 * 128, 1024);
    auto issue_s = [&](int x, int kt) {
      const uint64_t kb = dk + (uint64_t)(((kt & 1) * kBN2 * D * 2) >> 4);
      const uint64_t qb = dq + (uint64_t)((x * kBM * D * 2) >> 4);
      const uint32_t ts = tbase + x * kBN2;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        umma(ts, qb + (uint64_t)((((kk >> 2) * kBM * 128) + (kk & 3) * 32) >> 4),
             kb + (uint64_t)((((kk >> 2) * kBN2 * 128) + (kk & 3) * 32) >> 4), id_s, kk > 0);
      umma_commit(mbS0 + 8 * x);
      pend = 1;
    };
    auto issue_pv = [&](int x, int kt) {
      const uint64_t vb = dv + (uint64_t)(((kt & 1) * kBN2 * D * 2) >> 4);
      const uint32_t tS = tbase + x * kBN2, tO = tbase + 2 * kBN2 + x * 128;
#pragma unroll
      for (int kk = 0; kk < kBN2 / 16; ++kk)
        umma_ts(tO, tS + kk * 8, vb + (uint64_t)((kk * 16 * 128) >> 4), id_o, kt > 0 || kk > 0);
      umma_commit(mbO0 + 8 * x);
      pend = 1;
    };
    bool ok = true;
    if (n_kt > 0 && lane == 0) {
      ok = mbar_wait(mbK0, 0, a.wait_limit);
      if (ok) {
        tc_after();
        issue_s(0, 0);
        if (hasB) issue_s(1, 0);
        umma_commit(mbKf0);                      // K(0) free once both have completed
      } else {
        fail();
      }
    }
    for (int kt = 0; kt < n_kt; ++kt) {
      const int b = kt & 1;
      ok = __shfl_sync(0xffffffffu, ok, 0) && !*s_abort;
      if (!ok) break;
      if (lane == 0) {
        // A: softmax(kt) done and V(kt) in -> PV_A(kt); K(kt+1) in -> S_A(kt+1)
        ok = mbar_wait(mbP0 + 8 * b, (kt >> 1) & 1, a.wait_limit) &&
             mbar_wait(mbV0 + 8 * b, (kt >> 1) & 1, a.wait_limit);
        if (ok) {
          tc_after();
          issue_pv(0, kt);
          if (kt + 1 < n_kt) {
            ok = mbar_wait(mbK0 + 8 * (b ^ 1), ((kt + 1) >> 1) & 1, a.wait_limit);
            if (ok) issue_s(0, kt + 1);
          }
        }
        // B: the same
        if (ok && hasB) {
          ok = mbar_wait(mbP0 + 8 * (2 + b), (kt >> 1) & 1, a.wait_limit);
          if (ok) {
            tc_after();
            issue_pv(1, kt);
            if (kt + 1 < n_kt) issue_s(1, kt + 1);
          }
        }
        if (ok) {
          umma_commit(mbVf0 + 8 * b);            // V(kt) free once PV_A(kt), PV_B(kt) complete
          if (kt + 1 < n_kt) umma_commit(mbKf0 + 8 * (b ^ 1));
        } else {
          fail();
        }
      }
    }
    if (lane == 0 && *s_abort && pend) {
      // this thread's MMAs complete before the CTA's memory goes (bounded):
      // a commit after everything issued, on a barrier of its own
      umma_commit(smem_u32(mbar + 18));
      mbar_wait(smem_u32(mbar + 18), 0, kDrainPolls);
    }
    __syncwarp();
  } else {
    // ---- softmax warps: tile x = warp / 4, row = TMEM lane ----
    const int x = warp / kGroupWarps, quarter = warp % kGroupWarps;
    const RestoreTile& tl = x == 0 ? tA : tB;
    const int row = 32 * quarter + lane;
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const uint32_t tS = tbase + x * kBN2, tO = tbase + 2 * kBN2 + x * 128;
    const int tend = tl.tok0 + tl.n_tok;
    int time_r = -1, lo_r = 0, kend_r = 0;
    t_r = tl.tok0 + row / NH;
    const bool active = x == 0 || hasB;
    if (active && t_r < tend) {
      const RestoreQuery qq = a.queries[t_r];
      if (qq.pos >= 0 && qq.pos < a.max_pos) {
        time_r = qq.time;
        kend_r = qq.key_end;
        lo_r = a.window > 0 ? max(0, qq.pos - a.window + 1) : 0;
      }
    }
    const bool real = active && t_r < tend;
    const int w_kend = __reduce_min_sync(0xffffffffu, real ? kend_r : INT32_MAX);
    const int w_lo = __reduce_max_sync(0xffffffffu, real ? lo_r : INT32_MIN);
    const int w_time = __reduce_max_sync(0xffffffffu, real ? time_r : INT32_MIN);
    for (int kt = 0; active && kt < n_kt; ++kt) {
      const int b = kt & 1;
      const int k0 = key_lo + kt * kBN2;
      bool ok = mbar_wait(mbD0 + 8 * b, (kt >> 1) & 1, a.wait_limit) &&
                mbar_wait(mbS0 + 8 * x, kt & 1, a.wait_limit);
      ok = __all_sync(0xffffffffu, ok) && !*s_abort;
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_after();
      uint32_t sr[kBN2];
#pragma unroll
      for (int u = 0; u < kBN2 / 32; ++u) tmem_ld32(tS + lane_off + 32 * u, sr + 32 * u);
      tmem_wait_ld();
      const int* de = s_death + b * kBN2;
      const bool full = k0 >= w_lo && k0 + kBN2 <= w_kend && s_dmin[b] > w_time;   // warp-uniform
      if (!full) {
#pragma unroll
        for (int c = 0; c < kBN2; ++c) {
          const int j = k0 + c;
          const bool vis = j >= lo_r && j < kend_r && de[c] > time_r;
          if (!vis) sr[c] = __float_as_uint(-INFINITY);
        }
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < kBN2; c += 8)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          m4[u] = fmax3(m4[u], __uint_as_float(sr[c + 2 * u]), __uint_as_float(sr[c + 2 * u + 1]));
      const float mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
      // the reference max moves only when the row max grows by more than 2^8
      const float m_new = (mx > m_r + 8.f) ? mx : m_r;
      const float alpha = m_new == -INFINITY ? 1.f : ex2(m_r - m_new);
      const float msub = m_new == -INFINITY ? 0.f : m_new;
      uint64_t ps2[2] = {0, 0};
      const uint64_t neg_m = pack_f32x2(-msub, -msub);
#pragma unroll
      for (int u = 0; u < kBN2 / 32; ++u) {      // P over S, 32 keys (16 columns) at a time
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float d0, d1;
          unpack_f32x2(add_f32x2(pack_f32x2(__uint_as_float(sr[32 * u + c]),
                                            __uint_as_float(sr[32 * u + c + 1])), neg_m), d0, d1);
          const float p0 = ex2(d0), p1 = ex2(d1);
          ps2[(c / 2) & 1] = add_f32x2(ps2[(c / 2) & 1], pack_f32x2(p0, p1));
          pk[c / 2] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tS + lane_off + 16 * u, pk);
      }
      float ps_lo, ps_hi;
      unpack_f32x2(add_f32x2(ps2[0], ps2[1]), ps_lo, ps_hi);
      l_r = fmaf(l_r, alpha, ps_lo + ps_hi);
      m_r = m_new;
      if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O is stable once PV_X(kt-1) is done: rescale the row
        const bool okv = __all_sync(0xffffffffu, mbar_wait(mbO0 + 8 * x, (kt - 1) & 1, a.wait_limit));
        if (!okv) {
          if (lane == 0) fail();
          break;
        }
        tc_after();
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + lane_off + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + lane_off + c, o);
        }
      }
      tmem_wait_st();
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(mbP0 + 8 * (2 * x + b));
    }
    // the last PV of this tile
    if (active && n_kt > 0 && !*s_abort) {
      const bool okv = __all_sync(0xffffffffu, mbar_wait(mbO0 + 8 * x, (n_kt - 1) & 1, a.wait_limit));
      if (!okv && lane == 0) fail();
    }
  }
  tc_before();
  __syncthreads();
  tc_after();
  if (warp < 2 * kGroupWarps && n_kt > 0 && !*s_abort) {
    // epilogue: the row of O / l
    const int x = warp / kGroupWarps, quarter = warp % kGroupWarps;
    const RestoreTile& tl = x == 0 ? tA : tB;
    const int row = 32 * quarter + lane;
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const uint32_t tO = tbase + 2 * kBN2 + x * 128;
    const int hq = kvh * G + blockIdx.z * NH + row % NH;
    const bool real = (x == 0 || hasB) && t_r < tl.tok0 + tl.n_tok;
    float* po = a.out + ((int64_t)t_r * a.g.hq + hq) * D;
    const float inv = l_r > 0.f ? 1.f / l_r : 0.f;
    if (x == 0 || hasB) {
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + c, o);
        tmem_wait_ld();
        if (real) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(po + c + e) =
                make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                            __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
        }
      }
    }
  }
  tc_before();
  __syncthreads();
  if (control)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kCols2) : "memory");
}

template <int D, int NH>
cudaError_t launch_tc_nh(const RestoreArgs& a, int G, cudaStream_t st) {
  constexpr size_t smem = restore_tc_smem<D>();
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(k_restore_attn_tc<D, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    attr = true;
  }
  if (a.n_pairs > 0) {                          // two query tiles per CTA
    constexpr size_t smem2 = restore_tc2_smem<D>();
    static bool attr2 = false;
    if (!attr2) {
      cudaFuncSetAttribute(k_restore_attn_tc2<D, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem2);
      attr2 = true;
    }
    const dim3 grid2(a.n_pairs, a.g.hkv, G / NH);
    k_restore_attn_tc2<D, NH><<<grid2, kRestoreThreads2, smem2, st>>>(a);
    return cudaGetLastError();
  }
  const dim3 grid(a.n_tiles, a.g.hkv, G / NH);
  k_restore_attn_tc<D, NH><<<grid, kRestoreThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_tc(const RestoreArgs& a, cudaStream_t st) {
  const int G = a.g.hq / a.g.hkv;
  switch (G) {
    case 1: return launch_tc_nh<D, 1>(a, G, st);
    case 2: return launch_tc_nh<D, 2>(a, G, st);
    case 4: return launch_tc_nh<D, 4>(a, G, st);
    default: return launch_tc_nh<D, 8>(a, G, st);
  }
}

}  // namespace

bool make_restore_tensor_maps(const Geom& g, const void* k_era, const void* v_era, int64_t n_keys,
                              CUtensorMap* tk, CUtensorMap* tv) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void**>(&encode),
                                         12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !encode) {
      encode = nullptr;
      return false;
    }
  }
  if (n_keys < 1) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)g.d, (cuuint64_t)g.hkv, (cuuint64_t)n_keys};
  const cuuint64_t strides[2] = {(cuuint64_t)g.d * 2, (cuuint64_t)g.hkv * g.d * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kBN};
  const cuuint32_t estr[3] = {1, 1, 1};
  for (int i = 0; i < 2; ++i) {
    CUresult r = encode(i == 0 ? tk : tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void*>(i == 0 ? k_era : v_era), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
  }
  return true;
}

bool restore_mma_supported(const Geom& g) {
  const int G = g.hq / g.hkv;
  return g.dtype == AKV_DTYPE_BF16 && (g.d == 64 || g.d == 128) &&
         (G == 1 || G == 2 || G == 4 || G == 8 || G == 16);
}

int restore_tile_tokens(const Geom& g) {
  const int G = g.hq / g.hkv;
  return kBM / (G < 8 ? G : 8);
}

cudaError_t launch_restore(const RestoreArgs& a, cudaStream_t st) {
  if (a.n_keys > 0) {
    const int64_t total = (int64_t)a.n_keys * a.g.hkv * a.g.d;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, 152 * 32);
    if (a.g.dtype == AKV_DTYPE_BF16)
      k_restore_keys<__nv_bfloat16><<<blocks, 256, 0, st>>>(
          a.g, a.keys, a.n_keys, static_cast<const __nv_bfloat16*>(a.k_raw),
          static_cast<const __nv_bfloat16*>(a.v), static_cast<__nv_bfloat16*>(a.k_era),
          static_cast<__nv_bfloat16*>(a.v_era), a.n_tokens, a.cs, a.max_pos, a.err);
    else
      k_restore_keys<float><<<blocks, 256, 0, st>>>(
          a.g, a.keys, a.n_keys, static_cast<const float*>(a.k_raw),
          static_cast<const float*>(a.v), static_cast<float*>(a.k_era),
          static_cast<float*>(a.v_era), a.n_tokens, a.cs, a.max_pos, a.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.n_queries <= 0) return cudaSuccess;
  if (a.use_mma) return a.g.d == 64 ? launch_tc<64>(a, st) : launch_tc<128>(a, st);
  const int G = a.g.hq / a.g.hkv;
  if (a.g.dtype == AKV_DTYPE_BF16)
    return a.g.d == 64 ? launch_simple_g<__nv_bfloat16, 64>(a, G, st)
                       : launch_simple_g<__nv_bfloat16, 128>(a, G, st);
  return a.g.d == 64 ? launch_simple_g<float, 64>(a, G, st) : launch_simple_g<float, 128>(a, G, st);
}

}  // namespace akv
