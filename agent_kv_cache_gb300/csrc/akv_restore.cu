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

#include <cuda_bf16.h>

#include "akv.h"
#include "akv_internal.h"

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
// Tensor-core path (bf16, D in {64, 128}): FA2-style tiles on mma.sync.
// Block = 64 query rows: warp w takes head (w % NH) of the block's head
// subgroup and 16 consecutive tokens (group w / NH), NH = min(G, 4), so a
// K/V tile in shared memory serves NH heads.  64-key tiles, double-buffered
// with cp.async into rows whose 16-byte chunks are XOR-swizzled by row % 8
// (conflict-free ldmatrix).  S = Q K^T and O += P V (P reused from the
// accumulator registers as the A operand); interval mask per (row, key).
// ---------------------------------------------------------------------------

constexpr int kKT = 64;   // keys per tile

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
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
// byte offset of (row, 16-byte chunk) in a tile of rows of D bf16
template <int D>
__device__ __forceinline__ uint32_t rsw(int row, int chunk) {
  return (uint32_t)(row * (D * 2) + (((chunk & ~7) | ((chunk & 7) ^ (row & 7))) << 4));
}

template <int D, int NH>
__global__ void __launch_bounds__(128)
k_restore_attn_mma(const __grid_constant__ RestoreArgs a) {
  constexpr int KS = D / 16, NTD = D / 8, CH = D / 8, TILE = kKT * D * 2;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* s_k = smem;                       // [2][kKT][D]  (stage 0 also stages Q)
  unsigned char* s_v = smem + 2 * TILE;            // [2][kKT][D]
  int* s_birth = reinterpret_cast<int*>(smem + 4 * TILE);   // [2][kKT]
  int* s_death = s_birth + 2 * kKT;

  const RestoreTile tl = a.tiles[blockIdx.x];
  const int kvh = blockIdx.y;
  const int G = a.g.hq / a.g.hkv, H = a.g.hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int head = blockIdx.z * NH + warp % NH;
  const int tbase = tl.tok0 + (warp / NH) * 16;   // first token of this warp's rows
  const int tend = tl.tok0 + tl.n_tok;
  const int R = a.g.rope, RH = R / 2;
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(a.k_era);
  const __nv_bfloat16* vg = static_cast<const __nv_bfloat16*>(a.v_era);

  // stage rotated, scaled Q rows (bf16, swizzled) in s_k[0]; row = warp*16 + r
  for (int i = tid; i < 64 * (D / 2); i += 128) {
    const int row = i / (D / 2), d = i % (D / 2);
    const int w = row / 16, r = row % 16;
    const int t = tl.tok0 + (w / NH) * 16 + r;
    const int hq = kvh * G + blockIdx.z * NH + w % NH;
    float x = 0.f, y = 0.f;
    int dx = d, dy = d + D / 2;
    const bool ok = t < tend && a.queries[t].pos >= 0 && a.queries[t].pos < a.max_pos;
    if (t < tend && !ok && d == 0) atomicOr(a.err, AKV_DERR_INDEX);
    if (ok) {
      const RestoreQuery qq = a.queries[t];
      const __nv_bfloat16* qr = qg + ((int64_t)t * a.g.hq + hq) * D;
      if (d < RH) {                    // rotary pair (d, d + RH)
        dy = d + RH;
        const float2 c = a.cs[(int64_t)qq.pos * RH + d];
        const float qx = __bfloat162float(qr[d]), qy = __bfloat162float(qr[dy]);
        x = fmaf(qx, c.x, -qy * c.y) * a.scale_log2;
        y = fmaf(qx, c.y, qy * c.x) * a.scale_log2;
      } else {                         // two dims past the rotary part
        dx = R + 2 * (d - RH);
        dy = dx + 1;
        x = __bfloat162float(qr[dx]) * a.scale_log2;
        y = __bfloat162float(qr[dy]) * a.scale_log2;
      }
    } else if (d >= RH) {
      dx = R + 2 * (d - RH);
      dy = dx + 1;
    } else {
      dy = d + RH;
    }
    __nv_bfloat16* q0 = reinterpret_cast<__nv_bfloat16*>(s_k + rsw<D>(row, dx / 8)) + dx % 8;
    __nv_bfloat16* q1 = reinterpret_cast<__nv_bfloat16*>(s_k + rsw<D>(row, dy / 8)) + dy % 8;
    *q0 = __float2bfloat16_rn(x);
    *q1 = __float2bfloat16_rn(y);
  }
  __syncthreads();
  uint32_t qa[KS][4];
  {
    const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) ldsm_x4(smem_u32(s_k + rsw<D>(row, ks * 2 + (lane >> 4))), qa[ks]);
  }
  // per-row time and window bound (rows r0 = lane/4 and r1 = r0 + 8)
  int time0 = -1, time1 = -1, lo0 = 0, lo1 = 0;
  {
    const int t0 = tbase + (lane >> 2), t1 = t0 + 8;
    // a row past the tile or with a bad position sees no key (output 0)
    if (t0 < tend) {
      const RestoreQuery q0 = a.queries[t0];
      time0 = q0.pos >= 0 && q0.pos < a.max_pos ? q0.time : -1;
      lo0 = a.window > 0 ? q0.pos - a.window + 1 : 0;
    }
    if (t1 < tend) {
      const RestoreQuery q1 = a.queries[t1];
      time1 = q1.pos >= 0 && q1.pos < a.max_pos ? q1.time : -1;
      lo1 = a.window > 0 ? q1.pos - a.window + 1 : 0;
    }
  }
  __syncthreads();   // Q staging area is reused for key tiles

  auto load_tile = [&](int kt, int buf) {
    const int k0 = tl.key_lo + kt * kKT;
    for (int i = tid; i < kKT * CH; i += 128) {
      const int row = i / CH, ch = i % CH;
      const int j = k0 + row;
      const bool ok = j < tl.key_hi;
      const int64_t off = ((int64_t)(tl.era_off + (ok ? j : 0)) * H + kvh) * D + ch * 8;
      cp_async16(smem_u32(s_k + buf * TILE + rsw<D>(row, ch)), kg + off, ok);
      cp_async16(smem_u32(s_v + buf * TILE + rsw<D>(row, ch)), vg + off, ok);
    }
    for (int i = tid; i < kKT; i += 128) {
      const int j = k0 + i;
      int b = INT32_MAX, dth = 0;
      if (j < tl.key_hi) {
        const RestoreKey kk = a.keys[tl.era_off + j];
        b = kk.birth;
        dth = kk.death;
      }
      s_birth[buf * kKT + i] = b;
      s_death[buf * kKT + i] = dth;
    }
    cp_commit();
  };

  float o[NTD][4];
#pragma unroll
  for (int n = 0; n < NTD; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int n_kt = (tl.key_hi - tl.key_lo + kKT - 1) / kKT;
  if (n_kt > 0) load_tile(0, 0);
  for (int kt = 0; kt < n_kt; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < n_kt) {
      load_tile(kt + 1, buf ^ 1);
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    const uint32_t kb = smem_u32(s_k + buf * TILE), vb = smem_u32(s_v + buf * TILE);
    const int k0 = tl.key_lo + kt * kKT;
    // S = Q K^T: 16 rows x 64 keys per warp
    float sc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int n2 = 0; n2 < 4; ++n2) {
        uint32_t b[4];
        ldsm_x4(kb + rsw<D>(n2 * 16 + (lane & 7) + ((lane >> 4) & 1) * 8, ks * 2 + ((lane >> 3) & 1)), b);
        mma16816(sc[2 * n2], qa[ks], b[0], b[1]);
        mma16816(sc[2 * n2 + 1], qa[ks], b[2], b[3]);
      }
    }
    // interval mask (and window)
    const int* bi = s_birth + buf * kKT;
    const int* de = s_death + buf * kKT;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int kc = n * 8 + (lane & 3) * 2 + e;
        const int j = k0 + kc;
        const int b = bi[kc], dd = de[kc];
        if (!(b <= time0 && time0 < dd && j >= lo0)) sc[n][e] = -INFINITY;
        if (!(b <= time1 && time1 < dd && j >= lo1)) sc[n][2 + e] = -INFINITY;
      }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    const float a0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0);
    const float a1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
    m0 = n0;
    m1 = n1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      sc[n][0] = n0 == -INFINITY ? 0.f : exp2f(sc[n][0] - n0);
      sc[n][1] = n0 == -INFINITY ? 0.f : exp2f(sc[n][1] - n0);
      sc[n][2] = n1 == -INFINITY ? 0.f : exp2f(sc[n][2] - n1);
      sc[n][3] = n1 == -INFINITY ? 0.f : exp2f(sc[n][3] - n1);
      ps0 += sc[n][0] + sc[n][1];
      ps1 += sc[n][2] + sc[n][3];
    }
    l0 = fmaf(l0, a0, ps0);
    l1 = fmaf(l1, a1, ps1);
#pragma unroll
    for (int n = 0; n < NTD; ++n) {
      o[n][0] *= a0; o[n][1] *= a0; o[n][2] *= a1; o[n][3] *= a1;
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
      pa[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
      pa[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      pa[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int nd2 = 0; nd2 < NTD / 2; ++nd2) {
        uint32_t b[4];
        ldsm_x4_t(vb + rsw<D>(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, nd2 * 2 + (lane >> 4)), b);
        mma16816(o[2 * nd2], pa, b[0], b[1]);
        mma16816(o[2 * nd2 + 1], pa, b[2], b[3]);
      }
    }
    __syncthreads();   // this buffer is refilled next-but-one iteration
  }
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  const int t0 = tbase + (lane >> 2), t1 = t0 + 8;
  const int hq = kvh * G + head;
#pragma unroll
  for (int n = 0; n < NTD; ++n) {
    const int d = n * 8 + (lane & 3) * 2;
    if (t0 < tend) {
      float* po = a.out + ((int64_t)t0 * a.g.hq + hq) * D + d;
      po[0] = l0 > 0.f ? o[n][0] / l0 : 0.f;
      po[1] = l0 > 0.f ? o[n][1] / l0 : 0.f;
    }
    if (t1 < tend) {
      float* po = a.out + ((int64_t)t1 * a.g.hq + hq) * D + d;
      po[0] = l1 > 0.f ? o[n][2] / l1 : 0.f;
      po[1] = l1 > 0.f ? o[n][3] / l1 : 0.f;
    }
  }
}

template <int D, int NH>
cudaError_t launch_mma_nh(const RestoreArgs& a, int G, cudaStream_t st) {
  const size_t smem = 4 * (size_t)kKT * D * 2 + 4 * kKT * sizeof(int);
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(k_restore_attn_mma<D, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    attr = true;
  }
  const dim3 grid(a.n_tiles, a.g.hkv, G / NH);
  k_restore_attn_mma<D, NH><<<grid, 128, smem, st>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_mma(const RestoreArgs& a, cudaStream_t st) {
  const int G = a.g.hq / a.g.hkv;
  switch (G) {
    case 1: return launch_mma_nh<D, 1>(a, G, st);
    case 2: return launch_mma_nh<D, 2>(a, G, st);
    default: return launch_mma_nh<D, 4>(a, G, st);
  }
}

}  // namespace

bool restore_mma_supported(const Geom& g) {
  const int G = g.hq / g.hkv;
  return g.dtype == AKV_DTYPE_BF16 && (g.d == 64 || g.d == 128) &&
         (G == 1 || G == 2 || G == 4 || G == 8 || G == 16);
}

int restore_tile_tokens(const Geom& g) {
  const int G = g.hq / g.hkv;
  return 16 * (4 / (G < 4 ? G : 4));
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
  if (a.use_mma) return a.g.d == 64 ? launch_mma<64>(a, st) : launch_mma<128>(a, st);
  const int G = a.g.hq / a.g.hkv;
  if (a.g.dtype == AKV_DTYPE_BF16)
    return a.g.d == 64 ? launch_simple_g<__nv_bfloat16, 64>(a, G, st)
                       : launch_simple_g<__nv_bfloat16, 128>(a, G, st);
  return a.g.d == 64 ? launch_simple_g<float, 64>(a, G, st) : launch_simple_g<float, 128>(a, G, st);
}

}  // namespace akv
