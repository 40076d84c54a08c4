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

}  // namespace

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
  const int G = a.g.hq / a.g.hkv;
  if (a.g.dtype == AKV_DTYPE_BF16)
    return a.g.d == 64 ? launch_simple_g<__nv_bfloat16, 64>(a, G, st)
                       : launch_simple_g<__nv_bfloat16, 128>(a, G, st);
  return a.g.d == 64 ? launch_simple_g<float, 64>(a, G, st) : launch_simple_g<float, 128>(a, G, st);
}

}  // namespace akv
