// Decode attention over the active KV only, split over pages (flash-decode),
// plus the merge of the splits.
//
// Each (item, kv head) block reads the pages [p0, p1) of its sequence's
// active page list, masks dropped slots with the keep bits, and keeps an
// online softmax (running max m, sum l, weighted sum of V) per query head of
// its GQA group.  Scores are kept in log2 units: s = (q' . k) log2(e)/sqrt(D),
// weights are 2^(s - m).  q' = R(pos_q) q with pos_q the position of the
// last appended token.  Sources: "Cache Engineering for Agents" paper review,
// 3.3 (Eq. 3: the query is conditioned on the active cache) and A.4.1 (the
// decode reads the active KV only).
#include <cuda_bf16.h>

#include "akv.h"
#include "akv_internal.h"

namespace akv {
namespace {

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }

constexpr int kWarps = 4;

// Generic CUDA-core kernel: any pool dtype, page size, D in {64, 128}, G <= 16.
template <typename T, int D, int G>
__global__ void __launch_bounds__(kWarps * 32) k_decode_simple(DecodeArgs a) {
  constexpr int J = D / 32;
  __shared__ float s_q[G][D];
  __shared__ float s_m[kWarps][G], s_l[kWarps][G];
  __shared__ float s_acc[kWarps][G][D];
  const DecodeItem it = a.items[blockIdx.x];
  const int kvh = blockIdx.y;
  const Geom& g = a.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (it.pos_q >= 0 && it.pos_q < a.sa.max_slots) {
    // q' = R(pos_q) q on the first R dims (pairs (d, d + R/2)); the rest as is
    const int R = g.rope, RH = R / 2;
    const T* q = static_cast<const T*>(a.q) + ((int64_t)it.row * g.hq + (int64_t)kvh * G) * D;
    const float2* cs = a.cs + (int64_t)it.pos_q * RH;
    for (int i = tid; i < G * D; i += blockDim.x) {
      const int gq = i / D, d = i % D;
      if (d < RH) {
        const float x = to_f(q[gq * D + d]), y = to_f(q[gq * D + d + RH]);
        const float2 t = cs[d];
        s_q[gq][d] = fmaf(x, t.x, -y * t.y) * a.scale_log2;
        s_q[gq][d + RH] = fmaf(x, t.y, y * t.x) * a.scale_log2;
      } else if (d >= R) {
        s_q[gq][d] = to_f(q[gq * D + d]) * a.scale_log2;
      }
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
  const int32_t* active = a.sa.active + (int64_t)it.dslot * a.sa.seq_pages;
  const int32_t* pages = a.sa.pages + (int64_t)it.dslot * a.sa.seq_pages;
  const uint32_t* keep = a.sa.keep + (int64_t)it.dslot * a.sa.keep_words;
  const int64_t slab = (int64_t)(a.layer % g.phys_layers) * g.layer_stride;
  const T* kpool = static_cast<const T*>(g.k) + slab + (int64_t)kvh * g.head_stride;
  const T* vpool = static_cast<const T*>(g.v) + slab + (int64_t)kvh * g.head_stride;

  for (int p = it.p0 + warp; p < it.p1; p += kWarps) {
    const int kidx = active[p];
    const int page = (kidx >= 0 && kidx < a.sa.seq_pages) ? pages[kidx] : -1;
    if (page < 0 || page >= g.max_pages) {
      if (lane == 0) atomicOr(a.err, AKV_DERR_PAGE);
      continue;
    }
    for (int s = 0; s < g.s; ++s) {
      const int slot = kidx * g.s + s;
      if (slot < it.win_lo || !((keep[slot >> 5] >> (slot & 31)) & 1u)) continue;
      const T* kr = kpool + (int64_t)page * g.page_stride + (int64_t)s * D;
      const T* vr = vpool + (int64_t)page * g.page_stride + (int64_t)s * D;
      float kd[J], vd[J];
#pragma unroll
      for (int j = 0; j < J; ++j) { kd[j] = to_f(kr[lane + 32 * j]); vd[j] = to_f(vr[lane + 32 * j]); }
#pragma unroll
      for (int gq = 0; gq < G; ++gq) {
        float part = 0.f;
#pragma unroll
        for (int j = 0; j < J; ++j) part = fmaf(s_q[gq][lane + 32 * j], kd[j], part);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        const float mn = fmaxf(m[gq], part);
        const float alpha = exp2f(m[gq] - mn);
        const float w = exp2f(part - mn);
        l[gq] = fmaf(l[gq], alpha, w);
#pragma unroll
        for (int j = 0; j < J; ++j) acc[gq][j] = fmaf(acc[gq][j], alpha, w * vd[j]);
        m[gq] = mn;
      }
    }
  }

#pragma unroll
  for (int gq = 0; gq < G; ++gq) {
    if (lane == 0) { s_m[warp][gq] = m[gq]; s_l[warp][gq] = l[gq]; }
#pragma unroll
    for (int j = 0; j < J; ++j) s_acc[warp][gq][lane + 32 * j] = acc[gq][j];
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
    const int hq = kvh * G + gq;
    if (it.n_splits == 1) {
      a.out[((int64_t)it.row * g.hq + hq) * D + d] = L > 0.f ? A / L : 0.f;
    } else {
      const int64_t pi = ((int64_t)blockIdx.x * g.hkv + kvh) * G + gq;
      a.part_acc[pi * D + d] = A;
      if (d == 0) a.part_ml[pi] = make_float2(M, L);
    }
  }
}

// Merge of the splits of each (row, query head).
__global__ void k_combine(DecodeArgs a, const int32_t* __restrict__ row_item0,
                          const int32_t* __restrict__ row_splits) {
  const int row = blockIdx.x, hq = blockIdx.y;
  const int n = row_splits[row];
  if (n <= 1) return;
  const int i0 = row_item0[row];
  const int G = a.g.hq / a.g.hkv, D = a.g.d;
  const int kvh = hq / G, gq = hq % G;
  float M = -INFINITY;
  for (int c = 0; c < n; ++c)
    M = fmaxf(M, a.part_ml[((int64_t)(i0 + c) * a.g.hkv + kvh) * G + gq].x);
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
      for (int c = 0; c < n; ++c) {
        const int64_t pi = ((int64_t)(i0 + c) * a.g.hkv + kvh) * G + gq;
        const float2 ml = a.part_ml[pi];
        const float f = exp2f(ml.x - M);
        L = fmaf(ml.y, f, L);
        A = fmaf(a.part_acc[pi * D + d], f, A);
      }
    }
    a.out[((int64_t)row * a.g.hq + hq) * D + d] = L > 0.f ? A / L : 0.f;
  }
}

template <typename T, int D>
cudaError_t launch_simple_g(const DecodeArgs& a, int G, cudaStream_t st) {
  dim3 grid(a.n_items, a.g.hkv);
  switch (G) {
    case 1: k_decode_simple<T, D, 1><<<grid, kWarps * 32, 0, st>>>(a); break;
    case 2: k_decode_simple<T, D, 2><<<grid, kWarps * 32, 0, st>>>(a); break;
    case 4: k_decode_simple<T, D, 4><<<grid, kWarps * 32, 0, st>>>(a); break;
    case 8: k_decode_simple<T, D, 8><<<grid, kWarps * 32, 0, st>>>(a); break;
    case 16: k_decode_simple<T, D, 16><<<grid, kWarps * 32, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, bool need_combine, int n_rows,
                          const int32_t* row_item0, const int32_t* row_splits,
                          cudaStream_t st) {
  if (a.n_items <= 0) return cudaSuccess;
  const int G = a.g.hq / a.g.hkv;
  cudaError_t e;
  if (a.use_mma)
    e = launch_decode_mma(a, st);
  else if (a.g.dtype == AKV_DTYPE_BF16)
    e = a.g.d == 64 ? launch_simple_g<__nv_bfloat16, 64>(a, G, st)
                    : launch_simple_g<__nv_bfloat16, 128>(a, G, st);
  else
    e = a.g.d == 64 ? launch_simple_g<float, 64>(a, G, st)
                    : launch_simple_g<float, 128>(a, G, st);
  if (e != cudaSuccess) return e;
  if (need_combine) {
    k_combine<<<dim3(n_rows, a.g.hq), 128, 0, st>>>(a, row_item0, row_splits);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace akv
