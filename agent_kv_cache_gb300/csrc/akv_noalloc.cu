// Decode attention for callers that cannot allocate device memory.
//
// Some host applications reserve all of their device memory once at start-up
// (a fixed budget carved into their own pools) and forbid cudaMalloc/cudaFree
// afterwards: those calls synchronise the whole device, can fail under
// memory pressure in the middle of serving, and fragment memory the
// application has already planned.  A plugin running inside such a runtime
// owns its K/V pool and page metadata but cannot create an akv_cache (whose
// creation allocates metadata and workspace).  akv_decode_attention_noalloc()
// serves them: it takes only the caller's pointers, allocates nothing, and
// keeps its split-KV partial sums in the file-scope array below.
//
// The computation is the same as akv_decode_attention(): softmax attention
// of each query over the active tokens of its sequence, split over pages,
// then the splits merged.
#include <cmath>
#include <mutex>

#include <cuda_bf16.h>

#include "akv.h"

namespace {

// Scratch for split partials: 2 Mi floats (8 MiB).  Every GPU that loads
// this library holds it until the process exits.
constexpr int64_t kScratchFloats = AKV_NOALLOC_SCRATCH_BYTES / 4;
static __device__ __align__(256) float g_scratch[kScratchFloats];

constexpr int kRows = AKV_NOALLOC_MAX_SEQS;
constexpr int kWarps = 4;

struct Row { int32_t n_active, pos_q, item0, n_splits; };

struct Args {
  const void* k;
  const void* v;
  int64_t page_stride, head_stride;
  int32_t max_pages, hq, hkv, d, s;
  const int32_t* pages;
  const int32_t* active;
  const uint32_t* keep;
  int32_t row_stride, keep_stride;
  const void* q;
  float* out;
  float* acc;        // [items][hq][d]   (in the scratch array)
  float2* ml;        // [items][hq]      (after acc in the scratch array)
  float scale_log2;
  double theta;
  int32_t pps;       // pages per split
  int32_t n_rows;
  Row rows[kRows];
};

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }

template <typename T, int D, int G>
__global__ void __launch_bounds__(kWarps * 32) k_noalloc_decode(const __grid_constant__ Args a) {
  constexpr int H = D / 2, J = D / 32;
  __shared__ float s_q[G][D];
  __shared__ float s_m[kWarps][G], s_l[kWarps][G];
  __shared__ float s_acc[kWarps][G][D];
  const int split = blockIdx.x, kvh = blockIdx.y, row = blockIdx.z;
  const Row r = a.rows[row];
  if (split >= r.n_splits) return;
  const int p0 = split * a.pps, p1 = min(r.n_active, p0 + a.pps);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (r.pos_q >= 0) {
    // The angle pos * theta^(-2d/D) in fp64 (positions reach 10^5 radians),
    // reduced to one turn in fp64, then cos/sin in fp32: four fp64
    // operations per pair, on a part whose fp64 rate is low.  The
    // frequencies once per block.
    __shared__ double s_w[H];
    const double l2t = log2(a.theta);
    for (int d = tid; d < H; d += blockDim.x) s_w[d] = exp2(-2.0 * d / D * l2t);
    __syncthreads();
    const T* q = static_cast<const T*>(a.q) + ((int64_t)row * a.hq + (int64_t)kvh * G) * D;
    for (int i = tid; i < G * H; i += blockDim.x) {
      const int gq = i / H, d = i % H;
      const double ang = (double)r.pos_q * s_w[d];
      const double turns = rint(ang * 0.15915494309189535);       // ang / (2 pi)
      const float red = (float)fma(-turns, 6.283185307179586, ang);
      float sn, c;
      sincosf(red, &sn, &c);
      const float x = to_f(q[gq * D + d]), y = to_f(q[gq * D + d + H]);
      s_q[gq][d] = fmaf(x, c, -y * sn) * a.scale_log2;
      s_q[gq][d + H] = fmaf(x, sn, y * c) * a.scale_log2;
    }
  } else {
    // no token held (the host rejects active pages then): defined scores
    for (int i = tid; i < G * D; i += blockDim.x) s_q[i / D][i % D] = 0.f;
  }
  __syncthreads();

  float m[G], l[G], acc[G][J];
#pragma unroll
  for (int gq = 0; gq < G; ++gq) {
    m[gq] = -INFINITY; l[gq] = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) acc[gq][j] = 0.f;
  }
  const int32_t* active = a.active + (int64_t)row * a.row_stride;
  const int32_t* pages = a.pages + (int64_t)row * a.row_stride;
  const uint32_t* keep = a.keep + (int64_t)row * a.keep_stride;
  const T* kbase = static_cast<const T*>(a.k) + (int64_t)kvh * a.head_stride;
  const T* vbase = static_cast<const T*>(a.v) + (int64_t)kvh * a.head_stride;
  for (int p = p0 + warp; p < p1; p += kWarps) {
    const int kidx = active[p];
    if (kidx < 0 || kidx >= a.row_stride) continue;
    const int page = pages[kidx];
    if (page < 0 || page >= a.max_pages) continue;
    for (int s = 0; s < a.s; ++s) {
      const int slot = kidx * a.s + s;
      if ((slot >> 5) >= a.keep_stride || !((keep[slot >> 5] >> (slot & 31)) & 1u)) continue;
      const T* kr = kbase + (int64_t)page * a.page_stride + (int64_t)s * D;
      const T* vr = vbase + (int64_t)page * a.page_stride + (int64_t)s * D;
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
    if (r.n_splits == 1) {
      a.out[((int64_t)row * a.hq + hq) * D + d] = L > 0.f ? A / L : 0.f;
    } else {
      const int64_t pi = (int64_t)(r.item0 + split) * a.hq + hq;
      a.acc[pi * D + d] = A;
      if (d == 0) a.ml[pi] = make_float2(M, L);
    }
  }
}

__global__ void k_noalloc_merge(const __grid_constant__ Args a) {
  const int row = blockIdx.x, hq = blockIdx.y;
  const Row r = a.rows[row];
  if (r.n_splits <= 1) return;
  float M = -INFINITY;
  for (int c = 0; c < r.n_splits; ++c)
    M = fmaxf(M, a.ml[(int64_t)(r.item0 + c) * a.hq + hq].x);
  for (int d = threadIdx.x; d < a.d; d += blockDim.x) {
    float L = 0.f, A = 0.f;
    if (M != -INFINITY) {
      for (int c = 0; c < r.n_splits; ++c) {
        const int64_t pi = (int64_t)(r.item0 + c) * a.hq + hq;
        const float2 ml = a.ml[pi];
        const float f = exp2f(ml.x - M);
        L = fmaf(ml.y, f, L);
        A = fmaf(a.acc[pi * a.d + d], f, A);
      }
    }
    a.out[((int64_t)row * a.hq + hq) * a.d + d] = L > 0.f ? A / L : 0.f;
  }
}

template <typename T, int D>
cudaError_t launch_g(const Args& a, int G, int max_splits, cudaStream_t st) {
  const dim3 grid(max_splits, a.hkv, a.n_rows);
  switch (G) {
    case 1: k_noalloc_decode<T, D, 1><<<grid, kWarps * 32, 0, st>>>(a); break;
    case 2: k_noalloc_decode<T, D, 2><<<grid, kWarps * 32, 0, st>>>(a); break;
    case 4: k_noalloc_decode<T, D, 4><<<grid, kWarps * 32, 0, st>>>(a); break;
    case 8: k_noalloc_decode<T, D, 8><<<grid, kWarps * 32, 0, st>>>(a); break;
    case 16: k_noalloc_decode<T, D, 16><<<grid, kWarps * 32, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// Device address of g_scratch, looked up once per device.
std::mutex g_mu;
void* g_addr[256];
bool g_have[256];

int scratch_address(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return AKV_ECUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_have[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return AKV_ECUDA;
    g_addr[dev] = p;
    g_have[dev] = true;
  }
  *out = static_cast<float*>(g_addr[dev]);
  return AKV_OK;
}

}  // namespace

extern "C" int akv_decode_attention_noalloc(
    const void* k_slab, const void* v_slab, int32_t max_pages, int32_t hq, int32_t hkv,
    int32_t head_dim, int32_t page_size, int32_t dtype, double rope_theta,
    const int32_t* page_table, const int32_t* active_pages, const uint32_t* keep_bits,
    int32_t row_stride, int32_t keep_stride, const int32_t* n_active_pages,
    const int32_t* n_held, const void* q, float* out, int32_t n_seqs, void* stream) {
  if (n_seqs == 0) return AKV_OK;
  if (n_seqs < 0 || n_seqs > kRows) return AKV_ECAPACITY;   // more rows than the call can carry
  if (!k_slab || !v_slab || !page_table || !active_pages || !keep_bits || !n_active_pages ||
      !n_held || !q || !out)
    return AKV_EINVAL;
  const int G = hkv > 0 ? hq / hkv : 0;
  if (hkv < 1 || hq % hkv || !(G == 1 || G == 2 || G == 4 || G == 8 || G == 16)) return AKV_EINVAL;
  if (head_dim != 64 && head_dim != 128) return AKV_EINVAL;
  if (page_size < 1 || page_size > 64 || (page_size & (page_size - 1))) return AKV_EINVAL;
  if (dtype != AKV_DTYPE_BF16 && dtype != AKV_DTYPE_FP32) return AKV_EINVAL;
  if (max_pages < 1 || row_stride < 1 || keep_stride < 1 || !(rope_theta > 1.0)) return AKV_EINVAL;

  Args a{};
  int64_t total = 0, longest = 0;
  for (int i = 0; i < n_seqs; ++i) {
    if (n_active_pages[i] < 0 || n_active_pages[i] > row_stride) return AKV_EINVAL;
    if (n_held[i] < 0 || (int64_t)n_held[i] > (int64_t)keep_stride * 32) return AKV_EINVAL;
    // an active page needs a held token, whose position the query takes
    if (n_active_pages[i] > 0 && n_held[i] < 1) return AKV_EINVAL;
    total += n_active_pages[i];
    longest = n_active_pages[i] > longest ? n_active_pages[i] : longest;
  }
  // Pages per split: fill the GPU a few times over, then widen the splits
  // until the partials fit the scratch array (one split per sequence needs
  // no scratch at all, so every call fits).
  const int64_t per_item = (int64_t)hq * (head_dim + 2);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return AKV_ECUDA;
  int64_t pps = total * hkv / ((int64_t)sms * 8);
  if (pps < 4) pps = 4;
  for (;;) {
    int64_t items = 0;
    for (int i = 0; i < n_seqs; ++i) {
      const int64_t ns = (n_active_pages[i] + pps - 1) / pps;
      if (ns > 1) items += ns;
    }
    if (items * per_item <= kScratchFloats || pps >= longest) break;
    pps *= 2;
  }
  if (pps < 1) pps = 1;
  int max_splits = 1;
  int32_t item0 = 0;
  for (int i = 0; i < n_seqs; ++i) {
    int64_t ns = (n_active_pages[i] + pps - 1) / pps;
    if (ns < 1) ns = 1;
    a.rows[i] = Row{n_active_pages[i], n_held[i] - 1, ns > 1 ? item0 : 0, (int32_t)ns};
    if (ns > 1) item0 += (int32_t)ns;
    if (ns > max_splits) max_splits = (int)ns;
  }
  float* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != AKV_OK) return rc;
  a.k = k_slab;
  a.v = v_slab;
  a.head_stride = (int64_t)page_size * head_dim;
  a.page_stride = a.head_stride * hkv;
  a.max_pages = max_pages;
  a.hq = hq;
  a.hkv = hkv;
  a.d = head_dim;
  a.s = page_size;
  a.pages = page_table;
  a.active = active_pages;
  a.keep = keep_bits;
  a.row_stride = row_stride;
  a.keep_stride = keep_stride;
  a.q = q;
  a.out = out;
  a.acc = scratch;
  a.ml = reinterpret_cast<float2*>(scratch + (int64_t)item0 * hq * head_dim);
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)head_dim));
  a.theta = rope_theta;
  a.pps = (int32_t)pps;
  a.n_rows = n_seqs;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dtype == AKV_DTYPE_BF16)
    e = head_dim == 64 ? launch_g<__nv_bfloat16, 64>(a, G, max_splits, st)
                       : launch_g<__nv_bfloat16, 128>(a, G, max_splits, st);
  else
    e = head_dim == 64 ? launch_g<float, 64>(a, G, max_splits, st)
                       : launch_g<float, 128>(a, G, max_splits, st);
  if (e != cudaSuccess) return AKV_ECUDA;
  if (item0 > 0) {
    k_noalloc_merge<<<dim3(n_seqs, hq), 128, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return AKV_ECUDA;
  }
  return AKV_OK;
}
