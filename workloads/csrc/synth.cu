// Device copy of the seeded input generator of workloads/synth.py.
//
// SplitMix64 (Steele, Lea, Flood, OOPSLA 2014): the i-th output of a stream
// whose state starts at `key` is mix64(key + (i + 1) * GAMMA).  A 64-bit
// output is cut into three w-bit fields and mapped to the odd integer
// 2*(f0+f1+f2) - 3*(2^w - 1) divided by 2^w, which is exact in the pool dtype
// (w = 6 for bfloat16, 21 for float32), so no rounding is involved.
//
// This library only produces inputs; it holds nothing of the cache method.
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

struct Row { uint64_t key; int64_t start; int64_t out_off; };

template <typename T>
__global__ void k_fill(T* out, const Row* __restrict__ rows, int n_rows, int64_t count, int width) {
  const int64_t total = (int64_t)n_rows * count;
  const uint64_t m = (1ULL << width) - 1ULL;
  const int64_t bias = 3 * (int64_t)m;
  const float scale = 1.0f / (float)(1ULL << width);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / count, j = i - r * count;
    const Row row = rows[r];
    const uint64_t h = mix64(row.key + (uint64_t)(row.start + j + 1) * kGamma);
    const int64_t s = (int64_t)(h & m) + (int64_t)((h >> width) & m) + (int64_t)((h >> (2 * width)) & m);
    const float v = (float)(2 * s - bias) * scale;   // exact: |2s - bias| < 2^23
    if constexpr (sizeof(T) == 2) out[row.out_off + j] = __float2bfloat16_rn(v);
    else out[row.out_off + j] = v;
  }
}

}  // namespace

extern "C" int akv_synth_fill(void* out, int dtype_bf16, const void* rows, int n_rows,
                              int64_t count, int width, void* stream) {
  if (!out || !rows || n_rows <= 0 || count <= 0 || width < 1 || width > 21) return -1;
  const int64_t total = (int64_t)n_rows * count;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 152 * 64) blocks = 152 * 64;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype_bf16)
    k_fill<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<__nv_bfloat16*>(out),
                                                  static_cast<const Row*>(rows), n_rows, count, width);
  else
    k_fill<float><<<blocks, 256, 0, st>>>(static_cast<float*>(out), static_cast<const Row*>(rows),
                                          n_rows, count, width);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}
