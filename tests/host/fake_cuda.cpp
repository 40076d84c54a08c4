// Host-memory stand-in for the CUDA runtime calls and kernel launchers that
// the cache's host planner (akv_host.cpp, akv_prefix.cpp) makes, so that the
// planner -- page allocation and reference counts, copy-on-write decisions,
// interval sets, rollback of a call that fails, history keys -- builds and
// runs on a machine without a GPU.
//
// Test infrastructure only: device memory is host memory (zeroed), copies
// and sets are memcpy/memset, streams and events do nothing, and every
// kernel launcher returns success without doing anything.  So the metadata
// that kernels compute (device keep bits, device page-table rows, gather
// maps, K/V) is NOT produced here: only state the planner keeps on the host
// is meaningful in a build with this file.
#include <cstdlib>
#include <cstring>

#include <cuda_runtime_api.h>

#include "akv.h"
#include "akv_internal.h"

namespace {
long g_launches = 0;
bool g_tensor_cores = false;   // report the tensor-core decode kernels as usable
}

extern "C" {

long akv_fake_launches() { return g_launches; }
// Plans as for a GPU where the tensor-core decode kernels run (the planner's
// choices depend on it); off by default.
void akv_fake_set_tensor_cores(int on) { g_tensor_cores = on != 0; }

cudaError_t cudaMalloc(void** p, size_t n) {
  *p = std::calloc(1, n ? n : 1);
  return *p ? cudaSuccess : cudaErrorMemoryAllocation;
}
cudaError_t cudaHostAlloc(void** p, size_t n, unsigned int) { return cudaMalloc(p, n); }
cudaError_t cudaFree(void* p) { std::free(p); return cudaSuccess; }
cudaError_t cudaFreeHost(void* p) { std::free(p); return cudaSuccess; }
cudaError_t cudaHostGetDevicePointer(void** d, void* h, unsigned int) { *d = h; return cudaSuccess; }
cudaError_t cudaMemcpy(void* d, const void* s, size_t n, cudaMemcpyKind) {
  if (n) std::memmove(d, s, n);
  return cudaSuccess;
}
cudaError_t cudaMemcpyAsync(void* d, const void* s, size_t n, cudaMemcpyKind k, cudaStream_t) {
  return cudaMemcpy(d, s, n, k);
}
cudaError_t cudaMemset(void* d, int v, size_t n) { std::memset(d, v, n); return cudaSuccess; }
cudaError_t cudaMemsetAsync(void* d, int v, size_t n, cudaStream_t) { return cudaMemset(d, v, n); }
cudaError_t cudaStreamSynchronize(cudaStream_t) { return cudaSuccess; }
cudaError_t cudaDeviceSynchronize() { return cudaSuccess; }
cudaError_t cudaEventCreateWithFlags(cudaEvent_t* e, unsigned int) {
  *e = reinterpret_cast<cudaEvent_t>(std::calloc(1, 8));
  return cudaSuccess;
}
cudaError_t cudaEventDestroy(cudaEvent_t e) { std::free(e); return cudaSuccess; }
cudaError_t cudaEventRecord(cudaEvent_t, cudaStream_t) { return cudaSuccess; }
cudaError_t cudaEventSynchronize(cudaEvent_t) { return cudaSuccess; }
cudaError_t cudaGetDevice(int* d) { *d = 0; return cudaSuccess; }
cudaError_t cudaDeviceGetAttribute(int* v, cudaDeviceAttr a, int) {
  *v = a == cudaDevAttrMultiProcessorCount ? 152 : 0;
  return cudaSuccess;
}
const char* cudaGetErrorString(cudaError_t) { return "fake CUDA runtime"; }

}  // extern "C"

namespace akv {

// kernel launchers: nothing runs
cudaError_t launch_append(const Geom&, const SeqArrays&, const AppendItem*, const AppendBlock*, int,
                          const int32_t*, const int32_t*, const void*, const void*, int64_t,
                          const float2*, uint32_t*, AppendLimits, cudaStream_t) {
  ++g_launches;
  return cudaSuccess;
}
cudaError_t launch_copy_pages(const Geom&, const PagePair*, int, uint32_t*, cudaStream_t) {
  ++g_launches;
  return cudaSuccess;
}
// the byte copy and fill kernels move host metadata: done here
cudaError_t launch_copy_bytes(void* dst, const void* src, size_t n, cudaStream_t) {
  ++g_launches;
  if (n) std::memmove(dst, src, n);
  return cudaSuccess;
}
cudaError_t launch_fill_u32(uint32_t* dst, uint32_t v, size_t n, cudaStream_t) {
  ++g_launches;
  for (size_t i = 0; i < n; ++i) dst[i] = v;
  return cudaSuccess;
}
cudaError_t launch_drop(const Geom&, const SeqArrays&, const DropItem*, int, const int32_t*,
                        uint32_t*, cudaStream_t) {
  ++g_launches;
  return cudaSuccess;
}
cudaError_t launch_compact(const Geom&, const SeqArrays&, const ReposItem*, int, const int32_t*,
                           uint32_t*, cudaStream_t) {
  ++g_launches;
  return cudaSuccess;
}
cudaError_t launch_gather(const Geom&, const SeqArrays&, const ReposItem*, int, int, const float2*,
                          uint32_t*, uint32_t, cudaStream_t) {
  ++g_launches;
  return cudaSuccess;
}
cudaError_t launch_transplant(const Geom&, const MoveItem*, int, const MoveBlock*, int,
                              const float2*, int, uint32_t*, uint32_t, cudaStream_t) {
  ++g_launches;
  return cudaSuccess;
}
cudaError_t launch_decode(const DecodeArgs&, bool, int, const int32_t*, const int32_t*,
                          cudaStream_t) {
  ++g_launches;
  return cudaSuccess;
}
cudaError_t launch_decode_share(const DecodeArgs&, cudaStream_t) {
  ++g_launches;
  return cudaSuccess;
}
cudaError_t launch_restore(const RestoreArgs&, cudaStream_t) {
  ++g_launches;
  return cudaSuccess;
}
bool decode_mma_supported(const Geom& g) {
  return g_tensor_cores && g.dtype == AKV_DTYPE_BF16 && g.s % 16 == 0 && g.hq / g.hkv <= 8 &&
         (g.d == 64 || g.d == 128);
}
bool decode_share_supported(const Geom& g) {
  const int G = g.hq / g.hkv;
  return g_tensor_cores && g.dtype == AKV_DTYPE_BF16 && g.s == 16 && (g.d == 64 || g.d == 128) &&
         (G == 1 || G == 2 || G == 4 || G == 8);
}
int decode_mma_blocks_per_sm(int) { return 3; }
bool make_pool_tensor_maps(const Geom& g, CUtensorMap*, CUtensorMap*) { return decode_mma_supported(g); }
bool make_pool_tensor_maps4(const Geom& g, CUtensorMap*, CUtensorMap*) { return decode_mma_supported(g); }
bool restore_mma_supported(const Geom&) { return false; }
int restore_tile_tokens(const Geom&) { return 16; }
bool make_restore_tensor_maps(const Geom&, const void*, const void*, int64_t, CUtensorMap*,
                              CUtensorMap*) {
  return false;
}

}  // namespace akv
