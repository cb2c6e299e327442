// gc_ef_topk_compress_noalloc: EF Top-k / random-k compression whose scratch
// memory is a fixed array inside the library instead of a caller-provided
// workspace.
//
// Why it exists: some callers cannot allocate device memory when they need
// to compress.  A serving or training process whose memory manager has
// already reserved the GPU's memory (so a raw cudaMalloc fails or fragments
// its pool), plain C code that has no handle on that manager, and loops that
// must not pay for cudaMalloc/cudaFree (which can synchronize the whole
// device) all fall in this group.  They still pass their own inputs and
// outputs; only the scratch comes from here.
//
// The scratch is kStaticBytes of device memory that every GPU which loads
// libgc holds until the process exits.  All calls share it, so calls that
// overlap on the GPU (for example on two streams) race on it.  It keeps the
// previous call's contents; the compression path clears the parts that must
// start at zero (diagnostic words, per-tensor state, histograms) at the
// start of every call, as it does for a caller's workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "gc_common.cuh"
#include "gc_host.h"

namespace gc {

constexpr size_t kStaticBytes = (size_t)GC_NOALLOC_MAX_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kStaticBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current.  In host code the array's name is only a stand-in for the
// symbol, never a device address.
static void* g_scratch_addr[kMaxDevices];
static std::mutex g_scratch_mu;

static gc_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();  // reset the error state the failed lookup left behind
      return GC_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GC_OK;
}

}  // namespace gc

using namespace gc;

extern "C" gc_status gc_ef_topk_compress_noalloc(const gc_layout* dev, const gc_layout* host,
                                                 const float* g, float* e, int32_t* idx,
                                                 float* val, int8_t* q, float* scale,
                                                 uint64_t seed, uint64_t iter, uint32_t flags,
                                                 void* stream) {
  NvtxRange nvtx_range("gc_ef_topk_compress_noalloc");
  const gc_status lst = validate_layout(host, true);
  if (lst != GC_OK) return lst;
  const size_t need = topk_workspace_bytes(host, !(flags & GC_RANDK));
  if (need > kStaticBytes) return GC_ERR_WORKSPACE;  // layout too large for the built-in scratch
  void* scratch = nullptr;
  const gc_status st = scratch_for_current_device(&scratch);
  if (st != GC_OK) return st;
  return gc_ef_topk_compress(dev, host, g, e, idx, val, q, scale, seed, iter, flags, scratch,
                             kStaticBytes, stream);
}

extern "C" gc_status gc_ef_topk_compress_noalloc_status(void* stream, gc_diag* out) {
  NvtxRange nvtx_range("gc_ef_topk_compress_noalloc_status");
  if (!out) return GC_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const gc_status st = scratch_for_current_device(&scratch);
  if (st != GC_OK) return st;
  // the diagnostic words sit at the head of the scratch, as in a workspace
  return gc_get_device_status(scratch, kStaticBytes, stream, out);
}
