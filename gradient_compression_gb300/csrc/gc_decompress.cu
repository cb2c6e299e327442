// Receiver of sparse payloads (sm_103a): out += sum over workers of their
// sparse vectors (mbrenndoerfer.com "Gradient Compression": the received
// gradient is the union of different sparse vectors; inferensys.com zh
// glossary: all-gather of indices and values, then a local sum).
//
// Workers are applied in order w = 0..W-1, one launch each, so every output
// element receives its contributions in worker order (deterministic fp32
// sums).  Within a worker the indices of a tensor are distinct, so no
// atomics are needed.
#include <cstring>

#include "gc_common.cuh"
#include "gc_host.h"

namespace gc {

struct SparseArgs {
  int T;
  const int64_t* off;
  const int64_t* koff;
  const int32_t* idx;
  const float* val;
  const int8_t* q;
  const float* scale;
  float* out;
  uint32_t* diag;
  int64_t K;
};

constexpr int SP_THREADS = 256;
constexpr int SP_PER_THREAD = 4;

__global__ void __launch_bounds__(SP_THREADS) k_scatter_add(SparseArgs A) {
  const int64_t first = ((int64_t)blockIdx.x * SP_THREADS * SP_PER_THREAD) + threadIdx.x;
  int t = -1;
  int64_t t_end = -1, base = 0, n = 0;
#pragma unroll
  for (int j = 0; j < SP_PER_THREAD; ++j) {
    const int64_t p = first + (int64_t)j * SP_THREADS;
    if (p >= A.K) break;
    if (p >= t_end) {
      t = find_segment(A.koff, A.T, p);
      t_end = A.koff[t + 1];
      base = A.off[t];
      n = A.off[t + 1] - base;
    }
    const int32_t i = A.idx[p];
    if (i < 0 || (int64_t)i >= n) {
      atomicOr(A.diag + DIAG_ERR, GC_DIAG_INDEX_RANGE);
      continue;
    }
    const float v = A.val ? A.val[p] : __fmul_rn((float)A.q[p], A.scale[t]);
    float* o = A.out + base + i;
    *o = __fadd_rn(*o, v);
  }
}

}  // namespace gc

using namespace gc;

extern "C" gc_status gc_sparse_decompress_accumulate(const gc_layout* dev, const gc_layout* host,
                                                     int32_t W, const int32_t* const* idx,
                                                     const float* const* val,
                                                     const int8_t* const* q,
                                                     const float* const* scale, float* out,
                                                     void* workspace, size_t ws_bytes,
                                                     void* stream) {
  NvtxRange nvtx_range("gc_sparse_decompress_accumulate");
  gc_status st = validate_layout(host, true);
  if (st != GC_OK) return st;
  if (!dev || !dev->off || !dev->koff || dev->num_tensors != host->num_tensors) return GC_ERR_INVALID_ARG;
  if (W < 0 || !out || (W > 0 && !idx)) return GC_ERR_INVALID_ARG;
  const bool fp32 = val != nullptr;
  if (W > 0 && !fp32 && (!q || !scale)) return GC_ERR_INVALID_ARG;
  for (int w = 0; w < W; ++w) {
    if (!idx[w]) return GC_ERR_INVALID_ARG;
    if (fp32 ? !val[w] : (!q[w] || !scale[w])) return GC_ERR_INVALID_ARG;
  }
  if (!aligned16(out)) return GC_ERR_ALIGNMENT;
  if (!workspace || ((uintptr_t)workspace & 255u) || ws_bytes < DIAG_BYTES) return GC_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, DIAG_BYTES, s) != cudaSuccess) return GC_ERR_CUDA;
  const int64_t K = host->koff[host->num_tensors];
  if (K == 0) return GC_OK;
  SparseArgs A;
  memset(&A, 0, sizeof A);
  A.T = host->num_tensors;
  A.off = dev->off;
  A.koff = dev->koff;
  A.out = out;
  A.diag = static_cast<uint32_t*>(workspace);
  A.K = K;
  const int64_t per_block = (int64_t)SP_THREADS * SP_PER_THREAD;
  const unsigned grid = (unsigned)((K + per_block - 1) / per_block);
  for (int w = 0; w < W; ++w) {
    A.idx = idx[w];
    A.val = fp32 ? val[w] : nullptr;
    A.q = fp32 ? nullptr : q[w];
    A.scale = fp32 ? nullptr : scale[w];
    k_scatter_add<<<grid, SP_THREADS, 0, s>>>(A);
  }
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}
