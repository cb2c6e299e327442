// Host-side helpers of libgc: argument validation and workspace sizing.
#pragma once

#include <nvtx3/nvToolsExt.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gc.h"

namespace gc {

// Names the enclosing host scope (an entry point, or the enqueueing of one
// phase of it) in profiler timelines: an NVTX range, which costs nothing
// when no profiler is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0u; }

// Checks a host layout: T >= 1, off[0] >= 0, 1 <= n_t < 2^31; with
// `sparse`, also 0 <= k_t <= n_t, koff[0] >= 0 and koff[t+1] - koff[t] = k_t.
// off[0] > 0 or koff[0] > 0: the layout is a bucket, a contiguous range of
// tensors of a larger arena, addressed with that arena's element and entry
// offsets.
inline gc_status validate_layout(const gc_layout* h, bool sparse) {
  if (!h || h->num_tensors < 1 || !h->off) return GC_ERR_INVALID_ARG;
  if (sparse && (!h->k || !h->koff)) return GC_ERR_INVALID_ARG;
  if (h->off[0] < 0) return GC_ERR_LAYOUT;
  if (sparse && h->koff[0] < 0) return GC_ERR_LAYOUT;
  for (int t = 0; t < h->num_tensors; ++t) {
    const int64_t n = h->off[t + 1] - h->off[t];
    if (n < 1 || n > INT64_C(2147483647)) return GC_ERR_LAYOUT;
    if (sparse) {
      const int64_t k = h->k[t];
      if (k < 0 || k > n) return GC_ERR_LAYOUT;
      if (h->koff[t + 1] - h->koff[t] != k) return GC_ERR_LAYOUT;
    }
  }
  return GC_OK;
}

// Defined by the operation files.
size_t topk_workspace_bytes(const gc_layout* h, bool sampled);
size_t dense_workspace_bytes(const gc_layout* h);
size_t sparse_decompress_workspace_bytes(const gc_layout* h);

}  // namespace gc
