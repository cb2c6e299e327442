// libgc entry points that are not tied to one operation.
#include <cuda_runtime.h>

#include <cmath>

#include "gc_common.cuh"
#include "gc_host.h"

using namespace gc;

extern "C" gc_status gc_workspace_size(const gc_layout* host, int32_t op, uint32_t flags,
                                       size_t* bytes) {
  if (!bytes) return GC_ERR_INVALID_ARG;
  switch (op) {
    case GC_OP_TOPK:
    case GC_OP_MOMENTUM: {
      const gc_status st = validate_layout(host, true);
      if (st != GC_OK) return st;
      const bool sampled = !(op == GC_OP_TOPK && (flags & GC_RANDK));
      *bytes = topk_workspace_bytes(host, sampled);
      return GC_OK;
    }
    case GC_OP_SIGN:
    case GC_OP_QUANTIZE: {
      const gc_status st = validate_layout(host, false);
      if (st != GC_OK) return st;
      *bytes = dense_workspace_bytes(host);
      return GC_OK;
    }
    case GC_OP_DECOMPRESS: {
      gc_status st = validate_layout(host, false);
      if (st != GC_OK) return st;
      size_t b = dense_workspace_bytes(host);
      if (host->k && host->koff) {  // sparse receivers: window tables and starts
        st = validate_layout(host, true);
        if (st != GC_OK) return st;
        const size_t sb = sparse_decompress_workspace_bytes(host);
        b = sb > b ? sb : b;
      }
      *bytes = b;
      return GC_OK;
    }
    default:
      return GC_ERR_INVALID_ARG;
  }
}

extern "C" gc_status gc_get_device_status(const void* workspace, size_t ws_bytes, void* stream,
                                          gc_diag* out) {
  NvtxRange nvtx_range("gc_get_device_status");
  if (!workspace || ws_bytes < DIAG_BYTES || !out) return GC_ERR_INVALID_ARG;
  uint32_t w[5] = {0u, 0u, 0u, 0u, 0u};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(w, workspace, sizeof w, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GC_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GC_ERR_CUDA;
  out->error_bits = w[DIAG_ERR];
  out->exact_tensors = w[DIAG_EXACT];
  out->overflow_tensors = w[DIAG_OVF];
  out->one_launch = w[DIAG_PATH];
  return w[DIAG_ERR] ? GC_ERR_DEVICE : GC_OK;
}

extern "C" const char* gc_status_string(gc_status s) {
  switch (s) {
    case GC_OK: return "ok";
    case GC_ERR_INVALID_ARG: return "invalid argument";
    case GC_ERR_LAYOUT: return "invalid layout";
    case GC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case GC_ERR_ALIGNMENT: return "data pointer not 16-byte aligned";
    case GC_ERR_CUDA: return "CUDA launch or copy failed";
    case GC_ERR_DEVICE: return "device reported an error";
  }
  return "unknown status";
}

extern "C" int32_t gc_version(void) { return 100; }

extern "C" double gc_warmup_density(int64_t step, int64_t warmup_steps, double rho_start,
                                    double rho_final, int32_t kind, int32_t stages) {
  if (warmup_steps <= 0 || step >= warmup_steps) return rho_final;
  if (step < 0) step = 0;
  double f = (double)step / (double)warmup_steps;
  if (kind == 2 && stages > 0) f = floor(f * stages) / stages;
  if (kind == 0) return rho_start + (rho_final - rho_start) * f;
  return rho_start * pow(rho_final / rho_start, f);
}
