// Receiver of sparse payloads (sm_103a): out += sum over workers of their
// sparse vectors (mbrenndoerfer.com "Gradient Compression": the received
// gradient is the union of different sparse vectors; inferensys.com zh
// glossary: all-gather of indices and values, then a local sum).
//
// Every worker's entries of a tensor are in ascending index order (as every
// compressor here emits them).  The arena is cut into windows of a power of
// two elements per tensor, sized so that a window holds about DW_TARGET
// entries of each worker.  One CTA owns a window and adds the window's
// entries of up to DW_GROUP workers worker by worker, with a barrier between
// workers: each element receives its contributions in worker order (the
// sequential w = 0..W-1 sum, bit for bit), and windows are disjoint, so no
// two CTAs touch one element.  The additions are L2 atomics (one request per
// entry instead of a load and a store, and the L2 fetches one 32-byte sector
// for it instead of a whole line on a read miss), made exact where the
// hardware's flush of subnormals could change a sum.
//
// Each entry is a random 32-byte read-modify-write in DRAM; that, not the
// payload stream, bounds the pass.  Launches per group of DW_GROUP workers:
// window starts (a binary search per worker and window), then the window
// pass; a plan kernel builds the per-tensor window tables once per call.
#include <cstring>

#include "gc_common.cuh"
#include "gc_host.h"

namespace gc {

constexpr int DW_GROUP = 8;        // workers applied by one launch
constexpr int DW_THREADS = 256;
constexpr int64_t DW_TARGET = 192; // a window holds DW_TARGET / 2 .. DW_TARGET entries per worker

// Payload decoders (value of entry p of worker w in tensor t).
enum { DK_F32 = 0, DK_INT8 = 1, DK_QSGD = 2, DK_SIGN = 3 };

// log2 of tensor t's window size: floor(log2(DW_TARGET * n / k)), so that a
// window covers DW_TARGET / 2 .. DW_TARGET entries of a worker at density
// k / n; between 5 and 31.
__host__ __device__ inline int window_shift(int64_t n, int64_t k) {
  if (k <= 0) return 31;
  int64_t q = (DW_TARGET * n) / k;  // >= DW_TARGET
  int s = 0;
  while (s < 31 && (INT64_C(2) << s) <= q) ++s;
  return s < 5 ? 5 : s;
}
__host__ __device__ inline int64_t windows_of(int64_t n, int64_t k) {
  return k > 0 ? ((n - 1) >> window_shift(n, k)) + 1 : 0;
}

struct DecompArgs {
  int T;
  int W;  // workers in this launch (<= DW_GROUP)
  int s_levels;
  const int64_t* off;
  const int64_t* koff;
  const int32_t* idx[DW_GROUP];
  const float* val[DW_GROUP];
  const int8_t* q[DW_GROUP];
  const uint32_t* bits[DW_GROUP];
  const float* scale[DW_GROUP];
  float* out;
  uint32_t* diag;
  int64_t* wo;      // [T+1] first window of each tensor
  int32_t* wsh;     // [T]   log2 of the tensor's window size
  int64_t* kwoff;   // [T+1] first sign-bit word of each tensor (DK_SIGN)
  int64_t* starts;  // [DW_GROUP][NW+1] first entry of each window, per worker
  int64_t NW, K;        // windows; K = koff[T], the end of the entries
  int64_t off0, koff0;  // off[0] and koff[0] of the host layout (nonzero for a bucket)
};

// Window tables from the device layout (one CTA); a disagreement with the
// host's window count means the device and host layouts differ.
__global__ void __launch_bounds__(1024) k_dplan(DecompArgs A) {
  chain_wait();
  __shared__ int64_t s_w[32], s_b[32];
  int64_t carry = 0, carry_b = 0;
  for (int base = 0; base < A.T; base += blockDim.x) {
    const int t = base + threadIdx.x;
    int64_t nw = 0, nb = 0;
    if (t < A.T) {
      const int64_t n = A.off[t + 1] - A.off[t], k = A.koff[t + 1] - A.koff[t];
      A.wsh[t] = window_shift(n, k);
      nw = windows_of(n, k);
      nb = (k + 31) >> 5;
    }
    // block-wide exclusive scans of nw and nb
    int64_t x = nw, y = nb;
    const unsigned lane = lane_id(), w = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t a = __shfl_up_sync(FULL, x, d), b = __shfl_up_sync(FULL, y, d);
      if (lane >= (unsigned)d) {
        x += a;
        y += b;
      }
    }
    if (lane == 31) {
      s_w[w] = x;
      s_b[w] = y;
    }
    __syncthreads();
    int64_t bw = 0, bb = 0, tw = 0, tb = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
      if (i < (int)w) {
        bw += s_w[i];
        bb += s_b[i];
      }
      tw += s_w[i];
      tb += s_b[i];
    }
    if (t < A.T) {
      A.wo[t] = carry + bw + x - nw;
      A.kwoff[t] = carry_b + bb + y - nb;
    }
    carry += tw;
    carry_b += tb;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    A.wo[A.T] = carry;
    A.kwoff[A.T] = carry_b;
    if (carry != A.NW || A.off[0] != A.off0 || A.koff[0] != A.koff0 || A.koff[A.T] != A.K) {
      A.diag[DIAG_ERR] |= GC_DIAG_LAYOUT_MISMATCH;
      A.diag[DIAG_ABORT] = 1u;
    }
  }
}

// starts[w][gw] = first entry of worker w's tensor at or after window gw's
// first element (window 0 of a tensor starts at the tensor's first entry, so
// that every entry, even one with a negative index, lands in some window);
// starts[w][NW] = K.
__global__ void __launch_bounds__(256) k_dstarts(DecompArgs A) {
  chain_wait();
  if (A.diag[DIAG_ABORT]) return;
  const int64_t stride = A.NW + 1;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= stride * A.W) return;
  const int w = (int)(i / stride);
  const int64_t gw = i - (int64_t)w * stride;
  int64_t r;
  if (gw == A.NW) {
    r = A.K;
  } else {
    const int t = find_segment(A.wo, A.T, gw);
    const int64_t j = gw - A.wo[t];
    r = A.koff[t];
    if (j > 0) {
      const int64_t x = j << A.wsh[t];
      const int32_t* ix = A.idx[w];
      int64_t lo = A.koff[t], hi = A.koff[t + 1];  // first entry with index >= x
      while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)__ldg(ix + mid) < x)
          lo = mid + 1;
        else
          hi = mid;
      }
      r = lo;
    }
  }
  A.starts[i] = r;
}

template <int DK>
__device__ __forceinline__ float decode_entry(const DecompArgs& A, int w, int t, int64_t p) {
  if (DK == DK_F32) return A.val[w][p];
  if (DK == DK_INT8) return __fmul_rn((float)A.q[w][p], A.scale[w][t]);
  if (DK == DK_QSGD) {
    const int c = A.q[w][p];
    const int level = c < 0 ? -c : c;
    const float mag = __fdiv_rn(__fmul_rn((float)level, A.scale[w][t]), (float)A.s_levels);
    return c < 0 ? -mag : mag;
  }
  const int64_t j = p - A.koff[t];
  const uint32_t word = A.bits[w][A.kwoff[t] + (j >> 5)];
  const float mu = A.scale[w][t];
  return ((word >> (j & 31)) & 1u) ? mu : -mu;
}

// Reports an entry whose index lies outside its window: out of the tensor
// (GC_DIAG_INDEX_RANGE), or out of ascending order (GC_DIAG_INDEX_ORDER,
// the entry belongs to another window).  Such entries are skipped: adding
// them could race with the CTA that owns their window.
__device__ __forceinline__ void flag_entry(const DecompArgs& A, int64_t x, int64_t n) {
  atomicOr(A.diag + DIAG_ERR, (x < 0 || x >= n) ? GC_DIAG_INDEX_RANGE : GC_DIAG_INDEX_ORDER);
}

// No flush to zero can change a sum with this operand: zero, or at least
// 2^-103 in magnitude (two such operands are multiples of 2^-126, so their
// sum is zero or normal).
__device__ __forceinline__ bool ftz_safe(float x) { return x == 0.0f || fabsf(x) >= 0x1p-103f; }

// out[x] += v as one L2 atomic.  The hardware's fp32 atomic add rounds to
// nearest even but flushes subnormal operands and results to zero; where
// that can matter, the IEEE sum (from the returned old value) is written
// over it.  Nothing else updates out[x] before the caller's next barrier.
__device__ __forceinline__ void add_exact(float* o, float v) {
  const float old = atomicAdd(o, v);
  const float r = __fadd_rn(old, v);
  if (!(ftz_safe(old) && ftz_safe(v))) atomicExch(o, r);
}

// One CTA per window: the workers' entries of the window are added worker
// after worker, a barrier between workers, so each element receives its
// contributions in worker order.  Within a worker the window's indices are
// distinct, so the atomics of one phase never meet on an element.
template <int DK>
__global__ void __launch_bounds__(DW_THREADS) k_dphase(DecompArgs A) {
  chain_wait();
  __shared__ int64_t s_s[DW_GROUP], s_e[DW_GROUP];
  if (A.diag[DIAG_ABORT]) return;
  const int64_t gw = blockIdx.x;
  const int t = find_segment(A.wo, A.T, gw);
  const int64_t base = A.off[t], n = A.off[t + 1] - base;
  const int64_t wlo = (gw - A.wo[t]) << A.wsh[t];
  const int64_t whi = min(wlo + (INT64_C(1) << A.wsh[t]), n);
  const int64_t stride = A.NW + 1;
  if ((int)threadIdx.x < A.W) {
    s_s[threadIdx.x] = A.starts[(int64_t)threadIdx.x * stride + gw];
    s_e[threadIdx.x] = A.starts[(int64_t)threadIdx.x * stride + gw + 1];
  }
  __syncthreads();
  float* out = A.out + base;
  for (int w = 0; w < A.W; ++w) {
    const int32_t* ix = A.idx[w];
    for (int64_t p = s_s[w] + threadIdx.x; p < s_e[w]; p += DW_THREADS) {
      const int64_t x = ix[p];
      if (x < wlo || x >= whi) {
        flag_entry(A, x, n);
        continue;
      }
      if (p > s_s[w] && ix[p - 1] >= x) atomicOr(A.diag + DIAG_ERR, GC_DIAG_INDEX_ORDER);
      add_exact(out + x, decode_entry<DK>(A, w, t, p));
    }
    __syncthreads();  // worker w's sums are complete before worker w + 1 adds
  }
}

static size_t carve_decomp(int T, int64_t NW, size_t* o_wo, size_t* o_wsh, size_t* o_kw, size_t* o_st) {
  size_t p = DIAG_BYTES;
  auto take = [&p](size_t bytes) {
    const size_t at = p;
    p = align_up(p + bytes, 256);
    return at;
  };
  *o_wo = take(8 * (size_t)(T + 1));
  *o_wsh = take(4 * (size_t)T);
  *o_kw = take(8 * (size_t)(T + 1));
  *o_st = take(8 * (size_t)DW_GROUP * (size_t)(NW + 1));
  return p;
}

static int64_t windows_total(const gc_layout* h) {
  int64_t nw = 0;
  for (int t = 0; t < h->num_tensors; ++t) nw += windows_of(h->off[t + 1] - h->off[t], h->k[t]);
  return nw;
}

size_t sparse_decompress_workspace_bytes(const gc_layout* h) {
  size_t a, b, c, d;
  return carve_decomp(h->num_tensors, windows_total(h), &a, &b, &c, &d);
}

static gc_status run_decompress(int dk, const gc_layout* dev, const gc_layout* host, int32_t W,
                                const int32_t* const* idx, const float* const* val,
                                const int8_t* const* q, const uint32_t* const* bits,
                                const float* const* scale, int32_t s_levels, float* out,
                                void* workspace, size_t ws_bytes, void* stream) {
  gc_status st = validate_layout(host, true);
  if (st != GC_OK) return st;
  if (!dev || !dev->off || !dev->koff || dev->num_tensors != host->num_tensors) return GC_ERR_INVALID_ARG;
  if (W < 0 || !out || (W > 0 && !idx)) return GC_ERR_INVALID_ARG;
  for (int w = 0; w < W; ++w) {
    if (!idx[w]) return GC_ERR_INVALID_ARG;
    const bool ok = dk == DK_F32 ? (val && val[w])
                    : dk == DK_SIGN ? (bits && bits[w] && scale && scale[w])
                                    : (q && q[w] && scale && scale[w]);
    if (!ok) return GC_ERR_INVALID_ARG;
  }
  if (!aligned16(out)) return GC_ERR_ALIGNMENT;
  const int T = host->num_tensors;
  const int64_t NW = windows_total(host);
  size_t o_wo, o_wsh, o_kw, o_st;
  const size_t need = carve_decomp(T, NW, &o_wo, &o_wsh, &o_kw, &o_st);
  if (!workspace || ((uintptr_t)workspace & 255u) || ws_bytes < need) return GC_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!zero_chained(workspace, DIAG_BYTES, s)) return GC_ERR_CUDA;
  const int64_t K = host->koff[T];
  if (K == host->koff[0] || W == 0) return GC_OK;
  unsigned char* wsp = static_cast<unsigned char*>(workspace);
  DecompArgs A;
  memset(&A, 0, sizeof A);
  A.T = T;
  A.s_levels = s_levels;
  A.off = dev->off;
  A.koff = dev->koff;
  A.out = out;
  A.diag = reinterpret_cast<uint32_t*>(wsp);
  A.wo = reinterpret_cast<int64_t*>(wsp + o_wo);
  A.wsh = reinterpret_cast<int32_t*>(wsp + o_wsh);
  A.kwoff = reinterpret_cast<int64_t*>(wsp + o_kw);
  A.starts = reinterpret_cast<int64_t*>(wsp + o_st);
  A.NW = NW;
  A.K = K;
  A.off0 = host->off[0];
  A.koff0 = host->koff[0];
  launch_chained(k_dplan, 1, 1024, 0, s, A);
  for (int w0 = 0; w0 < W; w0 += DW_GROUP) {
    A.W = W - w0 < DW_GROUP ? W - w0 : DW_GROUP;
    for (int j = 0; j < DW_GROUP; ++j) {
      const bool in = j < A.W;
      A.idx[j] = in ? idx[w0 + j] : nullptr;
      A.val[j] = in && val ? val[w0 + j] : nullptr;
      A.q[j] = in && q ? q[w0 + j] : nullptr;
      A.bits[j] = in && bits ? bits[w0 + j] : nullptr;
      A.scale[j] = in && scale ? scale[w0 + j] : nullptr;
    }
    const int64_t nthr = (NW + 1) * A.W;
    launch_chained(k_dstarts, (unsigned)((nthr + 255) / 256), 256, 0, s, A);
    if (NW > 0) {
      switch (dk) {
        case DK_F32: launch_chained(k_dphase<DK_F32>, (unsigned)NW, DW_THREADS, 0, s, A); break;
        case DK_INT8: launch_chained(k_dphase<DK_INT8>, (unsigned)NW, DW_THREADS, 0, s, A); break;
        case DK_QSGD: launch_chained(k_dphase<DK_QSGD>, (unsigned)NW, DW_THREADS, 0, s, A); break;
        default: launch_chained(k_dphase<DK_SIGN>, (unsigned)NW, DW_THREADS, 0, s, A); break;
      }
    }
  }
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
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
  return run_decompress(val ? DK_F32 : DK_INT8, dev, host, W, idx, val, q, nullptr, scale, 0, out,
                        workspace, ws_bytes, stream);
}

extern "C" gc_status gc_sparse_decompress_accumulate_quantized(
    const gc_layout* dev, const gc_layout* host, int32_t W, int32_t kind, int32_t s_levels,
    const int32_t* const* idx, const int8_t* const* q, const uint32_t* const* bits,
    const float* const* scale, float* out, void* workspace, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("gc_sparse_decompress_accumulate_quantized");
  int dk;
  switch (kind) {
    case GC_KEPT_INT8: dk = DK_INT8; break;
    case GC_KEPT_QSGD:
      if (s_levels < 1 || s_levels > 127) return GC_ERR_INVALID_ARG;
      dk = DK_QSGD;
      break;
    case GC_KEPT_SIGN: dk = DK_SIGN; break;
    default: return GC_ERR_INVALID_ARG;
  }
  return run_decompress(dk, dev, host, W, idx, nullptr, q, bits, scale, s_levels, out, workspace,
                        ws_bytes, stream);
}
