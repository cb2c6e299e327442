// PowerSGD with error feedback (sm_103a).
//
// Method: mbrenndoerfer.com "Gradient Compression", PowerSGD section: each
// gradient matrix G (m x n) is sent as P (m x r) and Q (n x r) with
// G ~ P Q^T, found by power iteration (alternating updates of P and Q) with
// error feedback on G - P Q^T; chipfoundryservices.com glossary: rank-4
// PowerSGD.  One warm-started power-iteration step per call:
//   M = G + E;  P = M Q;  orthonormalize P (modified Gram-Schmidt);
//   Q = M^T P;  E = M - P Q^T.
//
// With r <= 4 the products are skinny (about one flop per byte of M), so
// they are HBM-bound streaming passes on the CUDA cores, not tensor-core
// GEMMs.  Passes over the matrices:
//   k_pmq   warp per PS_RB rows: M = G + E (stored into E), P_raw = M Q
//   k_porth one CTA per matrix: Gram-Schmidt on P (fixed-order sums)
//   k_pmtp  256 x 1024 tiles of M: partial column sums of M^T P
//   k_pqred fixed-order sum of the partials -> Q
//   k_pres  warp per row: E = M - P Q^T
// Reductions: fused multiply-add partial sums in fp32 over a few terms,
// added into a compensated fp32 accumulator per thread, then combined across
// lanes, warps and tiles by compensated fp32 additions in a fixed order
// (deterministic; no fp64 arithmetic, which is slow on this part);
// elementwise steps are single fp32 roundings in the order the method
// states them.
#include <cstring>

#include "gc_common.cuh"
#include "gc_host.h"

namespace gc {

constexpr int PS_RC = 256;   // rows per Q tile
constexpr int PS_CC = 1024;  // columns per Q tile (256 threads x 4)
// Launch shapes of the streaming passes (compile-time; the defaults are the
// measured best on the BERT-large weight matrices).
#ifndef GC_PS_RB
#define GC_PS_RB 2
#endif
#ifndef GC_PS_CU
#define GC_PS_CU 1
#endif
#ifndef GC_PS_RS
#define GC_PS_RS 4
#endif
#ifndef GC_PS_PMTP_MINB
#define GC_PS_PMTP_MINB 3
#endif
#ifndef GC_PS_RESVEC
#define GC_PS_RESVEC 0
#endif
constexpr int PS_RB = GC_PS_RB;        // rows per warp in P = M Q
constexpr int PS_CU = GC_PS_CU;        // 128-column groups per step in P = M Q
constexpr int PS_RS = GC_PS_RS;        // rows per step in M^T P
constexpr bool PS_RESVEC = GC_PS_RESVEC != 0;  // 16-byte accesses in E = M - P Q^T
// Terms summed in plain fp32 (fused multiply-adds) before each compensated
// addition in P = M Q and M^T P: the partial's rounding error is at most
// (PS_FLUSH - 1) u of the sum of |terms| (u = 2^-24), below 1e-6 of it.
constexpr int PS_FLUSH = 16;

struct PsArgs {
  int T;
  const int64_t* start;
  const int64_t* rows;
  const int64_t* cols;
  const float* g;
  float* e;
  float* q;
  float* p;
  float* p_raw;
  float* out;
  uint32_t* diag;
  int64_t* rowoff;   // [T+1] prefix of m
  int64_t* coloff;   // [T+1] prefix of n
  int64_t* tileoff;  // [T+1] prefix of Q tiles
  int64_t* partoff;  // [T+1] prefix of ceil(m / PS_RC) * n
  int64_t* blkoff;   // [T+1] prefix of ceil(m / PS_RB)
  float* part;       // partial column sums, [partoff][R]
  int64_t Mrows, Ncols, Tiles, Parts, Blocks;
};

__device__ __forceinline__ bool ps_aborted(const PsArgs& A) { return A.diag[DIAG_ABORT] != 0u; }

__global__ void __launch_bounds__(1024) k_psplan(PsArgs A) {
  __shared__ int64_t s_warp[32];
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  int64_t carry[5] = {0, 0, 0, 0, 0};
  int64_t* outs[5] = {A.rowoff, A.coloff, A.tileoff, A.partoff, A.blkoff};
  for (int base = 0; base < A.T; base += blockDim.x) {
    const int t = base + threadIdx.x;
    int64_t v[5] = {0, 0, 0, 0, 0};
    if (t < A.T) {
      const int64_t m = A.rows[t], n = A.cols[t];
      if (m < 1 || n < 1 || A.start[t] < 0) s_bad = 1;
      const int64_t rc = (m + PS_RC - 1) / PS_RC;
      v[0] = m;
      v[1] = n;
      v[2] = rc * ((n + PS_CC - 1) / PS_CC);
      v[3] = rc * n;
      v[4] = (m + PS_RB - 1) / PS_RB;
    }
    for (int w = 0; w < 5; ++w) {
      const unsigned lane = lane_id(), wi = threadIdx.x >> 5, nw = blockDim.x >> 5;
      int64_t x = v[w];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int64_t y = __shfl_up_sync(FULL, x, d);
        if (lane >= (unsigned)d) x += y;
      }
      if (lane == 31) s_warp[wi] = x;
      __syncthreads();
      if (wi == 0) {
        int64_t z = lane < nw ? s_warp[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int64_t y = __shfl_up_sync(FULL, z, d);
          if (lane >= (unsigned)d) z += y;
        }
        if (lane < nw) s_warp[lane] = z;
      }
      __syncthreads();
      const int64_t excl = (wi == 0 ? 0 : s_warp[wi - 1]) + x - v[w];
      const int64_t tot = s_warp[nw - 1];
      __syncthreads();
      if (t < A.T) outs[w][t] = carry[w] + excl;
      carry[w] += tot;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 0; w < 5; ++w) outs[w][A.T] = carry[w];
    if (s_bad || carry[0] != A.Mrows || carry[1] != A.Ncols || carry[2] != A.Tiles || carry[3] != A.Parts ||
        carry[4] != A.Blocks) {
      A.diag[DIAG_ERR] |= GC_DIAG_LAYOUT_MISMATCH;
      A.diag[DIAG_ABORT] = 1u;
    }
  }
}

struct Nm {
  float s = 0.0f, c = 0.0f;
  __device__ __forceinline__ void add(float x) {
    const float t = __fadd_rn(s, x);
    if (fabsf(s) >= fabsf(x))
      c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, t), x));
    else
      c = __fadd_rn(c, __fadd_rn(__fsub_rn(x, t), s));
    s = t;
  }
  // RN(s + c): the sum rounded once to fp32 (no fp64 arithmetic, which is
  // slow on this part)
  __device__ __forceinline__ float value() const { return __fadd_rn(s, c); }
  // Combine with the same accumulator of lane (lane ^ d): fp32 addition is
  // commutative and the compensation is symmetric in its operands, so both
  // partners end with identical values (fixed butterfly order).
  __device__ __forceinline__ void butterfly(int d) {
    const float os = __shfl_xor_sync(FULL, s, d);
    const float oc = __shfl_xor_sync(FULL, c, d);
    add(os);
    c = __fadd_rn(c, oc);
  }
};

// The R values of row j of Q or P (16- or 8-byte aligned for R = 4, 2).
template <int R>
__device__ __forceinline__ void load_row(const float* base, float v[R]) {
  if (R == 4) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(base));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else if (R == 2) {
    const float2 x = __ldg(reinterpret_cast<const float2*>(base));
    v[0] = x.x; v[1] = x.y;
  } else {
#pragma unroll
    for (int k = 0; k < R; ++k) v[k] = __ldg(base + k);
  }
}

// Store row i's P_raw from the lane-distributed accumulators (lane 0 writes).
template <int R>
__device__ __forceinline__ void pmq_emit(const PsArgs& A, int t, int64_t i, Nm acc[R], unsigned lane) {
#pragma unroll
  for (int k = 0; k < R; ++k) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) acc[k].butterfly(d);
    if (lane == 0) {
      const float pv = acc[k].value();
      A.p[(A.rowoff[t] + i) * R + k] = pv;
      if (A.p_raw) A.p_raw[(A.rowoff[t] + i) * R + k] = pv;
    }
  }
}

// M = G + E (stored into E) and P_raw = M Q.  A warp takes a block of PS_RB
// consecutive rows of one matrix; lane l owns 4 consecutive columns of every
// 128-column group, so each Q row it loads serves all the block's rows.
// Products are fused multiply-adds summed in fp32 over PS_FLUSH columns, then
// added to a compensated accumulator per row, then reduced across lanes (a
// fixed butterfly) and rounded once to fp32: a fixed order throughout.
// Matrices with misaligned rows take a scalar path, one row at a time.
template <int R>
__global__ void __launch_bounds__(256) k_pmq(PsArgs A) {
  if (ps_aborted(A)) return;
  const unsigned lane = lane_id();
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t gb = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); gb < A.Blocks; gb += nwarps) {
    const int t = find_segment(A.blkoff, A.T, gb);
    const int64_t m = A.rows[t], n = A.cols[t];
    const int64_t i0 = (gb - A.blkoff[t]) * PS_RB;
    const int nr = (int)min((int64_t)PS_RB, m - i0);
    const float* qt = A.q + A.coloff[t] * R;
    if ((A.start[t] & 3) == 0 && (n & 3) == 0) {
      Nm acc[PS_RB][R];
      float part[PS_RB][R];
#pragma unroll
      for (int r = 0; r < PS_RB; ++r)
#pragma unroll
        for (int k = 0; k < R; ++k) part[r][k] = 0.0f;
      const int64_t nv = n >> 2;
      int half = 0;
      for (int64_t v0 = lane; v0 < nv; v0 += 32 * PS_CU) {
        float4 mv[PS_CU][PS_RB];
#pragma unroll
        for (int cu = 0; cu < PS_CU; ++cu) {
          const int64_t v = v0 + 32 * cu;
#pragma unroll
          for (int r = 0; r < PS_RB; ++r) {
            if (r < nr && v < nv) {
              const int64_t o = A.start[t] + (i0 + r) * n + 4 * v;
              const float4 gv = ld_stream(reinterpret_cast<const float4*>(A.g + o));
              const float4 ev = ld_stream(reinterpret_cast<const float4*>(A.e + o));
              mv[cu][r].x = __fadd_rn(gv.x, ev.x);
              mv[cu][r].y = __fadd_rn(gv.y, ev.y);
              mv[cu][r].z = __fadd_rn(gv.z, ev.z);
              mv[cu][r].w = __fadd_rn(gv.w, ev.w);
              st_stream(reinterpret_cast<float4*>(A.e + o), mv[cu][r]);
            } else {
              mv[cu][r] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
          }
        }
#pragma unroll
        for (int cu = 0; cu < PS_CU; ++cu) {
          const int64_t v = v0 + 32 * cu;
          float qv[4][R];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (v < nv) {
              load_row<R>(qt + (4 * v + c) * R, qv[c]);
            } else {
#pragma unroll
              for (int k = 0; k < R; ++k) qv[c][k] = 0.0f;
            }
          }
#pragma unroll
          for (int r = 0; r < PS_RB; ++r) {
            const float mm[4] = {mv[cu][r].x, mv[cu][r].y, mv[cu][r].z, mv[cu][r].w};
#pragma unroll
            for (int k = 0; k < R; ++k)
#pragma unroll
              for (int c = 0; c < 4; ++c) part[r][k] = __fmaf_rn(mm[c], qv[c][k], part[r][k]);
          }
          if (++half * 4 >= PS_FLUSH) {
#pragma unroll
            for (int r = 0; r < PS_RB; ++r)
#pragma unroll
              for (int k = 0; k < R; ++k) {
                acc[r][k].add(part[r][k]);
                part[r][k] = 0.0f;
              }
            half = 0;
          }
        }
      }
#pragma unroll
      for (int r = 0; r < PS_RB; ++r) {
#pragma unroll
        for (int k = 0; k < R; ++k) acc[r][k].add(part[r][k]);
        if (r < nr) pmq_emit<R>(A, t, i0 + r, acc[r], lane);
      }
    } else {
      for (int r = 0; r < nr; ++r) {
        const int64_t i = i0 + r;
        const int64_t rb = A.start[t] + i * n;
        Nm acc[R];
        for (int64_t j0 = lane; j0 < n; j0 += 256) {
          float mv[8], qv[8][R];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int64_t j = j0 + 32 * u;
            if (j < n) {
              mv[u] = __fadd_rn(__ldcs(A.g + rb + j), __ldcs(A.e + rb + j));
              __stcs(A.e + rb + j, mv[u]);
              load_row<R>(qt + j * R, qv[u]);
            } else {
              mv[u] = 0.0f;
#pragma unroll
              for (int k = 0; k < R; ++k) qv[u][k] = 0.0f;
            }
          }
#pragma unroll
          for (int k = 0; k < R; ++k) {
            float part = 0.0f;
#pragma unroll
            for (int u = 0; u < 8; ++u) part = __fmaf_rn(mv[u], qv[u][k], part);
            acc[k].add(part);
          }
        }
        pmq_emit<R>(A, t, i, acc, lane);
      }
    }
  }
}

// Modified Gram-Schmidt on the columns of P, one CTA of 1024 threads per
// matrix.  Every reduction is one pass over P's rows, and the update that
// uses a reduction's result (P_ik -= d P_ij, or P_ik /= nrm) is applied to
// each row as the next pass reads it: the same per-element operations in the
// same order as separate update loops.  Per-thread sums are the error-free
// product (fp32 product plus its exact FMA remainder) added to a compensated
// fp32 accumulator (Ogita, Rump and Oishi, "Accurate sum and dot product",
// 2005, Dot2); threads are combined by a fixed compensated butterfly in each
// warp and then across warps.
template <int R>
__device__ __forceinline__ float pick(const float v[R], int k) {
  float r = v[0];
#pragma unroll
  for (int c = 1; c < R; ++c)
    if (c == k) r = v[c];
  return r;
}

template <int R>
__device__ __forceinline__ void porth_row(float* row, float v[R], int ukind, int uk, int uj, float uval) {
  if (R == 4) {
    const float4 x = *reinterpret_cast<const float4*>(row);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else if (R == 2) {
    const float2 x = *reinterpret_cast<const float2*>(row);
    v[0] = x.x; v[1] = x.y;
  } else {
#pragma unroll
    for (int k = 0; k < R; ++k) v[k] = row[k];
  }
  if (ukind != 0) {
    const float vk = pick<R>(v, uk);
    const float nv = (ukind == 1) ? __fsub_rn(vk, __fmul_rn(uval, pick<R>(v, uj))) : __fdiv_rn(vk, uval);
#pragma unroll
    for (int k = 0; k < R; ++k)
      if (k == uk) v[k] = nv;
    row[uk] = nv;
  }
}

template <int R>
__global__ void __launch_bounds__(1024) k_porth(PsArgs A) {
  __shared__ float s_ws[32], s_wc[32];
  __shared__ float s_tot;
  if (ps_aborted(A)) return;
  const int t = blockIdx.x;
  const int64_t m = A.rows[t];
  float* P = A.p + A.rowoff[t] * R;
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  int ukind = 0, uk = 0, uj = 0;  // pending update: 0 none, 1 P_k -= d P_j, 2 P_k /= nrm
  float uval = 0.0f;
  for (int k = 0; k < R; ++k) {
    for (int j = 0; j <= k; ++j) {  // j < k: d = <P_j, P_k>;  j == k: |P_k|^2
      Nm acc;
      for (int64_t i0 = threadIdx.x; i0 < m; i0 += 4 * 1024) {
        float v[4][R];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t i = i0 + 1024 * u;
          if (i < m) porth_row<R>(P + i * R, v[u], ukind, uk, uj, uval);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t i = i0 + 1024 * u;
          if (i < m) {
            const float a = pick<R>(v[u], j), b = pick<R>(v[u], k);
            const float pr = __fmul_rn(a, b);
            acc.add(pr);
            acc.c = __fadd_rn(acc.c, __fmaf_rn(a, b, -pr));
          }
        }
      }
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) acc.butterfly(d);
      if (lane == 0) {
        s_ws[warp] = acc.s;
        s_wc[warp] = acc.c;
      }
      __syncthreads();
      if (warp == 0) {
        Nm w;
        w.s = s_ws[lane];
        w.c = s_wc[lane];
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) w.butterfly(d);
        if (lane == 0) s_tot = w.value();
      }
      __syncthreads();
      const float tot = s_tot;
      __syncthreads();
      if (j < k) {
        ukind = 1; uk = k; uj = j; uval = tot;
      } else {
        const float nrm = __fsqrt_rn(tot);
        ukind = nrm > 0.0f ? 2 : 0; uk = k; uval = nrm;
      }
    }
  }
  if (ukind != 0)
    for (int64_t i = threadIdx.x; i < m; i += 1024) {
      float v[R];
      porth_row<R>(P + i * R, v, ukind, uk, uj, uval);
    }
}

// Partial column sums of M^T P over a tile of PS_RC rows x PS_CC columns;
// thread = 4 consecutive columns.  PS_RS rows are loaded per step; fused
// multiply-adds are summed in fp32 over PS_FLUSH rows, then added to
// compensated accumulators.
template <int R>
__global__ void __launch_bounds__(256, GC_PS_PMTP_MINB) k_pmtp(PsArgs A) {
  constexpr int RS = PS_RS;  // rows per step
  if (ps_aborted(A)) return;
  const int64_t tile = blockIdx.x;
  const int t = find_segment(A.tileoff, A.T, tile);
  const int64_t m = A.rows[t], n = A.cols[t];
  const int64_t nd = (n + PS_CC - 1) / PS_CC;
  const int64_t local = tile - A.tileoff[t];
  const int64_t c = local / nd, d = local % nd;
  const int64_t j0 = d * PS_CC + 4 * threadIdx.x;
  const int64_t i0 = c * PS_RC, i1 = min(m, i0 + PS_RC);
  const float* P = A.p + A.rowoff[t] * R;
  const bool vec = ((A.start[t] & 3) == 0) && ((n & 3) == 0);
  Nm acc[4][R];
  float part[4][R];
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
#pragma unroll
    for (int k = 0; k < R; ++k) part[cc][k] = 0.0f;
  if (j0 < n) {
    int step = 0;
    for (int64_t ib = i0; ib < i1; ib += RS) {
      float mm[RS][4], pv[RS][R];
#pragma unroll
      for (int u = 0; u < RS; ++u) {
        const int64_t i = ib + u;
        if (i < i1) {
          const int64_t rb = A.start[t] + i * n;
          if (vec) {
            const float4 mv = ld_stream(reinterpret_cast<const float4*>(A.e + rb + j0));
            mm[u][0] = mv.x; mm[u][1] = mv.y; mm[u][2] = mv.z; mm[u][3] = mv.w;
          } else {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) mm[u][cc] = (j0 + cc < n) ? A.e[rb + j0 + cc] : 0.0f;
          }
          load_row<R>(P + i * R, pv[u]);
        } else {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) mm[u][cc] = 0.0f;
#pragma unroll
          for (int k = 0; k < R; ++k) pv[u][k] = 0.0f;
        }
      }
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
#pragma unroll
        for (int k = 0; k < R; ++k)
#pragma unroll
          for (int u = 0; u < RS; ++u) part[cc][k] = __fmaf_rn(mm[u][cc], pv[u][k], part[cc][k]);
      if (++step * RS >= PS_FLUSH) {  // fp32 partials span PS_FLUSH rows
        step = 0;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int k = 0; k < R; ++k) {
            acc[cc][k].add(part[cc][k]);
            part[cc][k] = 0.0f;
          }
      }
    }
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
#pragma unroll
      for (int k = 0; k < R; ++k) acc[cc][k].add(part[cc][k]);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      if (j0 + cc >= n) break;
      float* dst = A.part + (A.partoff[t] + c * n + j0 + cc) * R;
#pragma unroll
      for (int k = 0; k < R; ++k) dst[k] = acc[cc][k].value();
    }
  }
}

// Q_jk = sum over row tiles of the partials, in tile order (compensated fp32).
template <int R>
__global__ void __launch_bounds__(256) k_pqred(PsArgs A) {
  if (ps_aborted(A)) return;
  for (int64_t gc = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gc < A.Ncols;
       gc += (int64_t)gridDim.x * blockDim.x) {
    const int t = find_segment(A.coloff, A.T, gc);
    const int64_t j = gc - A.coloff[t], n = A.cols[t];
    const int64_t nc = (A.rows[t] + PS_RC - 1) / PS_RC;
    Nm s[R];
    const float* src = A.part + (A.partoff[t] + j) * R;
    int64_t c = 0;
    for (; c + 8 <= nc; c += 8) {  // eight row tiles' loads in flight, summed in tile order
      float v[8][R];
#pragma unroll
      for (int u = 0; u < 8; ++u) load_row<R>(src + (c + u) * n * R, v[u]);
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int k = 0; k < R; ++k) s[k].add(v[u][k]);
    }
    for (; c < nc; ++c) {
      float v[R];
      load_row<R>(src + c * n * R, v);
#pragma unroll
      for (int k = 0; k < R; ++k) s[k].add(v[k]);
    }
#pragma unroll
    for (int k = 0; k < R; ++k) A.q[gc * R + k] = s[k].value();
  }
}

// s_ij = sum_k P_ik Q_jk accumulated in k order in fp32, then
//   E = M - s (residual) or out += s (receiver); warp per row, lane per
//   column (each lane's Q row is one 16-byte load, coalesced across the
//   warp); with PS_RESVEC aligned rows go 4 columns per lane instead.
template <int R, bool DECODE>
__device__ __forceinline__ float pres_one(float x, const float pv[R], const float qv[R]) {
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < R; ++k) s = __fadd_rn(s, __fmul_rn(pv[k], qv[k]));
  return DECODE ? __fadd_rn(x, s) : __fsub_rn(x, s);
}

template <int R, bool DECODE>
__global__ void __launch_bounds__(256) k_pres(PsArgs A) {
  if (ps_aborted(A)) return;
  const unsigned lane = lane_id();
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  float* dstbase = DECODE ? A.out : A.e;
  for (int64_t gr = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); gr < A.Mrows; gr += nwarps) {
    const int t = find_segment(A.rowoff, A.T, gr);
    const int64_t i = gr - A.rowoff[t], n = A.cols[t];
    const int64_t rb = A.start[t] + i * n;
    const float* qt = A.q + A.coloff[t] * R;
    float pv[R];
    load_row<R>(A.p + (A.rowoff[t] + i) * R, pv);
    if (PS_RESVEC && (rb & 3) == 0 && (n & 3) == 0) {
      float4* d4 = reinterpret_cast<float4*>(dstbase + rb);
      const int64_t nv = n >> 2;
      for (int64_t v0 = lane; v0 < nv; v0 += 64) {
        float4 x[2];
        float qv[2][4][R];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int64_t v = v0 + 32 * u;
          if (v < nv) {
            x[u] = ld_stream(d4 + v);
#pragma unroll
            for (int c = 0; c < 4; ++c) load_row<R>(qt + (4 * v + c) * R, qv[u][c]);
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int64_t v = v0 + 32 * u;
          if (v < nv) {
            float4 y;
            y.x = pres_one<R, DECODE>(x[u].x, pv, qv[u][0]);
            y.y = pres_one<R, DECODE>(x[u].y, pv, qv[u][1]);
            y.z = pres_one<R, DECODE>(x[u].z, pv, qv[u][2]);
            y.w = pres_one<R, DECODE>(x[u].w, pv, qv[u][3]);
            st_stream(d4 + v, y);
          }
        }
      }
    } else {
      for (int64_t j0 = lane; j0 < n; j0 += 128) {
        float qv[4][R], x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t j = j0 + 32 * u;
          if (j < n) {
            load_row<R>(qt + j * R, qv[u]);
            x[u] = __ldcs(dstbase + rb + j);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t j = j0 + 32 * u;
          if (j < n) __stcs(dstbase + rb + j, pres_one<R, DECODE>(x[u], pv, qv[u]));
        }
      }
    }
  }
}

// ============================================================================ host

struct PsTotals {
  int64_t M = 0, N = 0, Tiles = 0, Parts = 0, Blocks = 0, maxel = 0;
};

static gc_status ps_validate(const gc_matrix_layout* h, int32_t rank, PsTotals* z) {
  if (!h || h->num_tensors < 1 || !h->start || !h->rows || !h->cols) return GC_ERR_INVALID_ARG;
  if (rank != 1 && rank != 2 && rank != 4) return GC_ERR_INVALID_ARG;
  for (int t = 0; t < h->num_tensors; ++t) {
    const int64_t m = h->rows[t], n = h->cols[t];
    if (m < 1 || n < 1 || h->start[t] < 0 || m > (INT64_C(1) << 40) / n) return GC_ERR_LAYOUT;
    const int64_t rc = (m + PS_RC - 1) / PS_RC;
    z->M += m;
    z->N += n;
    z->Tiles += rc * ((n + PS_CC - 1) / PS_CC);
    z->Parts += rc * n;
    z->Blocks += (m + PS_RB - 1) / PS_RB;
  }
  return GC_OK;
}

struct PsCarve {
  size_t o_row, o_col, o_tile, o_part_off, o_blk, o_part, total;
};

static PsCarve ps_carve(int T, int R, const PsTotals& z) {
  PsCarve c;
  size_t p = DIAG_BYTES;
  auto take = [&p](size_t bytes) {
    const size_t at = p;
    p = align_up(p + bytes, 256);
    return at;
  };
  c.o_row = take(8 * (size_t)(T + 1));
  c.o_col = take(8 * (size_t)(T + 1));
  c.o_tile = take(8 * (size_t)(T + 1));
  c.o_part_off = take(8 * (size_t)(T + 1));
  c.o_blk = take(8 * (size_t)(T + 1));
  c.o_part = take(4 * (size_t)z.Parts * R);
  c.total = p;
  return c;
}

template <class K>
static int ps_grid(K kernel, int64_t warps_of_work) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0);
  if (per_sm < 1) per_sm = 1;
  int64_t want = (warps_of_work + 7) / 8;
  int64_t grid = (int64_t)sms * per_sm;
  if (grid > want) grid = want;
  if (grid < 1) grid = 1;
  return (int)grid;
}

template <int R>
static void ps_launch_compress(const PsArgs& A, cudaStream_t s) {
  k_psplan<<<1, 1024, 0, s>>>(A);
  k_pmq<R><<<ps_grid(k_pmq<R>, A.Blocks), 256, 0, s>>>(A);
  k_porth<R><<<A.T, 1024, 0, s>>>(A);
  k_pmtp<R><<<(unsigned)A.Tiles, 256, 0, s>>>(A);
  k_pqred<R><<<(unsigned)std::min<int64_t>((A.Ncols + 255) / 256, 65535), 256, 0, s>>>(A);
  k_pres<R, false><<<ps_grid(k_pres<R, false>, A.Mrows), 256, 0, s>>>(A);
}

static gc_status ps_setup(const gc_matrix_layout* dev, const gc_matrix_layout* host, int32_t rank,
                          void* ws, size_t ws_bytes, cudaStream_t s, PsArgs* A) {
  PsTotals z;
  const gc_status st = ps_validate(host, rank, &z);
  if (st != GC_OK) return st;
  if (!dev || !dev->start || !dev->rows || !dev->cols || dev->num_tensors != host->num_tensors)
    return GC_ERR_INVALID_ARG;
  const PsCarve c = ps_carve(host->num_tensors, rank, z);
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < c.total) return GC_ERR_WORKSPACE;
  unsigned char* w = static_cast<unsigned char*>(ws);
  memset(A, 0, sizeof *A);
  A->T = host->num_tensors;
  A->start = dev->start;
  A->rows = dev->rows;
  A->cols = dev->cols;
  A->diag = reinterpret_cast<uint32_t*>(w);
  A->rowoff = reinterpret_cast<int64_t*>(w + c.o_row);
  A->coloff = reinterpret_cast<int64_t*>(w + c.o_col);
  A->tileoff = reinterpret_cast<int64_t*>(w + c.o_tile);
  A->partoff = reinterpret_cast<int64_t*>(w + c.o_part_off);
  A->blkoff = reinterpret_cast<int64_t*>(w + c.o_blk);
  A->part = reinterpret_cast<float*>(w + c.o_part);
  A->Mrows = z.M;
  A->Ncols = z.N;
  A->Tiles = z.Tiles;
  A->Parts = z.Parts;
  A->Blocks = z.Blocks;
  if (cudaMemsetAsync(ws, 0, DIAG_BYTES, s) != cudaSuccess) return GC_ERR_CUDA;
  return GC_OK;
}

}  // namespace gc

using namespace gc;

extern "C" gc_status gc_powersgd_workspace_size(const gc_matrix_layout* host, int32_t rank,
                                                size_t* bytes) {
  if (!bytes) return GC_ERR_INVALID_ARG;
  PsTotals z;
  const gc_status st = ps_validate(host, rank, &z);
  if (st != GC_OK) return st;
  *bytes = ps_carve(host->num_tensors, rank, z).total;
  return GC_OK;
}

extern "C" gc_status gc_powersgd_compress(const gc_matrix_layout* dev, const gc_matrix_layout* host,
                                          int32_t rank, const float* g, float* e, float* q, float* p,
                                          float* p_raw, void* workspace, size_t ws_bytes,
                                          void* stream) {
  if (!g || !e || !q || !p) return GC_ERR_INVALID_ARG;
  if (!aligned16(g) || !aligned16(e) || !aligned16(q) || !aligned16(p)) return GC_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PsArgs A;
  const gc_status st = ps_setup(dev, host, rank, workspace, ws_bytes, s, &A);
  if (st != GC_OK) return st;
  A.g = g;
  A.e = e;
  A.q = q;
  A.p = p;
  A.p_raw = p_raw;
  if (rank == 1)
    ps_launch_compress<1>(A, s);
  else if (rank == 2)
    ps_launch_compress<2>(A, s);
  else
    ps_launch_compress<4>(A, s);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

extern "C" gc_status gc_powersgd_decompress_accumulate(const gc_matrix_layout* dev,
                                                       const gc_matrix_layout* host, int32_t rank,
                                                       const float* p, const float* q, float* out,
                                                       void* workspace, size_t ws_bytes,
                                                       void* stream) {
  if (!p || !q || !out) return GC_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(p)) return GC_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PsArgs A;
  const gc_status st = ps_setup(dev, host, rank, workspace, ws_bytes, s, &A);
  if (st != GC_OK) return st;
  A.p = const_cast<float*>(p);
  A.q = const_cast<float*>(q);
  A.out = out;
  k_psplan<<<1, 1024, 0, s>>>(A);
  if (rank == 1)
    k_pres<1, true><<<ps_grid(k_pres<1, true>, A.Mrows), 256, 0, s>>>(A);
  else if (rank == 2)
    k_pres<2, true><<<ps_grid(k_pres<2, true>, A.Mrows), 256, 0, s>>>(A);
  else
    k_pres<4, true><<<ps_grid(k_pres<4, true>, A.Mrows), 256, 0, s>>>(A);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}
