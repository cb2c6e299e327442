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
//   k_pmq   PS_RC x PS_CC tiles, Q^T in shared memory: M = G + E (stored
//           into E), row partials of P_raw = M Q per column tile
//   k_ppred fixed-order sum of the row partials -> P_raw
//   k_porth Gram-Schmidt on P (fixed-order sums): one CTA per matrix, or a
//           cluster of PORTH_CL CTAs for matrices of more than PORTH_BIG rows
//   k_pmtp  256 x 1024 tiles of M: partial column sums of M^T P
//   k_pqred fixed-order sum of the partials -> Q
//   k_pres  the same tiles, Q^T staged in shared memory: E = M - P Q^T
//           (the pending-residual entry point skips it: the next call's
//           k_pmq makes the residual from E = M, P and Q on the fly)
// Reductions: fused multiply-add partial sums in fp32 over a few terms,
// added into a compensated fp32 accumulator per thread, then combined across
// lanes, warps and tiles by compensated fp32 additions in a fixed order
// (deterministic; no fp64 arithmetic, which is slow on this part);
// elementwise steps are single fp32 roundings in the order the method
// states them.
#include <cooperative_groups.h>
#include <cstring>

#include "gc_common.cuh"
#include "gc_host.h"

namespace gc {

// Tiles of the three streaming passes: PS_RC rows x PS_CC columns (256
// threads x 4 columns); 128-row tiles measured the same as 256.
constexpr int PS_RC = 256;
constexpr int PS_CC = 1024;
// Terms summed in plain fp32 (fused multiply-adds) before each compensated
// addition in P = M Q and M^T P: the partial's rounding error is at most
// (PS_FLUSH - 1) u of the sum of |terms| (u = 2^-24), below 1e-6 of it.
constexpr int PS_FLUSH = 16;
// Gram-Schmidt of matrices with more than PORTH_BIG rows runs on a cluster of
// PORTH_CL CTAs (rows split over the cluster, sums combined through
// distributed shared memory).
constexpr int64_t PORTH_BIG = 8192;
constexpr int PORTH_CL = 8;

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
  const float* p_prev;  // pending residual: the previous call's P (E holds its M), else null
  float* out;
  uint32_t* diag;
  int64_t* rowoff;   // [T+1] prefix of m
  int64_t* coloff;   // [T+1] prefix of n
  int64_t* tileoff;  // [T+1] prefix of Q tiles
  int64_t* partoff;  // [T+1] prefix of ceil(m / PS_RC) * n
  int64_t* ppoff;    // [T+1] prefix of m * ceil(n / PS_CC)
  float* part;       // partial column sums of M^T P, [partoff][R]
  float* ppart;      // partial row sums of M Q per column tile, [ppoff][R]
  int64_t* bigoff;    // [T+1] prefix count of matrices with more than PORTH_BIG rows
  int64_t Mrows, Ncols, Tiles, Parts, PParts, Big;
};

__device__ __forceinline__ bool ps_aborted(const PsArgs& A) { return A.diag[DIAG_ABORT] != 0u; }

__global__ void __launch_bounds__(1024) k_psplan(PsArgs A) {
  chain_wait();
  __shared__ int64_t s_warp[32];
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  int64_t carry[6] = {0, 0, 0, 0, 0, 0};
  int64_t* outs[6] = {A.rowoff, A.coloff, A.tileoff, A.partoff, A.ppoff, A.bigoff};
  for (int base = 0; base < A.T; base += blockDim.x) {
    const int t = base + threadIdx.x;
    int64_t v[6] = {0, 0, 0, 0, 0, 0};
    if (t < A.T) {
      const int64_t m = A.rows[t], n = A.cols[t];
      if (m < 1 || n < 1 || A.start[t] < 0) s_bad = 1;
      const int64_t rc = (m + PS_RC - 1) / PS_RC;
      v[0] = m;
      v[1] = n;
      v[2] = rc * ((n + PS_CC - 1) / PS_CC);
      v[3] = rc * n;
      v[4] = m * ((n + PS_CC - 1) / PS_CC);
      v[5] = m > PORTH_BIG ? 1 : 0;
    }
    for (int w = 0; w < 6; ++w) {
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
    for (int w = 0; w < 6; ++w) outs[w][A.T] = carry[w];
    if (s_bad || carry[0] != A.Mrows || carry[1] != A.Ncols || carry[2] != A.Tiles || carry[3] != A.Parts ||
        carry[4] != A.PParts || carry[5] != A.Big) {
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

// Sums R compensated accumulators across the warp, in a fixed order, with
// a reduce-scatter: at the first levels a lane keeps half of its values and
// trades the other half with its partner, so R = 4 costs 6 compensated
// additions instead of 20.  Afterwards every lane holds the total for
// k = warp_rs_k<R>(lane).
template <int R>
__device__ __forceinline__ int warp_rs_k(unsigned lane) {
  return R == 4 ? (int)(((lane >> 4) & 1u) * 2u + ((lane >> 3) & 1u)) : (R == 2 ? (int)((lane >> 4) & 1u) : 0);
}

__device__ __forceinline__ void nm_trade(Nm& keep, const Nm& send, int d) {
  const float os = __shfl_xor_sync(FULL, send.s, d);
  const float oc = __shfl_xor_sync(FULL, send.c, d);
  keep.add(os);
  keep.c = __fadd_rn(keep.c, oc);
}

template <int R>
__device__ __forceinline__ Nm warp_reduce_scatter(Nm acc[R], unsigned lane) {
  Nm v;
  if (R == 4) {
    const bool h16 = (lane & 16u) != 0u, h8 = (lane & 8u) != 0u;
    Nm k0 = h16 ? acc[2] : acc[0], k1 = h16 ? acc[3] : acc[1];
    const Nm s0 = h16 ? acc[0] : acc[2], s1 = h16 ? acc[1] : acc[3];
    nm_trade(k0, s0, 16);
    nm_trade(k1, s1, 16);
    v = h8 ? k1 : k0;
    const Nm s = h8 ? k0 : k1;
    nm_trade(v, s, 8);
#pragma unroll
    for (int d = 4; d > 0; d >>= 1) v.butterfly(d);
  } else if (R == 2) {
    const bool h16 = (lane & 16u) != 0u;
    v = h16 ? acc[1] : acc[0];
    const Nm s = h16 ? acc[0] : acc[1];
    nm_trade(v, s, 16);
#pragma unroll
    for (int d = 8; d > 0; d >>= 1) v.butterfly(d);
  } else {
    v = acc[0];
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v.butterfly(d);
  }
  return v;
}

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

// s_ij = sum_k P_ik Q_jk accumulated in k order in fp32, as the method
// states, then E = M - s (residual) or out += s (receiver).
template <int R, bool DECODE>
__device__ __forceinline__ float pres_one(float x, const float pv[R], const float qv[R]) {
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < R; ++k) s = __fadd_rn(s, __fmul_rn(pv[k], qv[k]));
  return DECODE ? __fadd_rn(x, s) : __fsub_rn(x, s);
}

// M = G + E (stored into E) and partial sums of P_raw = M Q over the tiles
// of M^T P (PS_RC rows x PS_CC columns).  The tile's Q columns are staged
// transposed in shared memory; a warp takes a row and a lane 4 consecutive
// columns of each 128-column group (16-byte g, e and Q^T accesses, four
// groups of g and e in flight).  Fused multiply-adds are summed in fp32
// over PS_FLUSH columns into compensated accumulators, reduced across lanes
// by a fixed-order reduce-scatter, and one lane per k stores the row's
// partial for this column tile.  Matrices with misaligned rows go one column per lane.
// PEND: E holds the previous call's M, whose residual M - P_prev Q_prev^T is
// made here first, element by element with the arithmetic of k_pres (Q_prev
// is this call's warm start, the Q staged in shared memory), so the result
// is bit-identical to the eager residual.
template <int R, bool PEND>
__global__ void __launch_bounds__(256, PEND ? 3 : 1) k_pmq(PsArgs A) {
  chain_wait();
  constexpr int PG = 4;  // 128-column groups per step: PG * 4 = PS_FLUSH columns per lane
  static_assert(PG * 4 == PS_FLUSH, "one compensated addition per step");
  __shared__ __align__(16) float sq[R][PS_CC];
  if (ps_aborted(A)) return;
  for (int64_t tile = blockIdx.x; tile < A.Tiles; tile += gridDim.x) {
    const int t = find_segment(A.tileoff, A.T, tile);
    const int64_t m = A.rows[t], n = A.cols[t];
    const int64_t nd = (n + PS_CC - 1) / PS_CC;
    const int64_t local = tile - A.tileoff[t];
    const int64_t c = local / nd, d = local % nd;
    const int64_t jb = d * PS_CC;
    const int cw = (int)min((int64_t)PS_CC, n - jb);
    const int64_t i0 = c * PS_RC, i1 = min(m, i0 + PS_RC);
    const float* qt = A.q + (A.coloff[t] + jb) * R;
    for (int j = threadIdx.x; j < cw; j += blockDim.x) {
      float v[R];
      load_row<R>(qt + (int64_t)j * R, v);
#pragma unroll
      for (int k = 0; k < R; ++k) sq[k][j] = v[k];
    }
    __syncthreads();
    const unsigned lane = lane_id();
    const int warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
    const bool vec = ((A.start[t] & 3) == 0) && ((n & 3) == 0);
    for (int64_t i = i0 + warp; i < i1; i += nwarp) {
      const int64_t rb = A.start[t] + i * n + jb;
      Nm acc[R];
      float part[R];
#pragma unroll
      for (int k = 0; k < R; ++k) part[k] = 0.0f;
      float pv[R];
      if (PEND) load_row<R>(A.p_prev + (A.rowoff[t] + i) * R, pv);
      if (vec) {
        const float4* g4 = reinterpret_cast<const float4*>(A.g + rb);
        float4* e4 = reinterpret_cast<float4*>(A.e + rb);
        const int nv = cw >> 2;
        for (int v0 = (int)lane; v0 < nv; v0 += 32 * PG) {
          // every load of the step is issued before the first store (the
          // stores to E could alias later loads as far as the compiler knows)
          float4 mv[PG], ev[PG];
#pragma unroll
          for (int u = 0; u < PG; ++u) {
            const int vi = v0 + 32 * u;
            mv[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            ev[u] = mv[u];
            if (vi < nv) {
              mv[u] = ld_stream(g4 + vi);
              ev[u] = ld_stream(e4 + vi);
            }
          }
          if (PEND) {
#pragma unroll
            for (int u = 0; u < PG; ++u) {
              const int vi = v0 + 32 * u;
              if (vi < nv) {
                float qv[4][R];
#pragma unroll
                for (int k = 0; k < R; ++k) {
                  const float4 qk = *reinterpret_cast<const float4*>(&sq[k][4 * vi]);
                  qv[0][k] = qk.x; qv[1][k] = qk.y; qv[2][k] = qk.z; qv[3][k] = qk.w;
                }
                ev[u].x = pres_one<R, false>(ev[u].x, pv, qv[0]);
                ev[u].y = pres_one<R, false>(ev[u].y, pv, qv[1]);
                ev[u].z = pres_one<R, false>(ev[u].z, pv, qv[2]);
                ev[u].w = pres_one<R, false>(ev[u].w, pv, qv[3]);
              }
            }
          }
#pragma unroll
          for (int u = 0; u < PG; ++u) {
            const int vi = v0 + 32 * u;
            mv[u].x = __fadd_rn(mv[u].x, ev[u].x);
            mv[u].y = __fadd_rn(mv[u].y, ev[u].y);
            mv[u].z = __fadd_rn(mv[u].z, ev[u].z);
            mv[u].w = __fadd_rn(mv[u].w, ev[u].w);
            if (vi < nv) st_stream(e4 + vi, mv[u]);
          }
#pragma unroll
          for (int u = 0; u < PG; ++u) {
            const int vi = v0 + 32 * u;
            if (vi < nv) {
#pragma unroll
              for (int k = 0; k < R; ++k) {
                const float4 qk = *reinterpret_cast<const float4*>(&sq[k][4 * vi]);
                part[k] = __fmaf_rn(mv[u].x, qk.x, part[k]);
                part[k] = __fmaf_rn(mv[u].y, qk.y, part[k]);
                part[k] = __fmaf_rn(mv[u].z, qk.z, part[k]);
                part[k] = __fmaf_rn(mv[u].w, qk.w, part[k]);
              }
            }
          }
#pragma unroll
          for (int k = 0; k < R; ++k) {
            acc[k].add(part[k]);
            part[k] = 0.0f;
          }
        }
      } else {
        int fl = 0;
        for (int j = (int)lane; j < cw; j += 32) {
          float evj = __ldcs(A.e + rb + j);
          if (PEND) {
            float qv[R];
#pragma unroll
            for (int k = 0; k < R; ++k) qv[k] = sq[k][j];
            evj = pres_one<R, false>(evj, pv, qv);
          }
          const float mvj = __fadd_rn(__ldcs(A.g + rb + j), evj);
          __stcs(A.e + rb + j, mvj);
#pragma unroll
          for (int k = 0; k < R; ++k) part[k] = __fmaf_rn(mvj, sq[k][j], part[k]);
          if (++fl == PS_FLUSH) {
            fl = 0;
#pragma unroll
            for (int k = 0; k < R; ++k) {
              acc[k].add(part[k]);
              part[k] = 0.0f;
            }
          }
        }
#pragma unroll
        for (int k = 0; k < R; ++k) acc[k].add(part[k]);
      }
      const Nm tot = warp_reduce_scatter<R>(acc, lane);
      if ((lane & (R == 4 ? 7u : (R == 2 ? 15u : 31u))) == 0u)
        A.ppart[(A.ppoff[t] + i * nd + d) * R + warp_rs_k<R>(lane)] = tot.value();
    }
    __syncthreads();  // the next tile restages the shared Q^T
  }
}

// P_raw = sum over column tiles of the row partials, in tile order
// (compensated fp32); thread per row.
template <int R>
__global__ void __launch_bounds__(256) k_ppred(PsArgs A) {
  chain_wait();
  if (ps_aborted(A)) return;
  for (int64_t gr = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gr < A.Mrows;
       gr += (int64_t)gridDim.x * blockDim.x) {
    const int t = find_segment(A.rowoff, A.T, gr);
    const int64_t i = gr - A.rowoff[t];
    const int64_t nd = (A.cols[t] + PS_CC - 1) / PS_CC;
    const float* src = A.ppart + (A.ppoff[t] + i * nd) * R;
    Nm s[R];
    for (int64_t d = 0; d < nd; ++d) {
      float v[R];
      load_row<R>(src + d * R, v);
#pragma unroll
      for (int k = 0; k < R; ++k) s[k].add(v[k]);
    }
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const float pv = s[k].value();
      A.p[gr * R + k] = pv;
      if (A.p_raw) A.p_raw[gr * R + k] = pv;
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

// Gram-Schmidt of matrix t by one CTA (CL = 1) or by cluster rank `rank` of
// CL CTAs: thread g of the CL * blockDim.x threads owns rows g, g + CL *
// blockDim.x, ...  Each pass's block sum is a compensated pair; with CL > 1
// every CTA publishes its pair in shared memory (slot alternating by pass),
// the cluster barrier orders it, and every CTA adds the CL pairs in rank
// order, so all CTAs hold the same value.
template <int R, int CL>
__device__ __forceinline__ void porth_matrix(const PsArgs& A, int t, int rank) {
  __shared__ float s_ws[32], s_wc[32];
  __shared__ float s_tot;
  __shared__ float s_slot[2][2];
  const int64_t m = A.rows[t];
  float* P = A.p + A.rowoff[t] * R;
  const unsigned lane = lane_id(), warp = threadIdx.x >> 5;
  const int64_t nthr = (int64_t)CL * blockDim.x;
  const int64_t g0 = (int64_t)rank * blockDim.x + threadIdx.x;
  int ukind = 0, uk = 0, uj = 0;  // pending update: 0 none, 1 P_k -= d P_j, 2 P_k /= nrm
  float uval = 0.0f;
  int pass = 0;
  for (int k = 0; k < R; ++k) {
    for (int j = 0; j <= k; ++j, ++pass) {  // j < k: d = <P_j, P_k>;  j == k: |P_k|^2
      Nm acc;
      for (int64_t i0 = g0; i0 < m; i0 += 4 * nthr) {
        float v[4][R];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t i = i0 + nthr * u;
          if (i < m) porth_row<R>(P + i * R, v[u], ukind, uk, uj, uval);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t i = i0 + nthr * u;
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
        w.s = lane < (blockDim.x >> 5) ? s_ws[lane] : 0.0f;
        w.c = lane < (blockDim.x >> 5) ? s_wc[lane] : 0.0f;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) w.butterfly(d);
        if (lane == 0) {
          if (CL == 1) {
            s_tot = w.value();
          } else {
            s_slot[pass & 1][0] = w.s;
            s_slot[pass & 1][1] = w.c;
          }
        }
      }
      if (CL > 1) {
        cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
        cluster.sync();
        if (threadIdx.x == 0) {
          Nm z;
#pragma unroll
          for (int r = 0; r < CL; ++r) {
            const float* peer = cluster.map_shared_rank(&s_slot[pass & 1][0], r);
            z.add(peer[0]);
            z.c = __fadd_rn(z.c, peer[1]);
          }
          s_tot = z.value();
        }
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
  // no CTA may exit while a peer could still be reading its slots
  if (CL > 1) cooperative_groups::this_cluster().sync();
  if (ukind != 0)
    for (int64_t i = g0; i < m; i += nthr) {
      float v[R];
      porth_row<R>(P + i * R, v, ukind, uk, uj, uval);
    }
}

// One CTA per matrix: those of at most PORTH_BIG rows (big = 0), or the
// larger ones (big = 1, used only if the cluster launch is refused).
template <int R>
__global__ void __launch_bounds__(1024) k_porth(PsArgs A, int big) {
  chain_wait();
  if (ps_aborted(A)) return;
  const int t = blockIdx.x;
  if ((A.rows[t] > PORTH_BIG) != (big != 0)) return;
  porth_matrix<R, 1>(A, t, 0);
}

// One cluster of PORTH_CL CTAs per matrix of more than PORTH_BIG rows.  Every
// CTA of a cluster runs the same passes (the abort flag, set before this
// launch, reads the same in all of them), so all reach every barrier.
template <int R>
__global__ void __launch_bounds__(1024) k_porthc(PsArgs A) {
  chain_wait();
  if (ps_aborted(A)) return;
  const int64_t ci = blockIdx.x / PORTH_CL;
  const int t = find_segment(A.bigoff, A.T, ci);
  porth_matrix<R, PORTH_CL>(A, t, (int)(blockIdx.x % PORTH_CL));
}

// Partial column sums of M^T P over a tile of PS_RC rows x PS_CC columns;
// a thread owns 4 consecutive columns.  Aligned matrices stream M through a
// cp.async pipeline: each thread copies its own 16-byte slice of the next
// rows into shared memory PT_NS - 1 stages ahead (no registers held for
// data in flight, no thread reads another's slice), then computes from
// shared memory, with the tile's rows of P staged there once.  Fused
// multiply-adds are summed in fp32 over PS_FLUSH rows, then added to
// compensated accumulators; the tile's partials go to A.part.
constexpr int PT_RS = 2;  // rows per stage
constexpr int PT_NS = 5;  // stages (40 KB of shared memory per CTA, 8 rows in flight)

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

template <int R>
__device__ __forceinline__ void pmtp_rows(float part[4][R], const float mm[4], const float pv[R]) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
#pragma unroll
    for (int k = 0; k < R; ++k) part[cc][k] = __fmaf_rn(mm[cc], pv[k], part[cc][k]);
}

template <int R>
__device__ __forceinline__ void pmtp_flush(Nm acc[4][R], float part[4][R]) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
#pragma unroll
    for (int k = 0; k < R; ++k) {
      acc[cc][k].add(part[cc][k]);
      part[cc][k] = 0.0f;
    }
}

template <int R>
__global__ void __launch_bounds__(256, 3) k_pmtp(PsArgs A) {
  chain_wait();
  __shared__ __align__(16) float4 sbuf[PT_NS * PT_RS * 256];
  __shared__ __align__(16) float sp[PS_RC * R];  // the tile's rows of P
  if (ps_aborted(A)) return;
  const int tid = threadIdx.x;
  for (int64_t tile = blockIdx.x; tile < A.Tiles; tile += gridDim.x) {
    const int t = find_segment(A.tileoff, A.T, tile);
    const int64_t m = A.rows[t], n = A.cols[t];
    const int64_t nd = (n + PS_CC - 1) / PS_CC;
    const int64_t local = tile - A.tileoff[t];
    const int64_t c = local / nd, d = local % nd;
    const int64_t j0 = d * PS_CC + 4 * tid;
    const int64_t i0 = c * PS_RC, i1 = min(m, i0 + PS_RC);
    const float* P = A.p + A.rowoff[t] * R;
    const bool vec = ((A.start[t] & 3) == 0) && ((n & 3) == 0);
    __syncthreads();  // the previous tile's readers of sp are done
    for (int x = tid; x < (int)(i1 - i0) * R; x += blockDim.x) sp[x] = P[i0 * R + x];
    __syncthreads();
    if (j0 >= n) continue;
    Nm acc[4][R];
    float part[4][R];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
#pragma unroll
      for (int k = 0; k < R; ++k) part[cc][k] = 0.0f;
    if (vec) {
      const float* ecol = A.e + A.start[t] + j0;  // row i at ecol + i * n, 16-byte aligned
      const int nsteps = (int)((i1 - i0 + PT_RS - 1) / PT_RS);
      auto issue = [&](int st) {
        if (st < nsteps) {
#pragma unroll
          for (int u = 0; u < PT_RS; ++u) {
            const int64_t i = i0 + (int64_t)st * PT_RS + u;
            if (i < i1) cp_async16(&sbuf[((st % PT_NS) * PT_RS + u) * 256 + tid], ecol + i * n);
          }
        }
        cp_async_commit();
      };
#pragma unroll
      for (int st = 0; st < PT_NS - 1; ++st) issue(st);
      int fl = 0;
      for (int st = 0; st < nsteps; ++st) {
        issue(st + PT_NS - 1);
        cp_async_wait<PT_NS - 1>();  // this thread's copies of stage st have landed
#pragma unroll
        for (int u = 0; u < PT_RS; ++u) {
          const int64_t i = i0 + (int64_t)st * PT_RS + u;
          if (i < i1) {
            const float4 mv = sbuf[((st % PT_NS) * PT_RS + u) * 256 + tid];
            const float mm[4] = {mv.x, mv.y, mv.z, mv.w};
            float pv[R];
#pragma unroll
            for (int k = 0; k < R; ++k) pv[k] = sp[(i - i0) * R + k];
            pmtp_rows<R>(part, mm, pv);
          }
        }
        if (++fl * PT_RS >= PS_FLUSH) {
          fl = 0;
          pmtp_flush<R>(acc, part);
        }
      }
      cp_async_wait<0>();
    } else {
      int fl = 0;
      for (int64_t i = i0; i < i1; ++i) {
        const int64_t rb = A.start[t] + i * n;
        float mm[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) mm[cc] = (j0 + cc < n) ? A.e[rb + j0 + cc] : 0.0f;
        float pv[R];
#pragma unroll
        for (int k = 0; k < R; ++k) pv[k] = sp[(i - i0) * R + k];
        pmtp_rows<R>(part, mm, pv);
        if (++fl == PS_FLUSH) {
          fl = 0;
          pmtp_flush<R>(acc, part);
        }
      }
    }
    pmtp_flush<R>(acc, part);
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
  chain_wait();
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

// E = M - P Q^T (or out += P Q^T) over the same PS_RC x PS_CC tiles as
// M^T P.  The tile's Q columns are staged transposed in shared memory
// (Q^T[k][c]), so a lane reads the R values of its 4 consecutive columns
// with one conflict-free 16-byte load per k; a warp takes a row, and M (or
// out) moves in 16-byte vectors, four per lane in flight.  Matrices with
// misaligned rows go one column per lane.
template <int R, bool DECODE>
__global__ void __launch_bounds__(256) k_pres(PsArgs A) {
  chain_wait();
  constexpr int PG = 4;  // 128-column groups per step
  __shared__ __align__(16) float sq[R][PS_CC];
  if (ps_aborted(A)) return;
  const int64_t tile = blockIdx.x;
  const int t = find_segment(A.tileoff, A.T, tile);
  const int64_t m = A.rows[t], n = A.cols[t];
  const int64_t nd = (n + PS_CC - 1) / PS_CC;
  const int64_t local = tile - A.tileoff[t];
  const int64_t c = local / nd, d = local % nd;
  const int64_t jb = d * PS_CC;
  const int cw = (int)min((int64_t)PS_CC, n - jb);
  const int64_t i0 = c * PS_RC, i1 = min(m, i0 + PS_RC);
  const float* qt = A.q + (A.coloff[t] + jb) * R;
  for (int j = threadIdx.x; j < cw; j += blockDim.x) {
    float v[R];
    load_row<R>(qt + (int64_t)j * R, v);
#pragma unroll
    for (int k = 0; k < R; ++k) sq[k][j] = v[k];
  }
  __syncthreads();
  float* dstbase = DECODE ? A.out : A.e;
  const unsigned lane = lane_id();
  const int warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  const bool vec = ((A.start[t] & 3) == 0) && ((n & 3) == 0);
  for (int64_t i = i0 + warp; i < i1; i += nwarp) {
    const int64_t rb = A.start[t] + i * n + jb;
    float pv[R];
    load_row<R>(A.p + (A.rowoff[t] + i) * R, pv);
    if (vec) {
      float4* d4 = reinterpret_cast<float4*>(dstbase + rb);
      const int nv = cw >> 2;
      for (int v0 = (int)lane; v0 < nv; v0 += 32 * PG) {
        float4 x[PG];
#pragma unroll
        for (int u = 0; u < PG; ++u)
          if (v0 + 32 * u < nv) x[u] = ld_stream(d4 + v0 + 32 * u);
#pragma unroll
        for (int u = 0; u < PG; ++u) {
          const int vi = v0 + 32 * u;
          if (vi < nv) {
            float qv[4][R];
#pragma unroll
            for (int k = 0; k < R; ++k) {
              const float4 qk = *reinterpret_cast<const float4*>(&sq[k][4 * vi]);
              qv[0][k] = qk.x; qv[1][k] = qk.y; qv[2][k] = qk.z; qv[3][k] = qk.w;
            }
            float4 y;
            y.x = pres_one<R, DECODE>(x[u].x, pv, qv[0]);
            y.y = pres_one<R, DECODE>(x[u].y, pv, qv[1]);
            y.z = pres_one<R, DECODE>(x[u].z, pv, qv[2]);
            y.w = pres_one<R, DECODE>(x[u].w, pv, qv[3]);
            st_stream(d4 + vi, y);
          }
        }
      }
    } else {
      for (int j = (int)lane; j < cw; j += 32) {
        float qv[R];
#pragma unroll
        for (int k = 0; k < R; ++k) qv[k] = sq[k][j];
        __stcs(dstbase + rb + j, pres_one<R, DECODE>(__ldcs(dstbase + rb + j), pv, qv));
      }
    }
  }
}

// ============================================================================ host

struct PsTotals {
  int64_t M = 0, N = 0, Tiles = 0, Parts = 0, PParts = 0, Big = 0, maxel = 0;
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
    z->PParts += m * ((n + PS_CC - 1) / PS_CC);
    z->Big += m > PORTH_BIG ? 1 : 0;
  }
  return GC_OK;
}

struct PsCarve {
  size_t o_row, o_col, o_tile, o_part_off, o_pp_off, o_big, o_part, o_ppart, total;
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
  c.o_pp_off = take(8 * (size_t)(T + 1));
  c.o_big = take(8 * (size_t)(T + 1));
  c.o_part = take(4 * (size_t)z.Parts * R);
  c.o_ppart = take(4 * (size_t)z.PParts * R);
  c.total = p;
  return c;
}

// Resident CTAs of a tile kernel: k_pmq and k_pmtp stride over the tiles
// with a persistent grid (measured no slower than one tile per CTA, and
// k_pmq 6% faster); k_pres keeps one tile per CTA (the loop costs it
// registers and 15%).
template <class K>
static unsigned ps_tile_grid(K kernel, size_t smem, int64_t tiles) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, smem);
  if (per_sm < 1) per_sm = 1;
  const int64_t grid = std::min<int64_t>((int64_t)sms * per_sm, tiles);
  return (unsigned)std::max<int64_t>(grid, 1);
}

template <int R>
static void ps_launch_compress(const PsArgs& A, cudaStream_t s, bool lazy) {
  launch_chained(k_psplan, 1, 1024, 0, s, A);
  if (A.p_prev)
    launch_chained(k_pmq<R, true>, ps_tile_grid(k_pmq<R, true>, 0, A.Tiles), 256, 0, s, A);
  else
    launch_chained(k_pmq<R, false>, ps_tile_grid(k_pmq<R, false>, 0, A.Tiles), 256, 0, s, A);
  launch_chained(k_ppred<R>, (unsigned)std::min<int64_t>((A.Mrows + 255) / 256, 65535), 256, 0, s, A);
  launch_chained(k_porth<R>, A.T, 1024, 0, s, A, 0);
  if (A.Big > 0) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)(A.Big * PORTH_CL));
    cfg.blockDim = dim3(1024);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = PORTH_CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k_porthc<R>, A) != cudaSuccess) {
      (void)cudaGetLastError();  // cluster refused: one CTA per large matrix instead
      k_porth<R><<<A.T, 1024, 0, s>>>(A, 1);
    }
  }
  launch_chained(k_pmtp<R>, ps_tile_grid(k_pmtp<R>, 0, A.Tiles), 256, 0, s, A);
  launch_chained(k_pqred<R>, (unsigned)std::min<int64_t>((A.Ncols + 255) / 256, 65535), 256, 0, s, A);
  if (!lazy) launch_chained(k_pres<R, false>, (unsigned)A.Tiles, 256, 0, s, A);
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
  A->ppoff = reinterpret_cast<int64_t*>(w + c.o_pp_off);
  A->bigoff = reinterpret_cast<int64_t*>(w + c.o_big);
  A->ppart = reinterpret_cast<float*>(w + c.o_ppart);
  A->part = reinterpret_cast<float*>(w + c.o_part);
  A->Mrows = z.M;
  A->Ncols = z.N;
  A->Tiles = z.Tiles;
  A->Parts = z.Parts;
  A->PParts = z.PParts;
  A->Big = z.Big;
  if (!zero_chained(ws, DIAG_BYTES, s)) return GC_ERR_CUDA;
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
  NvtxRange nvtx_range("gc_powersgd_compress");
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
    ps_launch_compress<1>(A, s, false);
  else if (rank == 2)
    ps_launch_compress<2>(A, s, false);
  else
    ps_launch_compress<4>(A, s, false);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

extern "C" gc_status gc_powersgd_compress_lazy(const gc_matrix_layout* dev, const gc_matrix_layout* host,
                                               int32_t rank, const float* g, float* e, float* q, float* p,
                                               const float* p_prev, float* p_raw, void* workspace,
                                               size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("gc_powersgd_compress_lazy");
  if (!g || !e || !q || !p) return GC_ERR_INVALID_ARG;
  if (p_prev == p) return GC_ERR_INVALID_ARG;
  if (!aligned16(g) || !aligned16(e) || !aligned16(q) || !aligned16(p) || (p_prev && !aligned16(p_prev)))
    return GC_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PsArgs A;
  const gc_status st = ps_setup(dev, host, rank, workspace, ws_bytes, s, &A);
  if (st != GC_OK) return st;
  A.g = g;
  A.e = e;
  A.q = q;
  A.p = p;
  A.p_raw = p_raw;
  A.p_prev = p_prev;
  if (rank == 1)
    ps_launch_compress<1>(A, s, true);
  else if (rank == 2)
    ps_launch_compress<2>(A, s, true);
  else
    ps_launch_compress<4>(A, s, true);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

extern "C" gc_status gc_powersgd_residual_materialize(const gc_matrix_layout* dev,
                                                      const gc_matrix_layout* host, int32_t rank,
                                                      float* e, const float* p, const float* q,
                                                      void* workspace, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("gc_powersgd_residual_materialize");
  if (!e || !p || !q) return GC_ERR_INVALID_ARG;
  if (!aligned16(e) || !aligned16(q) || !aligned16(p)) return GC_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PsArgs A;
  const gc_status st = ps_setup(dev, host, rank, workspace, ws_bytes, s, &A);
  if (st != GC_OK) return st;
  A.e = e;
  A.p = const_cast<float*>(p);
  A.q = const_cast<float*>(q);
  launch_chained(k_psplan, 1, 1024, 0, s, A);
  if (rank == 1)
    launch_chained(k_pres<1, false>, (unsigned)A.Tiles, 256, 0, s, A);
  else if (rank == 2)
    launch_chained(k_pres<2, false>, (unsigned)A.Tiles, 256, 0, s, A);
  else
    launch_chained(k_pres<4, false>, (unsigned)A.Tiles, 256, 0, s, A);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

extern "C" gc_status gc_powersgd_decompress_accumulate(const gc_matrix_layout* dev,
                                                       const gc_matrix_layout* host, int32_t rank,
                                                       const float* p, const float* q, float* out,
                                                       void* workspace, size_t ws_bytes,
                                                       void* stream) {
  NvtxRange nvtx_range("gc_powersgd_decompress_accumulate");
  if (!p || !q || !out) return GC_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(p)) return GC_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PsArgs A;
  const gc_status st = ps_setup(dev, host, rank, workspace, ws_bytes, s, &A);
  if (st != GC_OK) return st;
  A.p = const_cast<float*>(p);
  A.q = const_cast<float*>(q);
  A.out = out;
  launch_chained(k_psplan, 1, 1024, 0, s, A);
  if (rank == 1)
    launch_chained(k_pres<1, true>, (unsigned)A.Tiles, 256, 0, s, A);
  else if (rank == 2)
    launch_chained(k_pres<2, true>, (unsigned)A.Tiles, 256, 0, s, A);
  else
    launch_chained(k_pres<4, true>, (unsigned)A.Tiles, 256, 0, s, A);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}
