// Dense compressors and receivers (sm_103a): 1-bit sign with EF, int8 and
// QSGD stochastic quantization, and their decoders.
//
// Method: mbrenndoerfer.com "Gradient Compression", 1-bit SGD
// (Q(g) = sign(g) ||g||_1 / d, one scalar per layer) and QSGD
// (Q_s(g) = ||g|| sgn(g) xi(g, s), stochastic rounding); inferensys.com
// genomic glossary "Gradient Compression", 8-bit quantization and
// stochastic rounding.
//
// Each compressor is two streaming passes over the arena (the per-tensor
// scale must be known before any code or residual can be written):
//   pass 1: acc = g (+ e, written back), per-unit partial of sum|acc| or
//           sum acc^2 (scaled compensated fp32 per lane, fp64 across
//           lanes), or the per-tensor max key (int8)
//   reduce: per tensor, unit partials summed in a fixed order in fp64
//   pass 2: bits / codes and the EF residual
// The single-pass sign variant (k_sign_lazy) writes bits, acc and the
// partials in one pass and leaves the residual's -+mean to the next call.
#include <cmath>
#include <cstring>

#include "gc_common.cuh"
#include "gc_host.h"

namespace gc {

enum { DOP_SIGN = 0, DOP_INT8 = 1, DOP_QSGD = 2 };

struct DenseArgs {
  int T;
  int op;
  int ef;
  int s_levels;
  const int64_t* off;
  const float* g;
  float* e;
  uint32_t* bits;
  int8_t* codes;
  float* scale;  // mean_abs (sign), max/127 (int8), norm (QSGD)
  uint64_t seed, iter;
  const uint64_t* iter_dev;  // iteration counter in device memory (graph capture), else null
  PhiloxKey pk;       // round keys of seed
  uint32_t* diag;
  uint32_t* maxkey;   // [T]
  int64_t* units_off; // [T+1]
  int64_t* woff;      // [T+1]
  double* upart;      // [U]
  int64_t U, W, N;
  int64_t off0;  // off[0] of the host layout (nonzero for a bucket)
};

__device__ __forceinline__ bool aborted(const DenseArgs& A) { return A.diag[DIAG_ABORT] != 0u; }

__global__ void __launch_bounds__(1024) k_dplan(DenseArgs A) {
  chain_wait();
  __shared__ int64_t s_warp[32];
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  int64_t carry_u = 0, carry_w = 0;
  for (int base = 0; base < A.T; base += blockDim.x) {
    const int t = base + threadIdx.x;
    int64_t nu = 0, nw = 0;
    if (t < A.T) {
      const int64_t n = A.off[t + 1] - A.off[t];
      if (n < 1 || n > INT64_C(2147483647)) s_bad = 1;
      nu = units_of(n);
      nw = (n + 31) >> 5;
    }
    // two block scans (same helper shape as the Top-k planner)
    for (int which = 0; which < 2; ++which) {
      const int64_t v = which == 0 ? nu : nw;
      const unsigned lane = lane_id(), w = threadIdx.x >> 5, nwp = blockDim.x >> 5;
      int64_t x = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int64_t y = __shfl_up_sync(FULL, x, d);
        if (lane >= (unsigned)d) x += y;
      }
      if (lane == 31) s_warp[w] = x;
      __syncthreads();
      if (w == 0) {
        int64_t z = lane < nwp ? s_warp[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int64_t y = __shfl_up_sync(FULL, z, d);
          if (lane >= (unsigned)d) z += y;
        }
        if (lane < nwp) s_warp[lane] = z;
      }
      __syncthreads();
      const int64_t excl = (w == 0 ? 0 : s_warp[w - 1]) + x - v;
      const int64_t tot = s_warp[nwp - 1];
      __syncthreads();
      if (which == 0) {
        if (t < A.T) A.units_off[t] = carry_u + excl;
        carry_u += tot;
      } else {
        if (t < A.T) A.woff[t] = carry_w + excl;
        carry_w += tot;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    A.units_off[A.T] = carry_u;
    A.woff[A.T] = carry_w;
    if (s_bad || carry_u != A.U || carry_w != A.W || A.off[0] != A.off0 || A.off[A.T] - A.off0 != A.N) {
      A.diag[DIAG_ERR] |= GC_DIAG_LAYOUT_MISMATCH;
      A.diag[DIAG_ABORT] = 1u;
    }
  }
}


__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(FULL, v, d);
  return v;
}

constexpr int DTHREADS = 256;
constexpr int DWARPS = DTHREADS / 32;

struct UnitRef {
  int t;
  int64_t base, lstart;
  int len;
};

__device__ __forceinline__ UnitRef unit_ref(const DenseArgs& A, int64_t u) {
  UnitRef r;
  r.t = find_segment(A.units_off, A.T, u);
  r.base = A.off[r.t];
  const int64_t n = A.off[r.t + 1] - r.base;
  r.lstart = (u - A.units_off[r.t]) << UNIT_SHIFT;
  r.len = (int)min((int64_t)UNIT, n - r.lstart);
  return r;
}

// Pass 1: acc (+ EF write-back) and the per-unit reduction input.
template <int OP, bool EF>
__global__ void __launch_bounds__(DTHREADS) k_dense1(DenseArgs A) {
  chain_wait();
  if (aborted(A)) return;
  const unsigned lane = lane_id();
  const int warp = threadIdx.x >> 5;
  const int64_t nwarps = (int64_t)gridDim.x * DWARPS;
  for (int64_t u = (int64_t)blockIdx.x * DWARPS + warp; u < A.U; u += nwarps) {
    const UnitRef r = unit_ref(A, u);
    const int64_t g0 = r.base + r.lstart;
    ScaledSum<OP == DOP_QSGD ? 2 : 1> acc_sum;  // sign: sum |acc|; QSGD: sum acc^2
    uint32_t mx = 0u;
    auto take1 = [&](float x) {
      if (OP == DOP_INT8) mx = max(mx, mag_key(x));
      else acc_sum.add1(x);
    };
    if ((g0 & 3) == 0) {
      const int nv = r.len >> 2;
      const float4* g4 = reinterpret_cast<const float4*>(A.g + g0);
      float4* e4 = reinterpret_cast<float4*>(A.e + g0);
      for (int v0 = 0; v0 < nv; v0 += 128) {
        float4 x[4], y[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int vi = v0 + 32 * j + (int)lane;
          x[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          if (vi < nv) {
            x[j] = ld_stream(g4 + vi);
            if (EF) y[j] = ld_stream(e4 + vi);
          }
        }
        uint32_t km = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int vi = v0 + 32 * j + (int)lane;
          if (vi < nv && EF) {
            x[j].x = __fadd_rn(x[j].x, y[j].x);
            x[j].y = __fadd_rn(x[j].y, y[j].y);
            x[j].z = __fadd_rn(x[j].z, y[j].z);
            x[j].w = __fadd_rn(x[j].w, y[j].w);
            st_stream(e4 + vi, x[j]);
          }
          km = max(km, max(max(mag_key(x[j].x), mag_key(x[j].y)), max(mag_key(x[j].z), mag_key(x[j].w))));
        }
        if (OP == DOP_INT8) {
          mx = max(mx, km);
        } else {
          // slots past the end hold zeros, which add nothing
          acc_sum.bound(km);
          const float m = acc_sum.mult();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc_sum.add(x[j].x, m);
            acc_sum.add(x[j].y, m);
            acc_sum.add(x[j].z, m);
            acc_sum.add(x[j].w, m);
          }
        }
      }
      const int rem = r.len & 3;
      if ((int)lane < rem) {
        const int64_t gi = g0 + 4 * nv + lane;
        float a = A.g[gi];
        if (EF) {
          a = __fadd_rn(a, A.e[gi]);
          A.e[gi] = a;
        }
        take1(a);
      }
    } else {
      for (int i = (int)lane; i < r.len; i += 32) {
        const int64_t gi = g0 + i;
        float a = A.g[gi];
        if (EF) {
          a = __fadd_rn(a, A.e[gi]);
          A.e[gi] = a;
        }
        take1(a);
      }
    }
    if (OP == DOP_INT8) {
      mx = warp_max_u32(mx);
      if (lane == 0) atomicMax(A.maxkey + r.t, mx);
    } else {
      const double part = warp_sum_f64(acc_sum.value());
      if (lane == 0) A.upart[u] = part;
    }
  }
}

// Per-tensor scale from the unit partials (fixed order, so deterministic).
__global__ void __launch_bounds__(256) k_dreduce(DenseArgs A) {
  chain_wait();
  __shared__ double s_part[256];
  if (aborted(A)) return;
  const int t = blockIdx.x;
  const int64_t n = A.off[t + 1] - A.off[t];
  if (A.op == DOP_INT8) {
    if (threadIdx.x == 0) A.scale[t] = __fdiv_rn(key_magnitude(A.maxkey[t]), 127.0f);
    return;
  }
  double s = 0.0;
  for (int64_t u = A.units_off[t] + threadIdx.x; u < A.units_off[t + 1]; u += blockDim.x) s += A.upart[u];
  s_part[threadIdx.x] = s;
  __syncthreads();
  for (int h = 128; h > 0; h >>= 1) {
    if ((int)threadIdx.x < h) s_part[threadIdx.x] += s_part[threadIdx.x + h];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double tot = s_part[0];
    A.scale[t] = (A.op == DOP_SIGN) ? __double2float_rn(tot / (double)n) : __double2float_rn(sqrt(tot));
  }
}

// Code of x for the dense quantizers; with DEC, *dec receives the decoded
// value (needed only for the EF residual).  dv divides by the tensor's scale;
// NZ: the caller has checked that the scale is not zero.
template <int OP, bool DEC, bool NZ = false>
__device__ __forceinline__ int dense_code(float x, const Divisor& dv, int s_levels, uint32_t r, float* dec) {
  const float sc = dv.b;
  if (OP == DOP_INT8) {
    int c = 0;
    if (NZ || sc != 0.0f) {
      // the scale is this call's max|acc| / 127, so |x| / s stays within an
      // ulp or two of 127 and inside stochastic_round's domain; no clamp is
      // needed before it (a non-finite x gives a NaN quotient, whose floor
      // comes out far above 127 and is cut to 127 here, as a clamp would)
      c = stochastic_round(dv.div(fabsf(x)), r);
      c = c > 127 ? 127 : c;
      c = signbit(x) ? -c : c;
    }
    if (DEC) *dec = __fmul_rn((float)c, sc);
    return c;
  }
  int level = 0;
  if (NZ || sc != 0.0f) {
    // the scale is this call's norm, within 1e-6 of ||acc|| >= |x|, so y
    // stays within a hair of s_levels (no clamp before stochastic_round; a
    // non-finite x gives a NaN y, whose floor is cut to s_levels by the min)
    const float y = dv.div(__fmul_rn(fabsf(x), (float)s_levels));
    level = min(s_levels, stochastic_round(y, r));
  }
  const bool neg = signbit(x);
  if (DEC) {
    const float mag = __fdiv_rn(__fmul_rn((float)level, sc), (float)s_levels);
    *dec = neg ? -mag : mag;
  }
  return neg ? -level : level;
}

// Pass 2 of the sign compressor: bits and residual.
template <bool EF>
__global__ void __launch_bounds__(DTHREADS) k_sign2(DenseArgs A) {
  chain_wait();
  if (aborted(A)) return;
  const unsigned lane = lane_id();
  const int warp = threadIdx.x >> 5;
  const int64_t nwarps = (int64_t)gridDim.x * DWARPS;
  const float* src = EF ? A.e : A.g;
  for (int64_t u = (int64_t)blockIdx.x * DWARPS + warp; u < A.U; u += nwarps) {
    const UnitRef r = unit_ref(A, u);
    const int64_t g0 = r.base + r.lstart;
    const float mu = A.scale[r.t];
    uint32_t* wbase = A.bits + A.woff[r.t] + (r.lstart >> 5);
    const int nwords = (r.len + 31) >> 5;
    if ((g0 & 3) == 0) {
      // 32 lanes x 4 elements = 4 words per step; 8 steps fill one word per lane
      const int nslots = (r.len + 3) >> 2;
      const float4* s4 = reinterpret_cast<const float4*>(src + g0);
      float4* e4 = reinterpret_cast<float4*>(A.e + g0);
      for (int v0 = 0; v0 < nslots; v0 += 256) {
        uint32_t myword = 0u;
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          const int vi = v0 + 32 * st + (int)lane;
          unsigned nib = 0u;
          if (vi < nslots) {
            const int li = vi * 4;
            if (li + 4 <= r.len) {
              float4 a = ld_stream(s4 + vi);
              nib = (signbit(a.x) ? 0u : 1u) | (signbit(a.y) ? 0u : 2u) | (signbit(a.z) ? 0u : 4u) |
                    (signbit(a.w) ? 0u : 8u);
              if (EF) {
                a.x = __fsub_rn(a.x, signbit(a.x) ? -mu : mu);
                a.y = __fsub_rn(a.y, signbit(a.y) ? -mu : mu);
                a.z = __fsub_rn(a.z, signbit(a.z) ? -mu : mu);
                a.w = __fsub_rn(a.w, signbit(a.w) ? -mu : mu);
                st_stream(e4 + vi, a);
              }
            } else {
              for (int j = 0; li + j < r.len; ++j) {
                const int64_t gi = g0 + li + j;
                const float a = src[gi];
                if (!signbit(a)) nib |= 1u << j;
                if (EF) A.e[gi] = __fsub_rn(a, signbit(a) ? -mu : mu);
              }
            }
          }
          uint32_t w = nib << (4 * (lane & 7));
          w |= __shfl_xor_sync(FULL, w, 1);
          w |= __shfl_xor_sync(FULL, w, 2);
          w |= __shfl_xor_sync(FULL, w, 4);
          const uint32_t mine = __shfl_sync(FULL, w, 8 * (lane & 3));
          if ((int)(lane >> 2) == st) myword = mine;
        }
        const int wi = (v0 >> 3) + (int)lane;  // 8 slots per word
        if (wi < nwords) wbase[wi] = myword;
      }
    } else {
      for (int i0 = 0; i0 < r.len; i0 += 32) {
        const int i = i0 + (int)lane;
        const bool valid = i < r.len;
        float a = 0.0f;
        if (valid) a = src[g0 + i];
        const unsigned w = __ballot_sync(FULL, valid && !signbit(a));
        if (valid && EF) A.e[g0 + i] = __fsub_rn(a, signbit(a) ? -mu : mu);
        if (lane == 0) wbase[i0 >> 5] = w;
      }
    }
  }
}

// Single-pass sign compression with the residual kept pending.  The sign
// bits depend only on acc, not on the scale, so bits, e and the scale's
// partial sums come out of one pass; the residual e = acc - (bit ? mu : -mu)
// is left to the next call (which receives this call's mu as `prev_mu` and
// applies it in registers before adding g) or to gc_sign_residual_materialize.
// With PREV, e holds the previous call's acc.
template <bool PREV>
__global__ void __launch_bounds__(DTHREADS) k_sign_lazy(DenseArgs A, const float* prev_mu) {
  chain_wait();
  if (aborted(A)) return;
  const unsigned lane = lane_id();
  const int warp = threadIdx.x >> 5;
  const int64_t nwarps = (int64_t)gridDim.x * DWARPS;
  for (int64_t u = (int64_t)blockIdx.x * DWARPS + warp; u < A.U; u += nwarps) {
    const UnitRef r = unit_ref(A, u);
    const int64_t g0 = r.base + r.lstart;
    const float mp = PREV ? prev_mu[r.t] : 0.0f;
    uint32_t* wbase = A.bits + A.woff[r.t] + (r.lstart >> 5);
    const int nwords = (r.len + 31) >> 5;
    ScaledSum<1> sum;
    auto acc_of = [&](float gv, float ev) {
      if (PREV) ev = __fsub_rn(ev, signbit(ev) ? -mp : mp);
      return __fadd_rn(gv, ev);
    };
    if ((g0 & 3) == 0) {
      const int nslots = (r.len + 3) >> 2;
      const float4* g4 = reinterpret_cast<const float4*>(A.g + g0);
      float4* e4 = reinterpret_cast<float4*>(A.e + g0);
      for (int v0 = 0; v0 < nslots; v0 += 256) {
        uint32_t myword = 0u;
#pragma unroll 2
        for (int st = 0; st < 8; ++st) {
          const int vi = v0 + 32 * st + (int)lane;
          unsigned nib = 0u;
          if (vi < nslots) {
            const int li = vi * 4;
            if (li + 4 <= r.len) {
              const float4 gv = ld_stream(g4 + vi);
              const float4 ev = ld_stream(e4 + vi);
              float4 a;
              a.x = acc_of(gv.x, ev.x);
              a.y = acc_of(gv.y, ev.y);
              a.z = acc_of(gv.z, ev.z);
              a.w = acc_of(gv.w, ev.w);
              st_stream(e4 + vi, a);
              nib = (signbit(a.x) ? 0u : 1u) | (signbit(a.y) ? 0u : 2u) | (signbit(a.z) ? 0u : 4u) |
                    (signbit(a.w) ? 0u : 8u);
              sum.bound(max(max(mag_key(a.x), mag_key(a.y)), max(mag_key(a.z), mag_key(a.w))));
              const float m = sum.mult();
              sum.add(a.x, m);
              sum.add(a.y, m);
              sum.add(a.z, m);
              sum.add(a.w, m);
            } else {
              for (int j = 0; li + j < r.len; ++j) {
                const int64_t gi = g0 + li + j;
                const float a = acc_of(A.g[gi], A.e[gi]);
                A.e[gi] = a;
                if (!signbit(a)) nib |= 1u << j;
                sum.add1(a);
              }
            }
          }
          uint32_t w = nib << (4 * (lane & 7));
          w |= __shfl_xor_sync(FULL, w, 1);
          w |= __shfl_xor_sync(FULL, w, 2);
          w |= __shfl_xor_sync(FULL, w, 4);
          const uint32_t mine = __shfl_sync(FULL, w, 8 * (lane & 3));
          if ((int)(lane >> 2) == st) myword = mine;
        }
        const int wi = (v0 >> 3) + (int)lane;
        if (wi < nwords) wbase[wi] = myword;
      }
    } else {
      for (int i0 = 0; i0 < r.len; i0 += 32) {
        const int i = i0 + (int)lane;
        const bool valid = i < r.len;
        float a = 0.0f;
        if (valid) {
          a = acc_of(A.g[g0 + i], A.e[g0 + i]);
          A.e[g0 + i] = a;
          sum.add1(a);
        }
        const unsigned w = __ballot_sync(FULL, valid && !signbit(a));
        if (lane == 0) wbase[i0 >> 5] = w;
      }
    }
    const double part = warp_sum_f64(sum.value());
    if (lane == 0) A.upart[u] = part;
  }
}

// e <- acc - (bit ? mu : -mu) per tensor (pending sign residual made explicit).
__global__ void __launch_bounds__(256) k_sign_materialize(const int64_t* off, int T, float* e,
                                                          const float* mu) {
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
    const float m = mu[t];
    const int64_t base = off[t], n = off[t + 1] - base;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
      const float a = e[base + i];
      e[base + i] = __fsub_rn(a, signbit(a) ? -m : m);
    }
  }
}

// Pass 2 of the int8 / QSGD quantizers: codes and residual.  A lane takes
// 4 float4 slots 32 apart per step; in full steps the four Philox blocks are
// independent chains that the compiler interleaves.
template <int OP, bool EF, bool NZ = false>
__device__ __forceinline__ void quant_slot(const DenseArgs& A, const Divisor& dv, float4 x, uint4 rw,
                                           char4* c4, float4* e4) {
  float4 d;
  char4 c;
  c.x = (signed char)dense_code<OP, EF, NZ>(x.x, dv, A.s_levels, rw.x, &d.x);
  c.y = (signed char)dense_code<OP, EF, NZ>(x.y, dv, A.s_levels, rw.y, &d.y);
  c.z = (signed char)dense_code<OP, EF, NZ>(x.z, dv, A.s_levels, rw.z, &d.z);
  c.w = (signed char)dense_code<OP, EF, NZ>(x.w, dv, A.s_levels, rw.w, &d.w);
  __stcs(reinterpret_cast<int*>(c4), *reinterpret_cast<int*>(&c));
  if (EF) {
    float4 res;
    res.x = __fsub_rn(x.x, d.x);
    res.y = __fsub_rn(x.y, d.y);
    res.z = __fsub_rn(x.z, d.z);
    res.w = __fsub_rn(x.w, d.w);
    st_stream(e4, res);
  }
}

// LO: the arena has fewer than 2^34 elements, so every Philox block index
// fits in 32 bits and the full steps take the shortened rounds of PhiloxLo.
template <int OP, bool EF, bool LO>
__global__ void __launch_bounds__(DTHREADS) k_quant2(DenseArgs A) {
  chain_wait();
  if (aborted(A)) return;
  const unsigned lane = lane_id();
  const int warp = threadIdx.x >> 5;
  const int64_t nwarps = (int64_t)gridDim.x * DWARPS;
  const float* src = EF ? A.e : A.g;
  const uint32_t purpose = (OP == DOP_INT8) ? PURPOSE_INT8 : PURPOSE_QSGD;
  const uint64_t iter = A.iter_dev ? *A.iter_dev : A.iter;
  const PhiloxLo plo(A.pk, iter, purpose);
  for (int64_t u = (int64_t)blockIdx.x * DWARPS + warp; u < A.U; u += nwarps) {
    const UnitRef r = unit_ref(A, u);
    const int64_t g0 = r.base + r.lstart;
    // |acc| <= ||acc|| gives a / N <= s (QSGD); |acc| <= max|acc| gives |acc| / s <= 127 (int8)
    const Divisor dv(A.scale[r.t], 256.0f);
    if ((g0 & 3) == 0) {
      const int nv = r.len >> 2;
      const float4* s4 = reinterpret_cast<const float4*>(src + g0);
      float4* e4 = reinterpret_cast<float4*>(A.e + g0);
      char4* c4 = reinterpret_cast<char4*>(A.codes + g0);
      const uint64_t b0 = (uint64_t)(g0 >> 2);
      for (int v0 = 0; v0 < nv; v0 += 128) {
        float4 x[4];
        if (v0 + 128 <= nv && dv.b == 0.0f) {
          // zero scale: every code is 0 and the residual stays acc
#pragma unroll
          for (int j = 0; j < 4; ++j) __stcs(reinterpret_cast<int*>(c4 + v0 + 32 * j + (int)lane), 0);
        } else if (v0 + 128 <= nv) {
#pragma unroll
          for (int j = 0; j < 4; ++j) x[j] = ld_stream(s4 + v0 + 32 * j + (int)lane);
          uint4 rw[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t b = b0 + (uint64_t)(v0 + 32 * j + (int)lane);
            rw[j] = LO ? plo.block(A.pk, (uint32_t)b) : philox_block(A.pk, iter, b, purpose);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int vi = v0 + 32 * j + (int)lane;
            quant_slot<OP, EF, true>(A, dv, x[j], rw[j], c4 + vi, e4 + vi);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int vi = v0 + 32 * j + (int)lane;
            if (vi < nv) x[j] = ld_stream(s4 + vi);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int vi = v0 + 32 * j + (int)lane;
            if (vi < nv) quant_slot<OP, EF>(A, dv, x[j], philox_block(A.pk, iter, b0 + (uint64_t)vi, purpose),
                                            c4 + vi, e4 + vi);
          }
        }
      }
      const int rem = r.len & 3;
      if ((int)lane < rem) {
        const int64_t gi = g0 + 4 * nv + lane;
        const float x = src[gi];
        float d;
        A.codes[gi] = (int8_t)dense_code<OP, EF>(x, dv, A.s_levels, philox_word(A.pk, iter, (uint64_t)gi, purpose), &d);
        if (EF) A.e[gi] = __fsub_rn(x, d);
      }
    } else {
      for (int i = (int)lane; i < r.len; i += 32) {
        const int64_t gi = g0 + i;
        const float x = src[gi];
        float d;
        A.codes[gi] = (int8_t)dense_code<OP, EF>(x, dv, A.s_levels, philox_word(A.pk, iter, (uint64_t)gi, purpose), &d);
        if (EF) A.e[gi] = __fsub_rn(x, d);
      }
    }
  }
}

// Receiver: out += decode(payload) for one worker.
template <int KIND>
__global__ void __launch_bounds__(DTHREADS) k_ddecode(DenseArgs A, const void* data, const float* scl,
                                                      float* out) {
  chain_wait();
  if (aborted(A)) return;
  const unsigned lane = lane_id();
  const int warp = threadIdx.x >> 5;
  const int64_t nwarps = (int64_t)gridDim.x * DWARPS;
  for (int64_t u = (int64_t)blockIdx.x * DWARPS + warp; u < A.U; u += nwarps) {
    const UnitRef r = unit_ref(A, u);
    const int64_t g0 = r.base + r.lstart;
    const float sc = scl[r.t];
    for (int i = (int)lane; i < r.len; i += 32) {
      const int64_t gi = g0 + i;
      float d;
      if (KIND == GC_DENSE_SIGN) {
        const uint32_t* bits = static_cast<const uint32_t*>(data) + A.woff[r.t] + (r.lstart >> 5);
        d = ((bits[i >> 5] >> (i & 31)) & 1u) ? sc : -sc;
      } else {
        const int c = static_cast<const int8_t*>(data)[gi];
        if (KIND == GC_DENSE_INT8) {
          d = __fmul_rn((float)c, sc);
        } else {
          const int level = c < 0 ? -c : c;
          const float mag = __fdiv_rn(__fmul_rn((float)level, sc), (float)A.s_levels);
          d = c < 0 ? -mag : mag;
        }
      }
      out[gi] = __fadd_rn(out[gi], d);
    }
  }
}

// ============================================================================ host

struct DenseTotals {
  int64_t U = 0, W = 0, N = 0;
};

static DenseTotals dense_totals(const gc_layout* h) {
  DenseTotals z;
  for (int t = 0; t < h->num_tensors; ++t) {
    const int64_t n = h->off[t + 1] - h->off[t];
    z.U += units_of(n);
    z.W += (n + 31) >> 5;
  }
  z.N = h->off[h->num_tensors] - h->off[0];
  return z;
}

struct DenseCarve {
  size_t o_max, zero_bytes, o_units, o_woff, o_part, total;
};

static DenseCarve carve_dense(int T, const DenseTotals& z) {
  DenseCarve c;
  size_t p = DIAG_BYTES;
  auto take = [&p](size_t bytes) {
    const size_t at = p;
    p = align_up(p + bytes, 256);
    return at;
  };
  c.o_max = take(4 * (size_t)T);
  c.zero_bytes = p;
  c.o_units = take(8 * (size_t)(T + 1));
  c.o_woff = take(8 * (size_t)(T + 1));
  c.o_part = take(8 * (size_t)z.U);
  c.total = p;
  return c;
}

size_t dense_workspace_bytes(const gc_layout* h) {
  return carve_dense(h->num_tensors, dense_totals(h)).total;
}

template <class K>
static int dense_grid(K kernel, int64_t units) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, DTHREADS, 0);
  if (per_sm < 1) per_sm = 1;
  int64_t want = (units + DWARPS - 1) / DWARPS;
  int64_t grid = (int64_t)sms * per_sm;
  if (grid > want) grid = want;
  if (grid < 1) grid = 1;
  return (int)grid;
}

static gc_status dense_setup(const gc_layout* dev, const gc_layout* host, void* ws, size_t ws_bytes,
                             cudaStream_t s, DenseArgs* A) {
  gc_status st = validate_layout(host, false);
  if (st != GC_OK) return st;
  if (!dev || !dev->off || dev->num_tensors != host->num_tensors) return GC_ERR_INVALID_ARG;
  const DenseTotals z = dense_totals(host);
  const DenseCarve c = carve_dense(host->num_tensors, z);
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < c.total) return GC_ERR_WORKSPACE;
  unsigned char* w = static_cast<unsigned char*>(ws);
  memset(A, 0, sizeof *A);
  A->T = host->num_tensors;
  A->off = dev->off;
  A->diag = reinterpret_cast<uint32_t*>(w);
  A->maxkey = reinterpret_cast<uint32_t*>(w + c.o_max);
  A->units_off = reinterpret_cast<int64_t*>(w + c.o_units);
  A->woff = reinterpret_cast<int64_t*>(w + c.o_woff);
  A->upart = reinterpret_cast<double*>(w + c.o_part);
  A->U = z.U;
  A->W = z.W;
  A->N = z.N;
  A->off0 = host->off[0];
  if (!zero_chained(ws, c.zero_bytes, s)) return GC_ERR_CUDA;
  launch_chained(k_dplan, 1, 1024, 0, s, *A);
  return GC_OK;
}

template <int OP, bool EF>
static void launch_quant(const DenseArgs& A, cudaStream_t s) {
  launch_chained(k_dense1<OP, EF>, dense_grid(k_dense1<OP, EF>, A.U), DTHREADS, 0, s, A);
  launch_chained(k_dreduce, A.T, 256, 0, s, A);
  if (OP == DOP_SIGN)
    launch_chained(k_sign2<EF>, dense_grid(k_sign2<EF>, A.U), DTHREADS, 0, s, A);
  else if (A.off0 + A.N < (int64_t(1) << 34))
    launch_chained(k_quant2<OP, EF, true>, dense_grid(k_quant2<OP, EF, true>, A.U), DTHREADS, 0, s, A);
  else
    launch_chained(k_quant2<OP, EF, false>, dense_grid(k_quant2<OP, EF, false>, A.U), DTHREADS, 0, s, A);
}

}  // namespace gc

using namespace gc;

extern "C" gc_status gc_sign_compress(const gc_layout* dev, const gc_layout* host, const float* g,
                                      float* e, uint32_t* bits, float* mean_abs, void* workspace,
                                      size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("gc_sign_compress");
  if (!g || !bits || !mean_abs) return GC_ERR_INVALID_ARG;
  if (!aligned16(g) || (e && !aligned16(e))) return GC_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DenseArgs A;
  gc_status st = dense_setup(dev, host, workspace, ws_bytes, s, &A);
  if (st != GC_OK) return st;
  A.op = DOP_SIGN;
  A.ef = e ? 1 : 0;
  A.g = g;
  A.e = e;
  A.bits = bits;
  A.scale = mean_abs;
  if (e)
    launch_quant<DOP_SIGN, true>(A, s);
  else
    launch_quant<DOP_SIGN, false>(A, s);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

static gc_status quantize_entry(const gc_layout* dev, const gc_layout* host, const float* g, float* e,
                                int8_t* codes, float* scale, int32_t mode, int32_t s_levels, uint64_t seed,
                                uint64_t iter, uint64_t* iter_dev, void* workspace, size_t ws_bytes,
                                void* stream) {
  if (!g || !codes || !scale) return GC_ERR_INVALID_ARG;
  if (mode != GC_Q_INT8 && mode != GC_Q_QSGD) return GC_ERR_INVALID_ARG;
  if (mode == GC_Q_QSGD && (s_levels < 1 || s_levels > 127)) return GC_ERR_INVALID_ARG;
  if (!aligned16(g) || (e && !aligned16(e)) || ((uintptr_t)codes & 3u)) return GC_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DenseArgs A;
  gc_status st = dense_setup(dev, host, workspace, ws_bytes, s, &A);
  if (st != GC_OK) return st;
  A.op = (mode == GC_Q_INT8) ? DOP_INT8 : DOP_QSGD;
  A.ef = e ? 1 : 0;
  A.s_levels = s_levels;
  A.g = g;
  A.e = e;
  A.codes = codes;
  A.scale = scale;
  A.seed = seed;
  A.pk = make_philox_key(seed);
  A.iter = iter;
  A.iter_dev = iter_dev;
  if (mode == GC_Q_INT8) {
    if (e) launch_quant<DOP_INT8, true>(A, s);
    else launch_quant<DOP_INT8, false>(A, s);
  } else {
    if (e) launch_quant<DOP_QSGD, true>(A, s);
    else launch_quant<DOP_QSGD, false>(A, s);
  }
  if (iter_dev) launch_chained(k_iter_advance, 1, 1, 0, s, iter_dev);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

extern "C" gc_status gc_quantize_stochastic(const gc_layout* dev, const gc_layout* host,
                                            const float* g, float* e, int8_t* codes, float* scale,
                                            int32_t mode, int32_t s_levels, uint64_t seed,
                                            uint64_t iter, void* workspace, size_t ws_bytes,
                                            void* stream) {
  NvtxRange nvtx_range("gc_quantize_stochastic");
  return quantize_entry(dev, host, g, e, codes, scale, mode, s_levels, seed, iter, nullptr, workspace,
                        ws_bytes, stream);
}

extern "C" gc_status gc_quantize_stochastic_dev_iter(const gc_layout* dev, const gc_layout* host,
                                                     const float* g, float* e, int8_t* codes, float* scale,
                                                     int32_t mode, int32_t s_levels, uint64_t seed,
                                                     uint64_t* iter_dev, void* workspace, size_t ws_bytes,
                                                     void* stream) {
  NvtxRange nvtx_range("gc_quantize_stochastic_dev_iter");
  if (!iter_dev || ((uintptr_t)iter_dev & 7u)) return GC_ERR_INVALID_ARG;
  return quantize_entry(dev, host, g, e, codes, scale, mode, s_levels, seed, 0, iter_dev, workspace,
                        ws_bytes, stream);
}

extern "C" gc_status gc_dense_decompress_accumulate(const gc_layout* dev, const gc_layout* host,
                                                    int32_t W, int32_t kind, int32_t s_levels,
                                                    const void* const* data,
                                                    const float* const* scale, float* out,
                                                    void* workspace, size_t ws_bytes,
                                                    void* stream) {
  NvtxRange nvtx_range("gc_dense_decompress_accumulate");
  if (W < 0 || !out || (W > 0 && (!data || !scale))) return GC_ERR_INVALID_ARG;
  if (kind != GC_DENSE_SIGN && kind != GC_DENSE_INT8 && kind != GC_DENSE_QSGD) return GC_ERR_INVALID_ARG;
  if (kind == GC_DENSE_QSGD && (s_levels < 1 || s_levels > 127)) return GC_ERR_INVALID_ARG;
  if (!aligned16(out)) return GC_ERR_ALIGNMENT;
  for (int w = 0; w < W; ++w)
    if (!data[w] || !scale[w]) return GC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DenseArgs A;
  gc_status st = dense_setup(dev, host, workspace, ws_bytes, s, &A);
  if (st != GC_OK) return st;
  A.s_levels = s_levels;
  for (int w = 0; w < W; ++w) {
    if (kind == GC_DENSE_SIGN)
      launch_chained(k_ddecode<GC_DENSE_SIGN>, dense_grid(k_ddecode<GC_DENSE_SIGN>, A.U), DTHREADS, 0, s, A, data[w],
                     scale[w], out);
    else if (kind == GC_DENSE_INT8)
      launch_chained(k_ddecode<GC_DENSE_INT8>, dense_grid(k_ddecode<GC_DENSE_INT8>, A.U), DTHREADS, 0, s, A, data[w],
                     scale[w], out);
    else
      launch_chained(k_ddecode<GC_DENSE_QSGD>, dense_grid(k_ddecode<GC_DENSE_QSGD>, A.U), DTHREADS, 0, s, A, data[w],
                     scale[w], out);
  }
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

extern "C" gc_status gc_sign_compress_lazy(const gc_layout* dev, const gc_layout* host,
                                           const float* g, float* e, const float* prev_mean_abs,
                                           uint32_t* bits, float* mean_abs, void* workspace,
                                           size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("gc_sign_compress_lazy");
  if (!g || !e || !bits || !mean_abs) return GC_ERR_INVALID_ARG;
  if (!aligned16(g) || !aligned16(e)) return GC_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DenseArgs A;
  gc_status st = dense_setup(dev, host, workspace, ws_bytes, s, &A);
  if (st != GC_OK) return st;
  A.op = DOP_SIGN;
  A.ef = 1;
  A.g = g;
  A.e = e;
  A.bits = bits;
  A.scale = mean_abs;
  if (prev_mean_abs)
    launch_chained(k_sign_lazy<true>, dense_grid(k_sign_lazy<true>, A.U), DTHREADS, 0, s, A, prev_mean_abs);
  else
    launch_chained(k_sign_lazy<false>, dense_grid(k_sign_lazy<false>, A.U), DTHREADS, 0, s, A,
                   (const float*)nullptr);
  launch_chained(k_dreduce, A.T, 256, 0, s, A);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

extern "C" gc_status gc_sign_residual_materialize(const gc_layout* dev, const gc_layout* host,
                                                  float* e, const float* mean_abs, void* stream) {
  NvtxRange nvtx_range("gc_sign_residual_materialize");
  const gc_status st = validate_layout(host, false);
  if (st != GC_OK) return st;
  if (!dev || !dev->off || dev->num_tensors != host->num_tensors || !e || !mean_abs) return GC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int T = host->num_tensors;
  k_sign_materialize<<<dim3(256, (unsigned)(T < 65535 ? T : 65535)), 256, 0, s>>>(dev->off, T, e, mean_abs);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}
