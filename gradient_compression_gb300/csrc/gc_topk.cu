// EF Top-k / random-k / momentum-corrected Top-k compression (sm_103a).
//
// Method: mbrenndoerfer.com "Gradient Compression", Top-K Sparsification
// (g^ = TopK(g + e), e = (g + e) - g^, fp32 value + int32 index payload);
// inferensys.com zh glossary (Random-k; Top-k + 8-bit); inferensys.com
// "Gradient Sparsification" (per-layer selection, momentum correction and
// factor masking).
//
// Pipeline for one call (all tensors of the arena at once, stream-ordered):
//   plan       per-tensor prefix tables (units, unit blocks, candidate and
//              sample regions) from the device layout
//   sample     a strided sample of acc per tensor, two shared-memory radix
//              levels -> a threshold estimate t_est below the k-th magnitude
//              (Top-k, momentum, threshold; random-k keys are uniform, so
//              t_est is set analytically by the plan)
//   [clip]     per-tensor ||g|| and the clipping multiplier (local clipping)
//   stream     THE pass over HBM: acc = g + e (or the momentum update),
//              write-back of e (u, v), and emission of every element whose
//              key >= t_est into an index-ordered per-unit candidate chunk,
//              plus the level-1 histogram of candidate keys
//   select     exact radix select (11 + 11 + 10 bits) of the k-th key over
//              the candidates; a tensor whose candidates are insufficient
//              (fewer than k, or overflow) is selected by full passes over
//              its acc instead (same result)
//   count/scan/write  index-ordered compaction of the kept set into the
//              payload, int8 stochastic rounding, and the residual scatter
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "gc_common.cuh"
#include "gc_host.h"

namespace gc {

enum { MODE_TOPK = 0, MODE_RANDK = 1, MODE_MOM = 2 };
// Quantizer of the kept values beyond int8 (A.int8): QSGD levels with the
// norm of the kept vector, or sign bits with the mean |kept value|.
enum { KQ_NONE = 0, KQ_QSGD = 2, KQ_SIGN = 3 };
enum { PH_C1 = 0, PH_C1D = 1, PH_C2 = 2, PH_C3 = 3 };

struct TopkArgs {
  int T;
  int mode;
  uint32_t flags;
  int int8;
  int ef;
  int unbiased;
  int masking;
  float beta;
  const int64_t* off;
  const int64_t* kk;
  const int64_t* koff;
  const float* g;
  float* e;
  float* u;
  float* v;
  int32_t* idx;
  float* val;
  int8_t* q;
  float* scale;
  uint64_t seed, iter;
  const uint64_t* iter_dev;  // iteration counter in device memory (graph capture), else null
  PhiloxKey pk;          // round keys of seed
  gc_residual_desc* rd;  // pending-residual descriptors (lazy mode), else null
  const float* tau;      // per-tensor magnitude thresholds (threshold mode), else null
  int64_t* count_out;    // per-tensor kept counts (threshold mode)
  int sampled;           // threshold estimated by sampling (Top-k and momentum)
  const float* clip;     // per-tensor maximum L2 norm of g (local clipping), else null
  float* norm_out;       // per-tensor ||g||_2 (local clipping)
  double* upart;         // per-unit partial sums of g^2 (local clipping); per-unit-block sums
                         // over the kept values (QSGD / sign of the kept values)
  int qkind;             // KQ_*: QSGD or sign of the kept values
  int slev;              // QSGD levels
  uint32_t* bits;        // sign bits of the kept values (KQ_SIGN)
  int64_t* kwoff;        // [T+1] first word of each tensor's kept-value sign bits
  // workspace
  uint32_t* diag;
  TensorState* ts;
  uint32_t* hist;
  int64_t* units_off;
  int64_t* ublk_off;
  int64_t* cand_off;
  int64_t* soff;
  uint2* chunk;
  uint32_t* ugt;
  uint32_t* ueq;
  uint32_t* bgt;
  uint32_t* beq;
  uint32_t* ckey;
  int32_t* cidx;
  float* cval;
  uint32_t* skey;
  int64_t* sblk;       // [T+1] first sampling CTA of each tensor (tensor order)
  int64_t* sord;       // [T]   where the tensor's CTAs start in the dispatch order (planner scratch)
  int2* smap;          // [SB]  sampling CTA (dispatch order) -> (tensor, its CTA index)
  uint32_t* scnt;      // [2T] per tensor: keys in its sample list, sampling CTAs finished (zeroed per call)
  int64_t U, UB, C, S, N, K, SB;
  int64_t off0, koff0;  // off[0] and koff[0] of the host layout (nonzero for a bucket)
  int ubu;              // units per unit block (UB_UNITS or UB_UNITS_DENSE)
  int ssplit;          // sampling CTAs per large sample (sample_ctas)
};

// ============================================================================ plan

// Exclusive block scans of NV values per thread at once (one pass of warp
// shuffles and three barriers for all of them); tot receives the totals.
template <int NV>
__device__ void block_excl_scan_multi(int64_t (&v)[NV], int64_t (*s_w)[32], int64_t (&tot)[NV]) {
  const unsigned lane = lane_id(), w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int64_t x[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) x[i] = v[i];
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int64_t y = __shfl_up_sync(FULL, x[i], d);
      if (lane >= (unsigned)d) x[i] += y;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int i = 0; i < NV; ++i) s_w[i][w] = x[i];
  }
  __syncthreads();
  if (w == 0) {
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      int64_t z = lane < nw ? s_w[i][lane] : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int64_t y = __shfl_up_sync(FULL, z, d);
        if (lane >= (unsigned)d) z += y;
      }
      if (lane < nw) s_w[i][lane] = z;  // inclusive warp prefix
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    tot[i] = s_w[i][nw - 1];
    v[i] = (w == 0 ? 0 : s_w[i][w - 1]) + x[i] - v[i];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(1024) k_plan(TopkArgs A) {
  chain_wait();
  __shared__ int64_t s_scan[8][32];
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  int64_t carry_u = 0, carry_b = 0, carry_c = 0, carry_s = 0, carry_w = 0, carry_sb = 0, carry_lb = 0, carry_xb = 0;
  const bool sampled = A.sampled != 0;
  for (int base = 0; base < A.T; base += blockDim.x) {
    const int t = base + threadIdx.x;
    int64_t nu = 0, nb = 0, nc = 0, ns = 0, nw = 0, nsb = 0, nlb = 0, nxb = 0;
    if (t < A.T) {
      const int64_t n = A.off[t + 1] - A.off[t];
      const int64_t k = A.kk[t];
      if (n < 1 || n > INT64_C(2147483647) || k < 0 || k > n || A.koff[t + 1] - A.koff[t] != k) s_bad = 1;
      nu = units_of(n);
      nb = ublocks_of(n, A.ubu);
      nc = cand_capacity(n, k);
      nw = k > 0 ? (k + 31) >> 5 : 0;
      nsb = sampled ? sample_ctas(n, k, A.ssplit) : 0;
      // long samples (the filtered search) are dispatched before short ones
      if (sample_splittable(n, k))
        nlb = nsb;
      else
        nxb = nsb;
      TensorState st;
      memset(&st, 0, sizeof st);
      if (sampled && k > 0) {
        int64_t runs, stride, m;
        sample_plan(n, k, &runs, &stride, &m);
        ns = m;
        // the sample key of rank j bounds t_est: j = k for a complete sample,
        // else the expected count lam of Top-k members in the sample plus five
        // standard deviations (and 6).  Fewer than k candidates then needs a
        // Poisson(lam) count of at least j (about 1e-7 at lam = 64 or 128); with four
        // (and 4) about one tensor-step in 10^4 fell short under error
        // feedback and took the full-pass path.  Each standard deviation of
        // margin costs about 7% more candidates.
        int64_t j = k;
        if (m < n) {
          const double lam = (double)k * (double)m / (double)n;
          j = (int64_t)ceil(lam + 5.0 * sqrt(lam) + 6.0);
        }
        st.s_runs = (uint32_t)runs;
        st.s_stride = (uint32_t)stride;
        st.s_j = (uint32_t)min(j, m + 1);
        // pilot rank whose count scales to about 4j over the whole sample
        const int64_t rp = (4 * j * (int64_t)SPILOT + runs - 1) / runs + 4;
        st.s_rp = (uint32_t)min(rp, (int64_t)SLIST);
      }
      if (k <= 0) st.flags = TS_NOEMIT;
      if (A.mode == MODE_RANDK && k > 0) {
        // keys ~kappa, kappa uniform on 32-bit words: emit kappa < tau with
        // tau chosen so that about k + 4 sqrt(k) + 16 elements qualify
        const double want = (double)k + 4.0 * sqrt((double)k) + 16.0;
        const double tau = floor(want * 4294967296.0 / (double)n);
        st.t_est = (tau >= 4294967296.0) ? 0u : ~((uint32_t)tau - 1u);
      }
      if (k >= n || (sampled && n <= NOSAMPLE_N)) st.t_est = 0u;  // every element a candidate
      if (A.tau && k > 0) {
        const float tau = A.tau[t];
        if (tau >= 0.0f) {
          st.t_est = mag_key(tau);  // |acc| >= tau  <=>  key(acc) >= key(tau)
        } else {                    // NaN or negative: reported, nothing kept
          st.flags = TS_NOEMIT;
          atomicOr(A.diag + DIAG_ERR, GC_DIAG_BAD_THRESHOLD);
        }
      }
      st.keff = (uint32_t)k;
      st.gmul = 1.0f;
      A.ts[t] = st;
      if (A.count_out && (st.flags & TS_NOEMIT)) A.count_out[t] = 0;
      if ((A.int8 || A.qkind != KQ_NONE) && k <= 0) A.scale[t] = 0.0f;
    }
    // all eight prefix tables in one block scan
    int64_t v[8] = {nu, nb, nc, ns, nw, nsb, nlb, nxb}, tot[8];
    block_excl_scan_multi<8>(v, s_scan, tot);
    if (t < A.T) {
      A.units_off[t] = carry_u + v[0];
      A.ublk_off[t] = carry_b + v[1];
      A.cand_off[t] = carry_c + v[2];
      A.soff[t] = carry_s + v[3];
      A.kwoff[t] = carry_w + v[4];
      A.sblk[t] = carry_sb + v[5];
      // dispatch order of the sampling CTAs: the long samples' CTAs first (a
      // short sample's CTA takes a fraction of a long one's time, so the
      // short ones fill the slots that free up instead of holding long ones
      // back to a second wave); short starts are offset by the long total below
      A.sord[t] = nlb > 0 ? carry_lb + v[6] : -1 - (carry_xb + v[7]);
    }
    carry_u += tot[0];
    carry_b += tot[1];
    carry_c += tot[2];
    carry_s += tot[3];
    carry_w += tot[4];
    carry_sb += tot[5];
    carry_lb += tot[6];
    carry_xb += tot[7];
  }
  __syncthreads();
  for (int t = threadIdx.x; t < A.T; t += blockDim.x) {
    const int64_t o = A.sord[t];
    const int64_t start = o >= 0 ? o : carry_lb + (-1 - o);
    const int64_t cnt = (t + 1 < A.T ? A.sblk[t + 1] : carry_sb) - A.sblk[t];
    for (int64_t c = 0; c < cnt && start + c < A.SB; ++c) A.smap[start + c] = make_int2(t, (int)c);
  }
  if (threadIdx.x == 0) {
    A.units_off[A.T] = carry_u;
    A.ublk_off[A.T] = carry_b;
    A.cand_off[A.T] = carry_c;
    A.soff[A.T] = carry_s;
    A.kwoff[A.T] = carry_w;
    A.sblk[A.T] = carry_sb;
    if (s_bad || carry_u != A.U || carry_b != A.UB || carry_c != A.C || carry_s != A.S || carry_sb != A.SB ||
        A.off[0] != A.off0 || A.off[A.T] - A.off0 != A.N || A.koff[0] != A.koff0 || A.koff[A.T] - A.koff0 != A.K) {
      A.diag[DIAG_ERR] |= GC_DIAG_LAYOUT_MISMATCH;
      A.diag[DIAG_ABORT] = 1u;
    }
  }
}

// ============================================================================ acc of one element

// Lazy mode.  An element whose stored value x is the acc of the call
// described by d was kept by that call iff its key is above the k-th key, or
// equal to it at an index up to the last kept tie.
__device__ __forceinline__ bool lazy_kept(float x, int64_t li, const gc_residual_desc& d) {
  const uint32_t key = mag_key(x);
  return (d.flags & 1u) && (key > d.thr || (key == d.thr && li <= (int64_t)d.last_tie));
}

// Residual of a kept element: +0, or acc - q*s with the int8 code redrawn
// from that call's Philox words (equal to what the eager update writes).
// Not inlined, so that the rare redraw stays out of the streaming loop.
__device__ __noinline__ float lazy_kept_residual(float x, int64_t gi, gc_residual_desc d) {
  if (!(d.flags & 2u)) return 0.0f;
  const int c = int8_code(x, d.scale, philox_word(d.seed, d.iter, (uint64_t)gi, PURPOSE_INT8));
  return __fsub_rn(x, __fmul_rn((float)c, d.scale));
}

// Exact EF residual of an element stored in pending form.
__device__ __forceinline__ float lazy_fix(float x, int64_t li, int64_t gi, const gc_residual_desc& d) {
  return lazy_kept(x, li, d) ? lazy_kept_residual(x, gi, d) : x;
}

// acc of element gi (local index li of tensor t) computed from the inputs
// (used by the sampler; the streaming pass computes the same expression).
template <int MODE>
__device__ __forceinline__ float acc_from_inputs(const TopkArgs& A, int t, int64_t li, int64_t gi) {
  if (MODE == MODE_MOM) {
    const float un = __fadd_rn(__fmul_rn(A.beta, A.u[gi]), A.g[gi]);
    return __fadd_rn(A.v[gi], un);
  }
  const float gv = __fmul_rn(A.ts[t].gmul, A.g[gi]);
  if (!A.ef) return gv;
  const float r = A.rd ? lazy_fix(A.e[gi], li, gi, A.rd[t]) : A.e[gi];
  return __fadd_rn(gv, r);
}

// After the streaming pass: the kept value source and the selection key.
template <int MODE>
__device__ __forceinline__ const float* value_source(const TopkArgs& A) {
  if (MODE == MODE_MOM) return A.v;
  return A.ef ? A.e : A.g;
}

// The call's iteration counter: the argument, or the device-resident counter
// of the *_dev_iter entry points (read where used, so a captured call sees
// each replay's value).
__device__ __forceinline__ uint64_t iter_of(const TopkArgs& A) { return A.iter_dev ? *A.iter_dev : A.iter; }

template <int MODE>
__device__ __forceinline__ uint32_t key_of(const TopkArgs& A, float value, int64_t gi) {
  if (MODE == MODE_RANDK) return ~philox_word(A.pk, iter_of(A), (uint64_t)gi, PURPOSE_RANDK);
  return mag_key(value);
}

__device__ __forceinline__ bool aborted(const TopkArgs& A) { return A.diag[DIAG_ABORT] != 0u; }

// ============================================================================ sampling

// Four consecutive acc values (elements li .. li+3 of tensor t, arena base
// `base`), read with one 16-byte load per input when aligned and complete.
template <int MODE>
__device__ __forceinline__ void acc4_from_inputs(const TopkArgs& A, int t, int64_t base, int64_t n,
                                                 int64_t li, bool vec, float gmul, float a[4], bool ok[4]) {
  const int64_t gi = base + li;
  if (vec && li + 4 <= n) {
    float4 g4 = ld_stream(reinterpret_cast<const float4*>(A.g + gi));
    if (MODE != MODE_MOM) {
      const float c = gmul;
      g4.x = __fmul_rn(c, g4.x);
      g4.y = __fmul_rn(c, g4.y);
      g4.z = __fmul_rn(c, g4.z);
      g4.w = __fmul_rn(c, g4.w);
    }
    if (MODE == MODE_MOM) {
      const float4 u4 = ld_stream(reinterpret_cast<const float4*>(A.u + gi));
      const float4 v4 = ld_stream(reinterpret_cast<const float4*>(A.v + gi));
      a[0] = __fadd_rn(v4.x, __fadd_rn(__fmul_rn(A.beta, u4.x), g4.x));
      a[1] = __fadd_rn(v4.y, __fadd_rn(__fmul_rn(A.beta, u4.y), g4.y));
      a[2] = __fadd_rn(v4.z, __fadd_rn(__fmul_rn(A.beta, u4.z), g4.z));
      a[3] = __fadd_rn(v4.w, __fadd_rn(__fmul_rn(A.beta, u4.w), g4.w));
    } else if (A.ef) {
      float4 e4 = ld_stream(reinterpret_cast<const float4*>(A.e + gi));
      if (A.rd) {
        const gc_residual_desc d = A.rd[t];
        e4.x = lazy_fix(e4.x, li + 0, gi + 0, d);
        e4.y = lazy_fix(e4.y, li + 1, gi + 1, d);
        e4.z = lazy_fix(e4.z, li + 2, gi + 2, d);
        e4.w = lazy_fix(e4.w, li + 3, gi + 3, d);
      }
      a[0] = __fadd_rn(g4.x, e4.x);
      a[1] = __fadd_rn(g4.y, e4.y);
      a[2] = __fadd_rn(g4.z, e4.z);
      a[3] = __fadd_rn(g4.w, e4.w);
    } else {
      a[0] = g4.x; a[1] = g4.y; a[2] = g4.z; a[3] = g4.w;
    }
    ok[0] = ok[1] = ok[2] = ok[3] = true;
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    ok[j] = li + j < n;
    a[j] = ok[j] ? acc_from_inputs<MODE>(A, t, li + j, gi + j) : 0.0f;
  }
}

// ============================================================================ local clipping


// Per-unit partial sums of g^2 (scaled compensated fp32 per lane, fp64 across lanes).
__global__ void __launch_bounds__(256) k_gnorm(TopkArgs A) {
  chain_wait();
  if (aborted(A)) return;
  const unsigned lane = lane_id();
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < A.U; u += nwarps) {
    const int t = find_segment(A.units_off, A.T, u);
    const int64_t base = A.off[t], n = A.off[t + 1] - base;
    const int64_t lstart = (u - A.units_off[t]) << UNIT_SHIFT;
    const int len = (int)min((int64_t)UNIT, n - lstart);
    const int64_t g0 = base + lstart;
    ScaledSum<2> acc;
    if ((g0 & 3) == 0) {
      const int nv = len >> 2;
      const float4* g4 = reinterpret_cast<const float4*>(A.g + g0);
      for (int v0 = 0; v0 < nv; v0 += 128) {
        float4 x[4];
        uint32_t km = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int vi = v0 + 32 * j + (int)lane;
          x[j] = vi < nv ? ld_stream(g4 + vi) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          km = max(km, max(max(mag_key(x[j].x), mag_key(x[j].y)), max(mag_key(x[j].z), mag_key(x[j].w))));
        acc.bound(km);
        const float m = acc.mult();
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // zeros past the end add nothing
          acc.add(x[j].x, m);
          acc.add(x[j].y, m);
          acc.add(x[j].z, m);
          acc.add(x[j].w, m);
        }
      }
      if ((int)lane < (len & 3)) acc.add1(A.g[g0 + 4 * nv + lane]);
    } else {
      for (int i = (int)lane; i < len; i += 32) acc.add1(A.g[g0 + i]);
    }
    double part = acc.value();
#pragma unroll
    for (int dd = 16; dd > 0; dd >>= 1) part += __shfl_xor_sync(FULL, part, dd);
    if (lane == 0) A.upart[u] = part;
  }
}

// Per tensor: N = ||g_t||_2 (fixed-order fp64 sum of the unit partials) and
// the clipping multiplier c = C / N when N > C, else 1.
__global__ void __launch_bounds__(256) k_gscale(TopkArgs A) {
  chain_wait();
  __shared__ double s_part[256];
  if (aborted(A)) return;
  const int t = blockIdx.x;
  double v = 0.0;
  for (int64_t u = A.units_off[t] + threadIdx.x; u < A.units_off[t + 1]; u += blockDim.x) v += A.upart[u];
  s_part[threadIdx.x] = v;
  __syncthreads();
  for (int h = 128; h > 0; h >>= 1) {
    if ((int)threadIdx.x < h) s_part[threadIdx.x] += s_part[threadIdx.x + h];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const float N = __double2float_rn(sqrt(s_part[0]));
    const float C = A.clip[t];
    float c = 1.0f;
    if (!(C >= 0.0f))
      atomicOr(A.diag + DIAG_ERR, GC_DIAG_BAD_THRESHOLD);
    else if (N > C)
      c = __fdiv_rn(C, N);
    A.norm_out[t] = N;
    A.ts[t].gmul = c;
  }
}

// ============================================================================ select

__device__ void block_scan_u32(uint32_t v, uint32_t* s_warp, uint32_t* excl, uint32_t* total) {
  const unsigned lane = lane_id(), w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned tw;
  const unsigned e = warp_excl_scan(v, lane, &tw);
  if (lane == 0) s_warp[w] = tw;
  __syncthreads();
  if (w == 0) {
    unsigned z = lane < nw ? s_warp[lane] : 0u, tz;
    const unsigned ez = warp_excl_scan(z, lane, &tz);
    if (lane < nw) s_warp[lane] = ez;
    if (lane == 0) s_warp[32] = tz;
  }
  __syncthreads();
  *excl = s_warp[w] + e;
  *total = s_warp[32];
  __syncthreads();
}

// Finds the bucket holding the rank-th largest key of a 2048-bin histogram
// (bins in key order; `row` in global or shared memory).  Returns the bin and
// the number of keys in the bins above it, or 0xFFFFFFFF when the histogram
// holds fewer than `rank` keys.  Called by all 256 threads of the block.
__device__ uint32_t find_bucket(const uint32_t* row, uint32_t rank, uint32_t* above,
                                uint32_t* s_warp, uint32_t* s_res) {
  // thread i owns `per` bins from 2047 - per*i downwards (keys in descending
  // order); blockDim.x is 256, 512 or 1024
  const int per = NBINS / (int)blockDim.x;
  uint32_t h[8], sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    h[j] = j < per ? row[NBINS - 1 - per * threadIdx.x - j] : 0u;
    sum += h[j];
  }
  uint32_t pre, total;
  block_scan_u32(sum, s_warp, &pre, &total);
  if (threadIdx.x == 0) s_res[0] = 0xFFFFFFFFu;
  __syncthreads();
  const uint32_t r0 = rank - 1u;
  if (rank >= 1u && rank <= total && r0 >= pre && r0 < pre + sum) {
    uint32_t acc = pre;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < per && r0 < acc + h[j]) {
        s_res[0] = NBINS - 1 - per * threadIdx.x - j;
        s_res[1] = acc;
        break;
      }
      acc += h[j];
    }
  }
  __syncthreads();
  const uint32_t b = s_res[0];
  *above = s_res[1];
  __syncthreads();
  return b;
}

// Threshold estimate t_est from a strided sample of acc, by CTAs of 512
// threads (two per SM; each warp keeps SR runs in flight): one per tensor,
// or for a sample of at least SFILTER_RUNS runs one per SAMPLE_RUNS_PER_CTA
// runs, which filter their shares and leave the search to the last of them.  The sample is runs
// of RUN = 128 consecutive elements (one warp, 16 bytes per lane per input)
// spaced `stride` apart; small tensors are sampled completely.
//
// t_est is the lower edge of the level-2 bucket (top 22 bits of the key) of
// the j-th largest sample key, so t_est <= that key.  It is found from a
// radix pass of two levels (top 11 bits, next 11 bits) over the sample keys
// that matter:
//  * filtered path (samples of at least SFILTER_RUNS runs): a pilot of
//    SPILOT runs spread evenly over the sample gives a floor F, the level-2
//    edge of the pilot key whose rank scales to about 4j in the whole sample;
//    one pass over the sample then keeps only the keys >= F (histogram of
//    their top bits, list in shared memory).  When at least j keys pass, the
//    j-th largest and its buckets lie among them and every key above it is
//    counted, so both levels give the same buckets as over the whole sample;
//  * direct path (small samples, or a filter that kept fewer than j keys or
//    more than the list holds): both levels over every sample key, the keys
//    stored in the sample key buffer between the levels.

// Keys of the sample runs r = (r0 + h * rstep) * rmul, h < SR, r0 + h * rstep < rend;
// bit c of okm[h] flags key[h][c] as a sample element.  Every run's loads
// are issued before any is used, so that a warp keeps SR runs in flight;
// runs that are not whole aligned float4s per lane (the tensor's tail, an
// unaligned tensor) and the pending-residual mode (which rebuilds e per
// element) take the per-run path.
template <int MODE>
constexpr int sample_runs_in_flight() { return MODE == MODE_MOM ? 2 : 4; }

template <int MODE, int SR>
__device__ __forceinline__ void sample_keys(const TopkArgs& A, int t, int64_t base, int64_t n, int64_t stride,
                                            int r0, int rstep, int rend, int rmul, bool vec, float gmul,
                                            unsigned lane, uint32_t key[SR][4], unsigned okm[SR]) {
  constexpr bool MOM = MODE == MODE_MOM;
  if (!MOM && A.rd) {
    // pending residual: one run at a time
#pragma unroll
    for (int h = 0; h < SR; ++h) {
      const int ri = r0 + h * rstep;
      float a[4];
      bool ok[4] = {false, false, false, false};
      if (ri < rend)
        acc4_from_inputs<MODE>(A, t, base, n, sample_run_start((int64_t)ri * rmul, stride) + 4 * lane, vec, gmul,
                               a, ok);
      okm[h] = (ok[0] ? 1u : 0u) | (ok[1] ? 2u : 0u) | (ok[2] ? 4u : 0u) | (ok[3] ? 8u : 0u);
#pragma unroll
      for (int c = 0; c < 4; ++c) key[h][c] = ok[c] ? mag_key(a[c]) : 0u;
    }
    return;
  }
  const float* gp = A.g + base;
  const float* ep = MOM ? A.u + base : A.e + base;  // second input (e, or u)
  const float* vp = A.v + base;
  const bool ef = MOM || A.ef;
  float4 x[SR], y[SR], z[SR];
  int li[SR];  // n < 2^31
#pragma unroll
  for (int h = 0; h < SR; ++h) {
    const int ri = r0 + h * rstep;
    li[h] = ri < rend ? (int)sample_run_start((int64_t)ri * rmul, stride) + 4 * (int)lane : (int)n;
    if (vec && (int64_t)li[h] + 4 <= n) {
      x[h] = ld_stream(reinterpret_cast<const float4*>(gp + li[h]));
      if (ef) y[h] = ld_stream(reinterpret_cast<const float4*>(ep + li[h]));
      if (MOM) z[h] = ld_stream(reinterpret_cast<const float4*>(vp + li[h]));
    } else {
      // tail or unaligned tensor: element loads, zero past the end
      float xs[4] = {0.f, 0.f, 0.f, 0.f}, ys[4] = {0.f, 0.f, 0.f, 0.f}, zs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if ((int64_t)li[h] + c < n) {
          xs[c] = gp[li[h] + c];
          if (ef) ys[c] = ep[li[h] + c];
          if (MOM) zs[c] = vp[li[h] + c];
        }
      }
      x[h] = make_float4(xs[0], xs[1], xs[2], xs[3]);
      y[h] = make_float4(ys[0], ys[1], ys[2], ys[3]);
      z[h] = make_float4(zs[0], zs[1], zs[2], zs[3]);
    }
  }
#pragma unroll
  for (int h = 0; h < SR; ++h) {
    const float g4[4] = {x[h].x, x[h].y, x[h].z, x[h].w}, e4[4] = {y[h].x, y[h].y, y[h].z, y[h].w};
    unsigned m = 0u;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float a;
      if (MOM) {
        const float v4[4] = {z[h].x, z[h].y, z[h].z, z[h].w};
        a = __fadd_rn(v4[c], __fadd_rn(__fmul_rn(A.beta, e4[c]), g4[c]));
      } else {
        const float gv = __fmul_rn(gmul, g4[c]);
        a = ef ? __fadd_rn(gv, e4[c]) : gv;
      }
      const bool ok = (int64_t)li[h] + c < n;
      m |= (ok ? 1u : 0u) << c;
      key[h][c] = ok ? mag_key(a) : 0u;
    }
    okm[h] = m;
  }
}

// The pilot of the filtered search: SPILOT runs spread evenly over the
// sample, their keys in sl; returns the floor F (the level-2 edge of the
// pilot key of rank rp).  Leaves sh zero.
template <int MODE>
__device__ uint32_t sample_pilot_floor(const TopkArgs& A, int t, int64_t base, int64_t n, int64_t stride, int runs,
                                       uint32_t rp, bool vec, float gmul, uint32_t* sh, uint32_t* sl,
                                       uint32_t* s_warp, uint32_t* s_res) {
  constexpr int SR = sample_runs_in_flight<MODE>();
  const unsigned lane = lane_id();
  const int nwarp = blockDim.x >> 5, w = threadIdx.x >> 5;
  uint32_t key[SR][4];
  unsigned okm[SR];
  const int ps = runs / SPILOT;
  for (int i0 = w; i0 < SPILOT; i0 += SR * nwarp) {
    sample_keys<MODE, SR>(A, t, base, n, stride, i0, nwarp, SPILOT, ps, vec, gmul, lane, key, okm);
#pragma unroll
    for (int h = 0; h < SR; ++h) {
      const int i = i0 + h * nwarp;
      if (i < SPILOT) {
#pragma unroll
        for (int c = 0; c < 4; ++c) sl[i * RUN + 4 * lane + c] = key[h][c];
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < SLIST; i += blockDim.x) atomicAdd(sh + (sl[i] >> 21), 1u);
  __syncthreads();
  uint32_t pabove;
  const uint32_t p1 = find_bucket(sh, rp, &pabove, s_warp, s_res);
  for (int i = threadIdx.x; i < NBINS; i += blockDim.x) sh[i] = 0u;
  __syncthreads();
  uint32_t F = 0u;
  if (p1 != 0xFFFFFFFFu) {
    for (int i = threadIdx.x; i < SLIST; i += blockDim.x) {
      const uint32_t kk = sl[i];
      if ((kk >> 21) == p1) atomicAdd(sh + ((kk >> 10) & 0x7FFu), 1u);
    }
    __syncthreads();
    uint32_t pabove2;
    const uint32_t p2 = find_bucket(sh, rp - pabove, &pabove2, s_warp, s_res);
    F = (p1 << 21) | (p2 == 0xFFFFFFFFu ? 0u : (p2 << 10));
    for (int i = threadIdx.x; i < NBINS; i += blockDim.x) sh[i] = 0u;
  }
  __syncthreads();
  return F;
}

// The filtered pass over sample runs [r_lo, r_hi): the keys >= F go to the
// level-1 histogram sh and to a list, at positions reserved with atomics on
// *cnt (a shared counter for a list in shared memory, or a global one for
// the tensor's list in the sample key buffer); positions at or above cap are
// counted but not stored.
template <int MODE>
__device__ void sample_filter_pass(const TopkArgs& A, int t, int64_t base, int64_t n, int64_t stride, int r_lo,
                                   int r_hi, bool vec, float gmul, uint32_t F, uint32_t* sh, uint32_t* list,
                                   uint32_t cap, uint32_t* cnt) {
  constexpr int SR = sample_runs_in_flight<MODE>();
  const unsigned lane = lane_id();
  const int nwarp = blockDim.x >> 5, w = threadIdx.x >> 5;
  uint32_t key[SR][4];
  unsigned okm[SR];
  for (int r0 = r_lo + w; r0 < r_hi; r0 += SR * nwarp) {
    sample_keys<MODE, SR>(A, t, base, n, stride, r0, nwarp, r_hi, 1, vec, gmul, lane, key, okm);
#pragma unroll
    for (int h = 0; h < SR; ++h) {
      unsigned msk = 0u;
#pragma unroll
      for (int c = 0; c < 4; ++c) msk |= (((okm[h] >> c) & 1u) && key[h][c] >= F ? 1u : 0u) << c;
      if (__any_sync(FULL, msk != 0u)) {
        unsigned pre, tot;
        warp_count_scan(__popc(msk), lane, &pre, &tot);
        uint32_t at = 0u;
        if (lane == 0) at = atomicAdd(cnt, tot);
        at = __shfl_sync(FULL, at, 0) + pre;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if ((msk >> c) & 1u) {
            atomicAdd(sh + (key[h][c] >> 21), 1u);
            if (at < cap) list[at] = key[h][c];
            ++at;
          }
        }
      }
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(512, 2) k_sample(TopkArgs A) {
  chain_wait();
  __shared__ uint32_t s_warp[33];
  __shared__ uint32_t s_res[2];
  __shared__ uint32_t s_cnt;
  __shared__ uint32_t s_last;
  __shared__ uint32_t sh[NBINS];
  __shared__ uint32_t sl[SLIST];
  if (aborted(A)) return;
  const int2 me = A.smap[blockIdx.x];
  const int t = me.x;
  const int cta = me.y;
  const int nctas = (int)(A.sblk[t + 1] - A.sblk[t]);
  TensorState* st = A.ts + t;
  if (st->flags & TS_NOEMIT) return;
  const int64_t base = A.off[t], n = A.off[t + 1] - base;
  const int64_t k = A.kk[t];
  if (k >= n) return;  // t_est set by the planner
  // threshold mode: never below the threshold's own key
  const uint32_t floor_key = A.tau ? mag_key(A.tau[t]) : 0u;
  const uint4 plan = *reinterpret_cast<const uint4*>(&st->s_runs);  // runs, stride, j, rp
  const int runs = (int)plan.x;
  const int64_t stride = plan.y, j = plan.z;
  const int64_t m = min((int64_t)runs * RUN, n);
  const float gmul = st->gmul;
  if (j > m) {
    if (threadIdx.x == 0 && cta == 0) st->t_est = floor_key;
    return;
  }
  const unsigned lane = lane_id();
  const bool vec = (base & 3) == 0;
  const int nwarp = blockDim.x >> 5, w = threadIdx.x >> 5;
  constexpr int SR = sample_runs_in_flight<MODE>();
  uint32_t key[SR][4];
  unsigned okm[SR];
  uint32_t b1 = 0xFFFFFFFFu, above = 0u, lvl2_n = 0u;
  const uint32_t* lvl2 = nullptr;  // keys for level 2 (shared list or sample buffer)
  bool have_b1 = false, lvl2_shared = false;
  uint32_t* sk = A.skey + A.soff[t];

  for (int i = threadIdx.x; i < NBINS; i += blockDim.x) sh[i] = 0u;
  if (threadIdx.x == 0) s_cnt = 0u;
  __syncthreads();
  if (nctas > 1) {
    // Several CTAs: each filters its share of the runs into the tensor's list
    // in the sample key buffer (room for the whole sample) and the tensor's
    // global histogram row; the last CTA to finish finds the threshold and
    // clears the row (the streaming pass reuses it).
    const uint32_t F = sample_pilot_floor<MODE>(A, t, base, n, stride, runs, plan.w, vec, gmul, sh, sl, s_warp,
                                                s_res);
    const int r_lo = (int)((int64_t)runs * cta / nctas), r_hi = (int)((int64_t)runs * (cta + 1) / nctas);
    sample_filter_pass<MODE>(A, t, base, n, stride, r_lo, r_hi, vec, gmul, F, sh, sk, (uint32_t)m,
                             A.scnt + 2 * t);
    __syncthreads();
    uint32_t* row = A.hist + (size_t)t * NBINS;
    for (int i = threadIdx.x; i < NBINS; i += blockDim.x)
      if (sh[i]) atomicAdd(row + i, sh[i]);
    __threadfence();  // every thread's list entries and histogram counts before the CTA's count
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(A.scnt + 2 * t + 1, 1u) == (uint32_t)(nctas - 1) ? 1u : 0u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const uint32_t c = __ldcg(A.scnt + 2 * t);
    for (int i = threadIdx.x; i < NBINS; i += blockDim.x) {
      sh[i] = __ldcg(row + i);
      row[i] = 0u;
    }
    __syncthreads();
    if (c >= (uint32_t)j) {
      have_b1 = true;
      lvl2 = sk;
      lvl2_n = c;
      b1 = find_bucket(sh, (uint32_t)j, &above, s_warp, s_res);
    }
    for (int i = threadIdx.x; i < NBINS; i += blockDim.x) sh[i] = 0u;
    __syncthreads();
  } else if (runs >= SFILTER_RUNS) {
    // One CTA, filtered search with the list in shared memory.
    const uint32_t F = sample_pilot_floor<MODE>(A, t, base, n, stride, runs, plan.w, vec, gmul, sh, sl, s_warp,
                                                s_res);
    sample_filter_pass<MODE>(A, t, base, n, stride, 0, runs, vec, gmul, F, sh, sl, (uint32_t)SLIST, &s_cnt);
    __syncthreads();
    const uint32_t c = s_cnt;
    if (c >= (uint32_t)j && c <= (uint32_t)SLIST) {
      have_b1 = true;
      lvl2_shared = true;
      lvl2 = sl;
      lvl2_n = c;
      b1 = find_bucket(sh, (uint32_t)j, &above, s_warp, s_res);
    }
    for (int i = threadIdx.x; i < NBINS; i += blockDim.x) sh[i] = 0u;
    __syncthreads();
  }
  if (!have_b1) {
    // direct path: level 1 over every sample key, keys kept in the sample buffer
    for (int r0 = w; r0 < runs; r0 += SR * nwarp) {
      sample_keys<MODE, SR>(A, t, base, n, stride, r0, nwarp, runs, 1, vec, gmul, lane, key, okm);
#pragma unroll
      for (int h = 0; h < SR; ++h) {
        const int64_t r = r0 + h * nwarp;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if ((okm[h] >> c) & 1u) {
            sk[r * RUN + 4 * lane + c] = key[h][c];
            atomicAdd(sh + (key[h][c] >> 21), 1u);
          }
        }
      }
    }
    __syncthreads();
    b1 = find_bucket(sh, (uint32_t)j, &above, s_warp, s_res);
    for (int i = threadIdx.x; i < NBINS; i += blockDim.x) sh[i] = 0u;
    __syncthreads();
    lvl2 = sk;
    lvl2_n = (uint32_t)m;
  }
  if (b1 == 0xFFFFFFFFu) {
    if (threadIdx.x == 0) {
      atomicOr(A.diag + DIAG_ERR, GC_DIAG_SELECT);
      st->t_est = floor_key;
    }
    return;
  }
  const uint32_t rank2 = (uint32_t)j - above;
  constexpr int U8 = 16;
  for (uint32_t i0 = 0; i0 < lvl2_n; i0 += blockDim.x * U8) {
    uint32_t kk[U8];
#pragma unroll
    for (int u = 0; u < U8; ++u) {
      const uint32_t i = i0 + u * blockDim.x + threadIdx.x;
      kk[u] = i < lvl2_n ? (lvl2_shared ? lvl2[i] : __ldcg(lvl2 + i)) : 0u;
    }
#pragma unroll
    for (int u = 0; u < U8; ++u) {
      const uint32_t i = i0 + u * blockDim.x + threadIdx.x;
      smem_hist_add(sh, (kk[u] >> 10) & 0x7FFu, i < lvl2_n && (kk[u] >> 21) == b1);
    }
  }
  __syncthreads();
  uint32_t above2;
  const uint32_t b2 = find_bucket(sh, rank2, &above2, s_warp, s_res);
  if (threadIdx.x == 0) {
    if (b2 == 0xFFFFFFFFu) {
      atomicOr(A.diag + DIAG_ERR, GC_DIAG_SELECT);
      st->t_est = max(b1 << 21, floor_key);
    } else {
      st->t_est = max((b1 << 21) | (b2 << 10), floor_key);
    }
  }
}

// One radix level of the k-th key search for tensor t, run by one CTA of 256
// threads: the histogram is read from `hrow` (the tensor's global row, or a
// copy of it in shared memory) and the global row is cleared for the next
// level.
__device__ void select_level(const TopkArgs& A, int t, int phase, const uint32_t* hrow, uint32_t* s_warp,
                             uint32_t* s_res) {
  TensorState* st = A.ts + t;
  const uint32_t flags = st->flags;
  if (flags & TS_NOEMIT) {
    if (phase == PH_C1 && A.rd && threadIdx.x == 0) A.rd[t] = gc_residual_desc{0u, 0u, 0, 0.0f, 0ull, 0ull};
    return;
  }
  uint32_t* row = A.hist + (size_t)t * NBINS;
  uint32_t rank = st->rank;

  if (phase == PH_C1) {
    const int64_t cap = A.cand_off[t + 1] - A.cand_off[t];
    const int64_t cnt = st->cand_count;
    const bool ovf = (flags & TS_OVERFLOW) || cnt > cap;
    int64_t kt = A.kk[t];
    bool force_dense = false;
    if (A.tau) {
      // threshold mode: candidates are the elements with key >= t_est >= key(tau).
      // Enough of them (>= k_t): keep the k_t largest.  Fewer, and t_est is
      // key(tau) itself: keep them all.  Fewer otherwise (or overflow): the
      // full-pass path counts |acc| >= tau exactly and decides there.
      const uint32_t tkey = mag_key(A.tau[t]);
      if (!ovf && cnt < kt) {
        if (st->t_est == tkey)
          kt = cnt;
        else
          force_dense = true;
      }
      if (!force_dense && !ovf) {
        if (threadIdx.x == 0) {
          st->keff = (uint32_t)kt;
          A.count_out[t] = kt;
          if (kt == 0) {
            st->flags = flags | TS_NOEMIT;
            if (A.int8) A.scale[t] = 0.0f;
            if (A.rd) A.rd[t] = gc_residual_desc{0u, 0u, 0, 0.0f, 0ull, 0ull};
          }
        }
        if (kt == 0) {
          for (int i = threadIdx.x; i < NBINS; i += blockDim.x) row[i] = 0u;
          return;
        }
      }
    }
    const bool dense = ovf || force_dense || cnt < kt || (A.flags & GC_FORCE_EXACT);
    if (dense) {
      for (int i = threadIdx.x; i < NBINS; i += blockDim.x) row[i] = 0u;
      if (threadIdx.x == 0) {
        st->flags = flags | TS_DENSE;
        st->maxkey = 0u;
        st->prefix = 0u;
        st->rank = (uint32_t)kt;
        atomicAdd(A.diag + DIAG_EXACT, 1u);
        if ((flags & TS_OVERFLOW) || cnt > cap) atomicAdd(A.diag + DIAG_OVF, 1u);
      }
      return;
    }
    rank = (uint32_t)kt;
  } else if (phase == PH_C1D) {
    if (!(flags & TS_DENSE)) return;
    if (A.tau) {
      const uint32_t kt = min(st->cnt_tau, (uint32_t)A.kk[t]);
      if (threadIdx.x == 0) {
        st->keff = kt;
        A.count_out[t] = kt;
        if (kt == 0) {
          st->flags = flags | TS_NOEMIT;
          if (A.int8) A.scale[t] = 0.0f;
        }
      }
      if (kt == 0) {
        for (int i = threadIdx.x; i < NBINS; i += blockDim.x) row[i] = 0u;
        return;
      }
      rank = kt;
    } else {
      rank = st->keff;
    }
  }

  uint32_t above;
  const uint32_t b = find_bucket(hrow, rank, &above, s_warp, s_res);
  for (int i = threadIdx.x; i < NBINS; i += blockDim.x) row[i] = 0u;
  if (threadIdx.x != 0) return;
  if (b == 0xFFFFFFFFu) {
    atomicOr(A.diag + DIAG_ERR, GC_DIAG_SELECT);
    st->flags = flags | TS_NOEMIT;  // never write a wrong payload
    return;
  }
  rank -= above;
  switch (phase) {
    case PH_C1:
    case PH_C1D:
      st->prefix = b;
      st->rank = rank;
      break;
    case PH_C2:
      st->prefix = (st->prefix << 11) | b;
      st->rank = rank;
      break;
    case PH_C3: {
      st->thr = (st->prefix << 10) | b;
      st->r_eq = rank;
      st->rank = rank;
      float sc = 0.0f;
      if (A.int8) {
        sc = __fdiv_rn(key_magnitude(st->maxkey), 127.0f);
        A.scale[t] = sc;
      }
      // last_tie is filled in by the payload write
      if (A.rd) A.rd[t] = gc_residual_desc{1u | (A.int8 ? 2u : 0u), st->thr, -1, sc, A.seed, iter_of(A)};
      break;
    }
  }
}

// One radix level of the k-th key search for every tensor (one CTA each).
__global__ void __launch_bounds__(256) k_select(TopkArgs A, int phase) {
  chain_wait();
  __shared__ uint32_t s_warp[33];
  __shared__ uint32_t s_res[3];
  if (aborted(A)) return;
  select_level(A, blockIdx.x, phase, A.hist + (size_t)blockIdx.x * NBINS, s_warp, s_res);
}


// ============================================================================ streaming pass

// Appends this lane's flagged entries (bit j of m -> entry j) to the warp's
// shared-memory chunk, in (lane, j) order, i.e. index order.
__device__ __forceinline__ void warp_append(float* sval, uint32_t* skey, uint16_t* spos, int& cnt,
                                            bool& ovf, unsigned m, const uint32_t* key,
                                            const float* val, int pos0, unsigned lane) {
  unsigned pre, tot;
  warp_count_scan(__popc(m), lane, &pre, &tot);
  if (ovf || cnt + (int)tot > WCAP) {
    ovf = true;
    return;
  }
  int o = cnt + (int)pre;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if ((m >> j) & 1u) {
      sval[o] = val[j];
      skey[o] = key[j];
      spos[o] = (uint16_t)(pos0 + j);
      ++o;
    }
  }
  cnt += (int)tot;
}

template <int MODE, bool EF, bool LOADG, bool LAZY>
__device__ __forceinline__ void stream_scalar(const TopkArgs& A, int64_t li, int64_t gi,
                                              const gc_residual_desc& d, float gmul, float* value,
                                              uint32_t* key) {
  float x = 0.0f;
  if (MODE == MODE_MOM) {
    const float un = __fadd_rn(__fmul_rn(A.beta, A.u[gi]), A.g[gi]);
    x = __fadd_rn(A.v[gi], un);
    A.u[gi] = un;
    A.v[gi] = x;
  } else if (LOADG) {
    x = __fmul_rn(gmul, A.g[gi]);
    if (EF) {
      x = __fadd_rn(x, LAZY ? lazy_fix(A.e[gi], li, gi, d) : A.e[gi]);
      A.e[gi] = x;
    }
  }
  *value = x;
  *key = (MODE == MODE_RANDK) ? ~philox_word(A.pk, iter_of(A), (uint64_t)gi, PURPOSE_RANDK)
                              : mag_key(x);
}

constexpr int STREAM_THREADS = 256;
constexpr int STREAM_WARPS = STREAM_THREADS / 32;
// Loads in flight per lane and resident blocks per SM of the streaming pass
// (compile-time; defaults measured best on the Llama-3-8B arena).
#ifndef GC_STREAM_UNROLL
#define GC_STREAM_UNROLL 2
#endif
#ifndef GC_STREAM_MINB
#define GC_STREAM_MINB 4
#endif
// Loads in flight per lane: eager Top-k GC_STREAM_UNROLL; the other modes
// and the lazy-residual pass (more registers per element) 4.
template <int MODE, bool LAZY>
constexpr int stream_unroll() { return (MODE == 0 && !LAZY) ? GC_STREAM_UNROLL : 4; }
constexpr size_t STREAM_SMEM = (size_t)STREAM_WARPS * WCAP * (4 + 4 + 2);

template <int MODE, bool EF, bool LOADG, bool LAZY>
__global__ void __launch_bounds__(STREAM_THREADS, MODE == MODE_TOPK ? (LAZY ? 3 : GC_STREAM_MINB) : 2) k_stream(TopkArgs A) {
  chain_wait();
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const unsigned lane = lane_id();
  float* sval = reinterpret_cast<float*>(smem) + warp * WCAP;
  uint32_t* skey = reinterpret_cast<uint32_t*>(smem + (size_t)STREAM_WARPS * WCAP * 4) + warp * WCAP;
  uint16_t* spos = reinterpret_cast<uint16_t*>(smem + (size_t)STREAM_WARPS * WCAP * 8) + warp * WCAP;
  if (aborted(A)) return;
  const uint64_t iter = iter_of(A);
  const int64_t nwarps = (int64_t)gridDim.x * STREAM_WARPS;
  int pushed_t = -1;        // tensor of the last maximum this warp pushed
  uint32_t pushed_max = 0u;  // and that maximum
  for (int64_t u = (int64_t)blockIdx.x * STREAM_WARPS + warp; u < A.U; u += nwarps) {
    const int t = find_segment(A.units_off, A.T, u);
    const int64_t base = A.off[t];
    const int64_t n = A.off[t + 1] - base;
    const int64_t lstart = (u - A.units_off[t]) << UNIT_SHIFT;
    const int len = (int)min((int64_t)UNIT, n - lstart);
    const int64_t g0 = base + lstart;
    const bool emit = !(A.ts[t].flags & TS_NOEMIT);
    const uint32_t test = A.ts[t].t_est;
    gc_residual_desc d;
    if (LAZY) d = A.rd[t];
    const float gmul = A.ts[t].gmul;
    int cnt = 0;
    bool ovf = false;
    if ((g0 & 3) == 0) {
      const int nv = len >> 2;
      const float4* g4 = reinterpret_cast<const float4*>(A.g + g0);
      float4* e4 = reinterpret_cast<float4*>(A.e + g0);
      float4* u4 = reinterpret_cast<float4*>(A.u + g0);
      float4* v4 = reinterpret_cast<float4*>(A.v + g0);
      constexpr int SU = stream_unroll<MODE, LAZY>();
      for (int v0 = 0; v0 < nv; v0 += 32 * SU) {
        float4 x[SU], y[SU], z[SU];
#pragma unroll
        for (int j = 0; j < SU; ++j) {
          const int vi = v0 + j * 32 + (int)lane;
          if (vi < nv) {
            if (LOADG || MODE == MODE_MOM) x[j] = ld_stream(g4 + vi);
            if (MODE == MODE_MOM) {
              y[j] = ld_stream(u4 + vi);
              z[j] = ld_stream(v4 + vi);
            } else if (EF) {
              y[j] = ld_stream(e4 + vi);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < SU; ++j) {
          const int vi = v0 + j * 32 + (int)lane;
          const bool valid = vi < nv;
          float a[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t kk[4];
          if (valid) {
            if (MODE == MODE_MOM) {
              float4 un, vn;
              un.x = __fadd_rn(__fmul_rn(A.beta, y[j].x), x[j].x);
              un.y = __fadd_rn(__fmul_rn(A.beta, y[j].y), x[j].y);
              un.z = __fadd_rn(__fmul_rn(A.beta, y[j].z), x[j].z);
              un.w = __fadd_rn(__fmul_rn(A.beta, y[j].w), x[j].w);
              vn.x = __fadd_rn(z[j].x, un.x);
              vn.y = __fadd_rn(z[j].y, un.y);
              vn.z = __fadd_rn(z[j].z, un.z);
              vn.w = __fadd_rn(z[j].w, un.w);
              st_stream(u4 + vi, un);
              st_stream(v4 + vi, vn);
              a[0] = vn.x; a[1] = vn.y; a[2] = vn.z; a[3] = vn.w;
            } else if (LOADG) {
              float4 s = x[j];
              s.x = __fmul_rn(gmul, s.x);
              s.y = __fmul_rn(gmul, s.y);
              s.z = __fmul_rn(gmul, s.z);
              s.w = __fmul_rn(gmul, s.w);
              if (EF) {
                if (LAZY) {
                  const int64_t li0 = lstart + 4 * vi;
                  const bool k0 = lazy_kept(y[j].x, li0 + 0, d), k1 = lazy_kept(y[j].y, li0 + 1, d);
                  const bool k2 = lazy_kept(y[j].z, li0 + 2, d), k3 = lazy_kept(y[j].w, li0 + 3, d);
                  if (k0 | k1 | k2 | k3) {
                    const int64_t gq = g0 + 4 * vi;
                    if (k0) y[j].x = lazy_kept_residual(y[j].x, gq + 0, d);
                    if (k1) y[j].y = lazy_kept_residual(y[j].y, gq + 1, d);
                    if (k2) y[j].z = lazy_kept_residual(y[j].z, gq + 2, d);
                    if (k3) y[j].w = lazy_kept_residual(y[j].w, gq + 3, d);
                  }
                }
                s.x = __fadd_rn(s.x, y[j].x);
                s.y = __fadd_rn(s.y, y[j].y);
                s.z = __fadd_rn(s.z, y[j].z);
                s.w = __fadd_rn(s.w, y[j].w);
                st_stream(e4 + vi, s);
              }
              a[0] = s.x; a[1] = s.y; a[2] = s.z; a[3] = s.w;
            }
          }
          unsigned m = 0u;
          if (MODE == MODE_RANDK) {
            const uint4 w = philox_block(A.pk, iter, (uint64_t)(g0 >> 2) + (uint64_t)vi, PURPOSE_RANDK);
            kk[0] = ~w.x; kk[1] = ~w.y; kk[2] = ~w.z; kk[3] = ~w.w;
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) kk[c] = mag_key(a[c]);
          }
          if (valid && emit) {
#pragma unroll
            for (int c = 0; c < 4; ++c) m |= (kk[c] >= test ? 1u : 0u) << c;
          }
          if (__any_sync(FULL, m != 0u))
            warp_append(sval, skey, spos, cnt, ovf, m, kk, a, vi * 4, lane);
        }
      }
      const int rem = len & 3;
      if (rem) {
        const int li = nv * 4 + (int)lane;
        const bool valid = (int)lane < rem;
        float a[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t kk[4] = {0u, 0u, 0u, 0u};
        if (valid) stream_scalar<MODE, EF, LOADG, LAZY>(A, lstart + li, g0 + li, d, gmul, &a[0], &kk[0]);
        const unsigned m = (valid && emit && kk[0] >= test) ? 1u : 0u;
        if (__any_sync(FULL, m != 0u)) warp_append(sval, skey, spos, cnt, ovf, m, kk, a, li, lane);
      }
    } else {
      for (int i0 = 0; i0 < len; i0 += 32) {
        const int li = i0 + (int)lane;
        const bool valid = li < len;
        float a[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t kk[4] = {0u, 0u, 0u, 0u};
        if (valid) stream_scalar<MODE, EF, LOADG, LAZY>(A, lstart + li, g0 + li, d, gmul, &a[0], &kk[0]);
        const unsigned m = (valid && emit && kk[0] >= test) ? 1u : 0u;
        if (__any_sync(FULL, m != 0u)) warp_append(sval, skey, spos, cnt, ovf, m, kk, a, li, lane);
      }
    }
    // flush the unit's candidates as one chunk
    __syncwarp();
    uint2 ch = make_uint2(0u, 0u);
    if (emit && cnt > 0 && !ovf) {
      uint32_t start = 0u;
      if (lane == 0) start = atomicAdd(&A.ts[t].cand_count, (uint32_t)cnt);
      start = __shfl_sync(FULL, start, 0);
      const int64_t cap = A.cand_off[t + 1] - A.cand_off[t];
      if ((int64_t)start + cnt > cap) {
        ovf = true;
      } else {
        const int64_t cb = A.cand_off[t] + start;
        uint32_t mx = 0u;
        uint32_t* row = A.hist + (size_t)t * NBINS;
        for (int j = (int)lane; j < cnt; j += 32) {
          const uint32_t key = skey[j];
          A.ckey[cb + j] = key;
          A.cidx[cb + j] = (int32_t)(lstart + spos[j]);
          A.cval[cb + j] = sval[j];
          // one atomic per distinct bin of the warp's candidates: the
          // candidates of a tensor crowd into a few bins, and an atomic per
          // candidate on those few addresses held the pass back (0.945 ->
          // 0.980 of the HBM copy peak on the Llama-3-8B arena)
          const unsigned peers = __match_any_sync(__activemask(), key >> 21);
          if ((int)lane == __ffs(peers) - 1) atomicAdd(row + (key >> 21), (uint32_t)__popc(peers));
          mx = max(mx, key);
        }
        mx = warp_max_u32(mx);
        // the tensor's maximum only grows: skip the atomic unless this warp
        // has not yet pushed a key as large for this tensor (one atomic per
        // unit on the tensor's one address cost 0.12 ms on the Llama-3-8B
        // arena; the pending-residual pass keeps it, the two registers made
        // it spill)
        if (LAZY) {
          if (lane == 0) atomicMax(&A.ts[t].maxkey, mx);
        } else {
          if (t != pushed_t) {
            pushed_t = t;
            pushed_max = 0u;
          }
          if (mx > pushed_max) {
            if (lane == 0) atomicMax(&A.ts[t].maxkey, mx);
            pushed_max = mx;
          }
        }
        ch = make_uint2(start, (uint32_t)cnt);
      }
    }
    if (lane == 0) {
      if (emit && ovf) atomicOr(&A.ts[t].flags, TS_OVERFLOW);
      A.chunk[u] = ch;
    }
    __syncwarp();
  }
}

// ============================================================================ unit-block kernels

struct UnitBlock {
  int t;
  int64_t u0;
  int nu;
  int64_t base, n;
};

__device__ __forceinline__ UnitBlock unit_block(const TopkArgs& A) {
  UnitBlock r;
  r.t = find_segment(A.ublk_off, A.T, (int64_t)blockIdx.x);
  r.u0 = A.units_off[r.t] + ((int64_t)blockIdx.x - A.ublk_off[r.t]) * A.ubu;
  const int64_t u1 = min(r.u0 + A.ubu, A.units_off[r.t + 1]);
  r.nu = (int)(u1 - r.u0);
  r.base = A.off[r.t];
  r.n = A.off[r.t + 1] - r.base;
  return r;
}

// Full-pass walk of one unit (tensors selected without candidates): the warp
// takes 128 elements per step, four consecutive per lane, and issues the
// loads of DSTEPS steps before using any.  f(o, key, x, ok) runs on every
// lane for each step in index order: o is the unit-local offset of the
// lane's first element, bit c of ok flags element o + c as inside the unit.
template <int MODE, bool LOADX, int DSTEPS = 4, class F>
__device__ __forceinline__ void dense_unit_walk(const TopkArgs& A, const float* src, int64_t g0, int len,
                                                unsigned lane, F&& f) {
  const bool vec = (g0 & 3) == 0;
  for (int i0 = 0; i0 < len; i0 += 128 * DSTEPS) {
    float x[DSTEPS][4];
#pragma unroll
    for (int st = 0; st < DSTEPS; ++st) {
      const int o = i0 + st * 128 + 4 * (int)lane;
#pragma unroll
      for (int c = 0; c < 4; ++c) x[st][c] = 0.0f;
      if (LOADX) {
        if (vec && o + 4 <= len) {
          const float4 v = __ldcs(reinterpret_cast<const float4*>(src + g0 + o));
          x[st][0] = v.x;
          x[st][1] = v.y;
          x[st][2] = v.z;
          x[st][3] = v.w;
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (o + c < len) x[st][c] = src[g0 + o + c];
        }
      }
    }
#pragma unroll
    for (int st = 0; st < DSTEPS; ++st) {
      const int o = i0 + st * 128 + 4 * (int)lane;
      uint32_t key[4];
      unsigned ok = 0u;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const bool in = o + c < len;
        ok |= (in ? 1u : 0u) << c;
        key[c] = in ? key_of<MODE>(A, x[st][c], g0 + o + c) : 0u;
      }
      f(o, key, x[st], ok);
    }
  }
}

// Histogram level `level` (1, 2, 3) of the keys matching the tensor's
// prefix.  Level 1 runs only for tensors selected by full passes (the
// candidate level-1 histogram comes from the streaming pass).
template <int MODE>
__global__ void __launch_bounds__(256) k_hist(TopkArgs A, int level) {
  chain_wait();
  __shared__ uint32_t sh[NBINS];
  __shared__ uint32_t s_max, s_tau;
  if (aborted(A)) return;
  const UnitBlock ub = unit_block(A);
  const TensorState st = A.ts[ub.t];
  if (st.flags & TS_NOEMIT) return;
  const bool dense = (st.flags & TS_DENSE) != 0u;
  if (level == 1 && !dense) return;
  for (int i = threadIdx.x; i < NBINS; i += blockDim.x) sh[i] = 0u;
  if (threadIdx.x == 0) {
    s_max = 0u;
    s_tau = 0u;
  }
  __syncthreads();
  // threshold mode, full-pass level 1: also count |acc| >= tau exactly
  const bool count_tau = level == 1 && A.tau != nullptr;
  const uint32_t tkey = count_tau ? mag_key(A.tau[ub.t]) : 0u;
  const int shift_prev = (level == 2) ? 21 : 10;
  const uint32_t mask = (level == 3) ? 0x3FFu : 0x7FFu;
  const int shift = (level == 1) ? 21 : ((level == 2) ? 10 : 0);
  if (dense) {
    const unsigned lane = lane_id();
    const float* src = value_source<MODE>(A);
    uint32_t mx = 0u;
    for (int ui = threadIdx.x >> 5; ui < ub.nu; ui += blockDim.x >> 5) {
      const int64_t lstart = (ub.u0 + ui - A.units_off[ub.t]) << UNIT_SHIFT;
      const int len = (int)min((int64_t)UNIT, ub.n - lstart);
      dense_unit_walk<MODE, MODE != MODE_RANDK>(
          A, src, ub.base + lstart, len, lane, [&](int, const uint32_t* key, const float*, unsigned ok) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const bool valid = (ok >> c) & 1u;
              const bool hit = valid && (level == 1 || (key[c] >> shift_prev) == st.prefix);
              if (valid) mx = max(mx, key[c]);
              if (count_tau) {
                const unsigned cnt = __popc(__ballot_sync(FULL, valid && key[c] >= tkey));
                if (lane == 0 && cnt) atomicAdd(&s_tau, cnt);
              }
              smem_hist_add(sh, (key[c] >> shift) & mask, hit);
            }
          });
    }
    if (level == 1) {
      mx = warp_max_u32(mx);
      if (lane == 0) atomicMax(&s_max, mx);
    }
  } else {
    // this CTA's slice of the tensor's candidate keys (order is irrelevant here)
    const int64_t nb = A.ublk_off[ub.t + 1] - A.ublk_off[ub.t];
    const int64_t bi = (int64_t)blockIdx.x - A.ublk_off[ub.t];
    const int64_t cnt = st.cand_count;
    const int64_t lo = cnt * bi / nb, hi = cnt * (bi + 1) / nb;
    const uint32_t* ck = A.ckey + A.cand_off[ub.t];
    constexpr int U8 = 8;
    for (int64_t i0 = lo; i0 < hi; i0 += (int64_t)blockDim.x * U8) {
      uint32_t kk[U8];
#pragma unroll
      for (int u = 0; u < U8; ++u) {
        const int64_t i = i0 + (int64_t)u * blockDim.x + threadIdx.x;
        kk[u] = i < hi ? __ldcs(ck + i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < U8; ++u) {
        const int64_t i = i0 + (int64_t)u * blockDim.x + threadIdx.x;
        if (i < hi && (kk[u] >> shift_prev) == st.prefix) atomicAdd(sh + ((kk[u] >> shift) & mask), 1u);
      }
    }
  }
  __syncthreads();
  uint32_t* row = A.hist + (size_t)ub.t * NBINS;
  for (int i = threadIdx.x; i < NBINS; i += blockDim.x)
    if (sh[i]) atomicAdd(row + i, sh[i]);
  if (level == 1 && threadIdx.x == 0) {
    atomicMax(&A.ts[ub.t].maxkey, s_max);
    if (count_tau && s_tau) atomicAdd(&A.ts[ub.t].cnt_tau, s_tau);
  }
}

// The candidate chunks of a warp's units are walked as one concatenated
// sequence, 32 entries per step with one entry per lane, so that loads are
// contiguous and no lane idles on a short chunk.  `off` is this lane's
// exclusive prefix of the chunk lengths; returns the lane whose chunk holds
// entry e (e below the total): the last lane with off <= e, which skips
// empty chunks.
__device__ __forceinline__ int chunk_owner(uint32_t off, uint32_t e) {
  int o = 0;
#pragma unroll
  for (int b = 16; b >= 1; b >>= 1)
    if (__shfl_sync(FULL, off, o + b) <= e) o += b;
  return o;
}

// Term of the kept-set reduction for one kept magnitude (the key holds |x|
// exactly): x^2 for the QSGD norm, |x| for the sign scale.  Both are exact
// in fp64.
__device__ __forceinline__ double kept_term(int qkind, uint32_t key) {
  const double m = (double)key_magnitude(key);
  return qkind == KQ_QSGD ? m * m : m;
}

// Sum of one fp64 value per thread over the CTA in a fixed order (a shuffle
// tree per warp, then the warps in index order), so that the result does
// not depend on timing.  Valid in thread 0.
__device__ double block_sum_f64(double v, double* s_d) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(FULL, v, d);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (lane_id() == 0) s_d[w] = v;
  __syncthreads();
  double r = 0.0;
  if (threadIdx.x == 0)
    for (int i = 0; i < nw; ++i) r += s_d[i];
  return r;
}

// Exclusive scan of the unit-block sums of each tensor (one CTA each).  Doing
// it in the last CTA of each tensor in k_count instead (one launch fewer)
// measured slower on the Llama-3-8B arena: 64.7 against 46.5 + 5.3 us.
// For QSGD / sign of the kept values it also sets the tensor's scale: the
// unit blocks' sums in a fixed order plus the kept ties, then
// N = (float)sqrt(sum x^2) or mu = (float)(sum |x| / k).
__global__ void __launch_bounds__(256) k_scan(TopkArgs A) {
  chain_wait();
  __shared__ uint32_t s_warp[33];
  __shared__ double s_d[32];
  if (aborted(A)) return;
  const int t = blockIdx.x;
  const int64_t b0 = A.ublk_off[t], b1 = A.ublk_off[t + 1];
  uint32_t carry_g = 0u, carry_e = 0u;
  for (int64_t c = b0; c < b1; c += blockDim.x) {
    const int64_t b = c + threadIdx.x;
    const uint32_t g = b < b1 ? A.bgt[b] : 0u;
    const uint32_t e = b < b1 ? A.beq[b] : 0u;
    uint32_t pg, tg, pe, te;
    block_scan_u32(g, s_warp, &pg, &tg);
    block_scan_u32(e, s_warp, &pe, &te);
    if (b < b1) {
      A.bgt[b] = carry_g + pg;
      A.beq[b] = carry_e + pe;
    }
    carry_g += tg;
    carry_e += te;
  }
  if (A.qkind != KQ_NONE) {
    double part = 0.0;
    for (int64_t b = b0 + threadIdx.x; b < b1; b += blockDim.x) part += A.upart[b];
    const double tot = block_sum_f64(part, s_d);
    if (threadIdx.x == 0) {
      const TensorState st = A.ts[t];
      if (!(st.flags & TS_NOEMIT)) {
        const double sum = tot + (double)st.r_eq * kept_term(A.qkind, st.thr);
        A.scale[t] = A.qkind == KQ_QSGD ? __double2float_rn(sqrt(sum))
                                        : __double2float_rn(sum / (double)st.keff);
      }
    }
  }
}

// Per-unit counts of keys above / equal to the k-th key, and their sums
// per unit block.  For QSGD / sign of the kept values, also each unit
// block's fp64 sum of x^2 or |x| over its elements above the k-th key (the
// kept ties, all of magnitude |k-th key|, are added per tensor by k_scan).
template <int MODE, bool KSUM>
__global__ void __launch_bounds__(256) k_count(TopkArgs A) {
  chain_wait();
  __shared__ uint32_t s_gt[UB_UNITS], s_eq[UB_UNITS];
  __shared__ uint32_t s_warp[33];
  __shared__ double s_d[32];
  if (aborted(A)) return;
  const UnitBlock ub = unit_block(A);
  const TensorState st = A.ts[ub.t];
  const int tid = threadIdx.x;
  constexpr bool kq = KSUM;  // QSGD / sign of the kept values (A.qkind != KQ_NONE)
  double ksum = 0.0;
  s_gt[tid] = 0u;
  s_eq[tid] = 0u;
  __syncthreads();
  if (!(st.flags & TS_NOEMIT)) {
    if (st.flags & TS_DENSE) {
      const unsigned lane = lane_id();
      const float* src = value_source<MODE>(A);
      for (int ui = tid >> 5; ui < ub.nu; ui += blockDim.x >> 5) {
        const int64_t lstart = (ub.u0 + ui - A.units_off[ub.t]) << UNIT_SHIFT;
        const int len = (int)min((int64_t)UNIT, ub.n - lstart);
        uint32_t gt = 0u, eq = 0u;
        dense_unit_walk<MODE, MODE != MODE_RANDK>(
            A, src, ub.base + lstart, len, lane, [&](int, const uint32_t* key, const float*, unsigned ok) {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const bool valid = (ok >> c) & 1u;
                gt += (valid && key[c] > st.thr) ? 1u : 0u;
                eq += (valid && key[c] == st.thr) ? 1u : 0u;
                if (kq && valid && key[c] > st.thr) ksum += kept_term(A.qkind, key[c]);
              }
            });
        gt = __reduce_add_sync(FULL, gt);
        eq = __reduce_add_sync(FULL, eq);
        if (lane == 0) {
          s_gt[ui] = gt;
          s_eq[ui] = eq;
        }
      }
    } else {
      // The warp's chunks (32 or 8 units) walked as one sequence, 32 entries per step
      // (see chunk_owner and k_write): loads contiguous across the lanes,
      // CP steps' loads in flight and the next CP steps' issued before these
      // are counted; a unit's counts are the differences of
      // the running counts at its chunk's start and at the next chunk's.  A
      // thread per unit issued a separate sector request per lane for every
      // load (25 us on ResNet-50 at 1%, the largest unit blocks the long pole).
      const unsigned lane = lane_id();
      const int wu = A.ubu >> 3;  // units per warp; lanes >= wu own empty chunks
      const int ui = (tid >> 5) * wu + (int)lane;
      const bool own = (int)lane < wu && ui < ub.nu;
      const uint2 ch = own ? A.chunk[ub.u0 + ui] : make_uint2(0u, 0u);
      const uint32_t* ckb = A.ckey + A.cand_off[ub.t];
      unsigned L;
      const uint32_t off = warp_excl_scan(ch.y, lane, &L);
      uint32_t Gc = 0u, Ec = 0u, gs = 0u, es = 0u;
      constexpr int CP = 4;
      uint32_t pk[CP], nk[CP];
      auto load_group = [&](uint32_t wg, uint32_t* gk) {
#pragma unroll
        for (int p = 0; p < CP; ++p) {
          const uint32_t e = wg + 32u * p + lane;
          const int o = chunk_owner(off, e);
          const uint32_t off_o = __shfl_sync(FULL, off, o), chx_o = __shfl_sync(FULL, ch.x, o);
          gk[p] = e < L ? __ldcs(ckb + chx_o + (e - off_o)) : 0u;
        }
      };
      if (L > 0u) load_group(0u, nk);
      for (uint32_t wg = 0; wg < L; wg += 32u * CP) {
#pragma unroll
        for (int p = 0; p < CP; ++p) pk[p] = nk[p];
        if (wg + 32u * CP < L) load_group(wg + 32u * CP, nk);  // the next group's loads first
#pragma unroll
        for (int p = 0; p < CP; ++p) {
          const uint32_t ws = wg + 32u * p;
          if (ws >= L) break;
          const bool act = ws + lane < L;
          const bool isgt = act && pk[p] > st.thr, iseq = act && pk[p] == st.thr;
          const unsigned gm = __ballot_sync(FULL, isgt), em = __ballot_sync(FULL, iseq);
          if (kq && isgt) ksum += kept_term(A.qkind, pk[p]);
          if (off - ws < 32u) {
            const unsigned below = (1u << (off - ws)) - 1u;
            gs = Gc + __popc(gm & below);
            es = Ec + __popc(em & below);
          }
          Gc += __popc(gm);
          Ec += __popc(em);
        }
      }
      if (off >= L) {  // empty chunks after the last entry
        gs = Gc;
        es = Ec;
      }
      const uint32_t gn = __shfl_down_sync(FULL, gs, 1), en = __shfl_down_sync(FULL, es, 1);
      if (own) {
        s_gt[ui] = (lane == 31 ? Gc : gn) - gs;
        s_eq[ui] = (lane == 31 ? Ec : en) - es;
      }
    }
  }
  __syncthreads();
  const uint32_t gt = s_gt[tid], eq = s_eq[tid];
  if (tid < ub.nu) {
    A.ugt[ub.u0 + tid] = gt;
    A.ueq[ub.u0 + tid] = eq;
  }
  uint32_t pre, tg, te;
  block_scan_u32(gt, s_warp, &pre, &tg);
  block_scan_u32(eq, s_warp, &pre, &te);
  if (tid == 0) {
    A.bgt[blockIdx.x] = tg;
    A.beq[blockIdx.x] = te;
  }
  if (kq) {
    const double r = block_sum_f64(ksum, s_d);
    if (tid == 0) A.upart[blockIdx.x] = r;
  }
}

// Writes one kept element: payload slot `pos` (absolute), residual.
template <int MODE, int KQ>
__device__ __forceinline__ void emit_kept(const TopkArgs& A, int t, int64_t base, int64_t n,
                                          int64_t li, float x, int64_t pos, float s, bool last_tie) {
  if (A.rd && last_tie) A.rd[t].last_tie = (int32_t)li;
  if (pos >= A.koff[t + 1]) {  // only reachable if the selection were inconsistent
    atomicOr(A.diag + DIAG_ERR, GC_DIAG_SELECT);
    return;
  }
  const int64_t gi = base + li;
  A.idx[pos] = (int32_t)li;
  if (MODE == MODE_RANDK) {
    if (A.unbiased) {
      const float c = __double2float_rn((double)n / (double)A.kk[t]);
      A.val[pos] = __fmul_rn(A.g[gi], c);
    } else {
      A.val[pos] = x;
      if (A.ef) A.e[gi] = 0.0f;
    }
    return;
  }
  float* res = (MODE == MODE_MOM) ? A.v : ((A.ef && !A.rd) ? A.e : nullptr);
  if (KQ == KQ_QSGD) {
    // s = N: level = min(L, SR((|x| L) / N)), decoded sgn ((level N) / L)
    const float L = (float)A.slev;
    int level = 0;
    if (s != 0.0f) {
      // (|x| L) / N <= L because |x| <= N; the clamp (which cannot change
      // min(L, .)) only guards the float -> int conversion
      const float y = fminf(__fdiv_rn(__fmul_rn(fabsf(x), L), s), L + 1.0f);
      level = min(A.slev, stochastic_round(y, philox_word(A.pk, iter_of(A), (uint64_t)gi, PURPOSE_QSGD)));
    }
    const bool neg = signbit(x);
    const float mag = __fdiv_rn(__fmul_rn((float)level, s), L);
    const float d = neg ? -mag : mag;
    A.q[pos] = (int8_t)(neg ? -level : level);
    if (A.val) A.val[pos] = d;
    if (res) res[gi] = __fsub_rn(x, d);
  } else if (KQ == KQ_SIGN) {
    // s = mu: bit j of the tensor's words = sign bit of x clear; decoded +-mu
    const bool neg = signbit(x);
    const int64_t j = pos - A.koff[t];
    if (!neg) atomicOr(A.bits + A.kwoff[t] + (j >> 5), 1u << (j & 31));
    const float d = neg ? -s : s;
    if (A.val) A.val[pos] = d;
    if (res) res[gi] = __fsub_rn(x, d);
  } else if (A.int8) {
    const int c = int8_code(x, s, philox_word(A.pk, iter_of(A), (uint64_t)gi, PURPOSE_INT8));
    const float d = __fmul_rn((float)c, s);
    A.q[pos] = (int8_t)c;
    if (A.val) A.val[pos] = d;
    if (res) res[gi] = __fsub_rn(x, d);
  } else {
    A.val[pos] = x;
    if (res) res[gi] = 0.0f;
  }
  if (MODE == MODE_MOM && A.masking) A.u[gi] = 0.0f;
}

template <int MODE, int KQ>
__global__ void __launch_bounds__(256, 3) k_write(TopkArgs A) {
  chain_wait();
  __shared__ uint32_t s_gt[UB_UNITS], s_eq[UB_UNITS];
  __shared__ uint32_t s_warp[33];
  if (aborted(A)) return;
  const UnitBlock ub = unit_block(A);
  const TensorState st = A.ts[ub.t];
  if (st.flags & TS_NOEMIT) return;
  const int tid = threadIdx.x;
  const uint32_t gt = tid < ub.nu ? A.ugt[ub.u0 + tid] : 0u;
  const uint32_t eq = tid < ub.nu ? A.ueq[ub.u0 + tid] : 0u;
  uint32_t pg, pe, tg, te;
  block_scan_u32(gt, s_warp, &pg, &tg);
  block_scan_u32(eq, s_warp, &pe, &te);
  s_gt[tid] = A.bgt[blockIdx.x] + pg;
  s_eq[tid] = A.beq[blockIdx.x] + pe;
  __syncthreads();
  const int64_t kbase = A.koff[ub.t];
  const float s = (A.int8 || KQ != KQ_NONE) ? A.scale[ub.t] : 0.0f;
  const uint32_t thr = st.thr, r_eq = st.r_eq;
  if (st.flags & TS_DENSE) {
    const unsigned lane = lane_id();
    const float* src = value_source<MODE>(A);
    for (int ui = tid >> 5; ui < ub.nu; ui += blockDim.x >> 5) {
      const int64_t lstart = (ub.u0 + ui - A.units_off[ub.t]) << UNIT_SHIFT;
      const int len = (int)min((int64_t)UNIT, ub.n - lstart);
      const uint32_t eqb = s_eq[ui];
      int64_t selpos = (int64_t)s_gt[ui] + min(eqb, r_eq);
      uint32_t eqrun = 0u;  // ties before this step in the unit
      dense_unit_walk<MODE, true, 2>(
          A, src, ub.base + lstart, len, lane, [&](int o, const uint32_t* key, const float* x, unsigned ok) {
            unsigned eqm = 0u, gtm = 0u;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const bool valid = (ok >> c) & 1u;
              eqm |= (valid && key[c] == thr ? 1u : 0u) << c;
              gtm |= (valid && key[c] > thr ? 1u : 0u) << c;
            }
            unsigned epre, etot;
            warp_count_scan(__popc(eqm), lane, &epre, &etot);
            unsigned selm = gtm;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint32_t rank = eqb + eqrun + epre + __popc(eqm & ((1u << c) - 1u));
              if (((eqm >> c) & 1u) && rank < r_eq) selm |= 1u << c;
            }
            unsigned spre, stot;
            warp_count_scan(__popc(selm), lane, &spre, &stot);
            for (unsigned m = selm; m != 0u; m &= m - 1u) {  // one emit site, no unrolling
              const int c = __ffs(m) - 1;
              const unsigned below = (1u << c) - 1u;
              const bool last = ((eqm >> c) & 1u) && eqb + eqrun + epre + __popc(eqm & below) + 1u == r_eq;
              const float xv = c == 0 ? x[0] : (c == 1 ? x[1] : (c == 2 ? x[2] : x[3]));
              emit_kept<MODE, KQ>(A, ub.t, ub.base, ub.n, lstart + o + c, xv, kbase + selpos + spre + __popc(selm & below),
                              s, last);
            }
            selpos += stot;
            eqrun += etot;
          });
    }
  } else {
    // Candidate path: the warp's chunks (32 or 8 units) are walked as one sequence (see
    // chunk_owner), 32 entries per step with loads and stores contiguous
    // across the lanes, and kept and tie counts inside a unit are
    // differences of running counts over the sequence, taken at the unit's
    // first entry.  A thread walking its own unit's chunk (the earlier path
    // for chunks of 40 or more candidates) issues a separate 32-byte sector
    // request per lane for every load and store; at 1% density on ResNet-50
    // that held the largest unit blocks at 35-43 us against 28 us here.
    const unsigned lane = lane_id();
    const unsigned lt = (1u << lane) - 1u;
    const int wu = A.ubu >> 3;  // units per warp; lanes >= wu own empty chunks
    const int ui = (tid >> 5) * wu + (int)lane;
    const bool own = (int)lane < wu && ui < ub.nu;
    const uint2 ch = own ? A.chunk[ub.u0 + ui] : make_uint2(0u, 0u);
    const uint32_t eqb = own ? s_eq[ui] : 0u;                 // ties before this unit
    const uint32_t sel0 = own ? s_gt[ui] + min(eqb, r_eq) : 0u;  // kept before this unit
    unsigned L;
    const uint32_t off = warp_excl_scan(ch.y, lane, &L);
    const int64_t cb = A.cand_off[ub.t];
    uint32_t Kc = 0u, Ec = 0u, ks = 0u, es = 0u;
    // WP steps' loads are issued before any of them is used (the entries'
    // owners and addresses depend only on the chunk table, not on data), and
    // the next WP steps' loads before this group is processed
    constexpr int WP = 4;
    uint32_t pkey[WP], nkey[WP];
    int32_t pli[WP], nli[WP];
    float px[WP], nx[WP];
    int pown[WP], nown[WP];
    auto load_group = [&](uint32_t wg, uint32_t* gk, int32_t* gl, float* gx, int* go) {
#pragma unroll
      for (int p = 0; p < WP; ++p) {
        const uint32_t e = wg + 32u * p + lane;
        const int o = chunk_owner(off, e);
        const uint32_t off_o = __shfl_sync(FULL, off, o), chx_o = __shfl_sync(FULL, ch.x, o);
        go[p] = o;
        gk[p] = 0u;
        gl[p] = 0;
        gx[p] = 0.0f;
        if (e < L) {
          const int64_t c = cb + chx_o + (e - off_o);
          gk[p] = __ldcs(A.ckey + c);
          gl[p] = __ldcs(A.cidx + c);
          gx[p] = __ldcs(A.cval + c);
        }
      }
    };
    if (L > 0u) load_group(0u, nkey, nli, nx, nown);
    for (uint32_t wg = 0; wg < L; wg += 32u * WP) {
#pragma unroll
      for (int p = 0; p < WP; ++p) {
        pkey[p] = nkey[p];
        pli[p] = nli[p];
        px[p] = nx[p];
        pown[p] = nown[p];
      }
      if (wg + 32u * WP < L) load_group(wg + 32u * WP, nkey, nli, nx, nown);
#pragma unroll
    for (int p = 0; p < WP; ++p) {
      const uint32_t ws = wg + 32u * p;
      if (ws >= L) break;
      const uint32_t e = ws + lane;
      const int o = pown[p];
      const uint32_t off_o = __shfl_sync(FULL, off, o);
      const uint32_t eqb_o = __shfl_sync(FULL, eqb, o), sel0_o = __shfl_sync(FULL, sel0, o);
      const uint32_t es_o = __shfl_sync(FULL, es, o), ks_o = __shfl_sync(FULL, ks, o);
      const bool act = e < L;
      const uint32_t key = pkey[p];
      const int32_t li = pli[p];
      const float x = px[p];
      const bool iseq = act && key == thr;
      const unsigned eqm = __ballot_sync(FULL, iseq);
      // the owner's first entry is in this step (off_o - ws <= 31 for every lane)
      const bool here = off_o >= ws;
      const unsigned below_o = (1u << ((off_o - ws) & 31u)) - 1u;
      const uint32_t eqr = eqb_o + (Ec + __popc(eqm & lt) - (here ? Ec + __popc(eqm & below_o) : es_o));
      const bool sel = act && (key > thr || (iseq && eqr < r_eq));
      const unsigned selm = __ballot_sync(FULL, sel);
      if (sel) {
        const uint32_t kin = Kc + __popc(selm & lt) - (here ? Kc + __popc(selm & below_o) : ks_o);
        emit_kept<MODE, KQ>(A, ub.t, ub.base, ub.n, li, x, kbase + sel0_o + kin, s, iseq && eqr + 1u == r_eq);
      }
      if (off - ws < 32u) {
        const unsigned below = (1u << (off - ws)) - 1u;
        ks = Kc + __popc(selm & below);
        es = Ec + __popc(eqm & below);
      }
      Kc += __popc(selm);
      Ec += __popc(eqm);
    }
    }
  }
}

// ============================================================================ one-launch path

// Small arenas (at most FNMAX elements in at most FTMAX tensors) spend most
// of the multi-kernel pipeline's time in launch gaps and short phases.  Here
// one cooperative launch, every CTA resident at once, runs the whole call,
// with grid-wide barriers between its phases:
//   1  acc = g + e, e <- acc; level-1 histogram (key >> 21) and largest key
//      per tensor
//   2  each CTA finds the level-1 bucket of its tensors' k-th key; level-2
//      histogram ((key >> 10) & 2047) of that bucket, re-reading acc (L1- or
//      L2-resident at these sizes)
//   3  level-2 bucket; level-3 histogram (key & 1023) of the 22-bit prefix
//      (skipped, with its barrier, when every tensor's level-1 bucket holds
//      at most FLMAX keys: phase 2 also lists those keys per tensor and
//      phase 4 finds both remaining buckets from the histogram and the list)
//   4  the k-th key and how many of its ties are kept; per-unit counts of
//      keys above and equal to it
//   5  index-ordered compaction into the payload, int8 codes, residual
// A CTA owns the same contiguous range of 2048-element units in every phase
// (a unit never straddles two tensors) and repeats the bucket searches of
// its own tensors from the global histograms, so the barriers (three or
// four) are the only waits between CTAs.  The keys, their total order (ties to the lower
// index) and the payload writer (emit_kept) are the pipeline's, so the
// results are identical to it.
constexpr int FTHREADS = 512;
constexpr int FUNIT_SHIFT = 11;
constexpr int FUNIT = 1 << FUNIT_SHIFT;  // one float4 per thread
constexpr int FTMAX = 1024;
constexpr int64_t FNMAX = int64_t(1) << 22;  // above ~7M elements the pipeline is faster (measured)
constexpr int FTCACHE = 64;                 // tensors one CTA's units may span
constexpr int FBATCH = 2;                   // units whose loads are in flight together (phase 1)
constexpr int FB = 2;                       // the same for the later phases (acc only)
constexpr uint32_t FSPIN_LIMIT = 1u << 20;  // polls of a barrier (about a second)
constexpr uint32_t FLMAX = 4096;  // level-1 bucket keys per tensor up to which level 3 reads the list
static_assert(FTHREADS * 4 == FUNIT, "one float4 per thread per unit");

struct FusedArgs {
  TopkArgs A;        // inputs, outputs and the fields emit_kept reads
  uint32_t* bar;     // arrivals at the grid barriers (zeroed per call)
  uint32_t* maxkey;  // [T] largest key per tensor (zeroed per call)
  uint32_t* h1;      // [T][NBINS] level-1 histograms (zeroed per call)
  uint32_t* h2;      // [T][NBINS] level 2, then [T][NBINS] level 3 (cleared in phase 1)
  uint32_t* ugt;     // [U] keys above the k-th key, per unit
  uint32_t* ueq;     // [U] keys equal to it, per unit
  uint32_t* lcnt;    // [T] keys of the k-th key's level-1 bucket per tensor, then a flag word
                     // set when one exceeds FLMAX (zeroed per call)
  uint32_t* lkey;    // [N] those keys, tensor t's from off[t] - off[0]
  int64_t U;
  uint32_t spin_limit;
};

// One tensor's k-th key search as seen by one CTA.
struct FSel {
  uint32_t b1, b2, r2, r3, thr, r_eq;
  float s;  // int8 scale
  int live;  // k_t > 0 and every level found its bucket
};

struct FUnitRef {
  int t;
  int64_t base;  // arena index of the tensor's element 0
  int64_t n;
  int64_t li0;   // local index of the unit's element 0
  int len;       // elements in the unit (1 .. FUNIT)
};

// Unit u, walking the tensor index t forward (units are visited in order).
__device__ __forceinline__ FUnitRef funit(const int64_t* s_off, const int32_t* s_uoff, int* t, int64_t u) {
  while ((int64_t)s_uoff[*t + 1] <= u) ++*t;
  FUnitRef r;
  r.t = *t;
  r.base = s_off[r.t];
  r.n = s_off[r.t + 1] - r.base;
  r.li0 = (u - (int64_t)s_uoff[r.t]) << FUNIT_SHIFT;
  r.len = (int)min((int64_t)FUNIT, r.n - r.li0);
  return r;
}

// This thread's elements li0 + 4 tid .. + 3 of the unit; returns how many
// exist.  One 16-byte load when the tensor starts on a 16-byte boundary.
template <bool STREAM>
__device__ __forceinline__ int fload4(const float* src, const FUnitRef& r, float x[4]) {
  const int o = 4 * (int)threadIdx.x;
  const int c = max(0, min(4, r.len - o));
  const int64_t gi = r.base + r.li0 + o;
  if (c == 4 && (gi & 3) == 0) {
    const float4* p = reinterpret_cast<const float4*>(src + gi);
    const float4 v = STREAM ? __ldcs(p) : *p;
    x[0] = v.x;
    x[1] = v.y;
    x[2] = v.z;
    x[3] = v.w;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = j < c ? src[gi + j] : 0.0f;
  }
  return c;
}

// The elements of up to NB consecutive units (fewer at u1), loads issued together.
template <int NB>
__device__ __forceinline__ void fload_batch(const float* src, const int64_t* s_off, const int32_t* s_uoff, int* t,
                                            int64_t ub, int64_t u1, float x[NB][4], int c[NB]) {
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    c[j] = 0;
    if (ub + j < u1) {
      const FUnitRef r = funit(s_off, s_uoff, t, ub + j);
      c[j] = fload4<false>(src, r, x[j]);
    }
  }
}

__device__ __forceinline__ void fstore4(float* dst, const FUnitRef& r, const float x[4], int c) {
  const int64_t gi = r.base + r.li0 + 4 * (int)threadIdx.x;
  if (c == 4 && (gi & 3) == 0) {
    *reinterpret_cast<float4*>(dst + gi) = make_float4(x[0], x[1], x[2], x[3]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < c) dst[gi + j] = x[j];
  }
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of the cooperative launch: false when the call is
// aborted.  Every wait is bounded: after spin_limit polls the CTA sets
// GC_DIAG_TIMEOUT and the abort word, which ends the other CTAs' waits too.
__device__ bool fused_barrier(const FusedArgs& F, uint32_t* target, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    *target += gridDim.x;
    __threadfence();
    atomicAdd(F.bar, 1u);
    int ok = 1;
    uint32_t spins = 0;
    while (ld_acquire_gpu(F.bar) < *target) {
      if (*reinterpret_cast<volatile uint32_t*>(F.A.diag + DIAG_ABORT) != 0u) {
        ok = 0;
        break;
      }
      if (++spins > F.spin_limit) {
        atomicOr(F.A.diag + DIAG_ERR, GC_DIAG_TIMEOUT);
        atomicExch(F.A.diag + DIAG_ABORT, 1u);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Adds the shared histogram to a global row and clears it (block-wide).
__device__ __forceinline__ void fflush_hist(uint32_t* s_hist, uint32_t* row) {
  __syncthreads();
  for (int b = threadIdx.x; b < NBINS; b += blockDim.x) {
    const uint32_t v = s_hist[b];
    if (v) {
      atomicAdd(row + b, v);
      s_hist[b] = 0u;
    }
  }
  __syncthreads();
}

// find_bucket on a global row written by other CTAs: copied through L2 into
// shared memory first.
__device__ __forceinline__ uint32_t ffind(const uint32_t* row, uint32_t rank, uint32_t* above, uint32_t* s_row,
                                          uint32_t* s_warp, uint32_t* s_res) {
  for (int b = threadIdx.x; b < NBINS; b += blockDim.x) s_row[b] = __ldcg(row + b);
  __syncthreads();
  return find_bucket(s_row, rank, above, s_warp, s_res);
}

template <bool EF>
__global__ void __launch_bounds__(FTHREADS, 2) k_fused(FusedArgs F) {
  __shared__ int64_t s_off[FTMAX + 1];
  __shared__ int32_t s_uoff[FTMAX + 1];
  __shared__ uint32_t s_hist[NBINS];
  __shared__ uint32_t s_row[NBINS];
  __shared__ uint32_t s_warp[33];
  __shared__ uint32_t s_res[3];
  __shared__ FSel s_sel[FTCACHE];
  __shared__ int s_ok;
  const TopkArgs& A = F.A;
  const int T = A.T;
  const int tid = threadIdx.x;
  const float* src = EF ? A.e : A.g;  // acc after phase 1

  // ---- layout: every CTA reads and checks all of it, so all agree
  if (tid == 0) s_ok = 1;
  for (int i = tid; i <= T; i += blockDim.x) s_off[i] = A.off[i];
  for (int i = tid; i < NBINS; i += blockDim.x) s_hist[i] = 0u;
  __syncthreads();
  uint32_t carry = 0u;
  for (int b0 = 0; b0 < T; b0 += blockDim.x) {
    const int t = b0 + tid;
    uint32_t nu = 0u;
    if (t < T) {
      const int64_t n = s_off[t + 1] - s_off[t];
      const int64_t k = A.kk[t];
      if (n < 1 || n > FNMAX || k < 0 || k > n || A.koff[t + 1] - A.koff[t] != k)
        s_ok = 0;
      else
        nu = (uint32_t)((n + FUNIT - 1) >> FUNIT_SHIFT);
    }
    uint32_t ex, tot;
    block_scan_u32(nu, s_warp, &ex, &tot);
    if (t < T) s_uoff[t] = (int32_t)(carry + ex);
    carry += tot;
  }
  if (tid == 0) {
    s_uoff[T] = (int32_t)carry;
    if (s_off[0] != A.off0 || s_off[T] - A.off0 != A.N || A.koff[0] != A.koff0 || A.koff[T] - A.koff0 != A.K ||
        (int64_t)carry != F.U)
      s_ok = 0;
  }
  __syncthreads();
  if (!s_ok) {
    if (blockIdx.x == 0 && tid == 0) {
      atomicOr(A.diag + DIAG_ERR, GC_DIAG_LAYOUT_MISMATCH);
      atomicExch(A.diag + DIAG_ABORT, 1u);
    }
    return;  // every CTA returns here: no barrier is waited on
  }
  if (blockIdx.x == 0 && tid == 0) A.diag[DIAG_PATH] = 1u;

  // ---- this CTA's units and tensors
  const int64_t G = gridDim.x;
  const int64_t u0 = F.U * (int64_t)blockIdx.x / G, u1 = F.U * ((int64_t)blockIdx.x + 1) / G;
  int tA = 0;
  {
    int lo = 0, hi = T;  // last t with s_uoff[t] <= u0
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if ((int64_t)s_uoff[mid] <= u0) lo = mid; else hi = mid;
    }
    tA = lo;
  }
  bool work = u1 > u0;
  if (work) {
    int tB = tA;
    while ((int64_t)s_uoff[tB + 1] <= u1 - 1) ++tB;
    if (tB - tA + 1 > FTCACHE) {  // the host sizes the grid so that this cannot happen
      if (tid == 0) atomicOr(A.diag + DIAG_ERR, GC_DIAG_SELECT);
      work = false;
    }
  }
  uint32_t target = 0u;  // barrier arrivals awaited (thread 0)

  // ---- phase 1: acc, e <- acc, level-1 histograms, largest keys
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + tid; i < 2 * (int64_t)T * NBINS; i += G * blockDim.x)
    __stcg(F.h2 + i, 0u);
  if (work) {
    int t = tA;
    uint32_t mx = 0u;
    for (int64_t ub = u0; ub < u1; ub += FBATCH) {
      FUnitRef r[FBATCH];
      float gx[FBATCH][4], ex[FBATCH][4];
      int c[FBATCH];
#pragma unroll
      for (int j = 0; j < FBATCH; ++j) {
        c[j] = 0;
        if (ub + j < u1) {
          r[j] = funit(s_off, s_uoff, &t, ub + j);
          c[j] = fload4<!EF>(A.g, r[j], gx[j]);
          if (EF) fload4<false>(A.e, r[j], ex[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < FBATCH; ++j) {
        if (ub + j >= u1) break;
        float a[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) a[q] = EF ? __fadd_rn(gx[j][q], ex[j][q]) : gx[j][q];
        if (EF) fstore4(A.e, r[j], a, c[j]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t key = mag_key(a[q]);
          smem_hist_add(s_hist, key >> 21, q < c[j]);
          if (q < c[j]) mx = max(mx, key);
        }
        if (ub + j + 1 == u1 || (int64_t)s_uoff[r[j].t + 1] == ub + j + 1) {  // the tensor's last unit here
          fflush_hist(s_hist, F.h1 + (size_t)r[j].t * NBINS);
          if (A.int8) {
            const uint32_t wm = warp_max_u32(mx);
            if ((tid & 31) == 0) s_warp[tid >> 5] = wm;
            __syncthreads();
            if (tid == 0) {
              uint32_t m = 0u;
              for (int w = 0; w < FTHREADS / 32; ++w) m = max(m, s_warp[w]);
              atomicMax(F.maxkey + r[j].t, m);
            }
            __syncthreads();
          }
          mx = 0u;
        }
      }
    }
  }
  if (!fused_barrier(F, &target, &s_ok)) return;

  // Phases 2-5 re-read acc; FB units' loads are issued together.
  // ---- phase 2: level-1 bucket; level-2 histograms
  if (work) {
    int tl = tA, t = tA;
    for (int64_t ub = u0; ub < u1; ub += FB) {
      float x[FB][4];
      int c[FB];
      fload_batch<FB>(src, s_off, s_uoff, &tl, ub, u1, x, c);
#pragma unroll
      for (int j = 0; j < FB; ++j) {
        const int64_t u = ub + j;
        if (u >= u1) break;
        const FUnitRef r = funit(s_off, s_uoff, &t, u);
        FSel* sl = s_sel + (r.t - tA);
        if (u == u0 || (int64_t)s_uoff[r.t] == u) {
          const int64_t k = A.kk[r.t];
          uint32_t above = 0u, b = 0xFFFFFFFFu;
          if (k > 0) b = ffind(F.h1 + (size_t)r.t * NBINS, (uint32_t)k, &above, s_row, s_warp, s_res);
          if (tid == 0) {
            sl->live = (k > 0 && b != 0xFFFFFFFFu) ? 1 : 0;
            if (k > 0 && b == 0xFFFFFFFFu) atomicOr(A.diag + DIAG_ERR, GC_DIAG_SELECT);
            sl->b1 = b;
            sl->r2 = (uint32_t)k - above;
          }
          __syncthreads();
        }
        if (!sl->live) continue;
        const uint32_t b1 = sl->b1;
        uint32_t* const lt = F.lkey + (s_off[r.t] - A.off0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t key = mag_key(x[j][q]);
          const bool in = q < c[j] && (key >> 21) == b1;
          smem_hist_add(s_hist, (key >> 10) & 0x7FFu, in);
          // the bucket's keys also go to the tensor's list (one atomic per
          // warp), so that level 3 can read them instead of re-reading acc
          const unsigned m = __ballot_sync(FULL, in);
          if (m) {
            const unsigned lane = tid & 31, lead = __ffs(m) - 1;
            uint32_t base = 0u;
            if (lane == lead) {
              base = atomicAdd(F.lcnt + r.t, (unsigned)__popc(m));
              if (base + (uint32_t)__popc(m) > FLMAX) atomicOr(F.lcnt + T, 1u);
            }
            base = __shfl_sync(FULL, base, lead);
            if (in) lt[base + __popc(m & ((1u << lane) - 1u))] = key;
          }
        }
        if (u + 1 == u1 || (int64_t)s_uoff[r.t + 1] == u + 1) fflush_hist(s_hist, F.h2 + (size_t)r.t * NBINS);
      }
    }
  }
  if (!fused_barrier(F, &target, &s_ok)) return;

  // Every tensor's level-1 bucket list within FLMAX keys: level 3 is searched
  // in those lists at the start of phase 4, and phase 3 with its barrier is
  // skipped.  The flag was final at the barrier, so every CTA decides alike.
  const bool lists = __ldcg(F.lcnt + T) == 0u;

  // ---- phase 3: level-2 bucket; level-3 histograms
  uint32_t* const h3 = F.h2 + (size_t)T * NBINS;
  if (work && !lists) {
    int tl = tA, t = tA;
    for (int64_t ub = u0; ub < u1; ub += FB) {
      float x[FB][4];
      int c[FB];
      fload_batch<FB>(src, s_off, s_uoff, &tl, ub, u1, x, c);
#pragma unroll
      for (int j = 0; j < FB; ++j) {
        const int64_t u = ub + j;
        if (u >= u1) break;
        const FUnitRef r = funit(s_off, s_uoff, &t, u);
        FSel* sl = s_sel + (r.t - tA);
        if (!sl->live) continue;
        if (u == u0 || (int64_t)s_uoff[r.t] == u) {
          uint32_t above = 0u;
          const uint32_t b = ffind(F.h2 + (size_t)r.t * NBINS, sl->r2, &above, s_row, s_warp, s_res);
          if (tid == 0) {
            if (b == 0xFFFFFFFFu) {
              atomicOr(A.diag + DIAG_ERR, GC_DIAG_SELECT);
              sl->live = 0;
            }
            sl->b2 = b;
            sl->r3 = sl->r2 - above;
          }
          __syncthreads();
          if (!sl->live) continue;
        }
        const uint32_t pfx = (sl->b1 << 11) | sl->b2;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t key = mag_key(x[j][q]);
          smem_hist_add(s_hist, key & 0x3FFu, q < c[j] && (key >> 10) == pfx);
        }
        if (u + 1 == u1 || (int64_t)s_uoff[r.t + 1] == u + 1) fflush_hist(s_hist, h3 + (size_t)r.t * NBINS);
      }
    }
  }
  if (!lists && !fused_barrier(F, &target, &s_ok)) return;

  // ---- phase 4: the k-th key, kept ties, scale; per-unit counts
  if (work) {
    int tl = tA, t = tA;
    for (int64_t ub = u0; ub < u1; ub += FB) {
      float x[FB][4];
      int c[FB];
      fload_batch<FB>(src, s_off, s_uoff, &tl, ub, u1, x, c);
#pragma unroll
      for (int j = 0; j < FB; ++j) {
        const int64_t u = ub + j;
        if (u >= u1) break;
        const FUnitRef r = funit(s_off, s_uoff, &t, u);
        FSel* sl = s_sel + (r.t - tA);
        const bool owner = (int64_t)s_uoff[r.t] == u;  // this CTA holds the tensor's first unit
        if (u == u0 || owner) {
          if (sl->live && lists) {
            // level 2 as phase 3 would find it, then level 3 over the list
            uint32_t above = 0u;
            const uint32_t b = ffind(F.h2 + (size_t)r.t * NBINS, sl->r2, &above, s_row, s_warp, s_res);
            if (tid == 0) {
              if (b == 0xFFFFFFFFu) {
                atomicOr(A.diag + DIAG_ERR, GC_DIAG_SELECT);
                sl->live = 0;
              }
              sl->b2 = b;
              sl->r3 = sl->r2 - above;
            }
            __syncthreads();
            if (sl->live) {
              const uint32_t pfx = (sl->b1 << 11) | sl->b2;
              const uint32_t nl = __ldcg(F.lcnt + r.t);
              const uint32_t* lt = F.lkey + (s_off[r.t] - A.off0);
              for (uint32_t i0 = 0; i0 < nl; i0 += 4 * blockDim.x) {  // at most two rounds of loads
                uint32_t kk[4];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  const uint32_t i = i0 + v * blockDim.x + tid;
                  kk[v] = i < nl ? __ldcg(lt + i) : 0u;
                }
#pragma unroll
                for (int v = 0; v < 4; ++v)
                  if (i0 + v * blockDim.x + tid < nl && (kk[v] >> 10) == pfx) atomicAdd(s_hist + (kk[v] & 0x3FFu), 1u);
              }
              __syncthreads();
              uint32_t above3 = 0u;
              const uint32_t b3 = find_bucket(s_hist, sl->r3, &above3, s_warp, s_res);
              for (int i = tid; i < 1024; i += blockDim.x) s_hist[i] = 0u;
              if (tid == 0) {
                if (b3 == 0xFFFFFFFFu) {
                  atomicOr(A.diag + DIAG_ERR, GC_DIAG_SELECT);
                  sl->live = 0;
                }
                sl->thr = (pfx << 10) | b3;
                sl->r_eq = sl->r3 - above3;
                sl->s = A.int8 ? __fdiv_rn(key_magnitude(__ldcg(F.maxkey + r.t)), 127.0f) : 0.0f;
              }
            }
          } else if (sl->live) {
            uint32_t above = 0u;
            const uint32_t b = ffind(h3 + (size_t)r.t * NBINS, sl->r3, &above, s_row, s_warp, s_res);
            if (tid == 0) {
              if (b == 0xFFFFFFFFu) {
                atomicOr(A.diag + DIAG_ERR, GC_DIAG_SELECT);
                sl->live = 0;
              }
              sl->thr = (((sl->b1 << 11) | sl->b2) << 10) | b;
              sl->r_eq = sl->r3 - above;
              sl->s = A.int8 ? __fdiv_rn(key_magnitude(__ldcg(F.maxkey + r.t)), 127.0f) : 0.0f;
            }
          }
          __syncthreads();
          if (owner && tid == 0 && A.int8) A.scale[r.t] = sl->live ? sl->s : 0.0f;
        }
        uint32_t v = 0u;
        if (sl->live) {
          const uint32_t thr = sl->thr;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t key = mag_key(x[j][q]);
            if (q < c[j]) v += (key > thr ? 1u : 0u) | (key == thr ? 0x10000u : 0u);
          }
        }
        uint32_t ex, tot;
        block_scan_u32(v, s_warp, &ex, &tot);  // unit counts < 2^16 each
        if (tid == 0) {
          F.ugt[u] = tot & 0xFFFFu;
          F.ueq[u] = tot >> 16;
        }
      }
    }
  }
  if (!fused_barrier(F, &target, &s_ok)) return;

  // ---- phase 5: payload and residual, in index order
  if (work) {
    int tl = tA, t = tA;
    uint32_t bgt = 0u, beq = 0u;  // this tensor's keys above / equal to the k-th key before the unit
    for (int64_t ub = u0; ub < u1; ub += FB) {
      float x[FB][4];
      int c[FB];
      fload_batch<FB>(src, s_off, s_uoff, &tl, ub, u1, x, c);
#pragma unroll
      for (int j = 0; j < FB; ++j) {
        const int64_t u = ub + j;
        if (u >= u1) break;
        const FUnitRef r = funit(s_off, s_uoff, &t, u);
        const FSel S = s_sel[r.t - tA];
        if (!S.live) continue;
        if (u == u0 || (int64_t)s_uoff[r.t] == u) {
          uint32_t pg = 0u, pe = 0u;
          for (int64_t w = (int64_t)s_uoff[r.t] + tid; w < u; w += blockDim.x) {
            pg += __ldcg(F.ugt + w);
            pe += __ldcg(F.ueq + w);
          }
          uint32_t ex;
          block_scan_u32(pg, s_warp, &ex, &bgt);
          block_scan_u32(pe, s_warp, &ex, &beq);
        }
        unsigned gtm = 0u, eqm = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t key = mag_key(x[j][q]);
          gtm |= (q < c[j] && key > S.thr ? 1u : 0u) << q;
          eqm |= (q < c[j] && key == S.thr ? 1u : 0u) << q;
        }
        uint32_t epre, etot;
        block_scan_u32((uint32_t)__popc(eqm), s_warp, &epre, &etot);
        unsigned selm = gtm;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (((eqm >> q) & 1u) && beq + epre + (uint32_t)__popc(eqm & ((1u << q) - 1u)) < S.r_eq) selm |= 1u << q;
        uint32_t spre, stot;
        block_scan_u32((uint32_t)__popc(selm), s_warp, &spre, &stot);
        const int64_t pos0 = A.koff[r.t] + (int64_t)bgt + (int64_t)min(beq, S.r_eq) + spre;
        for (unsigned m = selm; m != 0u; m &= m - 1u) {
          const int q = __ffs(m) - 1;
          const float xv = q == 0 ? x[j][0] : (q == 1 ? x[j][1] : (q == 2 ? x[j][2] : x[j][3]));
          emit_kept<MODE_TOPK, KQ_NONE>(A, r.t, r.base, r.n, r.li0 + 4 * tid + q, xv,
                                        pos0 + __popc(selm & ((1u << q) - 1u)), S.s, false);
        }
        bgt += __ldcg(F.ugt + u);
        beq += etot;
      }
    }
  }
}

// ============================================================================ host side

struct TopkLayoutTotals {
  int64_t U = 0, UB = 0, C = 0, S = 0, N = 0, K = 0, SB = 0, SBmax = 0;
  int split = 1;
  int ubu = UB_UNITS;
};

// Units per unit block: UB_UNITS_DENSE when the arena keeps at least 16
// elements per 4096-element unit on average (1% density and up), where a
// warp walking 32 units' candidates sets the count and write kernels' time;
// UB_UNITS otherwise, where small blocks would only add CTAs.  A function of
// the layout alone, so the workspace query and the call agree.
static int unit_block_units(const gc_layout* h) {
  int64_t K = 0, U = 0;
  for (int t = 0; t < h->num_tensors; ++t) {
    K += h->k[t];
    U += units_of(h->off[t + 1] - h->off[t]);
  }
  return K >= 16 * U ? UB_UNITS_DENSE : UB_UNITS;
}

// Sampling CTAs per large sample: enough to give about two CTAs per SM of
// the current device when the arena has few large tensors.
static int sampling_split(const gc_layout* h) {
  int large = 0;
  for (int t = 0; t < h->num_tensors; ++t)
    if (sample_splittable(h->off[t + 1] - h->off[t], h->k[t])) ++large;
  if (large == 0) return 1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();  // leave no error state behind
    sms = 152;
  }
  const int f = (2 * sms) / large;
  return f < 1 ? 1 : (f > 64 ? 64 : f);
}

// split_for_launch: also choose the sampling split for the current device
// (the workspace size does not depend on it).
static TopkLayoutTotals totals_of(const gc_layout* h, bool sampled, bool split_for_launch = false) {
  TopkLayoutTotals r;
  if (sampled && split_for_launch) r.split = sampling_split(h);
  r.ubu = unit_block_units(h);
  for (int t = 0; t < h->num_tensors; ++t) {
    const int64_t n = h->off[t + 1] - h->off[t];
    const int64_t k = h->k[t];
    r.U += units_of(n);
    r.UB += ublocks_of(n, r.ubu);
    r.C += cand_capacity(n, k);
    if (sampled && k > 0) {
      int64_t runs, stride, m;
      sample_plan(n, k, &runs, &stride, &m);
      r.S += m;
    }
    if (sampled) {
      r.SB += sample_ctas(n, k, r.split);
      r.SBmax += sample_ctas(n, k, 64);  // the dispatch table fits any device's split (at most 64)
    }
    r.K += k;
  }
  r.N = h->off[h->num_tensors] - h->off[0];
  return r;
}

struct TopkCarve {
  size_t zero_bytes = 0, total = 0;
  size_t o_ts, o_hist, o_scnt, o_units, o_ublk, o_cand, o_soff, o_chunk, o_ugt, o_ueq, o_bgt, o_beq, o_ckey,
      o_cidx, o_cval, o_skey, o_upart, o_kwoff, o_sblk, o_sord, o_smap;
};

static TopkCarve carve_topk(int T, const TopkLayoutTotals& z) {
  TopkCarve c;
  size_t p = DIAG_BYTES;
  auto take = [&p](size_t bytes) {
    const size_t at = p;
    p = align_up(p + bytes, 256);
    return at;
  };
  c.o_ts = take(sizeof(TensorState) * (size_t)T);
  c.o_hist = take((size_t)T * NBINS * 4);
  c.o_scnt = take(8 * (size_t)T);
  c.zero_bytes = p;
  c.o_units = take(8 * (size_t)(T + 1));
  c.o_ublk = take(8 * (size_t)(T + 1));
  c.o_cand = take(8 * (size_t)(T + 1));
  c.o_soff = take(8 * (size_t)(T + 1));
  c.o_chunk = take(8 * (size_t)z.U);
  c.o_ugt = take(4 * (size_t)z.U);
  c.o_ueq = take(4 * (size_t)z.U);
  c.o_bgt = take(4 * (size_t)z.UB);
  c.o_beq = take(4 * (size_t)z.UB);
  c.o_ckey = take(4 * (size_t)z.C);
  c.o_cidx = take(4 * (size_t)z.C);
  c.o_cval = take(4 * (size_t)z.C);
  c.o_skey = take(4 * (size_t)z.S);
  c.o_upart = take(8 * (size_t)z.U);
  c.o_kwoff = take(8 * (size_t)(T + 1));
  c.o_sblk = take(8 * (size_t)(T + 1));
  c.o_sord = take(8 * (size_t)T);
  c.o_smap = take(8 * (size_t)(z.SBmax > 0 ? z.SBmax : 1));
  c.total = p;
  return c;
}

// ---------------------------------------------------------------- one-launch path (host)

struct FusedCarve {
  int64_t U = 0;
  size_t zero_bytes = 0, total = 0;
  size_t o_bar = 0, o_max = 0, o_h1 = 0, o_lcnt = 0, o_h2 = 0, o_ugt = 0, o_ueq = 0, o_lkey = 0;
};

static bool fused_layout_fits(const gc_layout* h) {
  return h->num_tensors <= FTMAX && h->off[h->num_tensors] - h->off[0] <= FNMAX;
}

static FusedCarve carve_fused(const gc_layout* h) {
  FusedCarve c;
  const int T = h->num_tensors;
  for (int t = 0; t < T; ++t) c.U += (h->off[t + 1] - h->off[t] + FUNIT - 1) >> FUNIT_SHIFT;
  size_t p = DIAG_BYTES;
  auto take = [&p](size_t bytes) {
    const size_t at = p;
    p = align_up(p + bytes, 256);
    return at;
  };
  c.o_bar = take(4);
  c.o_max = take(4 * (size_t)T);
  c.o_h1 = take((size_t)T * NBINS * 4);
  c.o_lcnt = take(4 * ((size_t)T + 1));
  c.zero_bytes = p;
  c.o_h2 = take(2 * (size_t)T * NBINS * 4);
  c.o_ugt = take(4 * (size_t)c.U);
  c.o_ueq = take(4 * (size_t)c.U);
  c.o_lkey = take(4 * (size_t)(h->off[T] - h->off[0]));
  c.total = p;
  return c;
}

size_t topk_workspace_bytes(const gc_layout* h, bool sampled) {
  size_t b = carve_topk(h->num_tensors, totals_of(h, sampled)).total;
  if (sampled && fused_layout_fits(h)) b = std::max(b, carve_fused(h).total);
  return b;
}

template <class K>
static int stream_grid(K kernel, int64_t units) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, STREAM_THREADS, STREAM_SMEM);
  if (per_sm < 1) per_sm = 1;
  int64_t want = (units + STREAM_WARPS - 1) / STREAM_WARPS;
  int64_t grid = (int64_t)sms * per_sm;
  if (grid > want) grid = want;
  if (grid < 1) grid = 1;
  return (int)grid;
}

template <int MODE, bool EF, bool LOADG, bool LAZY = false>
static void launch_stream(const TopkArgs& A, cudaStream_t s) {
  auto kern = k_stream<MODE, EF, LOADG, LAZY>;
  launch_chained(kern, stream_grid(kern, A.U), STREAM_THREADS, STREAM_SMEM, s, A);
}

// Optional CUDA events recorded on the call's stream.  With n <= 5 they
// mark the phases (start, before the streaming pass, after it, after the
// k-th key search, after the payload write); with n > 5, event 0 marks the
// start and event j the end of the j-th enqueued operation.
struct PhaseEvents {
  void* const* ev = nullptr;
  int n = 0;
  mutable int ops = 0;
  void record(int i, cudaStream_t s) const {
    if (i < n && ev[i]) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s);
  }
  void start(cudaStream_t s) const { record(0, s); }
  // after each enqueued operation; `phase` > 0 if it ends that phase
  void done(int phase, cudaStream_t s) const {
    ++ops;
    if (n > 5)
      record(ops, s);
    else if (phase > 0)
      record(phase, s);
  }
};

// Grid of the cooperative launch: every CTA resident (at most the SMs times
// the CTAs that fit on one), at most one per unit, and no CTA's contiguous
// unit range spanning more than FTCACHE tensors.  0 if the path cannot run.
static int fused_grid(const gc_layout* h, int64_t U, bool ef) {
  int dev = 0, sms = 0, coop = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ef ? k_fused<true> : k_fused<false>, FTHREADS, 0) !=
          cudaSuccess) {
    cudaGetLastError();  // leave no error state behind
    return 0;
  }
  if (!coop || per_sm < 1 || U < 1) return 0;
  int64_t G = (int64_t)sms * per_sm;
  if (G > U) G = U;
  const int T = h->num_tensors;
  std::vector<int64_t> uoff(T + 1, 0);
  for (int t = 0; t < T; ++t) uoff[t + 1] = uoff[t] + ((h->off[t + 1] - h->off[t] + FUNIT - 1) >> FUNIT_SHIFT);
  int ta = 0;
  for (int64_t b = 0; b < G; ++b) {
    const int64_t u0 = U * b / G, u1 = U * (b + 1) / G;
    if (u1 <= u0) continue;
    while (uoff[ta + 1] <= u0) ++ta;
    int tb = ta;
    while (uoff[tb + 1] <= u1 - 1) ++tb;
    if (tb - ta + 1 > FTCACHE) return 0;
  }
  return (int)G;
}

static gc_status launch_fused(const TopkArgs& A0, const gc_layout* host, const FusedCarve& fc, int G, void* ws,
                              cudaStream_t s, const PhaseEvents& pe) {
  unsigned char* w = static_cast<unsigned char*>(ws);
  FusedArgs F;
  memset(&F, 0, sizeof F);
  F.A = A0;
  F.bar = reinterpret_cast<uint32_t*>(w + fc.o_bar);
  F.maxkey = reinterpret_cast<uint32_t*>(w + fc.o_max);
  F.h1 = reinterpret_cast<uint32_t*>(w + fc.o_h1);
  F.h2 = reinterpret_cast<uint32_t*>(w + fc.o_h2);
  F.ugt = reinterpret_cast<uint32_t*>(w + fc.o_ugt);
  F.ueq = reinterpret_cast<uint32_t*>(w + fc.o_ueq);
  F.lcnt = reinterpret_cast<uint32_t*>(w + fc.o_lcnt);
  F.lkey = reinterpret_cast<uint32_t*>(w + fc.o_lkey);
  F.U = fc.U;
  F.spin_limit = FSPIN_LIMIT;
  pe.start(s);
  if (cudaMemsetAsync(ws, 0, fc.zero_bytes, s) != cudaSuccess) return GC_ERR_CUDA;
  pe.done(0, s);
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(FTHREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  memset(&attr, 0, sizeof attr);
  attr.id = cudaLaunchAttributeCooperative;
  attr.val.cooperative = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  const cudaError_t err = F.A.ef ? cudaLaunchKernelEx(&cfg, k_fused<true>, F) : cudaLaunchKernelEx(&cfg, k_fused<false>, F);
  if (err != cudaSuccess) return GC_ERR_CUDA;
  for (int ph = 1; ph <= 4; ++ph) pe.done(ph, s);  // one launch: the inner phases take no time of their own
  (void)host;
  return GC_OK;
}

template <int MODE>
static void launch_pipeline(const TopkArgs& A, cudaStream_t s, const PhaseEvents& pe) {
  const int T = A.T;
  launch_chained(k_plan, 1, 1024, 0, s, A);
  if (A.clip) {
    launch_chained(k_gnorm, stream_grid(k_gnorm, A.U), 256, 0, s, A);
    launch_chained(k_gscale, T, 256, 0, s, A);
  }
  pe.done(A.sampled ? 0 : 1, s);
  if (A.sampled) {
    if (A.SB > 0) launch_chained(k_sample<MODE>, (unsigned)A.SB, 512, 0, s, A);
    pe.done(1, s);
  }
  if (MODE == MODE_MOM) {
    launch_stream<MODE_MOM, false, true>(A, s);
  } else if (MODE == MODE_TOPK) {
    if (A.ef && A.rd)
      launch_stream<MODE_TOPK, true, true, true>(A, s);
    else if (A.ef)
      launch_stream<MODE_TOPK, true, true>(A, s);
    else
      launch_stream<MODE_TOPK, false, true>(A, s);
  } else {
    if (A.unbiased)
      launch_stream<MODE_RANDK, false, false>(A, s);
    else if (A.ef)
      launch_stream<MODE_RANDK, true, true>(A, s);
    else
      launch_stream<MODE_RANDK, false, true>(A, s);
  }
  pe.done(2, s);
  const unsigned UBg = (unsigned)A.UB;
  // radix select: level 1 on the streaming pass's candidate histogram, then
  // a histogram pass and a select per level (running each tensor's select in
  // the last CTA of its histogram pass measured slower on the Llama arena:
  // 0.186 against 0.155 ms)
  launch_chained(k_select, T, 256, 0, s, A, (int)PH_C1);
  pe.done(0, s);
  launch_chained(k_hist<MODE>, UBg, 256, 0, s, A, 1);
  pe.done(0, s);
  launch_chained(k_select, T, 256, 0, s, A, (int)PH_C1D);
  pe.done(0, s);
  launch_chained(k_hist<MODE>, UBg, 256, 0, s, A, 2);
  pe.done(0, s);
  launch_chained(k_select, T, 256, 0, s, A, (int)PH_C2);
  pe.done(0, s);
  launch_chained(k_hist<MODE>, UBg, 256, 0, s, A, 3);
  pe.done(0, s);
  launch_chained(k_select, T, 256, 0, s, A, (int)PH_C3);
  pe.done(3, s);
  if (MODE != MODE_RANDK && A.qkind != KQ_NONE)
    launch_chained(k_count<MODE, MODE != MODE_RANDK>, UBg, 256, 0, s, A);
  else
    launch_chained(k_count<MODE, false>, UBg, 256, 0, s, A);
  pe.done(0, s);
  launch_chained(k_scan, T, 256, 0, s, A);
  pe.done(0, s);
  if (MODE != MODE_RANDK && A.qkind == KQ_QSGD)
    launch_chained(k_write<MODE, MODE != MODE_RANDK ? KQ_QSGD : KQ_NONE>, UBg, 256, 0, s, A);
  else if (MODE != MODE_RANDK && A.qkind == KQ_SIGN)
    launch_chained(k_write<MODE, MODE != MODE_RANDK ? KQ_SIGN : KQ_NONE>, UBg, 256, 0, s, A);
  else
    launch_chained(k_write<MODE, KQ_NONE>, UBg, 256, 0, s, A);
  pe.done(4, s);
}

// QSGD or sign quantization of the kept values (kind KQ_*), its levels and
// the sign-bit output.
struct KeptQuant {
  int kind = KQ_NONE;
  int slev = 0;
  uint32_t* bits = nullptr;
};

static gc_status run_topk(int mode, const gc_layout* dev, const gc_layout* host, const float* g,
                          float* e, float* u, float* v, float beta, int32_t* idx, float* val,
                          int8_t* q, float* scale, uint64_t seed, uint64_t iter, uint32_t flags,
                          void* ws, size_t ws_bytes, void* stream, const PhaseEvents& pe,
                          gc_residual_desc* rd = nullptr, const float* tau = nullptr,
                          int64_t* count_out = nullptr, const float* clip = nullptr,
                          float* norm_out = nullptr, uint64_t* iter_dev = nullptr,
                          const KeptQuant& kq = KeptQuant{}) {
  gc_status st = validate_layout(host, true);
  if (st != GC_OK) return st;
  if (!dev || !dev->off || !dev->k || !dev->koff || dev->num_tensors != host->num_tensors)
    return GC_ERR_INVALID_ARG;
  const bool int8 = (flags & GC_INT8) != 0u;
  if (!g || !idx) return GC_ERR_INVALID_ARG;
  if (int8 && (!q || !scale)) return GC_ERR_INVALID_ARG;
  if (kq.kind != KQ_NONE) {
    if (int8 || !scale || (kq.kind == KQ_QSGD && !q) || (kq.kind == KQ_SIGN && !kq.bits)) return GC_ERR_INVALID_ARG;
  } else if (!int8 && !val) {
    return GC_ERR_INVALID_ARG;
  }
  if (!aligned16(g) || (e && !aligned16(e)) || (u && !aligned16(u)) || (v && !aligned16(v)))
    return GC_ERR_ALIGNMENT;
  const bool sampled = mode != MODE_RANDK;
  const TopkLayoutTotals z = totals_of(host, sampled, true);
  const TopkCarve c = carve_topk(host->num_tensors, z);
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < c.total) return GC_ERR_WORKSPACE;
  if (z.K == 0 && z.N == 0) return GC_OK;

  unsigned char* w = static_cast<unsigned char*>(ws);
  TopkArgs A;
  memset(&A, 0, sizeof A);
  A.T = host->num_tensors;
  A.mode = mode;
  A.flags = flags;
  A.int8 = int8 ? 1 : 0;
  A.ef = (mode == MODE_MOM) ? 0 : ((flags & GC_EF) ? 1 : 0);
  A.unbiased = (flags & GC_UNBIASED) ? 1 : 0;
  A.masking = (flags & GC_NO_MASK) ? 0 : 1;
  A.beta = beta;
  A.off = dev->off;
  A.kk = dev->k;
  A.koff = dev->koff;
  A.g = g;
  A.e = e;
  A.u = u;
  A.v = v;
  A.idx = idx;
  A.val = val;
  A.q = q;
  A.scale = scale;
  A.seed = seed;
  A.pk = make_philox_key(seed);
  A.iter = iter;
  A.iter_dev = iter_dev;
  A.rd = rd;
  A.tau = tau;
  A.count_out = count_out;
  A.sampled = sampled ? 1 : 0;
  A.diag = reinterpret_cast<uint32_t*>(w);
  A.ts = reinterpret_cast<TensorState*>(w + c.o_ts);
  A.hist = reinterpret_cast<uint32_t*>(w + c.o_hist);
  A.units_off = reinterpret_cast<int64_t*>(w + c.o_units);
  A.ublk_off = reinterpret_cast<int64_t*>(w + c.o_ublk);
  A.cand_off = reinterpret_cast<int64_t*>(w + c.o_cand);
  A.soff = reinterpret_cast<int64_t*>(w + c.o_soff);
  A.chunk = reinterpret_cast<uint2*>(w + c.o_chunk);
  A.ugt = reinterpret_cast<uint32_t*>(w + c.o_ugt);
  A.ueq = reinterpret_cast<uint32_t*>(w + c.o_ueq);
  A.bgt = reinterpret_cast<uint32_t*>(w + c.o_bgt);
  A.beq = reinterpret_cast<uint32_t*>(w + c.o_beq);
  A.ckey = reinterpret_cast<uint32_t*>(w + c.o_ckey);
  A.cidx = reinterpret_cast<int32_t*>(w + c.o_cidx);
  A.cval = reinterpret_cast<float*>(w + c.o_cval);
  A.skey = reinterpret_cast<uint32_t*>(w + c.o_skey);
  A.upart = reinterpret_cast<double*>(w + c.o_upart);
  A.clip = clip;
  A.norm_out = norm_out;
  A.qkind = kq.kind;
  A.slev = kq.slev;
  A.bits = kq.bits;
  A.kwoff = reinterpret_cast<int64_t*>(w + c.o_kwoff);
  A.sblk = reinterpret_cast<int64_t*>(w + c.o_sblk);
  A.sord = reinterpret_cast<int64_t*>(w + c.o_sord);
  A.smap = reinterpret_cast<int2*>(w + c.o_smap);
  A.scnt = reinterpret_cast<uint32_t*>(w + c.o_scnt);
  A.U = z.U;
  A.UB = z.UB;
  A.C = z.C;
  A.S = z.S;
  A.N = z.N;
  A.K = z.K;
  A.off0 = host->off[0];
  A.koff0 = host->koff[0];
  A.ubu = z.ubu;
  A.SB = z.SB;
  A.ssplit = z.split;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mode == MODE_TOPK && !rd && !tau && !clip && kq.kind == KQ_NONE &&
      !(flags & (GC_FORCE_EXACT | GC_MULTI_KERNEL)) && fused_layout_fits(host)) {
    const FusedCarve fc = carve_fused(host);
    const int G = ws_bytes >= fc.total ? fused_grid(host, fc.U, A.ef != 0) : 0;
    if (G > 0) {
      const gc_status fst = launch_fused(A, host, fc, G, ws, s, pe);
      if (fst != GC_OK) return fst;
      if (iter_dev) k_iter_advance<<<1, 1, 0, s>>>(iter_dev);
      return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
    }
  }
  pe.start(s);
  if (!zero_chained(ws, c.zero_bytes, s)) return GC_ERR_CUDA;
  pe.done(0, s);
  if (kq.kind == KQ_SIGN) {
    // the payload write sets the bits of the positive kept values
    int64_t words = 0;
    for (int t = 0; t < host->num_tensors; ++t) words += (host->k[t] + 31) / 32;
    if (words > 0 && cudaMemsetAsync(kq.bits, 0, (size_t)words * 4u, s) != cudaSuccess) return GC_ERR_CUDA;
  }
  if (mode == MODE_TOPK)
    launch_pipeline<MODE_TOPK>(A, s, pe);
  else if (mode == MODE_RANDK)
    launch_pipeline<MODE_RANDK>(A, s, pe);
  else
    launch_pipeline<MODE_MOM>(A, s, pe);
  if (iter_dev) launch_chained(k_iter_advance, 1, 1, 0, s, iter_dev);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

}  // namespace gc

using namespace gc;

static gc_status topk_entry(const gc_layout* dev, const gc_layout* host, const float* g, float* e,
                            int32_t* idx, float* val, int8_t* q, float* scale, uint64_t seed,
                            uint64_t iter, uint32_t flags, void* workspace, size_t ws_bytes,
                            void* stream, const PhaseEvents& pe, uint64_t* iter_dev = nullptr) {
  const uint32_t known = GC_EF | GC_INT8 | GC_RANDK | GC_UNBIASED | GC_FORCE_EXACT | GC_MULTI_KERNEL;
  if (flags & ~known) return GC_ERR_INVALID_ARG;
  const bool randk = (flags & GC_RANDK) != 0u;
  if (randk && (flags & GC_INT8)) return GC_ERR_INVALID_ARG;
  if ((flags & GC_UNBIASED) && (!randk || (flags & GC_EF))) return GC_ERR_INVALID_ARG;
  if ((flags & GC_EF) && !e) return GC_ERR_INVALID_ARG;
  return run_topk(randk ? MODE_RANDK : MODE_TOPK, dev, host, g, (flags & GC_EF) ? e : nullptr,
                  nullptr, nullptr, 0.0f, idx, val, q, scale, seed, iter, flags, workspace,
                  ws_bytes, stream, pe, nullptr, nullptr, nullptr, nullptr, nullptr, iter_dev);
}

extern "C" gc_status gc_ef_topk_compress_dev_iter(const gc_layout* dev, const gc_layout* host,
                                                  const float* g, float* e, int32_t* idx, float* val,
                                                  int8_t* q, float* scale, uint64_t seed,
                                                  uint64_t* iter_dev, uint32_t flags, void* workspace,
                                                  size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("gc_ef_topk_compress_dev_iter");
  if (!iter_dev || ((uintptr_t)iter_dev & 7u)) return GC_ERR_INVALID_ARG;
  return topk_entry(dev, host, g, e, idx, val, q, scale, seed, 0, flags, workspace, ws_bytes, stream,
                    PhaseEvents{}, iter_dev);
}

extern "C" gc_status gc_ef_topk_compress(const gc_layout* dev, const gc_layout* host,
                                         const float* g, float* e, int32_t* idx, float* val,
                                         int8_t* q, float* scale, uint64_t seed, uint64_t iter,
                                         uint32_t flags, void* workspace, size_t ws_bytes,
                                         void* stream) {
  NvtxRange nvtx_range("gc_ef_topk_compress");
  return topk_entry(dev, host, g, e, idx, val, q, scale, seed, iter, flags, workspace, ws_bytes,
                    stream, PhaseEvents{});
}

extern "C" gc_status gc_ef_topk_compress_profiled(const gc_layout* dev, const gc_layout* host,
                                                  const float* g, float* e, int32_t* idx,
                                                  float* val, int8_t* q, float* scale,
                                                  uint64_t seed, uint64_t iter, uint32_t flags,
                                                  void* workspace, size_t ws_bytes, void* stream,
                                                  void* const* events, int32_t n_events) {
  NvtxRange nvtx_range("gc_ef_topk_compress_profiled");
  if (n_events < 0 || n_events > 32 || (n_events > 0 && !events)) return GC_ERR_INVALID_ARG;
  PhaseEvents pe;
  pe.ev = events;
  pe.n = n_events;
  return topk_entry(dev, host, g, e, idx, val, q, scale, seed, iter, flags, workspace, ws_bytes,
                    stream, pe);
}

extern "C" gc_status gc_ef_topk_compress_momentum(const gc_layout* dev, const gc_layout* host,
                                                  const float* g, float* u, float* v, float beta,
                                                  int32_t* idx, float* val, int8_t* q,
                                                  float* scale, uint64_t seed, uint64_t iter,
                                                  uint32_t flags, void* workspace,
                                                  size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("gc_ef_topk_compress_momentum");
  const uint32_t known = GC_INT8 | GC_NO_MASK | GC_FORCE_EXACT;
  if (flags & ~known) return GC_ERR_INVALID_ARG;
  if (!u || !v) return GC_ERR_INVALID_ARG;
  return run_topk(MODE_MOM, dev, host, g, nullptr, u, v, beta, idx, val, q, scale, seed, iter,
                  flags, workspace, ws_bytes, stream, PhaseEvents{});
}

// Kept-value quantizer of the *_quantized entry points: int8 goes through the
// GC_INT8 path, QSGD and sign through KeptQuant.
static gc_status kept_quant_of(int32_t kind, int32_t s_levels, uint32_t* bits, uint32_t* flags,
                               KeptQuant* kq) {
  switch (kind) {
    case GC_KEPT_INT8:
      *flags |= GC_INT8;
      return GC_OK;
    case GC_KEPT_QSGD:
      if (s_levels < 1 || s_levels > 127) return GC_ERR_INVALID_ARG;
      kq->kind = KQ_QSGD;
      kq->slev = s_levels;
      return GC_OK;
    case GC_KEPT_SIGN:
      if (!bits) return GC_ERR_INVALID_ARG;
      kq->kind = KQ_SIGN;
      kq->bits = bits;
      return GC_OK;
    default:
      return GC_ERR_INVALID_ARG;
  }
}

extern "C" gc_status gc_ef_topk_compress_quantized(const gc_layout* dev, const gc_layout* host,
                                                   const float* g, float* e, int32_t* idx,
                                                   float* val, int8_t* q, uint32_t* bits,
                                                   float* scale, int32_t kind, int32_t s_levels,
                                                   uint64_t seed, uint64_t iter, uint32_t flags,
                                                   void* workspace, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("gc_ef_topk_compress_quantized");
  const uint32_t known = GC_EF | GC_FORCE_EXACT;
  if (flags & ~known) return GC_ERR_INVALID_ARG;
  if ((flags & GC_EF) && !e) return GC_ERR_INVALID_ARG;
  KeptQuant kq;
  const gc_status st = kept_quant_of(kind, s_levels, bits, &flags, &kq);
  if (st != GC_OK) return st;
  return run_topk(MODE_TOPK, dev, host, g, (flags & GC_EF) ? e : nullptr, nullptr, nullptr, 0.0f,
                  idx, val, q, scale, seed, iter, flags, workspace, ws_bytes, stream, PhaseEvents{},
                  nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, kq);
}

extern "C" gc_status gc_ef_topk_compress_momentum_quantized(
    const gc_layout* dev, const gc_layout* host, const float* g, float* u, float* v, float beta,
    int32_t* idx, float* val, int8_t* q, uint32_t* bits, float* scale, int32_t kind,
    int32_t s_levels, uint64_t seed, uint64_t iter, uint32_t flags, void* workspace,
    size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("gc_ef_topk_compress_momentum_quantized");
  const uint32_t known = GC_NO_MASK | GC_FORCE_EXACT;
  if (flags & ~known) return GC_ERR_INVALID_ARG;
  if (!u || !v) return GC_ERR_INVALID_ARG;
  KeptQuant kq;
  const gc_status st = kept_quant_of(kind, s_levels, bits, &flags, &kq);
  if (st != GC_OK) return st;
  return run_topk(MODE_MOM, dev, host, g, nullptr, u, v, beta, idx, val, q, scale, seed, iter,
                  flags, workspace, ws_bytes, stream, PhaseEvents{}, nullptr, nullptr, nullptr,
                  nullptr, nullptr, nullptr, kq);
}

extern "C" gc_status gc_ef_topk_compress_lazy(const gc_layout* dev, const gc_layout* host,
                                              const float* g, float* e, gc_residual_desc* rd,
                                              int32_t* idx, float* val, int8_t* q, float* scale,
                                              uint64_t seed, uint64_t iter, uint32_t flags,
                                              void* workspace, size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("gc_ef_topk_compress_lazy");
  const uint32_t known = GC_EF | GC_INT8 | GC_FORCE_EXACT;
  if (flags & ~known) return GC_ERR_INVALID_ARG;
  if (!e || !rd) return GC_ERR_INVALID_ARG;
  return run_topk(MODE_TOPK, dev, host, g, e, nullptr, nullptr, 0.0f, idx, val, q, scale, seed,
                  iter, flags | GC_EF, workspace, ws_bytes, stream, PhaseEvents{}, rd);
}

namespace gc {

// e <- exact residual for every tensor with a pending selection.
__global__ void __launch_bounds__(256) k_materialize(const int64_t* off, int T, float* e,
                                                     const gc_residual_desc* rd) {
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
    const gc_residual_desc d = rd[t];
    if (!(d.flags & 1u)) continue;
    const int64_t base = off[t], n = off[t + 1] - base;
    for (int64_t li = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; li < n;
         li += (int64_t)gridDim.x * blockDim.x)
      e[base + li] = lazy_fix(e[base + li], li, base + li, d);
  }
}

__global__ void k_clear_desc(gc_residual_desc* rd, int T) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x)
    rd[t] = gc_residual_desc{0u, 0u, 0, 0.0f, 0ull, 0ull};
}

}  // namespace gc

extern "C" gc_status gc_ef_residual_materialize(const gc_layout* dev, const gc_layout* host, float* e,
                                                gc_residual_desc* rd, void* stream) {
  NvtxRange nvtx_range("gc_ef_residual_materialize");
  const gc_status st = validate_layout(host, false);
  if (st != GC_OK) return st;
  if (!dev || !dev->off || dev->num_tensors != host->num_tensors || !e || !rd) return GC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int T = host->num_tensors;
  k_materialize<<<dim3(256, (unsigned)std::min(T, 65535)), 256, 0, s>>>(dev->off, T, e, rd);
  k_clear_desc<<<(T + 255) / 256, 256, 0, s>>>(rd, T);
  return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

extern "C" gc_status gc_ef_threshold_compress(const gc_layout* dev, const gc_layout* host,
                                              const float* g, float* e, const float* tau,
                                              int64_t* count, int32_t* idx, float* val, int8_t* q,
                                              float* scale, uint64_t seed, uint64_t iter,
                                              uint32_t flags, void* workspace, size_t ws_bytes,
                                              void* stream) {
  NvtxRange nvtx_range("gc_ef_threshold_compress");
  const uint32_t known = GC_EF | GC_INT8 | GC_FORCE_EXACT;
  if (flags & ~known) return GC_ERR_INVALID_ARG;
  if (!tau || !count) return GC_ERR_INVALID_ARG;
  if ((flags & GC_EF) && !e) return GC_ERR_INVALID_ARG;
  return run_topk(MODE_TOPK, dev, host, g, (flags & GC_EF) ? e : nullptr, nullptr, nullptr, 0.0f,
                  idx, val, q, scale, seed, iter, flags, workspace, ws_bytes, stream, PhaseEvents{},
                  nullptr, tau, count);
}

extern "C" gc_status gc_ef_topk_compress_clipped(const gc_layout* dev, const gc_layout* host,
                                                 const float* g, float* e, const float* max_norm,
                                                 float* norm, int32_t* idx, float* val, int8_t* q,
                                                 float* scale, uint64_t seed, uint64_t iter,
                                                 uint32_t flags, void* workspace, size_t ws_bytes,
                                                 void* stream) {
  NvtxRange nvtx_range("gc_ef_topk_compress_clipped");
  const uint32_t known = GC_EF | GC_INT8 | GC_FORCE_EXACT;
  if (flags & ~known) return GC_ERR_INVALID_ARG;
  if (!(flags & GC_EF) || !e || !max_norm || !norm) return GC_ERR_INVALID_ARG;
  return run_topk(MODE_TOPK, dev, host, g, e, nullptr, nullptr, 0.0f, idx, val, q, scale, seed, iter,
                  flags, workspace, ws_bytes, stream, PhaseEvents{}, nullptr, nullptr, nullptr,
                  max_norm, norm);
}
