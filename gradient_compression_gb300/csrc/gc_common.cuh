// Device helpers shared by the libgc kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gc.h"

namespace gc {

constexpr unsigned FULL = 0xffffffffu;

// ---------------------------------------------------------------- chained launches
// The kernels of one call run back to back in one stream.  Each is issued as
// a programmatic dependent launch (launch_chained) and starts with
// chain_wait(): the wait returns once the kernels before it in the stream
// have completed and their writes are visible (at once for a plain launch),
// and the trigger after it lets the next kernel's CTAs be scheduled while
// this grid's last CTAs run, so the launch gap between two phases is hidden
// without any change to what either reads or writes.
__device__ __forceinline__ void chain_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// kern<<<grid, block, smem, s>>>(args...) as a programmatic dependent launch;
// a launch the runtime refuses with that attribute is issued plainly (a
// configuration error then stays for the caller's cudaGetLastError).
template <typename... P, typename... Arg>
static void launch_chained(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                           const Arg&... args) {
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, args...) != cudaSuccess) {
    (void)cudaGetLastError();
    kern<<<grid, block, smem, s>>>(args...);
  }
}

// Zeroes a call's workspace head (16-byte aligned, n16 16-byte words, then
// ntail bytes) as the first kernel of the call's chain.
static __global__ void __launch_bounds__(256) k_zero(uint4* p, size_t n16, unsigned char* tail, int ntail) {
  chain_wait();
  for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < n16; i += (size_t)gridDim.x * 256)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
  if (blockIdx.x == 0 && (int)threadIdx.x < ntail) tail[threadIdx.x] = 0;
}

// cudaMemsetAsync(p, 0, bytes, s) for a 16-byte aligned p, as a chained
// launch; false if the launch failed.
static bool zero_chained(void* p, size_t bytes, cudaStream_t s) {
  const size_t n16 = bytes / 16;
  const size_t blocks = (n16 + 255) / 256;
  const unsigned grid = blocks < 1 ? 1u : (blocks > 2048 ? 2048u : (unsigned)blocks);
  launch_chained(k_zero, grid, 256, 0, s, static_cast<uint4*>(p), n16, static_cast<unsigned char*>(p) + n16 * 16,
                 (int)(bytes % 16));
  return cudaGetLastError() == cudaSuccess;
}

// Work unit: one warp streams UNIT consecutive elements of one tensor.
constexpr int UNIT_SHIFT = 12;
constexpr int64_t UNIT = int64_t(1) << UNIT_SHIFT;
// Unit block: consecutive units of one tensor, one CTA of 8 warps in the
// selection kernels; on the candidate path a warp walks the candidate
// chunks of 1/8 of them.  UB_UNITS units per block (32 per warp), or
// UB_UNITS_DENSE (8 per warp) in arenas with many candidates per unit, where
// the longest walks set the kernels' time.
constexpr int UB_UNITS = 256;
constexpr int UB_UNITS_DENSE = 64;
// Radix digits of the 32-bit selection key: 11 + 11 + 10 bits.
constexpr int NBINS = 2048;
// Per-warp candidate staging capacity in shared memory (entries per unit).
constexpr int WCAP = 512;
// Tensors at most this long are sampled completely when the candidate
// threshold is estimated.
constexpr int64_t SMALL_N = 16384;
// Expected number of Top-k members in a tensor's sample: 128, or 64 for a
// tensor that keeps less than 0.2% of its elements, whose sample of 128 / rho
// elements would otherwise be an eighth of a 1M-element tensor.
__host__ __device__ inline int64_t sample_hits(int64_t n, int64_t k) { return 500 * k < n ? 64 : 128; }
constexpr int RUN = 128;  // sampled elements per contiguous run (one warp, one float4 per lane)
// Threshold estimate from the sample: pilot runs, shared-memory key list
// (the pilot's keys, then the keys above the pilot's floor), and the
// smallest sample that takes the filtered search.
constexpr int SPILOT = 64;
constexpr int SLIST = SPILOT * RUN;
constexpr int64_t SFILTER_RUNS = 256;

// Tensor state flags.
constexpr uint32_t TS_NOEMIT = 1u;    // k_t == 0: nothing is selected
constexpr uint32_t TS_DENSE = 2u;     // select with full passes over the tensor
constexpr uint32_t TS_OVERFLOW = 4u;  // candidate staging overflowed

// Diagnostic words at the head of every workspace.
constexpr int DIAG_ERR = 0, DIAG_EXACT = 1, DIAG_OVF = 2, DIAG_ABORT = 3, DIAG_PATH = 4;
constexpr size_t DIAG_BYTES = 256;

struct alignas(16) TensorState {
  uint32_t t_est;       // candidate threshold on the selection key
  uint32_t flags;       // TS_*
  uint32_t prefix;      // radix digits fixed so far
  uint32_t rank;        // 1-based rank still sought inside the current bucket
  uint32_t maxkey;      // largest key seen (int8 scale)
  uint32_t cand_count;  // candidates reserved by the streaming pass
  uint32_t thr;         // exact key of the k-th element
  uint32_t r_eq;        // how many elements with key == thr are kept (lowest indices)
  uint32_t keff;        // elements kept (k_t, or fewer under a threshold)
  float gmul;           // multiplier applied to g (local clipping), else 1
  uint32_t cnt_tau;     // elements with |acc| >= tau (threshold mode, full-pass path)
  uint32_t pad0;
  uint32_t s_runs;      // sample plan (set by the planner; 16-byte aligned): runs of RUN elements,
  uint32_t s_stride;    //   their spacing,
  uint32_t s_j;         //   the rank of the sample key that bounds t_est,
  uint32_t s_rp;        //   and the rank in the pilot of the filtered search
};
static_assert(sizeof(TensorState) == 64, "TensorState is 64 bytes");
static_assert(offsetof(TensorState, s_runs) % 16 == 0, "sample plan is one 16-byte load");

// ---------------------------------------------------------------- sizing
// Candidate capacity of a tensor, identical on host and device.  The sampled
// threshold yields about 1.5k candidates for a large tensor, with a relative
// spread of about 7%, so 3k + 4096 is many standard deviations above it.
__host__ __device__ inline int64_t cand_capacity(int64_t n, int64_t k) {
  if (k <= 0) return 0;
  if (n <= SMALL_N) return n;
  int64_t c = 3 * k + 4096;
  return c < n ? c : n;
}

__host__ __device__ inline int64_t units_of(int64_t n) { return (n + UNIT - 1) >> UNIT_SHIFT; }
__host__ __device__ inline int64_t ublocks_of(int64_t n, int ubu) {
  return (units_of(n) + ubu - 1) / ubu;
}

// Sample plan of a tensor: `runs` runs of RUN consecutive elements spaced
// `stride` apart (all of the tensor when it is small).  m = sampled count.
__host__ __device__ inline void sample_plan(int64_t n, int64_t k, int64_t* runs, int64_t* stride,
                                            int64_t* m) {
  if (n <= SMALL_N || k <= 0) {
    *stride = RUN;
    *runs = (n + RUN - 1) / RUN;
    *m = n;
    return;
  }
  const int64_t hits = sample_hits(n, k);
  int64_t want = (hits * n + k - 1) / k;  // ceil(hits / rho)
  int64_t r = (want + RUN - 1) / RUN;
  int64_t rmax = n / RUN;
  if (r > rmax) r = rmax;
  if (r < 1) r = 1;
  *runs = r;
  *stride = (n / r) & ~int64_t(3);  // keeps float4 alignment of every run; still >= RUN
  *m = r * RUN;
}

// CTAs that sample a tensor: one for a small sample; for a sample of at
// least SFILTER_RUNS runs, `split` of them but no fewer than
// SAMPLE_RUNS_PER_CTA runs each (each filters its share of the runs; the
// last to finish finds the threshold).  `split` spreads the arena's large
// samples over about two CTAs per SM: arenas with many large tensors keep
// one CTA per tensor.
constexpr int64_t SAMPLE_RUNS_PER_CTA = 128;
__host__ __device__ inline bool sample_splittable(int64_t n, int64_t k) {
  if (k <= 0 || k >= n) return false;
  int64_t runs, stride, m;
  sample_plan(n, k, &runs, &stride, &m);
  return runs >= SFILTER_RUNS;
}
// Tensors of at most NOSAMPLE_N elements are not sampled: every element is a
// candidate, which costs less than a sampling CTA; the bound is a warp's
// candidate staging of one unit (WCAP), so the streaming pass can stage them
// all.  A tensor with nothing to select (k = 0 or k = n) is not sampled
// either.
constexpr int64_t NOSAMPLE_N = WCAP;
__host__ __device__ inline int64_t sample_ctas(int64_t n, int64_t k, int split) {
  if (k <= 0 || k >= n || n <= NOSAMPLE_N) return 0;
  if (!sample_splittable(n, k)) return 1;
  int64_t runs, stride, m;
  sample_plan(n, k, &runs, &stride, &m);
  const int64_t most = runs / SAMPLE_RUNS_PER_CTA;
  return split < most ? (split > 1 ? split : 1) : (most > 1 ? most : 1);
}

// Element offset of sample run r inside its stride window: a hashed jitter
// (multiple of 4, run stays inside the window) so that runs of a tensor do
// not sit at a power-of-two spacing, which would map them all onto the same
// DRAM channels.  Zero when the tensor is sampled completely.
__host__ __device__ inline int64_t sample_run_start(int64_t r, int64_t stride) {
  const int64_t slack = (stride - RUN) >> 2;
  if (slack <= 0) return r * stride;
  const uint32_t h = (uint32_t)r * 2654435761u;
  return r * stride + 4 * (int64_t)(((uint64_t)h * (uint64_t)(slack + 1)) >> 32);
}

// ---------------------------------------------------------------- keys
// Top-k key: the fp32 bit pattern shifted left by one, which drops the sign
// bit; for finite values it orders by |x| and maps +0 and -0 together.
__device__ __forceinline__ uint32_t mag_key(float x) { return __float_as_uint(x) << 1; }
__device__ __forceinline__ float key_magnitude(uint32_t key) { return __uint_as_float(key >> 1); }

// ---------------------------------------------------------------- Philox
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// The four words of the block holding arena elements 4b .. 4b+3.
__device__ __forceinline__ uint4 philox_block(uint64_t seed, uint64_t iter, uint64_t b,
                                              uint32_t purpose) {
  return philox4x32_10(make_uint4((uint32_t)b, (uint32_t)(b >> 32), (uint32_t)iter, purpose),
                       (uint32_t)seed, (uint32_t)(seed >> 32));
}

__device__ __forceinline__ uint32_t uint4_word(uint4 w, int j) {
  return j == 0 ? w.x : (j == 1 ? w.y : (j == 2 ? w.z : w.w));
}

__device__ __forceinline__ uint32_t philox_word(uint64_t seed, uint64_t iter, uint64_t i,
                                                uint32_t purpose) {
  return uint4_word(philox_block(seed, iter, i >> 2, purpose), (int)(i & 3));
}

// The ten round keys of a seed, computed once on the host and passed in a
// kernel's parameters, so that each round XORs them straight from the
// parameter bank instead of stepping the key in registers.
struct PhiloxKey {
  uint32_t k[20];  // k[2r], k[2r + 1]: the two key words of round r
};

inline PhiloxKey make_philox_key(uint64_t seed) {
  PhiloxKey K;
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    K.k[2 * r] = k0;
    K.k[2 * r + 1] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return K;
}

__device__ __forceinline__ uint4 philox_block(const PhiloxKey& K, uint64_t iter, uint64_t b, uint32_t purpose) {
  uint4 c = make_uint4((uint32_t)b, (uint32_t)(b >> 32), (uint32_t)iter, purpose);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    // each 32 x 32 -> 64-bit product in one wide multiply
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x, p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ K.k[2 * r], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ K.k[2 * r + 1],
                   (uint32_t)p0);
  }
  return c;
}

__device__ __forceinline__ uint32_t philox_word(const PhiloxKey& K, uint64_t iter, uint64_t i, uint32_t purpose) {
  return uint4_word(philox_block(K, iter, i >> 2, purpose), (int)(i & 3));
}

// Philox4x32-10 blocks of one (key, iteration, purpose) whose block index b
// is below 2^32 (arenas of fewer than 2^34 elements): the counter is
// (b, 0, iter, purpose), so in the first round the product of the iteration
// word and in the second round the product of the first round's (constant)
// first word are the same for every block.  They are taken once here; the
// rounds are otherwise those of philox_block, which gives the same words.
struct PhiloxLo {
  uint32_t cp, c2, c3, c5;
  __device__ __forceinline__ PhiloxLo(const PhiloxKey& key, uint64_t iter, uint32_t purpose) {
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint32_t)iter;  // round 0: product of the iteration word
    const uint32_t x1 = (uint32_t)(p1 >> 32) ^ key.k[0];           // round 0 output x (counter y = 0)
    const uint32_t y1 = (uint32_t)p1;                              // round 0 output y
    const uint64_t q0 = (uint64_t)0xD2511F53u * x1;                // round 1: product of x
    cp = purpose ^ key.k[1];
    c2 = y1 ^ key.k[2];
    c3 = (uint32_t)(q0 >> 32) ^ key.k[3];
    c5 = (uint32_t)q0 ^ key.k[5];
  }
  // the same key as the constructor's
  __device__ __forceinline__ uint4 block(const PhiloxKey& K, uint32_t b) const {
    // round 0: x = b, y = 0, z = iter, w = purpose
    const uint64_t a0 = (uint64_t)0xD2511F53u * b;
    const uint32_t z1 = (uint32_t)(a0 >> 32) ^ cp, w1 = (uint32_t)a0;
    // round 1: its x-product is constant (c3 and, through w2, c5 carry it)
    const uint64_t a1 = (uint64_t)0xCD9E8D57u * z1;
    uint4 c = make_uint4((uint32_t)(a1 >> 32) ^ c2, (uint32_t)a1, w1 ^ c3, 0u);
    // round 2: w is round 1's constant low product, folded into c5
    {
      const uint64_t p0 = (uint64_t)0xD2511F53u * c.x, p1 = (uint64_t)0xCD9E8D57u * c.z;
      c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ K.k[4], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c5, (uint32_t)p0);
    }
#pragma unroll
    for (int r = 3; r < 10; ++r) {
      const uint64_t p0 = (uint64_t)0xD2511F53u * c.x, p1 = (uint64_t)0xCD9E8D57u * c.z;
      c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ K.k[2 * r], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ K.k[2 * r + 1],
                     (uint32_t)p0);
    }
    return c;
  }
};

constexpr uint32_t PURPOSE_INT8 = 1, PURPOSE_QSGD = 2, PURPOSE_RANDK = 3;

// Advances a device-resident iteration counter by one (the last kernel of a
// *_dev_iter call).
static __global__ void k_iter_advance(uint64_t* iter) {
  chain_wait();
  *iter += 1u;
}

// ---------------------------------------------------------------- rounding
// Stochastic rounding of 0 <= x < 2^23: floor(x) + 1 iff r * 2^-32 < frac(x),
// decided exactly.  x + 2^23 rounded toward zero is 2^23 + floor(x) (the
// sum's ulp is 1), which gives floor(x) both as an integer (its bit pattern
// minus that of 2^23) and as a float; frac = x - floor(x) and F = frac * 2^32
// are exact, and for an integer r, r < F iff r < ceil(F) <= 2^32 - 256.  One
// float-to-integer conversion per value.
__device__ __forceinline__ int stochastic_round(float x, uint32_t r) {
  const float t = __fadd_rz(x, 8388608.0f);
  const int fl = (int)(__float_as_uint(t) - 0x4B000000u);
  const float frac = __fsub_rn(x, __fsub_rn(t, 8388608.0f));
  const uint32_t c = __float2uint_ru(__fmul_rn(frac, 4294967296.0f));
  return fl + (r < c ? 1 : 0);
}

// int8 code of x for scale s (s == 0 gives 0).
__device__ __forceinline__ int int8_code(float x, float s, uint32_t r) {
  if (s == 0.0f) return 0;
  // |x| <= max|acc| keeps |x| / s near 127; the clamp (which cannot change
  // min(127, .)) only guards the float -> int conversion
  int m = stochastic_round(fminf(__fdiv_rn(fabsf(x), s), 128.0f), r);
  m = m > 127 ? 127 : m;
  return signbit(x) ? -m : m;
}

// Correctly rounded a / b for many a and one b, without a divide per a:
// with y = RN(1/b), q = RN(a y) is within one ulp of a / b, the remainder
// a - b q is exact (one FMA), and RN(q + (a - b q) y) is RN(a / b)
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  The theorem needs
// every intermediate in the normal range: b in [2^-125, 2^125], a >= 2^-100
// and q in [2^-99, 2^125]; anything else takes the IEEE division.  The
// bounds on a and q come from one per-divisor threshold on a.
struct Divisor {
  float b, rb, thr;
  // qmax: an upper bound of a / b over the values this divisor will see
  // (the fast path also needs q <= 2^125).  Values a >= thr take the fast
  // path: then a >= 2^-100 and q >= 2^-98 (1 - 2^-23) > 2^-99.
  __device__ __forceinline__ Divisor(float b_, float qmax) : b(b_) {
    const bool fast = b_ >= 0x1p-125f && b_ <= 0x1p125f && qmax <= 0x1p125f;
    rb = fast ? __frcp_rn(b_) : 0.0f;
    thr = fast ? fmaxf(0x1p-100f, __fmul_rn(b_, 0x1p-98f)) : __int_as_float(0x7f800000);
  }
  // a >= 0
  __device__ __forceinline__ float div(float a) const {
    if (a >= thr) {
      const float q = __fmul_rn(a, rb);
      return __fmaf_rn(__fmaf_rn(-q, b, a), rb, q);
    }
    if (a == 0.0f) return 0.0f;
    return __fdiv_rn(a, b);
  }
};

// ---------------------------------------------------------------- sums
// Per-lane sum of |x| (P = 1) or x^2 (P = 2) that neither overflows nor
// underflows in fp32 for any finite x: terms are taken relative to a running
// power of two 2^E that bounds every |x| seen so far (the scaled sum of
// squares of LAPACK's xLASSQ, after S. Hammarling), summed with Neumaier
// compensation, and the sum is rescaled exactly (a power of two) whenever E
// grows.  A term below 2^-126 of the bound may lose bits; its square is
// below 2^-252 of the largest square, far under fp64 resolution.
template <int P>
struct ScaledSum {
  float s = 0.0f, c = 0.0f;
  int E = -125;
  // mk: max of mag_key over the terms about to be added
  __device__ __forceinline__ void bound(uint32_t mk) {
    int eg = (int)(mk >> 24) - 126;  // |x| < 2^eg
    eg = eg < -125 ? -125 : (eg > 126 ? 126 : eg);
    if (eg > E) {
      const int sh = P * (E - eg);
      if (sh < -120) {
        s = 0.0f;  // the old terms are below 2^-110 of the new ones
        c = 0.0f;
      } else {
        const float f = __int_as_float((127 + sh) << 23);
        s = __fmul_rn(s, f);
        c = __fmul_rn(c, f);
      }
      E = eg;
    }
  }
  __device__ __forceinline__ float mult() const { return __int_as_float((127 - E) << 23); }
  __device__ __forceinline__ void add(float x, float m) {
    const float y = __fmul_rn(fabsf(x), m);
    const float v = (P == 2) ? __fmul_rn(y, y) : y;
    const float t = __fadd_rn(s, v);
    if (fabsf(s) >= v)
      c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, t), v));
    else
      c = __fadd_rn(c, __fadd_rn(__fsub_rn(v, t), s));
    s = t;
  }
  // one term at a time (tails)
  __device__ __forceinline__ void add1(float x) {
    bound(mag_key(x));
    add(x, mult());
  }
  __device__ __forceinline__ double value() const {
    return ((double)s + (double)c) * __longlong_as_double((long long)(1023 + P * E) << 52);
  }
};

// ---------------------------------------------------------------- lookup
// Largest t in [0, T) with offs[t] <= x (offs[0] <= x < offs[T]).
__device__ __forceinline__ int find_segment(const int64_t* __restrict__ offs, int T, int64_t x) {
  int lo = 0, hi = T;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(offs + mid) <= x)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------- warp scans
__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

// Exclusive prefix and total over the warp of small per-lane counts (0..7).
__device__ __forceinline__ void warp_count_scan(unsigned c, unsigned lane, unsigned* pre,
                                                unsigned* tot) {
  const unsigned b0 = __ballot_sync(FULL, c & 1u);
  const unsigned b1 = __ballot_sync(FULL, c & 2u);
  const unsigned b2 = __ballot_sync(FULL, c & 4u);
  const unsigned lt = (1u << lane) - 1u;
  *pre = __popc(b0 & lt) + 2u * __popc(b1 & lt) + 4u * __popc(b2 & lt);
  *tot = __popc(b0) + 2u * __popc(b1) + 4u * __popc(b2);
}

// Exclusive prefix and total of arbitrary per-lane unsigned values.
__device__ __forceinline__ unsigned warp_excl_scan(unsigned v, unsigned lane, unsigned* tot) {
  unsigned x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned y = __shfl_up_sync(FULL, x, d);
    if (lane >= (unsigned)d) x += y;
  }
  *tot = __shfl_sync(FULL, x, 31);
  return x - v;
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v = max(v, __shfl_xor_sync(FULL, v, d));
  return v;
}

// Shared-memory histogram add, aggregated over lanes that hit the same bin.
__device__ __forceinline__ void smem_hist_add(uint32_t* hist, uint32_t bin, bool pred) {
  const unsigned active = __ballot_sync(FULL, pred);
  if (pred) {
    const unsigned peers = __match_any_sync(active, bin);
    if ((int)lane_id() == __ffs(peers) - 1) atomicAdd(hist + bin, (uint32_t)__popc(peers));
  }
}

// Streaming (evict-first) 16-byte accesses.
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4* p, float4 v) { __stcs(p, v); }

}  // namespace gc
