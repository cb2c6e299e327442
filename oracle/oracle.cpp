// Oracle for error-feedback gradient compression.
//
// TEST INFRASTRUCTURE ONLY.  This file defines, slowly and plainly, what the
// GPU library must compute.  Only the tests, the smoke check and the
// benchmark's CPU-baseline leg may load it.  It shares no code, header,
// table or constant with the CUDA library and includes nothing from it.
//
// Everything is single-threaded and written in the order the method states
// it.  fp32 arithmetic is IEEE binary32 round-to-nearest-even, one rounding
// per written operation: this file must be built with -ffp-contract=off so
// that no a*b+c is fused.  Reductions that the method leaves unspecified are
// taken in fp64, in index order.
//
// Sources (page titles and sections):
//  [P1] inferensys.com "Gradient Compression" (zh glossary): Top-k, Random-k,
//       quantization (SignSGD, stochastic quantization), error feedback,
//       "Top-k + 8-bit" pipeline, all-gather of sparse payloads.
//  [P3] inferensys.com "Gradient Compression" (genomic glossary): per-layer
//       Top-k, 8-bit quantization (4x), stochastic rounding, QSGD, DGC
//       momentum correction and momentum factor masking.
//  [P4] mbrenndoerfer.com "Gradient Compression": eq. TopK(g_t + e_{t-1}),
//       residual eq. e_t = (g_t + e_{t-1}) - g^_t, sparse wire format
//       (fp32 value + int32 index), 1-bit SGD eq. sign(g)*||g||_1/d with a
//       per-layer scalar, QSGD eq. Q_s(g) and its stochastic-rounding toy
//       example (0.3 sent as 1 with probability 0.3).
//  [P5] inferensys.com "Gradient Sparsification": per-layer selection,
//       momentum correction (velocity from the dense local gradient),
//       momentum factor masking.
//
// Readings taken where the pages are silent (each is restated in the design
// notes): k_t = min(n_t, ceil(rho n_t)) is an input; ties in |x| go to the
// lower index and +0/-0 tie; payload indices are tensor-local int32 in
// ascending order; random draws come from Philox4x32-10 with
// counter (lo32(i/4), hi32(i/4), lo32(iter), purpose), key (lo32(seed),
// hi32(seed)) and word i mod 4, i the element's arena index; stochastic
// rounding acts on the magnitude and rounds up iff r * 2^-32 < frac.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------- bit views
inline uint32_t bits_of(float x) {
  uint32_t u;
  std::memcpy(&u, &x, sizeof u);
  return u;
}
inline float float_of(uint32_t u) {
  float x;
  std::memcpy(&x, &u, sizeof x);
  return x;
}
// |x| ordering key: the IEEE bit pattern without its sign bit.  For finite x
// this orders by magnitude; +0 and -0 get the same key.
inline uint32_t magnitude_key(float x) { return bits_of(x) & 0x7FFFFFFFu; }

// ---------------------------------------------------------------- Philox
// Philox4x32-10 as published by Salmon, Moraes, Dror and Shaw, "Parallel
// Random Numbers: As Easy as 1, 2, 3" (SC'11): ten rounds of the S-box
// (two 32x32->64 multiplies by the round multipliers, xor of the high
// halves with the other counter words and the key), with the key bumped by
// the Weyl constants between rounds.
void philox4x32_10(uint32_t ctr[4], uint32_t key[2]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t p0 = (uint64_t)M0 * (uint64_t)ctr[0];
    uint64_t p1 = (uint64_t)M1 * (uint64_t)ctr[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ ctr[1] ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ ctr[3] ^ k1;
    uint32_t n3 = lo0;
    ctr[0] = n0; ctr[1] = n1; ctr[2] = n2; ctr[3] = n3;
    k0 += W0;
    k1 += W1;
  }
}

// The random word for element i (arena index) of call (seed, iter) and use
// `purpose` (1: int8 stochastic rounding, 2: QSGD, 3: random-k keys).
uint32_t draw_u32(uint64_t seed, uint64_t iter, uint64_t i, uint32_t purpose) {
  uint64_t block = i >> 2;
  uint32_t ctr[4] = {(uint32_t)block, (uint32_t)(block >> 32), (uint32_t)iter, purpose};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  philox4x32_10(ctr, key);
  return ctr[i & 3];
}

const uint32_t PURPOSE_INT8 = 1, PURPOSE_QSGD = 2, PURPOSE_RANDK = 3;

// ---------------------------------------------------------------- rounding
// Stochastic rounding of x >= 0 to floor(x) or floor(x)+1 ([P4] QSGD section
// and its 0.3 example; [P1] stochastic quantization): round up with
// probability equal to the fractional part.  With r uniform on 32-bit words
// the test "r / 2^32 < frac" has exactly that probability (to 2^-32).  Both
// sides of the comparison are exact in double.
double stochastic_round(float x, uint32_t r) {
  float f = std::floor(x);
  float frac = x - f;  // exact: f <= x < f + 1 and both are fp32
  bool up = (double)r < (double)frac * 4294967296.0;
  return (double)f + (up ? 1.0 : 0.0);
}

// ---------------------------------------------------------------- selection
// Top-k order ([P4] TopK, [P1] Top-k): element i precedes j iff
// key_i > key_j, or the keys are equal and i < j.  This is a strict total
// order, so the first k elements are unique.
struct LargerFirst {
  const uint32_t* key;
  bool operator()(int64_t a, int64_t b) const {
    if (key[a] != key[b]) return key[a] > key[b];
    return a < b;
  }
};
// Random-k order ([P1] Random-k): the k smallest random keys, ties to the
// lower index.
struct SmallerFirst {
  const uint32_t* key;
  bool operator()(int64_t a, int64_t b) const {
    if (key[a] != key[b]) return key[a] < key[b];
    return a < b;
  }
};

// Returns the selected positions in ascending index order.
//   method 0: full sort of all n positions (brute force)
//   method 1: std::nth_element, then sort the first k by index
template <class Order>
std::vector<int64_t> select_k(int64_t n, int64_t k, const uint32_t* key, int method) {
  std::vector<int64_t> pos(n);
  for (int64_t i = 0; i < n; ++i) pos[i] = i;
  Order order{key};
  if (k <= 0) return {};
  if (k >= n) return pos;
  if (method == 0) {
    std::sort(pos.begin(), pos.end(), order);
  } else {
    std::nth_element(pos.begin(), pos.begin() + (k - 1), pos.end(), order);
  }
  pos.resize(k);
  std::sort(pos.begin(), pos.end());
  return pos;
}

// int8 stochastic quantization of one value with scale s (> 0):
// q = sgn(x) * min(127, SR(|x| / s)).  s == 0 gives q = 0.
int8_t int8_code(float x, float s, uint32_t r) {
  if (s == 0.0f) return 0;
  float y = std::fabs(x) / s;
  double m = stochastic_round(y, r);
  if (m > 127.0) m = 127.0;
  int v = (int)m;
  return (int8_t)(std::signbit(x) ? -v : v);
}

}  // namespace

extern "C" {

// ------------------------------------------------------------------ Philox
void oracle_philox4x32_10(const uint32_t* ctr_in, const uint32_t* key_in, uint32_t* out) {
  uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
  uint32_t k[2] = {key_in[0], key_in[1]};
  philox4x32_10(c, k);
  for (int j = 0; j < 4; ++j) out[j] = c[j];
}

void oracle_draw_u32(uint64_t seed, uint64_t iter, uint64_t first, int64_t count, uint32_t purpose,
                     uint32_t* out) {
  for (int64_t j = 0; j < count; ++j) out[j] = draw_u32(seed, iter, first + (uint64_t)j, purpose);
}

double oracle_stochastic_round(float x, uint32_t r) { return stochastic_round(x, r); }

// ------------------------------------------------------------------ selection
// largest = 1: Top-k by key (descending, ties to lower index);
// largest = 0: the k smallest keys (ties to lower index).
int oracle_select(int64_t n, int64_t k, const uint32_t* key, int32_t largest, int32_t method,
                  int64_t* out_pos) {
  if (n < 0 || k < 0 || k > n) return 1;
  std::vector<int64_t> s = largest ? select_k<LargerFirst>(n, k, key, method)
                                   : select_k<SmallerFirst>(n, k, key, method);
  for (size_t j = 0; j < s.size(); ++j) out_pos[j] = s[j];
  return 0;
}

// ------------------------------------------------------------------ EF Top-k
// One tensor of n elements whose first element has arena index `base`.
//   acc = g + e          ([P4] eq. TopK(g_t + e_{t-1}); EF off when e == NULL)
//   S   = Top-k of acc by |acc|
//   payload: idx = S in ascending order, val = acc[S]  ([P4] wire format)
//   e'  = acc off S, +0 on S  ([P4] residual eq.)
// With int8 ([P1] "Top-k + 8-bit" pipeline; [P3] 8-bit quantization and
// stochastic rounding): s = M / 127 with M the largest kept |acc| (the
// tensor's largest |acc|), q = sgn * min(127, SR(|acc| / s)),
// v' = q * s, e'[S] = acc - v' (the residual keeps the quantization error).
// `val`, when given, receives acc (fp32 mode) or v' (int8 mode).
int oracle_ef_topk_tensor(int64_t n, int64_t k, uint64_t base, const float* g, float* e,
                          int32_t* idx, float* val, int8_t* q, float* scale, uint64_t seed,
                          uint64_t iter, int32_t use_int8, int32_t method) {
  if (n < 0 || k < 0 || k > n) return 1;
  if (use_int8 && (!q || !scale)) return 1;
  std::vector<float> acc(n);
  for (int64_t i = 0; i < n; ++i) acc[i] = e ? g[i] + e[i] : g[i];
  std::vector<uint32_t> key(n);
  for (int64_t i = 0; i < n; ++i) key[i] = magnitude_key(acc[i]);
  std::vector<int64_t> S = select_k<LargerFirst>(n, k, key.data(), method);

  float s = 0.0f;
  if (use_int8) {
    uint32_t M = 0;
    for (int64_t i : S) M = std::max(M, key[i]);
    s = float_of(M) / 127.0f;
    *scale = s;
  }
  if (e)
    for (int64_t i = 0; i < n; ++i) e[i] = acc[i];
  for (size_t j = 0; j < S.size(); ++j) {
    int64_t i = S[j];
    idx[j] = (int32_t)i;
    if (use_int8) {
      int8_t c = int8_code(acc[i], s, draw_u32(seed, iter, base + (uint64_t)i, PURPOSE_INT8));
      float v = (float)c * s;
      q[j] = c;
      if (val) val[j] = v;
      if (e) e[i] = acc[i] - v;
    } else {
      if (val) val[j] = acc[i];
      if (e) e[i] = 0.0f;
    }
  }
  return 0;
}

// ------------------------------------------------------------------ clipping
// DGC local gradient clipping ([P3] DGC bullets: local gradient clipping
// normalizes the gradient magnitude before compression; [P1] gradient
// clipping is applied before quantization to control range), per tensor:
//   N = (float)sqrt(sum g^2)  (fp64 sum in index order)
//   g' = (N > C) ? (C / N) * g : g     (C / N rounded to fp32 first)
// then EF Top-k of g' (with int8 if requested).  norm_given != NULL
// replaces the computed N (to compare against a norm reduced elsewhere).
int oracle_clip_topk_tensor(int64_t n, int64_t k, uint64_t base, const float* g, float* e,
                            float max_norm, const float* norm_given, float* norm_out, int32_t* idx,
                            float* val, int8_t* q, float* scale, uint64_t seed, uint64_t iter,
                            int32_t use_int8) {
  if (n < 0 || k < 0 || k > n || !(max_norm >= 0.0f)) return 1;
  double ss = 0.0;
  for (int64_t i = 0; i < n; ++i) ss += (double)g[i] * (double)g[i];
  float N = (float)std::sqrt(ss);
  if (norm_out) *norm_out = N;
  if (norm_given) N = *norm_given;
  std::vector<float> gc(g, g + n);
  if (N > max_norm) {
    const float c = max_norm / N;
    for (int64_t i = 0; i < n; ++i) gc[i] = c * g[i];
  }
  return oracle_ef_topk_tensor(n, k, base, gc.data(), e, idx, val, q, scale, seed, iter, use_int8, 1);
}

// ------------------------------------------------------------------ threshold
// Threshold sparsification ([P3] "Threshold-based": gradients below a fixed
// or adaptive magnitude threshold are dropped; [P5] the threshold is
// dynamic): S = {i : |acc_i| >= tau}; if more than kmax elements pass, only
// the kmax largest are kept (Top-kmax, same order as Top-k).  Payload and
// residual as in EF Top-k.  Returns the number kept in *count.
int oracle_threshold_tensor(int64_t n, int64_t kmax, float tau, uint64_t base, const float* g,
                            float* e, int32_t* idx, float* val, int8_t* q, float* scale,
                            int64_t* count, uint64_t seed, uint64_t iter, int32_t use_int8) {
  if (n < 0 || kmax < 0 || kmax > n || !(tau >= 0.0f)) return 1;
  int64_t passing = 0;
  for (int64_t i = 0; i < n; ++i) {
    const float acc = e ? g[i] + e[i] : g[i];
    if (std::fabs(acc) >= tau) ++passing;
  }
  const int64_t k = passing < kmax ? passing : kmax;
  *count = k;
  // the kept set is then exactly the Top-k of acc with this k
  return oracle_ef_topk_tensor(n, k, base, g, e, idx, val, q, scale, seed, iter, use_int8, 1);
}

// Warm-up schedule ([P5] warm-up: sparsification introduced gradually, the
// ratio rising by a predefined linear, exponential or step schedule over the
// first iterations; [P3] DGC warm-up training).  Density (fraction kept) at
// `step` of a warm-up of `warmup_steps`, from rho_start to rho_final:
//   kind 0 linear:      rho_start + (rho_final - rho_start) * f
//   kind 1 exponential: rho_start * (rho_final / rho_start)^f   (geometric)
//   kind 2 step:        the exponential value at the start of the current
//                       one of `stages` equal stages, f = floor(f*stages)/stages
// with f = step / warmup_steps; rho_final from step >= warmup_steps on.
double oracle_warmup_density(int64_t step, int64_t warmup_steps, double rho_start, double rho_final,
                             int32_t kind, int32_t stages) {
  if (warmup_steps <= 0 || step >= warmup_steps) return rho_final;
  if (step < 0) step = 0;
  double f = (double)step / (double)warmup_steps;
  if (kind == 2) f = std::floor(f * stages) / stages;
  if (kind == 0) return rho_start + (rho_final - rho_start) * f;
  return rho_start * std::pow(rho_final / rho_start, f);
}

// ------------------------------------------------------------------ random-k
// [P1] Random-k: a per-iteration random mask picks exactly k of the n
// elements.  The mask is the k smallest Philox keys (purpose 3), a uniform
// k-subset.
//   EF mode (unbiased == 0): acc = g + e (e may be NULL), payload acc[S],
//     e' = acc off S, +0 on S (same bookkeeping as Top-k).
//   unbiased mode: no residual; payload g[S] * c with c = (float)(n / k)
//     computed in double, so that the expectation of the sent vector is g.
int oracle_randk_tensor(int64_t n, int64_t k, uint64_t base, const float* g, float* e,
                        int32_t* idx, float* val, uint64_t seed, uint64_t iter,
                        int32_t unbiased, int32_t method) {
  if (n < 0 || k < 0 || k > n) return 1;
  if (unbiased && e) return 1;
  std::vector<uint32_t> key(n);
  for (int64_t i = 0; i < n; ++i) key[i] = draw_u32(seed, iter, base + (uint64_t)i, PURPOSE_RANDK);
  std::vector<int64_t> S = select_k<SmallerFirst>(n, k, key.data(), method);
  if (unbiased) {
    float c = k > 0 ? (float)((double)n / (double)k) : 0.0f;
    for (size_t j = 0; j < S.size(); ++j) {
      idx[j] = (int32_t)S[j];
      val[j] = g[S[j]] * c;
    }
    return 0;
  }
  std::vector<float> acc(n);
  for (int64_t i = 0; i < n; ++i) acc[i] = e ? g[i] + e[i] : g[i];
  if (e)
    for (int64_t i = 0; i < n; ++i) e[i] = acc[i];
  for (size_t j = 0; j < S.size(); ++j) {
    int64_t i = S[j];
    idx[j] = (int32_t)i;
    val[j] = acc[i];
    if (e) e[i] = 0.0f;
  }
  return 0;
}

// ------------------------------------------------------------------ momentum
// DGC momentum correction ([P3] DGC bullets; [P5] momentum correction and
// momentum factor masking):
//   u' = beta * u + g          (velocity from the dense local gradient)
//   v' = v + u'                (accumulated, error-fed update)
//   S  = Top-k of v' by |v'|;  payload v'[S] (or its int8 code, as above)
//   v'[S] = +0 (int8: v' - v'_q);  u'[S] = +0 when masking != 0.
int oracle_momentum_topk_tensor(int64_t n, int64_t k, uint64_t base, const float* g, float* u,
                                float* v, float beta, int32_t masking, int32_t* idx, float* val,
                                int8_t* q, float* scale, uint64_t seed, uint64_t iter,
                                int32_t use_int8, int32_t method) {
  if (n < 0 || k < 0 || k > n) return 1;
  if (use_int8 && (!q || !scale)) return 1;
  for (int64_t i = 0; i < n; ++i) {
    float bu = beta * u[i];
    u[i] = bu + g[i];
    v[i] = v[i] + u[i];
  }
  std::vector<uint32_t> key(n);
  for (int64_t i = 0; i < n; ++i) key[i] = magnitude_key(v[i]);
  std::vector<int64_t> S = select_k<LargerFirst>(n, k, key.data(), method);
  float s = 0.0f;
  if (use_int8) {
    uint32_t M = 0;
    for (int64_t i : S) M = std::max(M, key[i]);
    s = float_of(M) / 127.0f;
    *scale = s;
  }
  for (size_t j = 0; j < S.size(); ++j) {
    int64_t i = S[j];
    idx[j] = (int32_t)i;
    if (use_int8) {
      int8_t c = int8_code(v[i], s, draw_u32(seed, iter, base + (uint64_t)i, PURPOSE_INT8));
      float d = (float)c * s;
      q[j] = c;
      if (val) val[j] = d;
      v[i] = v[i] - d;
    } else {
      if (val) val[j] = v[i];
      v[i] = 0.0f;
    }
    if (masking) u[i] = 0.0f;
  }
  return 0;
}

// ------------------------------------------------------------------ quantized kept values
// QSGD or sign quantization applied after Top-k ([P4] QSGD eq.
// Q_s(g) = ||g|| sgn(g) xi(g, s) and its stochastic rounding; [P4] 1-bit SGD
// eq. sign(g) ||g||_1 / d with one scalar; [P1] the Top-k + 8-bit pipeline,
// quantization applied to the values that sparsification kept).  The
// quantized vector is the kept one: its d entries are the k kept values x_j,
// in ascending index order.
//   kind 2, QSGD: N = (float)sqrt(sum_j x_j^2) (fp64 in index order);
//     y = (|x_j| * s_levels) / N; level = min(s_levels, SR(y)) with the
//     Philox word of purpose 2 at the element's arena index; code =
//     sgn * level (int8); decoded value sgn * ((level * N) / s_levels).
//     N == 0 gives level 0.
//   kind 3, sign: mu = (float)(sum_j |x_j| / k) (fp64 in index order, 0 when
//     k == 0); bit j = 1 iff x_j has a clear sign bit, packed LSB-first 32 per
//     word (pad bits 0); decoded value bit ? mu : -mu.
// res[i] (the EF residual or the velocity) becomes x - decoded on the kept
// set.  scale_given != NULL replaces the computed N or mu.
namespace {
const int32_t KEPT_QSGD = 2, KEPT_SIGN = 3;

int quantize_kept(int32_t kind, int32_t s_levels, const std::vector<int64_t>& S, const float* x,
                  float* res, uint64_t base, uint64_t seed, uint64_t iter, int8_t* q, uint32_t* bits,
                  float* val, float* scale_out, const float* scale_given) {
  const int64_t k = (int64_t)S.size();
  float sc;
  if (kind == KEPT_QSGD) {
    double ss = 0.0;
    for (int64_t i : S) ss += (double)x[i] * (double)x[i];
    sc = (float)std::sqrt(ss);
  } else {
    double sa = 0.0;
    for (int64_t i : S) sa += std::fabs((double)x[i]);
    sc = k > 0 ? (float)(sa / (double)k) : 0.0f;
  }
  if (scale_out) *scale_out = sc;
  if (scale_given) sc = *scale_given;
  if (kind == KEPT_SIGN)
    for (int64_t w = 0; w < (k + 31) / 32; ++w) bits[w] = 0u;
  for (int64_t j = 0; j < k; ++j) {
    const int64_t i = S[j];
    const bool neg = std::signbit(x[i]);
    float d;
    if (kind == KEPT_QSGD) {
      int level = 0;
      if (sc != 0.0f) {
        const float y = (std::fabs(x[i]) * (float)s_levels) / sc;
        double m = stochastic_round(y, draw_u32(seed, iter, base + (uint64_t)i, PURPOSE_QSGD));
        if (m > (double)s_levels) m = (double)s_levels;
        level = (int)m;
      }
      q[j] = (int8_t)(neg ? -level : level);
      const float mag = ((float)level * sc) / (float)s_levels;
      d = neg ? -mag : mag;
    } else {
      if (!neg) bits[j / 32] |= 1u << (j % 32);
      d = neg ? -sc : sc;
    }
    if (val) val[j] = d;
    if (res) res[i] = x[i] - d;
  }
  return 0;
}
}  // namespace

// EF Top-k, then QSGD (kind 2) or sign (kind 3) of the kept values:
//   acc = g + e (e may be NULL: no EF); S = Top-k of acc by |acc|;
//   idx = S ascending; codes / bits and scale[0] of quantize_kept over acc[S];
//   e' = acc off S, acc - decoded on S (the residual keeps the quantization
//   error, as with int8).  `val`, when given, receives the decoded values.
int oracle_ef_topk_quantized_tensor(int64_t n, int64_t k, uint64_t base, const float* g, float* e,
                                    int32_t* idx, float* val, int8_t* q, uint32_t* bits,
                                    float* scale_out, const float* scale_given, int32_t kind,
                                    int32_t s_levels, uint64_t seed, uint64_t iter, int32_t method) {
  if (n < 0 || k < 0 || k > n) return 1;
  if (kind != KEPT_QSGD && kind != KEPT_SIGN) return 1;
  if (kind == KEPT_QSGD && (!q || s_levels < 1 || s_levels > 127)) return 1;
  if (kind == KEPT_SIGN && !bits) return 1;
  std::vector<float> acc(n);
  for (int64_t i = 0; i < n; ++i) acc[i] = e ? g[i] + e[i] : g[i];
  std::vector<uint32_t> key(n);
  for (int64_t i = 0; i < n; ++i) key[i] = magnitude_key(acc[i]);
  std::vector<int64_t> S = select_k<LargerFirst>(n, k, key.data(), method);
  for (size_t j = 0; j < S.size(); ++j) idx[j] = (int32_t)S[j];
  std::vector<float> res(acc);
  quantize_kept(kind, s_levels, S, acc.data(), res.data(), base, seed, iter, q, bits, val, scale_out,
                scale_given);
  if (e)
    for (int64_t i = 0; i < n; ++i) e[i] = res[i];
  return 0;
}

// Momentum correction + Top-k, then QSGD or sign of the kept velocity
// (the update of oracle_momentum_topk_tensor; v'[S] = v' - decoded, u'[S] = +0
// with masking).
int oracle_momentum_topk_quantized_tensor(int64_t n, int64_t k, uint64_t base, const float* g,
                                          float* u, float* v, float beta, int32_t masking,
                                          int32_t* idx, float* val, int8_t* q, uint32_t* bits,
                                          float* scale_out, const float* scale_given, int32_t kind,
                                          int32_t s_levels, uint64_t seed, uint64_t iter,
                                          int32_t method) {
  if (n < 0 || k < 0 || k > n) return 1;
  if (kind != KEPT_QSGD && kind != KEPT_SIGN) return 1;
  if (kind == KEPT_QSGD && (!q || s_levels < 1 || s_levels > 127)) return 1;
  if (kind == KEPT_SIGN && !bits) return 1;
  for (int64_t i = 0; i < n; ++i) {
    float bu = beta * u[i];
    u[i] = bu + g[i];
    v[i] = v[i] + u[i];
  }
  std::vector<uint32_t> key(n);
  for (int64_t i = 0; i < n; ++i) key[i] = magnitude_key(v[i]);
  std::vector<int64_t> S = select_k<LargerFirst>(n, k, key.data(), method);
  for (size_t j = 0; j < S.size(); ++j) idx[j] = (int32_t)S[j];
  std::vector<float> x(v, v + n);
  quantize_kept(kind, s_levels, S, x.data(), v, base, seed, iter, q, bits, val, scale_out, scale_given);
  if (masking)
    for (int64_t i : S) u[i] = 0.0f;
  return 0;
}

// ------------------------------------------------------------------ sign
// 1-bit SGD ([P4] eq. Q(g) = sign(g) ||g||_1 / d, with a per-layer scalar):
//   acc = g + e (EF; e may be NULL)
//   mu  = (float)(sum_i |acc_i| / n), the sum in fp64 in index order
//   bit i = 1 iff acc_i has a clear sign bit (sign(+0) = +1), packed
//   LSB-first 32 per word, pad bits 0
//   e'  = acc - (bit ? mu : -mu)
// If mu_given != NULL it replaces the computed mu (used to compare bits and
// residuals against a scale produced elsewhere).
int oracle_sign_tensor(int64_t n, const float* g, float* e, uint32_t* bits, float* mu_out,
                       const float* mu_given) {
  if (n <= 0) return 1;
  std::vector<float> acc(n);
  for (int64_t i = 0; i < n; ++i) acc[i] = e ? g[i] + e[i] : g[i];
  double sum = 0.0;
  for (int64_t i = 0; i < n; ++i) sum += std::fabs((double)acc[i]);
  float mu = (float)(sum / (double)n);
  if (mu_given) mu = *mu_given;
  if (mu_out) *mu_out = (float)(sum / (double)n);
  int64_t words = (n + 31) / 32;
  for (int64_t w = 0; w < words; ++w) bits[w] = 0u;
  for (int64_t i = 0; i < n; ++i) {
    bool pos = !std::signbit(acc[i]);
    if (pos) bits[i / 32] |= (1u << (i % 32));
    if (e) e[i] = acc[i] - (pos ? mu : -mu);
  }
  return 0;
}

// ------------------------------------------------------------------ dense SR
// mode 0, int8 ([P3] 8-bit quantization, stochastic rounding):
//   s = M / 127, M = max |acc|; code = sgn * min(127, SR(|acc| / s)).
// mode 1, QSGD ([P4] eq. Q_s(g) = ||g|| sgn(g) xi(g, s)):
//   N = (float)sqrt(sum acc^2) (fp64 sum in index order);
//   x = (|acc| * s_levels) / N; level = min(s_levels, SR(x));
//   code = sgn * level; decoded value sgn * ((level * N) / s_levels).
// acc = g + e when e != NULL, and then e' = acc - decoded (EF).
// scale_given != NULL replaces the computed s or N.
int oracle_quantize_tensor(int64_t n, uint64_t base, const float* g, float* e, int8_t* codes,
                           float* scale_out, int32_t mode, int32_t s_levels, uint64_t seed,
                           uint64_t iter, const float* scale_given) {
  if (n <= 0) return 1;
  if (mode == 1 && (s_levels < 1 || s_levels > 127)) return 1;
  std::vector<float> acc(n);
  for (int64_t i = 0; i < n; ++i) acc[i] = e ? g[i] + e[i] : g[i];
  float sc;
  if (mode == 0) {
    uint32_t M = 0;
    for (int64_t i = 0; i < n; ++i) M = std::max(M, magnitude_key(acc[i]));
    sc = float_of(M) / 127.0f;
  } else {
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) ss += (double)acc[i] * (double)acc[i];
    sc = (float)std::sqrt(ss);
  }
  if (scale_out) *scale_out = sc;
  if (scale_given) sc = *scale_given;
  for (int64_t i = 0; i < n; ++i) {
    float d;
    if (mode == 0) {
      int8_t c = int8_code(acc[i], sc, draw_u32(seed, iter, base + (uint64_t)i, PURPOSE_INT8));
      codes[i] = c;
      d = (float)c * sc;
    } else {
      int level = 0;
      if (sc != 0.0f) {
        float x = (std::fabs(acc[i]) * (float)s_levels) / sc;
        double m = stochastic_round(x, draw_u32(seed, iter, base + (uint64_t)i, PURPOSE_QSGD));
        if (m > (double)s_levels) m = (double)s_levels;
        level = (int)m;
      }
      int c = std::signbit(acc[i]) ? -level : level;
      codes[i] = (int8_t)c;
      float mag = ((float)level * sc) / (float)s_levels;
      d = std::signbit(acc[i]) ? -mag : mag;
    }
    if (e) e[i] = acc[i] - d;
  }
  return 0;
}

// ------------------------------------------------------------------ PowerSGD
// PowerSGD with error feedback ([P4] PowerSGD section: G ~ P Q^T with
// P (m x r), Q (n x r), found by power iteration that alternates between
// updating P and Q, with error feedback on the residual G - P Q^T; [P2]
// rank-4 PowerSGD; [P3] low-rank compression).  One power-iteration step per
// call, warm-started from the previous call's Q (row-major n x r):
//   M = G + E                                         (fp32)
//   P = M Q            P_ik = (float) sum_j M_ij Q_jk (fp64 sum, j ascending)
//   orthonormalize P's columns (modified Gram-Schmidt), k = 0..r-1:
//     for j < k: d = (float) sum_i P_ij P_ik (fp64);  P_ik = P_ik - d * P_ij
//     nrm = (float) sqrt(sum_i P_ik^2) (fp64);  if nrm > 0: P_ik = P_ik / nrm
//   Q = M^T P          Q_jk = (float) sum_i M_ij P_ik (fp64 sum, i ascending)
//   E = M - P Q^T      with s_ij = 0; s_ij = s_ij + P_ik * Q_jk for k = 0..r-1 (fp32)
// G, E are row-major m x n; P is row-major m x r.  p_raw_out receives P
// before orthonormalization.  p_raw_given, p_given, q_given replace the
// computed P (before / after orthonormalization) and Q: used to compare
// each later step against values reduced elsewhere.
namespace {
double dot_rows(int64_t len, const float* a, int64_t sa, const float* b, int64_t sb) {
  double s = 0.0;
  for (int64_t i = 0; i < len; ++i) s += (double)a[i * sa] * (double)b[i * sb];
  return s;
}
}  // namespace

int oracle_powersgd_tensor(int64_t m, int64_t n, int32_t r, const float* g, float* e, float* q,
                           float* p, float* p_raw_out, const float* p_raw_given,
                           const float* p_given, const float* q_given) {
  if (m < 1 || n < 1 || r < 1 || r > 8) return 1;
  std::vector<float> M(m * n);
  for (int64_t x = 0; x < m * n; ++x) M[x] = g[x] + e[x];
  // P = M Q
  for (int64_t i = 0; i < m; ++i)
    for (int32_t k = 0; k < r; ++k) p[i * r + k] = (float)dot_rows(n, &M[i * n], 1, q + k, r);
  if (p_raw_out)
    for (int64_t x = 0; x < m * r; ++x) p_raw_out[x] = p[x];
  if (p_raw_given)
    for (int64_t x = 0; x < m * r; ++x) p[x] = p_raw_given[x];
  // modified Gram-Schmidt
  for (int32_t k = 0; k < r; ++k) {
    for (int32_t j = 0; j < k; ++j) {
      const float d = (float)dot_rows(m, p + j, r, p + k, r);
      for (int64_t i = 0; i < m; ++i) p[i * r + k] = p[i * r + k] - d * p[i * r + j];
    }
    const float nrm = (float)std::sqrt(dot_rows(m, p + k, r, p + k, r));
    if (nrm > 0.0f)
      for (int64_t i = 0; i < m; ++i) p[i * r + k] = p[i * r + k] / nrm;
  }
  if (p_given)
    for (int64_t x = 0; x < m * r; ++x) p[x] = p_given[x];
  // Q = M^T P
  for (int64_t jcol = 0; jcol < n; ++jcol)
    for (int32_t k = 0; k < r; ++k) q[jcol * r + k] = (float)dot_rows(m, &M[jcol], n, p + k, r);
  if (q_given)
    for (int64_t x = 0; x < n * r; ++x) q[x] = q_given[x];
  // E = M - P Q^T
  for (int64_t i = 0; i < m; ++i)
    for (int64_t jcol = 0; jcol < n; ++jcol) {
      float s = 0.0f;
      for (int32_t k = 0; k < r; ++k) s = s + p[i * r + k] * q[jcol * r + k];
      e[i * n + jcol] = M[i * n + jcol] - s;
    }
  return 0;
}

// Receiver of a PowerSGD payload: out += P Q^T (same fp32 accumulation).
int oracle_powersgd_decode_accumulate(int64_t m, int64_t n, int32_t r, const float* p,
                                      const float* q, float* out) {
  for (int64_t i = 0; i < m; ++i)
    for (int64_t jcol = 0; jcol < n; ++jcol) {
      float s = 0.0f;
      for (int32_t k = 0; k < r; ++k) s = s + p[i * r + k] * q[jcol * r + k];
      out[i * n + jcol] = out[i * n + jcol] + s;
    }
  return 0;
}

// ------------------------------------------------------------------ receivers
// Sum of W workers' sparse payloads into a dense arena ([P4]: the received
// gradient is the union of different sparse vectors; [P1]: all-gather of
// indices and values, then a local sum).  Workers are applied in order
// w = 0..W-1, tensors in order, entries in payload order; out += value with
// value = val (fp32) or q * scale[t] (int8).
int oracle_sparse_accumulate(int32_t T, const int64_t* off, const int64_t* koff, int32_t W,
                             const int32_t* const* idx, const float* const* val,
                             const int8_t* const* q, const float* const* scale, float* out) {
  for (int32_t w = 0; w < W; ++w) {
    for (int32_t t = 0; t < T; ++t) {
      int64_t n = off[t + 1] - off[t];
      for (int64_t j = koff[t]; j < koff[t + 1]; ++j) {
        int64_t i = idx[w][j];
        if (i < 0 || i >= n) return 2;
        float v = val ? val[w][j] : (float)q[w][j] * scale[w][t];
        out[off[t] + i] = out[off[t] + i] + v;
      }
    }
  }
  return 0;
}

// Receiver of W workers' quantized sparse payloads (the payloads of the
// quantized kept values above): as oracle_sparse_accumulate, with entry j of
// tensor t (j counted from koff[t]) decoded from its code:
//   kind 1, int8: q * scale[t]
//   kind 2, QSGD: sgn(q) * ((|q| * scale[t]) / s_levels), +0 for q = 0
//   kind 3, sign: bit j of tensor t's words ? scale[t] : -scale[t], tensor t's
//     words starting at sum_{t' < t} ceil(k_t' / 32).
int oracle_sparse_accumulate_quantized(int32_t T, const int64_t* off, const int64_t* koff, int32_t W,
                                       const int32_t* const* idx, const int8_t* const* q,
                                       const uint32_t* const* bits, const float* const* scale,
                                       int32_t kind, int32_t s_levels, float* out) {
  if (kind < 1 || kind > 3 || (kind == 2 && (s_levels < 1 || s_levels > 127))) return 1;
  for (int32_t w = 0; w < W; ++w) {
    int64_t word0 = 0;  // first sign-bit word of tensor t
    for (int32_t t = 0; t < T; ++t) {
      const int64_t n = off[t + 1] - off[t];
      for (int64_t p = koff[t]; p < koff[t + 1]; ++p) {
        const int64_t i = idx[w][p];
        if (i < 0 || i >= n) return 2;
        const float sc = scale[w][t];
        float v;
        if (kind == 1) {
          v = (float)q[w][p] * sc;
        } else if (kind == 2) {
          const int c = q[w][p];
          const int level = c < 0 ? -c : c;
          const float mag = ((float)level * sc) / (float)s_levels;
          v = c < 0 ? -mag : mag;
        } else {
          const int64_t j = p - koff[t];
          const bool bit = (bits[w][word0 + j / 32] >> (j % 32)) & 1u;
          v = bit ? sc : -sc;
        }
        out[off[t] + i] = out[off[t] + i] + v;
      }
      word0 += (koff[t + 1] - koff[t] + 31) / 32;
    }
  }
  return 0;
}

// Dense receivers: out += decode(payload) for one tensor.
//   sign: bit ? mu : -mu
//   int8: code * s
//   QSGD: sgn(code) * ((|code| * N) / s_levels)
int oracle_sign_decode_accumulate(int64_t n, const uint32_t* bits, float mu, float* out) {
  for (int64_t i = 0; i < n; ++i) {
    bool pos = (bits[i / 32] >> (i % 32)) & 1u;
    out[i] = out[i] + (pos ? mu : -mu);
  }
  return 0;
}

int oracle_codes_decode_accumulate(int64_t n, const int8_t* codes, float sc, int32_t mode,
                                   int32_t s_levels, float* out) {
  for (int64_t i = 0; i < n; ++i) {
    float d;
    if (mode == 0) {
      d = (float)codes[i] * sc;
    } else {
      int level = codes[i] < 0 ? -codes[i] : codes[i];
      float mag = ((float)level * sc) / (float)s_levels;
      d = codes[i] < 0 ? -mag : mag;
    }
    out[i] = out[i] + d;
  }
  return 0;
}

}  // extern "C"
