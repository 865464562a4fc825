// finalize.cuh -- the last step of the factored norm for one output row:
//
//   wnorm = sqrt(max(base + 2 s cross + s^2 ba, 0)),   g = m / max(wnorm, eps)
//
// ("Scaling DoRA", Chinese write-up section 1.2.2 and Algorithm 1 of section
// 5.1; English summary "Factored Norm").  The split partials of each term are
// summed in split order; the assembly is carried in double-float arithmetic
// (a value held as hi + lo, two fp32 words: about 44 significant bits), and
// the root and the divide are each an IEEE fp32 operation refined by one
// correction step on the double-float residual, then rounded once.  No fp64
// instructions: the fp64 units are scarce on this part.
//
// Used by the stand-alone finalize kernel and by the epilogue of the CTA-pair
// main pass, which finalizes each 128-row tile as its last K split lands.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace dora {

constexpr int kMaxFinalParts = 16;   // split partials per term

// exact sum of two floats (Knuth's TwoSum)
__device__ __forceinline__ void two_sum(float a, float b, float& hi, float& lo) {
  hi = __fadd_rn(a, b);
  const float bb = __fsub_rn(hi, a);
  lo = __fadd_rn(__fsub_rn(a, __fsub_rn(hi, bb)), __fsub_rn(b, bb));
}

struct df {
  float hi, lo;
};

__device__ __forceinline__ df df_add(df a, df b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  df r;
  two_sum(s, e, r.hi, r.lo);
  return r;
}

// a * c for a float c, exact product of the hi parts (FMA-based TwoProduct)
__device__ __forceinline__ df df_mul_f(df a, float c) {
  const float p = __fmul_rn(a.hi, c);
  const float e = fmaf(a.hi, c, -p);
  df r;
  two_sum(p, fmaf(a.lo, c, e), r.hi, r.lo);
  return r;
}

// v[0] + v[1] + ... in that order, carried as a double-float
__device__ __forceinline__ df df_sum_in_order(const float (&v)[kMaxFinalParts]) {
  df acc{0.f, 0.f};
#pragma unroll
  for (int i = 0; i < kMaxFinalParts; ++i) {
    float e;
    two_sum(acc.hi, v[i], acc.hi, e);
    acc.lo = __fadd_rn(acc.lo, e);
  }
  return acc;
}

// w2 = base + two_s * cross (+ s_sq * ba); then the root and m / max(root, eps)
__device__ __forceinline__ void finalize_row(df base, df cross, const df* ba, float two_s,
                                             float s_sq, float mj, float eps, float& wnorm_out,
                                             float& g_out) {
  df w2 = df_add(base, df_mul_f(cross, two_s));
  if (ba) w2 = df_add(w2, df_mul_f(*ba, s_sq));
  // clamp at zero under the root
  if (w2.hi < 0.f || (w2.hi == 0.f && w2.lo <= 0.f)) w2 = df{0.f, 0.f};
  // root: y = sqrt(hi) rounded, then y + (w2 - y^2) / (2 y)
  float wn_hi = 0.f, wn_lo = 0.f;
  if (w2.hi > 0.f) {
    const float y = __fsqrt_rn(w2.hi);
    const float res = __fadd_rn(fmaf(-y, y, w2.hi), w2.lo);     // w2 - y^2 (y^2 exact via FMA)
    two_sum(y, __fdiv_rn(res, __fmul_rn(2.f, y)), wn_hi, wn_lo);
  }
  // divisor max(wnorm, eps) as a double-float
  float d_hi = wn_hi, d_lo = wn_lo;
  if (wn_hi < eps || (wn_hi == eps && wn_lo < 0.f)) {
    d_hi = eps;
    d_lo = 0.f;
  }
  // quotient: q = m / d_hi rounded, then q + (m - q d) / d_hi
  const float q = __fdiv_rn(mj, d_hi);
  const float res = __fsub_rn(fmaf(-q, d_hi, mj), __fmul_rn(q, d_lo));   // m - q d
  wnorm_out = __fadd_rn(wn_hi, wn_lo);
  g_out = __fadd_rn(q, __fdiv_rn(res, d_hi));
}

}  // namespace dora
