// sv_df.cuh — double-float arithmetic on the fp32 pipes (a value is hi + lo,
// |lo| <= ulp(hi)/2), for the draws that must resolve a CDF edge more finely
// than fp32 can. The error-free transformations are Knuth's two-sum,
// Dekker's fast two-sum and the FMA-based exact product; every operation is
// written with explicitly rounded intrinsics so that the compiler cannot fuse
// or reorder them.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

struct df {
  float h, l;
};

__device__ __forceinline__ df df_make(float h) { return df{h, 0.f}; }

// s + e == a + b exactly.
__device__ __forceinline__ df two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return df{s, e};
}
// The same for |a| >= |b| (or a == 0).
__device__ __forceinline__ df fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return df{s, __fsub_rn(b, __fsub_rn(s, a))};
}
// p + e == a * b exactly (barring underflow).
__device__ __forceinline__ df two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return df{p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ df df_add(df a, df b) {
  const df s = two_sum(a.h, b.h);
  const df t = two_sum(a.l, b.l);
  df r = fast_two_sum(s.h, __fadd_rn(s.l, t.h));
  return fast_two_sum(r.h, __fadd_rn(r.l, t.l));
}
__device__ __forceinline__ df df_neg(df a) { return df{-a.h, -a.l}; }
__device__ __forceinline__ df df_sub(df a, df b) { return df_add(a, df_neg(b)); }
__device__ __forceinline__ df df_mul(df a, df b) {
  const df p = two_prod(a.h, b.h);
  const float t = __fmaf_rn(a.h, b.l, __fmul_rn(a.l, b.h));
  return fast_two_sum(p.h, __fadd_rn(p.l, t));
}
__device__ __forceinline__ df df_mul_f(df a, float b) {
  const df p = two_prod(a.h, b);
  return fast_two_sum(p.h, __fmaf_rn(a.l, b, p.l));
}
// a / b for b > 0: one Newton correction of the fp32 quotient.
__device__ __forceinline__ df df_div(df a, df b) {
  const float q1 = __fdiv_rn(a.h, b.h);
  const df r = df_sub(a, df_mul_f(b, q1));
  const float q2 = __fdiv_rn(r.h, b.h);
  return fast_two_sum(q1, q2);
}
// a > b, for normalised operands.
__device__ __forceinline__ bool df_gt(df a, df b) { return a.h > b.h || (a.h == b.h && a.l > b.l); }
__device__ __forceinline__ bool df_pos(df a) { return a.h > 0.f || (a.h == 0.f && a.l > 0.f); }

// 2^x for x = xh + xl <= 0, to about 1e-11 relative: x = k/32 + r with
// k = round(32 xh) and |r| <= 1/64, 2^(k/32) = 2^floor(k/32) * 2^((k mod 32)/32)
// from a table of double-floats, and 2^r = e^t, t = r ln 2, from its Taylor
// series to t^5 (the first omitted term is below 3e-15 for |t| < 0.011).
// The power of two is applied as an exact multiply; values below 2^-126 are
// returned as 0 (as the fp32 path's flush-to-zero exp2 does).
__device__ __forceinline__ df df_exp2(float xh, float xl, const float* tab_hi, const float* tab_lo) {
  if (!(xh >= -126.f)) return df{0.f, 0.f};
  constexpr float kLn2Hi = 0.693147182464599609375f;      // fl(ln 2)
  constexpr float kLn2Lo = -1.904654323148236017e-09f;     // ln 2 - fl(ln 2)
  const float kf = rintf(__fmul_rn(xh, 32.f));
  const float rh = __fmaf_rn(kf, -0.03125f, xh);           // exact
  const float th = __fmul_rn(rh, kLn2Hi);
  const float tl = __fadd_rn(__fmaf_rn(rh, kLn2Hi, -th), __fmaf_rn(rh, kLn2Lo, __fmul_rn(xl, kLn2Hi)));
  const df t = fast_two_sum(th, tl);
  // q = t^2/2 + t^3/6 + t^4/24 + t^5/120 on t.h
  float q = __fmaf_rn(t.h, 0.008333333767950534820556640625f, 0.041666667908430099487304688f);
  q = __fmaf_rn(t.h, q, 0.16666667163372039794921875f);
  q = __fmaf_rn(t.h, q, 0.5f);
  q = __fmul_rn(__fmul_rn(t.h, t.h), q);
  const int k = (int)kf;
  const int i = k & 31;
  const int n = k >> 5;  // floor(k / 32)
  const float Th = tab_hi[i], Tl = tab_lo[i];
  // T * (1 + t.h + (t.l + q))
  const float sl = __fadd_rn(t.l, q);
  const df p = two_prod(Th, t.h);
  df r = fast_two_sum(Th, p.h);
  const float corr = __fadd_rn(__fadd_rn(p.l, __fmul_rn(Th, sl)), __fmaf_rn(Tl, t.h, Tl));
  r = fast_two_sum(r.h, __fadd_rn(r.l, corr));
  if (n < -126) return df{0.f, 0.f};
  const float scale = __int_as_float((n + 127) << 23);  // 2^n, exact
  return df{__fmul_rn(r.h, scale), __fmul_rn(r.l, scale)};
}

}  // namespace sv
