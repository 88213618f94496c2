// sv_rowstat.cuh — per-row normaliser helpers shared by the Lookahead and
// multi-draft verify kernels: element access for fp32 and bf16 rows, and the
// online (max, sum of exp2) fold and combine.
#pragma once
#include <cstdint>

#include "sv_device.cuh"

namespace sv {
namespace rowstat {

// Element access for the two storage types: fp32, and bf16 kept as its raw
// 16-bit pattern (element 0 in the low half of a 32-bit word).
template <typename E>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kPerVec = 4;  // elements per 16-byte vector
  __device__ static float load(const float* p) { return __ldg(p); }
  __device__ static void unpack(const uint4& v, float* x) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
};
template <>
struct Elem<uint16_t> {
  static constexpr int kPerVec = 8;
  __device__ static float load(const uint16_t* p) { return __uint_as_float((uint32_t)__ldg(p) << 16); }
  __device__ static void unpack(const uint4& v, float* x) {
    x[0] = bf_lo(v.x);
    x[1] = bf_hi(v.x);
    x[2] = bf_lo(v.y);
    x[3] = bf_hi(v.y);
    x[4] = bf_lo(v.z);
    x[5] = bf_hi(v.z);
    x[6] = bf_lo(v.w);
    x[7] = bf_hi(v.w);
  }
};

// Folds the scaled values z[0..n) into a running (m, s): m = max z and
// s = sum 2^(z - m). A NaN reaches m and stays there; -inf values add 0; a row
// of -inf only leaves m = -inf, s = 0. All three are caught by the walk.
template <int n>
__device__ __forceinline__ void fold(float& m, float& s, const float* z) {
  float vm = z[0];
#pragma unroll
  for (int i = 1; i < n; ++i) vm = fmax_nan(vm, z[i]);
  const float mn = fmax_nan(m, vm);
  if (mn != m) {  // a new maximum (or a NaN)
    s *= ex2(m - mn);
    m = mn;
  }
  if (m != -INFINITY) {
#pragma unroll
    for (int i = 0; i < n; ++i) s += ex2(z[i] - m);
  }
}

// (m, s) <- the pair for the union of the two value sets.
__device__ __forceinline__ void combine(float& m, float& s, float m2, float s2) {
  const float mn = fmax_nan(m, m2);
  if (mn == -INFINITY) return;  // both sets hold only -inf
  s = s * ex2(m - mn) + s2 * ex2(m2 - mn);
  m = mn;
}

}  // namespace rowstat
}  // namespace sv
