// sv_greedy_rows.cu — a two-kernel greedy (Lookahead) verify, an alternative
// to the streaming kernel's greedy mode for calls of a few tens of MB, where
// fixed costs dominate ("Lookahead Decoding 完全拆解", verify branch: candidate
// token n must equal the argmax at position n; the longest matched prefix
// wins, then one bonus token).
//
//  gr_rows_kernel — one CTA per row of logits[B,G,N,V]: the row's argmax
//    (numeric order, so -0 ties +0; lowest index among equal maxima) in one
//    read with 16-byte loads, or a NaN mark.
//  gr_match_kernel — one warp per sequence: the longest matched prefix of
//    every candidate, the best candidate (lowest g on ties) and the outputs.
#include <cmath>

#include "sv_device.cuh"
#include "sv_greedy_rows.h"

namespace sv {
namespace gr {
namespace {

constexpr int kRowThreads = 256;
constexpr int kMatchThreads = 128;  // four sequences per CTA
constexpr int32_t kNanRow = -2;

template <typename E>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kPerVec = 4;
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

// (v, i) is the best value seen and its index; i < 0 until something is seen.
// Values arrive in increasing index order within a thread, so a later equal
// value never replaces an earlier one.
template <int n>
__device__ __forceinline__ void consider(float& v, int& i, bool& nan, const float* x, int e) {
  float vm = x[0];
#pragma unroll
  for (int k = 1; k < n; ++k) vm = fmax_nan(vm, x[k]);
  if (vm != vm) {
    nan = true;
    return;
  }
  if (vm > v || i < 0) {
    int k0 = 0;
#pragma unroll
    for (int k = n - 1; k >= 0; --k)
      if (x[k] == vm) k0 = k;
    v = vm;
    i = e + k0;
  }
}

// Eight bf16 values in their packed words: the maximum from packed
// comparisons, the elements unpacked only when it improves on (v, i).
__device__ __forceinline__ void consider_bf16x8(float& v, int& i, bool& nan, const uint4 q, int e) {
  const uint32_t mm = bf2_max_nan(bf2_max_nan(q.x, q.y), bf2_max_nan(q.z, q.w));
  const float vm = fmax_nan(bf_lo(mm), bf_hi(mm));
  if (vm != vm) {
    nan = true;
    return;
  }
  if (vm > v || i < 0) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    int k0 = 0;
#pragma unroll
    for (int k = 7; k >= 0; --k) {
      const float x = (k & 1) ? bf_hi(w[k >> 1]) : bf_lo(w[k >> 1]);
      if (x == vm) k0 = k;
    }
    v = vm;
    i = e + k0;
  }
}

// Whether (v2, i2) beats (v1, i1): a larger value, or an equal one earlier.
__device__ __forceinline__ bool better(float v2, int i2, float v1, int i1) {
  if (i2 < 0) return false;
  if (i1 < 0) return true;
  return v2 > v1 || (v2 == v1 && i2 < i1);
}

template <typename E>
__global__ void __launch_bounds__(kRowThreads, 8) gr_rows_kernel(const Params p) {
  using X = Elem<E>;
  constexpr int PV = X::kPerVec;
  constexpr int U = 4;
  const int tid = threadIdx.x;
  const int64_t r = blockIdx.x;
  const int V = (int)p.V;  // V < 2^31
  const E* row = static_cast<const E*>(p.logits) + r * p.V;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
  int head = (int)(((16u - (unsigned)(addr & 15u)) & 15u) / sizeof(E));
  if (head > V) head = V;
  const int nvec = (V - head) / PV;
  const int tail0 = head + nvec * PV;
  const uint4* vec = reinterpret_cast<const uint4*>(row + head);
  float v = -INFINITY;
  int i = -1;
  bool nan = false;
  // The head first (lowest indices), then the vectors, then the tail, so
  // that each thread sees its indices in increasing order.
  if (tid < head) {
    const float x = X::load(row + tid);
    consider<1>(v, i, nan, &x, tid);
  }
  for (int i0 = tid; i0 < nvec; i0 += U * kRowThreads) {
    uint4 q[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = i0 + u * kRowThreads;
      q[u] = k < nvec ? __ldg(vec + k) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = i0 + u * kRowThreads;
      if (k < nvec) {
        if constexpr (PV == 8) {
          consider_bf16x8(v, i, nan, q[u], head + k * PV);
        } else {
          float x[PV];
          X::unpack(q[u], x);
          consider<PV>(v, i, nan, x, head + k * PV);
        }
      }
    }
  }
  if (tail0 + tid < V) {
    const float x = X::load(row + tail0 + tid);
    consider<1>(v, i, nan, &x, tail0 + tid);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(v2, i2, v, i)) {
      v = v2;
      i = i2;
    }
  }
  nan = __any_sync(0xffffffffu, nan);
  __shared__ float rv[kRowThreads / 32];
  __shared__ int ri[kRowThreads / 32];
  __shared__ int rn[kRowThreads / 32];
  const int warp = tid >> 5, lane = tid & 31;
  if (lane == 0) {
    rv[warp] = v;
    ri[warp] = i;
    rn[warp] = nan;
  }
  __syncthreads();
  if (warp == 0) {
    v = lane < kRowThreads / 32 ? rv[lane] : -INFINITY;
    i = lane < kRowThreads / 32 ? ri[lane] : -1;
    nan = lane < kRowThreads / 32 ? rn[lane] != 0 : false;
#pragma unroll
    for (int o = kRowThreads / 64; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
      if (better(v2, i2, v, i)) {
        v = v2;
        i = i2;
      }
    }
    nan = __any_sync(0xffffffffu, nan);
    if (lane == 0) p.am[r] = nan ? kNanRow : i;
  }
}

// One warp per sequence; lane g handles candidates g, g+32, ...
__global__ void __launch_bounds__(kMatchThreads) gr_match_kernel(const Params p) {
  const int lane = threadIdx.x & 31;
  const int64_t b = (int64_t)blockIdx.x * (kMatchThreads / 32) + (threadIdx.x >> 5);
  grid_dependency_sync(false);
  if (b >= p.B) return;
  const int G = p.G, N = p.N;
  const int32_t* am = p.am + b * G * N;
  const int32_t* cand = p.cand + b * G * (N - 1);
  int bad = 0;
  for (int k = lane; k < G * N; k += 32) bad |= am[k] == kNanRow;
  for (int k = lane; k < G * (N - 1); k += 32) bad |= cand[k] < 0 || (int64_t)cand[k] >= p.V;
  int32_t* out = p.out_tokens + b * N;
  if (__any_sync(0xffffffffu, bad)) {
    for (int n = lane; n < N; n += 32) out[n] = -1;
    if (lane == 0) {
      p.out_accept_len[b] = -1;
      if (p.out_best) p.out_best[b] = -1;
      atomicOr(p.ctl + 3, kStatusInput);
    }
    return;
  }
  // key = L * 65536 + (65535 - g): the largest key is the longest prefix,
  // lowest g among equals (G <= 65535, N <= 32767).
  int key = -1;
  for (int g = lane; g < G; g += 32) {
    int L = 0;
    while (L < N - 1 && cand[g * (N - 1) + L] == am[g * N + L]) ++L;
    const int k = L * 65536 + (65535 - g);
    key = k > key ? k : key;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const int k2 = __shfl_xor_sync(0xffffffffu, key, o);
    key = k2 > key ? k2 : key;
  }
  const int L = key >> 16, g = 65535 - (key & 0xFFFF);
  for (int n = lane; n < N; n += 32)
    out[n] = n < L ? cand[g * (N - 1) + n] : (n == L ? am[g * N + L] : -1);
  if (lane == 0) {
    p.out_accept_len[b] = L;
    if (p.out_best) p.out_best[b] = g;
  }
}

template <typename E>
cudaError_t launch_t(const Params& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.G * p.N));
  cfg.blockDim = dim3(kRowThreads);
  cfg.stream = stream;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gr_rows_kernel<E>, p);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)((p.B + kMatchThreads / 32 - 1) / (kMatchThreads / 32)));
  cfg.blockDim = dim3(kMatchThreads);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gr_match_kernel, p);
}

}  // namespace

cudaError_t launch(const Params& p, int dtype, cudaStream_t stream) {
  return dtype == 1 ? launch_t<uint16_t>(p, stream) : launch_t<float>(p, stream);
}

}  // namespace gr
}  // namespace sv
