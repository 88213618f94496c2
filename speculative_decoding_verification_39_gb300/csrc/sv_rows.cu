// sv_rows.cu — the row pass of the two-kernel sampling verify (sm_103a).
//
// Every logit of a call is read once here. The call's rows are cut into work
// items, one CTA each: a chunk (at most 32 KB) of a long row, reduced by the
// whole CTA, or a group of whole short rows, one warp per row. Every thread
// issues all its 16-byte loads of the item at once (a chunk is 8 vectors per
// thread), so that each SM keeps ~100 KB of loads in flight; the few bytes of
// a row outside its 16-byte aligned interior are read element by element.
//
// Per row (chunk) the pass writes the largest raw logit m and
// s = sum 2^(l*c - fl(m*c)) with c = log2(e)/T ("Speculative Decoding ——
// LLM推理优化技术（一）" §4; kwkr.cn "投机解码" §3.4: softmax of l/T on both
// sides; fp32 per §3.2): the max first, then the sum against it, both from
// registers. A NaN or +inf logit reaches m and marks the row invalid; a row
// of -inf leaves m = -inf, s = 0; the decide kernel rejects all three. It
// also records the logit of the row's draft token (target row i and draft row
// i hold x_i), so that the accept scan needs no further read.
#include "sv_device.cuh"
#include "sv_v2.h"

namespace sv {
namespace v2 {
namespace {

constexpr int kWarpsR = kRowsThreads / 32;
constexpr int kVecsPerThread = 8;  // a 32 KB chunk over 256 threads

template <typename E>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kPerVec = 4;
  __device__ static float load(const char* row, int64_t e) { return __ldg(reinterpret_cast<const float*>(row) + e); }
  __device__ static float vmax(const uint4& v) {
    return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
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
  __device__ static float load(const char* row, int64_t e) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row) + e)) << 16);
  }
  __device__ static float vmax(const uint4& v) {
    const uint32_t m = bf2_max_nan(bf2_max_nan(v.x, v.y), bf2_max_nan(v.z, v.w));
    return fmax_nan(bf_lo(m), bf_hi(m));
  }
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

// The row of global row index g = b*R + i: target row i for i <= K, draft
// row i-K-1 after.
__device__ __forceinline__ const char* row_of(const Params& p, int64_t g) {
  const int64_t b = g / p.R;
  const int i = (int)(g - b * p.R);
  if (i <= p.K) return p.target + (b * (p.K + 1) + i) * p.V * p.esz;
  return p.draft + (b * p.K + (i - p.K - 1)) * p.V * p.esz;
}

// The draft token of global row g (target row i < K and draft row i hold
// x_i; target row K holds none: -1).
__device__ __forceinline__ int32_t token_of(const Params& p, int64_t g) {
  const int64_t b = g / p.R;
  const int i = (int)(g - b * p.R);
  if (i == p.K) return -1;
  return __ldg(p.tokens + b * p.K + (i < p.K ? i : i - p.K - 1));
}

// Records the logit of row g's draft token x when x lies in [e0, e1).
__device__ __forceinline__ void gather(const Params& p, int64_t g, const char* row, int64_t e0, int64_t e1,
                                       int32_t x) {
  if (x < e0 || (int64_t)x >= e1) return;
  const int64_t b = g / p.R;
  const int i = (int)(g - b * p.R);
  const float v = p.esz == 2 ? Elem<uint16_t>::load(row, x) : Elem<float>::load(row, x);
  p.gz[b * (2 * p.K) + (i < p.K ? i : p.K + (i - p.K - 1))] = v;
}

// Elements [e0, e1) of a row, by NT threads with index t: the aligned interior
// as 16-byte vectors, kVecsPerThread of them loaded at once per batch, and
// the unaligned head and tail element by element. Returns this thread's max
// (pass 1) and, against mref, its sum (pass 2), both over the same registers.
template <typename E, int NT>
__device__ __forceinline__ void segment(const char* row, int64_t e0, int64_t e1, int t, float c, float& m_out,
                                        float& s_out, float (*reduce_max)(float, float*), float* red) {
  using X = Elem<E>;
  constexpr int PV = X::kPerVec;
  constexpr uint32_t kNegInf = sizeof(E) == 2 ? 0xFF80FF80u : 0xFF800000u;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(row + e0 * (int64_t)sizeof(E));
  int64_t head = (int64_t)(((16u - (unsigned)(a0 & 15u)) & 15u) / sizeof(E));
  if (head > e1 - e0) head = e1 - e0;
  const int64_t nvec = (e1 - e0 - head) / PV;
  const int64_t tail0 = e0 + head + nvec * PV;
  const uint4* vec = reinterpret_cast<const uint4*>(row + (e0 + head) * (int64_t)sizeof(E));
  const float xh = t < head ? X::load(row, e0 + t) : -INFINITY;
  const float xt = tail0 + t < e1 ? X::load(row, tail0 + t) : -INFINITY;
  float m = fmax_nan(xh, xt), s = 0.f;
  // one batch covers a chunk of up to NT * kVecsPerThread vectors; longer
  // segments (very long fp32 rows) loop
  for (int64_t i0 = t; i0 < nvec || i0 == t; i0 += (int64_t)NT * kVecsPerThread) {
    uint4 v[kVecsPerThread];
#pragma unroll
    for (int u = 0; u < kVecsPerThread; ++u) {
      const int64_t i = i0 + (int64_t)u * NT;
      v[u] = i < nvec ? __ldg(vec + i) : make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
    }
    float bm = X::vmax(v[0]);
#pragma unroll
    for (int u = 1; u < kVecsPerThread; ++u) bm = fmax_nan(bm, X::vmax(v[u]));
    const float mn = fmax_nan(m, bm);
    if (nvec <= (int64_t)NT * kVecsPerThread) {
      // the whole segment is in registers (the same test in every thread, so
      // all of them reach the reduction's barrier): max, then sum against it
      m = reduce_max(mn, red);
      if (m > -INFINITY && m < INFINITY) {
        const float mref = __fmul_rn(m, c);
#pragma unroll
        for (int u = 0; u < kVecsPerThread; ++u) {
          float x[PV];
          X::unpack(v[u], x);
          float a = 0.f;
#pragma unroll
          for (int k = 0; k < PV; ++k) a += ex2(fmaf(x[k], c, -mref));
          s += a;
        }
        s += ex2(fmaf(xh, c, -mref)) + ex2(fmaf(xt, c, -mref));
      }
      m_out = m;
      s_out = s;
      return;
    }
    // a longer segment: online, rescaling at each new max (per thread)
    if (mn != m) {
      if (m > -INFINITY && m < INFINITY && mn < INFINITY) s *= ex2(__fsub_rn(__fmul_rn(m, c), __fmul_rn(mn, c)));
      m = mn;
    }
    if (m > -INFINITY && m < INFINITY) {
      const float mref = __fmul_rn(m, c);
#pragma unroll
      for (int u = 0; u < kVecsPerThread; ++u) {
        float x[PV];
        X::unpack(v[u], x);
#pragma unroll
        for (int k = 0; k < PV; ++k) s += ex2(fmaf(x[k], c, -mref));
      }
    }
  }
  // head and tail of a looped segment, against this thread's final max
  if (m > -INFINITY && m < INFINITY) {
    const float mref = __fmul_rn(m, c);
    s += ex2(fmaf(xh, c, -mref)) + ex2(fmaf(xt, c, -mref));
  }
  m_out = m;
  s_out = s;
}

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ float warp_max_only(float v, float*) { return warp_max_nan(v); }
__device__ float cta_max(float v, float* red) {
  v = warp_max_nan(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < kWarpsR; ++w) m = fmax_nan(m, red[w]);
  __syncthreads();
  return m;
}

// (m, s) <- the pair for the union of a's and b's values (per-thread
// references fl(m*c)).
__device__ __forceinline__ void combine(float& m, float& s, float m2, float s2, float c) {
  const float mn = fmax_nan(m, m2);
  if (!(mn > -INFINITY && mn < INFINITY)) {
    m = mn;
    return;
  }
  const float r = __fmul_rn(mn, c);
  float t = 0.f;
  if (m > -INFINITY) t += s * ex2(__fsub_rn(__fmul_rn(m, c), r));
  if (m2 > -INFINITY) t += s2 * ex2(__fsub_rn(__fmul_rn(m2, c), r));
  m = mn;
  s = t;
}

template <typename E>
__global__ void __launch_bounds__(kRowsThreads, 4) rows_kernel(const Params p) {
  __shared__ float red[kWarpsR];
  __shared__ float2 red2[kWarpsR];
  grid_dependency_sync(false);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float c = p.c;
  const int64_t it = blockIdx.x;
  const int64_t grp = it / p.NCH;
  const int k = (int)(it - grp * p.NCH);
  if (p.RPI == 1) {
    // one chunk of one row, the whole CTA
    const int64_t g = grp;
    const char* row = row_of(p, g);
    const int32_t x = tid == 0 ? token_of(p, g) : -1;
    const int64_t e0 = (int64_t)k * p.CE;
    const int64_t e1 = e0 + p.CE < p.V ? e0 + p.CE : p.V;
    float m, s;
    segment<E, kRowsThreads>(row, e0, e1, tid, c, m, s, cta_max, red);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the CTA's (m, s): every thread summed against the same reference when
    // the chunk fit one batch; the general combine handles both cases
    float mm = m, ss = s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, mm, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, ss, o);
      combine(mm, ss, m2, s2, c);
    }
    if (lane == 0) red2[warp] = make_float2(mm, ss);
    __syncthreads();
    if (tid == 0) {
      float M = red2[0].x, S = red2[0].y;
      for (int w = 1; w < kWarpsR; ++w) combine(M, S, red2[w].x, red2[w].y, c);
      p.part[g * p.NCH + k] = make_float2(M, S);
      gather(p, g, row, e0, e1, x);
    }
  } else {
    // short whole rows, one warp per row
    for (int r = warp; r < p.RPI; r += kWarpsR) {
      const int64_t g = grp * p.RPI + r;
      if (g >= p.B * p.R) break;
      const char* row = row_of(p, g);
      const int32_t x = lane == 0 ? token_of(p, g) : -1;
      float m, s;
      segment<E, 32>(row, 0, p.V, lane, c, m, s, warp_max_only, nullptr);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        combine(m, s, m2, s2, c);
      }
      if (lane == 0) {
        p.part[g] = make_float2(m, s);
        gather(p, g, row, 0, p.V, x);
      }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
}

}  // namespace

cudaError_t launch_rows(const Params& p, int dtype, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.items);
  cfg.blockDim = dim3(kRowsThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return dtype == 1 ? cudaLaunchKernelEx(&cfg, rows_kernel<uint16_t>, p)
                    : cudaLaunchKernelEx(&cfg, rows_kernel<float>, p);
}

}  // namespace v2
}  // namespace sv
