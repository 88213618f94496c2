// sv_rows.cu — the row pass of the two-kernel sampling verify (sm_103a).
//
// Every logit of a call is read once here. The call's rows are cut into work
// items: a chunk (at most 32 KB) of a long row, or a group of whole short
// rows. A persistent grid of CTAs takes the items in a fixed round-robin
// order; each CTA keeps two shared-memory stages, and its elected thread moves
// the next item HBM -> shared memory with 1-D bulk copies (cp.async.bulk,
// completing on the stage's mbarrier) while the CTA reduces the current one.
// Bytes of a row outside its 16-byte aligned interior (at most 15 at each
// end) are read directly.
//
// Per row (chunk) the pass writes the largest raw logit m and
// s = sum 2^(l*c - fl(m*c)) with c = log2(e)/T ("Speculative Decoding ——
// LLM推理优化技术（一）" §4; kwkr.cn "投机解码" §3.4: softmax of l/T on both
// sides; fp32 per §3.2), in two passes over shared memory: the max, then the
// sum against it. A NaN or +inf logit reaches m and marks the row invalid; a
// row of -inf leaves m = -inf, s = 0; the decide kernel rejects all three.
// It also records the logit of the row's draft token (target row i and draft
// row i hold x_i), so that the accept scan needs no further read.
#include "sv_device.cuh"
#include "sv_v2.h"

namespace sv {
namespace v2 {
namespace {

constexpr int kWarpsR = kRowsThreads / 32;
constexpr int kStagesR = 2;

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

// One segment of a work item: elements [e0, e1) of global row g, its aligned
// interior [ie0, ie0 + ibytes/esz) staged at byte offset `off` of the stage.
struct Seg {
  const char* row;
  int64_t g, e0, e1, ie0;
  uint32_t ibytes, off;
};

__device__ __forceinline__ Seg make_seg(const Params& p, int64_t g, int64_t e0, int64_t e1, uint32_t off) {
  Seg s;
  s.row = row_of(p, g);
  s.g = g;
  s.e0 = e0;
  s.e1 = e1;
  s.off = off;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(s.row + e0 * p.esz);
  const uintptr_t a1 = reinterpret_cast<uintptr_t>(s.row + e1 * p.esz);
  const uintptr_t A = (a0 + 15) & ~uintptr_t(15);
  const uintptr_t Z = a1 & ~uintptr_t(15);
  if (A < Z) {
    s.ibytes = (uint32_t)(Z - A);
    s.ie0 = e0 + (int64_t)((A - a0) / p.esz);
  } else {
    s.ibytes = 0;
    s.ie0 = e1;
  }
  return s;
}

// Rows in work item `it`: 1 for a chunk of a row, up to RPI whole rows.
__device__ __forceinline__ int item_rows(const Params& p, int64_t it) {
  if (p.RPI == 1) return 1;
  const int64_t g0 = (it / p.NCH) * p.RPI;
  const int64_t left = p.B * p.R - g0;
  return (int)(left < p.RPI ? left : p.RPI);
}

// Segment r of work item `it`; each row of a group has its own slot of
// row_slot bytes in the stage.
__device__ __forceinline__ Seg item_seg(const Params& p, int64_t it, int r) {
  const int64_t grp = it / p.NCH;
  const int k = (int)(it - grp * p.NCH);
  if (p.RPI == 1) {
    const int64_t e0 = (int64_t)k * p.CE;
    return make_seg(p, grp, e0, e0 + p.CE < p.V ? e0 + p.CE : p.V, 0);
  }
  return make_seg(p, grp * p.RPI + r, 0, p.V, (uint32_t)r * p.row_slot);
}

__device__ __forceinline__ void issue(const Params& p, int64_t it, char* stage, uint64_t* bar) {
  const int n = item_rows(p, it);
  uint32_t bytes = 0;
  for (int r = 0; r < n; ++r) bytes += item_seg(p, it, r).ibytes;
  mbar_arrive_expect_tx(bar, bytes);
  for (int r = 0; r < n; ++r) {
    const Seg sg = item_seg(p, it, r);
    if (sg.ibytes) bulk_g2s(stage + sg.off, sg.row + sg.ie0 * p.esz, sg.ibytes, bar);
  }
}

template <typename E, int NT>
__device__ __forceinline__ float seg_max(const Seg& s, const char* stage, int t) {
  using X = Elem<E>;
  float m = -INFINITY;
  const int64_t nh = s.ie0 - s.e0;
  const int64_t ni = (int64_t)s.ibytes / (int64_t)sizeof(E);
  const int64_t tail0 = s.ie0 + ni;
  if (t < nh) m = fmax_nan(m, X::load(s.row, s.e0 + t));
  if (tail0 + t < s.e1) m = fmax_nan(m, X::load(s.row, tail0 + t));
  const uint4* v = reinterpret_cast<const uint4*>(stage + s.off);
  const int64_t nv = (int64_t)s.ibytes / 16;
  for (int64_t i = t; i < nv; i += NT) m = fmax_nan(m, X::vmax(v[i]));
  return m;
}

template <typename E, int NT>
__device__ __forceinline__ float seg_sum(const Seg& s, const char* stage, int t, float c, float mref) {
  using X = Elem<E>;
  constexpr int PV = X::kPerVec;
  float acc = 0.f;
  const int64_t nh = s.ie0 - s.e0;
  const int64_t ni = (int64_t)s.ibytes / (int64_t)sizeof(E);
  const int64_t tail0 = s.ie0 + ni;
  if (t < nh) acc += ex2(fmaf(X::load(s.row, s.e0 + t), c, -mref));
  if (tail0 + t < s.e1) acc += ex2(fmaf(X::load(s.row, tail0 + t), c, -mref));
  const uint4* v = reinterpret_cast<const uint4*>(stage + s.off);
  const int64_t nv = (int64_t)s.ibytes / 16;
  for (int64_t i = t; i < nv; i += NT) {
    float x[PV];
    X::unpack(v[i], x);
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < PV; ++k) a += ex2(fmaf(x[k], c, -mref));
    acc += a;
  }
  return acc;
}

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// The draft token of global row g (target row i < K and draft row i hold
// x_i; target row K holds none: -1).
__device__ __forceinline__ int32_t token_of(const Params& p, int64_t g) {
  const int64_t b = g / p.R;
  const int i = (int)(g - b * p.R);
  if (i == p.K) return -1;
  return __ldg(p.tokens + b * p.K + (i < p.K ? i : i - p.K - 1));
}

// Records the logit of row sg.g's draft token x if it lies in [e0, e1): from
// the staged copy when it is in the aligned interior, else from global memory.
template <typename E>
__device__ __forceinline__ void gather(const Params& p, const Seg& sg, const char* stage, int32_t x) {
  if (x < sg.e0 || (int64_t)x >= sg.e1) return;
  const int64_t b = sg.g / p.R;
  const int i = (int)(sg.g - b * p.R);
  const int ii = i < p.K ? i : i - p.K - 1;
  const int64_t ni = (int64_t)sg.ibytes / (int64_t)sizeof(E);
  float v;
  if (x >= sg.ie0 && x < sg.ie0 + ni) {
    const char* a = stage + sg.off + (x - sg.ie0) * (int64_t)sizeof(E);
    v = sizeof(E) == 2 ? __uint_as_float((uint32_t)(*reinterpret_cast<const unsigned short*>(a)) << 16)
                       : *reinterpret_cast<const float*>(a);
  } else {
    v = Elem<E>::load(sg.row, x);
  }
  p.gz[b * (2 * p.K) + (i < p.K ? i : p.K + ii)] = v;
}

template <typename E>
__global__ void __launch_bounds__(kRowsThreads) rows_kernel(const Params p) {
  extern __shared__ __align__(16) char stages[];
  __shared__ uint64_t full[kStagesR];
  __shared__ float red[kWarpsR];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float c = p.c;
  const int64_t first = blockIdx.x, stride = gridDim.x;
  if (tid == 0) {
    for (int s = 0; s < kStagesR; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_sync(false);
  // prologue: the first kStagesR items in flight
  if (tid == 0) {
    for (int s = 0; s < kStagesR; ++s) {
      const int64_t it = first + s * stride;
      if (it < p.items) issue(p, it, stages + s * p.stage_bytes, &full[s]);
    }
  }
  // thread r keeps the draft token of row r of the item in hand, loaded one
  // item ahead so that its latency hides behind the current item's work
  int32_t tok_next = (first < p.items && tid < item_rows(p, first)) ? token_of(p, item_seg(p, first, tid).g) : -1;
  int n = 0;
  for (int64_t it = first; it < p.items; it += stride, ++n) {
    const int s = n % kStagesR;
    const uint32_t parity = (uint32_t)((n / kStagesR) & 1);
    char* stage = stages + s * p.stage_bytes;
    const int ns = item_rows(p, it);
    const int32_t tok = tok_next;
    const int64_t nx = it + stride;
    tok_next = (nx < p.items && tid < item_rows(p, nx)) ? token_of(p, item_seg(p, nx, tid).g) : -1;
    const bool ok = mbar_wait(&full[s], parity);
    if (!__syncthreads_and(ok)) {
      if (tid == 0) atomicOr(p.ctl + 3, kStatusTimeout);
      break;
    }
    if (p.RPI == 1) {
      // one chunk, the whole CTA
      const Seg sg = item_seg(p, it, 0);
      float m = warp_max_nan(seg_max<E, kRowsThreads>(sg, stage, tid));
      if (lane == 0) red[warp] = m;
      __syncthreads();
      m = red[0];
#pragma unroll
      for (int w = 1; w < kWarpsR; ++w) m = fmax_nan(m, red[w]);
      const float mref = __fmul_rn(m, c);
      float acc = (m > -INFINITY && m < INFINITY) ? seg_sum<E, kRowsThreads>(sg, stage, tid, c, mref) : 0.f;
      acc = warp_sum(acc);
      __syncthreads();  // everyone has read red[] as the max
      if (lane == 0) red[warp] = acc;
      __syncthreads();
      if (tid == 0) {
        float sum = 0.f;
        for (int w = 0; w < kWarpsR; ++w) sum += red[w];
        const int64_t k = it % p.NCH;
        p.part[sg.g * p.NCH + k] = make_float2(m, sum);
      }
    } else {
      // whole short rows, one warp per row
      for (int r = warp; r < ns; r += kWarpsR) {
        const Seg sg = item_seg(p, it, r);
        const float m = warp_max_nan(seg_max<E, 32>(sg, stage, lane));
        const float mref = __fmul_rn(m, c);
        float acc = (m > -INFINITY && m < INFINITY) ? seg_sum<E, 32>(sg, stage, lane, c, mref) : 0.f;
        acc = warp_sum(acc);
        if (lane == 0) p.part[sg.g] = make_float2(m, acc);
      }
    }
    if (tid < ns) gather<E>(p, item_seg(p, it, tid), stage, tok);
    __syncthreads();  // the stage is read: refill it
    if (tid == 0) {
      const int64_t nxt = it + kStagesR * stride;
      if (nxt < p.items) issue(p, nxt, stage, &full[s]);
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

cudaError_t launch_rows(const Params& p, int dtype, cudaStream_t stream) {
  const size_t smem = (size_t)kStagesR * p.stage_bytes;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.rows_grid);
  cfg.blockDim = dim3(kRowsThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const void* k = dtype == 1 ? reinterpret_cast<const void*>(rows_kernel<uint16_t>)
                             : reinterpret_cast<const void*>(rows_kernel<float>);
  cudaError_t e = raise_smem_limit_v2(k, smem);
  if (e != cudaSuccess) return e;
  return dtype == 1 ? cudaLaunchKernelEx(&cfg, rows_kernel<uint16_t>, p)
                    : cudaLaunchKernelEx(&cfg, rows_kernel<float>, p);
}

}  // namespace v2
}  // namespace sv
