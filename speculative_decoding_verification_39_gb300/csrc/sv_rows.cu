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

// ------------------------------------------------------------ top-p rows ---
// With top-p < 1 ("Speculative Decoding —— LLM推理优化技术（一）" §4; kwkr.cn
// "投机解码" §3.4: top-p applied to both p and q), each row also needs its
// nucleus: the largest key tau (the order-preserving key of the bf16 logit;
// equal logits share one) whose upper set {v : key(l_v) >= tau} holds mass
// >= top_p * s, and that mass cum. One CTA per row at a time (persistent
// CTAs, four per SM, taking rows g = blockIdx.x, + gridDim.x, ...); the row
// streams through registers in batches of 24 KB, and per batch each warp
// (on its own, with no barrier across the CTA)
//  - raises its running max M_w (NaN-propagating) and rescales its lanes'
//    running sums s = sum 2^(l c - fl(M_w c));
//  - counts its elements whose keys lie in its window of kTpWin keys below
//    key(M_w) (bin i holds key(M_w) - i). When M_w rises the window slides
//    up by as many keys: bins that fall off hold keys below the new window,
//    and no later element can bring them back.
// At the end of the row the CTA takes M = max M_w, rescales the sums to
// fl(M c) and merges the windows: as M_w <= M, warp w's window reaches at
// least as low as the row's window of kTpWin keys below key(M), so it holds
// every element of its own that lies in it. Bin i of the row's window weighs
// count * 2^(val(key) c - fl(M c)); the scan from the top key finds the cut. A row whose cut lies below the window
// (a flat row) is read twice more: once for the masses of coarse bins of 256
// keys below the window, once for the exact keys of the coarse bin that holds
// the cut.
constexpr int kTpThreads = 256;
constexpr int kTpWarps = kTpThreads / 32;
constexpr int kTpVecs = 6;    // 16-byte vectors per thread and batch: 24 KB per CTA
constexpr int kTpWin = 256;   // exact keys counted while the row streams (one bin per thread)
static_assert(kTpWin == kTpThreads, "one window bin per thread");

struct TpShared {
  union {
    uint32_t u[kTpWin];
    float f[kTpWin];
  } hist;
  float red[2][kTpWarps];
  float bf[2];
  int bi[2];
  uint32_t spare[32];                // the counts of elements outside the window (one word per lane, never read)
  uint32_t whist[kTpWarps][kTpWin];  // each warp's window of keys below its running max
  float wm[kTpWarps];                // each warp's max of the row
};

// key_bf16 of the value whose stored 16 bits are h.
__device__ __forceinline__ uint32_t key16(uint32_t h) {
  if (h == 0x8000u) h = 0u;
  return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
}

// The lowest key of the window whose top key is hi.
__device__ __forceinline__ uint32_t lo_key(uint32_t hi) {
  return hi >= (uint32_t)(kTpWin - 1) ? hi - (uint32_t)(kTpWin - 1) : 0u;
}

// Adds 1 to the shared-memory counter at `addr` when x >= lo, otherwise to
// `spare` (a word of this lane's own, never read): the address is selected,
// the atomic is unconditional, so the code has no branch (a predicated
// atomic is guarded by one). A NaN compares false.
__device__ __forceinline__ void red_add_ge(uint32_t addr, uint32_t spare, float x, float lo) {
  const uint32_t a = x >= lo ? addr : spare;
  asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(a) : "memory");
}

// (s0, s1) += (a0, a1): the packed fp32 pair add, rounded exactly as two
// scalar adds.
__device__ __forceinline__ void add_x2(float& s0, float& s1, float a0, float a1) {
  asm("{\n\t.reg .b64 ss, aa;\n\tmov.b64 ss, {%0, %1};\n\tmov.b64 aa, {%2, %3};\n\t"
      "add.rn.f32x2 ss, ss, aa;\n\tmov.b64 {%0, %1}, ss;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}

// One batch of the streaming pass: the exp2 sum of every element against
// mref into (s[0], s[1]), and a count at hbase - 4 * bin(h) for every element
// x >= lo_val (the window: keys follow the values). kPos: the window holds
// positive values only, so the bin is (M's bits) - (the element's bits);
// otherwise it is key(M) - key (hbase is set up to match).
template <bool kPos>
__device__ __forceinline__ void tp_batch(const uint4* v, float c, float mref, float lo_val, uint32_t hbase,
                                         uint32_t spare, float* s) {
#pragma unroll
  for (int u = 0; u < kTpVecs; ++u) {
    const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float x0 = bf_lo(w[j]), x1 = bf_hi(w[j]);
      add_x2(s[0], s[1], ex2(fmaf(x0, c, -mref)), ex2(fmaf(x1, c, -mref)));
      const uint32_t h0 = w[j] & 0xFFFFu, h1 = w[j] >> 16;
      red_add_ge(hbase - 4u * (kPos ? h0 : key16(h0)), spare, x0, lo_val);
      red_add_ge(hbase - 4u * (kPos ? h1 : key16(h1)), spare, x1, lo_val);
    }
  }
}

// Inclusive scan of v over the CTA in thread order; *total gets the sum.
// `par` picks the partials buffer (alternating calls need no extra barrier).
__device__ __forceinline__ float tp_scan(float v, float* total, TpShared& s, int& par) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float incl = warp_incl_scan(v, lane);
  if (lane == 31) s.red[par][warp] = incl;
  __syncthreads();
  float below = 0.f, t = 0.f;
#pragma unroll
  for (int w = 0; w < kTpWarps; ++w) {
    if (w < warp) below += s.red[par][w];
    t += s.red[par][w];
  }
  par ^= 1;
  *total = t;
  return below + incl;
}

// The lowest thread index whose flag is set (INT_MAX: none), for every thread.
__device__ __forceinline__ int tp_first(bool flag, TpShared& s) {
  if (threadIdx.x == 0) s.bi[0] = INT_MAX;
  __syncthreads();
  if (flag) atomicMin(&s.bi[0], (int)threadIdx.x);
  __syncthreads();
  const int r = s.bi[0];
  __syncthreads();
  return r;
}

// Every element of the row (8 at a time) to f(x[8]).
template <typename F>
__device__ __forceinline__ void tp_reread(const uint4* vp, int64_t nvec, F f) {
  for (int64_t i = threadIdx.x; i < nvec; i += kTpThreads) {
    float x[8];
    Elem<uint16_t>::unpack(__ldg(vp + i), x);
    f(x);
  }
}

__global__ void __launch_bounds__(kTpThreads, 4) topp_rows_kernel(const Params p) {
  __shared__ TpShared s;
  grid_dependency_sync(true);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float c = p.c;
  const int64_t rows = p.B * p.R;
  const int64_t nvec = p.V / 8;  // V is a multiple of 8 and rows start 16-byte aligned
  int par = 0;                   // which red[] buffer the next reduction uses
  const uint32_t spare = smem_u32(&s.spare[lane]);
  for (int64_t g = blockIdx.x; g < rows; g += gridDim.x) {
    const char* row = row_of(p, g);
    const uint4* vp = reinterpret_cast<const uint4*>(row);
    uint32_t* wh = s.whist[warp];
#pragma unroll
    for (int k = 0; k < kTpWin / 32; ++k) wh[lane + 32 * k] = 0u;
    __syncwarp();
    float Mw = -INFINITY;  // this warp's running max (the same in its lanes)
    uint32_t hw = 0u;      // key(Mw) once Mw > -inf
    float sth = 0.f;       // this thread's sum against fl(Mw c)
    // batches of kTpThreads * kTpVecs vectors; each warp keeps its own max and
    // window, so a batch takes no barrier across the CTA
    for (int64_t b0 = 0; b0 < nvec; b0 += (int64_t)kTpThreads * kTpVecs) {
      uint4 v[kTpVecs];
#pragma unroll
      for (int u = 0; u < kTpVecs; ++u) {
        const int64_t i = b0 + tid + (int64_t)u * kTpThreads;
        v[u] = i < nvec ? __ldg(vp + i) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
      }
      float bm = Elem<uint16_t>::vmax(v[0]);
#pragma unroll
      for (int u = 1; u < kTpVecs; ++u) bm = fmax_nan(bm, Elem<uint16_t>::vmax(v[u]));
      const float Mn = fmax_nan(Mw, warp_max_nan(bm));
      if (!(Mn < INFINITY)) {  // a NaN or +inf: the row is invalid
        Mw = Mn;
        break;
      }
      if (Mn == -INFINITY) continue;  // only -inf so far
      if (Mn != Mw) {
        if (Mw > -INFINITY) sth *= ex2(__fsub_rn(__fmul_rn(Mw, c), __fmul_rn(Mn, c)));
        const uint32_t nhi = key_bf16(Mn);
        if (Mw > -INFINITY && nhi != hw) {
          // slide the window up by dk keys: bin i now holds what bin i - dk held
          const uint32_t dk = nhi - hw;
          uint32_t t[kTpWin / 32];
#pragma unroll
          for (int k = 0; k < kTpWin / 32; ++k) {
            const uint32_t i = (uint32_t)(lane + 32 * k);
            t[k] = i >= dk ? wh[i - dk] : 0u;
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < kTpWin / 32; ++k) wh[lane + 32 * k] = t[k];
          __syncwarp();
        }
        hw = nhi;
        Mw = Mn;
      }
      const float mref = __fmul_rn(Mw, c);
      // The window [lo, hw] of keys holds exactly the elements x >= val(lo)
      // (x <= Mw always). Of positive values only (the usual case), the key
      // of an element is its 16 bits | 0x8000, so its bin is (Mw's bits) -
      // (its bits). Every lane runs the same code: no divergence.
      // (Keys below that of -inf, 0x7F, are NaN patterns: a window that
      // reaches them takes every value.)
      const uint32_t lo = lo_key(hw);
      const float lo_val = lo > 0x7Fu ? val_bf16(lo) : -INFINITY;
      const bool positive = lo > 0x8000u;
      const uint32_t hbase = smem_u32(wh) + (positive ? hw - 0x8000u : hw) * 4u;
      float acc[2] = {0.f, 0.f};
      if (positive)
        tp_batch<true>(v, c, mref, lo_val, hbase, spare, acc);
      else
        tp_batch<false>(v, c, mref, lo_val, hbase, spare, acc);
      sth += acc[0] + acc[1];
    }
    if (lane == 0) s.wm[warp] = Mw;
    __syncthreads();  // every count and every warp's max is in
    // the row's max (a NaN or +inf in any warp: the row is invalid)
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kTpWarps; ++w) M = fmax_nan(M, s.wm[w]);
    const bool valid = M < INFINITY;
    uint32_t hi = 0u;
    float S = 0.f, cum = 0.f;
    uint32_t tau = 0u;
    if (valid && M > -INFINITY) {
      const float mref = __fmul_rn(M, c);
      hi = key_bf16(M);
      // this thread's sum against fl(M c) (its warp's reference is at most that)
      sth = Mw > -INFINITY ? sth * ex2(__fsub_rn(__fmul_rn(Mw, c), mref)) : 0.f;
      float tot;
      (void)tp_scan(sth, &S, s, par);
      cum = S;
      const float target = p.top_p * S;
      const uint32_t lo = hi >= (uint32_t)(kTpWin - 1) ? hi - (uint32_t)(kTpWin - 1) : 0u;
      // the window: bin t is key hi - t, the warps' windows merged (warp w's
      // bin j holds key key(M_w) - j; as M_w <= M, its window reaches at
      // least as low as the row's, so it counted every element of its own
      // in the row's window)
      uint32_t cnt = 0u;
      if ((uint32_t)tid <= hi - lo) {
#pragma unroll
        for (int w = 0; w < kTpWarps; ++w) {
          const float mw = s.wm[w];
          if (mw > -INFINITY) {
            const uint32_t j = (uint32_t)tid - (hi - key_bf16(mw));  // wraps past kTpWin when below bin 0
            if (j < (uint32_t)kTpWin) cnt += s.whist[w][j];
          }
        }
      }
      float m = cnt ? (float)cnt * ex2(fmaf(val_bf16(hi - (uint32_t)tid), c, -mref)) : 0.f;
      float incl = tp_scan(m, &tot, s, par);
      int t = tp_first(incl >= target, s);
      if (t != INT_MAX) {
        if (tid == t) {
          s.bi[1] = (int)(hi - (uint32_t)t);
          s.bf[0] = incl;
        }
      } else if (lo == 0u) {  // every key seen: rounding left the mass short of top_p * s
        if (tid == 0) {
          s.bi[1] = 0;
          s.bf[0] = tot;
        }
      } else {
        // The cut lies below the window. Coarse bins: the masses of the keys
        // below the window, 256 keys per bin (thread t takes bin 255 - t, so
        // that thread order is descending keys).
        const float above = tot;
        s.hist.f[tid] = 0.f;
        __syncthreads();
        tp_reread(vp, nvec, [&](const float* x) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t key = key_bf16(x[k]);
            if (key < lo) atomicAdd(&s.hist.f[key >> 8], ex2(fmaf(x[k], c, -mref)));
          }
        });
        __syncthreads();
        m = s.hist.f[kTpWin - 1 - tid];
        incl = above + tp_scan(m, &tot, s, par);
        t = tp_first(incl >= target, s);
        if (t == INT_MAX) {  // rounding: keep everything
          if (tid == 0) {
            s.bi[1] = 0;
            s.bf[0] = above + tot;
          }
        } else {
          // the exact keys of coarse bin 255 - t (those below the window)
          const uint32_t lo2 = (uint32_t)(kTpWin - 1 - t) << 8;
          const uint32_t top2 = min(lo2 + 255u, lo - 1u);
          if (tid == t) s.bf[1] = incl - m;  // the mass above the coarse bin
          __syncthreads();
          const float above2 = s.bf[1];
          s.hist.u[tid] = 0u;
          __syncthreads();
          tp_reread(vp, nvec, [&](const float* x) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t key = key_bf16(x[k]);
              if (key >= lo2 && key <= top2) atomicAdd(&s.hist.u[top2 - key], 1u);
            }
          });
          __syncthreads();
          const uint32_t c2 = (uint32_t)tid <= top2 - lo2 ? s.hist.u[tid] : 0u;
          m = c2 ? (float)c2 * ex2(fmaf(val_bf16(top2 - (uint32_t)tid), c, -mref)) : 0.f;
          incl = above2 + tp_scan(m, &tot, s, par);
          t = tp_first(incl >= target, s);
          if (t != INT_MAX) {
            if (tid == t) {
              s.bi[1] = (int)(top2 - (uint32_t)t);
              s.bf[0] = incl;
            }
          } else if (tid == 0) {  // rounding: the whole coarse bin
            s.bi[1] = (int)lo2;
            s.bf[0] = above2 + tot;
          }
        }
      }
      __syncthreads();
      tau = (uint32_t)s.bi[1];
      cum = s.bf[0];
    }
    if (tid == 0) {
      p.rstat[g] = make_float4(M, S, cum, __uint_as_float(tau));
      gather(p, g, row, 0, p.V, token_of(p, g));
    }
    __syncthreads();  // the histogram and red[] are free for the next row
  }
}

}  // namespace

cudaError_t launch_rows(const Params& p, int dtype, cudaStream_t stream) {
  if (p.topp) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.rows_grid);
    cfg.blockDim = dim3(kTpThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, topp_rows_kernel, p);
  }
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
