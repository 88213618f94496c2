// sv_kernels.cu — the verify-step kernels of libspecverify (sm_103a).
//
// verify_kernel: one persistent kernel per call. Each CTA has one producer
// warp, eight consumer warps and one publisher warp around a ring of
// shared-memory stages. The producer takes the next chunk of the call (up to
// eight 32 KB tiles of one logit row) from a global work counter and moves
// each tile from HBM into a stage with a 1-D bulk copy that completes on the
// stage's mbarrier; the consumers reduce the tile and hand the stage back; the
// publisher combines the warps' partials per chunk and finishes rows. Chunks
// are numbered sequence-major, so the rows of one sequence are read close
// together in time and stay in L2 for the second look the draw needs.
//
// Cross-CTA hand-off is "the last arriver does the work", never a wait on
// another CTA's progress: the publisher that counts the last chunk of a row
// finalises the row (its normaliser, its top-p cut or its argmax), and the one
// that counts the last row of a sequence queues the sequence's tail (or the
// chunks of its split draw) on a global ticket queue, which CTAs drain once
// their own streaming is over. A split draw's last chunk finishes the draw.
//
// verify_seq_kernel (one CTA per sequence, the sequence staged in shared
// memory) and verify_warp_kernel (one warp per sequence, from global memory)
// serve sampling calls whose rows are short.
//
// Per-row quantities (sampling mode), with c = log2(e)/T:
//   M   = max_v l_v                       (raw stored logit)
//   Mc  = fl(M * c)
//   s   = sum_v 2^(l_v * c - Mc)           = sum_v exp((l_v - M)/T)
//   cum = sum_{v : l_v >= tau} 2^(l_v * c - Mc)   (= s without top-p)
// so p'(v) = 2^(l_v * c - Mc) / cum on the nucleus {l_v >= tau}, and
//   alpha_i = min(1, p'_i(x_i) / q'_i(x_i))
//           = min(1, 2^(a_p - a_q) * cum_q / cum_p),  a = fma(l_x, c, -Mc).
#include "sv_device.cuh"
#include "sv_kernels.h"
#include "sv_df.cuh"
#include "sv_refine.h"

#include <cfloat>
#include <climits>
#include <mutex>
#include <set>
#include <utility>

namespace sv {

// Raises a kernel's dynamic shared-memory limit to `bytes`, once per (kernel,
// device): the attribute belongs to the current device's context, so a
// process that calls on several devices raises it on each. Not a stream
// operation; kept out of later calls so that those can be graph-captured.
static cudaError_t raise_smem_limit(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done.insert({kernel, dev});
  return e;
}

// ------------------------------------------------------------------ layout ---

struct RowStat {
  float M;       // sampling: row max (NaN = invalid row); argmax: max value (NaN = invalid)
  float s;       // sampling: normaliser relative to Mc
  float cum;     // sampling: nucleus mass relative to Mc (= s without top-p)
  uint32_t tau;  // sampling: nucleus cut key (0 = keep all); argmax: the argmax index
};

__device__ __forceinline__ RowStat rs_load(const Params& p, int64_t idx) {
  const float4 v = __ldcg(p.rowstat + idx);
  RowStat r;
  r.M = v.x;
  r.s = v.y;
  r.cum = v.z;
  r.tau = __float_as_uint(v.w);
  return r;
}
__device__ __forceinline__ void rs_store(const Params& p, int64_t idx, const RowStat& r) {
  p.rowstat[idx] = make_float4(r.M, r.s, r.cum, __uint_as_float(r.tau));
}

struct TileDesc {
  const char* row;
  int64_t e0, e1;    // element range of the tile in its row
  int64_t ie0;       // first interior element
  int64_t w;         // chunk id (-1: no more work)
  int64_t rowid;     // b * RS + r
  uint32_t ibytes;   // interior bytes (multiple of 16), 0 if none
  int nh;            // head elements [e0, e0 + nh)
  int nt;            // tail elements [e1 - nt, e1)
  int last;          // last tile of its chunk
};

// Warp roles: warps 0-7 consume tiles, warp 8 (one lane) produces them,
// warp 9 (one lane) publishes chunk partials and finishes rows.
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kPublisherWarp = kConsumerWarps + 1;
constexpr int kAllThreads = (kConsumerWarps + 2) * 32;
constexpr int kPartSlots = 4;   // chunk partials in flight from consumers to the publisher
constexpr int kTaskSlots = 64;  // collective tasks in flight from the publisher to the consumers

struct alignas(16) Shared {
  uint64_t full[kMaxStages];     // tile landed in the stage (producer -> consumers)
  uint64_t empty[kMaxStages];    // stage read by all consumer warps (consumers -> producer)
  uint64_t pfull[kPartSlots];    // chunk partial written by all consumer warps
  uint64_t pempty[kPartSlots];   // chunk partial taken by the publisher
  uint64_t pdone;                // publisher finished
  uint64_t dbar[2];              // the draw's row pieces landed in ring half 0 / 1
  uint32_t dcount[2];            // pieces issued so far on dbar[0] / dbar[1]
  TileDesc td[kMaxStages];       // what the stage holds, decoded once by the producer
  float red_m[kPartSlots][kConsumerWarps];
  float red_s[kPartSlots][kConsumerWarps];
  int64_t red_i[kPartSlots][kConsumerWarps];
  int64_t pw[kPartSlots];        // chunk id of the partial (-1: consumers are done)
  int64_t prow[kPartSlots];      // row of that chunk (b * RS + r)
  int64_t tq[kTaskSlots];        // task: row id (top-p cut) or -(b+1) (sequence tail)
  float tq_m[kTaskSlots], tq_s[kTaskSlots];
  int tq_tail;                   // written by the publisher only
  int tq_head;                   // written by consumer thread 0 only
  int snap[2];                   // tq_tail as seen at a chunk boundary, by chunk parity
  union {
    uint32_t u[kHistBins];
    float f[kHistBins];
  } hist;
  float cells[kMaxCells];
  float scan[kConsumerWarps];
  float bf[8];
  int64_t bl[4];
  int bi[8];
  int flag;
};

size_t shared_bytes(int stages) { return (size_t)stages * kTileBytes + sizeof(Shared); }

template <typename E>
struct ET;
template <>
struct ET<float> {
  static constexpr int kSize = 4;
  static constexpr int kPerVec = 4;  // elements per 16-byte vector
  static constexpr int kKeyBits = 32;
  __device__ static float load(const char* row, int64_t e) { return __ldg(reinterpret_cast<const float*>(row) + e); }
  __device__ static uint32_t key(float x) { return key_f32(x); }
  __device__ static float val(uint32_t k) { return val_f32(k); }
};
template <>
struct ET<uint16_t> {
  static constexpr int kSize = 2;
  static constexpr int kPerVec = 8;
  static constexpr int kKeyBits = 16;
  __device__ static float load(const char* row, int64_t e) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row) + e)) << 16);
  }
  __device__ static uint32_t key(float x) { return key_bf16(x); }
  __device__ static float val(uint32_t k) { return val_bf16(k); }
};

// Start of row r of sequence b.
template <typename E, int MODE>
__device__ __forceinline__ const char* row_ptr(const Params& p, int64_t b, int r) {
  constexpr int S = ET<E>::kSize;
  if (MODE == kGreedy) return p.a + ((b * p.RS + r) * p.V) * S;
  if (r <= p.K) return p.a + ((b * (p.K + 1) + r) * p.V) * S;
  return p.d + ((b * p.K + (r - p.K - 1)) * p.V) * S;
}

// One ring stage's tile, decoded once by the producer. The interior is the
// 16-byte aligned part of the tile, moved by the bulk copy; the unaligned
// head and tail elements (rows whose byte length is not a multiple of 16)
// are read directly by the consumers.
// A chunk is up to CT consecutive tiles of one row, the unit of scheduling and
// of publishing a partial. Chunk ids run sequence-major: (b, r, ci).
struct ChunkId {
  int64_t b;
  int r;
  int64_t k0;  // first tile
  int n;       // tiles in the chunk
};

__device__ __forceinline__ ChunkId decode_chunk(const Params& p, int64_t w) {
  ChunkId c;
  const int64_t per = (int64_t)p.RS * p.NC;
  c.b = w / per;
  const int64_t rem = w - c.b * per;
  c.r = (int)(rem / p.NC);
  const int64_t ci = rem - (int64_t)c.r * p.NC;
  c.k0 = ci * p.CT;
  c.n = (int)min((int64_t)p.CT, p.NT - c.k0);
  return c;
}

template <typename E, int MODE>
__device__ __forceinline__ void decode_tile(const Params& p, const ChunkId& ch, int64_t k, TileDesc& t) {
  constexpr int S = ET<E>::kSize;
  t.row = row_ptr<E, MODE>(p, ch.b, ch.r);
  t.rowid = ch.b * p.RS + ch.r;
  t.e0 = k * p.TE;
  t.e1 = min(t.e0 + p.TE, p.V);
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(t.row + t.e0 * S);
  const uintptr_t a1 = reinterpret_cast<uintptr_t>(t.row + t.e1 * S);
  const uintptr_t A = (a0 + 15) & ~uintptr_t(15);
  const uintptr_t Z = a1 & ~uintptr_t(15);
  if (A < Z) {
    t.ibytes = (uint32_t)(Z - A);
    t.nh = (int)((A - a0) / S);
    t.nt = (int)((a1 - Z) / S);
    t.ie0 = t.e0 + t.nh;
  } else {
    t.ibytes = 0;
    t.nh = (int)(t.e1 - t.e0);
    t.nt = 0;
    t.ie0 = t.e1;
  }
}

// ------------------------------------------------ online (max, sum) ---------
// (m, s): m the running raw max, s = sum 2^(l*c - mref(m)) with
// mref(m) = fl(m*c). The reference is rounded explicitly (never fused into a
// neighbouring add), so that every rescale factor 2^(mref(m) - mref(m')) is
// exactly the shift between the references the terms were summed against.
__device__ __forceinline__ float mref(float m, float c) { return __fmul_rn(m, c); }
__device__ __forceinline__ float rescale(float m_old, float m_new, float c) {
  return (m_old == -INFINITY) ? 0.f : ex2(__fsub_rn(mref(m_old, c), mref(m_new, c)));
}
__device__ __forceinline__ void ms_combine(float& m, float& s, float m2, float s2, float c) {
  const float nm = fmax_nan(m, m2);
  if (nm == -INFINITY) {
    m = nm;
    s = 0.f;
    return;
  }
  s = s * rescale(m, nm, c) + s2 * rescale(m2, nm, c);
  m = nm;
}
__device__ __forceinline__ void ms_scalar(float& m, float& s, float x, float c) {
  const float nm = fmax_nan(m, x);
  if (nm != m) {  // also taken when nm is NaN
    s *= rescale(m, nm, c);
    m = nm;
  }
  if (m == -INFINITY) return;
  s += ex2(fmaf(x, c, -mref(m, c)));
}
__device__ __forceinline__ void ms_vec(float& m, float& s0, float& s1, const uint4 q, float c, uint16_t) {
  const uint32_t mm = bf2_max_nan(bf2_max_nan(q.x, q.y), bf2_max_nan(q.z, q.w));
  const float vmax = fmax_nan(bf_lo(mm), bf_hi(mm));
  const float nm = fmax_nan(m, vmax);
  if (nm != m) {
    const float f = rescale(m, nm, c);
    s0 *= f;
    s1 *= f;
    m = nm;
  }
  if (m == -INFINITY) return;
  const float nmc = -mref(m, c);
  s0 += ex2(fmaf(bf_lo(q.x), c, nmc));
  s1 += ex2(fmaf(bf_hi(q.x), c, nmc));
  s0 += ex2(fmaf(bf_lo(q.y), c, nmc));
  s1 += ex2(fmaf(bf_hi(q.y), c, nmc));
  s0 += ex2(fmaf(bf_lo(q.z), c, nmc));
  s1 += ex2(fmaf(bf_hi(q.z), c, nmc));
  s0 += ex2(fmaf(bf_lo(q.w), c, nmc));
  s1 += ex2(fmaf(bf_hi(q.w), c, nmc));
}
__device__ __forceinline__ void ms_vec(float& m, float& s0, float& s1, const uint4 q, float c, float) {
  const float x0 = __uint_as_float(q.x), x1 = __uint_as_float(q.y), x2 = __uint_as_float(q.z),
              x3 = __uint_as_float(q.w);
  const float vmax = fmax_nan(fmax_nan(x0, x1), fmax_nan(x2, x3));
  const float nm = fmax_nan(m, vmax);
  if (nm != m) {
    const float f = rescale(m, nm, c);
    s0 *= f;
    s1 *= f;
    m = nm;
  }
  if (m == -INFINITY) return;
  const float nmc = -mref(m, c);
  s0 += ex2(fmaf(x0, c, nmc));
  s1 += ex2(fmaf(x1, c, nmc));
  s0 += ex2(fmaf(x2, c, nmc));
  s1 += ex2(fmaf(x3, c, nmc));
}

// A thread's share of a tile, eight 16-byte vectors at a time: all eight are
// loaded first, one packed max covers them, the running reference moves once,
// and the exponentials are independent of each other (four accumulators).
// Vectors past the tile are -inf, which adds nothing.
constexpr int kVecBatch = 8;
__device__ __forceinline__ uint4 neg_inf_vec(uint16_t) { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
__device__ __forceinline__ uint4 neg_inf_vec(float) { return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u); }
__device__ __forceinline__ float vec_max(const uint4& q, uint16_t) {
  const uint32_t mm = bf2_max_nan(bf2_max_nan(q.x, q.y), bf2_max_nan(q.z, q.w));
  return fmax_nan(bf_lo(mm), bf_hi(mm));
}
__device__ __forceinline__ float vec_max(const uint4& q, float) {
  return fmax_nan(fmax_nan(__uint_as_float(q.x), __uint_as_float(q.y)),
                  fmax_nan(__uint_as_float(q.z), __uint_as_float(q.w)));
}
__device__ __forceinline__ void vec_exp_add(const uint4& q, float c, float nmc, float s[4], uint16_t) {
  s[0] += ex2(fmaf(bf_lo(q.x), c, nmc));
  s[1] += ex2(fmaf(bf_hi(q.x), c, nmc));
  s[2] += ex2(fmaf(bf_lo(q.y), c, nmc));
  s[3] += ex2(fmaf(bf_hi(q.y), c, nmc));
  s[0] += ex2(fmaf(bf_lo(q.z), c, nmc));
  s[1] += ex2(fmaf(bf_hi(q.z), c, nmc));
  s[2] += ex2(fmaf(bf_lo(q.w), c, nmc));
  s[3] += ex2(fmaf(bf_hi(q.w), c, nmc));
}
__device__ __forceinline__ void vec_exp_add(const uint4& q, float c, float nmc, float s[4], float) {
  s[0] += ex2(fmaf(__uint_as_float(q.x), c, nmc));
  s[1] += ex2(fmaf(__uint_as_float(q.y), c, nmc));
  s[2] += ex2(fmaf(__uint_as_float(q.z), c, nmc));
  s[3] += ex2(fmaf(__uint_as_float(q.w), c, nmc));
}
template <typename E>
__device__ __forceinline__ void ms_tile(const uint4* sv, int nvec, int tid, float c, float& m, float s[4]) {
  for (int v0 = tid; v0 < nvec; v0 += kVecBatch * kConsumerThreads) {
    uint4 q[kVecBatch];
#pragma unroll
    for (int k = 0; k < kVecBatch; ++k) {
      const int v = v0 + k * kConsumerThreads;
      q[k] = v < nvec ? sv[v] : neg_inf_vec(E());
    }
    float vmax = vec_max(q[0], E());
#pragma unroll
    for (int k = 1; k < kVecBatch; ++k) vmax = fmax_nan(vmax, vec_max(q[k], E()));
    const float nm = fmax_nan(m, vmax);
    if (nm != m) {  // also taken when nm is NaN
      const float f = rescale(m, nm, c);
      s[0] *= f;
      s[1] *= f;
      s[2] *= f;
      s[3] *= f;
      m = nm;
    }
    if (m == -INFINITY) continue;
    const float nmc = -mref(m, c);
#pragma unroll
    for (int k = 0; k < kVecBatch; ++k) vec_exp_add(q[k], c, nmc, s, E());
  }
}

// ---------------------------------------------------- argmax (lowest index) --
// (v, i): best value and its index; i < 0 means "nothing seen but -inf".
__device__ __forceinline__ bool am_better(float v2, int64_t i2, float v1, int64_t i1) {
  if (i2 < 0) return false;
  if (i1 < 0) return true;
  return (v2 > v1) || (v2 == v1 && i2 < i1);
}
__device__ __forceinline__ void am_scalar(float& v, int64_t& i, bool& nan, float x, int64_t e) {
  if (x != x) {
    nan = true;
    return;
  }
  if (am_better(x, e, v, i)) {
    v = x;
    i = e;
  }
}
__device__ __forceinline__ void am_vec(float& v, int64_t& i, bool& nan, const uint4 q, int64_t e, uint16_t) {
  const uint32_t mm = bf2_max_nan(bf2_max_nan(q.x, q.y), bf2_max_nan(q.z, q.w));
  const float vmax = fmax_nan(bf_lo(mm), bf_hi(mm));
  if (vmax != vmax) {
    nan = true;
    return;
  }
  if (vmax > v || i < 0) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    int k = 0;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      const float x = (j & 1) ? bf_hi(w[j >> 1]) : bf_lo(w[j >> 1]);
      if (x == vmax) k = j;
    }
    v = vmax;
    i = e + k;
  }
}
__device__ __forceinline__ void am_vec(float& v, int64_t& i, bool& nan, const uint4 q, int64_t e, float) {
  const float x[4] = {__uint_as_float(q.x), __uint_as_float(q.y), __uint_as_float(q.z), __uint_as_float(q.w)};
  const float vmax = fmax_nan(fmax_nan(x[0], x[1]), fmax_nan(x[2], x[3]));
  if (vmax != vmax) {
    nan = true;
    return;
  }
  if (vmax > v || i < 0) {
    int k = 0;
#pragma unroll
    for (int j = 3; j >= 0; --j)
      if (x[j] == vmax) k = j;
    v = vmax;
    i = e + k;
  }
}

// ---------------------------------------------- weights for the inverse CDF --
// Eight consecutive elements starting at e (a multiple of 8); -inf past V.
template <typename E>
__device__ __forceinline__ void load8(const char* row, int64_t e, int64_t V, bool aligned, float out[8]) {
  if (aligned && e + 8 <= V) {
    if (ET<E>::kSize == 2) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(row + e * 2));
      out[0] = bf_lo(q.x); out[1] = bf_hi(q.x); out[2] = bf_lo(q.y); out[3] = bf_hi(q.y);
      out[4] = bf_lo(q.z); out[5] = bf_hi(q.z); out[6] = bf_lo(q.w); out[7] = bf_hi(q.w);
    } else {
      const uint4 q0 = __ldg(reinterpret_cast<const uint4*>(row + e * 4));
      const uint4 q1 = __ldg(reinterpret_cast<const uint4*>(row + e * 4 + 16));
      out[0] = __uint_as_float(q0.x); out[1] = __uint_as_float(q0.y);
      out[2] = __uint_as_float(q0.z); out[3] = __uint_as_float(q0.w);
      out[4] = __uint_as_float(q1.x); out[5] = __uint_as_float(q1.y);
      out[6] = __uint_as_float(q1.z); out[7] = __uint_as_float(q1.w);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) out[k] = (e + k < V) ? ET<E>::load(row, e + k) : -INFINITY;
  }
}

// The smallest stored value whose key is >= k (keys at or below key(-inf)
// hold no value but NaN, which valid rows do not contain): x >= key_floor(k)
// exactly when key(x) >= k.
template <typename E>
__device__ __forceinline__ float key_floor(uint32_t k) {
  return k <= ET<E>::key(-INFINITY) ? -INFINITY : ET<E>::val(k);
}

// Eight consecutive elements of a row piece staged in shared memory (the
// piece starts at element e0 of the row; -inf past V).
template <typename E>
__device__ __forceinline__ void load8_smem(const char* piece, int64_t e_in_piece, int64_t e, int64_t V,
                                           float out[8]) {
  if (ET<E>::kSize == 2) {
    const uint4 q = *reinterpret_cast<const uint4*>(piece + e_in_piece * 2);
    out[0] = bf_lo(q.x); out[1] = bf_hi(q.x); out[2] = bf_lo(q.y); out[3] = bf_hi(q.y);
    out[4] = bf_lo(q.z); out[5] = bf_hi(q.z); out[6] = bf_lo(q.w); out[7] = bf_hi(q.w);
  } else {
    const uint4 q0 = *reinterpret_cast<const uint4*>(piece + e_in_piece * 4);
    const uint4 q1 = *reinterpret_cast<const uint4*>(piece + e_in_piece * 4 + 16);
    out[0] = __uint_as_float(q0.x); out[1] = __uint_as_float(q0.y);
    out[2] = __uint_as_float(q0.z); out[3] = __uint_as_float(q0.w);
    out[4] = __uint_as_float(q1.x); out[5] = __uint_as_float(q1.y);
    out[6] = __uint_as_float(q1.z); out[7] = __uint_as_float(q1.w);
  }
  if (e + 8 > V) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (e + k >= V) out[k] = -INFINITY;
  }
}

// The sampler's weights over one row: w_v = p'(v) up to a constant, or, with
// two rows, w_v = max(0, p'(v) - q'(v)).
template <typename E, bool kResidual, bool kTopp>
struct Weights {
  const char* rp;
  const char* rq;
  int64_t V;
  float c, nMcp, nMcq, ip, iq;
  float tp, tq;  // the nucleus: elements below tp (tq) weigh nothing in p' (q'); -inf without top-p
  bool aligned;
  static constexpr bool kRes = kResidual;
  __device__ __forceinline__ void w8(int64_t e, float w[8]) const {
    float lp[8], lq[8];
    load8<E>(rp, e, V, aligned, lp);
    if (kResidual) load8<E>(rq, e, V, aligned, lq);
    weigh(lp, lq, w);
  }
  // The same weights for elements staged in shared memory.
  __device__ __forceinline__ void w8_staged(const char* sp, const char* sq, int64_t e_in_piece, int64_t e,
                                            float w[8]) const {
    float lp[8], lq[8];
    load8_smem<E>(sp, e_in_piece, e, V, lp);
    if (kResidual) load8_smem<E>(sq, e_in_piece, e, V, lq);
    weigh(lp, lq, w);
  }
  __device__ __forceinline__ void weigh(const float lp[8], const float lq[8], float w[8]) const {
    if (kResidual) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float ep = ex2(fmaf(lp[k], c, nMcp));
        float eq = ex2(fmaf(lq[k], c, nMcq));
        if (kTopp) {
          ep = lp[k] >= tp ? ep : 0.f;
          eq = lq[k] >= tq ? eq : 0.f;
        }
        w[k] = fmaxf(0.f, fmaf(ep, ip, -eq * iq));
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float ep = ex2(fmaf(lp[k], c, nMcp));
        w[k] = (!kTopp || lp[k] >= tp) ? ep : 0.f;
      }
    }
  }
};

// Cell sums of one piece staged in shared memory (row p at sp, row q at sq,
// elements e0 .. of the row) for cells [cfirst, clast), written to dst[cell]:
// a warp takes four of its cells at a time, all their weights first, then the
// four warp reductions interleaved. Lane l sums elements l*8m .. of a cell.
template <typename E, class WF>
__device__ __forceinline__ void cells_piece(const WF& wf, const char* sp, const char* sq, int cfirst, int clast,
                                            int64_t e0, int64_t CE, float* dst, int warp, int lane) {
  const int64_t m = CE / 256;
  constexpr int UC = 4;
  for (int cb = cfirst + warp; cb < clast; cb += kConsumerWarps * UC) {
    float acc[UC];
#pragma unroll
    for (int k = 0; k < UC; ++k) {
      const int cc = cb + k * kConsumerWarps;
      float a = 0.f;
      if (cc < clast) {
        for (int64_t q = 0; q < m; ++q) {
          const int64_t e = (int64_t)cc * CE + (lane * m + q) * 8;
          float w[8];
          wf.w8_staged(sp, sq, e - e0, e, w);
          a += ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
        }
      }
      acc[k] = a;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int k = 0; k < UC; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
    }
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < UC; ++k) {
        const int cc = cb + k * kConsumerWarps;
        if (cc < clast) dst[cc] = acc[k];
      }
    }
  }
}

// Inverse-CDF draw by the 256 consumer threads: the smallest t with
// sum_{v<=t} w_v > u * sum_v w_v. Returns -1 when every weight is zero.
// The row is cut into cells of CE = 256*m elements (at most kMaxCells cells);
// pass A sums each cell, then one warp scans the cell sums to find the cell
// holding the crossing and rescans that cell alone (cdf_cross). Pass A may
// be split over CTAs by ranges of cells (draw_chunk).
// Pass A over cells [cbeg, cend) from shared memory, sums to dst[cell]: the
// row (or the two rows) is moved in pieces of whole cells into the two halves
// of the idle tile ring by bulk copies, the next piece landing while the
// current one is summed. Returns false (having touched nothing) when it cannot
// run: unaligned rows, or a ring too small for one cell per row.
template <typename E, class WF>
__device__ bool cells_staged(const WF& wf, int64_t V, int64_t CE, int cbeg, int cend, float* dst, char* ring,
                             size_t ring_bytes, Shared& sh, int tid, const uint32_t* ctl_status) {
  constexpr int S = ET<E>::kSize;
  constexpr int nrows = WF::kRes ? 2 : 1;
  if (!wf.aligned || ring_bytes == 0) return false;
  const size_t half = (ring_bytes / 2) & ~size_t(15);
  int64_t cells_per_piece = (int64_t)(half / nrows / S) / CE;
  if (cells_per_piece < 1) return false;
  const int64_t P = cells_per_piece * CE;  // elements per row per piece
  const int64_t ebeg = (int64_t)cbeg * CE, eend = min(V, (int64_t)cend * CE);
  const int64_t npieces = (eend - ebeg + P - 1) / P;
  const int warp = tid >> 5, lane = tid & 31;
  cbar();  // everyone has read dcount, and nothing reads the ring any more
  const uint32_t c0 = sh.dcount[0], c1 = sh.dcount[1];
  auto issue = [&](int64_t k) {  // thread 0 only
    const int buf = (int)(k & 1);
    const int64_t e0 = ebeg + k * P;
    const int64_t n = min(P, eend - e0);
    const uint32_t bytes = (uint32_t)(n * S);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(&sh.dbar[buf], bytes * (uint32_t)nrows);
    char* dst = ring + (size_t)buf * half;
    bulk_g2s(dst, wf.rp + e0 * S, bytes, &sh.dbar[buf]);
    if (nrows == 2) bulk_g2s(dst + (size_t)P * S, wf.rq + e0 * S, bytes, &sh.dbar[buf]);
  };
  if (tid == 0) {
    issue(0);
    if (npieces > 1) issue(1);
  }
  bool ok = true;
  for (int64_t k = 0; k < npieces; ++k) {
    const int buf = (int)(k & 1);
    const uint32_t use = (buf ? c1 : c0) + (uint32_t)(k >> 1);  // uses of this barrier before this one
    if (!mbar_wait(&sh.dbar[buf], use & 1u)) ok = false;
    if (cbar_or(!ok)) {
      ok = false;
      break;
    }
    const char* sp = ring + (size_t)buf * half;
    const char* sq = sp + (size_t)P * S;
    const int64_t e0 = ebeg + k * P;
    const int cfirst = (int)(e0 / CE);
    const int clast = (int)min((int64_t)cend, (e0 + P) / CE);
    cells_piece<E>(wf, sp, sq, cfirst, clast, e0, CE, dst, warp, lane);
    cbar();  // the half is free again
    if (tid == 0 && k + 2 < npieces) issue(k + 2);
  }
  if (tid == 0) {
    const int64_t used0 = (npieces + 1) / 2, used1 = npieces / 2;
    sh.dcount[0] = c0 + (uint32_t)used0;
    sh.dcount[1] = c1 + (uint32_t)used1;
    if (!ok) {  // a wait ran out: let what is in flight land, then report
      atomicOr(const_cast<uint32_t*>(ctl_status), kStatusTimeout);
      (void)mbar_wait(&sh.dbar[0], (c0 + (uint32_t)used0 - 1u) & 1u);
      if (used1) (void)mbar_wait(&sh.dbar[1], (c1 + (uint32_t)used1 - 1u) & 1u);
    }
  }
  cbar();
  return ok;
}

// Pass A over cells [cbeg, cend) from global memory, sums to dst[cell]: four
// cells per warp at a time so that their loads are in flight together.
template <typename E, class WF>
__device__ void cells_global(const WF& wf, int64_t CE, int cbeg, int cend, float* dst, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t m = CE / 256;
  constexpr int U = 4;
  for (int c0 = cbeg + warp; c0 < cend; c0 += kConsumerWarps * U) {
    float sum[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int cc = c0 + k * kConsumerWarps;
      float acc = 0.f;
      if (cc < cend) {
        for (int64_t q = 0; q < m; ++q) {
          float w[8];
          wf.w8(cc * CE + (lane * m + q) * 8, w);
          acc += ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
        }
      }
      sum[k] = acc;
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const float t = warp_sum(sum[k]);
      const int cc = c0 + k * kConsumerWarps;
      if (lane == 0 && cc < cend) dst[cc] = t;
    }
  }
}

// The crossing, from the cell sums in sh.cells[0, ncells): one warp scans
// them, finds the cell holding u * Z and walks it. Returns the token to every
// consumer thread (-1 when every weight is zero).
// Out of line: it runs once per draw, and inlined into the streaming kernel
// its double-float arithmetic pushed registers of the streaming loop to spill.
template <typename E, class WF>
__device__ __noinline__ int64_t cdf_cross(const WF& wf, int64_t V, float u, Shared& sh, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t CE = cell_elems(V);
  const int64_t m = CE / 256;
  const int ncells = (int)((V + CE - 1) / CE);
  if (warp == 0) {
    // The running sums over the cells are carried in double-float: they reach
    // the size of Z, where fp32 would round at ~6e-8*Z.
    const int cpl = (ncells + 31) / 32;
    const int c0 = min(ncells, lane * cpl), c1 = min(ncells, c0 + cpl);
    df ls{0.f, 0.f};
    for (int cc = c0; cc < c1; ++cc) ls = df_add(ls, df{sh.cells[cc], 0.f});
    df incl = ls;
    // (not unrolled: this runs once per draw, cold in the instruction cache)
#pragma unroll 1
    for (int o = 1; o < 32; o <<= 1) {
      df t2;
      t2.h = __shfl_up_sync(0xffffffffu, incl.h, o);
      t2.l = __shfl_up_sync(0xffffffffu, incl.l, o);
      if (lane >= o) incl = df_add(incl, t2);
    }
    df Zd;
    Zd.h = __shfl_sync(0xffffffffu, incl.h, 31);
    Zd.l = __shfl_sync(0xffffffffu, incl.l, 31);
    const float Z = Zd.h;
    int64_t t = -1;
    int settled = 0;  // the fp32 walk found the token clear of its interval's edges
    if (Z > 0.f) {
      const df Tg = df_mul_f(Zd, u);
      df run = df_sub(incl, ls);
      int hit = -1;
      for (int cc = c0; cc < c1; ++cc) {
        const df nr = df_add(run, df{sh.cells[cc], 0.f});
        if (df_gt(nr, Tg)) {
          hit = cc;
          break;
        }
        run = nr;
      }
      const unsigned bal = __ballot_sync(0xffffffffu, hit >= 0);
      int cstar;
      float Tl = 0.f;  // what is left of the target inside the crossing cell
      bool last_positive = false;
      if (bal) {
        const int fl = __ffs(bal) - 1;
        cstar = __shfl_sync(0xffffffffu, hit, fl);
        df rn;
        rn.h = __shfl_sync(0xffffffffu, run.h, fl);
        rn.l = __shfl_sync(0xffffffffu, run.l, fl);
        const df rem = df_sub(Tg, rn);
        Tl = rem.h + rem.l;
      } else {  // u*Z at or past the total after rounding: the last positive weight
        int last = -1;
        for (int cc = c0; cc < c1; ++cc)
          if (sh.cells[cc] > 0.f) last = cc;
        for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
        cstar = last;
        last_positive = true;
      }
      // the crossing cell: lane l owns elements [cstar*CE + l*8m, +8m)
      const int64_t base = (int64_t)cstar * CE + (int64_t)lane * 8 * m;
      float ls2 = 0.f;
      for (int64_t q = 0; q < m; ++q) {
        float w[8];
        wf.w8(base + q * 8, w);
        if (q == 0) {  // kept in shared memory for the walk below (no second load)
#pragma unroll
          for (int k = 0; k < 8; ++k) sh.hist.f[lane * 8 + k] = w[k];
        }
        ls2 += ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
      }
      __syncwarp();
      const float incl2 = warp_incl_scan(ls2, lane);
      const float excl2 = incl2 - ls2;
      int64_t mine = -1;
      if (!last_positive) {
        const unsigned bal2 = __ballot_sync(0xffffffffu, excl2 + ls2 > Tl);
        if (bal2) {
          const int fl2 = __ffs(bal2) - 1;
          if (lane == fl2) {
            float acc = excl2;
            int64_t lastpos = -1;
            for (int64_t q = 0; q < m && mine < 0; ++q) {
              float w[8];
              if (q == 0) {
#pragma unroll
                for (int k = 0; k < 8; ++k) w[k] = sh.hist.f[lane * 8 + k];
              } else {
                wf.w8(base + q * 8, w);
              }
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                if (mine < 0) {
                  const float prev = acc;
                  acc += w[k];
                  if (w[k] > 0.f) lastpos = base + q * 8 + k;
                  if (acc > Tl) {
                    mine = base + q * 8 + k;
                    // u*Z within the refine margin of an edge of the token's
                    // interval: too close for fp32 to be sure
                    settled = fminf(acc - Tl, Tl - prev) >= rf::kRefineMargin * Z;
                  }
                }
              }
            }
            if (mine < 0) mine = lastpos;  // rounding inside the lane
          }
          mine = __shfl_sync(0xffffffffu, mine, fl2);
          settled = __shfl_sync(0xffffffffu, settled, fl2);
        } else {
          last_positive = true;
        }
      }
      if (last_positive) {
        int64_t lastpos = -1;
        for (int64_t q = 0; q < m; ++q) {
          float w[8];
          wf.w8(base + q * 8, w);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (w[k] > 0.f) lastpos = base + q * 8 + k;
        }
        for (int o = 16; o > 0; o >>= 1) {
          const long long other = __shfl_xor_sync(0xffffffffu, (long long)lastpos, o);
          lastpos = max((long long)lastpos, other);
        }
        mine = lastpos;
      }
      t = mine;
      if (last_positive) settled = 0;
    }
    if (lane == 0) {
      sh.bl[0] = t;
      sh.bi[7] = settled;
    }
  }
  cbar();
  const int64_t t = sh.bl[0];
  cbar();
  return t;
}

// The whole draw in this CTA.
template <typename E, class WF>
__device__ int64_t cdf_draw(const WF& wf, int64_t V, float u, Shared& sh, int tid, char* ring, size_t ring_bytes,
                            const uint32_t* ctl_status) {
  const int64_t CE = cell_elems(V);
  const int ncells = (int)((V + CE - 1) / CE);
  if (!cells_staged<E>(wf, V, CE, 0, ncells, sh.cells, ring, ring_bytes, sh, tid, ctl_status))
    cells_global<E>(wf, CE, 0, ncells, sh.cells, tid);
  cbar();
  return cdf_cross<E>(wf, V, u, sh, tid);
}

// ------------------------------------------------ block-wide helpers ---------
// Exclusive prefix of one float per consumer thread; also returns the total.
__device__ __forceinline__ float block_excl_scan(float v, float& total, Shared& sh, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  const float incl = warp_incl_scan(v, lane);
  if (lane == 31) sh.scan[warp] = incl;
  cbar();
  float off = 0.f, tot = 0.f;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) {
    const float x = sh.scan[w];
    if (w < warp) off += x;
    tot += x;
  }
  cbar();
  total = tot;
  return off + incl - v;
}

// Calls f(element value) for every element of a row, spread over the
// consumer threads (16-byte loads when the row is aligned).
template <typename E, class F>
__device__ __forceinline__ void for_each_elem(const char* row, int64_t V, int tid, F&& f) {
  constexpr int PV = ET<E>::kPerVec;
  auto apply = [&](const uint4 q) {
    if (PV == 8) {
      f(bf_lo(q.x)); f(bf_hi(q.x)); f(bf_lo(q.y)); f(bf_hi(q.y));
      f(bf_lo(q.z)); f(bf_hi(q.z)); f(bf_lo(q.w)); f(bf_hi(q.w));
    } else {
      f(__uint_as_float(q.x)); f(__uint_as_float(q.y)); f(__uint_as_float(q.z)); f(__uint_as_float(q.w));
    }
  };
  if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) {
    const int64_t nv = V / PV;
    const uint4* rv = reinterpret_cast<const uint4*>(row);
    int64_t v = tid;
    // four 16-byte loads in flight per thread before any is used
    for (; v + 3 * kConsumerThreads < nv; v += 4 * kConsumerThreads) {
      uint4 q[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) q[k] = __ldg(rv + v + k * kConsumerThreads);
#pragma unroll
      for (int k = 0; k < 4; ++k) apply(q[k]);
    }
    for (; v < nv; v += kConsumerThreads) apply(__ldg(rv + v));
    for (int64_t e = nv * PV + tid; e < V; e += kConsumerThreads) f(ET<E>::load(row, e));
  } else {
    for (int64_t e = tid; e < V; e += kConsumerThreads) f(ET<E>::load(row, e));
  }
}

// Top-p cut of one row: the largest key tau whose upper set
// {v : key(l_v) >= tau} holds mass >= top_p * s, and that mass.
// Windows of kHistBins bins are laid below the current upper key; a bin is
// one exact key (counts times the key's weight) or, for fp32 rows first, a
// run of 2^sh keys (weights added per element). The window that holds the
// crossing is refined until the bins are exact keys.
template <typename E>
__device__ void topp_cut(const Params& p, Shared& sh, const char* row, float M, float s, int tid, uint32_t& tau,
                         float& cum) {
  const float c = p.c, nMc = -mref(M, p.c);
  const float target = p.top_p * s;
  uint32_t hi = ET<E>::key(M);
  int shf = (ET<E>::kKeyBits == 16) ? 0 : 16;
  float above = 0.f;
  for (int iter = 0; iter < 4096; ++iter) {
    const uint64_t span = (uint64_t)kHistBins << shf;
    const uint32_t lo = ((uint64_t)hi + 1 >= span) ? (uint32_t)((uint64_t)hi + 1 - span) : 0u;
    const int nb = (int)(((uint64_t)hi - lo) >> shf) + 1;
    for (int k = tid; k < kHistBins; k += kConsumerThreads) sh.hist.u[k] = 0u;
    cbar();
    const int s_ = shf;
    for_each_elem<E>(row, p.V, tid, [&](float x) {
      const uint32_t k = ET<E>::key(x);
      if (k >= lo && k <= hi) {
        const int bin = (int)((hi - k) >> s_);
        if (s_ == 0)
          atomicAdd(&sh.hist.u[bin], 1u);
        else
          atomicAdd(&sh.hist.f[bin], ex2(fmaf(x, c, nMc)));
      }
    });
    cbar();
    constexpr int PER = kHistBins / kConsumerThreads;
    float m[PER];
    float ls = 0.f;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int bin = tid * PER + j;
      float mj = 0.f;
      if (bin < nb) {
        if (shf == 0) {
          const uint32_t cnt = sh.hist.u[bin];
          mj = cnt ? (float)cnt * ex2(fmaf(ET<E>::val(hi - (uint32_t)bin), c, nMc)) : 0.f;
        } else {
          mj = sh.hist.f[bin];
        }
      }
      m[j] = mj;
      ls += mj;
    }
    float total;
    const float excl = block_excl_scan(ls, total, sh, tid);
    if (tid == 0) sh.bi[0] = INT_MAX;
    cbar();
    float run = excl;
    int hit = -1;
    float before = 0.f, mh = 0.f;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      if (hit < 0 && above + run + m[j] >= target) {
        hit = tid * PER + j;
        before = run;
        mh = m[j];
      }
      run += m[j];
    }
    if (hit >= 0) atomicMin(&sh.bi[0], hit);
    cbar();
    const int b = sh.bi[0];
    if (b != INT_MAX && hit == b) {
      sh.bf[0] = before;
      sh.bf[1] = mh;
    }
    cbar();
    if (b != INT_MAX) {
      const float bb = sh.bf[0], bm = sh.bf[1];
      if (shf == 0) {
        tau = hi - (uint32_t)b;
        cum = above + bb + bm;
        cbar();
        return;
      }
      above += bb;
      hi = hi - ((uint32_t)b << shf);
      shf = (shf > 11) ? shf - 11 : 0;
    } else {
      above += total;
      if (lo == 0u) {  // every key seen: rounding left the mass short of top_p * s
        tau = 0u;
        cum = above;
        cbar();
        return;
      }
      hi = lo - 1u;
    }
    cbar();
  }
  tau = 0u;
  cum = s;
}

// ------------------------------------------------------ sequence tails -------

// What a sequence's accept scan decided, for its draw.
struct DrawJob {
  float uK;          // the draw's uniform
  float nMcp, nMcq;  // -M c of the p and q rows
  float ip, iq;      // 1 / nucleus mass of the p and q rows
  float tp, tq;      // nucleus thresholds (-inf without top-p)
  int j;             // the rejected position (K: bonus draw)
};

__device__ __forceinline__ bool rows_aligned(const Params& p, int esz) {
  return (p.V * esz) % 16 == 0 && (reinterpret_cast<uintptr_t>(p.a) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(p.d) & 15) == 0;
}

template <typename E, bool kTopp>
__device__ __forceinline__ Weights<E, true, kTopp> residual_weights(const Params& p, int64_t b, const DrawJob& jb) {
  return Weights<E, true, kTopp>{row_ptr<E, kSample>(p, b, jb.j), row_ptr<E, kSample>(p, b, p.K + 1 + jb.j), p.V,
                                 p.c, jb.nMcp, jb.nMcq, jb.ip, jb.iq, jb.tp, jb.tq, rows_aligned(p, ET<E>::kSize)};
}
template <typename E, bool kTopp>
__device__ __forceinline__ Weights<E, false, kTopp> target_weights(const Params& p, int64_t b, const DrawJob& jb) {
  return Weights<E, false, kTopp>{row_ptr<E, kSample>(p, b, jb.j), nullptr, p.V, p.c, jb.nMcp, 0.f, 1.f, 0.f, jb.tp,
                                  -INFINITY, rows_aligned(p, ET<E>::kSize)};
}

// The draw of sequence b in this CTA alone: the residual at a rejection
// (p'_j itself if that is all zero), or p'_K for the bonus token.
// Appends a draw the fp32 walk could not settle to the refine kernel's list
// (the draw's rows, their largest raw logits and nucleus cuts, its uniform).
template <typename E>
__device__ __forceinline__ void flag_draw(const Params& p, int64_t b, const DrawJob& jb) {
  if (!p.rf_ctl) return;
  rf::Rec r{};
  r.b = (int32_t)b;
  r.j = jb.j;
  r.resid = jb.j < p.K ? 1 : 0;
  r.mp = rs_load(p, b * p.RS + jb.j).M;
  r.mq = jb.j < p.K ? rs_load(p, b * p.RS + p.K + 1 + jb.j).M : 0.f;
  r.taup = jb.tp;
  r.tauq = jb.j < p.K ? jb.tq : -INFINITY;
  r.u = jb.uK;
  rf::flag(p.rf_ctl, p.rf_recs, p.B, r);
}

template <typename E, bool kTopp>
__device__ int64_t draw_whole(const Params& p, Shared& sh, int64_t b, const DrawJob& jb, int tid, char* ring,
                              size_t ring_bytes) {
  int64_t t = -1;
  int settled = 1;
  if (jb.j < p.K) {
    t = cdf_draw<E>(residual_weights<E, kTopp>(p, b, jb), p.V, jb.uK, sh, tid, ring, ring_bytes, p.ctl + 3);
    settled = t >= 0 && sh.bi[7];  // a residual of zero mass in fp32 may not be zero exactly
  }
  if (t < 0) {
    t = cdf_draw<E>(target_weights<E, kTopp>(p, b, jb), p.V, jb.uK, sh, tid, ring, ring_bytes, p.ctl + 3);
    if (jb.j == p.K) settled = sh.bi[7];
  }
  if (!settled && tid == 0) flag_draw<E>(p, b, jb);
  return t;
}

constexpr uint32_t kTailClaimed = 0x80000000u;
constexpr uint32_t kTailChunk = 0x40000000u;

template <typename E>
__device__ __forceinline__ bool seq_decide(const Params& p, Shared& sh, int64_t b, int tid, DrawJob& jb) {
  const int K = p.K;
  const float c = p.c;
  if (tid == 0) sh.bi[1] = K;
  cbar();
  int bad = 0;
  for (int i = tid; i < K; i += kConsumerThreads) {
    const int32_t x = p.tokens[b * K + i];
    const float u = p.uniforms[b * (K + 1) + i];
    const RowStat rp = rs_load(p, b * p.RS + i);
    const RowStat rq = rs_load(p, b * p.RS + K + 1 + i);
    if (x < 0 || (int64_t)x >= p.V || !(u >= 0.f && u < 1.f) || rp.M != rp.M || rq.M != rq.M) {
      bad = 1;
      continue;
    }
    const float lp = ET<E>::load(row_ptr<E, kSample>(p, b, i), x);
    const float lq = ET<E>::load(row_ptr<E, kSample>(p, b, K + 1 + i), x);
    float alpha;
    const bool in_p = !p.topp || ET<E>::key(lp) >= rp.tau;
    const bool in_q = !p.topp || ET<E>::key(lq) >= rq.tau;
    if (!in_p || lp == -INFINITY) {
      alpha = 0.f;
    } else if (!in_q || lq == -INFINITY) {
      alpha = 1.f;
    } else {
      const float ap = fmaf(lp, c, -mref(rp.M, c));
      const float aq = fmaf(lq, c, -mref(rq.M, c));
      alpha = fminf(1.f, ex2(ap - aq) * (rq.cum / rp.cum));
    }
    if (!(u < alpha)) atomicMin(&sh.bi[1], i);
  }
  {
    const RowStat rk = rs_load(p, b * p.RS + K);
    const float uK = p.uniforms[b * (K + 1) + K];
    if (tid == 0 && (rk.M != rk.M || !(uK >= 0.f && uK < 1.f))) bad = 1;
  }
  bad = cbar_or(bad);
  const int j = sh.bi[1];
  cbar();
  if (bad) return false;
  const RowStat rp = rs_load(p, b * p.RS + j);
  const RowStat rq = rs_load(p, b * p.RS + K + 1 + (j < K ? j : 0));
  jb.uK = p.uniforms[b * (K + 1) + K];
  jb.j = j;
  jb.nMcp = -mref(rp.M, c);
  jb.ip = 1.f / rp.cum;
  jb.tp = p.topp ? key_floor<E>(rp.tau) : -INFINITY;
  jb.nMcq = -mref(rq.M, c);
  jb.iq = 1.f / rq.cum;
  jb.tq = p.topp ? key_floor<E>(rq.tau) : -INFINITY;
  return true;
}

// Sequence b's outputs other than the drawn token (all -1 for bad input).
__device__ __forceinline__ void seq_write_prefix(const Params& p, int64_t b, bool ok, int j, int tid) {
  const int K = p.K;
  int32_t* out = p.out_tokens + b * (K + 1);
  if (!ok) {
    for (int i = tid; i <= K; i += kConsumerThreads) out[i] = -1;
    if (tid == 0) {
      p.out_accept_len[b] = -1;
      atomicOr(p.ctl + 3, kStatusInput);
    }
    return;
  }
  for (int i = tid; i <= K; i += kConsumerThreads)
    if (i != j) out[i] = i < j ? p.tokens[b * K + i] : -1;
  if (tid == 0) p.out_accept_len[b] = j;
}

// Sequence b's tail when its draw is not split (p.DC == 0): the accept scan
// and the whole draw in this CTA.
template <typename E>
__device__ void seq_sample(const Params& p, Shared& sh, int64_t b, int tid) {
  DrawJob jb;
  const bool ok = seq_decide<E>(p, sh, b, tid, jb);
  seq_write_prefix(p, b, ok, jb.j, tid);
  if (!ok) return;
  // The tile ring is idle while sequence tails run (they run only after the
  // CTA's streaming is over), so the draw stages its rows there.
  char* ring = reinterpret_cast<char*>(&sh) - (size_t)p.stages * kTileBytes;
  const size_t ring_bytes = (size_t)p.stages * kTileBytes;
  const int64_t t = p.topp ? draw_whole<E, true>(p, sh, b, jb, tid, ring, ring_bytes)
                           : draw_whole<E, false>(p, sh, b, jb, tid, ring, ring_bytes);
  if (tid == 0) p.out_tokens[b * (p.K + 1) + jb.j] = (int32_t)t;
}

template <typename E>
__device__ void seq_argmax_limit(const Params& p, Shared& sh, int64_t b, int tid) {
  const int K = p.K;
  if (tid == 0) sh.bi[1] = K;
  cbar();
  int bad = 0;
  for (int i = tid; i <= K; i += kConsumerThreads) {
    const RowStat r = rs_load(p, b * p.RS + i);
    if (r.M != r.M) bad = 1;
    if (i < K) {
      const int32_t x = p.tokens[b * K + i];
      if (x < 0 || (int64_t)x >= p.V) bad = 1;
      else if ((uint32_t)x != r.tau) atomicMin(&sh.bi[1], i);
    }
  }
  bad = cbar_or(bad);
  const int j = sh.bi[1];
  int32_t* out = p.out_tokens + b * (K + 1);
  if (bad) {
    for (int i = tid; i <= K; i += kConsumerThreads) out[i] = -1;
    if (tid == 0) {
      p.out_accept_len[b] = -1;
      atomicOr(p.ctl + 3, kStatusInput);
    }
    return;
  }
  const RowStat rj = rs_load(p, b * p.RS + j);
  for (int i = tid; i <= K; i += kConsumerThreads)
    out[i] = i < j ? p.tokens[b * K + i] : (i == j ? (int32_t)rj.tau : -1);
  if (tid == 0) p.out_accept_len[b] = j;
}

__device__ void seq_greedy(const Params& p, Shared& sh, int64_t b, int tid) {
  const int G = p.G, N = p.N;
  if (tid == 0) sh.bi[1] = -1;
  cbar();
  int bad = 0;
  for (int r = tid; r < G * N; r += kConsumerThreads) {
    const RowStat rs = rs_load(p, b * p.RS + r);
    if (rs.M != rs.M) bad = 1;
  }
  for (int k = tid; k < G * (N - 1); k += kConsumerThreads) {
    const int32_t x = p.tokens[b * G * (N - 1) + k];
    if (x < 0 || (int64_t)x >= p.V) bad = 1;
  }
  bad = cbar_or(bad);
  int32_t* out = p.out_tokens + b * N;
  if (bad) {
    for (int n = tid; n < N; n += kConsumerThreads) out[n] = -1;
    if (tid == 0) {
      p.out_accept_len[b] = -1;
      if (p.out_best) p.out_best[b] = -1;
      atomicOr(p.ctl + 3, kStatusInput);
    }
    return;
  }
  for (int g = tid; g < G; g += kConsumerThreads) {
    const int32_t* cg = p.tokens + (b * G + g) * (N - 1);
    const float4* rg = p.rowstat + b * p.RS + (int64_t)g * N;
    int L = 0;
    while (L < N - 1 && (uint32_t)cg[L] == __float_as_uint(__ldcg(rg + L).w)) ++L;
    atomicMax(&sh.bi[1], L * 65536 + (65535 - g));
  }
  cbar();
  const int key = sh.bi[1];
  const int L = key >> 16, g = 65535 - (key & 0xFFFF);
  const int32_t* cg = p.tokens + (b * G + g) * (N - 1);
  const float4* rg = p.rowstat + b * p.RS + (int64_t)g * N;
  for (int n = tid; n < N; n += kConsumerThreads)
    out[n] = n < L ? cg[n] : (n == L ? (int32_t)__float_as_uint(__ldcg(rg + L).w) : -1);
  if (tid == 0) {
    p.out_accept_len[b] = L;
    if (p.out_best) p.out_best[b] = g;
  }
}

// ------------------------------------------------------------- row tails -----

template <typename E, int MODE>
__device__ __forceinline__ void seq_tail(const Params& p, Shared& sh, int64_t b, int tid) {
  __threadfence();
  if (MODE == kSample) seq_sample<E>(p, sh, b, tid);
  else if (MODE == kArgmaxLimit) seq_argmax_limit<E>(p, sh, b, tid);
  else seq_greedy(p, sh, b, tid);
  cbar();
}

// A finished sampling row: its record for the sequence tail and, if asked,
// the caller-visible {m, lse, P_S, tau}.
template <typename E>
__device__ void store_sample_row(const Params& p, int64_t row, float M, float s, float cum, uint32_t tau) {
  const bool valid = (M > -INFINITY) && (M < INFINITY);  // NaN fails both
  RowStat rs;
  rs.M = valid ? M : __int_as_float(0x7fc00000);
  rs.s = s;
  rs.cum = cum;
  rs.tau = tau;
  rs_store(p, row, rs);
  if (p.out_row_stats) {
    float4 o;
    o.x = valid ? __fdiv_rn(M, p.T) : __int_as_float(0x7fc00000);
    o.y = valid ? (mref(M, p.c) + lg2(s)) * 0.69314718055994531f : __int_as_float(0x7fc00000);
    o.z = valid ? cum / s : __int_as_float(0x7fc00000);
    o.w = (valid && p.topp) ? ET<E>::val(tau) : -INFINITY;
    reinterpret_cast<float4*>(p.out_row_stats)[row] = o;
  }
}

// Publisher side: hand a collective task to the consumers.
__device__ void enqueue_task(const Params& p, Shared& sh, int64_t task, float m, float s) {
  const int t = sh.tq_tail;
  if (t - *reinterpret_cast<volatile int*>(&sh.tq_head) >= kTaskSlots) {  // full: wait for the consumers
    const uint64_t t0 = globaltimer_ns();
    while (t - *reinterpret_cast<volatile int*>(&sh.tq_head) >= kTaskSlots) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicOr(p.ctl + 3, kStatusTimeout);
        return;
      }
    }
  }
  sh.tq[t % kTaskSlots] = task;
  sh.tq_m[t % kTaskSlots] = m;
  sh.tq_s[t % kTaskSlots] = s;
  __threadfence_block();
  *reinterpret_cast<volatile int*>(&sh.tq_tail) = t + 1;
}

// Sequence tails go to a queue in global memory: ctl[4] counts the entries
// written, ctl[5] the entries taken, tq_global[k] holds b+1 (0 = not yet
// written). CTAs take entries only once their own streaming work is done, so
// a tail never holds up tiles that other sequences are waiting for.
// A sequence whose draw is split over p.DC CTAs queues p.DC chunk entries
// instead (kTailChunk | b*DC + c + 1), each running the accept scan and one
// range of the draw's cells.
__device__ __forceinline__ void tail_enqueue(const Params& p, int64_t b) {
  if (p.DC > 0) {  // one fence for all the entries, then plain stores
    const uint32_t k = atomicAdd(p.ctl + 4, (uint32_t)p.DC);
    fence_acq_rel_gpu();
    for (int c = 0; c < p.DC; ++c) st_relaxed_gpu(p.tail_q + k + c, kTailChunk | (uint32_t)(b * p.DC + c + 1));
    return;
  }
  const uint32_t k = atomicAdd(p.ctl + 4, 1u);
  st_release_gpu(p.tail_q + k, (uint32_t)(b + 1));
}

// A tail that this CTA runs itself (its streaming is over, so running it here
// holds up nothing): the queue entry is only marked as claimed, which keeps
// the count of entries equal to the number of sequences.
__device__ __forceinline__ void tail_claim(const Params& p, int64_t b) {
  const uint32_t k = atomicAdd(p.ctl + 4, 1u);
  st_release_gpu(p.tail_q + k, kTailClaimed | (uint32_t)(b + 1));
}

// One more row of sequence b is final. Returns true if it was the last one.
__device__ __forceinline__ bool seq_row_final(const Params& p, int64_t b) {
  const uint32_t old = atom_add_acq_rel(p.seq_cnt + b, 1u);
  if (old == (uint32_t)p.RS - 1u) {
    p.seq_cnt[b] = 0u;
    return true;
  }
  return false;
}

// Publisher side: the last row of a sequence queues its tail, globally while
// this CTA still streams, locally once it does not.
__device__ __forceinline__ void seq_arrive(const Params& p, Shared& sh, int64_t b, bool local) {
  if (!seq_row_final(p, b)) return;
  if (local && p.DC == 0) {
    enqueue_task(p, sh, -(b + 1), 0.f, 0.f);
    tail_claim(p, b);
  } else {
    tail_enqueue(p, b);
  }
}

// Publisher side: the row's result is complete (m, s for sampling; best
// value and index for argmax). Finish the row here unless it needs the
// collective top-p pass.
template <typename E, int MODE>
__device__ void publisher_row_done(const Params& p, Shared& sh, int64_t row, float2 r, bool local) {
  if (MODE == kSample) {
    const float m = r.x, s = r.y;
    const bool valid = (m > -INFINITY) && (m < INFINITY);
    if (valid && p.topp) {
      enqueue_task(p, sh, row, m, s);
      return;
    }
    store_sample_row<E>(p, row, m, s, s, 0u);
  } else {
    const int64_t i = (int64_t)__float_as_int(r.y);
    RowStat rs;
    rs.M = r.x;  // NaN marks a row with a NaN logit
    rs.s = 0.f;
    rs.cum = 0.f;
    rs.tau = (uint32_t)(i < 0 ? 0 : i);  // all -inf: every element ties, index 0 wins
    rs_store(p, row, rs);
  }
  seq_arrive(p, sh, row / p.RS, local);
}

// Publisher side: every chunk of `row` is published; combine the partials.
template <typename E, int MODE>
__device__ void publisher_finish_row(const Params& p, Shared& sh, int64_t row, bool local) {
  p.row_cnt[row] = 0u;
  const float2* part = p.part + row * p.NC;
  if (MODE == kSample) {
    float m = -INFINITY, s = 0.f;
    for (int64_t k = 0; k < p.NC; k += 4) {
      float2 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = (k + j < p.NC) ? __ldcg(part + k + j) : make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int j = 0; j < 4; ++j) ms_combine(m, s, v[j].x, v[j].y, p.c);
    }
    publisher_row_done<E, MODE>(p, sh, row, make_float2(m, s), local);
  } else {
    float v = -INFINITY;
    int64_t i = -1;
    bool nan = false;
    for (int64_t k = 0; k < p.NC; k += 4) {
      float2 pv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        pv[j] = (k + j < p.NC) ? __ldcg(part + k + j) : make_float2(-INFINITY, __int_as_float(-1));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t pi = (int64_t)__float_as_int(pv[j].y);
        if (pv[j].x != pv[j].x) nan = true;
        else if (am_better(pv[j].x, pi, v, i)) {
          v = pv[j].x;
          i = pi;
        }
      }
    }
    publisher_row_done<E, MODE>(p, sh, row,
                                make_float2(nan ? __int_as_float(0x7fc00000) : v, __int_as_float((int)i)), local);
  }
}

// Consumer side: one queued task, run by all 256 consumer threads: a top-p
// cut (row >= 0) or, once streaming is over, a sequence tail (-(b+1)).
// `local` says the CTA's streaming is over.
template <typename E, int MODE>
__device__ void run_task(const Params& p, Shared& sh, int64_t task, float m, float s, int tid, bool local) {
  if (task < 0) {
    seq_tail<E, MODE>(p, sh, -task - 1, tid);
    return;
  }
  if (MODE == kSample) {
    const int64_t b = task / p.RS;
    const int r = (int)(task % p.RS);
    __threadfence();
    uint32_t tau = 0u;
    float cum = s;
    topp_cut<E>(p, sh, row_ptr<E, MODE>(p, b, r), m, s, tid, tau, cum);
    if (tid == 0) {
      store_sample_row<E>(p, task, m, s, cum, tau);
      int run_here = 0;
      if (seq_row_final(p, b)) {
        if (local && p.DC == 0) {
          tail_claim(p, b);
          run_here = 1;
        } else {
          tail_enqueue(p, b);
        }
      }
      sh.flag = run_here;
    }
    cbar();
    const int run_here = sh.flag;
    cbar();
    if (run_here) seq_tail<E, MODE>(p, sh, b, tid);
  }
}

// One chunk of sequence b's split draw (sampling mode, p.DC > 0). Every chunk
// CTA runs the short accept scan itself, so no decision is handed over;
// chunk 0 writes the outputs other than the drawn token. Each sums the cells
// [c*CPC, (c+1)*CPC) of the draw into p.dcells; the CTA that completes the last
// chunk scans all the cells and writes the drawn token.
template <typename E, bool kTopp>
__device__ void draw_chunk(const Params& p, Shared& sh, int64_t b, int c, int tid) {
  DrawJob jb;
  const bool ok = seq_decide<E>(p, sh, b, tid, jb);
  if (c == 0) seq_write_prefix(p, b, ok, jb.j, tid);
  if (!ok) jb.j = -1;
  const int64_t CE = cell_elems(p.V);
  const int ncells = (int)((p.V + CE - 1) / CE);
  float* cells = p.dcells + b * ncells;
  char* ring = reinterpret_cast<char*>(&sh) - (size_t)p.stages * kTileBytes;
  const size_t ring_bytes = (size_t)p.stages * kTileBytes;
  const int cbeg = min(ncells, c * p.CPC), cend = min(ncells, (c + 1) * p.CPC);
  if (ok && cbeg < cend) {
    if (jb.j < p.K) {
      const Weights<E, true, kTopp> wf = residual_weights<E, kTopp>(p, b, jb);
      if (!cells_staged<E>(wf, p.V, CE, cbeg, cend, cells, ring, ring_bytes, sh, tid, p.ctl + 3))
        cells_global<E>(wf, CE, cbeg, cend, cells, tid);
    } else {
      const Weights<E, false, kTopp> wf = target_weights<E, kTopp>(p, b, jb);
      if (!cells_staged<E>(wf, p.V, CE, cbeg, cend, cells, ring, ring_bytes, sh, tid, p.ctl + 3))
        cells_global<E>(wf, CE, cbeg, cend, cells, tid);
    }
  }
  __threadfence();
  cbar();
  if (tid == 0) {
    const uint32_t old = atom_add_acq_rel(p.dcnt + b, 1u);
    const int last = old == (uint32_t)p.DC - 1u;
    if (last) p.dcnt[b] = 0u;
    sh.flag = last;
  }
  cbar();
  const int last = sh.flag;
  cbar();
  if (!last || !ok) return;
  for (int i = tid; i < ncells; i += kConsumerThreads) sh.cells[i] = __ldcg(cells + i);
  cbar();
  int64_t t = -1;
  int settled = 1;
  if (jb.j < p.K) {
    t = cdf_cross<E>(residual_weights<E, kTopp>(p, b, jb), p.V, jb.uK, sh, tid);
    settled = t >= 0 && sh.bi[7];
  }
  if (t < 0) {  // the bonus draw, or a residual that is all zero: p'_j
    t = jb.j < p.K
            ? cdf_draw<E>(target_weights<E, kTopp>(p, b, jb), p.V, jb.uK, sh, tid, ring, ring_bytes, p.ctl + 3)
            : cdf_cross<E>(target_weights<E, kTopp>(p, b, jb), p.V, jb.uK, sh, tid);
    if (jb.j == p.K) settled = sh.bi[7];
  }
  if (tid == 0) {
    p.out_tokens[b * (p.K + 1) + jb.j] = (int32_t)t;
    if (!settled) flag_draw<E>(p, b, jb);
  }
}

// Consumer side, after the CTA's streaming is done: take tickets for queued
// sequence tails and draw chunks until every entry of the call has been
// taken. Ticket k is the k-th entry queued; it may not be written yet, but
// whoever will write it holds what it waits for and needs nothing from this
// CTA, so the wait ends.
template <typename E, int MODE>
__device__ void drain_tails(const Params& p, Shared& sh, int tid) {
  const int64_t entries = p.B * (MODE == kSample && p.DC > 0 ? (int64_t)p.DC : 1);
  for (;;) {
    if (tid == 0) {
      const uint32_t k = atomicAdd(p.ctl + 5, 1u);
      int64_t e = -1;  // -1: none left; -2: skip; >= 0: b, or kTailChunk | (b*DC + c)
      if ((int64_t)k < entries) {
        uint32_t v = ld_acquire_gpu(p.tail_q + k);
        if (v == 0u) {
          const uint64_t t0 = globaltimer_ns();
          while (v == 0u && globaltimer_ns() - t0 < kWaitLimitNs) v = ld_acquire_gpu(p.tail_q + k);
        }
        if (v == 0u) atomicOr(p.ctl + 3, kStatusTimeout);
        else if (v & kTailClaimed) e = -2;  // run by the CTA that completed it
        else if (v & kTailChunk) e = (int64_t)kTailChunk | (int64_t)((v & ~kTailChunk) - 1u);
        else e = (int64_t)v - 1;
        p.tail_q[k] = 0u;
      }
      sh.bl[1] = e;
    }
    cbar();
    const int64_t e = sh.bl[1];
    cbar();
    if (e == -2) continue;
    if (e < 0) return;
    if (MODE == kSample && (e & kTailChunk)) {
      const int64_t bc = e & ~(int64_t)kTailChunk;
      if (p.topp)
        draw_chunk<E, true>(p, sh, bc / p.DC, (int)(bc % p.DC), tid);
      else
        draw_chunk<E, false>(p, sh, bc / p.DC, (int)(bc % p.DC), tid);
    } else {
      seq_tail<E, MODE>(p, sh, e, tid);
    }
  }
}

template <typename E, int MODE>
__device__ __forceinline__ int drain_tasks(const Params& p, Shared& sh, int head, int snap, int tid, bool local) {
  while (head < snap) {
    const int i = head % kTaskSlots;
    run_task<E, MODE>(p, sh, sh.tq[i], sh.tq_m[i], sh.tq_s[i], tid, local);
    ++head;
  }
  if (tid == 0) *reinterpret_cast<volatile int*>(&sh.tq_head) = head;
  return head;
}

// --------------------------------------------------------------- kernel -------

// The producer: one thread takes chunks from the call's work counter (one
// fetch ahead) and streams their tiles into the ring, one stage per tile,
// each stage one bulk copy completing on the stage's "full" barrier.
template <typename E, int MODE>
__device__ void producer_loop(const Params& p, char* ring, Shared& sh) {
  unsigned long long* next = reinterpret_cast<unsigned long long*>(p.ctl);
  int last_parity[kMaxStages];
  for (int i = 0; i < kMaxStages; ++i) last_parity[i] = -1;
  bool aborted = false;
  int slot = 0;
  uint32_t ph = 0u;
  bool wrapped = false;  // every stage has been used once
  // Two work indices are always in flight ahead of the chunk being streamed,
  // so the round trip of the counter never stalls the ring.
  int64_t w = (int64_t)atomicAdd(next, 1ull);
  int64_t w1 = w < p.W ? (int64_t)atomicAdd(next, 1ull) : w;
  while (!aborted) {
    const int64_t w2 = w1 < p.W ? (int64_t)atomicAdd(next, 1ull) : w1;
    ChunkId ch;
    if (w < p.W) ch = decode_chunk(p, w);
    const int n = w < p.W ? ch.n : 1;  // the end of work takes one stage too
    for (int j = 0; j < n; ++j) {
      if (wrapped && !mbar_wait(&sh.empty[slot], ph ^ 1u)) {
        aborted = true;
        break;
      }
      TileDesc& t = sh.td[slot];
      if (w >= p.W) {
        t.w = -1;
        mbar_arrive(&sh.full[slot]);
        break;
      }
      decode_tile<E, MODE>(p, ch, ch.k0 + j, t);
      t.w = w;
      t.last = (j == n - 1);
      if (t.ibytes) {
        const char* src = t.row + t.ie0 * ET<E>::kSize;
        mbar_arrive_expect_tx(&sh.full[slot], t.ibytes);
        bulk_g2s(ring + (size_t)slot * kTileBytes, src, t.ibytes, &sh.full[slot]);
        last_parity[slot] = (int)ph;
      } else {
        mbar_arrive(&sh.full[slot]);
      }
      if (++slot == p.stages) {
        slot = 0;
        ph ^= 1u;
        wrapped = true;
      }
    }
    if (w >= p.W) break;
    w = w1;
    w1 = w2;
  }
  if (aborted) {  // a wait ran out: let copies still in flight land before the CTA exits
    atomicOr(p.ctl + 3, kStatusTimeout);
    for (int i = 0; i < p.stages; ++i)
      if (last_parity[i] >= 0) (void)mbar_wait(&sh.full[i], (uint32_t)last_parity[i]);
  }
  // The last producer to finish re-arms the work counter for the next call.
  __threadfence();
  const uint32_t prev = atomicAdd(p.ctl + 2, 1u);
  if (prev == gridDim.x - 1) {
    *next = 0ull;
    p.ctl[2] = 0u;
    __threadfence();
  }
}

// The publisher: combines the consumer warps' chunk partials, stores the
// chunk's partial and counts it against its row (release/acquire atomic,
// whose result is looked at one chunk later so that its round trip overlaps
// the next chunk). The last chunk of a row finishes the row.
template <typename E, int MODE>
__device__ void publisher_loop(const Params& p, Shared& sh) {
  // The row a chunk completes is finished one chunk later, so that the
  // counter's round trip overlaps the next chunk and the CTA's last row is
  // known to be its last (its sequence tail can then run here).
  int64_t pend_row = -1;
  uint32_t pend_old = 0u;
  float2 pend_res = make_float2(0.f, 0.f);
  auto finish_pending = [&](bool local) {
    if (pend_row < 0 || pend_old != (uint32_t)(p.NC - 1)) return;
    if (p.NC == 1) publisher_row_done<E, MODE>(p, sh, pend_row, pend_res, local);
    else publisher_finish_row<E, MODE>(p, sh, pend_row, local);
  };
  for (int64_t c = 0;; ++c) {
    const int ps = (int)(c % kPartSlots);
    const uint32_t pph = (uint32_t)((c / kPartSlots) & 1);
    if (!mbar_wait(&sh.pfull[ps], pph)) {
      atomicOr(p.ctl + 3, kStatusTimeout);
      break;
    }
    const int64_t w = sh.pw[ps];
    if (w < 0) break;
    float2 res;
    if (MODE == kSample) {
      float M = sh.red_m[ps][0], S = sh.red_s[ps][0];
      for (int k = 1; k < kConsumerWarps; ++k) ms_combine(M, S, sh.red_m[ps][k], sh.red_s[ps][k], p.c);
      res = make_float2(M, S);
    } else {
      float V_ = sh.red_m[ps][0];
      int64_t I = sh.red_i[ps][0];
      bool N_ = V_ != V_;
      for (int k = 1; k < kConsumerWarps; ++k) {
        const float v2 = sh.red_m[ps][k];
        if (v2 != v2) N_ = true;
        else if (am_better(v2, sh.red_i[ps][k], V_, I)) {
          V_ = v2;
          I = sh.red_i[ps][k];
        }
      }
      if (N_) V_ = __int_as_float(0x7fc00000);
      res = make_float2(V_, __int_as_float((int)I));
    }
    const int64_t row = sh.prow[ps];
    mbar_arrive(&sh.pempty[ps]);
    uint32_t old = 0u;  // a row that is a single chunk is complete with it
    if (p.NC > 1) {
      p.part[w] = res;
      old = atom_add_acq_rel(p.row_cnt + row, 1u);
    }
    finish_pending(false);
    pend_row = row;
    pend_old = old;
    pend_res = res;
  }
  // The consumers are done streaming: a sequence completed from here on runs here.
  finish_pending(true);
  mbar_arrive(&sh.pdone);
}

// The consumers: per-thread accumulation over every tile of a chunk; at the
// end of a chunk, per-warp partials go to the publisher and one barrier (which
// carries the abort vote of the bounded waits) lets all consumers see the
// same task-queue snapshot.
template <typename E, int MODE>
__device__ __forceinline__ void consumer_loop(const Params& p, const char* ring, Shared& sh, int tid) {
  constexpr int PV = ET<E>::kPerVec;
  const int warp = tid >> 5, lane = tid & 31;
  float m = -INFINITY;                      // sampling: online (max, sum)
  float sa[4] = {0.f, 0.f, 0.f, 0.f};
  float av = -INFINITY;                     // argmax: value, index, NaN seen
  int64_t ai = -1;
  bool an = false;
  int timed_out = 0;
  int64_t chunks = 0;
  int head = 0;
  int slot = 0;
  uint32_t ph = 0u;
  for (;;) {
    const int cur = slot;
    if (!mbar_wait(&sh.full[cur], ph)) {
      timed_out = 1;
      break;
    }
    if (++slot == p.stages) {
      slot = 0;
      ph ^= 1u;
    }
    const TileDesc t = sh.td[cur];  // a copy: the stage (and its descriptor) is released below
    const int64_t w = t.w;
    if (w < 0) break;  // no more work
    const bool last = t.last != 0;
    const uint4* sv = reinterpret_cast<const uint4*>(ring + (size_t)cur * kTileBytes);
    const int nvec = (int)(t.ibytes >> 4);
    if (MODE == kSample) {
      ms_tile<E>(sv, nvec, tid, p.c, m, sa);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[cur]);
      if (t.nh | t.nt) {
        // head and tail elements (rows not 16-byte aligned) join one
        // accumulator, so that a new maximum among them rescales everything
        sa[0] += (sa[1] + sa[2]) + sa[3];
        sa[1] = sa[2] = sa[3] = 0.f;
        if (tid < t.nh) ms_scalar(m, sa[0], ET<E>::load(t.row, t.e0 + tid), p.c);
        if (tid >= 32 && tid < 32 + t.nt) ms_scalar(m, sa[0], ET<E>::load(t.row, t.e1 - t.nt + (tid - 32)), p.c);
      }
    } else {
      for (int v0 = tid; v0 < nvec; v0 += kVecBatch * kConsumerThreads) {
        uint4 q[kVecBatch];
#pragma unroll
        for (int k = 0; k < kVecBatch; ++k) {
          const int v = v0 + k * kConsumerThreads;
          q[k] = v < nvec ? sv[v] : neg_inf_vec(E());
        }
        float vmax = vec_max(q[0], E());
#pragma unroll
        for (int k = 1; k < kVecBatch; ++k) vmax = fmax_nan(vmax, vec_max(q[k], E()));
        if (vmax != vmax) {
          an = true;
        } else if (vmax > av || ai < 0) {  // a new best somewhere in the batch: find its first occurrence
#pragma unroll
          for (int k = 0; k < kVecBatch; ++k) {
            const int v = v0 + k * kConsumerThreads;
            if (v < nvec) am_vec(av, ai, an, q[k], t.ie0 + (int64_t)v * PV, E());
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[cur]);
      if (tid < t.nh) am_scalar(av, ai, an, ET<E>::load(t.row, t.e0 + tid), t.e0 + tid);
      if (tid >= 32 && tid < 32 + t.nt) {
        const int64_t e = t.e1 - t.nt + (tid - 32);
        am_scalar(av, ai, an, ET<E>::load(t.row, e), e);
      }
    }
    if (!last) continue;

    // ---- end of a chunk
    const int ps = (int)(chunks % kPartSlots);
    const uint32_t pph = (uint32_t)((chunks / kPartSlots) & 1);
    float rm, rs_;
    int64_t ri = -1;
    if (MODE == kSample) {
      float s = (sa[0] + sa[1]) + (sa[2] + sa[3]);
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
        ms_combine(m, s, m2, s2, p.c);
      }
      rm = m;
      rs_ = s;
      m = -INFINITY;
      sa[0] = sa[1] = sa[2] = sa[3] = 0.f;
    } else {
      for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, av, o);
        const long long i2 = __shfl_xor_sync(0xffffffffu, (long long)ai, o);
        if (am_better(v2, i2, av, ai)) {
          av = v2;
          ai = i2;
        }
      }
      an = __any_sync(0xffffffffu, an);
      rm = an ? __int_as_float(0x7fc00000) : av;
      rs_ = 0.f;
      ri = ai;
      av = -INFINITY;
      ai = -1;
      an = false;
    }
    if (chunks >= kPartSlots && !mbar_wait(&sh.pempty[ps], pph ^ 1u)) timed_out = 1;
    if (lane == 0) {
      sh.red_m[ps][warp] = rm;
      sh.red_s[ps][warp] = rs_;
      sh.red_i[ps][warp] = ri;
      if (warp == 0) {
        sh.pw[ps] = w;
        sh.prow[ps] = t.rowid;
      }
      mbar_arrive(&sh.pfull[ps]);
    }
    const int par = (int)(chunks & 1);
    ++chunks;
    if (tid == 0) {
      sh.snap[par] = *reinterpret_cast<volatile int*>(&sh.tq_tail);
      __threadfence_block();
    }
    if (cbar_or(timed_out)) {
      if (tid == 0) atomicOr(p.ctl + 3, kStatusTimeout);
      return;
    }
    head = drain_tasks<E, MODE>(p, sh, head, sh.snap[par], tid, false);
  }
  // End of work (or a wait that ran out): tell the publisher, wait for it to
  // finish, and run what it queued.
  if (!timed_out) {
    const int ps = (int)(chunks % kPartSlots);
    const uint32_t pph = (uint32_t)((chunks / kPartSlots) & 1);
    if (chunks >= kPartSlots && !mbar_wait(&sh.pempty[ps], pph ^ 1u)) timed_out = 1;
    if (lane == 0) {
      if (warp == 0) sh.pw[ps] = -1;
      mbar_arrive(&sh.pfull[ps]);
    }
  }
  if (cbar_or(timed_out)) {
    if (tid == 0) atomicOr(p.ctl + 3, kStatusTimeout);
    return;
  }
  const int done = mbar_wait(&sh.pdone, 0u) ? 1 : 0;
  if (tid == 0) {
    sh.snap[0] = *reinterpret_cast<volatile int*>(&sh.tq_tail);
    __threadfence_block();
  }
  if (cbar_or(!done)) {
    if (tid == 0) atomicOr(p.ctl + 3, kStatusTimeout);
    return;
  }
  drain_tasks<E, MODE>(p, sh, head, sh.snap[0], tid, true);
  drain_tails<E, MODE>(p, sh, tid);
  // The last CTA out re-arms the tail queue for the next call.
  if (tid == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(p.ctl + 6, 1u);
    if (prev == gridDim.x - 1) {
      p.ctl[4] = 0u;
      p.ctl[5] = 0u;
      p.ctl[6] = 0u;
      __threadfence();
    }
  }
}

template <typename E, int MODE>
__global__ void __launch_bounds__(kAllThreads, 2) verify_kernel(const Params p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  char* ring = reinterpret_cast<char*>(smem);
  Shared& sh = *reinterpret_cast<Shared*>(smem + (size_t)p.stages * kTileBytes);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&sh.full[i], 1u);
      mbar_init(&sh.empty[i], (uint32_t)kConsumerWarps);
    }
    for (int i = 0; i < kPartSlots; ++i) {
      mbar_init(&sh.pfull[i], (uint32_t)kConsumerWarps);
      mbar_init(&sh.pempty[i], 1u);
    }
    mbar_init(&sh.pdone, 1u);
    mbar_init(&sh.dbar[0], 1u);
    mbar_init(&sh.dbar[1], 1u);
    sh.dcount[0] = sh.dcount[1] = 0u;
    sh.tq_tail = 0;
    sh.tq_head = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_sync();
  const int warp = tid >> 5;
  if (warp == kProducerWarp) {
    if ((tid & 31) == 0) producer_loop<E, MODE>(p, ring, sh);
    return;
  }
  if (warp == kPublisherWarp) {
    if ((tid & 31) == 0) publisher_loop<E, MODE>(p, sh);
    return;
  }
  consumer_loop<E, MODE>(p, ring, sh, tid);
}

// ------------------------------------------- whole sequences in one CTA -----
//
// For short rows (a whole sequence of 2K+1 rows fits in 48 KB), one work item
// is one sequence: the producer moves its target block and its draft block
// into a shared-memory stage with two bulk copies; the consumers compute every
// row's (max, sum), the accept scan and the draw from shared memory. No row or
// sequence crosses a CTA, so there are no partials, counters or queues.

constexpr int kSeqStageBytes = 49152;
constexpr int kSeqStages = 2;
constexpr int kSeqMaxRows = 64;
constexpr int kSeqThreads = kConsumerThreads + 32;
constexpr int kSeqMaxCells = kSeqStageBytes / 2 / 256;

struct alignas(16) SeqShared {
  uint64_t full[kSeqStages];
  uint64_t empty[kSeqStages];
  int64_t seq[kSeqStages];  // sequence in the stage (-1: no more work)
  float rm[kSeqMaxRows];    // per row: max and sum relative to mref(max)
  float rsum[kSeqMaxRows];
  float cells[kSeqMaxCells];
  float wl[256];            // the crossing cell's weights
  float bf[4];
  int bi[4];
  int64_t bl[2];
};

size_t seq_shared_bytes() { return (size_t)kSeqStages * kSeqStageBytes + sizeof(SeqShared); }

template <typename E>
__device__ __forceinline__ float smem_elem(const char* row, int64_t e) {
  if (ET<E>::kSize == 2)
    return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(row)[e] << 16);
  return reinterpret_cast<const float*>(row)[e];
}

template <typename E>
__device__ void seq_producer(const Params& p, char* ring, SeqShared& sh) {
  constexpr int S = ET<E>::kSize;
  unsigned long long* next = reinterpret_cast<unsigned long long*>(p.ctl);
  const uint32_t tbytes = (uint32_t)((p.K + 1) * p.V * S), dbytes = (uint32_t)(p.K * p.V * S);
  int stage = 0;
  uint32_t ph = 0u;
  bool wrapped = false, aborted = false;
  int last_parity[kSeqStages] = {-1, -1};
  int64_t b = (int64_t)atomicAdd(next, 1ull);
  for (;;) {
    const int64_t bn = b < p.B ? (int64_t)atomicAdd(next, 1ull) : b;
    if (wrapped && !mbar_wait(&sh.empty[stage], ph ^ 1u)) {
      aborted = true;
      break;
    }
    if (b >= p.B) {
      sh.seq[stage] = -1;
      mbar_arrive(&sh.full[stage]);
      break;
    }
    sh.seq[stage] = b;
    char* dst = ring + (size_t)stage * kSeqStageBytes;
    mbar_arrive_expect_tx(&sh.full[stage], tbytes + dbytes);
    bulk_g2s(dst, p.a + b * (int64_t)tbytes, tbytes, &sh.full[stage]);
    bulk_g2s(dst + tbytes, p.d + b * (int64_t)dbytes, dbytes, &sh.full[stage]);
    last_parity[stage] = (int)ph;
    if (++stage == kSeqStages) {
      stage = 0;
      ph ^= 1u;
      wrapped = true;
    }
    b = bn;
  }
  if (aborted) {
    atomicOr(p.ctl + 3, kStatusTimeout);
    for (int i = 0; i < kSeqStages; ++i)
      if (last_parity[i] >= 0) (void)mbar_wait(&sh.full[i], (uint32_t)last_parity[i]);
  }
  __threadfence();
  const uint32_t prev = atomicAdd(p.ctl + 2, 1u);
  if (prev == gridDim.x - 1) {
    *next = 0ull;
    p.ctl[2] = 0u;
    __threadfence();
  }
}

// One staged sequence, by the 256 consumer threads.
template <typename E>
__device__ void seq_in_smem(const Params& p, SeqShared& sh, const char* st, int64_t b, int tid) {
  constexpr int S = ET<E>::kSize;
  constexpr int PV = ET<E>::kPerVec;
  const int warp = tid >> 5, lane = tid & 31;
  const int K = p.K, R = p.RS;
  const int64_t V = p.V;
  const float c = p.c;
  const int64_t tb = (K + 1) * V * S;
  auto rowp = [&](int r) { return r <= K ? st + r * V * S : st + tb + (r - K - 1) * V * S; };
  // ---- per-row (max, sum): one warp per row
  const int nvec = (int)(V / PV);
  for (int r = warp; r < R; r += kConsumerWarps) {
    const uint4* rv = reinterpret_cast<const uint4*>(rowp(r));
    float m = -INFINITY, sa[4] = {0.f, 0.f, 0.f, 0.f};
    for (int v0 = lane; v0 < nvec; v0 += 32 * kVecBatch) {
      uint4 q[kVecBatch];
#pragma unroll
      for (int k = 0; k < kVecBatch; ++k) {
        const int v = v0 + 32 * k;
        q[k] = v < nvec ? rv[v] : neg_inf_vec(E());
      }
      float vmax = vec_max(q[0], E());
#pragma unroll
      for (int k = 1; k < kVecBatch; ++k) vmax = fmax_nan(vmax, vec_max(q[k], E()));
      const float nm = fmax_nan(m, vmax);
      if (nm != m) {
        const float f = rescale(m, nm, c);
        sa[0] *= f; sa[1] *= f; sa[2] *= f; sa[3] *= f;
        m = nm;
      }
      if (m == -INFINITY) continue;
      const float nmc = -mref(m, c);
#pragma unroll
      for (int k = 0; k < kVecBatch; ++k) vec_exp_add(q[k], c, nmc, sa, E());
    }
    float sum = (sa[0] + sa[1]) + (sa[2] + sa[3]);
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, sum, o);
      ms_combine(m, sum, m2, s2, c);
    }
    if (lane == 0) {
      sh.rm[r] = m;
      sh.rsum[r] = sum;
    }
  }
  if (tid == 0) sh.bi[1] = K;
  cbar();
  // ---- row stats out, validity, accept scan
  int bad = 0;
  for (int r = tid; r < R; r += kConsumerThreads) {
    const float M = sh.rm[r], s = sh.rsum[r];
    const bool valid = (M > -INFINITY) && (M < INFINITY);
    if (!valid) bad = 1;
    if (p.out_row_stats) {
      float4 o;
      o.x = valid ? __fdiv_rn(M, p.T) : __int_as_float(0x7fc00000);
      o.y = valid ? (mref(M, c) + lg2(s)) * 0.69314718055994531f : __int_as_float(0x7fc00000);
      o.z = valid ? 1.f : __int_as_float(0x7fc00000);
      o.w = -INFINITY;
      reinterpret_cast<float4*>(p.out_row_stats)[b * R + r] = o;
    }
  }
  for (int i = tid; i < K; i += kConsumerThreads) {
    const int32_t x = p.tokens[b * K + i];
    const float u = p.uniforms[b * (K + 1) + i];
    if (x < 0 || (int64_t)x >= V || !(u >= 0.f && u < 1.f)) {
      bad = 1;
      continue;
    }
    const float Mp = sh.rm[i], Mq = sh.rm[K + 1 + i];
    if (!(Mp > -INFINITY && Mp < INFINITY && Mq > -INFINITY && Mq < INFINITY)) continue;  // counted above
    const float lp = smem_elem<E>(rowp(i), x), lq = smem_elem<E>(rowp(K + 1 + i), x);
    float alpha;
    if (lp == -INFINITY) alpha = 0.f;
    else if (lq == -INFINITY) alpha = 1.f;
    else alpha = fminf(1.f, ex2(fmaf(lp, c, -mref(Mp, c)) - fmaf(lq, c, -mref(Mq, c))) * (sh.rsum[K + 1 + i] / sh.rsum[i]));
    if (!(u < alpha)) atomicMin(&sh.bi[1], i);
  }
  const float uK = p.uniforms[b * (K + 1) + K];
  if (tid == 0 && !(uK >= 0.f && uK < 1.f)) bad = 1;
  bad = cbar_or(bad);
  const int j = sh.bi[1];
  int32_t* out = p.out_tokens + b * (K + 1);
  if (bad) {
    for (int i = tid; i <= K; i += kConsumerThreads) out[i] = -1;
    if (tid == 0) {
      p.out_accept_len[b] = -1;
      atomicOr(p.ctl + 3, kStatusInput);
    }
    return;
  }
  // ---- the draw, from shared memory: cells of 256 elements, eight per lane
  const char* rp = rowp(j);
  const char* rq = j < K ? rowp(K + 1 + j) : nullptr;
  const float nMp = -mref(sh.rm[j], c), ip = 1.f / sh.rsum[j];
  const float nMq = rq ? -mref(sh.rm[K + 1 + j], c) : 0.f, iq = rq ? 1.f / sh.rsum[K + 1 + j] : 0.f;
  const int ncells = (int)((V + 255) / 256);
  int64_t t = -1;
  for (int attempt = 0; attempt < 2 && t < 0; ++attempt) {
    const bool resid = (attempt == 0) && rq != nullptr;
    auto w8 = [&](int64_t e, float w[8]) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int64_t ek = e + k;
        if (ek >= V) {
          w[k] = 0.f;
          continue;
        }
        const float ep = ex2(fmaf(smem_elem<E>(rp, ek), c, nMp));
        w[k] = resid ? fmaxf(0.f, fmaf(ep, ip, -ex2(fmaf(smem_elem<E>(rq, ek), c, nMq)) * iq)) : ep;
      }
    };
    for (int cc = warp; cc < ncells; cc += kConsumerWarps) {
      float w[8];
      w8((int64_t)cc * 256 + lane * 8, w);
      const float a = warp_sum(((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7])));
      if (lane == 0) sh.cells[cc] = a;
    }
    cbar();
    if (warp == 0) {
      const int cpl = (ncells + 31) / 32;
      const int c0 = min(ncells, lane * cpl), c1 = min(ncells, c0 + cpl);
      float ls = 0.f;
      for (int cc = c0; cc < c1; ++cc) ls += sh.cells[cc];
      const float incl = warp_incl_scan(ls, lane);
      const float Z = __shfl_sync(0xffffffffu, incl, 31);
      int64_t tt = -1;
      if (Z > 0.f) {
        const float Tg = uK * Z;
        float run = incl - ls;
        int hit = -1;
        for (int cc = c0; cc < c1; ++cc) {
          if (run + sh.cells[cc] > Tg) {
            hit = cc;
            break;
          }
          run += sh.cells[cc];
        }
        const unsigned bal = __ballot_sync(0xffffffffu, hit >= 0);
        int cstar;
        float Tl = 0.f;
        bool lastpos_mode = false;
        if (bal) {
          const int fl = __ffs(bal) - 1;
          cstar = __shfl_sync(0xffffffffu, hit, fl);
          Tl = Tg - __shfl_sync(0xffffffffu, run, fl);
        } else {
          int last = -1;
          for (int cc = c0; cc < c1; ++cc)
            if (sh.cells[cc] > 0.f) last = cc;
          for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
          cstar = last;
          lastpos_mode = true;
        }
        const int64_t base = (int64_t)cstar * 256 + lane * 8;
        float w[8];
        w8(base, w);
        const float l8 = ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
        const float incl2 = warp_incl_scan(l8, lane);
        const float excl2 = incl2 - l8;
        int64_t mine = -1, lastp = -1;
        float acc = excl2;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (w[k] > 0.f) lastp = base + k;
          acc += w[k];
          if (mine < 0 && !lastpos_mode && acc > Tl) mine = base + k;
        }
        const unsigned bal2 = __ballot_sync(0xffffffffu, mine >= 0);
        if (bal2) {
          tt = __shfl_sync(0xffffffffu, (long long)mine, __ffs(bal2) - 1);
        } else {  // rounding or u*Z past the total: the last positive weight
          long long lp = lastp;
          for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
          tt = lp;
        }
      }
      if (lane == 0) sh.bl[0] = tt;
    }
    cbar();
    t = sh.bl[0];
    cbar();
    if (!resid) break;  // the bonus or the fallback to p'_j always has mass
    if (t < 0) {        // a residual that is all zero: draw from p'_j instead
      rq = nullptr;
    }
  }
  for (int i = tid; i <= K; i += kConsumerThreads)
    out[i] = i < j ? p.tokens[b * K + i] : (i == j ? (int32_t)t : -1);
  if (tid == 0) p.out_accept_len[b] = j;
}

template <typename E>
__device__ void seq_consumer(const Params& p, const char* ring, SeqShared& sh, int tid) {
  const int lane = tid & 31;
  int stage = 0;
  uint32_t ph = 0u;
  for (;;) {
    const int cur = stage;
    const int ok = mbar_wait(&sh.full[cur], ph) ? 1 : 0;
    if (++stage == kSeqStages) {
      stage = 0;
      ph ^= 1u;
    }
    if (cbar_or(!ok)) {
      if (tid == 0) atomicOr(p.ctl + 3, kStatusTimeout);
      return;
    }
    const int64_t b = sh.seq[cur];
    if (b < 0) return;
    seq_in_smem<E>(p, sh, ring + (size_t)cur * kSeqStageBytes, b, tid);
    cbar();  // every consumer is done with the stage
    if (lane == 0) mbar_arrive(&sh.empty[cur]);
  }
}

template <typename E>
__global__ void __launch_bounds__(kSeqThreads, 2) verify_seq_kernel(const Params p) {
  extern __shared__ __align__(1024) unsigned char smem[];
  char* ring = reinterpret_cast<char*>(smem);
  SeqShared& sh = *reinterpret_cast<SeqShared*>(smem + (size_t)kSeqStages * kSeqStageBytes);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < kSeqStages; ++i) {
      mbar_init(&sh.full[i], 1u);
      mbar_init(&sh.empty[i], (uint32_t)kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_sync();
  if (tid >= kConsumerThreads) {
    if (tid == kConsumerThreads) seq_producer<E>(p, ring, sh);
    return;
  }
  seq_consumer<E>(p, ring, sh, tid);
}

bool seq_mode_fits(int64_t K, int64_t V, int esz) {
  const int64_t R = 2 * K + 1;
  return R <= kSeqMaxRows && R * V * esz <= kSeqStageBytes && (V * esz) % 16 == 0;
}

// Every kernel is launched with programmatic stream serialization: it may be
// scheduled while the kernel before it on the stream is still finishing, and
// waits for that kernel (grid_dependency_sync) before it touches global
// memory, so only its launch and shared-memory set-up overlap.
template <typename Kern>
static cudaError_t launch_pdl(Kern* k, int grid, int threads, size_t smem, cudaStream_t stream, const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

template <typename E>
static cudaError_t launch_seq_t(const Params& p, int grid, cudaStream_t stream) {
  const size_t smem = seq_shared_bytes();
  auto* k = verify_seq_kernel<E>;
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(k), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, grid, kSeqThreads, smem, stream, p);
}

cudaError_t launch_seq(const Params& p, int dtype, int grid, cudaStream_t stream) {
  return dtype == 1 ? launch_seq_t<uint16_t>(p, grid, stream) : launch_seq_t<float>(p, grid, stream);
}

// ------------------------------------------------- warp-per-sequence mode ---
// Sampling without top-p for short rows (V <= 1024 and the whole sequence
// within 64 KB, rows 16-byte aligned): each warp verifies whole sequences on
// its own, straight from global memory, with warp shuffles only — no shared
// ring, no block barrier, no cross-CTA hand-off. Many sequences are in flight
// per SM at once, which is what short rows need: their per-sequence work is a
// chain of short dependent steps.

constexpr int kWarpThreads = 128;
constexpr int kWarpSeqWarps = kWarpThreads / 32;
constexpr int kWarpMaxRows = 64;
constexpr int64_t kWarpMaxV = 1024;

// Online (max, sum 2^(x c - M c)) of NR rows at once (their loads in flight
// together), every lane ending with the row's totals.
template <typename E, int NR>
__device__ __forceinline__ void warp_rows_ms(const char* row0, const char* row1, int nvec, float c, int lane,
                                             float* m_out, float* s_out) {
  const char* rows[2] = {row0, row1};
  float m[NR], sa[NR][4];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    m[r] = -INFINITY;
    sa[r][0] = sa[r][1] = sa[r][2] = sa[r][3] = 0.f;
  }
  constexpr int kB = 8;  // vectors per lane per row per batch (a whole fp32 row of 1024)
  for (int v0 = lane; v0 < nvec; v0 += 32 * kB) {
    uint4 q[NR][kB];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
#pragma unroll
      for (int k = 0; k < kB; ++k) {
        const int v = v0 + 32 * k;
        q[r][k] = v < nvec ? __ldg(reinterpret_cast<const uint4*>(rows[r]) + v) : neg_inf_vec(E());
      }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      float vmax = vec_max(q[r][0], E());
#pragma unroll
      for (int k = 1; k < kB; ++k) vmax = fmax_nan(vmax, vec_max(q[r][k], E()));
      const float nm = fmax_nan(m[r], vmax);
      if (nm != m[r]) {
        const float f = rescale(m[r], nm, c);
        sa[r][0] *= f; sa[r][1] *= f; sa[r][2] *= f; sa[r][3] *= f;
        m[r] = nm;
      }
      if (m[r] == -INFINITY) continue;
      const float nmc = -mref(m[r], c);
#pragma unroll
      for (int k = 0; k < kB; ++k) vec_exp_add(q[r][k], c, nmc, sa[r], E());
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float mm = m[r], sum = (sa[r][0] + sa[r][1]) + (sa[r][2] + sa[r][3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, mm, o), s2 = __shfl_xor_sync(0xffffffffu, sum, o);
      ms_combine(mm, sum, m2, s2, c);
    }
    m_out[r] = mm;
    s_out[r] = sum;
  }
}

// The draw by one warp over rows of at most kWarpMaxV elements: the smallest
// t with sum_{v<=t} w_v > u * Z (-1 when every weight is zero), w the residual
// max(0, p' - q') (kRes) or p' up to a constant. A group is one 16-byte vector
// of each row; lane l owns groups l, l+32, ... and keeps their sums, so the
// scan that finds the crossing needs no second read; only the crossing
// group's elements are read again.
template <typename E, bool kRes>
__device__ int64_t warp_draw(const char* rp, const char* rq, int64_t V, float c, float nMcp, float nMcq, float ip,
                             float iq, float u, int lane, int& settled) {
  constexpr int PV = ET<E>::kPerVec;
  constexpr int kMaxG = (int)(kWarpMaxV / 4 / 32);  // groups per lane
  const int ng = (int)(V / PV);
  auto weights = [&](const uint4 a, const uint4 bq, float w[PV]) {
    float lp[PV], lq[PV];
    if constexpr (PV == 8) {
      lp[0] = bf_lo(a.x); lp[1] = bf_hi(a.x); lp[2] = bf_lo(a.y); lp[3] = bf_hi(a.y);
      lp[4] = bf_lo(a.z); lp[5] = bf_hi(a.z); lp[6] = bf_lo(a.w); lp[7] = bf_hi(a.w);
      lq[0] = bf_lo(bq.x); lq[1] = bf_hi(bq.x); lq[2] = bf_lo(bq.y); lq[3] = bf_hi(bq.y);
      lq[4] = bf_lo(bq.z); lq[5] = bf_hi(bq.z); lq[6] = bf_lo(bq.w); lq[7] = bf_hi(bq.w);
    } else {
      lp[0] = __uint_as_float(a.x); lp[1] = __uint_as_float(a.y); lp[2] = __uint_as_float(a.z); lp[3] = __uint_as_float(a.w);
      lq[0] = __uint_as_float(bq.x); lq[1] = __uint_as_float(bq.y); lq[2] = __uint_as_float(bq.z); lq[3] = __uint_as_float(bq.w);
    }
#pragma unroll
    for (int k = 0; k < PV; ++k) {
      const float ep = ex2(fmaf(lp[k], c, nMcp));
      w[k] = kRes ? fmaxf(0.f, fmaf(ep, ip, -ex2(fmaf(lq[k], c, nMcq)) * iq)) : ep;
    }
  };
  auto gsum = [&](const float w[PV]) {
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < PV; ++k) a += w[k];
    return a;
  };
  const uint4* pv = reinterpret_cast<const uint4*>(rp);
  const uint4* qv = reinterpret_cast<const uint4*>(rq);
  uint4 a[kMaxG], bq[kMaxG];
#pragma unroll
  for (int i = 0; i < kMaxG; ++i) {
    const int g = i * 32 + lane;
    a[i] = g < ng ? __ldg(pv + g) : neg_inf_vec(E());
    bq[i] = (kRes && g < ng) ? __ldg(qv + g) : neg_inf_vec(E());
  }
  float part[kMaxG];
  float zl = 0.f;
  int64_t lastpos = -1;
#pragma unroll
  for (int i = 0; i < kMaxG; ++i) {
    float w[PV];
    weights(a[i], bq[i], w);
    part[i] = gsum(w);
    zl += part[i];
#pragma unroll
    for (int k = 0; k < PV; ++k)
      if (w[k] > 0.f) lastpos = (int64_t)(i * 32 + lane) * PV + k;
  }
  // the running sums in double-float: they reach the size of Z, where fp32
  // would round at ~6e-8*Z
  df Zd{zl, 0.f};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    df t2;
    t2.h = __shfl_xor_sync(0xffffffffu, Zd.h, o);
    t2.l = __shfl_xor_sync(0xffffffffu, Zd.l, o);
    Zd = df_add(Zd, t2);
  }
  const float Z = Zd.h;
  settled = 0;
  if (!(Z > 0.f)) return -1;
  const df Tg = df_mul_f(Zd, u);
  df run{0.f, 0.f}, before{0.f, 0.f};
  int gstar = -1;  // the group holding the crossing, and the sum before it
#pragma unroll
  for (int i = 0; i < kMaxG; ++i) {
    df incl{part[i], 0.f};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      df t2;
      t2.h = __shfl_up_sync(0xffffffffu, incl.h, o);
      t2.l = __shfl_up_sync(0xffffffffu, incl.l, o);
      if (lane >= o) incl = df_add(incl, t2);
    }
    df tot;
    tot.h = __shfl_sync(0xffffffffu, incl.h, 31);
    tot.l = __shfl_sync(0xffffffffu, incl.l, 31);
    if (gstar < 0 && df_gt(df_add(run, tot), Tg)) {
      const unsigned bal = __ballot_sync(0xffffffffu, df_gt(df_add(run, incl), Tg));
      const int fl = __ffs(bal) - 1;
      gstar = i * 32 + fl;
      const df bl = df_add(run, df_sub(incl, df{part[i], 0.f}));
      before.h = __shfl_sync(0xffffffffu, bl.h, fl);
      before.l = __shfl_sync(0xffffffffu, bl.l, fl);
    }
    run = df_add(run, tot);
  }
  if (gstar >= 0) {  // one lane walks the crossing group, read again
    int64_t t = -1;
    int ok = 0;
    if (lane == 0) {
      float w[PV];
      weights(__ldg(pv + gstar), kRes ? __ldg(qv + gstar) : neg_inf_vec(E()), w);
      const df rem = df_sub(Tg, before);
      const float Tl = rem.h + rem.l;  // what is left of the target inside the group
      float acc = 0.f;
      int64_t lp = -1;
#pragma unroll
      for (int k = 0; k < PV; ++k) {
        if (t < 0) {
          const float prev = acc;
          acc += w[k];
          if (w[k] > 0.f) lp = (int64_t)gstar * PV + k;
          if (acc > Tl) {
            t = (int64_t)gstar * PV + k;
            ok = fminf(acc - Tl, Tl - prev) >= rf::kRefineMargin * Z;
          }
        }
      }
      if (t < 0) t = lp;  // rounding inside the group
    }
    settled = __shfl_sync(0xffffffffu, ok, 0);
    return __shfl_sync(0xffffffffu, (long long)t, 0);
  }
  // u*Z at or past the total after rounding: the last positive weight
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lastpos = max((long long)lastpos, __shfl_xor_sync(0xffffffffu, (long long)lastpos, o));
  return lastpos;
}

template <typename E>
__global__ void __launch_bounds__(kWarpThreads, 4) verify_warp_kernel(const Params p) {
  __shared__ float s_m[kWarpSeqWarps][kWarpMaxRows], s_s[kWarpSeqWarps][kWarpMaxRows];
  constexpr int S = ET<E>::kSize;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.K, R = p.RS;
  const int64_t V = p.V;
  const float c = p.c;
  const int nvec = (int)(V / ET<E>::kPerVec);
  float* rm = s_m[warp];
  float* rsum = s_s[warp];
  // No early trigger: this grid may leave SMs empty, and the next one should
  // spread over all of them rather than fill the free slots of this one.
  grid_dependency_sync(false);
  for (int64_t b = (int64_t)blockIdx.x * kWarpSeqWarps + warp; b < p.B; b += (int64_t)gridDim.x * kWarpSeqWarps) {
    auto rowp = [&](int r) {
      return r <= K ? p.a + ((b * (K + 1) + r) * V) * S : p.d + ((b * K + (r - K - 1)) * V) * S;
    };
    // this lane's first position's token and uniform, read while the rows stream
    const int32_t x0 = lane < K ? __ldg(p.tokens + b * K + lane) : 0;
    const float u0 = lane < K ? __ldg(p.uniforms + b * (K + 1) + lane) : 0.f;
    const float uK = __ldg(p.uniforms + b * (K + 1) + K);
    // ---- per-row (max, sum), two rows' loads in flight together
    for (int r = 0; r < R; r += 2) {
      float m2[2], s2[2];
      if (r + 1 < R)
        warp_rows_ms<E, 2>(rowp(r), rowp(r + 1), nvec, c, lane, m2, s2);
      else
        warp_rows_ms<E, 1>(rowp(r), nullptr, nvec, c, lane, m2, s2);
      if (lane == 0) {
        rm[r] = m2[0];
        rsum[r] = s2[0];
        if (r + 1 < R) {
          rm[r + 1] = m2[1];
          rsum[r + 1] = s2[1];
        }
      }
    }
    __syncwarp();
    // ---- row stats out, validity, accept scan
    int bad = 0;
    for (int r = lane; r < R; r += 32) {
      const float M = rm[r], sm = rsum[r];
      const bool valid = (M > -INFINITY) && (M < INFINITY);
      if (!valid) bad = 1;
      if (p.out_row_stats) {
        float4 o;
        o.x = valid ? __fdiv_rn(M, p.T) : __int_as_float(0x7fc00000);
        o.y = valid ? (mref(M, c) + lg2(sm)) * 0.69314718055994531f : __int_as_float(0x7fc00000);
        o.z = valid ? 1.f : __int_as_float(0x7fc00000);
        o.w = -INFINITY;
        reinterpret_cast<float4*>(p.out_row_stats)[b * R + r] = o;
      }
    }
    int jl = K;
    for (int i = lane; i < K; i += 32) {
      const int32_t x = i == lane ? x0 : p.tokens[b * K + i];
      const float u = i == lane ? u0 : p.uniforms[b * (K + 1) + i];
      if (x < 0 || (int64_t)x >= V || !(u >= 0.f && u < 1.f)) {
        bad = 1;
        continue;
      }
      const float Mp = rm[i], Mq = rm[K + 1 + i];
      if (!(Mp > -INFINITY && Mp < INFINITY && Mq > -INFINITY && Mq < INFINITY)) continue;  // counted above
      const float lp = ET<E>::load(rowp(i), x), lq = ET<E>::load(rowp(K + 1 + i), x);
      float alpha;
      if (lp == -INFINITY) alpha = 0.f;
      else if (lq == -INFINITY) alpha = 1.f;
      else alpha = fminf(1.f, ex2(fmaf(lp, c, -mref(Mp, c)) - fmaf(lq, c, -mref(Mq, c))) * (rsum[K + 1 + i] / rsum[i]));
      if (!(u < alpha) && i < jl) jl = i;
    }
    if (lane == 0 && !(uK >= 0.f && uK < 1.f)) bad = 1;
    const int j = (int)__reduce_min_sync(0xffffffffu, (unsigned)jl);
    int32_t* out = p.out_tokens + b * (K + 1);
    if (__any_sync(0xffffffffu, bad)) {
      for (int i = lane; i <= K; i += 32) out[i] = -1;
      if (lane == 0) {
        p.out_accept_len[b] = -1;
        atomicOr(p.ctl + 3, kStatusInput);
      }
      continue;
    }
    // ---- the draw
    const float nMp = -mref(rm[j], c), ip = 1.f / rsum[j];
    int64_t t = -1;
    int settled = 1, st2 = 0;
    if (j < K) {
      const float nMq = -mref(rm[K + 1 + j], c), iq = 1.f / rsum[K + 1 + j];
      t = warp_draw<E, true>(rowp(j), rowp(K + 1 + j), V, c, nMp, nMq, ip, iq, uK, lane, settled);
    }
    if (t < 0) {  // the bonus draw, or a residual that is all zero in fp32 (which stays unsettled)
      t = warp_draw<E, false>(rowp(j), nullptr, V, c, nMp, 0.f, 1.f, 0.f, uK, lane, st2);
      if (j == K) settled = st2;
    }
    for (int i = lane; i <= K; i += 32) out[i] = i < j ? p.tokens[b * K + i] : (i == j ? (int32_t)t : -1);
    if (lane == 0) {
      p.out_accept_len[b] = j;
      if (!settled && p.rf_ctl) {  // the refine kernel redoes this draw
        rf::Rec r{};
        r.b = (int32_t)b;
        r.j = j;
        r.resid = j < K ? 1 : 0;
        r.mp = rm[j];
        r.mq = j < K ? rm[K + 1 + j] : 0.f;
        r.taup = r.tauq = -INFINITY;
        r.u = uK;
        rf::flag(p.rf_ctl, p.rf_recs, p.B, r);
      }
    }
    __syncwarp();
  }
}

bool warp_mode_fits(int64_t K, int64_t V, int esz) {
  const int64_t R = 2 * K + 1;
  return R <= kWarpMaxRows && V <= kWarpMaxV && (V * esz) % 16 == 0 && R * V * esz <= 65536;
}

template <typename E>
static cudaError_t launch_warp_t(const Params& p, int grid, cudaStream_t stream) {
  return launch_pdl(verify_warp_kernel<E>, grid, kWarpThreads, 0, stream, p);
}

cudaError_t launch_warp(const Params& p, int dtype, int grid, cudaStream_t stream) {
  return dtype == 1 ? launch_warp_t<uint16_t>(p, grid, stream) : launch_warp_t<float>(p, grid, stream);
}

int warp_mode_seqs_per_cta() { return kWarpSeqWarps; }

// ------------------------------------------------------------ self-test ------
// The bounded-wait path, made to run out on purpose without any fault: one
// thread waits for a control word that nothing ever sets, gives up after
// limit_ns like every wait in the kernels, and records a timeout in the
// status word the host reads.
__global__ void wait_selftest_kernel(uint32_t* ctl, uint64_t limit_ns) {
  if (threadIdx.x != 0) return;
  const uint64_t t0 = globaltimer_ns();
  uint32_t v = ld_acquire_gpu(ctl + kCtlNeverSet);
  while (v == 0u && globaltimer_ns() - t0 < limit_ns) v = ld_acquire_gpu(ctl + kCtlNeverSet);
  if (v == 0u) atomicOr(ctl + 3, kStatusTimeout);
}

cudaError_t launch_wait_selftest(uint32_t* ctl, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(ctl, limit_ns);
  return cudaGetLastError();
}

// ------------------------------------------------------------- launching ------

template <typename E, int MODE>
static cudaError_t launch_t(const Params& p, int grid, cudaStream_t stream) {
  const size_t smem = shared_bytes(p.stages);
  auto* k = verify_kernel<E, MODE>;
  cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(k), shared_bytes(kMaxStages));
  if (e != cudaSuccess) return e;
  return launch_pdl(k, grid, kAllThreads, smem, stream, p);
}

int kernel_threads() { return kAllThreads; }

cudaError_t launch(const Params& p, int dtype, int mode, int grid, cudaStream_t stream) {
  if (dtype == 1) {
    if (mode == kSample) return launch_t<uint16_t, kSample>(p, grid, stream);
    if (mode == kArgmaxLimit) return launch_t<uint16_t, kArgmaxLimit>(p, grid, stream);
    return launch_t<uint16_t, kGreedy>(p, grid, stream);
  }
  if (mode == kSample) return launch_t<float, kSample>(p, grid, stream);
  if (mode == kArgmaxLimit) return launch_t<float, kArgmaxLimit>(p, grid, stream);
  return launch_t<float, kGreedy>(p, grid, stream);
}

}  // namespace sv
