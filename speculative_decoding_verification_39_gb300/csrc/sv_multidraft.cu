// sv_multidraft.cu — the multi-draft sampling verify on sm_103a.
//
// G drafts, each drawn from its own draft distribution, are tested position by
// position as in the Lookahead sampling verify ("Lookahead Decoding 完全拆解",
// section "采样模式的验证"), but with full draft distributions: draft g's
// token x is accepted with probability min(1, p(x)/q_g(x)), and a rejection
// replaces p by norm(max(0, p - q_g)) — the single-draft rule of
// "Speculative Decoding —— LLM推理优化技术（一）" §2.1, applied once per
// rejected draft.
//
// Two kernels on the caller's stream:
//  md_rows_kernel — one CTA per row, target rows [B,G,N,V] then draft rows
//    [B,G,N-1,V]: the row's normaliser (M = max l*c, S = sum 2^(l*c - M)) in
//    one read, and the logit of every draft's token at the row's position.
//  md_walk_kernel — one CTA per sequence. The current distribution at a
//    position is a chain: the owner's target p, then one residual step per
//    rejected draft, each link holding the draft row, its (M, 1/S) and the
//    1/Z of its residual. Thread 0 evaluates the chain at a draft's token from
//    the gathered logits to decide acceptance; after a rejection the whole CTA
//    evaluates the chain over the row to get the new residual's mass. The
//    draw walks the final chain by chunk sums, a block scan and one chunk
//    walk. Both sides evaluate the chain with the same expression, so a
//    rejected token has exactly zero residual weight afterwards.
#include <climits>
#include <cmath>
#include <mutex>
#include <set>

#include "sv_device.cuh"
#include "sv_multidraft.h"
#include "sv_rowstat.cuh"

namespace sv {
namespace md {
namespace {

using rowstat::combine;
using rowstat::Elem;
using rowstat::fold;

constexpr int kRowThreads = 256;
constexpr int kWalkThreads = 512;
constexpr int kWalkWarps = kWalkThreads / 32;
constexpr float kLn2 = 0.693147180559945309f;

// One CTA per row: r < B*G*N is target row (b*G + a)*N + n, the rest are
// draft rows (b*G + j)*(N-1) + n.
template <typename E>
__global__ void __launch_bounds__(kRowThreads, 8) md_rows_kernel(const Params p) {
  using X = Elem<E>;
  constexpr int PV = X::kPerVec;
  constexpr int U = 4;
  const int tid = threadIdx.x;
  const int G = p.G, N = p.N;
  const int64_t V = p.V;
  const int64_t RT = p.B * G * N;
  const int64_t r = blockIdx.x;
  const E* row;
  if (r < RT) {
    const int n = (int)(r % N);
    const int64_t ba = r / N;
    const int64_t b = ba / G;
    row = static_cast<const E*>(p.target) + r * V;
    if (n < N - 1 && tid < G) {
      const int32_t t = p.tokens[(b * G + tid) * (N - 1) + n];
      p.gp[(ba * (N - 1) + n) * G + tid] = (t >= 0 && (int64_t)t < V) ? X::load(row + t) * p.c : 0.f;
    }
  } else {
    const int64_t rd = r - RT;
    const int n = (int)(rd % (N - 1));
    const int64_t bj = rd / (N - 1);
    const int64_t b = bj / G;
    row = static_cast<const E*>(p.draft) + rd * V;
    if (tid < G) {
      const int32_t t = p.tokens[(b * G + tid) * (N - 1) + n];
      p.gq[(bj * (N - 1) + n) * G + tid] = (t >= 0 && (int64_t)t < V) ? X::load(row + t) * p.c : 0.f;
    }
  }

  // (V < 2^31, so indices within a row fit in 32 bits.)
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
  int head = (int)(((16u - (unsigned)(addr & 15u)) & 15u) / sizeof(E));
  if (head > (int)V) head = (int)V;
  const int nvec = ((int)V - head) / PV;
  const int tail0 = head + nvec * PV;
  const uint4* vec = reinterpret_cast<const uint4*>(row + head);
  float m = -INFINITY, s = 0.f;
  if (tid < head) {
    const float z = X::load(row + tid) * p.c;
    fold<1>(m, s, &z);
  }
  if (tail0 + tid < (int)V) {
    const float z = X::load(row + tail0 + tid) * p.c;
    fold<1>(m, s, &z);
  }
  for (int i0 = tid; i0 < nvec; i0 += U * kRowThreads) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * kRowThreads;
      v[u] = i < nvec ? __ldg(vec + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (i0 + u * kRowThreads < nvec) {
        float x[PV];
        X::unpack(v[u], x);
#pragma unroll
        for (int k = 0; k < PV; ++k) x[k] *= p.c;
        fold<PV>(m, s, x);
      }
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    combine(m, s, m2, s2);
  }
  __shared__ float2 red[kRowThreads / 32];
  const int warp = tid >> 5, lane = tid & 31;
  if (lane == 0) red[warp] = make_float2(m, s);
  __syncthreads();
  if (warp == 0) {
    const float2 w = lane < kRowThreads / 32 ? red[lane] : make_float2(-INFINITY, 0.f);
    m = w.x;
    s = w.y;
#pragma unroll
    for (int o = kRowThreads / 64; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      combine(m, s, m2, s2);
    }
    if (lane == 0) {
      p.rowstat[r] = make_float2(m, s);
      if (p.out_row_lse) p.out_row_lse[r] = (m + lg2(s)) * kLn2;
    }
  }
}

// The residual chain of the current position, in shared memory.
struct Chain {
  int64_t roff[kMaxG];  // element offset of each link's draft row from the draft base
  int jd[kMaxG];        // its draft index
  float qm[kMaxG];      // its M
  float qsi[kMaxG];     // its 1/S
  float rzi[kMaxG];     // 1/Z of the residual the link produced
  int nr;               // links in use
};

// The current distribution at element v: p = 2^(l*c - M)/S of the target
// row, then p <- max(0, p - q_i(v)) / Z_i for each link i.
template <typename E>
__device__ __forceinline__ float chain_at(const E* trow, const E* dbase, float c, float tm, float tsi,
                                          const Chain& ch, int nr, int64_t v) {
  using X = Elem<E>;
  float pv = ex2(X::load(trow + v) * c - tm) * tsi;
  for (int i = 0; i < nr; ++i) {
    const float qv = ex2(X::load(dbase + ch.roff[i] + v) * c - ch.qm[i]) * ch.qsi[i];
    pv = fmaxf(0.f, pv - qv) * ch.rzi[i];
  }
  return pv;
}

// Sum over the CTA; every thread gets the total.
__device__ __forceinline__ float block_sum(float v, float* red, float* out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float t = lane < kWalkWarps ? red[lane] : 0.f;
    t = warp_sum(t);
    if (lane == 0) *out = t;
  }
  __syncthreads();
  return *out;
}

// One CTA per sequence b.
template <typename E>
__global__ void __launch_bounds__(kWalkThreads, 1) md_walk_kernel(const Params p) {
  using X = Elem<E>;
  __shared__ float2 stt[kMaxRowsPerSeq];    // target rows, a*N + n
  __shared__ float2 std_[kMaxRowsPerSeq];   // draft rows, j*(N-1) + n
  __shared__ float gps[kMaxGather];         // (a*(N-1) + n)*G + k
  __shared__ float gqs[kMaxGather];         // (j*(N-1) + n)*G + k
  __shared__ int32_t cs[kMaxRowsPerSeq];    // draft tokens, k*(N-1) + n
  __shared__ float us[kMaxRowsPerSeq + 1];  // the uniforms
  __shared__ int alive[kMaxG];
  __shared__ Chain ch;
  __shared__ float red[kWalkWarps], wtot[kWalkWarps];
  __shared__ float sh_sum;
  __shared__ int sh_lead, sh_acc, sh_cross, sh_lastpos, sh_tok;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, N = p.N;
  const int R = G * N, RD = G * (N - 1), NU = RD + 1, NG = G * RD;
  const int64_t V = p.V;
  const int64_t b = blockIdx.x;
  const float c = p.c;
  const E* tbase = static_cast<const E*>(p.target);
  const E* dbase = static_cast<const E*>(p.draft);

  int bad = 0;
  for (int i = tid; i < RD; i += kWalkThreads) {
    const int32_t t = p.tokens[b * RD + i];
    cs[i] = t;
    bad |= (t < 0 || (int64_t)t >= V);
  }
  for (int i = tid; i < NU; i += kWalkThreads) {
    const float u = p.uniforms[b * NU + i];
    us[i] = u;
    bad |= !(u >= 0.f && u < 1.f);
  }
  if (tid < G) alive[tid] = 1;
  grid_dependency_sync(false);
  const int64_t RT = p.B * R;
  for (int i = tid; i < R; i += kWalkThreads) {
    const float2 v = p.rowstat[b * R + i];
    stt[i] = v;
    bad |= !(v.x > -INFINITY && v.x < INFINITY);
  }
  for (int i = tid; i < RD; i += kWalkThreads) {
    const float2 v = p.rowstat[RT + b * RD + i];
    std_[i] = v;
    bad |= !(v.x > -INFINITY && v.x < INFINITY);
  }
  for (int i = tid; i < NG; i += kWalkThreads) {
    gps[i] = p.gp[b * NG + i];
    gqs[i] = p.gq[b * NG + i];
  }
  if (tid == 0) {
    sh_lead = 0;
    ch.nr = 0;
  }
  if (__syncthreads_or(bad)) {
    for (int i = tid; i < N; i += kWalkThreads) p.out_tokens[b * N + i] = -1;
    if (tid == 0) {
      p.out_accept_len[b] = -1;
      if (p.out_best) p.out_best[b] = -1;
      atomicOr(p.ctl + 3, kStatusInput);
    }
    return;
  }

  // The walk. Every branch below depends only on shared state written before
  // a barrier, so the whole CTA takes it together.
  int j = N - 1;
  for (int n = 0; n < N - 1; ++n) {
    const int a = sh_lead;
    const float2 tms = stt[a * N + n];
    const float tsi = 1.f / tms.y;
    const E* trow = tbase + ((b * G + a) * N + n) * V;
    int acc = -1;
    for (int k = 0; k < G; ++k) {
      if (!alive[k]) continue;
      const float2 qms = std_[k * (N - 1) + n];
      const float qsi = 1.f / qms.y;
      if (tid == 0) {
        // The chain at draft k's token, from the gathered logits.
        const int nr = ch.nr;
        float pc = ex2(gps[(a * (N - 1) + n) * G + k] - tms.x) * tsi;
        for (int i = 0; i < nr; ++i) {
          const float qv = ex2(gqs[(ch.jd[i] * (N - 1) + n) * G + k] - ch.qm[i]) * ch.qsi[i];
          pc = fmaxf(0.f, pc - qv) * ch.rzi[i];
        }
        const float qk = ex2(gqs[(k * (N - 1) + n) * G + k] - qms.x) * qsi;
        const float alpha = pc > 0.f ? (qk > 0.f ? fminf(1.f, pc / qk) : 1.f) : 0.f;
        sh_acc = us[n * G + k] < alpha;
      }
      __syncthreads();
      if (sh_acc) {
        acc = k;
        break;
      }
      // Rejected: the mass of max(0, p - q_k) over the row.
      const E* krow = dbase + ((b * G + k) * (N - 1) + n) * V;
      const int nr = ch.nr;
      float z = 0.f;
      for (int64_t v = tid; v < V; v += kWalkThreads) {
        const float pv = chain_at(trow, dbase, c, tms.x, tsi, ch, nr, v);
        const float qv = ex2(X::load(krow + v) * c - qms.x) * qsi;
        z += fmaxf(0.f, pv - qv);
      }
      z = block_sum(z, red, &sh_sum);
      if (tid == 0 && z > 0.f) {  // a zero residual keeps p
        ch.roff[nr] = ((b * G + k) * (N - 1) + n) * V;
        ch.jd[nr] = k;
        ch.qm[nr] = qms.x;
        ch.qsi[nr] = qsi;
        ch.rzi[nr] = 1.f / z;
        ch.nr = nr + 1;
      }
      __syncthreads();
    }
    if (acc < 0) {
      j = n;
      break;
    }
    const int32_t xa = cs[acc * (N - 1) + n];
    const int keep = tid < G ? (alive[tid] && cs[tid * (N - 1) + n] == xa) : 0;
    __syncthreads();
    if (tid < G) alive[tid] = keep;
    if (tid == 0) {
      sh_lead = acc;
      ch.nr = 0;
    }
    __syncthreads();
  }

  // The draw at position j (the bonus at N-1, from the owner's plain row).
  const int lead = sh_lead;
  const float2 tms = stt[lead * N + j];
  const float tsi = 1.f / tms.y;
  const E* trow = tbase + ((b * G + lead) * N + j) * V;
  const float target_u = us[RD];
  const int64_t CH = (V + kWalkThreads - 1) / kWalkThreads;
  const int64_t lo = (int64_t)tid * CH < V ? (int64_t)tid * CH : V;
  const int64_t hi = lo + CH < V ? lo + CH : V;
  int nr = j < N - 1 ? ch.nr : 0;
  if (tid == 0) sh_tok = (int)(V - 1);
  for (int attempt = 0; attempt < 2; ++attempt) {
    float s = 0.f;
    for (int64_t v = lo; v < hi; ++v) s += chain_at(trow, dbase, c, tms.x, tsi, ch, nr, v);
    const float inw = warp_incl_scan(s, lane);
    if (lane == 31) wtot[warp] = inw;
    if (tid == 0) {
      sh_cross = INT_MAX;
      sh_lastpos = -1;
    }
    __syncthreads();
    if (warp == 0) {
      float t = lane < kWalkWarps ? wtot[lane] : 0.f;
      t = warp_incl_scan(t, lane);
      __syncwarp();
      if (lane < kWalkWarps) wtot[lane] = t;
    }
    __syncthreads();
    const float base = warp > 0 ? wtot[warp - 1] : 0.f;
    const float incl = base + inw;
    const float Z = wtot[kWalkWarps - 1];
    if (!(Z > 0.f) && attempt == 0 && nr > 0) {  // rounding only: fall back to p
      nr = 0;
      __syncthreads();
      continue;
    }
    const float target = target_u * Z;
    if (s > 0.f && incl > target) atomicMin(&sh_cross, tid);
    if (s > 0.f) atomicMax(&sh_lastpos, tid);
    __syncthreads();
    const int cross = sh_cross;
    const int owner = cross != INT_MAX ? cross : sh_lastpos;
    if (tid == owner) {
      float C = incl - s;
      int64_t tok = -1, last = -1;
      for (int64_t v = lo; v < hi; ++v) {
        const float w = chain_at(trow, dbase, c, tms.x, tsi, ch, nr, v);
        if (w > 0.f) last = v;
        C += w;
        if (cross != INT_MAX && C > target) {
          tok = v;
          break;
        }
      }
      sh_tok = (int)(tok >= 0 ? tok : last);
    }
    break;
  }
  __syncthreads();

  for (int i = tid; i < N; i += kWalkThreads)
    p.out_tokens[b * N + i] = i < j ? cs[lead * (N - 1) + i] : (i == j ? sh_tok : -1);
  if (tid == 0) {
    p.out_accept_len[b] = j;
    if (p.out_best) p.out_best[b] = lead;
  }
}

// ------------------------------------------------------ resident walk ---
// The walk with the current distribution of the position held in shared
// memory (V floats): a position starts from the owner's target row, p(v) =
// 2^(fl(l c) - M) / S; a rejected draft k replaces it in place by
// max(0, p - q_k) * (1/Z) — one read of draft k's row; the accept test reads
// p(x) from the same array and computes q_k(x) with the same expression as
// the update, so a rejected token keeps exactly zero weight. A residual of
// zero mass (rare: p <= q_k everywhere) keeps p, which is then rebuilt from
// the target row and the position's earlier links.
constexpr int kResThreads = 1024;
constexpr int kResWarps = kResThreads / 32;

// f(v, l) over every element of a row, 16-byte vectors first (four in
// flight per thread) when the row is aligned; f gets 8 (bf16) or 4 (fp32)
// consecutive elements at once through fv(v0, x[]) and single ones through f1.
template <typename E, typename FV, typename F1>
__device__ __forceinline__ void row_pass(const E* row, int64_t V, bool vec, FV fv, F1 f1) {
  using X = Elem<E>;
  constexpr int PV = X::kPerVec;
  const int tid = threadIdx.x;
  int64_t done = 0;
  if (vec) {
    const int64_t nv = V / PV;
    const uint4* vp = reinterpret_cast<const uint4*>(row);
    for (int64_t i0 = tid; i0 < nv; i0 += 4 * kResThreads) {
      uint4 u[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t i = i0 + (int64_t)k * kResThreads;
        u[k] = i < nv ? __ldg(vp + i) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t i = i0 + (int64_t)k * kResThreads;
        if (i < nv) {
          float x[PV];
          X::unpack(u[k], x);
          fv(i * PV, x);
        }
      }
    }
    done = nv * PV;
  }
  for (int64_t v = done + tid; v < V; v += kResThreads) f1(v, X::load(row + v));
}

template <typename E>
__global__ void __launch_bounds__(kResThreads, 1) md_walk_res_kernel(const Params p) {
  using X = Elem<E>;
  constexpr int PV = X::kPerVec;
  extern __shared__ __align__(16) float P[];  // [V] the current distribution
  __shared__ float2 stt[kMaxRowsPerSeq];    // target rows, a*N + n
  __shared__ float2 std_[kMaxRowsPerSeq];   // draft rows, j*(N-1) + n
  __shared__ int32_t cs[kMaxRowsPerSeq];    // draft tokens, k*(N-1) + n
  __shared__ float us[kMaxRowsPerSeq + 1];  // the uniforms
  __shared__ int alive[kMaxG];
  __shared__ Chain ch;
  __shared__ float red[kResWarps], wtot[kResWarps];
  __shared__ float sh_sum;
  __shared__ int sh_acc, sh_cross, sh_lastpos, sh_tok;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, N = p.N;
  const int R = G * N, RD = G * (N - 1), NU = RD + 1;
  const int64_t V = p.V;
  const int64_t b = blockIdx.x;
  const float c = p.c;
  const E* tbase = static_cast<const E*>(p.target);
  const E* dbase = static_cast<const E*>(p.draft);
  // rows start on 16-byte boundaries when V fills whole vectors and the
  // bases are aligned
  const bool vec = (V % PV) == 0 && (reinterpret_cast<uintptr_t>(tbase) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(dbase) & 15u) == 0;

  int bad = 0;
  for (int i = tid; i < RD; i += kResThreads) {
    const int32_t t = p.tokens[b * RD + i];
    cs[i] = t;
    bad |= (t < 0 || (int64_t)t >= V);
  }
  for (int i = tid; i < NU; i += kResThreads) {
    const float u = p.uniforms[b * NU + i];
    us[i] = u;
    bad |= !(u >= 0.f && u < 1.f);
  }
  if (tid < G) alive[tid] = 1;
  grid_dependency_sync(false);
  const int64_t RT = p.B * R;
  for (int i = tid; i < R; i += kResThreads) {
    const float2 v = p.rowstat[b * R + i];
    stt[i] = v;
    bad |= !(v.x > -INFINITY && v.x < INFINITY);
  }
  for (int i = tid; i < RD; i += kResThreads) {
    const float2 v = p.rowstat[RT + b * RD + i];
    std_[i] = v;
    bad |= !(v.x > -INFINITY && v.x < INFINITY);
  }
  if (__syncthreads_or(bad)) {
    for (int i = tid; i < N; i += kResThreads) p.out_tokens[b * N + i] = -1;
    if (tid == 0) {
      p.out_accept_len[b] = -1;
      if (p.out_best) p.out_best[b] = -1;
      atomicOr(p.ctl + 3, kStatusInput);
    }
    return;
  }

  // P <- the target row (b, a, n): 2^(fl(l c) - M) / S
  auto load_target = [&](int a, int n) {
    const float2 tms = stt[a * N + n];
    const float tsi = 1.f / tms.y;
    const E* trow = tbase + ((b * G + a) * N + n) * V;
    row_pass<E>(
        trow, V, vec,
        [&](int64_t v0, const float* x) {
#pragma unroll
          for (int k = 0; k < PV; k += 4) {
            float4 o;
            o.x = ex2(__fmul_rn(x[k], c) - tms.x) * tsi;
            o.y = ex2(__fmul_rn(x[k + 1], c) - tms.x) * tsi;
            o.z = ex2(__fmul_rn(x[k + 2], c) - tms.x) * tsi;
            o.w = ex2(__fmul_rn(x[k + 3], c) - tms.x) * tsi;
            *reinterpret_cast<float4*>(P + v0 + k) = o;
          }
        },
        [&](int64_t v, float l) { P[v] = ex2(__fmul_rn(l, c) - tms.x) * tsi; });
  };

  int j = N - 1;
  int lead = 0;
  for (int n = 0; n < N - 1; ++n) {
    load_target(lead, n);
    if (tid == 0) ch.nr = 0;
    __syncthreads();
    int acc = -1;
    for (int k = 0; k < G; ++k) {
      if (!alive[k]) continue;
      const float2 qms = std_[k * (N - 1) + n];
      const float qsi = 1.f / qms.y;
      const E* krow = dbase + ((b * G + k) * (N - 1) + n) * V;
      if (tid == 0) {
        const int32_t x = cs[k * (N - 1) + n];
        const float pc = P[x];
        const float qk = ex2(__fmul_rn(X::load(krow + x), c) - qms.x) * qsi;
        const float alpha = pc > 0.f ? (qk > 0.f ? fminf(1.f, pc / qk) : 1.f) : 0.f;
        sh_acc = us[n * G + k] < alpha;
      }
      __syncthreads();
      if (sh_acc) {
        acc = k;
        break;
      }
      // Rejected: P <- max(0, P - q_k), then scaled by 1/Z.
      float z = 0.f;
      row_pass<E>(
          krow, V, vec,
          [&](int64_t v0, const float* x) {
#pragma unroll
            for (int kk = 0; kk < PV; kk += 4) {
              float4 o = *reinterpret_cast<const float4*>(P + v0 + kk);
              o.x = fmaxf(0.f, o.x - ex2(__fmul_rn(x[kk], c) - qms.x) * qsi);
              o.y = fmaxf(0.f, o.y - ex2(__fmul_rn(x[kk + 1], c) - qms.x) * qsi);
              o.z = fmaxf(0.f, o.z - ex2(__fmul_rn(x[kk + 2], c) - qms.x) * qsi);
              o.w = fmaxf(0.f, o.w - ex2(__fmul_rn(x[kk + 3], c) - qms.x) * qsi);
              z += (o.x + o.y) + (o.z + o.w);
              *reinterpret_cast<float4*>(P + v0 + kk) = o;
            }
          },
          [&](int64_t v, float l) {
            const float r = fmaxf(0.f, P[v] - ex2(__fmul_rn(l, c) - qms.x) * qsi);
            z += r;
            P[v] = r;
          });
      z = warp_sum(z);
      if (lane == 0) red[warp] = z;
      __syncthreads();
      if (warp == 0) {
        float t = red[lane];
        t = warp_sum(t);
        if (lane == 0) sh_sum = t;
      }
      __syncthreads();
      z = sh_sum;
      const int nr = ch.nr;
      if (z > 0.f) {
        const float rz = 1.f / z;
        for (int64_t v = tid; v < V; v += kResThreads) P[v] *= rz;
        if (tid == 0) {
          ch.roff[nr] = ((b * G + k) * (N - 1) + n) * V;
          ch.jd[nr] = k;
          ch.qm[nr] = qms.x;
          ch.qsi[nr] = qsi;
          ch.rzi[nr] = rz;
          ch.nr = nr + 1;
        }
      } else {
        // a residual of zero mass keeps p: rebuild it from the target row and
        // the position's earlier links
        const float2 tms = stt[lead * N + n];
        const float tsi = 1.f / tms.y;
        const E* trow = tbase + ((b * G + lead) * N + n) * V;
        for (int64_t v = tid; v < V; v += kResThreads) P[v] = chain_at(trow, dbase, c, tms.x, tsi, ch, nr, v);
      }
      __syncthreads();
    }
    if (acc < 0) {
      j = n;
      break;
    }
    const int32_t xa = cs[acc * (N - 1) + n];
    const int keep = tid < G ? (alive[tid] && cs[tid * (N - 1) + n] == xa) : 0;
    __syncthreads();
    if (tid < G) alive[tid] = keep;
    lead = acc;
    __syncthreads();
  }
  if (j == N - 1) {  // every position accepted: the bonus from the owner's last row
    load_target(lead, N - 1);
    __syncthreads();
  }

  // The draw from P: warp w sums [w*SW, (w+1)*SW) with its lanes on
  // consecutive elements; the crossing warp walks its segment 32 at a time.
  const float target_u = us[RD];
  const int64_t SW = ((V + kResWarps - 1) / kResWarps + 31) / 32 * 32;
  const int64_t lo = min((int64_t)warp * SW, V), hi = min(lo + SW, V);
  float s = 0.f;
  for (int64_t v = lo + lane; v < hi; v += 32) s += P[v];
  s = warp_sum(s);
  if (lane == 0) wtot[warp] = s;
  if (tid == 0) {
    sh_cross = INT_MAX;
    sh_lastpos = -1;
    sh_tok = (int)(V - 1);
  }
  __syncthreads();
  if (warp == 0) {
    float t = wtot[lane];
    t = warp_incl_scan(t, lane);
    __syncwarp();
    wtot[lane] = t;
  }
  __syncthreads();
  const float base = warp > 0 ? wtot[warp - 1] : 0.f;
  const float Z = wtot[kResWarps - 1];
  const float target = target_u * Z;
  if (lane == 0) {
    if (s > 0.f && base + s > target) atomicMin(&sh_cross, warp);
    if (s > 0.f) atomicMax(&sh_lastpos, warp);
  }
  __syncthreads();
  const int cw = sh_cross != INT_MAX ? sh_cross : sh_lastpos;
  if (warp == cw && cw >= 0) {
    // the crossing within the segment; if rounding leaves none, the last
    // positive weight of the segment
    float C = base;
    int tok = -1, last = -1;
    for (int64_t v0 = lo; v0 < hi && tok < 0; v0 += 32) {
      const int64_t v = v0 + lane;
      const float w = v < hi ? P[v] : 0.f;
      const float incl = C + warp_incl_scan(w, lane);
      const uint32_t pos = __ballot_sync(0xffffffffu, w > 0.f);
      if (pos) last = (int)(v0 + 31 - __clz(pos));
      const uint32_t m = __ballot_sync(0xffffffffu, sh_cross != INT_MAX && w > 0.f && incl > target);
      if (m) tok = (int)(v0 + __ffs(m) - 1);
      C = __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) sh_tok = tok >= 0 ? tok : last;
  }
  __syncthreads();

  for (int i = tid; i < N; i += kResThreads)
    p.out_tokens[b * N + i] = i < j ? cs[lead * (N - 1) + i] : (i == j ? sh_tok : -1);
  if (tid == 0) {
    p.out_accept_len[b] = j;
    if (p.out_best) p.out_best[b] = lead;
  }
}

// Dynamic shared memory of the resident walk, and whether it fits.
inline size_t res_smem_bytes(int64_t V) { return (size_t)((V + 3) / 4 * 4) * sizeof(float); }

template <typename E>
cudaError_t launch_t(const Params& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.G * (2 * p.N - 1)));
  cfg.blockDim = dim3(kRowThreads);
  cfg.stream = stream;
  cudaError_t e = cudaLaunchKernelEx(&cfg, md_rows_kernel<E>, p);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)p.B);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the resident walk where the row fits in shared memory next to the
  // kernel's static arrays
  static const size_t kResBudget = 200 * 1024;
  if (res_smem_bytes(p.V) <= kResBudget) {
    static std::mutex mu;
    static std::set<int> raised;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
      std::lock_guard<std::mutex> lk(mu);
      if (!raised.count(dev)) {
        e = cudaFuncSetAttribute(md_walk_res_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kResBudget);
        if (e != cudaSuccess) return e;
        raised.insert(dev);
      }
    }
    cfg.blockDim = dim3(kResThreads);
    cfg.dynamicSmemBytes = res_smem_bytes(p.V);
    return cudaLaunchKernelEx(&cfg, md_walk_res_kernel<E>, p);
  }
  cfg.blockDim = dim3(kWalkThreads);
  return cudaLaunchKernelEx(&cfg, md_walk_kernel<E>, p);
}

}  // namespace

cudaError_t launch(const Params& p, int dtype, cudaStream_t stream) {
  return dtype == 1 ? launch_t<uint16_t>(p, stream) : launch_t<float>(p, stream);
}

}  // namespace md
}  // namespace sv
