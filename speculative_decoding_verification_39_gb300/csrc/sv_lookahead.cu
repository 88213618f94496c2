// sv_lookahead.cu — the Lookahead sampling-mode verify ("Lookahead Decoding
// 完全拆解", section "采样模式的验证") on sm_103a.
//
// The candidates were produced greedily, so the draft distribution of every
// candidate token is one-hot: token x is accepted with probability
// min(1, p(x)/1) = p(x), and a rejection leaves p with x removed and
// renormalised (the residual norm(max(0, p - q)) of "Speculative Decoding ——
// LLM推理优化技术（一）" §2.1, with q one-hot on x).
//
// Two kernels on the caller's stream:
//  la_rows_kernel — one CTA per row of logits[B,G,N,V]. One read of the row
//    gives its normaliser: M = max_v l_v*c and S = sum_v 2^(l_v*c - M), with
//    c = log2(e)/T. The same CTA picks up, for that row's position, the logit
//    of every candidate's token, so the walk needs nothing else from the rows.
//  la_walk_kernel — one CTA per sequence. Warp 0 walks the positions: the
//    candidates still matching the accepted prefix are tested in order of g,
//    candidate k with alpha = w_k / (S - D), where w_k = 2^(l_k*c - M) and D
//    is the mass of the distinct tokens already rejected at that position.
//    The CTA then draws the token at the stopping position from the owner's
//    row with the rejected tokens skipped (or the bonus from row N-1): a sum
//    over contiguous per-thread chunks of the row, a block scan, and one
//    thread's walk through the chunk holding the crossing. The first kernel
//    has just read that row, so the draw reads it from L2.
#include <climits>
#include <cmath>

#include "sv_device.cuh"
#include "sv_lookahead.h"
#include "sv_rowstat.cuh"

namespace sv {
namespace la {
namespace {

using rowstat::combine;
using rowstat::Elem;
using rowstat::fold;

constexpr int kRowThreads = 256;
constexpr int kWalkThreads = 512;
constexpr int kWalkWarps = kWalkThreads / 32;
constexpr float kLn2 = 0.693147180559945309f;

// One CTA per row r = (b*G + a)*N + n.
template <typename E>
__global__ void __launch_bounds__(kRowThreads, 8) la_rows_kernel(const Params p) {
  using X = Elem<E>;
  constexpr int PV = X::kPerVec;
  constexpr int U = 4;  // vectors in flight per thread
  const int tid = threadIdx.x;
  const int G = p.G, N = p.N;
  const int64_t V = p.V;
  const int64_t r = blockIdx.x;
  const int n = (int)(r % N);
  const int64_t ba = r / N;  // b*G + a
  const int64_t b = ba / G;
  const E* row = static_cast<const E*>(p.logits) + r * V;

  // The logit of candidate k's token at this position (k < G), for the walk.
  // An id outside [0, V) is not read; the walk rejects that sequence.
  if (n < N - 1 && tid < G) {
    const int32_t t = p.cand[(b * G + tid) * (N - 1) + n];
    const float z = (t >= 0 && (int64_t)t < V) ? X::load(row + t) * p.c : 0.f;
    p.gath[(ba * (N - 1) + n) * G + tid] = z;
  }

  // The row: a head up to the first 16-byte boundary, whole vectors, a tail.
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
  // The walk may be scheduled now; it waits for this grid to complete.
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

// One CTA per sequence b.
template <typename E>
__global__ void __launch_bounds__(kWalkThreads, 1) la_walk_kernel(const Params p) {
  using X = Elem<E>;
  __shared__ float2 st[kMaxRowsPerSeq];     // the sequence's row normalisers, row a*N + n
  __shared__ float gz[kMaxGather];          // gathered l*c, at (a*(N-1) + n)*G + k
  __shared__ int32_t cs[kMaxRowsPerSeq];    // candidate tokens, at k*(N-1) + n
  __shared__ float us[kMaxRowsPerSeq + 1];  // the uniforms
  __shared__ int32_t xs[kMaxG];             // candidate tokens at the stopping position
  __shared__ int32_t excl[kMaxG];           // distinct rejected tokens there, ascending
  __shared__ float wtot[kWalkWarps];        // inclusive scan of per-warp sums
  __shared__ int sh_j, sh_lead, sh_nex, sh_cross, sh_lastpos, sh_tok;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, N = p.N;
  const int R = G * N, NC = G * (N - 1), NU = NC + 1, NG = G * NC;
  const int64_t V = p.V;
  const int64_t b = blockIdx.x;

  // Inputs first (they do not depend on the row kernel), then its results.
  int bad = 0;
  for (int i = tid; i < NC; i += kWalkThreads) {
    const int32_t t = p.cand[b * NC + i];
    cs[i] = t;
    bad |= (t < 0 || (int64_t)t >= V);
  }
  for (int i = tid; i < NU; i += kWalkThreads) {
    const float u = p.uniforms[b * NU + i];
    us[i] = u;
    bad |= !(u >= 0.f && u < 1.f);
  }
  grid_dependency_sync(false);
  for (int i = tid; i < R; i += kWalkThreads) {
    const float2 v = p.rowstat[b * R + i];
    st[i] = v;
    bad |= !(v.x > -INFINITY && v.x < INFINITY);  // a NaN, a +inf, or a row of -inf only
  }
  for (int i = tid; i < NG; i += kWalkThreads) gz[i] = p.gath[b * NG + i];
  if (__syncthreads_or(bad)) {
    for (int i = tid; i < N; i += kWalkThreads) p.out_tokens[b * N + i] = -1;
    if (tid == 0) {
      p.out_accept_len[b] = -1;
      if (p.out_best) p.out_best[b] = -1;
      atomicOr(p.ctl + 3, kStatusInput);
    }
    return;
  }

  // The walk: lane k holds candidate k. Every branch below is warp-uniform.
  if (warp == 0) {
    const bool mine = lane < G;
    bool alive = mine;
    int lead = 0, j = N - 1;
    uint32_t rej = 0u;   // candidates rejected at the current position
    int32_t xstop = -1;  // this lane's token at the stopping position
    for (int n = 0; n < N - 1; ++n) {
      const float2 ms = st[lead * N + n];
      const int32_t x = mine ? cs[lane * (N - 1) + n] : -1;
      const float w = mine ? ex2(gz[(lead * (N - 1) + n) * G + lane] - ms.x) : 0.f;
      const uint32_t live = __ballot_sync(0xffffffffu, alive);
      float gone = 0.f;  // mass of the distinct tokens rejected so far at n
      int acc = -1;
      rej = 0u;
      for (int k = 0; k < G; ++k) {
        if (!((live >> k) & 1u)) continue;
        const int32_t xk = __shfl_sync(0xffffffffu, x, k);
        const float wk = __shfl_sync(0xffffffffu, w, k);
        // A token rejected before has probability 0 now.
        const bool seen = __ballot_sync(0xffffffffu, ((rej >> lane) & 1u) && x == xk) != 0u;
        float alpha = 0.f;
        if (!seen && wk > 0.f) {
          const float den = ms.y - gone;
          alpha = den <= wk ? 1.f : wk / den;
        }
        if (us[n * G + k] < alpha) {
          acc = k;
          break;
        }
        if (!seen) gone += wk;
        rej |= 1u << k;
      }
      if (acc < 0) {
        j = n;
        xstop = x;
        break;
      }
      const int32_t xa = __shfl_sync(0xffffffffu, x, acc);
      alive = alive && x == xa;
      lead = acc;
    }
    if (mine) xs[lane] = xstop;
    __syncwarp();
    if (lane == 0) {
      int ne = 0;
      if (j < N - 1) {
        for (int k = 0; k < G; ++k) {
          if (!((rej >> k) & 1u)) continue;
          const int32_t t = xs[k];
          bool dup = false;
          for (int i = 0; i < ne; ++i) dup |= excl[i] == t;
          if (dup) continue;
          int pos = ne++;
          while (pos > 0 && excl[pos - 1] > t) {
            excl[pos] = excl[pos - 1];
            --pos;
          }
          excl[pos] = t;
        }
      }
      sh_j = j;
      sh_lead = lead;
      sh_nex = ne;
      sh_tok = (int)(V - 1);
    }
  }
  __syncthreads();

  // The draw at position j from the owner's row: weights 2^(l*c - M), zero at
  // the rejected tokens. If those held all the mass (rounding only), the
  // draw falls back to the whole row.
  const int j = sh_j, lead = sh_lead;
  const float M = st[lead * N + j].x;
  const float target_u = us[NC];
  const E* row = static_cast<const E*>(p.logits) + ((b * G + lead) * N + j) * V;
  const int64_t CH = (V + kWalkThreads - 1) / kWalkThreads;
  const int64_t lo = (int64_t)tid * CH < V ? (int64_t)tid * CH : V;
  const int64_t hi = lo + CH < V ? lo + CH : V;
  int nex = sh_nex;
  for (int attempt = 0; attempt < 2; ++attempt) {
    int e = 0;
    while (e < nex && excl[e] < lo) ++e;
    int64_t nx = e < nex ? excl[e] : INT64_MAX;
    float s = 0.f;
#pragma unroll 4
    for (int64_t v = lo; v < hi; ++v) {
      float w = ex2(X::load(row + v) * p.c - M);
      if (v == nx) {
        w = 0.f;
        ++e;
        nx = e < nex ? excl[e] : INT64_MAX;
      }
      s += w;
    }
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
    if (!(Z > 0.f) && attempt == 0 && nex > 0) {
      nex = 0;
      __syncthreads();  // every thread has read wtot before it is rewritten
      continue;
    }
    // The chunk holding the crossing: the first one whose inclusive sum
    // passes u*Z. With none (rounding at u near 1), the last positive weight.
    const float target = target_u * Z;
    if (s > 0.f && incl > target) atomicMin(&sh_cross, tid);
    if (s > 0.f) atomicMax(&sh_lastpos, tid);
    __syncthreads();
    const int cross = sh_cross;
    const int owner = cross != INT_MAX ? cross : sh_lastpos;
    if (tid == owner) {
      float C = incl - s;  // the sum before this chunk
      int64_t tok = -1, last = -1;
      e = 0;
      while (e < nex && excl[e] < lo) ++e;
      nx = e < nex ? excl[e] : INT64_MAX;
      for (int64_t v = lo; v < hi; ++v) {
        float w = ex2(X::load(row + v) * p.c - M);
        if (v == nx) {
          w = 0.f;
          ++e;
          nx = e < nex ? excl[e] : INT64_MAX;
        }
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

template <typename E>
cudaError_t launch_t(const Params& p, cudaStream_t stream) {
  // The row kernel is an ordinary launch: it must not start before the
  // previous call on this stream has finished reading the scratch it writes.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.G * p.N));
  cfg.blockDim = dim3(kRowThreads);
  cfg.stream = stream;
  cudaError_t e = cudaLaunchKernelEx(&cfg, la_rows_kernel<E>, p);
  if (e != cudaSuccess) return e;
  // The walk may be scheduled while the row kernel finishes; it waits for it
  // (griddepcontrol.wait) before reading the row kernel's results.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)p.B);
  cfg.blockDim = dim3(kWalkThreads);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, la_walk_kernel<E>, p);
}

}  // namespace

cudaError_t launch(const Params& p, int dtype, cudaStream_t stream) {
  return dtype == 1 ? launch_t<uint16_t>(p, stream) : launch_t<float>(p, stream);
}

}  // namespace la
}  // namespace sv
