// sv_decide.cu — the decision and draw of the two-kernel sampling verify
// (sm_103a). One thread-block cluster of D CTAs per sequence b.
//
// Every CTA of the cluster combines the row pass's chunk partials into the
// normalisers of the sequence's 2K+1 rows, gathers the logits of the draft
// tokens and runs the accept scan ("Speculative Decoding —— LLM推理优化技术
// （一）" §2.1-2.3; kwkr.cn "投机解码" §3.1): alpha_i = min(1, p_i(x_i) /
// q_i(x_i)), accept while u_i < alpha_i. All CTAs reach the same j (same
// inputs, same arithmetic). The draw then splits the row into cells of 256
// elements, the cluster's ranks taking contiguous runs of cells:
//
//  the draw — fp32 weights w = max(0, p_j - q_j) after a rejection, or the
//    unnormalised p_K for the bonus; per-cell sums; the ranks' totals are
//    exchanged through distributed shared memory; the rank whose run holds
//    u_K * Z finds the crossing cell and walks it. The token stands when u_K*Z
//    is at least 1e-7 * Z from both edges of the token's CDF interval;
//    otherwise (and for a residual of zero mass, or a draw past the last
//    partial sum) the draw is appended to the refine kernel's list, which
//    redoes it in double-float arithmetic (sv_refine.cu).
//
// The selected token is the smallest t with sum_{v<=t} w_v > u_K * Z (the
// ascending-vocabulary inverse CDF); if rounding leaves u_K * Z at or past the
// last partial sum, the largest t with w_t > 0; a residual of zero mass draws
// from p_j ("Speculative Decoding" §4).
#include <climits>
#include <mutex>
#include <set>
#include <utility>

#include "sv_device.cuh"
#include "sv_df.cuh"
#include "sv_refine.h"
#include "sv_v2.h"

namespace sv {
namespace v2 {
namespace {

constexpr float kLn2 = 0.693147180559945309f;

__device__ __forceinline__ int nwarps() { return (int)(blockDim.x >> 5); }

// -------------------------------------------------------------- elements ---
template <typename E>
struct Elem;
template <>
struct Elem<float> {
  __device__ static float load(const char* row, int64_t e) { return __ldg(reinterpret_cast<const float*>(row) + e); }
  // 8 elements from e (e + 8 <= V and 16-byte aligned).
  __device__ static void load8v(const char* row, int64_t e, float* x) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(row + e * 4));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(row + e * 4) + 1);
    x[0] = __uint_as_float(a.x);
    x[1] = __uint_as_float(a.y);
    x[2] = __uint_as_float(a.z);
    x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b.x);
    x[5] = __uint_as_float(b.y);
    x[6] = __uint_as_float(b.z);
    x[7] = __uint_as_float(b.w);
  }
};
template <>
struct Elem<uint16_t> {
  __device__ static float load(const char* row, int64_t e) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row) + e)) << 16);
  }
  __device__ static void load8v(const char* row, int64_t e, float* x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + e * 2));
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

// A draw row as this CTA sees it: elements [s0, s1) (the 16-byte aligned
// part of its slice) from a copy in shared memory at `sm`, the rest from
// global memory at `g`.
struct RowView {
  const char* g;
  const char* sm;
  int64_t s0, s1;
};

template <typename E>
__device__ __forceinline__ float view_load(const RowView& r, int64_t e) {
  if (e >= r.s0 && e < r.s1) {
    const char* a = r.sm + (e - r.s0) * (int64_t)sizeof(E);
    return sizeof(E) == 2 ? __uint_as_float((uint32_t)(*reinterpret_cast<const unsigned short*>(a)) << 16)
                          : *reinterpret_cast<const float*>(a);
  }
  return Elem<E>::load(r.g, e);
}

// Elements e .. e+7 of a row; -inf past V.
template <typename E>
__device__ __forceinline__ void load8(const RowView& r, int64_t e, int64_t V, float* x) {
  if (e >= r.s0 && e + 8 <= r.s1 && ((((e - r.s0) * (int64_t)sizeof(E)) & 15) == 0)) {
    const char* a = r.sm + (e - r.s0) * (int64_t)sizeof(E);
    if (sizeof(E) == 2) {
      const uint4 v = *reinterpret_cast<const uint4*>(a);
      x[0] = bf_lo(v.x);
      x[1] = bf_hi(v.x);
      x[2] = bf_lo(v.y);
      x[3] = bf_hi(v.y);
      x[4] = bf_lo(v.z);
      x[5] = bf_hi(v.z);
      x[6] = bf_lo(v.w);
      x[7] = bf_hi(v.w);
    } else {
      const uint4 v0 = reinterpret_cast<const uint4*>(a)[0];
      const uint4 v1 = reinterpret_cast<const uint4*>(a)[1];
      x[0] = __uint_as_float(v0.x);
      x[1] = __uint_as_float(v0.y);
      x[2] = __uint_as_float(v0.z);
      x[3] = __uint_as_float(v0.w);
      x[4] = __uint_as_float(v1.x);
      x[5] = __uint_as_float(v1.y);
      x[6] = __uint_as_float(v1.z);
      x[7] = __uint_as_float(v1.w);
    }
  } else if (e + 8 <= V && (e + 8 <= r.s0 || e >= r.s1) &&
             ((reinterpret_cast<uintptr_t>(r.g + e * (int64_t)sizeof(E)) & 15u) == 0)) {
    Elem<E>::load8v(r.g, e, x);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = e + k < V ? view_load<E>(r, e + k) : -INFINITY;
  }
}

// ---------------------------------------------------------------- weights ---
// fp32 weights of the fast draw. Residual: max(0, 2^(l_p c - Mc_p)/s_p -
// 2^(l_q c - Mc_q)/s_q); bonus (or a residual of zero mass): 2^(l_p c - Mc_p).
// With top-p, an element outside a row's nucleus (l < tp, resp. tq) has
// weight 0 in that row.
struct FastW {
  float c, mcp, ip, mcq, iq, tp, tq;
  bool resid;
  // (the cut selects the exponent, -inf outside the nucleus: no branch)
  __device__ __forceinline__ float w(float lp, float lq) const {
    const float ep = ex2(lp >= tp ? fmaf(lp, c, -mcp) : -INFINITY);
    if (!resid) return ep;
    const float eq = ex2(lq >= tq ? fmaf(lq, c, -mcq) : -INFINITY);
    return fmaxf(0.f, fmaf(ep, ip, -eq * iq));
  }
};

__device__ __forceinline__ df warp_incl_scan_df(df v, int lane) {
#pragma unroll 1  // once per CTA, cold in the instruction cache
  for (int o = 1; o < 32; o <<= 1) {
    df t;
    t.h = __shfl_up_sync(0xffffffffu, v.h, o);
    t.l = __shfl_up_sync(0xffffffffu, v.l, o);
    if (lane >= o) v = df_add(v, t);
  }
  return v;
}

// Per-CTA state of the decide kernel. The arrays sized by K and by the
// cells per rank live in dynamic shared memory (see Layout); this part is
// fixed.
struct Smem {
  // exchanged through distributed shared memory
  float x_tot_h, x_tot_l;   // this rank's total weight (double-float)
  int res_tok, res_precise; // on rank 0: the token and whether to redo the draw
  int bad, j;
  uint64_t slice_bar;       // the slice copies of the draw rows landed
};

// Dynamic shared memory, in floats: rM[R] rS[R] rT[R] gz[2K] us[K+1] xs[K]
// cs_h cs_l cp_h cp_l [cpr each], then (16-byte aligned) the copies of this
// CTA's slice of the two draw rows. rS is the nucleus mass (the whole row's
// sum without top-p), rT the smallest logit in the nucleus (-inf: all).
struct Layout {
  float *rM, *rS, *rT, *gz, *us;
  int32_t* xs;
  float *cs_h, *cs_l, *cp_h, *cp_l;
  char* slice;
  __device__ Layout(float* d, int K, int R, int cpr) {
    rM = d;
    rS = rM + R;
    rT = rS + R;
    gz = rT + R;
    us = gz + 2 * K;
    xs = reinterpret_cast<int32_t*>(us + K + 1);
    cs_h = reinterpret_cast<float*>(xs + K);
    cs_l = cs_h + cpr;
    cp_h = cs_l + cpr;
    cp_l = cp_h + cpr;
    slice = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(cp_l + cpr) + 15) & ~uintptr_t(15));
  }
};

// Floats of the Layout arrays (the slice area follows them).
__host__ __device__ inline size_t layout_floats(int K, int R, int cpr) {
  return (size_t)3 * R + 2 * (size_t)K + (K + 1) + K + 4 * (size_t)cpr;
}

// What the draw works on: the rows, this rank's cells, the uniform.
struct DrawCtx {
  RowView prow;
  RowView qrow;
  int64_t V;
  int cb, ce, D;
  uint32_t rank;
  float u;
  bool resid;
};

// Cell sums of cells [cb, ce) of this rank (fast draw), into cs_h.
template <typename E>
__device__ __forceinline__ void fast_cells(const FastW& fw, const DrawCtx& x, const Layout& L, int warp, int lane) {
  for (int cell = x.cb + warp; cell < x.ce; cell += nwarps()) {
    const int64_t e = (int64_t)cell * kCellElems + lane * 8;
    float lp[8], lq[8];
    load8<E>(x.prow, e, x.V, lp);
    if (fw.resid) {
      // the draft's logits matter only where the target's lie in its
      // nucleus (a weight is 0 where p' is): with top-p most vectors need
      // none; without it (tp = -inf) every vector does
      bool need = false;
#pragma unroll
      for (int k = 0; k < 8; ++k) need |= lp[k] >= fw.tp;
      if (need) {
        load8<E>(x.qrow, e, x.V, lq);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) lq[k] = -INFINITY;
      }
    }
    float w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = fw.w(lp[k], fw.resid ? lq[k] : 0.f);
    float s = ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
    s = warp_sum(s);
    if (lane == 0) L.cs_h[cell - x.cb] = s;
  }
}

template <typename E>
__global__ void __launch_bounds__(kDecideThreads, 4) decide_kernel(const Params p) {
  __shared__ Smem sm;
  extern __shared__ float dyn[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const int D = p.D;
  const int64_t b = blockIdx.x / D;
  const int K = p.K, R = p.R;
  const int64_t V = p.V;
  const float c = p.c;
  const Layout L(dyn, K, R, p.cpr);
  if (tid == 0) {
    mbar_init(&sm.slice_bar, 1);
    fence_mbar_init();
  }
  grid_dependency_sync(true);

  // ---- inputs and row normalisers ------------------------------------------
  int bad = 0;
  for (int i = tid; i < K; i += (int)blockDim.x) {
    const int32_t t = p.tokens[b * K + i];
    L.xs[i] = t;
    bad |= (t < 0 || (int64_t)t >= V);
  }
  for (int i = tid; i <= K; i += (int)blockDim.x) {
    const float u = p.uniforms[b * (K + 1) + i];
    L.us[i] = u;
    bad |= !(u >= 0.f && u < 1.f);
  }
  for (int i = tid; i < R && p.topp; i += (int)blockDim.x) {
    const float4 r = p.rstat[b * R + i];
    const uint32_t tau = __float_as_uint(r.w);
    L.rM[i] = r.x;
    L.rS[i] = r.z;
    // the smallest bf16 value whose key is >= tau (tau = 0: every value)
    L.rT[i] = tau <= key_bf16(-INFINITY) ? -INFINITY : val_bf16(tau);
    bad |= !(r.x > -INFINITY && r.x < INFINITY && r.z > 0.f);
  }
  for (int i = tid; i < R && !p.topp; i += (int)blockDim.x) {
    const float2* pp = p.part + (b * R + i) * p.NCH;
    float m = pp[0].x, s = pp[0].y;
    for (int k = 1; k < p.NCH; ++k) {
      const float2 q = pp[k];
      const float mn = fmax_nan(m, q.x);
      if (mn > -INFINITY && mn < INFINITY) {
        const float r = __fmul_rn(mn, c);
        float t = 0.f;
        if (m > -INFINITY) t += s * ex2(__fsub_rn(__fmul_rn(m, c), r));
        if (q.x > -INFINITY) t += q.y * ex2(__fsub_rn(__fmul_rn(q.x, c), r));
        s = t;
      }
      m = mn;
    }
    L.rM[i] = m;
    L.rS[i] = s;
    L.rT[i] = -INFINITY;
    bad |= !(m > -INFINITY && m < INFINITY && s > 0.f);
  }
  // the logits of the draft tokens, recorded by the row pass
  for (int i = tid; i < 2 * K; i += (int)blockDim.x) L.gz[i] = p.gz[b * (2 * K) + i];
  bad = __syncthreads_or(bad);

  // ---- accept scan (warp 0) and the row statistics (rank 0) ----------------
  if (warp == 0) {
    int j = K;
    if (!bad) {
      for (int i0 = 0; i0 < K; i0 += 32) {
        const int i = i0 + lane;
        bool rej = false;
        if (i < K) {
          // alpha = min(1, p(x)/q(x)); p(x) = 0 gives 0 and q(x) = 0 < p(x)
          // gives 1 (the pages' p/(q+eps)). Ratios of weights that would
          // underflow fp32 are taken in the log2 domain instead.
          const float lp = L.gz[i], lq = L.gz[K + i];
          float alpha;
          if (!(lp > -INFINITY && lp >= L.rT[i])) {  // p(x) = 0
            alpha = 0.f;
          } else if (!(lq > -INFINITY && lq >= L.rT[K + 1 + i])) {  // q(x) = 0
            alpha = 1.f;
          } else {
            const float xp = fmaf(lp, c, -__fmul_rn(L.rM[i], c));
            const float xq = fmaf(lq, c, -__fmul_rn(L.rM[K + 1 + i], c));
            if (xp > -120.f && xq > -120.f) {
              const float pw = ex2(xp) / L.rS[i];
              const float qw = ex2(xq) / L.rS[K + 1 + i];
              alpha = fminf(1.f, pw / qw);
            } else {
              alpha = ex2(fminf(0.f, (xp - lg2(L.rS[i])) - (xq - lg2(L.rS[K + 1 + i]))));
            }
          }
          rej = !(L.us[i] < alpha);
        }
        const uint32_t m = __ballot_sync(0xffffffffu, rej);
        if (m) {
          j = i0 + __ffs(m) - 1;
          break;
        }
      }
    }
    if (lane == 0) {
      sm.j = j;
      sm.bad = bad;
      sm.res_precise = 0;
    }
  }
  if (rank == 0 && p.out_row_stats && !bad) {
    for (int i = tid; i < R; i += (int)blockDim.x) {
      const float mc = __fmul_rn(L.rM[i], c);
      float4 o;
      o.x = L.rM[i] / p.T;
      if (p.topp) {
        const float4 r = p.rstat[b * R + i];
        o.y = (mc + lg2(r.y)) * kLn2;
        o.z = r.z / r.y;
        o.w = val_bf16(__float_as_uint(r.w));
      } else {
        o.y = (mc + lg2(L.rS[i])) * kLn2;
        o.z = 1.f;
        o.w = -INFINITY;
      }
      reinterpret_cast<float4*>(p.out_row_stats)[b * R + i] = o;
    }
  }
  __syncthreads();
  const int j = sm.j;

  // ---- the fast draw ----------------------------------------------------------
  DrawCtx x;
  x.resid = j < K;
  x.V = V;
  x.cb = (int)rank * p.cpr;
  x.ce = min(x.cb + p.cpr, p.ncell);
  x.D = D;
  x.rank = rank;
  x.u = bad ? 0.f : L.us[K];
  const int cb = x.cb, ce = x.ce;
  x.prow.g = p.target + ((b * (K + 1) + j) * V) * p.esz;
  x.qrow.g = x.resid ? p.draft + ((b * K + j) * V) * p.esz : x.prow.g;
  x.prow.sm = x.qrow.sm = L.slice;
  x.prow.s0 = x.prow.s1 = x.qrow.s0 = x.qrow.s1 = 0;
  // the rows whose slices are copied: the target's, and the draft's after a
  // rejection without top-p (with top-p the draft's few logits inside the
  // target's nucleus are read directly)
  const int ncopy = x.resid && !p.topp ? 2 : 1;
  if (p.prefetch && !bad && ce > cb) {
    // This CTA's slice of the draw rows, HBM/L2 -> shared memory: the
    // 16-byte aligned part of [cb*256, ce*256) of each row, one bulk copy
    // each; the few elements outside it are read directly.
    const int64_t e_lo = (int64_t)cb * kCellElems;
    const int64_t e_hi = min((int64_t)ce * kCellElems, V);
    const uint32_t cap = (uint32_t)(p.cpr * kCellElems * p.esz);
    RowView* rv[2] = {&x.prow, &x.qrow};
    uint32_t total = 0;
    for (int k = 0; k < ncopy; ++k) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(rv[k]->g + e_lo * p.esz);
      const uintptr_t a1 = reinterpret_cast<uintptr_t>(rv[k]->g + e_hi * p.esz);
      const uintptr_t A = (a0 + 15) & ~uintptr_t(15), Z = a1 & ~uintptr_t(15);
      if (A < Z) {
        rv[k]->s0 = e_lo + (int64_t)((A - a0) / p.esz);
        rv[k]->s1 = rv[k]->s0 + (int64_t)((Z - A) / p.esz);
        rv[k]->sm = L.slice + k * (size_t)cap;
        total += (uint32_t)(Z - A);
      }
    }
    if (tid == 0) {
      mbar_arrive_expect_tx(&sm.slice_bar, total);
      for (int k = 0; k < ncopy; ++k)
        if (rv[k]->s1 > rv[k]->s0)
          bulk_g2s(const_cast<char*>(rv[k]->sm), rv[k]->g + rv[k]->s0 * p.esz,
                   (uint32_t)((rv[k]->s1 - rv[k]->s0) * p.esz), &sm.slice_bar);
    }
    if (!__syncthreads_and(mbar_wait(&sm.slice_bar, 0))) {
      // a copy did not land in time: read the rows from global memory
      x.prow.s0 = x.prow.s1 = x.qrow.s0 = x.qrow.s1 = 0;
      if (tid == 0) atomicOr(p.ctl + 3, kStatusTimeout);
    }
  }
  if (!x.resid) x.qrow = x.prow;

  FastW fw;
  fw.c = c;
  fw.mcp = __fmul_rn(L.rM[j], c);
  fw.ip = 1.f / L.rS[j];
  fw.mcq = x.resid ? __fmul_rn(L.rM[K + 1 + j], c) : 0.f;
  fw.iq = x.resid ? 1.f / L.rS[K + 1 + j] : 0.f;
  fw.tp = L.rT[j];
  fw.tq = x.resid ? L.rT[K + 1 + j] : -INFINITY;
  fw.resid = x.resid;
  if (!bad) fast_cells<E>(fw, x, L, warp, lane);
  __syncthreads();
  if (warp == 0) {
    // inclusive prefix of this rank's cells and its total, in double-float:
    // the running sums reach the size of Z, where fp32 would round at ~6e-8*Z
    df carry{0.f, 0.f};
    for (int c0 = 0; c0 < ce - cb; c0 += 32) {
      const bool in = c0 + lane < ce - cb;
      const df v{in ? L.cs_h[c0 + lane] : 0.f, 0.f};
      const df incl = df_add(carry, warp_incl_scan_df(v, lane));
      if (in) {
        L.cp_h[c0 + lane] = incl.h;
        L.cp_l[c0 + lane] = incl.l;
      }
      carry.h = __shfl_sync(0xffffffffu, incl.h, 31);
      carry.l = __shfl_sync(0xffffffffu, incl.l, 31);
    }
    if (lane == 0) {
      sm.x_tot_h = carry.h;
      sm.x_tot_l = carry.l;
    }
  }
  __syncthreads();
  cluster_sync();  // (1) rank totals visible
  if (warp == 0 && !bad) {
    // The ranks' running sums, in rank order, identical in every CTA: lane q
    // reads rank q's total, one warp scan gives every prefix at once.
    const df mine = lane < D ? df{dsmem_ld_f32(&sm.x_tot_h, (uint32_t)lane), dsmem_ld_f32(&sm.x_tot_l, (uint32_t)lane)}
                             : df{0.f, 0.f};
    const df incl = warp_incl_scan_df(mine, lane);
    const df Z{__shfl_sync(0xffffffffu, incl.h, 31), __shfl_sync(0xffffffffu, incl.l, 31)};
    const df target = df_mul_f(Z, x.u);
    const df excl = df_sub(incl, mine);
    const df Pme{__shfl_sync(0xffffffffu, excl.h, (int)rank), __shfl_sync(0xffffffffu, excl.l, (int)rank)};
    const uint32_t om = __ballot_sync(0xffffffffu, lane < D && df_gt(incl, target));
    const int owner = om ? __ffs(om) - 1 : -1;
    const bool need_precise_all = !df_pos(Z) || owner < 0;
    if ((int)rank == owner && !need_precise_all) {
      // the crossing cell: the first whose inclusive sum exceeds the target
      int cc = -1;
      for (int c0 = 0; c0 < ce - cb && cc < 0; c0 += 32) {
        const bool hit =
            c0 + lane < ce - cb && df_gt(df_add(Pme, df{L.cp_h[c0 + lane], L.cp_l[c0 + lane]}), target);
        const uint32_t m = __ballot_sync(0xffffffffu, hit);
        if (m) cc = c0 + __ffs(m) - 1;
      }
      int tok = -1;
      bool precise = true;
      if (cc >= 0) {
        // what is left of the target inside the crossing cell, exactly enough
        // in fp32 (it is below the cell's sum)
        const df base = cc > 0 ? df_add(Pme, df{L.cp_h[cc - 1], L.cp_l[cc - 1]}) : Pme;
        const df rem = df_sub(target, base);
        const float Rm = rem.h + rem.l;
        const int64_t e = (int64_t)(cb + cc) * kCellElems + lane * 8;
        float lp[8], lq[8], w[8];
        load8<E>(x.prow, e, V, lp);
        if (fw.resid) load8<E>(x.qrow, e, V, lq);
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = fw.w(lp[k], fw.resid ? lq[k] : 0.f);
        const float s = ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
        const float incl = warp_incl_scan(s, lane);
        const uint32_t m = __ballot_sync(0xffffffffu, incl > Rm);
        int found = 0;
        float margin = 0.f;
        if (m && lane == __ffs(m) - 1) {
          float C = incl - s;
          for (int k = 0; k < 8; ++k) {
            const float prev = C;
            C = C + w[k];
            if (C > Rm) {
              tok = (int)(e + k);
              margin = fminf(C - Rm, Rm - prev);
              found = 1;
              break;
            }
          }
        }
        const uint32_t fm = __ballot_sync(0xffffffffu, found);
        if (fm) {
          const int src = __ffs(fm) - 1;
          tok = __shfl_sync(0xffffffffu, tok, src);
          margin = __shfl_sync(0xffffffffu, margin, src);
          precise = !(margin >= rf::kRefineMargin * Z.h);
        }
      }
      if (lane == 0) {
        dsmem_st_s32(&sm.res_tok, 0, tok);
        if (precise) dsmem_st_s32(&sm.res_precise, 0, 1);
      }
    }
    if (rank == 0 && lane == 0 && need_precise_all) sm.res_precise = 1;
  }
  cluster_sync();  // (2) the fast draw's verdict is on rank 0
  if (rank == 0 && tid == 0 && !bad && sm.res_precise) {
    // too close to a CDF edge for fp32 (or a residual of zero mass, or
    // rounding in the walk): the refine kernel redoes this draw
    rf::Rec r{};
    r.b = (int32_t)b;
    r.j = j;
    r.resid = x.resid ? 1 : 0;
    r.mp = L.rM[j];
    r.mq = x.resid ? L.rM[K + 1 + j] : 0.f;
    r.taup = L.rT[j];
    r.tauq = x.resid ? L.rT[K + 1 + j] : -INFINITY;
    r.u = x.u;
    rf::flag(p.rf_ctl, p.rf_recs, p.B, r);
  }

  // ---- outputs (rank 0) ------------------------------------------------------
  if (rank == 0) {
    if (bad) {
      for (int i = tid; i <= K; i += (int)blockDim.x) p.out_tokens[b * (K + 1) + i] = -1;
      if (tid == 0) {
        p.out_accept_len[b] = -1;
        atomicOr(p.ctl + 3, kStatusInput);
      }
    } else {
      const int tok = sm.res_tok;
      for (int i = tid; i <= K; i += (int)blockDim.x)
        p.out_tokens[b * (K + 1) + i] = i < j ? L.xs[i] : (i == j ? tok : -1);
      if (tid == 0) p.out_accept_len[b] = j;
    }
  }
  cluster_sync();  // no CTA leaves while another may still read its shared memory
}

}  // namespace

size_t decide_smem_bytes(const Params& p) {
  size_t b = sizeof(float) * layout_floats(p.K, p.R, p.cpr) + 16;
  if (p.prefetch) b += (p.topp ? 1 : 2) * (size_t)p.cpr * kCellElems * p.esz;
  return b;
}

cudaError_t launch_decide(const Params& p, int dtype, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.D));
  cfg.blockDim = dim3((unsigned)p.dthreads);
  cfg.dynamicSmemBytes = decide_smem_bytes(p);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.D;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const void* kf = dtype == 1 ? reinterpret_cast<const void*>(decide_kernel<uint16_t>)
                              : reinterpret_cast<const void*>(decide_kernel<float>);
  cudaError_t e = raise_smem_limit_v2(kf, cfg.dynamicSmemBytes);
  if (e != cudaSuccess) return e;
  e = dtype == 1 ? cudaLaunchKernelEx(&cfg, decide_kernel<uint16_t>, p)
                             : cudaLaunchKernelEx(&cfg, decide_kernel<float>, p);
  if (e != cudaSuccess) {  // without programmatic serialisation
    cudaGetLastError();
    cfg.numAttrs = 1;
    e = dtype == 1 ? cudaLaunchKernelEx(&cfg, decide_kernel<uint16_t>, p)
                   : cudaLaunchKernelEx(&cfg, decide_kernel<float>, p);
  }
  return e;
}

cudaError_t launch_rows(const Params& p, int dtype, cudaStream_t stream);

bool fits(int64_t K, int64_t V) {
  // within what portable clusters of 8 cover (larger clusters only spread the work thinner)
  return K >= 1 && K <= kMaxK && V >= 2 && V <= (int64_t)8 * kMaxCellsPerCta * kCellElems;
}

bool fits_topp(int64_t K, int64_t V, int esz) { return fits(K, V) && esz == 2 && V % 8 == 0; }

void plan(Params& p, int sms) {
  const int64_t rowbytes = p.V * p.esz;
  const int64_t rows = p.B * p.R;
  if (p.topp) {
    // whole rows, one CTA each at a time (persistent CTAs, see below)
    p.NCH = 1;
    p.CE = p.V;
    p.RPI = 1;
  } else if (rowbytes <= kChunkBytes / 2) {
    // short rows: groups of whole rows, about one chunk's worth each
    p.NCH = 1;
    p.CE = p.V;
    int64_t rpi = kChunkBytes / (rowbytes + 16);
    if (rpi > kMaxRowsPerItem) rpi = kMaxRowsPerItem;
    // keep a few items per CTA slot when the call has the rows for it
    const int64_t want = (int64_t)sms * 3 * 4;
    if (rows / rpi < want) rpi = rows / want;
    if (rpi < 1) rpi = 1;
    p.RPI = (int)rpi;
  } else {
    const int64_t per = p.esz == 2 ? 8 : 4;  // elements per 16 bytes
    int64_t nch = (rowbytes + kChunkBytes - 1) / kChunkBytes;
    if (nch > kMaxChunks) nch = kMaxChunks;
    int64_t ce = (p.V + nch - 1) / nch;
    ce = (ce + per - 1) / per * per;
    p.CE = ce;
    p.NCH = (int)((p.V + ce - 1) / ce);
    p.RPI = 1;
  }
  p.items = (rows + p.RPI - 1) / p.RPI * p.NCH;
  p.row_slot = (uint32_t)((rowbytes + 15) / 16 * 16 + 16);
  p.stage_bytes = p.RPI == 1 ? (uint32_t)((p.CE * p.esz + 31) / 16 * 16) : (uint32_t)p.RPI * p.row_slot;
  // persistent CTAs: as many as the stages' shared memory lets reside, up to
  // four per SM
  int per_sm = (int)((200 * 1024) / (2 * (int64_t)p.stage_bytes));
  per_sm = per_sm < 1 ? 1 : (per_sm > 4 ? 4 : per_sm);
  p.rows_grid = (int64_t)sms * per_sm;
  if (p.topp) p.rows_grid = (int64_t)sms * 4;  // the top-p row pass: four CTAs per SM
  if (p.rows_grid > p.items) p.rows_grid = p.items;
  p.ncell = (int)((p.V + kCellElems - 1) / kCellElems);
  // about 32 cells per rank (one warp scan of its cell sums); with top-p,
  // where only the target row's slice is copied, about 80, so that the
  // clusters are smaller and more of them reside at once
  const int per_rank = p.topp ? 80 : 32;
  int d = (p.ncell + per_rank - 1) / per_rank;
  d = d < 1 ? 1 : (d > kMaxCluster ? kMaxCluster : d);
  // cluster sizes of 1, 2, 4, 8 or 16
  int dd = 1;
  while (dd < d) dd <<= 1;
  p.D = dd;
  p.cpr = (p.ncell + p.D - 1) / p.D;
  // threads: one warp per cell of the slice, 2 to 8 warps
  int w = p.cpr < 2 ? 2 : (p.cpr > 8 ? 8 : p.cpr);
  p.dthreads = w * 32;
  // the slice copies when the copied rows' slices fit 96 KB
  p.prefetch = (p.topp ? 1 : 2) * (int64_t)p.cpr * kCellElems * p.esz <= 96 * 1024 ? 1 : 0;
  for (int i = 0; i < 32; ++i) {
    const double v = exp2((double)i / 32.0);
    p.tab_hi[i] = (float)v;
    p.tab_lo[i] = (float)(v - (double)p.tab_hi[i]);
  }
  const double cd = 1.4426950408889634 / (double)p.T;
  p.c_hi = (float)cd;
  p.c_lo = (float)(cd - (double)p.c_hi);
}

cudaError_t raise_smem_limit_v2(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  // the most any call of this kernel may ask for on this device
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  (void)bytes;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - 1024);
  if (e != cudaSuccess) return e;
  // clusters of 16 (a non-portable size) for the decide kernel's long rows
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) done.insert({kernel, dev});
  return e;
}

size_t part_bytes(const Params& p) {
  const size_t b = p.topp ? (size_t)(p.B * p.R) * sizeof(float4) : (size_t)(p.B * p.R * p.NCH) * sizeof(float2);
  return (b + 255) / 256 * 256;
}
size_t scratch_bytes(const Params& p) { return part_bytes(p) + (size_t)p.B * 2 * p.K * sizeof(float); }

cudaError_t launch(const Params& p, int dtype, cudaStream_t stream) {
  cudaError_t e = launch_rows(p, dtype, stream);
  if (e != cudaSuccess) return e;
  return launch_decide(p, dtype, stream);
}

}  // namespace v2
}  // namespace sv
