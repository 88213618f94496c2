// sv_refine.cu — the refine kernel: sampling draws that an fp32 draw could not
// settle, redone in double-float arithmetic (sm_103a).
//
// The draw ("Speculative Decoding —— LLM推理优化技术（一）" §2.1-2.3, kwkr.cn
// "投机解码" §3.1, §3.4): after a rejection at j, the token is the smallest t
// with sum_{v<=t} w_v > u*Z for w = max(0, p'_j - q'_j) (p'_j itself if that
// is all zero, "Speculative Decoding" §4), else the bonus from p'_K; p' and q'
// are softmax(l/T), restricted to the nucleus {l >= tau} and renormalised
// with top-p. Here e_v = 2^((l_v - M)*log2(e)/T) is evaluated as a
// double-float (the difference l - M and its product with the double-float
// log2(e)/T carried exactly, 2^x by df_exp2), the normalisers S = sum of e
// over the nucleus in double-float, and the residual weights as
// max(0, e_p - (S_p/S_q) e_q), proportional to max(0, p' - q').
//
// One thread-block cluster of CL CTAs per flagged draw (CL up to 16); CTA r
// of the cluster owns elements [r*RL, (r+1)*RL) of the draw's rows. Per draw:
//  1. every CTA evaluates e_p (and e_q) over its range once, keeps the
//     double-float values in shared memory and sums them; the CTAs exchange
//     the sums through distributed shared memory, so that every CTA holds the
//     same S_p / S_q;
//  2. every CTA sums the weights of its range in chunks of 8m elements and
//     scans the chunk sums; the CTAs exchange their range totals, giving the
//     base of each range, Z and u*Z; the CTA whose range crosses u*Z finds
//     its thread whose chunks cross, and that thread walks them element by
//     element. A residual of zero mass repeats step 2 with w = e_p.
// Clusters take flagged draws in turn (draw f on cluster f mod clusters).
// Where the range is too long for the double-float values to stay in shared
// memory, step 2 evaluates them again from global memory.
#include <climits>
#include <map>
#include <mutex>
#include <tuple>

#include "sv_device.cuh"
#include "sv_df.cuh"
#include "sv_refine.h"

namespace sv {
namespace rf {
namespace {

constexpr int kWarps = kThreads / 32;
constexpr int kMaxChunks = 2048;  // chunk sums kept per CTA

template <typename E>
__device__ __forceinline__ float load_elem(const char* row, int64_t e) {
  if (sizeof(E) == 2)
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row) + e)) << 16);
  return __ldg(reinterpret_cast<const float*>(row) + e);
}

// The 8 elements of a group as stored words (bf16: one 16-byte vector, fp32:
// two), so that a loop over the elements can pick element k with selects
// instead of indexing a register array.
template <typename E>
struct Raw;
template <>
struct Raw<uint16_t> {
  uint4 a;
  __device__ __forceinline__ float at(int k) const {
    const uint32_t w = k < 4 ? (k < 2 ? a.x : a.y) : (k < 6 ? a.z : a.w);
    return __uint_as_float((k & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
};
template <>
struct Raw<float> {
  uint4 a, b;
  __device__ __forceinline__ float at(int k) const {
    const uint4& v = k < 4 ? a : b;
    const int j = k & 3;
    return __uint_as_float(j < 2 ? (j == 0 ? v.x : v.y) : (j == 2 ? v.z : v.w));
  }
};

// Elements e..e+7 of a row as stored words (-inf from hi on).
template <typename E>
__device__ __forceinline__ void load_raw(const char* row, int64_t e, int64_t hi, bool vec, Raw<E>& r) {
  if constexpr (sizeof(E) == 2) {
    if (vec && e + 8 <= hi) {
      r.a = __ldg(reinterpret_cast<const uint4*>(row + e * 2));
    } else {
      const unsigned short* s = reinterpret_cast<const unsigned short*>(row);
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t l0 = e + 2 * k < hi ? (uint32_t)__ldg(s + e + 2 * k) : 0xFF80u;
        const uint32_t l1 = e + 2 * k + 1 < hi ? (uint32_t)__ldg(s + e + 2 * k + 1) : 0xFF80u;
        w[k] = l0 | (l1 << 16);
      }
      r.a = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    if (vec && e + 8 <= hi) {
      r.a = __ldg(reinterpret_cast<const uint4*>(row + e * 4));
      r.b = __ldg(reinterpret_cast<const uint4*>(row + e * 4 + 16));
    } else {
      const float* s = reinterpret_cast<const float*>(row);
      uint32_t w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) w[k] = e + k < hi ? __float_as_uint(__ldg(s + e + k)) : 0xFF800000u;
      r.a = make_uint4(w[0], w[1], w[2], w[3]);
      r.b = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

struct Ctx {
  float mp, mq, taup, tauq;
  df rho;
  float c_hi, c_lo;
  const float* th;
  const float* tl;
  // e = 2^((l - M) c) in the nucleus {l >= tau}, else 0
  __device__ __forceinline__ df e(float l, float M, float tau) const {
    if (!(l >= tau)) return df{0.f, 0.f};
    const df d = two_sum(l, -M);
    const float xh = __fmul_rn(d.h, c_hi);
    const float xl = __fadd_rn(__fmaf_rn(d.h, c_hi, -xh), __fmaf_rn(d.h, c_lo, __fmul_rn(d.l, c_hi)));
    return df_exp2(xh, xl, th, tl);
  }
  // the residual weight from the two e values
  __device__ __forceinline__ df resid_w(df ep, df eq) const {
    const df r = df_sub(ep, df_mul(rho, eq));
    return df_pos(r) ? r : df{0.f, 0.f};
  }
};

__device__ __forceinline__ df shfl_xor_df(df v, int o) {
  return df{__shfl_xor_sync(0xffffffffu, v.h, o), __shfl_xor_sync(0xffffffffu, v.l, o)};
}
// (The shuffle loops of this file are not unrolled: the code after the
// element loops runs once per launch, cold in the instruction cache, where
// fewer distinct instructions matter more than the loop's few extra ones.)
__device__ __forceinline__ df warp_incl_scan_df(df v, int lane) {
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    df t;
    t.h = __shfl_up_sync(0xffffffffu, v.h, o);
    t.l = __shfl_up_sync(0xffffffffu, v.l, o);
    if (lane >= o) v = df_add(v, t);
  }
  return v;
}

// Shared state of a CTA besides the dynamic arrays.
struct Shared {
  float xs[2][4];                // exchange slots, read by the other CTAs of the cluster
  float wh[kWarps], wl[kWarps];  // per-warp partials
  float wh2[kWarps], wl2[kWarps];
  int wi[kWarps];
  float bh[4], bl[4];            // values broadcast to the CTA
  int bi[4];
  float sh[2], sl[2];            // block_sum2's results
  float th[32], tl[32];          // 2^(i/32) as double-floats
};

// Sums of two double-floats over the CTA (a fixed shuffle tree, the same in
// every CTA); every thread gets both.
__device__ __forceinline__ void block_sum2(df& a, df& b, Shared& s) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll 1
  for (int o = 16; o > 0; o >>= 1) {
    a = df_add(a, shfl_xor_df(a, o));
    b = df_add(b, shfl_xor_df(b, o));
  }
  if (lane == 0) {
    s.wh[warp] = a.h;
    s.wl[warp] = a.l;
    s.wh2[warp] = b.h;
    s.wl2[warp] = b.l;
  }
  __syncthreads();
  if (warp == 0) {
    df x = lane < kWarps ? df{s.wh[lane], s.wl[lane]} : df{0.f, 0.f};
    df y = lane < kWarps ? df{s.wh2[lane], s.wl2[lane]} : df{0.f, 0.f};
#pragma unroll 1
    for (int o = 16; o > 0; o >>= 1) {
      x = df_add(x, shfl_xor_df(x, o));
      y = df_add(y, shfl_xor_df(y, o));
    }
    if (lane == 0) {
      s.sh[0] = x.h;
      s.sl[0] = x.l;
      s.sh[1] = y.h;
      s.sl[1] = y.l;
    }
  }
  __syncthreads();
  a = df{s.sh[0], s.sl[0]};
  b = df{s.sh[1], s.sl[1]};
  __syncthreads();
}

// Draws f = cluster, cluster + clusters, ... of the flagged list.
template <typename E>
__global__ void __launch_bounds__(kThreads, 1) refine_kernel(const Params p) {
  extern __shared__ __align__(16) float dyn[];
  __shared__ Shared s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 32) {
    s.th[tid] = p.tab_hi[tid];
    s.tl[tid] = p.tab_lo[tid];
  }
  __syncthreads();
  grid_dependency_sync(true);
  uint32_t total = ld_acquire_gpu(&p.ctl[0]);
  if (total > (uint32_t)p.B) total = (uint32_t)p.B;
  if (total == 0) return;  // the same word for every CTA: nothing to redo, no cluster barrier taken
  if (blockIdx.x == 0 && tid == 0 && p.stats) atomicAdd(p.stats, total);
  const int CL = p.CL;
  const uint32_t rank = cluster_rank();
  const uint32_t clus = cluster_id_x(), nclus = cluster_count_x();
  const int64_t V = p.V;
  const int64_t lo = min((int64_t)rank * p.RL, V), hi = min(lo + p.RL, V);
  const int NG = (int)((hi - lo + 7) / 8);  // groups of 8 elements in this CTA's range
  const int NGc = (int)(p.RL / 8);          // stride of the e arrays
  const int m = p.m;
  const int NC = (NG + m - 1) / m;          // chunks of m groups in this range
  const bool cache = p.cache != 0, vec = p.vec != 0;
  // dynamic shared memory: [cache] e_p and e_q as hi/lo arrays (element k of
  // group g at k*NGc + g, so that a warp's 32 groups hit 32 banks); the chunk sums
  const int ca = cache ? 8 * NGc : 0;
  float* cph = dyn;
  float* cpl = cph + ca;
  float* cqh = cpl + ca;
  float* cql = cqh + ca;
  float* csh = cql + ca;
  float* csl = csh + p.NC;
  Ctx x;
  x.c_hi = p.c_hi;
  x.c_lo = p.c_lo;
  x.th = s.th;
  x.tl = s.tl;
  x.rho = df{0.f, 0.f};
  int xc = 0;  // exchanges so far: slot xc & 1 is free to write
  for (uint32_t f = clus; f < total; f += nclus) {
    const Rec r = p.recs[f];
    const char* prow = p.target + ((r.b * (int64_t)(p.K + 1) + r.j) * V) * p.esz;
    const char* qrow = r.resid ? p.draft + ((r.b * (int64_t)p.K + r.j) * V) * p.esz : prow;
    x.mp = r.mp;
    x.mq = r.mq;
    x.taup = r.taup;
    x.tauq = r.tauq;
    bool resid = r.resid != 0;
    // the weight of element k of group g: from the kept e values or evaluated
    // again from global memory
    auto weight1 = [&](int g, int k) -> df {
      if (cache) {
        const df ep{cph[k * NGc + g], cpl[k * NGc + g]};
        return resid ? x.resid_w(ep, df{cqh[k * NGc + g], cql[k * NGc + g]}) : ep;
      }
      const int64_t v = lo + 8 * (int64_t)g + k;
      const df ep = x.e(v < hi ? load_elem<E>(prow, v) : -INFINITY, x.mp, x.taup);
      if (!resid) return ep;
      return x.resid_w(ep, x.e(v < hi ? load_elem<E>(qrow, v) : -INFINITY, x.mq, x.tauq));
    };
    __syncthreads();  // the previous draw is done with the shared arrays
    // ---- step 1: e over the range (kept), and the residual's normalisers ----
    if (resid || cache) {
      df sp{0.f, 0.f}, sq{0.f, 0.f};
      // group g is processed while group g + kThreads is loading; the element
      // loop is not unrolled, so the double-float exp is one copy of code
      Raw<E> cp, cq, np, nq;
      if (tid < NG) {
        load_raw<E>(prow, lo + 8 * (int64_t)tid, hi, vec, cp);
        if (resid) load_raw<E>(qrow, lo + 8 * (int64_t)tid, hi, vec, cq);
      }
      for (int g = tid; g < NG; g += kThreads) {
        const int gn = g + kThreads;
        if (gn < NG) {
          load_raw<E>(prow, lo + 8 * (int64_t)gn, hi, vec, np);
          if (resid) load_raw<E>(qrow, lo + 8 * (int64_t)gn, hi, vec, nq);
        }
        // two elements per iteration: independent chains for the scheduler,
        // while the exp stays a few copies of code
#pragma unroll 1
        for (int k = 0; k < 8; k += 2) {
          const df ep0 = x.e(cp.at(k), x.mp, x.taup);
          const df ep1 = x.e(cp.at(k + 1), x.mp, x.taup);
          sp = df_add(sp, df_add(ep0, ep1));
          if (cache) {
            cph[k * NGc + g] = ep0.h;
            cpl[k * NGc + g] = ep0.l;
            cph[(k + 1) * NGc + g] = ep1.h;
            cpl[(k + 1) * NGc + g] = ep1.l;
          }
          if (resid) {
            const df eq0 = x.e(cq.at(k), x.mq, x.tauq);
            const df eq1 = x.e(cq.at(k + 1), x.mq, x.tauq);
            sq = df_add(sq, df_add(eq0, eq1));
            if (cache) {
              cqh[k * NGc + g] = eq0.h;
              cql[k * NGc + g] = eq0.l;
              cqh[(k + 1) * NGc + g] = eq1.h;
              cql[(k + 1) * NGc + g] = eq1.l;
            }
          }
        }
        cp = np;
        cq = nq;
      }
      if (resid) {  // uniform: the record is the cluster's
        block_sum2(sp, sq, s);
        const int b = xc++ & 1;
        if (tid == 0) {
          s.xs[b][0] = sp.h;
          s.xs[b][1] = sp.l;
          s.xs[b][2] = sq.h;
          s.xs[b][3] = sq.l;
        }
        cluster_sync();
        if (warp == 0) {
          // lane q holds rank q's sums; one shuffle tree, the same in every CTA
          df Sp{0.f, 0.f}, Sq{0.f, 0.f};
          if (lane < CL) {
            Sp = df{dsmem_ld_f32(&s.xs[b][0], (uint32_t)lane), dsmem_ld_f32(&s.xs[b][1], (uint32_t)lane)};
            Sq = df{dsmem_ld_f32(&s.xs[b][2], (uint32_t)lane), dsmem_ld_f32(&s.xs[b][3], (uint32_t)lane)};
          }
#pragma unroll 1
          for (int o = 16; o > 0; o >>= 1) {
            Sp = df_add(Sp, shfl_xor_df(Sp, o));
            Sq = df_add(Sq, shfl_xor_df(Sq, o));
          }
          if (lane == 0) {
            const df rr = df_div(Sp, Sq);
            s.bh[0] = rr.h;
            s.bl[0] = rr.l;
          }
        }
        __syncthreads();
        x.rho = df{s.bh[0], s.bl[0]};
      }
    }
    // ---- step 2: chunk sums, the cluster's scan, the crossing ------------------
    int32_t* out = p.out_tokens + (int64_t)r.b * (p.K + 1) + r.j;
    for (int pass = 0; pass < 2; ++pass) {
      int lastp = -1;  // the last positive weight this thread saw
      for (int c = tid; c < NC; c += kThreads) {
        df cs{0.f, 0.f};
        for (int i = 0; i < m; ++i) {
          const int g = c * m + i;
          if (g >= NG) break;
#pragma unroll 1
          for (int k = 0; k < 8; k += 2) {
            const df w0 = weight1(g, k);
            const df w1 = weight1(g, k + 1);
            cs = df_add(cs, df_add(w0, w1));
            if (df_pos(w0)) lastp = (int)(lo + 8 * (int64_t)g + k);
            if (df_pos(w1)) lastp = (int)(lo + 8 * (int64_t)g + k + 1);
          }
        }
        csh[c] = cs.h;
        csl[c] = cs.l;
      }
      __syncthreads();
      // thread t scans chunks [c0, c1): a contiguous run, in element order
      const int cpt = (NC + kThreads - 1) / kThreads;
      const int c0 = min(tid * cpt, NC), c1 = min(c0 + cpt, NC);
      df run{0.f, 0.f};
      for (int c = c0; c < c1; ++c) run = df_add(run, df{csh[c], csl[c]});
      df incl = warp_incl_scan_df(run, lane);
      int lm = lastp;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lm = max(lm, __shfl_xor_sync(0xffffffffu, lm, o));
      if (lane == 31) {
        s.wh[warp] = incl.h;
        s.wl[warp] = incl.l;
      }
      if (lane == 0) s.wi[warp] = lm;
      __syncthreads();
      if (warp == 0) {
        // the warps' totals scanned by one warp: each warp's base, the CTA's
        // total and its last positive index
        const df tw = lane < kWarps ? df{s.wh[lane], s.wl[lane]} : df{0.f, 0.f};
        int lw = lane < kWarps ? s.wi[lane] : -1;
        const df wi = warp_incl_scan_df(tw, lane);
        const df we = df_sub(wi, tw);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lw = max(lw, __shfl_xor_sync(0xffffffffu, lw, o));
        __syncwarp();
        if (lane < kWarps) {
          s.wh2[lane] = we.h;
          s.wl2[lane] = we.l;
        }
        if (lane == 31) {
          s.sh[0] = wi.h;
          s.sl[0] = wi.l;
          s.bi[2] = lw;
        }
      }
      __syncthreads();
      const df tot{s.sh[0], s.sl[0]};
      const int L = s.bi[2];
      incl = df_add(df{s.wh2[warp], s.wl2[warp]}, incl);  // this CTA's sum up to the end of thread t's run
      // exchange the range totals and last positive indices
      const int b = xc++ & 1;
      if (tid == 0) {
        s.xs[b][0] = tot.h;
        s.xs[b][1] = tot.l;
        s.xs[b][2] = __int_as_float(L);
      }
      cluster_sync();
      if (warp == 0) {
        // lane q holds rank q's total: one warp scan gives Z, this rank's
        // base and the owner (the first rank whose running sum passes u*Z)
        df t{0.f, 0.f};
        int a2 = -1;
        if (lane < CL) {
          t = df{dsmem_ld_f32(&s.xs[b][0], (uint32_t)lane), dsmem_ld_f32(&s.xs[b][1], (uint32_t)lane)};
          a2 = dsmem_ld_s32(&s.xs[b][2], (uint32_t)lane);
        }
        const df inc = warp_incl_scan_df(t, lane);
        const df Z{__shfl_sync(0xffffffffu, inc.h, 31), __shfl_sync(0xffffffffu, inc.l, 31)};
        const df exc = df_sub(inc, t);
        const df base{__shfl_sync(0xffffffffu, exc.h, (int)rank), __shfl_sync(0xffffffffu, exc.l, (int)rank)};
        int Lall = a2;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Lall = max(Lall, __shfl_xor_sync(0xffffffffu, Lall, o));
        const df target = df_mul_f(Z, r.u);
        const uint32_t om = __ballot_sync(0xffffffffu, lane < CL && df_gt(inc, target));
        const int owner = om ? __ffs(om) - 1 : -1;
        if (lane == 0) {
          s.bh[1] = Z.h;
          s.bl[1] = Z.l;
          s.bh[2] = base.h;
          s.bl[2] = base.l;
          s.bh[3] = target.h;
          s.bl[3] = target.l;
          s.bi[0] = owner;
          s.bi[1] = Lall;
        }
      }
      __syncthreads();
      if (pass == 0 && resid && !df_pos(df{s.bh[1], s.bl[1]})) {
        resid = false;  // a residual of zero mass: the draw is from p itself
        continue;
      }
      const int owner = s.bi[0];
      if (owner < 0) {
        // u*Z at or past the last partial sum: the last positive weight
        if (rank == 0 && tid == 0) *out = s.bi[1];
        break;
      }
      if ((int)rank != owner) break;
      const df base{s.bh[2], s.bl[2]}, target{s.bh[3], s.bl[3]};
      const uint32_t mk = __ballot_sync(0xffffffffu, c0 < c1 && df_gt(df_add(base, incl), target));
      if (lane == 0) s.wi[warp] = mk ? warp * 32 + __ffs(mk) - 1 : INT_MAX;
      __syncthreads();
      int first = INT_MAX;
      for (int w = 0; w < kWarps; ++w) first = min(first, s.wi[w]);
      if (first == INT_MAX) {
        // rounding between the cluster's totals and this CTA's scan: the
        // range's last positive weight
        if (tid == 0) *out = L;
        break;
      }
      if (tid == first) {  // where the crossing thread's run starts, in this CTA's sum
        const df ex = df_sub(incl, run);
        s.bh[0] = ex.h;
        s.bl[0] = ex.l;
      }
      __syncthreads();
      if (warp == 0) {
        // warp 0 walks that run 32 elements at a time: the first element whose
        // running sum passes u*Z
        const int fc0 = min(first * cpt, NC), fc1 = min(fc0 + cpt, NC);
        const int64_t E0 = lo + 8 * (int64_t)fc0 * m, E1 = min(lo + 8 * (int64_t)fc1 * m, hi);
        df C = df_add(base, df{s.bh[0], s.bl[0]});
        int t = -1, lw = -1;
        for (int64_t e0 = E0; e0 < E1 && t < 0; e0 += 32) {
          const int64_t e = e0 + lane;
          df w{0.f, 0.f};
          if (e < E1) {
            const int off = (int)(e - lo);
            w = weight1(off >> 3, off & 7);
          }
          const df Ce = df_add(C, warp_incl_scan_df(w, lane));
          const uint32_t pos = __ballot_sync(0xffffffffu, df_pos(w));
          if (pos) lw = (int)(e0 + 31 - __clz(pos));
          const uint32_t cr = __ballot_sync(0xffffffffu, e < E1 && df_gt(Ce, target));
          if (cr) t = (int)(e0 + __ffs(cr) - 1);
          C = df{__shfl_sync(0xffffffffu, Ce.h, 31), __shfl_sync(0xffffffffu, Ce.l, 31)};
        }
        // rounding between the scan and the walk: the run's last positive weight
        if (lane == 0) *out = t >= 0 ? t : (lw >= 0 ? lw : L);
      }
      break;
    }
  }
  cluster_sync();  // no CTA leaves while another may still read its exchange slots
  // ---- the last CTA out leaves the control words at zero ------------------------
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&p.ctl[1], 1u) == gridDim.x - 1) {
      p.ctl[0] = 0;
      __threadfence();
      p.ctl[1] = 0;
    }
  }
}

}  // namespace

void fill_table(Params& p, float temperature) {
  for (int i = 0; i < 32; ++i) {
    const double v = exp2((double)i / 32.0);
    p.tab_hi[i] = (float)v;
    p.tab_lo[i] = (float)(v - (double)p.tab_hi[i]);
  }
  const double cd = 1.4426950408889634 / (double)temperature;
  p.c_hi = (float)cd;
  p.c_lo = (float)(cd - (double)p.c_hi);
}

namespace {

// Launch shape per (device, V, element size).
struct Shape {
  int CL = 0, m = 1, NC = 0, cache = 0, clusters = 0;
  int64_t RL = 0;
  size_t smem = 0;
};
std::mutex g_mu;
std::map<std::tuple<int, int64_t, int>, Shape> g_shapes;

// The most dynamic shared memory the kernel may ask for on this device (the
// attribute is raised once per device and kernel).
template <typename E>
cudaError_t prepare(int dev, size_t& budget) {
  static std::map<int, size_t> done;
  auto it = done.find(dev);
  if (it != done.end()) {
    budget = it->second;
    return cudaSuccess;
  }
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  const size_t b = (size_t)optin > sizeof(Shared) + 2048 ? (size_t)optin - sizeof(Shared) - 2048 : 0;
  e = cudaFuncSetAttribute(refine_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)b);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(refine_kernel<E>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) {
    cudaGetLastError();  // only portable sizes then
  }
  done[dev] = b;
  budget = b;
  return cudaSuccess;
}

// CL: the smallest power of two that gives each CTA at most 4096 elements,
// capped at kMaxCluster, halved until the device can hold such a cluster.
template <typename E>
cudaError_t plan(int dev, int64_t V, Shape& sh) {
  size_t budget = 0;
  cudaError_t e = prepare<E>(dev, budget);
  if (e != cudaSuccess) return e;
  int want = 1;
  while (want < kMaxCluster && (int64_t)want * 4096 < V) want <<= 1;
  for (int CL = want; CL >= 1; CL >>= 1) {
    Shape t;
    t.CL = CL;
    t.RL = ((V + CL - 1) / CL + 7) / 8 * 8;
    const int64_t NGc = t.RL / 8;
    t.m = (int)((NGc + kMaxChunks - 1) / kMaxChunks);
    t.NC = (int)((NGc + t.m - 1) / t.m);
    const size_t sums = (size_t)t.NC * 8;
    t.cache = (size_t)NGc * 128 + sums <= budget;
    t.smem = (t.cache ? (size_t)NGc * 128 : 0) + sums;
    if (t.smem > budget) continue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)CL);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = t.smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, refine_kernel<E>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    if (n < 1) continue;
    t.clusters = n;
    sh = t;
    return cudaSuccess;
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace

cudaError_t launch(Params& p, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  Shape sh;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const auto key = std::make_tuple(dev, p.V, p.esz);
    auto it = g_shapes.find(key);
    if (it != g_shapes.end()) {
      sh = it->second;
    } else {
      e = p.esz == 2 ? plan<uint16_t>(dev, p.V, sh) : plan<float>(dev, p.V, sh);
      if (e != cudaSuccess) return e;
      g_shapes[key] = sh;
    }
  }
  p.CL = sh.CL;
  p.RL = sh.RL;
  p.m = sh.m;
  p.NC = sh.NC;
  p.cache = sh.cache;
  p.vec = (reinterpret_cast<uintptr_t>(p.target) % 16 == 0 && reinterpret_cast<uintptr_t>(p.draft) % 16 == 0 &&
           (p.V * p.esz) % 16 == 0)
              ? 1
              : 0;
  const int64_t clusters = p.B < sh.clusters ? p.B : sh.clusters;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * sh.CL));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sh.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)sh.CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  auto go = [&](cudaLaunchConfig_t& c) {
    return p.esz == 2 ? cudaLaunchKernelEx(&c, refine_kernel<uint16_t>, p)
                      : cudaLaunchKernelEx(&c, refine_kernel<float>, p);
  };
  e = go(cfg);
  if (e != cudaSuccess) {  // without programmatic serialisation
    cudaGetLastError();
    cfg.numAttrs = 1;
    e = go(cfg);
  }
  return e;
}

}  // namespace rf
}  // namespace sv
