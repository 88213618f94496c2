// sv_refine.cu — the refine kernel: sampling draws that an fp32 draw could not
// settle, redone in double-float arithmetic over the whole GPU (sm_103a).
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
// One CTA per SM, launched cooperatively, so that the CTAs can wait for one
// another at grid barriers (bounded: a wait gives up after 2 s and the call
// reports SV_ERR_TIMEOUT). Each CTA owns one contiguous range of every row;
// every flagged draw of the call is handled in the same three phases —
// normaliser partials, range totals, the crossing — so that the number of
// barriers does not grow with the number of flagged draws.
#include <climits>

#include "sv_device.cuh"
#include "sv_df.cuh"
#include "sv_refine.h"

namespace sv {
namespace rf {
namespace {

constexpr int kWarps = kThreads / 32;
constexpr int kRecFloats = 12;  // per (flagged draw, CTA) partials
constexpr int kGroup = 4;       // flagged draws whose loads a thread keeps in flight together
constexpr int kPer = 4;         // elements per row and draw a thread loads at a time

template <typename E>
__device__ __forceinline__ float load_elem(const char* row, int64_t e) {
  if (sizeof(E) == 2)
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row) + e)) << 16);
  return __ldg(reinterpret_cast<const float*>(row) + e);
}

struct Ctx {
  const char* prow;
  const char* qrow;
  float mp, mq, taup, tauq;
  df rho;
  bool resid;  // weights max(0, e_p - rho e_q); otherwise e_p
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
  // the weight of an element with target logit lp and draft logit lq
  __device__ __forceinline__ df w_of(float lp, float lq) const {
    const df ep = e(lp, mp, taup);
    if (!resid) return ep;
    const df r = df_sub(ep, df_mul(rho, e(lq, mq, tauq)));
    return df_pos(r) ? r : df{0.f, 0.f};
  }
  template <typename E>
  __device__ __forceinline__ df w(int64_t v) const {
    return w_of(load_elem<E>(prow, v), resid ? load_elem<E>(qrow, v) : -INFINITY);
  }
};

__device__ __forceinline__ df warp_sum_df(df v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    df t;
    t.h = __shfl_xor_sync(0xffffffffu, v.h, o);
    t.l = __shfl_xor_sync(0xffffffffu, v.l, o);
    v = df_add(v, t);
  }
  return v;
}
__device__ __forceinline__ df warp_incl_scan_df(df v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    df t;
    t.h = __shfl_up_sync(0xffffffffu, v.h, o);
    t.l = __shfl_up_sync(0xffffffffu, v.l, o);
    if (lane >= o) v = df_add(v, t);
  }
  return v;
}

// Sum over the CTA, in a fixed order; every thread gets it.
__device__ __forceinline__ df block_sum_df(df v, float* sh, int tid) {
  v = warp_sum_df(v);
  const int lane = tid & 31, warp = tid >> 5;
  __syncthreads();
  if (lane == 0) {
    sh[2 * warp] = v.h;
    sh[2 * warp + 1] = v.l;
  }
  __syncthreads();
  df s{0.f, 0.f};
  for (int w = 0; w < kWarps; ++w) s = df_add(s, df{sh[2 * w], sh[2 * w + 1]});
  return s;
}

// Over the G CTAs' partials of one flagged draw (record fields oh, oh+1 as a
// double-float, ol the last-positive index; ol < 0: none), in CTA order, one
// CTA per thread (G <= kThreads): every thread gets the total, the exclusive
// prefix of CTA `me`, the first CTA whose inclusive prefix exceeds u*total
// (-1: none, or u < 0 to skip) and the largest last-positive index. All loads
// are issued at once.
struct Scan {
  df total, excl_me;
  int owner, last;
};
__device__ Scan cta_scan(const float* part, int f, int G, int oh, int ol, float u, int me, float* wh, float* wl,
                         int* wi, int* wj) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* q = part + ((int64_t)f * G + tid) * kRecFloats;
  df v{0.f, 0.f};
  int lt = -1;
  if (tid < G) {
    v = df{__ldcg(q + oh), __ldcg(q + oh + 1)};
    if (ol >= 0) lt = __float_as_int(__ldcg(q + ol));
  }
  df incl = warp_incl_scan_df(v, lane);
  int lm = lt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lm = max(lm, __shfl_xor_sync(0xffffffffu, lm, o));
  __syncthreads();
  if (lane == 31) {
    wh[warp] = incl.h;
    wl[warp] = incl.l;
  }
  if (lane == 0) wi[warp] = lm;
  __syncthreads();
  df base{0.f, 0.f}, total{0.f, 0.f};
  int last = -1;
  for (int w = 0; w < kWarps; ++w) {
    const df tw{wh[w], wl[w]};
    if (w < warp) base = df_add(base, tw);
    total = df_add(total, tw);
    last = max(last, wi[w]);
  }
  incl = df_add(base, incl);
  Scan r;
  r.total = total;
  r.last = last;
  const df target = df_mul_f(total, u < 0.f ? 0.f : u);
  const uint32_t m = __ballot_sync(0xffffffffu, tid < G && u >= 0.f && df_gt(incl, target));
  __syncthreads();
  if (lane == 0) wj[warp] = m ? warp * 32 + __ffs(m) - 1 : INT_MAX;
  if (tid == me) {
    const df ex = df_sub(incl, v);
    wh[kWarps] = ex.h;
    wl[kWarps] = ex.l;
  }
  __syncthreads();
  int own = INT_MAX;
  for (int w = 0; w < kWarps; ++w) own = min(own, wj[w]);
  r.owner = own == INT_MAX ? -1 : own;
  r.excl_me = df{wh[kWarps], wl[kWarps]};
  __syncthreads();  // the scratch may be reused by the next call
  return r;
}

// Every CTA waits until all have arrived k times; false if the wait gave up
// (or another CTA's did).
__device__ bool grid_barrier(uint32_t* ctl, uint32_t k, int* sh_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&ctl[1], 1u);
    const uint32_t target = k * gridDim.x;
    int ok = 1;
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(&ctl[1]) < target) {
      if (ld_relaxed_gpu(&ctl[3])) {
        ok = 0;
        break;
      }
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicExch(&ctl[3], 1u);
        ok = 0;
        break;
      }
    }
    __threadfence();
    *sh_ok = ok;
  }
  __syncthreads();
  return *sh_ok != 0;
}

template <typename E>
__global__ void __launch_bounds__(kThreads, 1) refine_kernel(const Params p) {
  __shared__ float red[2 * kWarps];
  __shared__ Rec rec[kMaxBatch];
  __shared__ float rho_h[kMaxBatch], rho_l[kMaxBatch];
  __shared__ int zero[kMaxBatch];
  __shared__ int lastw[kWarps];
  __shared__ float wt_h[kWarps + 1], wt_l[kWarps + 1];
  __shared__ int wsi[kWarps], wsj[kWarps];
  __shared__ int sh_ok, sh_tok;
  grid_dependency_sync(true);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, cta = blockIdx.x;
  const int64_t V = p.V;
  uint32_t total = ld_acquire_gpu(&p.ctl[0]);
  if (total > (uint32_t)p.B) total = (uint32_t)p.B;
  if (cta == 0 && tid == 0 && total && p.stats) atomicAdd(p.stats, total);
  // this CTA's range of every row: [lo, hi), a multiple of 8 elements long
  const int64_t RL = ((V + G - 1) / G + 7) / 8 * 8;
  const int64_t lo = min((int64_t)cta * RL, V), hi = min(lo + RL, V);
  uint32_t nbar = 0;
  bool ok = true;
  Ctx x;
  x.c_hi = p.c_hi;
  x.c_lo = p.c_lo;
  x.th = p.tab_hi;
  x.tl = p.tab_lo;
  auto setup = [&](const Rec& r, bool resid) {
    x.prow = p.target + ((r.b * (int64_t)(p.K + 1) + r.j) * V) * p.esz;
    x.qrow = r.resid ? p.draft + ((r.b * (int64_t)p.K + r.j) * V) * p.esz : x.prow;
    x.mp = r.mp;
    x.mq = r.mq;
    x.taup = r.taup;
    x.tauq = r.tauq;
    x.resid = resid;
  };
  for (uint32_t f0 = 0; f0 < total && ok; f0 += kMaxBatch) {
    const int nb = (int)min((uint32_t)kMaxBatch, total - f0);
    for (int f = tid; f < nb; f += kThreads) rec[f] = p.recs[f0 + f];
    __syncthreads();
    // ---- phase 1: the residual draws' normalisers, per range ----------------
    // Draws go four at a time: every thread first loads its elements of all
    // four (so that their latencies overlap), then sums.
    for (int g0 = 0; g0 < nb; g0 += kGroup) {
      df sp[kGroup], sq[kGroup];
#pragma unroll
      for (int q = 0; q < kGroup; ++q) sp[q] = sq[q] = df{0.f, 0.f};
      for (int64_t v0 = lo + tid; v0 < hi; v0 += kPer * kThreads) {
        float lp[kGroup][kPer], lq[kGroup][kPer];
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
          const bool on = g0 + q < nb && rec[g0 + q].resid;
          const Rec& r = rec[on ? g0 + q : g0];
          const char* pr = p.target + ((r.b * (int64_t)(p.K + 1) + r.j) * V) * p.esz;
          const char* qr = p.draft + ((r.b * (int64_t)p.K + (r.resid ? r.j : 0)) * V) * p.esz;
#pragma unroll
          for (int u = 0; u < kPer; ++u) {
            const int64_t v = v0 + (int64_t)u * kThreads;
            lp[q][u] = (on && v < hi) ? load_elem<E>(pr, v) : -INFINITY;
            lq[q][u] = (on && v < hi) ? load_elem<E>(qr, v) : -INFINITY;
          }
        }
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
          if (!(g0 + q < nb && rec[g0 + q].resid)) continue;
          setup(rec[g0 + q], false);
#pragma unroll
          for (int u = 0; u < kPer; ++u) {
            sp[q] = df_add(sp[q], x.e(lp[q][u], x.mp, x.taup));
            sq[q] = df_add(sq[q], x.e(lq[q][u], x.mq, x.tauq));
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kGroup; ++q) {
        if (!(g0 + q < nb && rec[g0 + q].resid)) continue;  // uniform: rec is in shared memory
        const df a = block_sum_df(sp[q], red, tid);
        const df bq = block_sum_df(sq[q], red, tid);
        if (tid == 0) {
          float* qq = p.part + ((int64_t)(g0 + q) * G + cta) * kRecFloats;
          qq[0] = a.h;
          qq[1] = a.l;
          qq[2] = bq.h;
          qq[3] = bq.l;
        }
      }
    }
    ok = grid_barrier(p.ctl, ++nbar, &sh_ok);
    if (!ok) break;
    for (int f = 0; f < nb; ++f) {
      if (!rec[f].resid) continue;  // uniform: rec is in shared memory
      const Scan sa = cta_scan(p.part, f, G, 0, -1, -1.f, 0, wt_h, wt_l, wsi, wsj);
      const Scan sb = cta_scan(p.part, f, G, 2, -1, -1.f, 0, wt_h, wt_l, wsi, wsj);
      if (tid == 0) {
        const df r = df_div(sa.total, sb.total);
        rho_h[f] = r.h;
        rho_l[f] = r.l;
      }
    }
    __syncthreads();
    // ---- phase 2: range totals of the weights; a second pass, from p itself,
    // settles residuals of zero mass ----------------------------------------
    // per (draw, CTA) record of 12 floats: [0..3] S_p, S_q; [4..5] total and
    // [6] last positive index of pass 0; [7..8] and [9] of pass 1
    for (int pass = 0; pass < 2 && ok; ++pass) {
      int any = 0;
      for (int g0 = 0; g0 < nb; g0 += kGroup) {
        df t[kGroup];
        int last[kGroup];
        bool in[kGroup];
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
          t[q] = df{0.f, 0.f};
          last[q] = -1;
          in[q] = g0 + q < nb && (pass == 0 || (rec[g0 + q].resid && zero[g0 + q]));
          any |= in[q];
        }
        for (int64_t v0 = lo + tid; v0 < hi; v0 += kPer * kThreads) {
          float lp[kGroup][kPer], lq[kGroup][kPer];
#pragma unroll
          for (int q = 0; q < kGroup; ++q) {
            const Rec& r = rec[in[q] ? g0 + q : g0];
            const bool rs = in[q] && pass == 0 && r.resid;
            const char* pr = p.target + ((r.b * (int64_t)(p.K + 1) + r.j) * V) * p.esz;
            const char* qr = p.draft + ((r.b * (int64_t)p.K + (r.resid ? r.j : 0)) * V) * p.esz;
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
              const int64_t v = v0 + (int64_t)u * kThreads;
              lp[q][u] = (in[q] && v < hi) ? load_elem<E>(pr, v) : -INFINITY;
              lq[q][u] = (rs && v < hi) ? load_elem<E>(qr, v) : -INFINITY;
            }
          }
#pragma unroll
          for (int q = 0; q < kGroup; ++q) {
            if (!in[q]) continue;
            setup(rec[g0 + q], pass == 0 && rec[g0 + q].resid);
            x.rho = df{rho_h[g0 + q], rho_l[g0 + q]};
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
              const df w = x.w_of(lp[q][u], lq[q][u]);
              if (df_pos(w)) last[q] = (int)(v0 + (int64_t)u * kThreads);
              t[q] = df_add(t[q], w);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
          if (!in[q]) continue;  // uniform: rec and zero are in shared memory
          int l = last[q];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) l = max(l, __shfl_xor_sync(0xffffffffu, l, o));
          const df tt = block_sum_df(t[q], red, tid);
          if (lane == 0) lastw[warp] = l;
          __syncthreads();
          if (tid == 0) {
            int l2 = -1;
            for (int w = 0; w < kWarps; ++w) l2 = max(l2, lastw[w]);
            float* qq = p.part + ((int64_t)(g0 + q) * G + cta) * kRecFloats;
            qq[4 + 3 * pass] = tt.h;
            qq[5 + 3 * pass] = tt.l;
            qq[6 + 3 * pass] = __int_as_float(l2);
          }
          __syncthreads();
        }
      }
      if (pass == 1 && !any) break;
      ok = grid_barrier(p.ctl, ++nbar, &sh_ok);
      if (!ok) break;
      // ---- the crossing of each draw this pass settles --------------------------
      for (int f = 0; f < nb; ++f) {
        const bool in_pass = pass == 0 || (rec[f].resid && zero[f]);
        if (!in_pass) continue;
        const Scan sc = cta_scan(p.part, f, G, 4 + 3 * pass, 6 + 3 * pass, rec[f].u, cta, wt_h, wt_l, wsi, wsj);
        const df Z = sc.total;
        if (pass == 0) {
          const int z = rec[f].resid && !df_pos(Z);
          if (tid == 0) zero[f] = z;
          if (z) continue;  // settled in the second pass
        }
        const df target = df_mul_f(Z, rec[f].u);
        const df Pme = sc.excl_me;
        const int owner = sc.owner;
        const Rec& r = rec[f];
        int32_t* out = p.out_tokens + (int64_t)r.b * (p.K + 1) + r.j;
        if (owner < 0) {
          // u*Z at or past the last partial sum: the last positive weight
          if (cta == 0 && tid == 0) *out = sc.last;
          continue;
        }
        if (cta != owner) continue;
        setup(r, pass == 0 && r.resid);
        x.rho = df{rho_h[f], rho_l[f]};
        // pieces of 256 elements, one per warp, kWarps at a time
        df base = Pme;
        int tok = -1;
        if (tid == 0) sh_tok = -1;
        __syncthreads();
        for (int64_t s0 = lo; s0 < hi && tok < 0; s0 += 256 * kWarps) {
          const int64_t e = s0 + (int64_t)warp * 256 + lane * 8;
          float lp[8], lq[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            lp[k] = e + k < hi ? load_elem<E>(x.prow, e + k) : -INFINITY;
            lq[k] = (e + k < hi && x.resid) ? load_elem<E>(x.qrow, e + k) : -INFINITY;
          }
          df w[8];
          df sl{0.f, 0.f};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            w[k] = x.w_of(lp[k], lq[k]);
            sl = df_add(sl, w[k]);
          }
          const df incl = warp_incl_scan_df(sl, lane);
          if (lane == 31) {
            wt_h[warp] = incl.h;
            wt_l[warp] = incl.l;
          }
          __syncthreads();
          // the bases of the pieces, in order; the first piece that crosses
          df bw = base;
          int cw = -1;
          for (int q = 0; q < kWarps; ++q) {
            const df nb2 = df_add(bw, df{wt_h[q], wt_l[q]});
            if (q == warp) {
              // this warp's base is bw
              const uint32_t m = __ballot_sync(0xffffffffu, df_gt(df_add(bw, incl), target));
              if (m && cw < 0) {
                int t = -1;
                if (lane == __ffs(m) - 1) {
                  df C = df_add(bw, df_sub(incl, sl));
                  for (int k = 0; k < 8 && t < 0; ++k) {
                    C = df_add(C, w[k]);
                    if (df_gt(C, target)) t = (int)(e + k);
                  }
                  for (int k = 7; k >= 0 && t < 0; --k)  // rounding between scan and walk
                    if (df_pos(w[k])) t = (int)(e + k);
                }
                const uint32_t fm = __ballot_sync(0xffffffffu, t >= 0);
                const int tv = __shfl_sync(0xffffffffu, t, fm ? __ffs(fm) - 1 : 0);
                if (fm && lane == 0) sh_tok = tv;
              }
            }
            if (cw < 0 && df_gt(nb2, target)) cw = q;
            bw = nb2;
          }
          __syncthreads();
          if (cw >= 0) tok = sh_tok;
          base = bw;
          __syncthreads();
        }
        if (tok < 0)  // rounding between the ranks' totals and the walk: the range's last positive weight
          tok = __float_as_int(__ldcg(p.part + ((int64_t)f * G + cta) * kRecFloats + 6 + 3 * pass));
        if (tid == 0) *out = tok;
      }
      __syncthreads();
    }
    if (!ok) break;
    ok = grid_barrier(p.ctl, ++nbar, &sh_ok);  // the partials may be reused
  }
  // ---- the last CTA out leaves the control words at zero ------------------------
  __syncthreads();
  if (tid == 0) {
    if (!ok) atomicOr(p.status, kStatusTimeout);
    __threadfence();
    if (atomicAdd(&p.ctl[2], 1u) == (uint32_t)G - 1) {
      p.ctl[0] = 0;
      p.ctl[1] = 0;
      p.ctl[3] = 0;
      __threadfence();
      p.ctl[2] = 0;
    }
  }
}

}  // namespace

size_t part_bytes(int grid) { return (size_t)kMaxBatch * grid * kRecFloats * sizeof(float); }

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

cudaError_t launch(const Params& p, int grid, cudaStream_t stream) {
  if (grid > kThreads) grid = kThreads;  // one CTA per thread in cta_scan
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  auto go = [&](cudaLaunchConfig_t& c) {
    return p.esz == 2 ? cudaLaunchKernelEx(&c, refine_kernel<uint16_t>, p)
                      : cudaLaunchKernelEx(&c, refine_kernel<float>, p);
  };
  cudaError_t e = go(cfg);
  if (e != cudaSuccess) {  // without programmatic serialisation
    cudaGetLastError();
    cfg.numAttrs = 1;
    e = go(cfg);
  }
  return e;
}

}  // namespace rf
}  // namespace sv
