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
  template <typename E>
  __device__ __forceinline__ df w(int64_t v) const {
    const df ep = e(load_elem<E>(prow, v), mp, taup);
    if (!resid) return ep;
    const df r = df_sub(ep, df_mul(rho, e(load_elem<E>(qrow, v), mq, tauq)));
    return df_pos(r) ? r : df{0.f, 0.f};
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
  __shared__ int sh_ok;
  grid_dependency_sync(true);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, cta = blockIdx.x;
  const int64_t V = p.V;
  uint32_t total = ld_acquire_gpu(&p.ctl[0]);
  if (total > (uint32_t)p.B) total = (uint32_t)p.B;
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
    for (int f = 0; f < nb; ++f) {
      if (!rec[f].resid) continue;
      setup(rec[f], false);
      df sp{0.f, 0.f}, sq{0.f, 0.f};
      for (int64_t v = lo + tid; v < hi; v += kThreads) {
        sp = df_add(sp, x.e(load_elem<E>(x.prow, v), x.mp, x.taup));
        sq = df_add(sq, x.e(load_elem<E>(x.qrow, v), x.mq, x.tauq));
      }
      sp = block_sum_df(sp, red, tid);
      sq = block_sum_df(sq, red, tid);
      if (tid == 0) {
        float* q = p.part + ((int64_t)f * G + cta) * kRecFloats;
        q[0] = sp.h;
        q[1] = sp.l;
        q[2] = sq.h;
        q[3] = sq.l;
      }
    }
    ok = grid_barrier(p.ctl, ++nbar, &sh_ok);
    if (!ok) break;
    for (int f = tid; f < nb; f += kThreads) {
      if (!rec[f].resid) continue;
      df a{0.f, 0.f}, bq{0.f, 0.f};
      for (int c = 0; c < G; ++c) {
        const float* q = p.part + ((int64_t)f * G + c) * kRecFloats;
        a = df_add(a, df{__ldcg(q + 0), __ldcg(q + 1)});
        bq = df_add(bq, df{__ldcg(q + 2), __ldcg(q + 3)});
      }
      const df r = df_div(a, bq);
      rho_h[f] = r.h;
      rho_l[f] = r.l;
    }
    __syncthreads();
    // ---- phase 2: range totals of the weights; a second pass, from p itself,
    // settles residuals of zero mass ----------------------------------------
    // per (draw, CTA) record of 12 floats: [0..3] S_p, S_q; [4..5] total and
    // [6] last positive index of pass 0; [7..8] and [9] of pass 1
    for (int pass = 0; pass < 2 && ok; ++pass) {
      int any = 0;
      for (int f = 0; f < nb; ++f) {
        const bool in_pass = pass == 0 || (rec[f].resid && zero[f]);
        if (!in_pass) continue;
        any = 1;
        setup(rec[f], pass == 0 && rec[f].resid);
        x.rho = df{rho_h[f], rho_l[f]};
        df t{0.f, 0.f};
        int last = -1;
        for (int64_t v = lo + tid; v < hi; v += kThreads) {
          const df w = x.w<E>(v);
          if (df_pos(w)) last = (int)v;
          t = df_add(t, w);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
        t = block_sum_df(t, red, tid);
        if (lane == 0) lastw[warp] = last;
        __syncthreads();
        if (tid == 0) {
          int l2 = -1;
          for (int w = 0; w < kWarps; ++w) l2 = max(l2, lastw[w]);
          float* q = p.part + ((int64_t)f * G + cta) * kRecFloats;
          q[4 + 3 * pass] = t.h;
          q[5 + 3 * pass] = t.l;
          q[6 + 3 * pass] = __int_as_float(l2);
        }
        __syncthreads();
      }
      if (pass == 1 && !any) break;
      ok = grid_barrier(p.ctl, ++nbar, &sh_ok);
      if (!ok) break;
      // ---- the crossing of each draw this pass settles --------------------------
      for (int f = 0; f < nb; ++f) {
        const bool in_pass = pass == 0 || (rec[f].resid && zero[f]);
        if (!in_pass) continue;
        df Z{0.f, 0.f};
        for (int c = 0; c < G; ++c) {
          const float* q = p.part + ((int64_t)f * G + c) * kRecFloats;
          Z = df_add(Z, df{__ldcg(q + 4 + 3 * pass), __ldcg(q + 5 + 3 * pass)});
        }
        if (pass == 0) {
          const int z = rec[f].resid && !df_pos(Z);
          __syncthreads();
          if (tid == 0) zero[f] = z;
          if (z) continue;  // settled in the second pass
        }
        const df target = df_mul_f(Z, rec[f].u);
        df P{0.f, 0.f}, Pme{0.f, 0.f};
        int owner = -1, last_cta = -1, last_tok = -1;
        for (int c = 0; c < G; ++c) {
          const float* q = p.part + ((int64_t)f * G + c) * kRecFloats;
          const df tq{__ldcg(q + 4 + 3 * pass), __ldcg(q + 5 + 3 * pass)};
          if (c == cta) Pme = P;
          P = df_add(P, tq);
          if (owner < 0 && df_gt(P, target)) owner = c;
          const int lt = __float_as_int(__ldcg(q + 6 + 3 * pass));
          if (lt >= 0) {
            last_cta = c;
            last_tok = lt;
          }
        }
        const Rec& r = rec[f];
        int32_t* out = p.out_tokens + (int64_t)r.b * (p.K + 1) + r.j;
        if (owner < 0) {
          // u*Z at or past the last partial sum: the last positive weight
          if (cta == last_cta && tid == 0) *out = last_tok;
          continue;
        }
        if (cta != owner || warp != 0) continue;
        setup(r, pass == 0 && r.resid);
        x.rho = df{rho_h[f], rho_l[f]};
        df base = Pme;
        int tok = -1, lastpos = -1;
        bool done = false;
        for (int64_t g0 = lo; g0 < hi && !done; g0 += 256) {
          const int64_t e = g0 + lane * 8;
          df w[8];
          df s{0.f, 0.f};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            w[k] = (e + k < hi) ? x.w<E>(e + k) : df{0.f, 0.f};
            if (df_pos(w[k])) lastpos = (int)(e + k);
            s = df_add(s, w[k]);
          }
          const df incl = warp_incl_scan_df(s, lane);
          const uint32_t m = __ballot_sync(0xffffffffu, df_gt(df_add(base, incl), target));
          if (m) {
            int t = -1;
            if (lane == __ffs(m) - 1) {
              df C = df_add(base, df_sub(incl, s));
              for (int k = 0; k < 8 && t < 0; ++k) {
                C = df_add(C, w[k]);
                if (df_gt(C, target)) t = (int)(e + k);
              }
              for (int k = 7; k >= 0 && t < 0; --k)  // rounding between scan and walk
                if (df_pos(w[k])) t = (int)(e + k);
            }
            const uint32_t fm = __ballot_sync(0xffffffffu, t >= 0);
            if (fm) tok = __shfl_sync(0xffffffffu, t, __ffs(fm) - 1);
            done = true;
          }
          df tot;
          tot.h = __shfl_sync(0xffffffffu, incl.h, 31);
          tot.l = __shfl_sync(0xffffffffu, incl.l, 31);
          base = df_add(base, tot);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
        if (lane == 0) *out = tok >= 0 ? tok : lastpos;
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
