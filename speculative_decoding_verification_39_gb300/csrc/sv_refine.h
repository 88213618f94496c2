// sv_refine.h — the draws that fp32 cannot settle, redone in double-float
// arithmetic (sv_refine.cu). Not part of the public ABI.
//
// A sampling draw finds the smallest t with sum_{v<=t} w_v > u*Z in fp32.
// When u*Z lands within kRefineMargin*Z of an edge of the chosen token's CDF
// interval (or the weights sum to zero, or the walk meets rounding), the draw
// kernel appends a record here; the refine kernel, launched after it on the
// same stream, recomputes those draws with double-float weights and sums and
// overwrites their tokens.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {
namespace rf {

// fp32 draws closer than this (times Z) to a CDF edge are redone. The fp32
// weights carry ~6e-8 relative error each (rounding, ex2.approx) and
// log2(e)/T rounded to fp32 (a relative error of up to 3e-8, the same in
// every weight and normaliser) shifts the CDF by up to a few 1e-8 of Z;
// with the running sums in double-float, 1e-7 of Z leaves room for both.
constexpr float kRefineMargin = 1e-7f;
constexpr int kThreads = 512;
// Largest thread-block cluster the refine kernel asks for (a non-portable
// size; smaller ones are used where the device cannot schedule it).
constexpr int kMaxCluster = 16;

// One flagged draw: sequence b drew position j from target row (b, j)
// (minus draft row (b, j) after a rejection) with uniform u; M are the
// rows' largest raw logits; tau the nucleus cut (stored logit value, -inf
// without top-p).
struct Rec {
  int32_t b, j, resid, pad;
  float mp, mq, taup, tauq, u;
  float pad2[3];
};

// Control words of the refine kernel, zero between calls: [0] flagged
// draws, [1] CTAs finished, [2..3] unused.
constexpr int kCtlWords = 4;

struct Params {
  const char* target;  // [B,K+1,V]
  const char* draft;   // [B,K,V]
  int64_t B, V;
  int K, esz;
  float c_hi, c_lo;    // log2(e)/T as a double-float
  float tab_hi[32], tab_lo[32];
  uint32_t* ctl;       // kCtlWords words
  uint32_t* stats;     // nullable: a running count of the draws refined
  Rec* recs;           // [B]
  int32_t* out_tokens; // [B, K+1]
  // launch shape (filled by launch())
  int CL;      // CTAs per draw: one thread-block cluster
  int m;       // groups of 8 elements per chunk
  int NC;      // chunks per CTA
  int cache;   // 1: the double-float e values of the range stay in shared memory
  int vec;     // 1: rows start on 16-byte boundaries (128-bit loads)
  int64_t RL;  // elements per CTA, a multiple of 8
};

// Appends a flagged draw (device side; any thread).
__device__ __forceinline__ void flag(uint32_t* ctl, Rec* recs, int64_t B, const Rec& r) {
  const uint32_t slot = atomicAdd(ctl, 1u);
  if (slot < (uint32_t)B) recs[slot] = r;
}

void fill_table(Params& p, float temperature);
// Plans the launch shape for p.V / p.esz on the current device and launches
// one grid of clusters (as many as can be resident, at most B) on `stream`.
cudaError_t launch(Params& p, cudaStream_t stream);

}  // namespace rf
}  // namespace sv
