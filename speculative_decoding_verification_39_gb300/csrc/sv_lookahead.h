// sv_lookahead.h — internal interface of the Lookahead sampling-mode verify
// kernels (sv_lookahead.cu), used by the C ABI in sv_api.cu.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {
namespace la {

constexpr int kMaxG = 32;             // candidates per sequence: one lane of the walking warp each
constexpr int kMaxRowsPerSeq = 1024;  // G * N
constexpr int kMaxGather = 4096;      // G * G * (N - 1) gathered candidate logits per sequence

struct Params {
  const void* logits;       // [B,G,N,V], dtype as launched
  const int32_t* cand;      // [B,G,N-1]
  const float* uniforms;    // [B,(N-1)*G+1]
  int64_t B;
  int64_t V;
  int32_t G;
  int32_t N;
  float c;                  // log2(e) / T
  float2* rowstat;          // scratch [B*G*N]: {M = max_v l_v*c, S = sum_v 2^(l_v*c - M)}
  float* gath;              // scratch [B*G*(N-1)*G]: l*c of candidate k's token in row (b, a, n)
  uint32_t* ctl;            // scratch control block; ctl[3] is the sticky status word
  int32_t* out_tokens;      // [B,N]
  int32_t* out_accept_len;  // [B]
  int32_t* out_best;        // [B] or null
  float* out_row_lse;       // [B,G,N] or null: log sum_v exp(l_v/T) of every row
};

// Whether (G, N) is within the kernels' per-sequence limits.
inline bool fits(int64_t G, int64_t N) {
  return G >= 1 && G <= kMaxG && N >= 2 && G * N <= kMaxRowsPerSeq && G * G * (N - 1) <= kMaxGather;
}

// Enqueues both kernels on `stream`. dtype 0 = fp32, 1 = bf16.
cudaError_t launch(const Params& p, int dtype, cudaStream_t stream);

}  // namespace la
}  // namespace sv
