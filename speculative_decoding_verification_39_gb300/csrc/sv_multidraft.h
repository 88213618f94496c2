// sv_multidraft.h — internal interface of the multi-draft sampling verify
// kernels (sv_multidraft.cu), used by the C ABI in sv_api.cu.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {
namespace md {

constexpr int kMaxG = 32;             // drafts per sequence
constexpr int kMaxRowsPerSeq = 1024;  // G * N
constexpr int kMaxGather = 2048;      // G * G * (N - 1), for each of the target and the draft gathers

struct Params {
  const void* target;       // [B,G,N,V]
  const void* draft;        // [B,G,N-1,V]
  const int32_t* tokens;    // [B,G,N-1]
  const float* uniforms;    // [B,(N-1)*G+1]
  int64_t B;
  int64_t V;
  int32_t G;
  int32_t N;
  float c;                  // log2(e) / T
  float2* rowstat;          // scratch [B*G*N + B*G*(N-1)]: target rows, then draft rows; {M, S}
  float* gp;                // scratch [B*G*(N-1)*G]: l*c of draft k's token in target row (b, a, n)
  float* gq;                // scratch [B*G*(N-1)*G]: l*c of draft k's token in draft row (b, j, n)
  uint32_t* ctl;            // scratch control block; ctl[3] is the sticky status word
  int32_t* out_tokens;      // [B,N]
  int32_t* out_accept_len;  // [B]
  int32_t* out_best;        // [B] or null
  float* out_row_lse;       // [B*G*N + B*G*(N-1)] or null, rows in rowstat's order
};

inline bool fits(int64_t G, int64_t N) {
  return G >= 1 && G <= kMaxG && N >= 2 && G * N <= kMaxRowsPerSeq && G * G * (N - 1) <= kMaxGather;
}

cudaError_t launch(const Params& p, int dtype, cudaStream_t stream);

}  // namespace md
}  // namespace sv
