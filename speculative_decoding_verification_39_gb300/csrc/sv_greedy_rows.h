// sv_greedy_rows.h — internal interface of the two-kernel greedy verify
// (sv_greedy_rows.cu), used by the C ABI in sv_api.cu.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {
namespace gr {

struct Params {
  const void* logits;       // [B,G,N,V]
  const int32_t* cand;      // [B,G,N-1]
  int64_t B;
  int64_t V;
  int32_t G;
  int32_t N;
  int32_t* am;              // scratch [B*G*N]: each row's argmax, or -2 for a row holding a NaN
  uint32_t* ctl;            // scratch control block; ctl[3] is the sticky status word
  int32_t* out_tokens;      // [B,N]
  int32_t* out_accept_len;  // [B]
  int32_t* out_best;        // [B] or null
};

cudaError_t launch(const Params& p, int dtype, cudaStream_t stream);

}  // namespace gr
}  // namespace sv
