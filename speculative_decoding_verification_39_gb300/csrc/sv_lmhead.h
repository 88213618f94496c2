// sv_lmhead.h — the LM-head GEMM of the verify on hidden states
// (sv_lmhead.cu): logits = h · Wᵀ on the sm_103a tensor cores (tcgen05, fp32
// accumulators in tensor memory), written as fp32 for the sampling verify.
// Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {
namespace lm {

constexpr int kTileM = 128;  // rows of a tile: a CTA's vocabulary entries (tensor-memory lanes), or positions
constexpr int kTileK = 64;   // hidden dimension per shared-memory stage
constexpr int kThreads = 256;

struct Params {
  const uint16_t* h[2];  // bf16 hidden states: [Mrows[i], D] (target rows, then draft rows)
  const uint16_t* w[2];  // bf16 LM heads [V, D]
  float* out[2];         // fp32 logits [Mrows[i], V]
  int64_t Mrows[2];
  int64_t V, D;
  uint32_t* status;      // sticky status word (a wait that ran out)
};

// D a multiple of kTileK; one launch covers both heads.
bool fits(int64_t D);
cudaError_t launch(const Params& p, cudaStream_t stream);

}  // namespace lm
}  // namespace sv
