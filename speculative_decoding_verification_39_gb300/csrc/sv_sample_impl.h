// sv_sample_impl.h — the sampling verify behind both of its C entry points
// (sv_verify_sample in sv_api.cu, sv_verify_sample_noalloc in sv_noalloc.cu).
// The two differ only in where their scratch memory comes from, so the
// argument checks, the choice of kernels and their launch shapes are one
// function here, given a scratch provider. Not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

// A scratch area laid out as [control block: 256 B][counters][data]:
// `base` its start, `data_off` the offset of the data region.
struct ScratchArea {
  char* base;
  size_t data_off;
  bool clear_counters;  // the control block and counters are not known to be zero: clear them before use
};

// Fills *out with an area holding at least `cnt_words` 32-bit counters and
// `data_bytes` of data for work on `stream`; returns an sv_status.
typedef int (*ScratchGet)(void* ctx, cudaStream_t stream, size_t cnt_words, size_t data_bytes, ScratchArea* out);

// Adds n to the count sv_launch_count reports (kernels launched by entry
// points outside sv_api.cu).
void note_launches(int n);

int verify_sample_impl(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                       const float* uniforms, int64_t B, int32_t K, int64_t V, int32_t dtype, float temperature,
                       float top_p, int32_t* out_tokens, int32_t* out_accept_len, float* out_row_stats,
                       cudaStream_t stream, ScratchGet get, void* ctx);

}  // namespace sv
