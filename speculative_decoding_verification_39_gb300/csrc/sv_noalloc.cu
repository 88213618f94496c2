// sv_noalloc.cu — sv_verify_sample_noalloc: the sampling-mode verify for
// callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: code running inside a
// caller-managed memory pool or arena that must account for every byte,
// allocator hooks and custom allocators that would recurse into themselves,
// and deployments that pre-reserve all device memory at start-up and treat
// any later allocation as a failure. sv_verify_sample allocates (and caches)
// a scratch area per stream on its first call; this entry point instead runs
// the same kernels, chosen by the same rule and with the same launch shapes, on
// a fixed scratch array that is part of the library image itself, so a call
// allocates nothing, ever.
//
// The array below is a file-scope __device__ object of kNoAllocScratchBytes
// (4 MiB). Every GPU that loads the library holds it until the process exits.
// Host code must not pass the array's name to a kernel: on the host it is only
// a stand-in, not a device address. The device address is looked up once per
// device with cudaGetSymbolAddress (with that device current) on the first call
// on that device, and cached.
#include <cstdint>
#include <mutex>

#include "../../include/specverify.h"
#include "sv_sample_impl.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;
constexpr size_t kCtl = 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Set-up, once per device, with that device current: the array's device
// address on the current device.
int device_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SV_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return SV_ERR_CUDA;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return SV_OK;
}

// The scratch provider of this entry point: the fixed array, laid out as
// control block | counters | data, or SV_ERR_SCRATCH_LIMIT when the call
// needs more than it holds. The array keeps whatever the last call left, so
// the control block and the counters are cleared on the caller's stream (a
// memset, not an allocation) before the kernels run.
int fixed_scratch(void*, cudaStream_t, size_t cnt_words, size_t data_bytes, sv::ScratchArea* out) {
  const size_t data_off = kCtl + up256(cnt_words * 4);
  if (data_off + data_bytes > kNoAllocScratchBytes) return SV_ERR_SCRATCH_LIMIT;
  void* base = nullptr;
  const int rc = device_scratch(&base);
  if (rc != SV_OK) return rc;
  out->base = static_cast<char*>(base);
  out->data_off = data_off;
  out->clear_counters = true;
  return SV_OK;
}

}  // namespace

extern "C" int sv_verify_sample_noalloc(const void* target_logits, const void* draft_logits,
                                        const int32_t* draft_tokens, const float* uniforms, int64_t B, int32_t K,
                                        int64_t V, int32_t dtype, float temperature, float top_p,
                                        int32_t* out_tokens, int32_t* out_accept_len, float* out_row_stats,
                                        void* stream) {
  // The same checks, kernels and launch shapes as sv_verify_sample; only the
  // scratch differs. Calls whose kernels overlap on the GPU (other streams,
  // other threads) would race on the one array.
  return sv::verify_sample_impl(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype, temperature,
                                top_p, out_tokens, out_accept_len, out_row_stats, static_cast<cudaStream_t>(stream),
                                fixed_scratch, nullptr);
}
