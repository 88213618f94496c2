// sv_noalloc.cu — sv_verify_sample_noalloc: the sampling-mode verify for
// callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: code running inside a
// caller-managed memory pool or arena that must account for every byte,
// allocator hooks and custom allocators that would recurse into themselves,
// and deployments that pre-reserve all device memory at start-up and treat
// any later allocation as a failure. sv_verify_sample allocates (and caches)
// a scratch area per stream on its first call; this entry point instead runs
// the same kernel on a fixed scratch array that is part of the library image
// itself, so a call allocates nothing, ever.
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
#include "sv_kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;
constexpr size_t kCtl = 256;
constexpr int kMaxDevices = 64;
constexpr int kStages = 3;      // the launch shape sv_verify_sample uses by default
constexpr int kCtasPerSm = 2;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Set-up, once per device, with that device current.
int device_scratch(int dev, void** out, int* sms) {
  if (dev < 0 || dev >= kMaxDevices) return SV_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return SV_ERR_CUDA;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return SV_ERR_CUDA;
    }
    g_addr[dev] = p;
    g_sms[dev] = n;
  }
  *out = g_addr[dev];
  *sms = g_sms[dev];
  return SV_OK;
}

}  // namespace

extern "C" int sv_verify_sample_noalloc(const void* target_logits, const void* draft_logits,
                                        const int32_t* draft_tokens, const float* uniforms, int64_t B, int32_t K,
                                        int64_t V, int32_t dtype, float temperature, float top_p,
                                        int32_t* out_tokens, int32_t* out_accept_len, float* out_row_stats,
                                        void* stream) {
  // The same host-side checks as sv_verify_sample.
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B < 0 || K < 1 || V < 2 || V >= ((int64_t)1 << 31) || K > (1 << 20)) return SV_ERR_ARG;
  if (!(temperature >= 0.f) || temperature == __builtin_inff()) return SV_ERR_ARG;
  if (!(top_p > 0.f && top_p <= 1.f)) return SV_ERR_ARG;
  if (B == 0) return SV_OK;
  const bool limit = temperature == 0.f;
  if (!target_logits || !draft_tokens || !out_tokens || !out_accept_len) return SV_ERR_ARG;
  if (!limit && (!draft_logits || !uniforms)) return SV_ERR_ARG;
  const size_t esz = dtype == SV_BF16 ? 2 : 4;
  auto misaligned = [](const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; };
  if (misaligned(target_logits, esz) || (!limit && misaligned(draft_logits, esz))) return SV_ERR_DTYPE;
  if (misaligned(draft_tokens, 4) || misaligned(out_tokens, 4) || misaligned(out_accept_len, 4) ||
      (uniforms && misaligned(uniforms, 4)) || (out_row_stats && misaligned(out_row_stats, 16)))
    return SV_ERR_ARG;
  const float c = limit ? 0.f : (float)(1.4426950408889634 / (double)temperature);
  if (!limit && !(c < __builtin_inff())) return SV_ERR_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  void* base = nullptr;
  int sms = 1;
  int rc = device_scratch(dev, &base, &sms);
  if (rc != SV_OK) return rc;

  sv::Params p{};
  p.a = static_cast<const char*>(target_logits);
  p.d = static_cast<const char*>(limit ? target_logits : draft_logits);
  p.tokens = draft_tokens;
  p.uniforms = uniforms;
  p.out_tokens = out_tokens;
  p.out_accept_len = out_accept_len;
  p.out_best = nullptr;
  p.out_row_stats = limit ? nullptr : out_row_stats;
  p.B = B;
  p.V = V;
  p.K = K;
  p.RS = limit ? K + 1 : 2 * K + 1;
  p.c = c;
  p.T = temperature;
  p.top_p = top_p;
  p.topp = (!limit && top_p < 1.f) ? 1 : 0;
  p.stages = kStages;
  const int64_t rows = B * (int64_t)p.RS;
  p.TE = sv::kTileBytes / (int64_t)esz;
  p.NT = (V + p.TE - 1) / p.TE;
  const int64_t slots = (int64_t)sms * kCtasPerSm;
  int64_t ct = rows * p.NT / (slots * 4);
  ct = ct < 1 ? 1 : (ct > 8 ? 8 : ct);
  if (p.NT <= 4) ct = p.NT;  // as sv_verify_sample chooses
  if (ct > p.NT) ct = p.NT;
  p.NC = (p.NT + ct - 1) / ct;
  p.CT = (p.NT + p.NC - 1) / p.NC;
  p.W = rows * p.NC;
  // Draw splitting as sv_verify_sample chooses it.
  const int64_t CE = sv::cell_elems(V);
  const int64_t ncells = (V + CE - 1) / CE;
  p.DC = 0;
  p.CPC = 0;
  if (!limit) {
    const int64_t half = sv::draw_cells_per_chunk(kStages, (int)esz, V);
    int64_t dc = half > 0 ? (ncells + half - 1) / half : 0;
    // Only calls that leave most CTAs idle at their end gain from the split.
    const int64_t cover = (slots + B - 1) / B;
    if (B * 2 > slots) dc = 0;
    if (dc > cover) dc = cover;
    if (dc >= 2 && B * (1 + dc) < (int64_t(1) << 30)) {
      p.DC = (int)dc;
      p.CPC = (int)((ncells + dc - 1) / dc);
    }
  }

  // Layout inside the fixed array: control block, counters, data.
  const size_t cnt_bytes = up256((size_t)(rows + B * (3 + (int64_t)p.DC)) * 4);
  const size_t part_bytes = up256((size_t)p.W * 8);
  const size_t rowstat_bytes = up256((size_t)rows * 16);
  const size_t dcells_bytes = p.DC ? up256((size_t)B * (size_t)ncells * 4) : 0;
  const size_t need = kCtl + cnt_bytes + part_bytes + rowstat_bytes + dcells_bytes;
  if (need > kNoAllocScratchBytes) return SV_ERR_SCRATCH_LIMIT;
  char* s = static_cast<char*>(base);
  p.ctl = reinterpret_cast<uint32_t*>(s);
  p.row_cnt = reinterpret_cast<uint32_t*>(s + kCtl);
  p.seq_cnt = p.row_cnt + rows;
  p.tail_q = p.seq_cnt + B;
  p.dcnt = p.tail_q + B * (1 + p.DC);
  p.part = reinterpret_cast<float2*>(s + kCtl + cnt_bytes);
  p.rowstat = reinterpret_cast<float4*>(s + kCtl + cnt_bytes + part_bytes);
  p.dcells = reinterpret_cast<float*>(s + kCtl + cnt_bytes + part_bytes + rowstat_bytes);

  // The array keeps whatever the last call left: the control block and the
  // counters must start at zero, so clear them on the caller's stream (a
  // memset, not an allocation). Calls whose kernels overlap on the GPU (other
  // streams, other threads) would race on this one array.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(s, 0, kCtl + cnt_bytes, st) != cudaSuccess) return SV_ERR_CUDA;
  int64_t grid = slots;
  if (grid > p.W) grid = p.W;
  if (grid < 1) grid = 1;
  if (sv::launch(p, dtype, limit ? sv::kArgmaxLimit : sv::kSample, (int)grid, st) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}
