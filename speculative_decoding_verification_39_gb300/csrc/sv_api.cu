// sv_api.cu — the C ABI of libspecverify (declared in include/specverify.h):
// host-side argument checks, the per-(device, stream) scratch areas and the
// launch of the verify kernel.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/specverify.h"
#include "sv_kernels.h"
#include "sv_lmhead.h"
#include "sv_greedy_rows.h"
#include "sv_lookahead.h"
#include "sv_multidraft.h"
#include "sv_refine.h"
#include "sv_sample_impl.h"
#include "sv_v2.h"

namespace {

constexpr int kDefaultStages = 3;
constexpr int kDefaultCtasPerSm = 2;
constexpr int64_t kMaxV = (int64_t)1 << 31;

std::atomic<int> g_stages{kDefaultStages};
std::atomic<int> g_ctas_per_sm{kDefaultCtasPerSm};
std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_greedy_path{0};  // 0: row argmax + match kernels; 1: the streaming kernel
std::atomic<int> g_sample_path{0};  // 0: by size; 1: the streaming kernel; 2: row pass + cluster decide

// A scratch area has three parts at fixed places: the control block, a
// counter region and a data region. Every counter is back at zero when a call
// completes (the kernel resets what it used), and the counter region never
// holds anything else, so calls of any shape can follow each other without a
// memset. The data region (per-tile partials, per-row results) is written
// before it is read in every call.
struct Scratch {
  void* base = nullptr;
  size_t cnt_words = 0;   // capacity of the counter region, in 32-bit words
  size_t data_bytes = 0;  // capacity of the data region
  size_t bytes = 0;
};

std::mutex g_mu;
std::map<std::pair<int, uintptr_t>, Scratch> g_scratch;
// The fp32 logits of sv_verify_sample_lmhead when the caller gives no buffer:
// one workspace per (device, stream), grown on demand, freed by sv_release.
std::map<std::pair<int, uintptr_t>, std::pair<void*, size_t>> g_lm_ws;
std::map<int, int> g_sm_count;

constexpr size_t kCtlBytes = 256;
// Word of the control block that counts the draws the refine kernel redid
// (cumulative per scratch area; word 3 is the sticky status).
constexpr int kCtlRefined = 12;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t counter_offset() { return kCtlBytes; }
size_t data_offset(const Scratch& s) { return kCtlBytes + align256(s.cnt_words * 4); }

// Returns the scratch of the current device and `stream`, grown (and zeroed)
// if it has fewer than `cnt_words` counters or `data_bytes` of data room.
int get_scratch(cudaStream_t stream, size_t cnt_words, size_t data_bytes, Scratch* out, int* device) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  *device = dev;
  std::lock_guard<std::mutex> lk(g_mu);
  Scratch& s = g_scratch[{dev, reinterpret_cast<uintptr_t>(stream)}];
  if (s.cnt_words < cnt_words || s.data_bytes < data_bytes) {
    if (s.base) {
      cudaStreamSynchronize(stream);
      cudaFree(s.base);
      s = Scratch{};
    }
    Scratch n;
    n.cnt_words = cnt_words < 65536 ? 65536 : cnt_words;
    n.data_bytes = align256(data_bytes < (1u << 20) ? (1u << 20) : data_bytes);
    n.bytes = data_offset(n) + n.data_bytes;
    if (cudaMalloc(&n.base, n.bytes) != cudaSuccess) {
      cudaGetLastError();
      return SV_ERR_NOMEM;
    }
    if (cudaMemsetAsync(n.base, 0, n.bytes, stream) != cudaSuccess) return SV_ERR_CUDA;
    s = n;
  }
  *out = s;
  return SV_OK;
}

int sm_count(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_sm_count.find(dev);
  if (it != g_sm_count.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  g_sm_count[dev] = n;
  return n;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The refine kernel after a sampling call: it redoes, in double-float
// arithmetic, the draws the call's fp32 walks could not settle.
int launch_refine(const void* target, const void* draft, int64_t B, int K, int64_t V, int esz, float temperature,
                  uint32_t* rf_ctl, sv::rf::Rec* recs, uint32_t* status, int32_t* out_tokens, cudaStream_t stream) {
  sv::rf::Params r{};
  r.target = static_cast<const char*>(target);
  r.draft = static_cast<const char*>(draft);
  r.B = B;
  r.V = V;
  r.K = K;
  r.esz = esz;
  sv::rf::fill_table(r, temperature);
  r.ctl = rf_ctl;
  r.stats = status + (kCtlRefined - 3);
  r.recs = recs;
  r.out_tokens = out_tokens;
  if (sv::rf::launch(r, stream) != cudaSuccess) return SV_ERR_CUDA;
  g_launches.fetch_add(1);
  return SV_OK;
}

int run(sv::Params& p, int dtype, int mode, int64_t rows_total, cudaStream_t stream, sv::ScratchGet get, void* ctx,
        bool allow_seq = true) {
  const int esz = dtype == SV_BF16 ? 2 : 4;
  p.TE = sv::kTileBytes / esz;
  p.NT = (p.V + p.TE - 1) / p.TE;
  p.stages = g_stages.load();
  int dev0 = 0;
  if (cudaGetDevice(&dev0) != cudaSuccess) return SV_ERR_CUDA;
  const int64_t slots = (int64_t)sm_count(dev0) * g_ctas_per_sm.load();
  // Chunks of up to 8 tiles, small enough that every CTA gets about four of
  // them, and of near-equal size within a row.
  int64_t ct = rows_total * p.NT / (slots * 4);
  ct = ct < 1 ? 1 : (ct > 8 ? 8 : ct);
  // A row of up to four tiles is one chunk: its CTA finishes it alone, with
  // no partial to store and no row counter to count it against.
  if (p.NT <= 4) ct = p.NT;
  if (ct > p.NT) ct = p.NT;
  p.NC = (p.NT + ct - 1) / ct;
  p.CT = (p.NT + p.NC - 1) / p.NC;
  p.W = rows_total * p.NC;
  // Sampling draws over more cells than one ring half holds are split over
  // CTAs: into at most one chunk per half-ring of cells, and into no more
  // chunks than it takes for the call's draws to cover the CTAs once.
  const int64_t CE = sv::cell_elems(p.V);
  const int64_t ncells = (p.V + CE - 1) / CE;
  p.DC = 0;
  p.CPC = 0;
  if (mode == sv::kSample) {
    const int64_t half = sv::draw_cells_per_chunk(p.stages, esz, p.V);
    int64_t dc = half > 0 ? (ncells + half - 1) / half : 0;
    // Only calls that leave most CTAs idle at their end gain from the split.
    const int64_t cover = (slots + p.B - 1) / p.B;
    if (p.B * 2 > slots) dc = 0;
    if (dc > cover) dc = cover;
    if (dc >= 2 && p.B * (1 + dc) < (int64_t(1) << 30)) {
      p.DC = (int)dc;
      p.CPC = (int)((ncells + dc - 1) / dc);
    }
  }
  const bool refine = mode == sv::kSample;
  const size_t cnt_words = (size_t)rows_total + (size_t)p.B * (3 + (size_t)p.DC) + (refine ? sv::rf::kCtlWords : 0);
  const size_t part_bytes = align256((size_t)p.W * 8);
  const size_t rowstat_bytes = align256((size_t)rows_total * 16);
  const size_t dcells_bytes = p.DC ? align256((size_t)p.B * (size_t)ncells * 4) : 0;
  const size_t recs_bytes = refine ? align256((size_t)p.B * sizeof(sv::rf::Rec)) : 0;
  const size_t data_bytes = part_bytes + rowstat_bytes + dcells_bytes + recs_bytes;
  sv::ScratchArea sa;
  int rc = get(ctx, stream, cnt_words, data_bytes, &sa);
  if (rc != SV_OK) return rc;
  char* b = sa.base;
  if (sa.clear_counters && cudaMemsetAsync(b, 0, sa.data_off, stream) != cudaSuccess) return SV_ERR_CUDA;
  p.ctl = reinterpret_cast<uint32_t*>(b);
  p.row_cnt = reinterpret_cast<uint32_t*>(b + counter_offset());
  p.seq_cnt = p.row_cnt + rows_total;
  p.tail_q = p.seq_cnt + p.B;
  p.dcnt = p.tail_q + p.B * (1 + p.DC);
  p.part = reinterpret_cast<float2*>(b + sa.data_off);
  p.rowstat = reinterpret_cast<float4*>(b + sa.data_off + part_bytes);
  p.dcells = reinterpret_cast<float*>(b + sa.data_off + part_bytes + rowstat_bytes);
  p.rf_ctl = refine ? p.dcnt + p.B : nullptr;
  p.rf_recs = refine ? reinterpret_cast<sv::rf::Rec*>(b + sa.data_off + part_bytes + rowstat_bytes + dcells_bytes)
                     : nullptr;
  // Short rows: one warp per sequence (rows of at most 1024 elements), else
  // one CTA per sequence with the whole sequence staged in shared memory.
  const bool short_ok = mode == sv::kSample && !p.topp && aligned_to(p.a, 16) && aligned_to(p.d, 16);
  const bool warp_mode = short_ok && sv::warp_mode_fits(p.K, p.V, esz);
  const bool seq_mode = allow_seq && short_ok && !warp_mode && sv::seq_mode_fits(p.K, p.V, esz);
  int64_t grid = slots;
  const int64_t items = warp_mode ? (p.B + sv::warp_mode_seqs_per_cta() - 1) / sv::warp_mode_seqs_per_cta()
                                  : (seq_mode ? p.B : p.W);
  if (grid > items) grid = items;
  if (grid < 1) grid = 1;
  cudaError_t e = warp_mode  ? sv::launch_warp(p, dtype, (int)grid, stream)
                  : seq_mode ? sv::launch_seq(p, dtype, (int)grid, stream)
                             : sv::launch(p, dtype, mode, (int)grid, stream);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  g_launches.fetch_add(1);
  if (refine)
    return launch_refine(p.a, p.d, p.B, p.K, p.V, esz, p.T, p.rf_ctl, p.rf_recs, p.ctl + 3, p.out_tokens, stream);
  return SV_OK;
}

// The allocating provider: the per-(device, stream) scratch area.
int cached_scratch(void*, cudaStream_t stream, size_t cnt_words, size_t data_bytes, sv::ScratchArea* out) {
  Scratch sc;
  int dev = 0;
  const int rc = get_scratch(stream, cnt_words, data_bytes, &sc, &dev);
  if (rc != SV_OK) return rc;
  out->base = static_cast<char*>(sc.base);
  out->data_off = data_offset(sc);
  out->clear_counters = false;  // zeroed when allocated; every kernel leaves its counters at zero
  return SV_OK;
}

}  // namespace

int sv::verify_sample_impl(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                           const float* uniforms, int64_t B, int32_t K, int64_t V, int32_t dtype, float temperature,
                           float top_p, int32_t* out_tokens, int32_t* out_accept_len, float* out_row_stats,
                           cudaStream_t st, sv::ScratchGet get, void* ctx) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B < 0 || K < 1 || V < 2 || V >= kMaxV || K > (1 << 20)) return SV_ERR_ARG;
  if (!(temperature >= 0.f) || std::isinf(temperature)) return SV_ERR_ARG;
  if (!(top_p > 0.f && top_p <= 1.f)) return SV_ERR_ARG;
  if (B == 0) return SV_OK;
  const bool limit = temperature == 0.f;
  if (!target_logits || !draft_tokens || !out_tokens || !out_accept_len) return SV_ERR_ARG;
  if (!limit && (!draft_logits || !uniforms)) return SV_ERR_ARG;
  const size_t esz = dtype == SV_BF16 ? 2 : 4;
  if (!aligned_to(target_logits, esz) || (!limit && !aligned_to(draft_logits, esz))) return SV_ERR_DTYPE;
  if (!aligned_to(draft_tokens, 4) || !aligned_to(out_tokens, 4) || !aligned_to(out_accept_len, 4) ||
      (uniforms && !aligned_to(uniforms, 4)) || (out_row_stats && !aligned_to(out_row_stats, 16)))
    return SV_ERR_ARG;
  const float c = limit ? 0.f : (float)(1.4426950408889634 / (double)temperature);
  if (!limit && !std::isfinite(c)) return SV_ERR_ARG;
  // The row pass + cluster decide kernels re-read the draw rows after the
  // whole call has streamed: cheap while the call's logits stay in L2 (the
  // streaming kernel draws each sequence as soon as its rows are in, which
  // wins for larger calls).
  // Rows of at most 1024 elements go to the streaming kernel's one-warp-per-
  // sequence mode, which reads a whole sequence with one round of loads.
  const bool two_kernel_size = (double)B * (2.0 * K + 1.0) * (double)V * (double)esz <= 96.0 * 1024 * 1024;
  const bool warp_rows = sv::warp_mode_fits(K, V, (int)esz) && aligned_to(target_logits, 16) &&
                         aligned_to(draft_logits, 16);
  const int path = g_sample_path.load();
  // Top-p: the row pass holds each row in one cluster's registers while it
  // takes the nucleus cut, so the rows are read once at every size.
  const bool topp = top_p < 1.f;
  const bool v2_topp = !limit && topp && path != 1 && sv::v2::fits_topp(K, V, (int)esz) &&
                       aligned_to(target_logits, 16) && aligned_to(draft_logits, 16);
  if (v2_topp || (!limit && !topp && sv::v2::fits(K, V) &&
                  (path == 2 || (path == 0 && two_kernel_size && !warp_rows)))) {
    sv::v2::Params q{};
    q.topp = topp ? 1 : 0;
    q.top_p = top_p;
    q.target = static_cast<const char*>(target_logits);
    q.draft = static_cast<const char*>(draft_logits);
    q.tokens = draft_tokens;
    q.uniforms = uniforms;
    q.out_tokens = out_tokens;
    q.out_accept_len = out_accept_len;
    q.out_row_stats = out_row_stats;
    q.B = B;
    q.V = V;
    q.K = K;
    q.R = 2 * K + 1;
    q.esz = (int)esz;
    q.c = c;
    q.T = temperature;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
    sv::v2::plan(q, sm_count(dev));
    if (q.items >= (int64_t(1) << 31) || B * q.D >= (int64_t(1) << 31)) return SV_ERR_ARG;
    const size_t v2_bytes = align256(sv::v2::scratch_bytes(q));
    const size_t recs_bytes = align256((size_t)B * sizeof(sv::rf::Rec));
    sv::ScratchArea sa;
    const int rc = get(ctx, st, sv::rf::kCtlWords, v2_bytes + recs_bytes, &sa);
    if (rc != SV_OK) return rc;
    if (sa.clear_counters && cudaMemsetAsync(sa.base, 0, sa.data_off, st) != cudaSuccess) return SV_ERR_CUDA;
    q.ctl = reinterpret_cast<uint32_t*>(sa.base);
    q.part = reinterpret_cast<float2*>(sa.base + sa.data_off);
    q.rstat = reinterpret_cast<float4*>(sa.base + sa.data_off);
    q.gz = reinterpret_cast<float*>(sa.base + sa.data_off + sv::v2::part_bytes(q));
    q.rf_ctl = reinterpret_cast<uint32_t*>(sa.base + counter_offset());
    q.rf_recs = reinterpret_cast<sv::rf::Rec*>(sa.base + sa.data_off + v2_bytes);
    if (sv::v2::launch(q, dtype, st) != cudaSuccess) return SV_ERR_CUDA;
    g_launches.fetch_add(2);
    return launch_refine(target_logits, draft_logits, B, K, V, (int)esz, temperature, q.rf_ctl, q.rf_recs, q.ctl + 3,
                         out_tokens, st);
  }
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
  p.G = 0;
  p.N = 0;
  p.RS = limit ? K + 1 : 2 * K + 1;
  p.c = c;
  p.T = temperature;
  p.top_p = top_p;
  p.topp = (!limit && top_p < 1.f) ? 1 : 0;
  // the sequence-in-shared-memory mode has no refine hand-off: only on request
  return run(p, dtype, limit ? sv::kArgmaxLimit : sv::kSample, B * (int64_t)p.RS, st, get, ctx, path == 1);
}

extern "C" int sv_verify_sample(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                                const float* uniforms, int64_t B, int32_t K, int64_t V, int32_t dtype,
                                float temperature, float top_p, int32_t* out_tokens, int32_t* out_accept_len,
                                float* out_row_stats, void* stream) {
  return sv::verify_sample_impl(target_logits, draft_logits, draft_tokens, uniforms, B, K, V, dtype, temperature,
                                top_p, out_tokens, out_accept_len, out_row_stats, static_cast<cudaStream_t>(stream),
                                cached_scratch, nullptr);
}

extern "C" int sv_verify_greedy(const void* logits, const int32_t* cand, int64_t B, int32_t G, int32_t N, int64_t V,
                                int32_t dtype, int32_t* out_tokens, int32_t* out_accept_len, int32_t* out_best_cand,
                                void* stream) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B < 0 || G < 1 || G > 65535 || N < 2 || N > 32767 || V < 2 || V >= kMaxV) return SV_ERR_ARG;
  if ((int64_t)G * N > (1 << 24)) return SV_ERR_ARG;
  if (B == 0) return SV_OK;
  if (!logits || !cand || !out_tokens || !out_accept_len) return SV_ERR_ARG;
  const size_t esz = dtype == SV_BF16 ? 2 : 4;
  if (!aligned_to(logits, esz)) return SV_ERR_DTYPE;
  if (!aligned_to(cand, 4) || !aligned_to(out_tokens, 4) || !aligned_to(out_accept_len, 4) ||
      (out_best_cand && !aligned_to(out_best_cand, 4)))
    return SV_ERR_ARG;
  if (g_greedy_path.load() == 0 && B * (int64_t)G * N < kMaxV) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Scratch sc;
    int dev = 0;
    const int rc = get_scratch(st, 0, (size_t)B * G * N * 4, &sc, &dev);
    if (rc != SV_OK) return rc;
    char* base = static_cast<char*>(sc.base);
    sv::gr::Params q{};
    q.logits = logits;
    q.cand = cand;
    q.B = B;
    q.V = V;
    q.G = G;
    q.N = N;
    q.am = reinterpret_cast<int32_t*>(base + data_offset(sc));
    q.ctl = reinterpret_cast<uint32_t*>(base);
    q.out_tokens = out_tokens;
    q.out_accept_len = out_accept_len;
    q.out_best = out_best_cand;
    if (sv::gr::launch(q, dtype, st) != cudaSuccess) return SV_ERR_CUDA;
    g_launches.fetch_add(2);
    return SV_OK;
  }
  sv::Params p{};
  p.a = static_cast<const char*>(logits);
  p.d = p.a;
  p.tokens = cand;
  p.uniforms = nullptr;
  p.out_tokens = out_tokens;
  p.out_accept_len = out_accept_len;
  p.out_best = out_best_cand;
  p.out_row_stats = nullptr;
  p.B = B;
  p.V = V;
  p.K = 0;
  p.G = G;
  p.N = N;
  p.RS = G * N;
  p.c = 0.f;
  p.T = 0.f;
  p.top_p = 1.f;
  p.topp = 0;
  return run(p, dtype, sv::kGreedy, B * (int64_t)p.RS, static_cast<cudaStream_t>(stream), cached_scratch, nullptr);
}

extern "C" int sv_verify_lookahead_sample(const void* logits, const int32_t* cand, const float* uniforms, int64_t B,
                                          int32_t G, int32_t N, int64_t V, int32_t dtype, float temperature,
                                          int32_t* out_tokens, int32_t* out_accept_len, int32_t* out_best_cand,
                                          float* out_row_lse, void* stream) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B < 0 || B >= kMaxV || V < 2 || V >= kMaxV || !sv::la::fits(G, N)) return SV_ERR_ARG;
  if (B * (int64_t)G * N >= kMaxV) return SV_ERR_ARG;
  if (!(temperature > 0.f) || std::isinf(temperature)) return SV_ERR_ARG;
  if (B == 0) return SV_OK;
  if (!logits || !cand || !uniforms || !out_tokens || !out_accept_len) return SV_ERR_ARG;
  const size_t esz = dtype == SV_BF16 ? 2 : 4;
  if (!aligned_to(logits, esz)) return SV_ERR_DTYPE;
  if (!aligned_to(cand, 4) || !aligned_to(uniforms, 4) || !aligned_to(out_tokens, 4) ||
      !aligned_to(out_accept_len, 4) || (out_best_cand && !aligned_to(out_best_cand, 4)) ||
      (out_row_lse && !aligned_to(out_row_lse, 4)))
    return SV_ERR_ARG;
  const float c = (float)(1.4426950408889634 / (double)temperature);
  if (!std::isfinite(c)) return SV_ERR_ARG;
  const int64_t rows = B * G * N;
  const size_t rowstat_bytes = align256((size_t)rows * 8);
  const size_t gath_bytes = align256((size_t)B * G * (N - 1) * G * 4);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Scratch sc;
  int dev = 0;
  int rc = get_scratch(st, 0, rowstat_bytes + gath_bytes, &sc, &dev);
  if (rc != SV_OK) return rc;
  char* base = static_cast<char*>(sc.base);
  sv::la::Params p{};
  p.logits = logits;
  p.cand = cand;
  p.uniforms = uniforms;
  p.B = B;
  p.V = V;
  p.G = G;
  p.N = N;
  p.c = c;
  p.rowstat = reinterpret_cast<float2*>(base + data_offset(sc));
  p.gath = reinterpret_cast<float*>(base + data_offset(sc) + rowstat_bytes);
  p.ctl = reinterpret_cast<uint32_t*>(base);
  p.out_tokens = out_tokens;
  p.out_accept_len = out_accept_len;
  p.out_best = out_best_cand;
  p.out_row_lse = out_row_lse;
  if (sv::la::launch(p, dtype, st) != cudaSuccess) return SV_ERR_CUDA;
  g_launches.fetch_add(2);
  return SV_OK;
}

extern "C" int sv_verify_multidraft_sample(const void* target, const void* draft, const int32_t* draft_tokens,
                                           const float* uniforms, int64_t B, int32_t G, int32_t N, int64_t V,
                                           int32_t dtype, float temperature, int32_t* out_tokens,
                                           int32_t* out_accept_len, int32_t* out_best_cand, float* out_row_lse,
                                           void* stream) {
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B < 0 || B >= kMaxV || V < 2 || V >= kMaxV || !sv::md::fits(G, N)) return SV_ERR_ARG;
  if (B * (int64_t)G * (2 * N - 1) >= kMaxV) return SV_ERR_ARG;
  if (!(temperature > 0.f) || std::isinf(temperature)) return SV_ERR_ARG;
  if (B == 0) return SV_OK;
  if (!target || !draft || !draft_tokens || !uniforms || !out_tokens || !out_accept_len) return SV_ERR_ARG;
  const size_t esz = dtype == SV_BF16 ? 2 : 4;
  if (!aligned_to(target, esz) || !aligned_to(draft, esz)) return SV_ERR_DTYPE;
  if (!aligned_to(draft_tokens, 4) || !aligned_to(uniforms, 4) || !aligned_to(out_tokens, 4) ||
      !aligned_to(out_accept_len, 4) || (out_best_cand && !aligned_to(out_best_cand, 4)) ||
      (out_row_lse && !aligned_to(out_row_lse, 4)))
    return SV_ERR_ARG;
  const float c = (float)(1.4426950408889634 / (double)temperature);
  if (!std::isfinite(c)) return SV_ERR_ARG;
  const int64_t rows = B * G * (2 * N - 1);
  const size_t rowstat_bytes = align256((size_t)rows * 8);
  const size_t gath_bytes = align256((size_t)B * G * (N - 1) * G * 4);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Scratch sc;
  int dev = 0;
  int rc = get_scratch(st, 0, rowstat_bytes + 2 * gath_bytes, &sc, &dev);
  if (rc != SV_OK) return rc;
  char* base = static_cast<char*>(sc.base);
  sv::md::Params p{};
  p.target = target;
  p.draft = draft;
  p.tokens = draft_tokens;
  p.uniforms = uniforms;
  p.B = B;
  p.V = V;
  p.G = G;
  p.N = N;
  p.c = c;
  p.rowstat = reinterpret_cast<float2*>(base + data_offset(sc));
  p.gp = reinterpret_cast<float*>(base + data_offset(sc) + rowstat_bytes);
  p.gq = reinterpret_cast<float*>(base + data_offset(sc) + rowstat_bytes + gath_bytes);
  p.ctl = reinterpret_cast<uint32_t*>(base);
  p.out_tokens = out_tokens;
  p.out_accept_len = out_accept_len;
  p.out_best = out_best_cand;
  p.out_row_lse = out_row_lse;
  if (sv::md::launch(p, dtype, st) != cudaSuccess) return SV_ERR_CUDA;
  g_launches.fetch_add(2);
  return SV_OK;
}

extern "C" int sv_get_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  Scratch sc;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_scratch.find({dev, reinterpret_cast<uintptr_t>(s)});
    if (it == g_scratch.end()) return SV_OK;
    sc = it->second;
  }
  uint32_t status = 0;
  char* ctl = static_cast<char*>(sc.base);
  if (cudaMemcpy(&status, ctl + 12, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return SV_ERR_CUDA;
  if (status == 0) return SV_OK;
  if (status & 2u) {  // a wait ran out: counters may be left half-way, start clean
    if (cudaMemset(sc.base, 0, sc.bytes) != cudaSuccess) return SV_ERR_CUDA;
    return SV_ERR_TIMEOUT;
  }
  if (cudaMemset(ctl + 12, 0, 4) != cudaSuccess) return SV_ERR_CUDA;
  return SV_ERR_INPUT;
}

extern "C" int sv_selftest_wait_timeout(int64_t limit_ns, void* stream) {
  if (limit_ns < 0 || limit_ns > 2000000000LL) return SV_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Scratch sc;
  int dev = 0;
  const int rc = get_scratch(st, 1, 1, &sc, &dev);
  if (rc != SV_OK) return rc;
  if (sv::launch_wait_selftest(static_cast<uint32_t*>(sc.base), (uint64_t)limit_ns, st) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

extern "C" const char* sv_status_string(int status) {
  switch (status) {
    case SV_OK: return "ok";
    case SV_ERR_ARG: return "invalid argument";
    case SV_ERR_DTYPE: return "unsupported dtype or misaligned logits";
    case SV_ERR_CUDA: return "CUDA runtime error";
    case SV_ERR_INPUT: return "bad input in at least one sequence";
    case SV_ERR_TIMEOUT: return "a bounded device wait ran out";
    case SV_ERR_NOMEM: return "scratch allocation failed";
    case SV_ERR_SCRATCH_LIMIT: return "the call needs more than the fixed no-allocation scratch";
    default: return "unknown status";
  }
}

extern "C" int sv_release(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int rc = SV_OK;
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : g_scratch) {
    if (!kv.second.base) continue;
    cudaSetDevice(kv.first.first);
    cudaDeviceSynchronize();
    if (cudaFree(kv.second.base) != cudaSuccess) rc = SV_ERR_CUDA;
  }
  g_scratch.clear();
  for (auto& kv : g_lm_ws) {
    if (!kv.second.first) continue;
    cudaSetDevice(kv.first.first);
    cudaDeviceSynchronize();
    if (cudaFree(kv.second.first) != cudaSuccess) rc = SV_ERR_CUDA;
  }
  g_lm_ws.clear();
  cudaSetDevice(cur);
  return rc;
}

extern "C" int sv_set_launch_shape(int32_t stages, int32_t ctas_per_sm) {
  if (stages < 0 || stages > sv::kMaxStages || ctas_per_sm < 0 || ctas_per_sm > 4) return SV_ERR_ARG;
  g_stages.store(stages == 0 ? kDefaultStages : stages);
  g_ctas_per_sm.store(ctas_per_sm == 0 ? kDefaultCtasPerSm : ctas_per_sm);
  return SV_OK;
}

extern "C" uint64_t sv_launch_count(void) { return g_launches.load(); }

void sv::note_launches(int n) { g_launches.fetch_add((uint64_t)n); }

extern "C" int sv_set_greedy_path(int32_t path) {
  if (path < 0 || path > 1) return SV_ERR_ARG;
  g_greedy_path.store(path);
  return SV_OK;
}

extern "C" int sv_set_sample_path(int32_t path) {
  if (path < 0 || path > 2) return SV_ERR_ARG;
  g_sample_path.store(path);
  return SV_OK;
}

extern "C" int64_t sv_refined_draws(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  Scratch sc;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_scratch.find({dev, reinterpret_cast<uintptr_t>(s)});
    if (it == g_scratch.end()) return 0;
    sc = it->second;
  }
  uint32_t n = 0;
  if (cudaMemcpy(&n, static_cast<char*>(sc.base) + 4 * kCtlRefined, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return -1;
  return (int64_t)n;
}

namespace {


int lm_workspace(cudaStream_t stream, size_t bytes, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  auto& w = g_lm_ws[{dev, reinterpret_cast<uintptr_t>(stream)}];
  if (w.second < bytes) {
    if (w.first) {
      cudaStreamSynchronize(stream);
      cudaFree(w.first);
      w = {nullptr, 0};
    }
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
      cudaGetLastError();
      return SV_ERR_NOMEM;
    }
    w = {p, bytes};
  }
  *out = w.first;
  return SV_OK;
}

}  // namespace

extern "C" int sv_verify_sample_lmhead(const void* h_target, const void* h_draft, const void* w_target,
                                       const void* w_draft, const int32_t* draft_tokens, const float* uniforms,
                                       int64_t B, int32_t K, int64_t D, int64_t V, float temperature, float top_p,
                                       int32_t* out_tokens, int32_t* out_accept_len, float* out_logits,
                                       void* stream) {
  if (B < 0 || K < 1 || V < 2 || V >= kMaxV || K > (1 << 20) || !sv::lm::fits(D)) return SV_ERR_ARG;
  // the tensor copies address rows and columns with signed 32-bit coordinates
  if (B > (int64_t(1) << 31) || B * (2 * (int64_t)K + 1) >= (int64_t(1) << 31) || D >= (int64_t(1) << 31))
    return SV_ERR_ARG;
  if (!(temperature > 0.f) || std::isinf(temperature)) return SV_ERR_ARG;
  if (!(top_p > 0.f && top_p <= 1.f)) return SV_ERR_ARG;
  if (B == 0) return SV_OK;
  if (!h_target || !h_draft || !w_target || !w_draft || !draft_tokens || !uniforms || !out_tokens ||
      !out_accept_len)
    return SV_ERR_ARG;
  if (!aligned_to(h_target, 16) || !aligned_to(h_draft, 16) || !aligned_to(w_target, 16) || !aligned_to(w_draft, 16))
    return SV_ERR_DTYPE;
  if (out_logits && !aligned_to(out_logits, 16)) return SV_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t mt = B * (K + 1), md = B * (int64_t)K;
  float* logits = out_logits;
  if (!logits) {
    void* w = nullptr;
    const int rc = lm_workspace(st, (size_t)(mt + md) * (size_t)V * sizeof(float), &w);
    if (rc != SV_OK) return rc;
    logits = static_cast<float*>(w);
  }
  // the sticky status word of this stream's scratch
  Scratch sc;
  int dev = 0;
  int rc = get_scratch(st, 1, 1, &sc, &dev);
  if (rc != SV_OK) return rc;
  sv::lm::Params q{};
  q.h[0] = static_cast<const uint16_t*>(h_target);
  q.h[1] = static_cast<const uint16_t*>(h_draft);
  q.w[0] = static_cast<const uint16_t*>(w_target);
  q.w[1] = static_cast<const uint16_t*>(w_draft);
  q.out[0] = logits;
  q.out[1] = logits + mt * V;
  q.Mrows[0] = mt;
  q.Mrows[1] = md;
  q.V = V;
  q.D = D;
  q.status = static_cast<uint32_t*>(sc.base) + 3;
  if (sv::lm::launch(q, st) != cudaSuccess) return SV_ERR_CUDA;
  g_launches.fetch_add(1);
  return sv::verify_sample_impl(q.out[0], q.out[1], draft_tokens, uniforms, B, K, V, SV_F32, temperature, top_p,
                                out_tokens, out_accept_len, nullptr, st, cached_scratch, nullptr);
}
