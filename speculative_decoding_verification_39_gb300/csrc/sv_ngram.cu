// sv_ngram.cu — the Lookahead n-gram pool on the GPU ("Lookahead Decoding
// 完全拆解", section "N-gram 池与身份判定"): the n-grams the lookahead branch
// collects (W new ones of N tokens per step), keyed by first token; only those
// whose first token equals the last generated token become candidates for the
// verify branch, at most G of them; n-grams that are not adopted stay.
//
// Layout of a pool of B sequences over a vocabulary of V (caller-owned device
// memory, sv_ngram_pool_bytes bytes):
//   dir   uint32 [B][V]             n-grams ever inserted under each first token
//   slots int32  [B][V][cap][N-1]   ring of the tokens after the first
// Under key k with n = dir[b][k] insertions, the held n-grams are insertions
// max(0, n-cap) .. n-1, insertion i in slot i % cap: inserting into a full key
// overwrites the oldest. An n-gram already held is not inserted again (it
// keeps its place); an n-gram with a token outside [0, V) is ignored.
// Candidates are the newest first.
//
// One warp per sequence, in both kernels: a step's n-grams go in in order, so
// two n-grams of one step under one key see each other.
#include <cstdint>

#include "../../include/specverify.h"
#include "sv_device.cuh"
#include "sv_sample_impl.h"

namespace sv {
namespace ng {
namespace {

constexpr int kWarpsPerCta = 8;

struct Pool {
  uint32_t* dir;
  int32_t* slots;
  int64_t B, V;
  int N, cap;
  __device__ int32_t* slot(int64_t b, int64_t key, int s) const {
    return slots + ((b * V + key) * cap + s) * (int64_t)(N - 1);
  }
};

__global__ void __launch_bounds__(kWarpsPerCta * 32) insert_kernel(Pool P, const int32_t* ngrams, int W) {
  grid_dependency_sync(true);
  const int lane = threadIdx.x & 31;
  const int64_t b = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (b >= P.B) return;
  const int N = P.N, T = N - 1;
  for (int w = 0; w < W; ++w) {
    const int32_t* g = ngrams + (b * W + w) * (int64_t)N;
    int bad = 0;
    for (int t = lane; t < N; t += 32) bad |= (g[t] < 0 || (int64_t)g[t] >= P.V);
    if (__any_sync(0xffffffffu, bad)) continue;
    const int32_t key = g[0];
    uint32_t* dp = P.dir + b * P.V + key;
    const uint32_t n = *reinterpret_cast<volatile uint32_t*>(dp);
    const int held = n < (uint32_t)P.cap ? (int)n : P.cap;
    // is the n-gram already held? lanes compare (entry, token) pairs
    int differs = 0;  // per entry bit, for entries in the lane's pairs
    uint32_t dup = 0;
    for (int h = 0; h < held; ++h) {
      const int32_t* e = P.slot(b, key, (int)((n - 1 - (uint32_t)h) % (uint32_t)P.cap));
      differs = 0;
      for (int t = lane; t < T; t += 32) differs |= (reinterpret_cast<const volatile int32_t*>(e)[t] != g[1 + t]);
      if (!__any_sync(0xffffffffu, differs)) {
        dup = 1;
        break;
      }
    }
    if (dup) continue;
    int32_t* dst = P.slot(b, key, (int)(n % (uint32_t)P.cap));
    for (int t = lane; t < T; t += 32) reinterpret_cast<volatile int32_t*>(dst)[t] = g[1 + t];
    __syncwarp();
    if (lane == 0) *reinterpret_cast<volatile uint32_t*>(dp) = n + 1;
    __threadfence_block();
    __syncwarp();
  }
}

// The same insertions with the step's keys staged in shared memory (W <= 32,
// N <= 33, cap <= 32): one round of loads brings every involved key's count
// and slots and the step's n-grams in, the warp resolves the W n-grams in
// order there (an n-gram sees the ones before it under its key), and one
// round of stores writes back the keys that changed. Per warp, in dynamic
// shared memory (words): cnt[W] | key[W] | tok[W][N] | ent[W][cap][N-1].
__device__ __forceinline__ int stage_words(int W, int N, int cap) { return 2 * W + W * N + W * cap * (N - 1); }

__global__ void __launch_bounds__(kWarpsPerCta * 32) insert_staged_kernel(Pool P, const int32_t* ngrams, int W) {
  extern __shared__ int32_t stage[];
  grid_dependency_sync(true);
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + wib;
  if (b >= P.B) return;
  const int N = P.N, T = N - 1, cap = P.cap;
  int32_t* cnt = stage + (int64_t)wib * stage_words(W, N, cap);
  int32_t* key = cnt + W;
  int32_t* tok = key + W;
  int32_t* ent = tok + W * N;
  // the step's n-grams
  for (int i = lane; i < W * N; i += 32) tok[i] = ngrams[b * (int64_t)W * N + i];
  __syncwarp();
  // lane w: its n-gram's key (-1: some token outside [0, V)) and the first
  // n-gram of the step under the same key (its representative)
  int k = -1, rep = -1;
  if (lane < W) {
    bool ok = true;
    for (int t = 0; t < N; ++t) {
      const int32_t v = tok[lane * N + t];
      ok = ok && v >= 0 && (int64_t)v < P.V;
    }
    k = ok ? tok[lane * N] : -1;
  }
  for (int w = 0; w < W; ++w) {
    const int kw = __shfl_sync(0xffffffffu, k, w);
    if (lane < W && rep < 0 && k >= 0 && kw == k) rep = w;
  }
  if (lane < W) key[lane] = rep == lane ? k : -1;  // only representatives load and store
  __syncwarp();
  // one round of loads: the representatives' counts and slots
  if (lane < W && key[lane] >= 0) cnt[lane] = (int32_t)P.dir[b * P.V + key[lane]];
  for (int i = lane; i < W * cap * T; i += 32) {
    const int r = i / (cap * T), rest = i - r * cap * T;
    if (key[r] >= 0) ent[i] = P.slot(b, key[r], rest / T)[rest % T];
  }
  __syncwarp();
  // in order, in shared memory
  uint32_t dirty = 0;  // representatives whose key changed
  for (int w = 0; w < W; ++w) {
    const int kw = __shfl_sync(0xffffffffu, k, w);
    const int r = __shfl_sync(0xffffffffu, rep, w);
    if (kw < 0) continue;  // an n-gram with a token outside [0, V): ignored
    const uint32_t n = (uint32_t)cnt[r];
    const int held = n < (uint32_t)cap ? (int)n : cap;
    bool dup = false;
    for (int h = 0; h < held && !dup; ++h) {
      const int s = (int)((n - 1 - (uint32_t)h) % (uint32_t)cap);
      const bool differs = lane < T && ent[(r * cap + s) * T + lane] != tok[w * N + 1 + lane];
      dup = !__any_sync(0xffffffffu, differs);
    }
    if (dup) continue;  // already held: it keeps its place
    const int s = (int)(n % (uint32_t)cap);
    if (lane < T) ent[(r * cap + s) * T + lane] = tok[w * N + 1 + lane];
    __syncwarp();
    if (lane == 0) cnt[r] = (int32_t)(n + 1);
    __syncwarp();
    dirty |= 1u << r;
  }
  // one round of stores: the changed keys' slots and counts
  for (int i = lane; i < W * cap * T; i += 32) {
    const int r = i / (cap * T), rest = i - r * cap * T;
    if ((dirty >> r) & 1u) P.slot(b, key[r], rest / T)[rest % T] = ent[i];
  }
  if (lane < W && ((dirty >> lane) & 1u)) P.dir[b * P.V + key[lane]] = (uint32_t)cnt[lane];
}

__global__ void __launch_bounds__(kWarpsPerCta * 32) lookup_kernel(Pool P, const int32_t* last, int G,
                                                                    int32_t* cand, int32_t* count) {
  grid_dependency_sync(true);
  const int lane = threadIdx.x & 31;
  const int64_t b = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (b >= P.B) return;
  const int T = P.N - 1;
  int32_t* out = cand + b * (int64_t)G * T;
  const int32_t key = last[b];
  if (key < 0 || (int64_t)key >= P.V) {
    for (int i = lane; i < G * T; i += 32) out[i] = -1;
    if (lane == 0) count[b] = -1;
    return;
  }
  const uint32_t n = P.dir[b * P.V + key];
  int c = n < (uint32_t)P.cap ? (int)n : P.cap;
  if (c > G) c = G;
  for (int i = lane; i < G * T; i += 32) {
    const int k = i / T, t = i - k * T;
    int32_t v;
    if (c == 0) {
      v = key;  // no candidate: the last token repeated
    } else {
      const int kk = k < c ? k : 0;  // unused slots copy the newest candidate
      v = P.slot(b, key, (int)((n - 1 - (uint32_t)kk) % (uint32_t)P.cap))[t];
    }
    out[i] = v;
  }
  if (lane == 0) count[b] = c;
}

bool shape_ok(int64_t B, int64_t V, int32_t N, int32_t cap) {
  return B >= 0 && V >= 1 && V < ((int64_t)1 << 31) && N >= 2 && N <= 4096 && cap >= 1 && cap <= 4096;
}

Pool make_pool(void* mem, int64_t B, int64_t V, int32_t N, int32_t cap) {
  Pool P;
  P.dir = static_cast<uint32_t*>(mem);
  const size_t dir_bytes = ((size_t)B * V * 4 + 255) / 256 * 256;
  P.slots = reinterpret_cast<int32_t*>(static_cast<char*>(mem) + dir_bytes);
  P.B = B;
  P.V = V;
  P.N = N;
  P.cap = cap;
  return P;
}

cudaError_t launch_pdl(const void* kernel, unsigned grid, void** args, cudaStream_t st, size_t smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWarpsPerCta * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelExC(&cfg, kernel, args);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace
}  // namespace ng
}  // namespace sv

extern "C" int64_t sv_ngram_pool_bytes(int64_t B, int64_t V, int32_t N, int32_t cap) {
  if (!sv::ng::shape_ok(B, V, N, cap)) return -1;
  const int64_t dir = ((int64_t)B * V * 4 + 255) / 256 * 256;
  return dir + (int64_t)B * V * cap * (int64_t)(N - 1) * 4;
}

extern "C" int sv_ngram_pool_reset(void* pool, int64_t B, int64_t V, int32_t N, int32_t cap, void* stream) {
  if (!sv::ng::shape_ok(B, V, N, cap) || (B > 0 && !pool)) return SV_ERR_ARG;
  if (B == 0) return SV_OK;
  // only the insertion counters: slots are never read past them
  const size_t dir = (size_t)B * V * 4;
  return cudaMemsetAsync(pool, 0, dir, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

extern "C" int sv_ngram_pool_insert(void* pool, int64_t B, int64_t V, int32_t N, int32_t cap, const int32_t* ngrams,
                                    int32_t W, void* stream) {
  if (!sv::ng::shape_ok(B, V, N, cap) || W < 0) return SV_ERR_ARG;
  if (B == 0 || W == 0) return SV_OK;
  if (!pool || !ngrams || (reinterpret_cast<uintptr_t>(pool) & 255) || (reinterpret_cast<uintptr_t>(ngrams) & 3))
    return SV_ERR_ARG;
  sv::ng::Pool P = sv::ng::make_pool(pool, B, V, N, cap);
  int W_ = W;
  void* args[] = {&P, &ngrams, &W_};
  const unsigned grid = (unsigned)((B + sv::ng::kWarpsPerCta - 1) / sv::ng::kWarpsPerCta);
  const size_t staged = (size_t)sv::ng::kWarpsPerCta * (size_t)(2 * W + W * N + W * cap * (N - 1)) * 4;
  if (W <= 32 && N <= 33 && cap <= 32 && staged <= 48 * 1024)
    return sv::ng::launch_pdl(reinterpret_cast<const void*>(sv::ng::insert_staged_kernel), grid, args,
                              static_cast<cudaStream_t>(stream), staged) == cudaSuccess
               ? SV_OK
               : SV_ERR_CUDA;
  return sv::ng::launch_pdl(reinterpret_cast<const void*>(sv::ng::insert_kernel), grid, args,
                            static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

extern "C" int sv_ngram_pool_lookup(const void* pool, int64_t B, int64_t V, int32_t N, int32_t cap,
                                    const int32_t* last, int32_t G, int32_t* cand, int32_t* count, void* stream) {
  if (!sv::ng::shape_ok(B, V, N, cap) || G < 1) return SV_ERR_ARG;
  if (B == 0) return SV_OK;
  if (!pool || !last || !cand || !count || (reinterpret_cast<uintptr_t>(pool) & 255) ||
      (reinterpret_cast<uintptr_t>(last) & 3) || (reinterpret_cast<uintptr_t>(cand) & 3) ||
      (reinterpret_cast<uintptr_t>(count) & 3))
    return SV_ERR_ARG;
  sv::ng::Pool P = sv::ng::make_pool(const_cast<void*>(pool), B, V, N, cap);
  int G_ = G;
  void* args[] = {&P, &last, &G_, &cand, &count};
  const unsigned grid = (unsigned)((B + sv::ng::kWarpsPerCta - 1) / sv::ng::kWarpsPerCta);
  return sv::ng::launch_pdl(reinterpret_cast<const void*>(sv::ng::lookup_kernel), grid, args,
                            static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}
