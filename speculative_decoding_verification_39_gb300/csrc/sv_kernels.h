// sv_kernels.h — internal interface between the C ABI (sv_api.cu) and the
// kernels (sv_kernels.cu). Not installed; not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "sv_refine.h"

namespace sv {

enum Mode { kSample = 0, kArgmaxLimit = 1, kGreedy = 2 };
constexpr int kMaxStages = 6;  // 6 x 32 KB + control stays under the 227 KB a CTA may use
constexpr int kTileBytes = 32768;  // one ring stage holds one tile

constexpr int kMaxCells = 1024;    // inverse-CDF cells per row

// Elements per inverse-CDF cell: 256 * m, the fewest that keep a row of V
// elements within kMaxCells cells.
__host__ __device__ inline int64_t cell_elems(int64_t V) {
  const int64_t m = (V + 256LL * kMaxCells - 1) / (256LL * kMaxCells);
  return 256 * (m > 1 ? m : 1);
}

// Cells of a residual draw (two rows) that fit one half of a ring of
// `stages` tiles: the unit of work of a draw split over CTAs.
inline int64_t draw_cells_per_chunk(int stages, int esz, int64_t V) {
  const int64_t half = ((int64_t)stages * kTileBytes / 2) & ~int64_t(15);
  return half / 2 / esz / cell_elems(V);
}

struct Params {
  const char* a;           // target logits [B,K+1,V] (sampling) or logits [B,G,N,V] (greedy)
  const char* d;           // draft logits [B,K,V] (sampling, T > 0)
  const int32_t* tokens;   // draft tokens [B,K] or candidates [B,G,N-1]
  const float* uniforms;   // [B,K+1]
  int32_t* out_tokens;
  int32_t* out_accept_len;
  int32_t* out_best;       // nullable (greedy)
  float* out_row_stats;    // nullable (sampling)
  int64_t B, V;
  int K, G, N;
  int RS;                  // rows per sequence
  int64_t NT;              // tiles per row
  int64_t TE;              // elements per tile
  int64_t CT;              // tiles per chunk (the unit of scheduling)
  int64_t NC;              // chunks per row = ceil(NT / CT)
  int64_t W;               // chunks in the call = B * RS * NC
  float c;                 // log2(e) / T
  float T;
  float top_p;
  int topp;                // top_p < 1
  uint32_t* ctl;           // [0..1] work counter (u64), [2] finished producers, [3] status bits,
                           // [4] tails queued, [5] tails taken, [6] finished CTAs, [8] never set
  uint32_t* row_cnt;       // [B*RS] chunks published per row
  uint32_t* seq_cnt;       // [B] rows finished per sequence
  uint32_t* tail_q;        // [B * max(1, DC)] queued sequence tails or draw chunks (0 = empty)
  float2* part;            // [W] per-chunk partials
  float4* rowstat;         // [B*RS] per-row results
  int stages;
  // Draws split over CTAs (sampling mode, T > 0): DC chunks of CPC cells per
  // sequence; 0 = each sequence's tail draws alone.
  int DC;
  int CPC;
  float* dcells;           // [B][kMaxCells] cell sums
  uint32_t* dcnt;          // [B] chunks done
  // Draws the fp32 walk cannot settle go to the refine kernel's list (null:
  // the greedy modes, which draw nothing).
  uint32_t* rf_ctl;
  rf::Rec* rf_recs;
};

size_t shared_bytes(int stages);
cudaError_t launch(const Params& p, int dtype, int mode, int grid, cudaStream_t stream);

// Sampling mode for short rows: one CTA per sequence, the whole sequence
// staged in shared memory. seq_mode_fits() says whether a shape qualifies
// (2K+1 <= 64 rows, the sequence within 48 KB, rows 16-byte aligned).
bool seq_mode_fits(int64_t K, int64_t V, int esz);
// Sampling mode for rows of at most 1024 elements: one warp per sequence,
// from global memory (2K+1 <= 64 rows, the sequence within 64 KB, rows
// 16-byte aligned).
bool warp_mode_fits(int64_t K, int64_t V, int esz);
cudaError_t launch_warp(const Params& p, int dtype, int grid, cudaStream_t stream);
int warp_mode_seqs_per_cta();

// A control word no kernel ever writes (the self-test waits for it).
constexpr int kCtlNeverSet = 8;
// Self-test of the bounded waits: a one-thread kernel that waits limit_ns for
// ctl[kCtlNeverSet] and then records a timeout in ctl[3].
cudaError_t launch_wait_selftest(uint32_t* ctl, uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_seq(const Params& p, int dtype, int grid, cudaStream_t stream);
int kernel_threads();

}  // namespace sv
