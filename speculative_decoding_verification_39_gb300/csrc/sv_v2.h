// sv_v2.h — internal interface of the two-kernel sampling verify
// (sv_rows.cu, sv_decide.cu), used by the C ABI in sv_api.cu and
// sv_noalloc.cu. Not installed; not part of the public ABI.
//
// rows kernel   — one CTA per chunk of a logit row (or per group of short
//                 rows): the chunk's max and sum of 2^(l*c - fl(max*c)), one
//                 read of every logit.
// decide kernel — one thread-block cluster of D CTAs per sequence: combines
//                 the chunk partials into row normalisers, runs the accept
//                 scan, draws the residual or bonus token in fp32 over the
//                 cluster's slices of the row, and redoes the draw in
//                 double-float arithmetic when the fp32 draw lands too close
//                 to a CDF edge to be trusted.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "sv_refine.h"

namespace sv {
namespace v2 {

constexpr int kRowsThreads = 256;
constexpr int kDecideThreads = 256;
constexpr int kMaxK = 1024;         // draft tokens per sequence on this path
constexpr int kCellElems = 256;     // inverse-CDF cell: 32 lanes x 8 elements
constexpr int kMaxCellsPerCta = 512;
constexpr int kMaxCluster = 16;     // CTAs per sequence in the decide kernel (above 8: a non-portable size)
constexpr int kMaxChunks = 64;      // chunks per row
constexpr int kMaxRowsPerItem = 64; // whole short rows per work item of the row pass
// Chunks hold at most this many bytes of a row.
constexpr int64_t kChunkBytes = 32768;

struct Params {
  const char* target;       // [B,K+1,V]
  const char* draft;        // [B,K,V]
  const int32_t* tokens;    // [B,K]
  const float* uniforms;    // [B,K+1]
  int32_t* out_tokens;      // [B,K+1]
  int32_t* out_accept_len;  // [B]
  float* out_row_stats;     // nullable [B,2K+1,4]
  int64_t B, V;
  int K, R;                 // R = 2K+1 rows per sequence
  int esz;                  // 2 (bf16) or 4 (fp32)
  float c;                  // fl(log2(e)/T)
  float c_hi, c_lo;         // log2(e)/T as a double-float
  float T;
  // rows kernel layout: each work item is either one chunk of a row
  // (NCH > 1 or RPI == 1) or a group of RPI whole rows (NCH == 1).
  int64_t CE;               // elements per chunk (V when NCH == 1)
  int NCH;                  // chunks per row
  int RPI;                  // rows per work item (1 unless rows are short)
  int64_t items;            // work items = ceil(B*R / RPI) * NCH
  uint32_t row_slot;        // bytes of a stage per row of a group (RPI > 1)
  uint32_t stage_bytes;     // bytes of one shared-memory stage
  int64_t rows_grid;        // persistent CTAs of the row pass
  float2* part;             // [B*R*NCH] {max raw logit, sum 2^(l*c - fl(max*c))} (top_p == 1)
  // top-p < 1 (bf16 rows): the row pass takes whole rows, one CTA each, and
  // writes each row's statistics whole
  int topp;
  float top_p;
  float4* rstat;            // [B*R] {M, s, cum, tau key as bits} (topp)
  float* gz;                // [B, 2K] raw logit of x_i: target row i at [b*2K + i], draft row i at [b*2K + K + i]
  uint32_t* ctl;            // ctl[3]: sticky status bits
  uint32_t* rf_ctl;         // the refine kernel's control words (zero between calls)
  rf::Rec* rf_recs;         // its list of flagged draws [B]
  // decide kernel
  int D;                    // CTAs per cluster (one cluster per sequence)
  int ncell;                // cells per row = ceil(V / kCellElems)
  int cpr;                  // cells per cluster rank = ceil(ncell / D)
  int dthreads;             // threads per CTA of the decide kernel
  int prefetch;             // copy each CTA's slice of the draw rows into shared memory
  float tab_hi[32], tab_lo[32];  // 2^(i/32) as double-floats
};

// Shapes this path takes (the rest go to the streaming kernel).
bool fits(int64_t K, int64_t V);
// With top-p < 1: bf16 rows whose byte length is a multiple of 16.
bool fits_topp(int64_t K, int64_t V, int esz);
// Fills the layout fields (CE, NCH, RPI, items, stage sizes, grids, D,
// ncell, cpr, the table) from B, K, V, esz, T and the device's SM count.
void plan(Params& p, int sms);
// Scratch bytes: the chunk partials, then the gathered logits.
size_t part_bytes(const Params& p);
size_t scratch_bytes(const Params& p);
// Raises a kernel's dynamic shared-memory limit, once per (kernel, device).
cudaError_t raise_smem_limit_v2(const void* kernel, size_t bytes);
cudaError_t launch(const Params& p, int dtype, cudaStream_t stream);

}  // namespace v2
}  // namespace sv
