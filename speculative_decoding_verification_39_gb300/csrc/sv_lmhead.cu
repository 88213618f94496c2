// sv_lmhead.cu — the LM-head GEMM of the verify on hidden states (sm_103a).
//
// The sampling verify of "Speculative Decoding —— LLM推理优化技术（一）"
// §2.1-2.3 takes the target's and the draft's logits as given; with the
// models' last hidden states h and their LM heads W instead, the logits are
// h · Wᵀ (one row per position, one column per vocabulary entry). This kernel
// computes them on the fifth-generation tensor cores:
//
//  - one CTA (256 threads) per 128-entry tile of the vocabulary of one head
//    (blockIdx.y: 0 target, 1 draft), covering up to 384 positions per pass in
//    three 128 x 128 fp32 accumulators in tensor memory (512 columns,
//    allocated by warp 0 with tcgen05.alloc), so that W is read once;
//  - the hidden dimension goes in 64-wide slices through two shared-memory
//    stages (the W tile, then the h tiles, each 128 rows x 128 bytes in the
//    128-byte-swizzled K-major layout): while one thread issues the slice's
//    tcgen05.mma (K = 16 each, bf16 inputs, fp32 accumulate) and commits them
//    to the stage's mbarrier, every thread loads the next slice into the
//    other stage, waiting (bounded) only for the MMAs that last read it;
//  - the epilogue: warp w reads tensor-memory lanes 32(w mod 4) .. +31 (one
//    position per thread) with tcgen05.ld and writes the fp32 logits.
//
// Products of bf16 values are exact in fp32 and the accumulation is fp32, so
// the logits equal h · Wᵀ up to fp32 summation rounding (exactly, when the
// partial sums are integers below 2^24).
#include "sv_device.cuh"
#include "sv_lmhead.h"

namespace sv {
namespace lm {
namespace {

constexpr uint32_t kTileBytes = kTileM * kTileK * 2;  // 16 KB, the same for the W tile
constexpr int kMT = 3;                                 // M tiles per pass: 3 x 128 TMEM columns
constexpr int kStages = 2;
constexpr uint32_t kStageBytes = kTileBytes * (1 + kMT);  // the W tile, then the h tiles
constexpr uint32_t kTmemCols = 512;                    // the power of two above 3 x 128
constexpr int kChunksPerThread = (1 + kMT) * kTileM * 8 / kThreads;
static_assert((1 + kMT) * kTileM * 8 % kThreads == 0, "whole chunks per thread");
// Byte offset of the 16-byte chunk kc (elements 8kc..8kc+7) of row `row` of a
// 128 x 64 bf16 tile in the 128-byte-swizzled K-major layout: each row is one
// 128-byte line (the whole 64-wide slice), its chunks permuted by XOR with
// (row mod 8), so that the eight rows of an 8-row group, which the tensor
// core reads together, fall on different banks. 8-row groups are 1024 bytes
// apart; the tile starts on a 1024-byte boundary.
__device__ __forceinline__ uint32_t tile_off(int row, int kc) {
  return (uint32_t)(row * 128 + ((kc ^ (row & 7)) << 4));
}

// Shared-memory matrix descriptor of a 128-byte-swizzled K-major operand:
// start address (>> 4; advanced by 32 bytes per K step of 16 inside the
// swizzle atom), leading byte offset 16 (unused by this layout), stride byte
// offset 1024 (the 8-row groups), the descriptor version of the sm_100
// family (bit 46), base offset 0, layout type 2 (128-byte swizzle, bits 61-63).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)(16u >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTileN >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t taddr, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(taddr),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void proxy_fence_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
}

// Chunk c of a stage load: tile t = c / 1024 (0: the W tile, 1..3: h tiles),
// row (c / 8) % 128 of it, 16-byte chunk c % 8 of the 64-wide slice.
__global__ void __launch_bounds__(kThreads, 1) lmhead_kernel(const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t bar[kStages];
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int head = blockIdx.y;
  const int64_t M = p.Mrows[head];
  const int64_t n0 = (int64_t)blockIdx.x * kTileN;
  const uint16_t* H = p.h[head];
  const uint16_t* W = p.w[head];
  const int64_t V = p.V, D = p.D;
  grid_dependency_sync(true);
  if (M <= 0) return;  // (uniform per CTA, before any allocation)
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"((uint32_t)kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = tmem_base;
  // the stages on a 1024-byte boundary (the swizzle atom)
  uint8_t* sbase = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
  const int nk = (int)(D / kTileK);
  uint32_t par[kStages] = {0u, 0u};  // the parity of each barrier's next completion
  bool ok = true;

  for (int64_t mg = 0; mg < M && ok; mg += (int64_t)kMT * kTileM) {
    const int nt = (int)min((int64_t)kMT, (M - mg + kTileM - 1) / kTileM);  // M tiles in this group
    // slice kb of the W tile and the nt h tiles into stage s: every thread
    // loads its 16 chunks first, then stores them (loads in flight together)
    auto load = [&](int kb, int s) {
      uint8_t* st = sbase + (size_t)s * kStageBytes;
      uint4 v[kChunksPerThread];
#pragma unroll
      for (int i = 0; i < kChunksPerThread; ++i) {
        const int c = tid + i * kThreads;
        const int t = c >> 10, row = (c >> 3) & (kTileM - 1), kc = c & 7;
        const int64_t k0 = (int64_t)kb * kTileK + kc * 8;
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (t == 0) {
          if (n0 + row < V) v[i] = __ldg(reinterpret_cast<const uint4*>(W + (n0 + row) * D + k0));
        } else if (t <= nt) {
          const int64_t m = mg + (int64_t)(t - 1) * kTileM + row;
          if (m < M) v[i] = __ldg(reinterpret_cast<const uint4*>(H + m * D + k0));
        }
      }
#pragma unroll
      for (int i = 0; i < kChunksPerThread; ++i) {
        const int c = tid + i * kThreads;
        const int t = c >> 10, row = (c >> 3) & (kTileM - 1), kc = c & 7;
        if (t <= nt) *reinterpret_cast<uint4*>(st + (size_t)t * kTileBytes + tile_off(row, kc)) = v[i];
      }
    };
    load(0, 0);
    proxy_fence_smem();  // the tensor cores read shared memory through the async proxy
    __syncthreads();
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb & 1;
      if (tid == 0) {
        tc_fence_after();
        const uint32_t st = smem_u32(sbase) + (uint32_t)s * kStageBytes;
        for (int t = 0; t < nt; ++t) {
#pragma unroll
          for (int j = 0; j < kTileK / 16; ++j)  // K = 16 per instruction: 32 bytes of each 128-byte row
            mma_bf16(taddr + (uint32_t)(t * kTileN), smem_desc(st + (uint32_t)(t + 1) * kTileBytes + j * 32),
                     smem_desc(st + j * 32), kIdesc, (kb > 0 || j > 0) ? 1u : 0u);
        }
        mma_commit(&bar[s]);
      }
      if (kb + 1 < nk) {
        if (kb >= 1) {
          // stage s ^ 1 was read by the MMAs of slice kb - 1: let them finish
          ok = __syncthreads_and(mbar_wait(&bar[s ^ 1], par[s ^ 1]));
          par[s ^ 1] ^= 1u;
          if (!ok) break;
        }
        load(kb + 1, s ^ 1);
        proxy_fence_smem();
        __syncthreads();
      }
    }
    // the last one or two commits, in order
    for (int kb = (nk >= 2 ? nk - 2 : nk - 1); kb < nk && ok; ++kb) {
      const int s = kb & 1;
      ok = __syncthreads_and(mbar_wait(&bar[s], par[s]));
      par[s] ^= 1u;
    }
    tc_fence_after();
    if (!ok) break;
    // epilogue: warp w reads TMEM lanes 32(w % 4) .. +31 of M tiles w / 4
    // and w / 4 + 2 (one position per thread), 32 columns at a time
    const int q = warp & 3;
    for (int t = warp >> 2; t < nt; t += 2) {
      const int64_t m = mg + (int64_t)t * kTileM + q * 32 + lane;
      float* out = p.out[head] + m * V;
#pragma unroll 1
      for (int c0 = 0; c0 < kTileN; c0 += 32) {
        float v[32];
        tmem_ld32(taddr + ((uint32_t)(q * 32) << 16) + (uint32_t)(t * kTileN + c0), v);
        if (m < M) {
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const int64_t n = n0 + c0 + k;
            if (n < V) out[n] = v[k];
          }
        }
      }
    }
    // the accumulators and stages are free for the next group
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (!ok && tid == 0) atomicOr(p.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"((uint32_t)kTmemCols)
                 : "memory");
  }
}

}  // namespace

bool fits(int64_t D) { return D >= kTileK && D % kTileK == 0; }

cudaError_t launch(const Params& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.V + kTileN - 1) / kTileN), 2u);
  cfg.blockDim = dim3(kThreads);
  // two stages of 64 KB; one CTA per SM, so that its 512 TMEM columns are
  // always free
  const int smem = (int)(kStages * kStageBytes + 1024);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaFuncSetAttribute(lmhead_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, lmhead_kernel, p);
}

}  // namespace lm
}  // namespace sv
