// sv_lmhead.cu — the LM-head GEMM of the verify on hidden states (sm_103a).
//
// The sampling verify of "Speculative Decoding —— LLM推理优化技术（一）"
// §2.1-2.3 takes the target's and the draft's logits as given; with the
// models' last hidden states h and their LM heads W instead, the logits are
// h · Wᵀ (one row per position, one column per vocabulary entry). This kernel
// computes them on the fifth-generation tensor cores:
//
//  - one CTA per 128 x 128 tile of logits (128 positions x 128 vocabulary
//    entries) of one head (blockIdx.z: 0 target, 1 draft);
//  - the fp32 accumulator lives in tensor memory (128 lanes x 128 columns,
//    allocated by warp 0 with tcgen05.alloc);
//  - per 64-wide slice of the hidden dimension, the CTA stages the h tile and
//    the W tile in shared memory in the canonical no-swizzle K-major layout
//    (8 x 8 core matrices of 128 contiguous bytes), and one thread issues four
//    tcgen05.mma of K = 16 (bf16 inputs, fp32 accumulate) and commits them to
//    an mbarrier that the CTA waits on before it overwrites the tiles;
//  - the epilogue: warp w reads tensor-memory lanes 32w..32w+31 (one position
//    per thread) with tcgen05.ld and writes the fp32 logits.
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
constexpr uint32_t kLBO = 128;                        // K-adjacent core matrices
constexpr uint32_t kSBO = 1024;                       // 8-row groups

// Byte offset of the 16-byte chunk kc (elements 8kc..8kc+7) of row `row` of a
// 128 x 64 bf16 tile in the canonical no-swizzle K-major layout.
__device__ __forceinline__ uint32_t tile_off(int row, int kc) {
  return (uint32_t)(((row >> 3) * 8 + kc) * 128 + (row & 7) * 16);
}

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (all >> 4), the descriptor version of the sm_100 family (bit 46),
// base offset 0, no swizzling.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((kLBO >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((kSBO >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
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

__global__ void __launch_bounds__(kThreads, 4) lmhead_kernel(const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int head = blockIdx.z;
  const int64_t M = p.Mrows[head];
  const int64_t m0 = (int64_t)blockIdx.y * kTileM;
  const int64_t n0 = (int64_t)blockIdx.x * kTileN;
  if (m0 >= M) return;  // the draft head has fewer positions (uniform per CTA, before any allocation)
  const uint16_t* H = p.h[head];
  const uint16_t* W = p.w[head];
  const int64_t V = p.V, D = p.D;
  grid_dependency_sync(true);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"((uint32_t)kTileN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = tmem_base;
  uint8_t* As = smem;
  uint8_t* Bs = smem + kTileBytes;
  const uint32_t a_s = smem_u32(As), b_s = smem_u32(Bs);
  const int nk = (int)(D / kTileK);
  bool ok = true;
  for (int kb = 0; kb < nk; ++kb) {
    // stage the two tiles: 128 rows x 8 chunks of 16 bytes each
#pragma unroll
    for (int i = 0; i < (kTileM * 8) / kThreads; ++i) {
      const int c = tid + i * kThreads;
      const int row = c >> 3, kc = c & 7;
      const int64_t k0 = (int64_t)kb * kTileK + kc * 8;
      uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = make_uint4(0u, 0u, 0u, 0u);
      if (m0 + row < M) va = __ldg(reinterpret_cast<const uint4*>(H + (m0 + row) * D + k0));
      if (n0 + row < V) vb = __ldg(reinterpret_cast<const uint4*>(W + (n0 + row) * D + k0));
      *reinterpret_cast<uint4*>(As + tile_off(row, kc)) = va;
      *reinterpret_cast<uint4*>(Bs + tile_off(row, kc)) = vb;
    }
    proxy_fence_smem();  // the tensor cores read shared memory through the async proxy
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < kTileK / 16; ++j)  // K = 16 per instruction: two core matrices, 256 bytes
        mma_bf16(taddr, smem_desc(a_s + j * 256), smem_desc(b_s + j * 256), kIdesc, (kb > 0 || j > 0) ? 1u : 0u);
      mma_commit(&bar);
    }
    // the MMAs read the tiles: wait for them before the next slice overwrites
    // the tiles (and, after the last slice, before reading the accumulator)
    ok = __syncthreads_and(mbar_wait(&bar, (uint32_t)(kb & 1)));
    if (!ok) break;
  }
  tc_fence_after();
  if (ok) {
    const int64_t m = m0 + warp * 32 + lane;
    float* out = p.out[head] + m * V;
#pragma unroll 1
    for (int c0 = 0; c0 < kTileN; c0 += 32) {
      float v[32];
      tmem_ld32(taddr + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
      if (m < M) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int64_t n = n0 + c0 + k;
          if (n < V) out[n] = v[k];
        }
      }
    }
  } else if (tid == 0) {
    atomicOr(p.status, kStatusTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"((uint32_t)kTileN)
                 : "memory");
  }
}

}  // namespace

bool fits(int64_t D) { return D >= kTileK && D % kTileK == 0; }

cudaError_t launch(const Params& p, cudaStream_t stream) {
  const int64_t mmax = p.Mrows[0] > p.Mrows[1] ? p.Mrows[0] : p.Mrows[1];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.V + kTileN - 1) / kTileN), (unsigned)((mmax + kTileM - 1) / kTileM), 2u);
  cfg.blockDim = dim3(kThreads);
  // two 16 KB tiles; 56 KB keeps at most four CTAs on an SM, so that their
  // tensor-memory allocations (128 columns each) always fit its 512 columns
  cfg.dynamicSmemBytes = 56 * 1024;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaFuncSetAttribute(lmhead_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 56 * 1024);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, lmhead_kernel, p);
}

}  // namespace lm
}  // namespace sv
