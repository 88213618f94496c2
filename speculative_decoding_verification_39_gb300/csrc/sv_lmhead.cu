// sv_lmhead.cu — the LM-head GEMM of the verify on hidden states (sm_103a).
//
// The sampling verify of "Speculative Decoding —— LLM推理优化技术（一）"
// §2.1-2.3 takes the target's and the draft's logits as given; with the
// models' last hidden states h and their LM heads W instead, the logits are
// h · Wᵀ (one row per position, one column per vocabulary entry). This kernel
// computes them on the fifth-generation tensor cores, as D = W_tile · hᵀ:
//
//  - one CTA (256 threads) per 128-entry tile of the vocabulary of one head
//    (blockIdx.y: 0 target, 1 draft); the tile is the MMA's A operand (M =
//    128, one tensor-memory lane per vocabulary entry) and up to 384
//    positions per pass are its B operand (N = 256, then the rest), so that
//    a pass holds every position's accumulator (fp32, 384 of the 512
//    tensor-memory columns) and W is read once;
//  - the hidden dimension goes in 64-wide slices through a ring of three
//    shared-memory stages (the W tile, then up to three 128-row h tiles,
//    each 128 rows x 128 bytes in the 128-byte-swizzled K-major layout that
//    the tensor copy writes). One thread issues the tensor copies
//    (cp.async.bulk.tensor, completing on the stage's "full" mbarrier),
//    another the tcgen05.mma (K = 16 each, bf16 inputs, fp32 accumulate),
//    whose commit frees the stage on its "empty" mbarrier;
//  - with clusters of two CTAs (neighbouring vocabulary tiles, the same
//    positions), each CTA copies half of the h tiles and the copy engine
//    multicasts them into both CTAs' stages, halving the h traffic from L2;
//    a stage is then free once both CTAs' MMAs have read it;
//  - the epilogue: warp w reads tensor-memory lanes 32(w mod 4) .. +31 (one
//    vocabulary entry per thread) 32 positions at a time with tcgen05.ld, and
//    the warp's stores to one position's row are 128 contiguous bytes.
// Every mbarrier wait is bounded; a wait that runs out sets the status word
// and the kernel winds down, freeing its tensor memory.
//
// Products of bf16 values are exact in fp32 and the accumulation is fp32, so
// the logits equal h · Wᵀ up to fp32 summation rounding (exactly, when the
// partial sums are integers below 2^24).
#include <cuda.h>  // CUtensorMap and its enums; the encoder is fetched through the runtime

#include "sv_device.cuh"
#include "sv_lmhead.h"

namespace sv {
namespace lm {
namespace {

constexpr uint32_t kTileBytes = kTileM * kTileK * 2;       // 16 KB: one 128 x 64 bf16 box
constexpr int kMT = 3;                                      // h tiles (128 positions each) per pass
constexpr int kPass = kMT * kTileM;                         // positions per pass
constexpr int kStages = 3;
constexpr uint32_t kStageBytes = kTileBytes * (1 + kMT);    // the W tile, then the h tiles
constexpr uint32_t kTmemCols = 512;                         // the power of two above 384
constexpr int kSmemBytes = (int)(kStages * kStageBytes) + 1024;  // + the 1024-byte alignment

struct Maps {
  CUtensorMap h[2];  // [Mrows, D] per head, 128 x 64 boxes
  CUtensorMap w[2];  // [V, D] per head, 128 x 64 boxes
};

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
// N >> 3 at bits 17-22, M >> 4 at bits 24-28 (M = 128).
__device__ __forceinline__ uint32_t idesc(uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t taddr, uint64_t adesc, uint64_t bdesc, uint32_t id,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(taddr),
      "l"(adesc), "l"(bdesc), "r"(id), "r"(accumulate)
      : "memory");
}
// Arrive (once) on this CTA's mbarrier when every MMA this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// The same on the mbarrier at this offset in every CTA of `mask`.
__device__ __forceinline__ void mma_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// The 128 x 64 box at (x = column, y = row) of `map` into `dst` (1024-byte
// aligned), completing on `bar`; x is a multiple of 64 elements (128 bytes).
__device__ __forceinline__ void tma_load(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// The same box into `dst` of every CTA in `mask`, completing on each one's `bar`.
__device__ __forceinline__ void tma_load_mc(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "h"(mask)
      : "memory");
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

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

// CS: CTAs per cluster: 1, or 2 with the h tiles multicast between them.
template <int CS>
__global__ void __launch_bounds__(kThreads, 1) lmhead_kernel(const __grid_constant__ Maps maps, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t full[kStages], empty[kStages], accb;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int head = blockIdx.y;
  const int64_t M = p.Mrows[head];
  const int64_t n0 = (int64_t)blockIdx.x * kTileM;
  const int64_t V = p.V;
  const uint32_t rank = CS > 1 ? cluster_rank() : 0u;
  const uint16_t mask = (uint16_t)((1u << CS) - 1u);
  const CUtensorMap* hm = &maps.h[head];
  const CUtensorMap* wm = &maps.w[head];
  grid_dependency_sync(true);
  if (M <= 0) return;  // the same for both CTAs of a cluster (one head), before any allocation
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 32) {
    prefetch_map(wm);
    prefetch_map(hm);
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);    // the producer's arrival (plus the stage's bytes)
      mbar_init(&empty[s], CS);  // one MMA commit per CTA of the cluster
    }
    mbar_init(&accb, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  if (CS > 1)
    cluster_sync();  // the peer's barriers are initialised before any copy or commit reaches them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t taddr = tmem_base;
  // the stages on a 1024-byte boundary (the swizzle atom)
  uint8_t* sbase = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sbase);
  const int nk = (int)(p.D / kTileK);
  uint32_t it0 = 0;  // slices of all earlier passes (the position in the stage ring)
  uint32_t pass = 0;
  bool ok = true;    // this thread's waits all ended in time
  for (int64_t mg = 0; mg < M; mg += kPass, it0 += (uint32_t)nk, ++pass) {
    const int rows = (int)min((int64_t)kPass, M - mg);
    const int nt = (rows + kTileM - 1) / kTileM;
    if (warp == 0 && lane == 0) {
      // producer: slice kb of the W tile and the pass's h tiles into stage it % kStages
      for (int kb = 0; kb < nk; ++kb) {
        const uint32_t it = it0 + (uint32_t)kb, s = it % kStages, use = it / kStages;
        if (use > 0 && !mbar_wait(&empty[s], (use - 1u) & 1u)) {
          ok = false;
          break;
        }
        uint8_t* st = sbase + s * kStageBytes;
        mbar_arrive_expect_tx(&full[s], kTileBytes * (uint32_t)(1 + nt));
        tma_load(st, wm, kb * kTileK, (int)n0, &full[s]);
        for (int t = 0; t < nt; ++t) {
          uint8_t* dst = st + (size_t)(1 + t) * kTileBytes;
          const int y = (int)(mg + (int64_t)t * kTileM);
          if (CS == 1)
            tma_load(dst, hm, kb * kTileK, y, &full[s]);
          else if (t % CS == (int)rank)
            tma_load_mc(dst, hm, kb * kTileK, y, &full[s], mask);
        }
      }
    } else if (warp == 1 && lane == 0) {
      // MMA issuer: positions 0..255 of the pass (N = na) to columns 0.., the
      // rest (N = nb) to columns 256..
      const uint32_t na = (uint32_t)min(256, (rows + 15) & ~15);
      const uint32_t nb = rows > 256 ? (uint32_t)((rows - 256 + 15) & ~15) : 0u;
      for (int kb = 0; kb < nk; ++kb) {
        const uint32_t it = it0 + (uint32_t)kb, s = it % kStages, use = it / kStages;
        if (!mbar_wait(&full[s], use & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = sb + s * kStageBytes;
#pragma unroll
        for (int j = 0; j < kTileK / 16; ++j) {  // K = 16 per instruction: 32 bytes of each 128-byte row
          const uint64_t a = smem_desc(st + (uint32_t)j * 32u);
          const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
          mma_bf16(taddr, a, smem_desc(st + kTileBytes + (uint32_t)j * 32u), idesc(na), acc);
          if (nb)
            mma_bf16(taddr + 256u, a, smem_desc(st + kTileBytes + 256u * 128u + (uint32_t)j * 32u), idesc(nb), acc);
        }
        if (CS > 1)
          mma_commit_mc(&empty[s], mask);
        else
          mma_commit(&empty[s]);
      }
      mma_commit(&accb);  // every MMA this pass issued (also after a failed wait)
    }
    __syncwarp();
    const bool got = mbar_wait(&accb, pass & 1u);
    if (!__syncthreads_and(got && ok)) {
      ok = false;
      break;
    }
    tc_fence_after();
    // epilogue: warp w reads lanes 32(w % 4) .. +31 (vocabulary entries) and
    // chunks w / 4, w / 4 + 2, ... of 32 columns (positions)
    const int q = warp & 3;
    const int64_t n = n0 + q * 32 + lane;
    float* out = p.out[head];
    const int nch = (rows + 31) >> 5;
#pragma unroll 1
    for (int ch = warp >> 2; ch < nch; ch += 2) {
      float v[32];
      tmem_ld32(taddr + ((uint32_t)(q * 32) << 16) + (uint32_t)(ch * 32), v);
      if (n < V) {
        const int64_t m0 = mg + (int64_t)ch * 32;
        float* o = out + m0 * V + n;
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (m0 + k < M) o[(int64_t)k * V] = v[k];
      }
    }
    // the accumulators are free for the next pass
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  // Before this CTA exits, every commit (its own and the peer's) has arrived
  // on its barriers: the producer waits for the last use of each stage.
  if (ok && warp == 0 && lane == 0) {
    for (uint32_t it = it0 > (uint32_t)kStages ? it0 - (uint32_t)kStages : 0u; it < it0; ++it) {
      if (!mbar_wait(&empty[it % kStages], (it / kStages) & 1u)) {
        ok = false;
        break;
      }
    }
  }
  tc_fence_before();
  const bool all_ok = __syncthreads_and(ok);
  if (!all_ok && tid == 0) atomicOr(p.status, kStatusTimeout);
  if (CS > 1) cluster_sync();  // no copy or commit of the peer reaches this CTA after it exits
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kTmemCols) : "memory");
  }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver (through the runtime: no link
// against the driver library); null when the driver has none.
EncodeTiled encoder() {
  static const EncodeTiled fn = []() -> EncodeTiled {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<EncodeTiled>(f);
  }();
  return fn;
}

// A row-major [rows, D] bf16 matrix in 128 x 64 boxes, 128-byte swizzle;
// rows past the end read as zeros.
bool encode_rows(CUtensorMap* map, const uint16_t* base, int64_t rows, int64_t D) {
  const EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t dim[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t stride[1] = {(cuuint64_t)D * 2u};
  const cuuint32_t box[2] = {(cuuint32_t)kTileK, (cuuint32_t)kTileM};
  const cuuint32_t estride[2] = {1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dim, stride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_maps(Maps& maps, const Params& p) {
  for (int i = 0; i < 2; ++i) {
    if (p.Mrows[i] <= 0) return false;
    if (!encode_rows(&maps.h[i], p.h[i], p.Mrows[i], p.D) || !encode_rows(&maps.w[i], p.w[i], p.V, p.D))
      return false;
  }
  return true;
}

template <int CS>
cudaError_t launch_cs(const Maps& maps, const Params& p, cudaStream_t stream) {
  const unsigned tiles = (unsigned)((p.V + kTileM - 1) / kTileM);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((tiles + CS - 1) / CS * CS, 2u);  // whole clusters (a tile past V stores nothing)
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;  // one CTA per SM: its 512 tensor-memory columns are always free
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int na = 1;
  if (CS > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CS;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    na = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaFuncSetAttribute(lmhead_kernel<CS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, lmhead_kernel<CS>, maps, p);
}

constexpr int kCluster = 2;  // CTAs per cluster of the product launch

}  // namespace

bool fits(int64_t D) { return D >= kTileK && D % kTileK == 0; }

cudaError_t launch(const Params& p, cudaStream_t stream) {
  Maps maps;
  if (!encode_maps(maps, p)) return cudaErrorNotSupported;
  return launch_cs<kCluster>(maps, p, stream);
}

}  // namespace lm
}  // namespace sv
