// projection_tc.cu -- the input projection on the 5th-generation tensor cores.
//
// P[m][n] = bias[n] + sum_k x16[m][k] * Wx16[n][k] for all m = t*B + b at
// once: the input half of every step does not depend on h_{t-1}, so it is
// taken out of the serial loop as one dense matrix product (work independent
// of the previous step batched across steps: Abstract of "Optimizing
// Performance of Recurrent Neural Networks on GPUs").  x is rounded to fp16 (RNE) by a
// staging kernel into a K-padded buffer; Wx is stored fp16, K-padded, at
// set_weights time; accumulation is fp32 in tensor memory.
//
// One CTA computes one 128 x BN tile of P (BN = 128, 96 or 64, chosen per
// launch so the tiles fill the SMs in as few waves as possible -- at
// M = 1024, N = 1792, 96-wide tiles give exactly one CTA per SM of 152):
//   warp 0 / lane 0  TMA producer: 64-wide K slices of the A (x16) and B (Wx16)
//                    tiles into a 4-stage smem ring (128-byte swizzle),
//                    completion signalled on a per-stage mbarrier;
//   warp 1 / lane 0  MMA issuer: 4 x tcgen05.mma (M=128, N=BN, K=16) per
//                    slice into a TMEM accumulator, tcgen05.commit frees the
//                    slice's stage;
//   warps 0-3        epilogue: tcgen05.ld of the warp's 32 TMEM lanes (rows),
//                    + bias, fp32 stores to P (and the sentinel fill of y).
// Every mbarrier wait is bounded; a timeout sets the status word and the CTA
// still waits for its issued work, frees its TMEM and returns.
//
// In the forward the GEMM is launched as the programmatic dependent of the x
// staging kernel: its launch, TMEM allocation and first weight stages overlap
// the staging, and the producer waits for the staging grid
// (griddepcontrol.wait) before its first x16 load (-2 us of the ~30 us
// projection stage at M = 1024).
//
// The same kernel, without bias and with bf16 operands, computes the weight
// and input gradients of the backward pass (launch_gemm_tc): C[m][n] =
// sum_k A[m][k] * B[n][k] with both operands K-major.
#include <cuda.h>

#include <cstdint>
#include <cstdio>

#include "device_common.cuh"
#include "prnn_internal.h"
#include "tc_common.cuh"

namespace prnn {

namespace {

using namespace tc;

constexpr int BM = 128, BK = 64;
// The projection GEMM starts as the programmatic dependent of the x staging
// kernel (its set-up and first weight stages overlap the staging).
constexpr bool kProjectionPdl = true;
// P written through shared memory by TMA stores (whole 128-byte lines)
// instead of each thread storing its own row of the tile.
constexpr bool kTmaStoreEpilogue = true;
constexpr int kThreads = 128;
constexpr uint32_t kTileA = BM * BK * 2;  // 16 KiB
constexpr long long kWaitNs = 200LL * 1000 * 1000;                   // 200 ms per wait
// Per tile width: B tile bytes, stage bytes (a multiple of 1024, so every
// tile of the ring stays 1024-byte aligned for the 128-byte swizzle), TMEM
// columns (a power of two >= 32 holding the BN fp32 accumulator columns).
// ST: the ring's depth, chosen per launch (see launch_tc).
template <int BN, int ST>
struct TileCfg {
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 128, "tile width");
  static_assert(ST >= 2 && ST <= 8, "ring depth");
  static constexpr uint32_t kTileB = BN * BK * 2;
  static constexpr uint32_t kStageBytes = kTileA + kTileB;
  static constexpr uint32_t kTmemCols = BN <= 64 ? 64 : 128;
  static constexpr int kStages = ST;
  static constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + 1024;  // + alignment slack
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

struct TcKernelArgs {
  int M, N, Kp;
  const float* bias;     // [N] or nullptr (no bias)
  float* P;
  float* y_fill;
  int* status;
  uint32_t idesc;
  int tma_out;           // 1: P written by TMA tensor stores through shared memory (tmC)
};

// Store one 32-float x 128-row block of P from shared memory (128-byte
// swizzled rows) at column c0, row r0; the tensor map clips what lies
// outside P.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0,
                                             int r0) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(r0)
               : "memory");
}

template <int BN, int ST>
__global__ void __launch_bounds__(kThreads, 1)
    proj_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcKernelArgs a) {
  constexpr uint32_t kTileB = TileCfg<BN, ST>::kTileB;
  constexpr uint32_t kStageBytes = TileCfg<BN, ST>::kStageBytes;
  constexpr uint32_t kTmemCols = TileCfg<BN, ST>::kTmemCols;
  constexpr int kStages = TileCfg<BN, ST>::kStages;
  (void)kTileB;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_err;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int nkb = a.Kp / BK;
  // 1024-byte aligned ring of stages: [A tile | B tile] per stage
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&done_bar, 1);
    s_err = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
  const uint64_t deadline = global_ns() + (uint64_t)kWaitNs;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer ----
    // B (the weights) does not depend on the kernel before this one: its
    // first stages are requested before waiting for that kernel (a no-op
    // unless this grid was launched as its programmatic dependent), then A
    const int pre = nkb < kStages ? nkb : kStages;
    for (int kb = 0; kb < pre; ++kb) {
      mbar_arrive_expect_tx(&full_bar[kb], kStageBytes);
      tma_load_2d(base + (uint32_t)kb * kStageBytes + kTileA, &tmB, &full_bar[kb], kb * BK, n0);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int issued = 0;
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % kStages;
      const int round = kb / kStages;
      if (round > 0 && !mbar_wait(&empty_bar[s], (round - 1) & 1, deadline)) {
        atomicExch(&s_err, 1);
        break;
      }
      const uint32_t sa = base + (uint32_t)s * kStageBytes;
      if (kb >= pre) {
        mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
        tma_load_2d(sa + kTileA, &tmB, &full_bar[s], kb * BK, n0);
      }
      tma_load_2d(sa, &tmA, &full_bar[s], kb * BK, m0);
      ++issued;
    }
    // every issued load lands before the CTA may leave
    for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb)
      mbar_wait(&full_bar[kb % kStages], (kb / kStages) & 1, deadline + (uint64_t)kWaitNs);
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    const uint32_t idesc = a.idesc;
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % kStages;
      if (!mbar_wait(&full_bar[s], (kb / kStages) & 1, deadline)) {
        atomicExch(&s_err, 1);
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t sa = base + (uint32_t)s * kStageBytes;
#pragma unroll
      for (int k = 0; k < BK / 16; ++k) {
        // advancing K by 16 fp16 = 32 bytes inside the 128-byte swizzle atom
        const uint64_t adesc = sw128_kmajor_desc(sa + (uint32_t)k * 32u);
        const uint64_t bdesc = sw128_kmajor_desc(sa + kTileA + (uint32_t)k * 32u);
        umma_f16(tmem, adesc, bdesc, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      }
      umma_commit(&empty_bar[s]);  // stage free once these MMAs have read it
    }
    umma_commit(&done_bar);        // accumulator complete (or all issued MMAs retired)
  }

  // ---- epilogue: all four warps, warp w owns TMEM lanes / tile rows 32w..32w+31 ----
  __syncwarp();
  const bool ok = mbar_wait(&done_bar, 0, deadline + (uint64_t)kWaitNs);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (!ok) atomicExch(&s_err, 1);
  __syncthreads();
  const bool good = (s_err == 0);
  if (good && a.tma_out) {
    // The ring is idle once the accumulator is complete: column block j of
    // the tile (32 columns x 128 rows) is staged at base + j * 16 KiB, row r
    // at 128 r bytes with 16-byte chunk c at c ^ (r % 8) (the 128-byte
    // swizzle of the output tensor map), then written by one TMA store.  A
    // warp's 8-lane phases hit 8 different chunks: no bank conflicts.
    const int r = warp * 32 + lane;
#pragma unroll 1
    for (int j = 0; j < BN / 32; ++j) {
      uint32_t v[32];
      tmem_load_32cols(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(j * 32), v);
      const int nb = n0 + j * 32;
      unsigned char* blk = smem_raw + (base - smem_u32(smem_raw)) + (size_t)j * 16384;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float4 o;
        o.x = __uint_as_float(v[4 * c + 0]);
        o.y = __uint_as_float(v[4 * c + 1]);
        o.z = __uint_as_float(v[4 * c + 2]);
        o.w = __uint_as_float(v[4 * c + 3]);
        if (a.bias) {
          const int n = nb + 4 * c;
          o.x += n + 0 < a.N ? __ldg(a.bias + n + 0) : 0.f;
          o.y += n + 1 < a.N ? __ldg(a.bias + n + 1) : 0.f;
          o.z += n + 2 < a.N ? __ldg(a.bias + n + 2) : 0.f;
          o.w += n + 3 < a.N ? __ldg(a.bias + n + 3) : 0.f;
        }
        *reinterpret_cast<float4*>(blk + r * 128 + ((c ^ (r & 7)) << 4)) = o;
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) {
      for (int j = 0; j < BN / 32; ++j) tma_store_2d(&tmC, base + (uint32_t)j * 16384u, n0 + 32 * j, m0);
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    // the sentinel fill of y: row segments, consecutive lanes on consecutive
    // float4s (the fill depends on nothing in the tile)
    if (a.y_fill) {
      const float sv = __uint_as_float(kSentinel);
      const float4 s4 = make_float4(sv, sv, sv, sv);
      constexpr int kQ = BN / 4;
      for (int i = tid; i < BM * kQ; i += kThreads) {
        const int m = m0 + i / kQ, n = n0 + 4 * (i % kQ);
        if (m >= a.M) break;
        float* yrow = a.y_fill + (size_t)m * a.N;
        if (n + 3 < a.N) {
          *reinterpret_cast<float4*>(yrow + n) = s4;
        } else {
          for (int q = 0; q < 4; ++q)
            if (n + q < a.N) yrow[n + q] = sv;
        }
      }
    }
    // the stores must have read the staged tile before the CTA leaves
    if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  } else if (good) {
    const int m = m0 + warp * 32 + lane;
    const bool vec = (a.N & 3) == 0;
#pragma unroll 1
    for (int j = 0; j < BN / 32; ++j) {
      uint32_t r[32];
      tmem_load_32cols(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(j * 32), r);
      const int nb = n0 + j * 32;
      if (m < a.M) {
        float* prow = a.P + (size_t)m * a.N;
        float* yrow = a.y_fill ? a.y_fill + (size_t)m * a.N : nullptr;
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const int n = nb + c;
          if (vec && n + 3 < a.N) {
            const float4 bv = a.bias ? __ldg(reinterpret_cast<const float4*>(a.bias + n))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 o;
            o.x = __uint_as_float(r[c + 0]) + bv.x;
            o.y = __uint_as_float(r[c + 1]) + bv.y;
            o.z = __uint_as_float(r[c + 2]) + bv.z;
            o.w = __uint_as_float(r[c + 3]) + bv.w;
            *reinterpret_cast<float4*>(prow + n) = o;
            if (yrow) {
              const float sv = __uint_as_float(kSentinel);
              *reinterpret_cast<float4*>(yrow + n) = make_float4(sv, sv, sv, sv);
            }
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (n + q < a.N) {
                prow[n + q] = __uint_as_float(r[c + q]) + (a.bias ? __ldg(a.bias + n + q) : 0.f);
                if (yrow) yrow[n + q] = __uint_as_float(kSentinel);
              }
            }
          }
        }
      }
    }
  } else if (tid == 0) {
    report_timeout(a.status, -1, blockIdx.y * gridDim.x + blockIdx.x);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// x [M][K] fp32 -> x16 [M][Kp] fp16 (round to nearest even), zero for k >= K.
// Each thread converts 8 consecutive values: two 16-byte loads when the row
// holds all 8 and rows are 16-byte aligned (K % 4 == 0, x 16-byte aligned),
// else scalar loads.
__global__ void stage_x_f16_kernel(const float* __restrict__ x, __half* __restrict__ x16, int M,
                                   int K, int Kp) {
  // the GEMM launched after this kernel may start its set-up and weight
  // loads now; it waits for this grid's completion before reading x16
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int groups = Kp / 8;
  const size_t total = (size_t)M * groups;
  const bool vec_rows = (K & 3) == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int m = (int)(i / groups), k0 = (int)(i % groups) * 8;
    const float* row = x + (size_t)m * K;
    float v[8];
    if (vec_rows && k0 + 8 <= K) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(row + k0));
      const float4 b = __ldg(reinterpret_cast<const float4*>(row + k0 + 4));
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = k0 + j < K ? row[k0 + j] : 0.f;
    }
    __align__(16) __half h[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) h[j] = __float2half_rn(v[j]);
    *reinterpret_cast<uint4*>(x16 + (size_t)m * Kp + k0) = *reinterpret_cast<const uint4*>(h);
  }
}

// Driver entry point for tensor-map encoding, fetched through the runtime so
// the library needs no link-time dependency on libcuda.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D fp16 (or bf16) K-major map: dims {Kp, rows}, box {64, 128}, 128-byte
// swizzle, out-of-range rows read as zeros.
bool encode_kmajor(CUtensorMap* map, const void* base, int Kp, int rows, int box_rows,
                   bool bf16 = false) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)Kp, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)Kp * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// P [M][N] fp32 as the destination of 32-column x 128-row TMA stores from
// 128-byte swizzled shared memory (needs N % 4 == 0 and a 16-byte aligned P).
bool encode_out(CUtensorMap* map, float* P, int N, int M) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (N & 3) != 0 || (reinterpret_cast<uintptr_t>(P) & 15u) != 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)N * 4};
  const cuuint32_t box[2] = {32, (cuuint32_t)BM};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, P, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool projection_tc_supported() { return encode_fn() != nullptr; }

namespace {

// Tile width for an M x N product: the fewest waves of one CTA per SM, each
// wave costing in proportion to the tile's width (its MMAs and loads).
int sm_count() {
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    sms = 1;
  return sms;
}

int pick_bn(int M, int N, int sms) {
  int best = 128;
  long long best_cost = -1;
  for (int bn : {128, 96, 64}) {
    const long long tiles = (long long)((M + BM - 1) / BM) * ((N + bn - 1) / bn);
    const long long cost = ((tiles + sms - 1) / sms) * bn;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

// after_producer: launch as the programmatic dependent of the kernel before
// it on the stream (that kernel must not write B, P or the y fill)
template <int BN, int ST>
cudaError_t launch_tc_bn(const CUtensorMap& tmA, const CUtensorMap& tmC, const void* Bp, int Kp,
                         int N, bool bf16, const TcKernelArgs& ka, bool after_producer,
                         cudaStream_t s) {
  CUtensorMap tmB;
  if (!encode_kmajor(&tmB, Bp, Kp, N, BN, bf16)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(proj_tc_kernel<BN, ST>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)TileCfg<BN, ST>::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((ka.N + BN - 1) / BN, (ka.M + BM - 1) / BM);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = TileCfg<BN, ST>::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_producer ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, proj_tc_kernel<BN, ST>, tmA, tmB, tmC, ka);
}

cudaError_t launch_tc(const void* A, const void* B, int M, int N, int Kp, bool bf16,
                      TcKernelArgs ka, bool after_producer, cudaStream_t s) {
  CUtensorMap tmA, tmC;
  if (!encode_kmajor(&tmA, A, Kp, M, BM, bf16)) return cudaErrorInvalidValue;
  // the TMA-store epilogue where P's rows allow it; otherwise per-thread row
  // stores (tmC is then unused: any valid map stands in)
  ka.tma_out = kTmaStoreEpilogue && encode_out(&tmC, ka.P, N, M) ? 1 : 0;
  if (!ka.tma_out) tmC = tmA;
  const int sms = sm_count();
  const int bn = pick_bn(M, N, sms);
  ka.idesc = bf16 ? bf16_idesc(BM, bn) : f16_idesc(BM, bn);
  // The ring's depth. With more tiles than SMs a 3-stage ring (97-113 KB)
  // lets two CTAs share an SM, so one CTA's epilogue and prologue hide
  // behind the other's main loop: at M = 8192, K = 4096 the GEMM took 245 us
  // against 303 us with 4 stages (and 566 us with 6). Within one wave the
  // second CTA slot has no tile to run, and 4 stages measured faster there
  // (16.0 against 18.0 us at M = 1024, K = 1792).
  const long long tiles = (long long)((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  const bool multi_wave = tiles > sms;
  switch (bn) {
    case 64:
      return multi_wave ? launch_tc_bn<64, 3>(tmA, tmC, B, Kp, N, bf16, ka, after_producer, s)
                        : launch_tc_bn<64, 4>(tmA, tmC, B, Kp, N, bf16, ka, after_producer, s);
    case 96:
      return multi_wave ? launch_tc_bn<96, 3>(tmA, tmC, B, Kp, N, bf16, ka, after_producer, s)
                        : launch_tc_bn<96, 4>(tmA, tmC, B, Kp, N, bf16, ka, after_producer, s);
    default:
      return multi_wave ? launch_tc_bn<128, 3>(tmA, tmC, B, Kp, N, bf16, ka, after_producer, s)
                        : launch_tc_bn<128, 4>(tmA, tmC, B, Kp, N, bf16, ka, after_producer, s);
  }
}

}  // namespace

cudaError_t launch_projection_tc(const ProjTcArgs& a, int* status, cudaStream_t s) {
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  if (a.Kp % BK != 0 || a.Kp < a.K) return cudaErrorInvalidValue;
  // 1. x -> fp16, K-padded
  {
    const size_t total = (size_t)a.M * (a.Kp / 8);
    const int blocks = (int)((total + 255) / 256 < 8192 ? (total + 255) / 256 : 8192);
    stage_x_f16_kernel<<<blocks, 256, 0, s>>>(a.x, reinterpret_cast<__half*>(a.x16), a.M, a.K,
                                              a.Kp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // 2. tensor-core GEMM
  TcKernelArgs ka{a.M, a.N, a.Kp, a.bias, a.P, a.y_fill, status, 0u, 0};
  return launch_tc(a.x16, a.Wx16, a.M, a.N, a.Kp, false, ka, kProjectionPdl, s);
}

cudaError_t launch_gemm_tc(const GemmTcArgs& g, int* status, cudaStream_t s) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  if (g.Kp % BK != 0) return cudaErrorInvalidValue;
  TcKernelArgs ka{g.M, g.N, g.Kp, nullptr, g.C, nullptr, status, 0u, 0};
  return launch_tc(g.A, g.B, g.M, g.N, g.Kp, g.bf16, ka, false, s);
}

}  // namespace prnn
