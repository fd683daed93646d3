// k_dense.cu — the shared experts of a batch as two dense bf16 GEMMs on the
// 5th-generation tensor cores (Deltafin analysis §2.1 and §5.1: two shared
// experts added to every token's routed output; SwiGLU as silu(gate) * up,
// then down).
//
//   GEMM 1  [gate; up] (R x H each, R = shared experts x their intermediate)
//           times x (T x H): per 128-row tile 64 gate rows and the matching 64
//           up rows, so that the epilogue forms h = silu(g) * u for its 64
//           intermediate rows, and writes h as three bf16 parts (high,
//           middle, low: 24 significant bits, as fp32 carries) in three B
//           rows per token.
//   GEMM 2  down (H x R) times those rows: the three columns of a token
//           summed in the epilogue = y[t][row].
// bf16 x bf16 products are exact and the accumulators fp32 (tensor memory).
//
// The router logits of a batch run here too (GEMM 3): the fp32 router
// weights are held as three bf16 parts side by side along K ([E][3H]: high,
// middle, low; their sum is the fp32 weight), the K loop walks 3H columns
// with x's column index taken modulo H, so the accumulator sums x . (high +
// middle + low) = x . w with exact products. The K range is split over CTAs
// so that the grid fills the SMs; split s writes its own partial plane
// part[s][t][e], and the top-k kernel sums the planes in order (the same
// sums every run).
//
// One 128 x 96 (GEMM 1: 96 tokens), 128 x 96 (GEMM 2: 32 tokens) or 128 x 128
// (GEMM 3: 128 tokens) output tile per
// CTA, 192 threads: warp 0 loads A and B tiles
// of 64 columns by TMA (128-byte swizzle) into a ring of stages, warp 1
// issues tcgen05.mma (M = 128, N = 128, K = 16) and commits each stage back,
// warps 2-5 read the accumulator (tcgen05.ld; warp w reaches tensor memory
// lanes 32 (w % 4) .. + 31) and write the results. Every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "mxfrag.cuh"
#include "pipeline.cuh"
#include "umma.cuh"

namespace dfm {
namespace {

constexpr int kDM = 128, kDN = 128, kDK = 64;  // tile rows, B rows (columns of D), K per stage
// GEMM 1: 96 tokens a tile (at batch 512, 288 tiles fill 1.9 waves of 152 SMs
// where 128-token tiles left the second of two waves a quarter full)
constexpr int kDN0 = 96;
constexpr int kDN1 = 96;                       // GEMM 2: B rows of 32 tokens x 3 parts
// Stages a CTA: 6 with one CTA an SM, 3 with two (each with half the shared
// and tensor memory, so that one CTA's tile prologue and epilogue overlap the
// other's stream). Grids of more tiles than SMs take two CTAs an SM:
// measured at batch 512 the shared GEMMs went from ~86 to ~61 us each, while
// the router (140 CTAs) and the shared GEMMs of 8 tokens (48-56 tiles) were
// slower with half the stages.
constexpr int kDStagesMax = 6;
constexpr int kDABytes = kDM * kDK * 2;        // 16 KB
constexpr int kDBBytes = kDN * kDK * 2;        // 16 KB
constexpr int kDThr = 6 * 32;
constexpr uint32_t kDCols = 128;               // tensor memory columns: the fp32 accumulator
constexpr int kXsLd = kDN + 1;                 // padded row of the up-value exchange

struct DenseArgs {
  ChunkMap a0, a1;  // A: GEMM 1 gate and up [R][H]; GEMM 2 down [H][R] (a0); GEMM 3 [E][3H]
  ChunkMap b;       // B: GEMM 1 and 3 x [T][H]; GEMM 2 hh [3T][R]
  int mode;         // 0: gate/up, 1: down, 2: router logits
  int K, T, R, H;
  int tiles;        // GEMM 3: output tiles a K split (the grid is tiles x splits)
  int per;          // GEMM 3: K blocks of 64 a split
  int E;            // GEMM 3: experts (rows of A)
  uint16_t* hh;     // GEMM 1 out: [T][3][R] bf16 (high, middle, low)
  float* y;         // GEMM 2 out: [T][H] fp32; GEMM 3 out: [split][T][E] fp32
  uint32_t* err;
};

template <int NS>
struct DSmem {
  uint64_t full[NS], empty[NS], done;
  uint64_t xdone;  // the two up-row warps have handed their values over
  uint32_t tmem;
  int err;
};

template <int NS>
constexpr size_t dense_smem_bytes() {
  return (size_t)NS * (kDABytes + kDBBytes) + sizeof(DSmem<NS>);
}
static_assert(dense_smem_bytes<kDStagesMax>() <= 227 * 1024, "shared memory");
static_assert(2 * (dense_smem_bytes<kDStagesMax / 2>() + 1024) <= 228 * 1024, "two CTAs an SM");
static_assert((size_t)64 * kXsLd * 4 <= (size_t)(kDStagesMax / 2) * kDABytes, "exchange buffer");

__device__ __forceinline__ uint32_t uni_d(uint32_t v) { return __shfl_sync(0xffffffffu, v, 0); }

__device__ __forceinline__ void tma_2d(uint32_t dst, const ChunkMap* map, int x, int y,
                                       uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n\t}" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t bf16_bits(float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&b);
}

template <int NS>
__global__ void __launch_bounds__(kDThr, kDStagesMax / NS) dense_kernel(const __grid_constant__ DenseArgs a) {
  constexpr int kDStages = NS;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sa = smem;
  uint8_t* sb = smem + (size_t)kDStages * kDABytes;
  DSmem<NS>* sm = reinterpret_cast<DSmem<NS>*>(sb + (size_t)kDStages * kDBBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bn = a.mode == 1 ? kDN1 : a.mode == 0 ? kDN0 : kDN;          // B rows of a tile
  const int n_rows = a.mode == 1 ? 3 * a.T : a.T;  // B rows
  const int ntn = (n_rows + bn - 1) / bn;
  const int split = a.mode == 2 ? (int)blockIdx.x / a.tiles : 0;
  const int tile = (int)blockIdx.x - split * (a.mode == 2 ? a.tiles : 0);
  const int mt = tile / ntn, nt = tile - mt * ntn;
  // this CTA's K blocks: kb0 .. kb0 + NK - 1 (GEMM 3: one split; x's column
  // block is the A block modulo the H / 64 blocks of one part)
  const int kb0 = split * (a.mode == 2 ? a.per : 0);
  const int NK = a.mode == 2 ? min(a.per, a.K / kDK - kb0) : a.K / kDK;
  const int xkb = a.H / kDK;

  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm->tmem)),
                 "r"(kDCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < kDStages; ++i) {
      mbar_init(&sm->full[i], 1);
      mbar_init(&sm->empty[i], 1);
    }
    mbar_init(&sm->done, 1);
    mbar_init(&sm->xdone, 2);
    sm->err = 0;
    fence_barrier_init();
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&sm->tmem);
  pdl_wait();

  if (warp == 0) {
    // ---- loads: A (64 gate + 64 up rows, or 128 down rows) and B, 64 columns a stage
    for (int it = 0; it < NK; ++it) {
      const int s = it % kDStages;
      bool ok = it < kDStages || mbar_wait(&sm->empty[s], ((it / kDStages) - 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        sm->err = 1;
        break;
      }
      const uint32_t bar = uni_d(smem_u32(&sm->full[s]));
      const uint32_t da = uni_d(smem_u32(sa + (size_t)s * kDABytes));
      const uint32_t db = uni_d(smem_u32(sb + (size_t)s * kDBBytes));
      if (lane == 0) mbar_arrive_expect_tx(&sm->full[s], kDABytes + bn * kDK * 2);
      __syncwarp();
      if (a.mode == 0) {
        tma_2d(da, &a.a0, kDK * it, 64 * mt, bar);
        tma_2d(da + kDABytes / 2, &a.a1, kDK * it, 64 * mt, bar);
        tma_2d(db, &a.b, kDK * it, bn * nt, bar);
      } else if (a.mode == 1) {
        tma_2d(da, &a.a0, kDK * it, kDM * mt, bar);
        tma_2d(db, &a.b, kDK * it, bn * nt, bar);
      } else {
        const int kb = kb0 + it;
        tma_2d(da, &a.a0, kDK * kb, kDM * mt, bar);
        tma_2d(db, &a.b, kDK * (kb % xkb), bn * nt, bar);
      }
    }
  } else if (warp == 1) {
    // ---- MMAs: four K = 16 steps a stage into the fp32 accumulator
    const uint32_t idesc = umma::idesc_bf16_f32(kDM, bn);
    int it = 0;
    for (; it < NK; ++it) {
      const int s = it % kDStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm->full[s], (it / kDStages) & 1))) {
        sm->err = 1;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint64_t ad = umma::smem_desc_sw128(smem_u32(sa + (size_t)s * kDABytes));
      const uint64_t bd = umma::smem_desc_sw128(smem_u32(sb + (size_t)s * kDBBytes));
      const uint32_t first = it == 0 ? 1u : 0u;
      asm volatile(
          "{\n\t"
          ".reg .pred e, p0, pt;\n\t"
          ".reg .b32 r;\n\t"
          ".reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
          "elect.sync r|e, 0xffffffff;\n\t"
          "setp.eq.u32 p0, %4, 0;\n\t"
          "setp.eq.u32 pt, %4, %4;\n\t"
          "add.u64 a1, %1, 2;\n\tadd.u64 a2, %1, 4;\n\tadd.u64 a3, %1, 6;\n\t"
          "add.u64 b1, %2, 2;\n\tadd.u64 b2, %2, 4;\n\tadd.u64 b3, %2, 6;\n\t"
          "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n\t"
          "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, pt;\n\t"
          "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, pt;\n\t"
          "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, pt;\n\t"
          "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"
          "}" ::"r"(uni_d(tmem)),
          "l"(ad), "l"(bd), "r"(idesc), "r"(first), "r"(uni_d(smem_u32(&sm->empty[s])))
          : "memory");
    }
    if (it == NK) {
      asm volatile(
          "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
          "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
              smem_u32(&sm->done))
          : "memory");
    }
    // the MMAs issued must land before the tensor memory is released
    if (it > 0) (void)mbar_wait(&sm->empty[(it - 1) % kDStages], ((it - 1) / kDStages) & 1);
  } else {
    // ---- epilogue: warps 2-5, row m = tensor memory lane
    const int q = warp & 3, m = 32 * q + lane;
    const bool got = __all_sync(0xffffffffu, mbar_wait(&sm->done, 0));
    if (got) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t d = tmem + ((uint32_t)(32 * q) << 16);
      float* xs = reinterpret_cast<float*>(sa);  // the stages are idle once the MMAs are done
      if (a.mode == 0) {
        // up rows (m >= 64) hand their values to the gate rows (m - 64), in
        // the stage memory the tensor copies wrote last
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (m >= 64) {
          for (int c0 = 0; c0 < kDN0; c0 += 16) {
            uint32_t r[16];
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                "%12,%13,%14,%15}, [%16];"
                : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                  "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                  "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                : "r"(d + (uint32_t)c0));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int i = 0; i < 16; ++i) xs[(m - 64) * kXsLd + c0 + i] = __uint_as_float(r[i]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm->xdone);
        } else if (!__all_sync(0xffffffffu, mbar_wait(&sm->xdone, 0))) {
          sm->err = 1;
        } else {
          const int row = 64 * mt + m;  // intermediate index
          for (int c0 = 0; c0 < kDN0; c0 += 16) {
            uint32_t r[16];
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                "%12,%13,%14,%15}, [%16];"
                : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                  "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                  "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                : "r"(d + (uint32_t)c0));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int t = kDN0 * nt + c0 + i;
              if (t < a.T) {
                const float h = silu_f(__uint_as_float(r[i])) * xs[m * kXsLd + c0 + i];
                const uint32_t hi = bf16_bits(h);
                const float r1 = h - __uint_as_float(hi << 16);  // exact
                const uint32_t mid = bf16_bits(r1);
                const uint32_t lo = bf16_bits(r1 - __uint_as_float(mid << 16));
                uint16_t* dst = a.hh + (size_t)t * 3 * a.R + row;
                dst[0] = (uint16_t)hi;
                dst[a.R] = (uint16_t)mid;
                dst[2 * (size_t)a.R] = (uint16_t)lo;
              }
            }
          }
        }
      } else if (a.mode == 2) {
        // partial logits of this split: lanes are experts (consecutive
        // addresses for a token), columns tokens
        const int e = kDM * mt + m;
        float* dst = a.y + (size_t)split * a.T * a.E;
        for (int c0 = 0; c0 < kDN; c0 += 16) {
          uint32_t r[16];
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
              "%12,%13,%14,%15}, [%16];"
              : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
              : "r"(d + (uint32_t)c0));
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int t = kDN * nt + c0 + i;
            if (t < a.T && e < a.E) dst[(size_t)t * a.E + e] = __uint_as_float(r[i]);
          }
        }
      } else {
        const int row = kDM * mt + m;  // output row of H
        // 48 columns at a time: 16 tokens x (high, middle, low)
        for (int c0 = 0; c0 < kDN1; c0 += 48) {
          uint32_t r[48];
#pragma unroll
          for (int j = 0; j < 3; ++j)
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                "%12,%13,%14,%15}, [%16];"
                : "=r"(r[16 * j + 0]), "=r"(r[16 * j + 1]), "=r"(r[16 * j + 2]),
                  "=r"(r[16 * j + 3]), "=r"(r[16 * j + 4]), "=r"(r[16 * j + 5]),
                  "=r"(r[16 * j + 6]), "=r"(r[16 * j + 7]), "=r"(r[16 * j + 8]),
                  "=r"(r[16 * j + 9]), "=r"(r[16 * j + 10]), "=r"(r[16 * j + 11]),
                  "=r"(r[16 * j + 12]), "=r"(r[16 * j + 13]), "=r"(r[16 * j + 14]),
                  "=r"(r[16 * j + 15])
                : "r"(d + (uint32_t)(c0 + 16 * j)));
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int i = 0; i < 48; i += 3) {
            const int t = (kDN1 * nt + c0 + i) / 3;
            if (t < a.T)
              a.y[(size_t)t * a.H + row] =
                  __uint_as_float(r[i]) + __uint_as_float(r[i + 1]) + __uint_as_float(r[i + 2]);
          }
        }
      }
    } else {
      sm->err = 1;
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (threadIdx.x == 0 && *(volatile int*)&sm->err) atomicOr(a.err, DEV_ERR_TIMEOUT);
  if (warp == 2)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kDCols)
                 : "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 dense_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return encode;
}

// 2-d bf16 [rows][cols] row-major, boxes of 64 columns x box_rows rows,
// 128-byte swizzle; rows past `rows` read as zeros.
bool map_bf16(ChunkMap* out, const void* base, int cols, int rows, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = dense_encoder();
  if (!encode || ((uintptr_t)base & 15) || (cols % 64) || rows <= 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return encode(reinterpret_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The three bf16 parts of fp32 router weights: high = bf16(w), middle =
// bf16(w - high), low = bf16(w - high - middle); both differences are exact
// in fp32, and high + middle + low = w for every finite w whose low part is
// not below the bf16 subnormal range. Row e of `out` holds [high | middle |
// low] (3H columns).
__global__ void router_parts_kernel(const float* __restrict__ w, size_t n, int H,
                                    uint16_t* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t e = i / H, j = i - e * H;
    const float v = w[i];
    const uint32_t hi = bf16_bits(v);
    const float r1 = v - __uint_as_float(hi << 16);
    const uint32_t mid = bf16_bits(r1);
    const uint32_t lo = bf16_bits(r1 - __uint_as_float(mid << 16));
    uint16_t* row = out + e * 3 * (size_t)H;
    row[j] = (uint16_t)hi;
    row[H + j] = (uint16_t)mid;
    row[2 * (size_t)H + j] = (uint16_t)lo;
  }
}

template <int NS>
cudaError_t launch_dense_ns(const DenseArgs& a, int tiles, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(dense_kernel<NS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)dense_smem_bytes<NS>());
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dense_kernel<NS><<<tiles, kDThr, dense_smem_bytes<NS>(), s>>>(a);
  return cudaGetLastError();
}

int dense_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

cudaError_t launch_dense(const DenseArgs& a, int tiles, cudaStream_t s) {
  return tiles > dense_sms() ? launch_dense_ns<kDStagesMax / 2>(a, tiles, s)
                             : launch_dense_ns<kDStagesMax>(a, tiles, s);
}

}  // namespace

bool dense_supported(int H, int R) { return H % kDM == 0 && R % 64 == 0 && R > 0; }

bool make_shared_maps(const uint16_t* gate, const uint16_t* up, const uint16_t* down, int H,
                      int R, const uint16_t* hh, int max_rows, SharedMaps* out) {
  return map_bf16(&out->gate, gate, H, R, 64) && map_bf16(&out->up, up, H, R, 64) &&
         map_bf16(&out->down, down, R, H, kDM) && map_bf16(&out->hh, hh, R, max_rows, kDN1);
}

cudaError_t launch_shared_gemm_gateup(const SharedMaps& m, const uint16_t* x, int T, int H,
                                      int R, uint16_t* hh, uint32_t* err, cudaStream_t s) {
  DenseArgs a{};
  a.a0 = m.gate;
  a.a1 = m.up;
  if (!map_bf16(&a.b, x, H, T, kDN0)) return cudaErrorInvalidValue;
  a.mode = 0;
  a.K = H;
  a.T = T;
  a.R = R;
  a.H = H;
  a.hh = hh;
  a.err = err;
  return launch_dense(a, (R / 64) * ((T + kDN0 - 1) / kDN0), s);
}

cudaError_t launch_shared_gemm_down(const SharedMaps& m, int T, int H, int R, float* y,
                                    uint32_t* err, cudaStream_t s) {
  DenseArgs a{};
  a.a0 = m.down;
  a.a1 = m.down;
  a.b = m.hh;
  a.mode = 1;
  a.K = R;
  a.T = T;
  a.R = R;
  a.H = H;
  a.y = y;
  a.err = err;
  return launch_dense(a, (H / kDM) * ((3 * T + kDN1 - 1) / kDN1), s);
}

// ---- router logits of a batch (GEMM 3) --------------------------------------
int router_tc_splits(int E, int H, int T, int sms, size_t max_rows) {
  if (T < 1) return 0;
  const int tiles = ((E + kDM - 1) / kDM) * ((T + kDN - 1) / kDN);
  const int KB = 3 * H / kDK;
  size_t n = (size_t)std::max(1, sms / tiles);
  n = std::min(n, (size_t)KB);
  if (max_rows) n = std::min(n, max_rows / (size_t)T);
  if (n < 1) return 0;
  const int per = (KB + (int)n - 1) / (int)n;
  return (KB + per - 1) / per;
}

size_t router_tc_part_rows(int E, int H, int Tmin, int Tmax, int sms) {
  size_t rows = 0;
  for (int T = Tmin; T <= Tmax; ++T)
    rows = std::max(rows, (size_t)router_tc_splits(E, H, T, sms, 0) * T);
  return rows;
}

cudaError_t launch_router_parts(const float* w, int E, int H, uint16_t* out, cudaStream_t s) {
  const size_t n = (size_t)E * H;
  const int blocks = (int)std::min<size_t>((n + 255) / 256, 4096);
  router_parts_kernel<<<blocks, 256, 0, s>>>(w, n, H, out);
  return cudaGetLastError();
}

bool make_router_map(const uint16_t* parts, int E, int H, ChunkMap* out) {
  return map_bf16(out, parts, 3 * H, E, kDM);
}

int launch_router_tc(const ChunkMap& map, const uint16_t* x, int T, int E, int H, float* part,
                     size_t max_rows, int sms, uint32_t* err, cudaStream_t s) {
  const int nsplit = router_tc_splits(E, H, T, sms, max_rows);
  if (nsplit < 1) return -1;
  DenseArgs a{};
  a.a0 = map;
  a.a1 = map;
  if (!map_bf16(&a.b, x, H, T, kDN)) return -1;
  a.mode = 2;
  a.K = 3 * H;
  a.T = T;
  a.R = 0;
  a.H = H;
  a.E = E;
  a.tiles = ((E + kDM - 1) / kDM) * ((T + kDN - 1) / kDN);
  const int KB = 3 * H / kDK;
  a.per = (KB + nsplit - 1) / nsplit;
  a.y = part;
  a.err = err;
  return launch_dense(a, a.tiles * nsplit, s) == cudaSuccess ? nsplit : -1;
}

}  // namespace dfm
