// k_shared.cu — bf16 shared-expert GEMVs and RMSNorm.
//
// The shared experts run for every token next to the routed ones ("add the
// two shared experts", Deltafin analysis §5.1). Their n_shared gate/up
// matrices are concatenated along rows and their down matrices along
// columns, so the shared part is one SwiGLU FFN of intermediate n_shared*Is.
#include <cuda_bf16.h>

#include "internal.h"

namespace dfm {
namespace {

constexpr int kSharedTT = 8;  // tokens per smem tile

__device__ __forceinline__ void bf16x8_to_f32(uint4 q, float (&f)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Each warp: intermediate rows i0, i0+1 (gate and up) over all of H.
// hsh[t][i] = silu(gate_i . x_t) * (up_i . x_t)
__global__ void __launch_bounds__(256)
shared_gateup_kernel(const uint16_t* __restrict__ gate,
                     const uint16_t* __restrict__ up, int R, int H,
                     const uint16_t* __restrict__ x, int T,
                     float* __restrict__ hsh) {
  extern __shared__ uint16_t xs16[];  // [kSharedTT][H] bf16
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i0 = (blockIdx.x * 8 + warp) * 2;
  for (int t0 = 0; t0 < T; t0 += kSharedTT) {
    const int tt = min(kSharedTT, T - t0);
    __syncthreads();
    for (int v = threadIdx.x; v < tt * H / 8; v += blockDim.x)
      reinterpret_cast<uint4*>(xs16)[v] =
          reinterpret_cast<const uint4*>(x + (size_t)t0 * H)[v];
    __syncthreads();
    if (i0 >= R) continue;
    float acc[4][kSharedTT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int t = 0; t < kSharedTT; ++t) acc[r][t] = 0.f;
    const uint16_t* rows[4] = {gate + (size_t)i0 * H, gate + (size_t)(i0 + 1) * H,
                               up + (size_t)i0 * H, up + (size_t)(i0 + 1) * H};
    for (int j = 8 * lane; j < H; j += 256) {
      float wf[4][8];
#pragma unroll
      for (int r = 0; r < 4; ++r)
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(rows[r] + j)), wf[r]);
#pragma unroll
      for (int t = 0; t < kSharedTT; ++t) {
        if (t < tt) {
          float xf[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(xs16 + t * H + j), xf);
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[r][t] = fmaf(wf[r][q], xf[q], acc[r][t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kSharedTT; ++t) {
      if (t < tt) {
        const float g0 = warp_sum(acc[0][t]), g1 = warp_sum(acc[1][t]);
        const float u0 = warp_sum(acc[2][t]), u1 = warp_sum(acc[3][t]);
        if (lane == 0) {
          hsh[(size_t)(t0 + t) * R + i0] = silu_f(g0) * u0;
          hsh[(size_t)(t0 + t) * R + i0 + 1] = silu_f(g1) * u1;
        }
      }
    }
  }
}

// Each warp: 4 rows of down [H][K] over all of K. ysh[t][row] = down_row . h_t
__global__ void __launch_bounds__(256)
shared_down_kernel(const uint16_t* __restrict__ down, int H, int K,
                   const float* __restrict__ hsh, int T,
                   float* __restrict__ ysh) {
  extern __shared__ float hs[];  // [kSharedTT][K]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = (blockIdx.x * 8 + warp) * 4;
  for (int t0 = 0; t0 < T; t0 += kSharedTT) {
    const int tt = min(kSharedTT, T - t0);
    __syncthreads();
    for (int v = threadIdx.x; v < tt * K / 4; v += blockDim.x)
      reinterpret_cast<float4*>(hs)[v] =
          reinterpret_cast<const float4*>(hsh + (size_t)t0 * K)[v];
    __syncthreads();
    if (r0 >= H) continue;
    float acc[4][kSharedTT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int t = 0; t < kSharedTT; ++t) acc[r][t] = 0.f;
    for (int j = 8 * lane; j < K; j += 256) {
      float wf[4][8];
#pragma unroll
      for (int r = 0; r < 4; ++r)
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(down + (size_t)(r0 + r) * K + j)),
                      wf[r]);
#pragma unroll
      for (int t = 0; t < kSharedTT; ++t) {
        if (t < tt) {
          const float4 h0 = *reinterpret_cast<const float4*>(hs + t * K + j);
          const float4 h1 = *reinterpret_cast<const float4*>(hs + t * K + j + 4);
          const float hf[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[r][t] = fmaf(wf[r][q], hf[q], acc[r][t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kSharedTT; ++t) {
      if (t < tt) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float v = warp_sum(acc[r][t]);
          if (lane == 0) ysh[(size_t)(t0 + t) * H + r0 + r] = v;
        }
      }
    }
  }
}

// xn = RNE_bf16(x / sqrt(mean(x^2) + eps)); one block per token.
__global__ void __launch_bounds__(256)
rmsnorm_kernel(const uint16_t* __restrict__ x, int H, float eps,
               uint16_t* __restrict__ xn) {
  __shared__ float ws[8];
  const int t = blockIdx.x;
  const uint16_t* xr = x + (size_t)t * H;
  float ss = 0.f;
  for (int j = threadIdx.x; j < H; j += blockDim.x) {
    const float v = __uint_as_float((uint32_t)xr[j] << 16);
    ss = fmaf(v, v, ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += ws[w];
  const float denom = sqrtf(tot / (float)H + eps);
  for (int j = threadIdx.x; j < H; j += blockDim.x) {
    const float v = __uint_as_float((uint32_t)xr[j] << 16);
    xn[(size_t)t * H + j] = __bfloat16_as_ushort(__float2bfloat16_rn(v / denom));
  }
}

}  // namespace

cudaError_t launch_shared_gateup(const uint16_t* gate, const uint16_t* up,
                                 int R, int H, const uint16_t* x, int T,
                                 float* hsh, cudaStream_t s) {
  const size_t smem = (size_t)kSharedTT * H * sizeof(uint16_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(
        shared_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int warps = (R + 1) / 2;
  shared_gateup_kernel<<<(warps + 7) / 8, 256, smem, s>>>(gate, up, R, H, x, T, hsh);
  return cudaGetLastError();
}

cudaError_t launch_shared_down(const uint16_t* down, int H, int K,
                               const float* hsh, int T, float* ysh,
                               cudaStream_t s) {
  const size_t smem = (size_t)kSharedTT * K * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(
        shared_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int warps = (H + 3) / 4;
  shared_down_kernel<<<(warps + 7) / 8, 256, smem, s>>>(down, H, K, hsh, T, ysh);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const uint16_t* x, int T, int H, float eps,
                           uint16_t* xn, cudaStream_t s) {
  rmsnorm_kernel<<<T, 256, 0, s>>>(x, H, eps, xn);
  return cudaGetLastError();
}

}  // namespace dfm
