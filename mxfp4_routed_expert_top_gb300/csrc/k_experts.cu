// k_experts.cu — the routed-expert kernels: MXFP4 dequant-fused gate/up GEMV
// with SwiGLU epilogue, down GEMV, and the weighted combine.
//
// The operation is the Deltafin README's fused MXFP4 dequant+GEMV ("Techniques
// / Compute": decode the 4-bit weights and multiply in one pass, apply the
// e8m0 scale on the exponent), restated for HBM streaming on sm_103a:
//   * one 16-byte load per lane = one 32-element MX block of one row;
//   * E2M1 pairs decoded in registers by the hardware cvt (e2m1x2 -> f16x2);
//   * the 32 products of a block are summed in fp32 and the block's scale
//     2^(s-127) is applied once to the block sum (exact: a power of two);
//   * x for a lane's block stays in registers across the 32 rows of a group.
#include <cuda_fp16.h>

#include <cuda_bf16.h>

#include "internal.h"

namespace dfm {
namespace {

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
  // 2^(e-127): normal for 1..254, 2^-127 (subnormal) for 0, NaN for 255
  uint32_t bits = e == 0 ? 0x00400000u : (e == 255 ? 0x7FC00000u : e << 23);
  return __uint_as_float(bits);
}

// Four bytes = eight E2M1 codes -> four f16x2 (low nibble in the low half).
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t h) {
  float a, b;
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
      : "=f"(a), "=f"(b)
      : "r"(h));
  return make_float2(a, b);
}

// Sum over the 32 elements of one block: sum_j E2M1(q_j) * x_j (unscaled).
__device__ __forceinline__ float block_dot(const uint4 q, const float (&x)[32]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float d0 = 0.f, d1 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h[4];
    decode_word(w[i], h);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 f = h2_to_f2(h[j]);
      d0 = fmaf(f.x, x[8 * i + 2 * j], d0);
      d1 = fmaf(f.y, x[8 * i + 2 * j + 1], d1);
    }
  }
  return d0 + d1;
}

// Transpose-reduce over the 16 lanes of a half-warp: on entry lane b holds
// v[p] = partial of pair p; on exit v[0] = sum over the 16 lanes of pair b.
__device__ __forceinline__ float halfwarp_transpose_reduce(float (&v)[16],
                                                           int b) {
#pragma unroll
  for (int m = 8, n = 8; m >= 1; m >>= 1, n >>= 1) {
    const bool upper = (b & m) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < n) {
        float send = upper ? v[i] : v[i + n];
        float keep = upper ? v[i + n] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
      }
    }
  }
  return v[0];
}

// One warp: the 16 pairs of group G, chunk c of an MXFP4 matrix in the
// pair-chunk layout, against TG right-hand sides held in registers. On exit
// acc[t][p] holds this lane's partial of pair p (row 2p + r of the group).
template <int TG>
__device__ __forceinline__ void mx_group_chunk(const uint8_t* __restrict__ codes,
                                               const uint8_t* __restrict__ scales,
                                               int K, int G, int c, int lane,
                                               const float (&x)[TG][32],
                                               float (&acc)[TG][16]) {
  const int r = lane >> 4, b = lane & 15;
  const int nbc = mx_nbc(K, c);
#pragma unroll
  for (int t = 0; t < TG; ++t)
#pragma unroll
    for (int p = 0; p < 16; ++p) acc[t][p] = 0.f;
  if (b >= nbc) return;
  const size_t lane_off = (size_t)(c << 9) + (size_t)((r * nbc + b) << 4);
  const uint4 s16 = ldg_stream(scales + (size_t)G * 32 * mx_nb(K) + lane_off);
  const uint32_t sw[4] = {s16.x, s16.y, s16.z, s16.w};
  const uint8_t* cp = codes + (size_t)(16 * G) * K + lane_off;
#pragma unroll
  for (int p0 = 0; p0 < 16; p0 += 8) {
    uint4 q[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) q[u] = ldg_stream(cp + (size_t)(p0 + u) * K);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p = p0 + u;
      const float sc = e8m0_to_f32((sw[p >> 2] >> (8 * (p & 3))) & 0xFFu);
#pragma unroll
      for (int t = 0; t < TG; ++t) acc[t][p] = block_dot(q[u], x[t]) * sc;
    }
  }
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

constexpr int kMaxChunkWarps = 16;  // K up to 8192

// ---------------------------------------------------------------------------
// gate/up: grid (I/16 groups, items). Block = one warp per K-chunk of H.
// Output hbuf[a][16G + p] = silu(g) * u for each assignment a of the item.
// ---------------------------------------------------------------------------
template <int TG>
__global__ void __launch_bounds__(kMaxChunkWarps * 32)
gateup_kernel(const uint8_t* __restrict__ arena, size_t span_bytes, int H,
              int I, int k, const uint16_t* __restrict__ x,
              const Item* __restrict__ items, const int32_t* __restrict__ n_items,
              const int32_t* __restrict__ sorted, float* __restrict__ hbuf) {
  if ((int)blockIdx.y >= *n_items) return;
  const Item it = items[blockIdx.y];
  const int G = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = warp;
  const SpanLayout L = span_layout(H, I);
  const uint8_t* span = arena + (size_t)it.e * span_bytes;
  const int b = lane & 15;
  const bool act = b < mx_nbc(H, c);

  int a_t[TG];
  float xr[TG][32];
#pragma unroll
  for (int t = 0; t < TG; ++t) {
    a_t[t] = t < it.cnt ? sorted[it.pos + t] : -1;
    if (a_t[t] >= 0 && act) {
      const uint16_t* xp = x + (size_t)(a_t[t] / k) * H + (size_t)(16 * c + b) * 32;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        uint4 q = *reinterpret_cast<const uint4*>(xp + 8 * v);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          xr[t][8 * v + 2 * j] = __uint_as_float(w[j] << 16);
          xr[t][8 * v + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) xr[t][j] = 0.f;
    }
  }
  float acc[TG][16];
  mx_group_chunk<TG>(span + L.gu_codes, span + L.gu_scales, H, G, c, lane, xr, acc);

  __shared__ float red[kMaxChunkWarps][kMaxTG][32];
#pragma unroll
  for (int t = 0; t < TG; ++t) {
    float s = halfwarp_transpose_reduce(acc[t], lane & 15);
    red[warp][t][lane] = s;  // lane = 16 r + pair
  }
  __syncthreads();
  const int nw = blockDim.x >> 5;
  for (int o = threadIdx.x; o < TG * 16; o += blockDim.x) {
    const int t = o >> 4, p = o & 15;
    const int a = t < it.cnt ? sorted[it.pos + t] : -1;
    if (a >= 0) {
      float g = 0.f, u = 0.f;
      for (int w = 0; w < nw; ++w) { g += red[w][t][p]; u += red[w][t][16 + p]; }
      hbuf[(size_t)a * I + 16 * G + p] = silu_f(g) * u;
    }
  }
}

// ---------------------------------------------------------------------------
// down: grid (H/32 groups, items). Block = one warp per K-chunk of I.
// Output part[a][32G + 2p + r] = (Wd_e h_a) for each assignment a.
// ---------------------------------------------------------------------------
template <int TG>
__global__ void __launch_bounds__(kMaxChunkWarps * 32)
down_kernel(const uint8_t* __restrict__ arena, size_t span_bytes, int H, int I,
            const Item* __restrict__ items, const int32_t* __restrict__ n_items,
            const int32_t* __restrict__ sorted, const float* __restrict__ hbuf,
            float* __restrict__ part) {
  if ((int)blockIdx.y >= *n_items) return;
  const Item it = items[blockIdx.y];
  const int G = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = warp;
  const SpanLayout L = span_layout(H, I);
  const uint8_t* span = arena + (size_t)it.e * span_bytes;
  const int b = lane & 15;
  const bool act = b < mx_nbc(I, c);

  int a_t[TG];
  float xr[TG][32];
#pragma unroll
  for (int t = 0; t < TG; ++t) {
    a_t[t] = t < it.cnt ? sorted[it.pos + t] : -1;
    if (a_t[t] >= 0 && act) {
      const float4* hp = reinterpret_cast<const float4*>(
          hbuf + (size_t)a_t[t] * I + (size_t)(16 * c + b) * 32);
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        float4 f = hp[v];
        xr[t][4 * v] = f.x; xr[t][4 * v + 1] = f.y;
        xr[t][4 * v + 2] = f.z; xr[t][4 * v + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) xr[t][j] = 0.f;
    }
  }
  float acc[TG][16];
  mx_group_chunk<TG>(span + L.dn_codes, span + L.dn_scales, I, G, c, lane, xr, acc);

  __shared__ float red[kMaxChunkWarps][kMaxTG][32];
#pragma unroll
  for (int t = 0; t < TG; ++t) {
    float s = halfwarp_transpose_reduce(acc[t], lane & 15);
    red[warp][t][lane] = s;
  }
  __syncthreads();
  const int nw = blockDim.x >> 5;
  for (int o = threadIdx.x; o < TG * 32; o += blockDim.x) {
    const int t = o >> 5, l = o & 31;  // l = 16 r + p
    const int a = t < it.cnt ? sorted[it.pos + t] : -1;
    if (a >= 0) {
      float s = 0.f;
      for (int w = 0; w < nw; ++w) s += red[w][t][l];
      const int row = 32 * G + 2 * (l & 15) + (l >> 4);
      part[(size_t)a * H + row] = s;
    }
  }
}

// out[t][j] = residual + sum_i w[t][i] part[t k + i][j] + ysh[t][j]
__global__ void combine_kernel(const float* __restrict__ part,
                               const float* __restrict__ w, int k, int H,
                               const float* __restrict__ ysh,
                               const uint16_t* __restrict__ residual,
                               float* __restrict__ out_f32,
                               uint16_t* __restrict__ out_bf16) {
  const int t = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= H) return;
  float y = 0.f;
  for (int i = 0; i < k; ++i)
    y = fmaf(w[(size_t)t * k + i], part[((size_t)t * k + i) * H + j], y);
  if (ysh) y += ysh[(size_t)t * H + j];
  if (residual) y += __uint_as_float((uint32_t)residual[(size_t)t * H + j] << 16);
  if (out_f32) out_f32[(size_t)t * H + j] = y;
  if (out_bf16) {
    out_bf16[(size_t)t * H + j] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
  }
}

}  // namespace

cudaError_t launch_gateup(const uint8_t* arena, size_t span_bytes, int H,
                          int I, int k, const uint16_t* x, const Item* items,
                          const int32_t* n_items, int max_items,
                          const int32_t* sorted, float* hbuf, int tg,
                          cudaStream_t s) {
  dim3 grid(I / 16, max_items), block(mx_nchunks(H) * 32);
  if (tg == 1)
    gateup_kernel<1><<<grid, block, 0, s>>>(arena, span_bytes, H, I, k, x,
                                            items, n_items, sorted, hbuf);
  else
    gateup_kernel<2><<<grid, block, 0, s>>>(arena, span_bytes, H, I, k, x,
                                            items, n_items, sorted, hbuf);
  return cudaGetLastError();
}

cudaError_t launch_down(const uint8_t* arena, size_t span_bytes, int H, int I,
                        const Item* items, const int32_t* n_items,
                        int max_items, const int32_t* sorted,
                        const float* hbuf, float* part, int tg,
                        cudaStream_t s) {
  dim3 grid(H / 32, max_items), block(mx_nchunks(I) * 32);
  if (tg == 1)
    down_kernel<1><<<grid, block, 0, s>>>(arena, span_bytes, H, I, items,
                                          n_items, sorted, hbuf, part);
  else
    down_kernel<2><<<grid, block, 0, s>>>(arena, span_bytes, H, I, items,
                                          n_items, sorted, hbuf, part);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* part, const float* w, int T, int k,
                           int H, const float* ysh, const uint16_t* residual,
                           float* out_f32, uint16_t* out_bf16, cudaStream_t s) {
  dim3 grid((H + 255) / 256, T);
  combine_kernel<<<grid, 256, 0, s>>>(part, w, k, H, ysh, residual, out_f32,
                                      out_bf16);
  return cudaGetLastError();
}

}  // namespace dfm
