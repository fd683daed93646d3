// k_router.cu — router GEMV, top-k selection with softmax over the selected
// logits, and grouping of token->expert assignments by expert.
//
// "The router picks 16 of the 896 experts; only those are read" (Deltafin
// README, "How it works"; Deltafin analysis §5.1). Selection ties go to the
// lower expert id; ids come out in descending logit order.
#include <math.h>

#include "internal.h"

namespace dfm {
namespace {

constexpr int kRouterRowsPerBlock = 8;  // one warp per row
constexpr int kRouterTT = 8;            // tokens per smem tile

// part[split][t][e] = sum over the split's K range of Wr[e][j] x[t][j]
__global__ void __launch_bounds__(256)
router_kernel(const float* __restrict__ Wr, int E, int H,
              const uint16_t* __restrict__ x, int T, float* __restrict__ part,
              int split_len) {
  extern __shared__ float xs[];  // [kRouterTT][split_len]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterRowsPerBlock + warp;
  const int split = blockIdx.y;
  const int k0 = split * split_len;
  const int len = min(split_len, H - k0);
  for (int t0 = 0; t0 < T; t0 += kRouterTT) {
    const int tt = min(kRouterTT, T - t0);
    __syncthreads();
    for (int i = threadIdx.x; i < tt * len; i += blockDim.x) {
      const int t = i / len, j = i - t * len;
      xs[t * split_len + j] =
          __uint_as_float((uint32_t)x[(size_t)(t0 + t) * H + k0 + j] << 16);
    }
    __syncthreads();
    if (e < E) {
      float acc[kRouterTT];
#pragma unroll
      for (int t = 0; t < kRouterTT; ++t) acc[t] = 0.f;
      const float* wr = Wr + (size_t)e * H + k0;
      for (int j = 4 * lane; j < len; j += 128) {
        const float4 w4 = __ldg(reinterpret_cast<const float4*>(wr + j));
#pragma unroll
        for (int t = 0; t < kRouterTT; ++t) {
          if (t < tt) {
            const float4 x4 = *reinterpret_cast<const float4*>(xs + t * split_len + j);
            acc[t] = fmaf(w4.x, x4.x, acc[t]);
            acc[t] = fmaf(w4.y, x4.y, acc[t]);
            acc[t] = fmaf(w4.z, x4.z, acc[t]);
            acc[t] = fmaf(w4.w, x4.w, acc[t]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kRouterTT; ++t) {
        float v = acc[t];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0 && t < tt)
          part[((size_t)split * T + t0 + t) * E + e] = v;
      }
    }
  }
}

__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
  return v > bv || (v == bv && e < be);
}

// One block of 128 threads per token: sum the split partials (fixed order),
// then warp 0 selects the top k and the softmax weights.
__global__ void __launch_bounds__(128)
topk_kernel(const float* __restrict__ part, int nsplit, int T, int E, int k,
            float* __restrict__ logits_out, int32_t* __restrict__ ids,
            float* __restrict__ w, Item* items, int32_t* n_items,
            int32_t* sorted) {
  __shared__ float lg[1024];
  const int t = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float v = 0.f;
    for (int s = 0; s < nsplit; ++s) v += part[((size_t)s * T + t) * E + e];
    lg[e] = v;
    if (logits_out) logits_out[(size_t)t * E + e] = v;
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  float sel_v = 0.f;
  int sel_e = 0;
  for (int i = 0; i < k; ++i) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const float v = lg[e];
      if (better(v, e, bv, be)) { bv = v; be = e; }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (better(ov, oe, bv, be)) { bv = ov; be = oe; }
    }
    if (lane == i) { sel_v = bv; sel_e = be; }
    __syncwarp();
    if (lane == 0) lg[be] = -INFINITY;
    __syncwarp();
  }
  const float vmax = __shfl_sync(0xffffffffu, sel_v, 0);
  const float ex = lane < k ? expf(sel_v - vmax) : 0.f;
  float z = ex;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane < k) {
    ids[(size_t)t * k + lane] = sel_e;
    w[(size_t)t * k + lane] = ex / z;
    if (items && T == 1) {
      items[lane] = Item{sel_e, lane, 1, 0};
      sorted[lane] = lane;
    }
  }
  if (items && T == 1 && lane == 0) *n_items = k;
}

// Block-wide exclusive scan of one value per thread (blockDim.x <= 1024).
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  __syncthreads();
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    if (lane < nw) warp_sums[lane] = s;  // inclusive warp prefix
  }
  __syncthreads();
  const int base = warp ? warp_sums[warp - 1] : 0;
  if (total) *total = warp_sums[(blockDim.x >> 5) - 1];
  return base + incl - v;
}

// Single block of 1024 threads. Counting sort of the T*k assignments by
// expert; each expert's segment is then put in ascending assignment order,
// so the result does not depend on atomic ordering.
__global__ void __launch_bounds__(1024)
group_kernel(const int32_t* __restrict__ ids, int T, int k, int E,
             int32_t* offs, int32_t* tok, int32_t* slot, int32_t* n_union,
             Item* items, int32_t* n_items, int32_t* sorted, int tg) {
  __shared__ int cnt[1024];
  __shared__ int fill[1024];
  __shared__ int warp_sums[32];
  __shared__ int tot;
  const int tid = threadIdx.x;
  const int A = T * k;
  cnt[tid] = 0;
  __syncthreads();
  for (int a = tid; a < A; a += blockDim.x) atomicAdd(&cnt[ids[a]], 1);
  __syncthreads();
  const int c = tid < E ? cnt[tid] : 0;
  const int start = block_exclusive_scan(c, warp_sums, nullptr);
  if (tid < E) {
    fill[tid] = start;
    if (offs) offs[tid] = start;
  }
  if (tid == 0 && offs) offs[E] = A;
  __syncthreads();
  for (int a = tid; a < A; a += blockDim.x) {
    const int p = atomicAdd(&fill[ids[a]], 1);
    sorted[p] = a;
  }
  __syncthreads();
  __threadfence_block();
  // order each segment by assignment index (insertion sort, one thread each)
  if (tid < E) {
    for (int i = start + 1; i < start + c; ++i) {
      const int v = sorted[i];
      int j = i - 1;
      while (j >= start && sorted[j] > v) { sorted[j + 1] = sorted[j]; --j; }
      sorted[j + 1] = v;
    }
  }
  __syncthreads();
  if (tok) {
    for (int p = tid; p < A; p += blockDim.x) {
      tok[p] = sorted[p] / k;
      slot[p] = sorted[p] % k;
    }
  }
  // work items: ceil(count / tg) per expert, in expert order
  const int ni = (c + tg - 1) / tg;
  const int ibase = block_exclusive_scan(ni, warp_sums, &tot);
  if (tid < E) {
    for (int q = 0; q < ni; ++q)
      items[ibase + q] = Item{tid, start + q * tg, min(tg, c - q * tg), 0};
  }
  const int nz = block_exclusive_scan(c > 0 ? 1 : 0, warp_sums, nullptr);
  __syncthreads();
  if (tid == 0) *n_items = tot;
  if (tid == E - 1 && n_union) *n_union = nz + (c > 0 ? 1 : 0);
}

}  // namespace

cudaError_t launch_router(const float* Wr, int E, int H, const uint16_t* x,
                          int T, float* part, RouterSplit sp, cudaStream_t s) {
  const int split_len = sp.split_len;
  const size_t smem = (size_t)kRouterTT * split_len * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(router_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((E + kRouterRowsPerBlock - 1) / kRouterRowsPerBlock, sp.nsplit);
  router_kernel<<<grid, 256, smem, s>>>(Wr, E, H, x, T, part, split_len);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* part, int nsplit, int T, int E, int k,
                        float* logits_out, int32_t* ids, float* w, Item* items,
                        int32_t* n_items, int32_t* sorted, cudaStream_t s) {
  topk_kernel<<<T, 128, 0, s>>>(part, nsplit, T, E, k, logits_out, ids, w,
                                items, n_items, sorted);
  return cudaGetLastError();
}

cudaError_t launch_group(const int32_t* ids, int T, int k, int E,
                         int32_t* offs, int32_t* tok, int32_t* slot,
                         int32_t* n_union, Item* items, int32_t* n_items,
                         int32_t* sorted, int tg, cudaStream_t s) {
  group_kernel<<<1, 1024, 0, s>>>(ids, T, k, E, offs, tok, slot, n_union,
                                  items, n_items, sorted, tg);
  return cudaGetLastError();
}

}  // namespace dfm
