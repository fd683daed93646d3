// select.cuh — top-k selection of one token's logits by a thread block:
// bitonic sorting networks on warp shuffles.
//
// Each token's router chooses 16 of the 896 experts, and only the chosen
// experts' weights are touched (Deltafin README, "How it works"). Order:
// larger logit first, equal logits by lower expert id, so the selection
// equals a full sort of the logits.
#pragma once

#include <math.h>
#include <stdint.h>

namespace dfm {

__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
  return v > bv || (v == bv && e < be);
}

// ---- top-k by bitonic sorting networks on warp shuffles ----
// Order: larger logit first, equal logits by lower expert id. Padding entries
// are (-inf, INT_MAX). A warp holds a list of 32 entries, one per lane.

// Compare-exchange with lane ^ mask: keep the better entry of the pair if
// `keep_better`, else the worse one.
__device__ __forceinline__ void bitonic_cas(float& v, int& e, int mask, bool keep_better) {
  const float ov = __shfl_xor_sync(0xffffffffu, v, mask);
  const int oe = __shfl_xor_sync(0xffffffffu, e, mask);
  if (better(ov, oe, v, e) == keep_better) { v = ov; e = oe; }
}

// Sorts L independent 32-entry lists (one entry per lane each), best first.
template <int L>
__device__ __forceinline__ void warp_sort32(float (&v)[L], int (&e)[L]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      // runs of `size` lanes alternate direction until the last stage
      const bool best_first = (lane & size) == 0 || size == 32;
      const bool keep_better = ((lane & stride) == 0) == best_first;
#pragma unroll
      for (int j = 0; j < L; ++j) bitonic_cas(v[j], e[j], stride, keep_better);
    }
  }
}

// (va, ea) <- the best 32 of two sorted lists, sorted: the first list against
// the second reversed gives, entry by entry, a bitonic sequence holding the
// best 32 of the union; a bitonic merge sorts it.
__device__ __forceinline__ void warp_merge32(float& va, int& ea, float vb, int eb) {
  const int lane = threadIdx.x & 31;
  const float rv = __shfl_sync(0xffffffffu, vb, 31 - lane);
  const int re = __shfl_sync(0xffffffffu, eb, 31 - lane);
  if (better(rv, re, va, ea)) { va = rv; ea = re; }
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1)
    bitonic_cas(va, ea, stride, (lane & stride) == 0);
}

// Top k (k <= 32) of the E <= 1024 values value(i), i in [0, E), by a block
// of NW warps. Warp w sorts the 32/NW lists i = 32 (w L + j) + lane and
// merges them; the warps' lists are then merged in a tree through shared
// memory (cand_v / cand_e: NW * 32 entries). On return lane r < k of warp 0
// holds the entry of rank r. Every thread of the block must call.
template <int NW, typename F>
__device__ void block_topk(F value, int E, float* cand_v, int* cand_e,
                           float& out_v, int& out_e) {
  constexpr int L = 32 / NW;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float v[L];
  int e[L];
#pragma unroll
  for (int j = 0; j < L; ++j) {
    const int i = 32 * (warp * L + j) + lane;
    v[j] = i < E ? value(i) : -INFINITY;
    e[j] = i < E ? i : 0x7fffffff;
  }
  warp_sort32<L>(v, e);
#pragma unroll
  for (int w = 1; w < L; w <<= 1)
#pragma unroll
    for (int j = 0; j + w < L; j += 2 * w) warp_merge32(v[j], e[j], v[j + w], e[j + w]);
  cand_v[warp * 32 + lane] = v[0];
  cand_e[warp * 32 + lane] = e[0];
#pragma unroll
  for (int w = 1; w < NW; w <<= 1) {
    __syncthreads();
    if (warp % (2 * w) == 0) {
      warp_merge32(v[0], e[0], cand_v[(warp + w) * 32 + lane], cand_e[(warp + w) * 32 + lane]);
      cand_v[warp * 32 + lane] = v[0];
      cand_e[warp * 32 + lane] = e[0];
    }
  }
  out_v = v[0];
  out_e = e[0];
}

// Sum over the nsplit partial-logit planes p[s * stride] in plane order, the
// first eight loads issued together (one round trip instead of nsplit).
template <bool L2_ONLY>
__device__ __forceinline__ float sum_planes(const float* p, size_t stride, int nsplit) {
  float q[8];
#pragma unroll
  for (int s = 0; s < 8; ++s)
    if (s < nsplit) q[s] = L2_ONLY ? __ldcg(p + (size_t)s * stride) : p[(size_t)s * stride];
  float v = 0.f;
#pragma unroll
  for (int s = 0; s < 8; ++s)
    if (s < nsplit) v += q[s];
  for (int s = 8; s < nsplit; ++s) v += L2_ONLY ? __ldcg(p + (size_t)s * stride) : p[(size_t)s * stride];
  return v;
}

// Softmax over the k <= 32 selected logits held by lanes 0..k-1 of a warp in
// rank order (the largest at lane 0): the weight of this lane's entry (0 for
// lanes >= k). Every lane of the warp must call.
__device__ __forceinline__ float selected_softmax(int k, float sel_v) {
  const int lane = threadIdx.x & 31;
  const float vmax = __shfl_sync(0xffffffffu, sel_v, 0);
  const float ex = lane < k ? expf(sel_v - vmax) : 0.f;
  float z = ex;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  return ex / z;
}

}  // namespace dfm
