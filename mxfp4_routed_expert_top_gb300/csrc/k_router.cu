// k_router.cu — router GEMV, top-k selection with softmax over the selected
// logits, and grouping of token->expert assignments by expert.
//
// Each token's router chooses 16 of the 896 experts, and only the chosen
// experts' weights are touched (Deltafin README, "How it works"; Deltafin
// analysis §5.1). Selection ties go to the lower expert id; ids come out in
// descending logit order.
#include <math.h>

#include <algorithm>

#include "internal.h"
#include "pipeline.cuh"
#include "select.cuh"

namespace dfm {
namespace {

constexpr int kRouterRowsPerBlock = 8;  // one warp per (row, column split)
constexpr int kRouterMaxV = 16;         // float4 loads per lane: split <= 2048
constexpr int kRouterThreads = 32 * kRouterRowsPerBlock;
constexpr int kTopkThreads = 256;       // top-k blocks of the batch path

// Softmax over the k selected logits (warp 0, lanes 0..k-1 hold them) and
// the writes of ids / weights (and, for a single token, the work items).
__device__ void write_selection(int t, int k, float sel_v, int sel_e,
                                int32_t* ids, float* w, Item* items,
                                int32_t* n_items, int32_t* sorted) {
  const int lane = threadIdx.x & 31;
  const float wt = selected_softmax(k, sel_v);
  if (lane < k) {
    ids[(size_t)t * k + lane] = sel_e;
    w[(size_t)t * k + lane] = wt;
    if (items) {
      items[lane] = Item{sel_e, lane, 1, 0};
      sorted[lane] = lane;
    }
  }
  if (items && lane == 0) *n_items = k;
}

struct TopkFuse {  // fused top-k of a single token by the router's last block
  unsigned int* counter;  // zero between calls; reset by the last block
  int k;
  int32_t* ids;
  float* w;
  Item* items;
  int32_t* n_items;
  int32_t* sorted;
};

// part[split][t][e] = sum over the split's columns of Wr[e][j] x[t][j].
// One warp per (row, split); every weight load of the warp is issued before
// the first FMA. Tokens go in passes of NT, each weight register feeding the
// NT accumulators of a pass, so the weights are read once per call. For one
// token at most 80 registers a thread (three blocks an SM, so that the K3
// router's 448 blocks run as a single wave on 152 SMs), else at most 128 (two).
template <int NT>
__global__ void __launch_bounds__(kRouterThreads, NT == 1 ? 3 : 2)
router_kernel(const float* __restrict__ Wr, int E, int H,
              const uint16_t* __restrict__ x, int T, float* __restrict__ part,
              int split_len, TopkFuse fz) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterRowsPerBlock + warp;
  const int split = blockIdx.y;
  const int k0 = split * split_len;
  const int len = min(split_len, H - k0);
  // each pass's slice of x, [NT][split_len] bf16, is staged in shared
  // memory (all its loads issued at once; the first pass while the weight
  // loads are in flight)
  extern __shared__ __align__(16) uint16_t xs[];
  float4 w4[kRouterMaxV];
  if (e < E) {
    const float* wr = Wr + (size_t)e * H + k0 + 4 * lane;
#pragma unroll
    for (int i = 0; i < kRouterMaxV; ++i)
      w4[i] = (4 * lane + 128 * i < len) ? __ldg(reinterpret_cast<const float4*>(wr + 128 * i))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // x and the outputs' readers come from the preceding kernels; the weights
  // (read above) do not
  pdl_wait();
  // The next kernel may start now. Triggering only after the wait makes the
  // start of any later kernel of the chain (each starts only after the one
  // before it has triggered) imply that x is complete: the decode phase
  // kernels' shared-expert CTAs read x without waiting, and x may come from
  // the kernel before this one (the stack's RMSNorm, which triggers early).
  pdl_launch_dependents();
  const int q8 = len >> 3;  // 8 bf16 a copy (len is a multiple of 32)
  for (int t0 = 0; t0 < T; t0 += NT) {
    const int nt = min(NT, T - t0);
    if (t0 > 0) __syncthreads();  // the previous pass has read its slice
    for (int q = threadIdx.x; q < nt * q8; q += blockDim.x) {
      const int t = q / q8, c = q - t * q8;
      reinterpret_cast<uint4*>(xs + (size_t)t * split_len)[c] =
          __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + t) * H + k0) + c);
    }
    __syncthreads();
    if (e >= E) continue;
    {
      float acc[NT];
#pragma unroll
      for (int u = 0; u < NT; ++u) acc[u] = 0.f;
#pragma unroll
      for (int i = 0; i < kRouterMaxV; ++i) {
        if (4 * lane + 128 * i < len) {
#pragma unroll
          for (int u = 0; u < NT; ++u) {
            if (t0 + u < T) {
              const uint2 xv = *reinterpret_cast<const uint2*>(
                  xs + (size_t)u * split_len + 4 * lane + 128 * i);
              acc[u] = fmaf(w4[i].x, __uint_as_float(xv.x << 16), acc[u]);
              acc[u] = fmaf(w4[i].y, __uint_as_float(xv.x & 0xFFFF0000u), acc[u]);
              acc[u] = fmaf(w4[i].z, __uint_as_float(xv.y << 16), acc[u]);
              acc[u] = fmaf(w4[i].w, __uint_as_float(xv.y & 0xFFFF0000u), acc[u]);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < NT; ++u) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
        if (lane == 0 && t0 + u < T) part[((size_t)split * T + t0 + u) * E + e] = acc[u];
      }
    }
  }
  if (!fz.counter) return;

  // ---- single token: the last block to finish selects the experts ----
  __shared__ unsigned int ticket;
  __shared__ float cand_v[kRouterThreads];
  __shared__ int cand_e[kRouterThreads];
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    ticket = atomicAdd(fz.counter, 1u);
  }
  __syncthreads();
  if (ticket != gridDim.x * gridDim.y - 1) return;
  __threadfence();
  const int nsplit = gridDim.y;
  float sel_v = 0.f;
  int sel_e = 0;
  block_topk<kRouterThreads / 32>(
      [&](int i) { return sum_planes<true>(part + i, E, nsplit); },
      E, cand_v, cand_e, sel_v, sel_e);
  if (warp == 0) {
    write_selection(0, fz.k, sel_v, sel_e, fz.ids, fz.w, fz.items, fz.n_items,
                    fz.sorted);
    if (lane == 0) *fz.counter = 0u;
  }
}

// One block of kTopkThreads per token: sum the split partials (fixed order),
// select the top k and the softmax weights.
__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const float* __restrict__ part, int nsplit, int T, int E, int k,
            float* __restrict__ logits_out, int32_t* __restrict__ ids,
            float* __restrict__ w, Item* items, int32_t* n_items,
            int32_t* sorted) {
  __shared__ float cand_v[kTopkThreads];
  __shared__ int cand_e[kTopkThreads];
  // the next kernel may start now: it waits for this grid before it reads
  // (and this grid started only after the router had passed its own wait)
  pdl_launch_dependents();
  pdl_wait();  // the router's partial logits
  const int t = blockIdx.x;
  float sel_v = 0.f;
  int sel_e = 0;
  block_topk<kTopkThreads / 32>(
      [&](int e) {
        const float v = sum_planes<false>(part + (size_t)t * E + e, (size_t)T * E, nsplit);
        if (logits_out) logits_out[(size_t)t * E + e] = v;
        return v;
      },
      E, cand_v, cand_e, sel_v, sel_e);
  if (threadIdx.x < 32)
    write_selection(t, k, sel_v, sel_e, ids, w, (items && T == 1) ? items : nullptr,
                    n_items, sorted);
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
             Item* items, int32_t* n_items, int32_t* sorted, int tg, uint32_t* err,
             int32_t* inv) {
  __shared__ int cnt[1024];
  __shared__ int fill[1024];
  __shared__ int warp_sums[32];
  __shared__ int tot;
  // the sorted list is built in shared memory when it fits (the segment
  // sorts then run at shared-memory latency), else in place in global memory
  constexpr int kSortSmem = 8192;
  __shared__ int ssort[kSortSmem];
  const int tid = threadIdx.x;
  const int A = T * k;
  int* const buf = A <= kSortSmem ? ssort : sorted;
  cnt[tid] = 0;
  pdl_launch_dependents();  // the next kernel waits for this grid itself
  pdl_wait();  // the selected ids
  __syncthreads();
  // an id outside [0, E) (the single-step entry points take the caller's
  // ids) is left out of every segment and recorded in the error word
  bool bad = false;
  // eight loads a thread issued together (one round trip, not eight)
  for (int a0 = tid; a0 < A; a0 += 8 * blockDim.x) {
    int ev[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int a = a0 + u * (int)blockDim.x;
      ev[u] = a < A ? ids[a] : 0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (a0 + u * (int)blockDim.x >= A) break;
      if ((unsigned)ev[u] < (unsigned)E) atomicAdd(&cnt[ev[u]], 1);
      else bad = true;
    }
  }
  if (bad && err) atomicOr(err, DEV_ERR_RANGE);
  __syncthreads();
  const int c = tid < E ? cnt[tid] : 0;
  const int start = block_exclusive_scan(c, warp_sums, &tot);
  const int nvalid = tot;  // assignments with an id in range
  if (tid < E) {
    fill[tid] = start;
    if (offs) offs[tid] = start;
  }
  __syncthreads();
  if (tid == 0 && offs) offs[E] = tot;  // A when every id is in range
  for (int a0 = tid; a0 < A; a0 += 8 * blockDim.x) {
    int ev[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int a = a0 + u * (int)blockDim.x;
      ev[u] = a < A ? ids[a] : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if ((unsigned)ev[u] >= (unsigned)E) continue;  // out of range, or past A
      const int p = atomicAdd(&fill[ev[u]], 1);
      buf[p] = a0 + u * (int)blockDim.x;
    }
  }
  __syncthreads();
  __threadfence_block();
  // order each segment by assignment index (insertion sort, one thread each)
  if (tid < E) {
    for (int i = start + 1; i < start + c; ++i) {
      const int v = buf[i];
      int j = i - 1;
      while (j >= start && buf[j] > v) { buf[j + 1] = buf[j]; --j; }
      buf[j + 1] = v;
    }
  }
  if (inv)
    for (int a = tid; a < A; a += blockDim.x) inv[a] = -1;
  __syncthreads();
  if (buf != sorted)
    for (int p = tid; p < nvalid; p += blockDim.x) sorted[p] = buf[p];
  if (inv)
    for (int p = tid; p < nvalid; p += blockDim.x) inv[buf[p]] = p;
  if (tok) {
    for (int p = tid; p < nvalid; p += blockDim.x) {
      tok[p] = buf[p] / k;
      slot[p] = buf[p] % k;
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
                          int T, float* part, RouterSplit sp, cudaStream_t s,
                          const RouterFuse* fuse, bool after_previous) {
  TopkFuse fz{nullptr, 0, nullptr, nullptr, nullptr, nullptr, nullptr};
  if (fuse && T == 1)
    fz = TopkFuse{fuse->counter, fuse->k, fuse->ids, fuse->w, fuse->items,
                  fuse->n_items, fuse->sorted};
  dim3 grid((E + kRouterRowsPerBlock - 1) / kRouterRowsPerBlock, sp.nsplit);
  const int nt = T == 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;
  const size_t xs = (size_t)nt * sp.split_len * sizeof(uint16_t);  // <= 8 * 2048 * 2
  const dim3 block(kRouterThreads);
  auto go = [&](auto kernel) {
    if (after_previous)
      return launch_after_previous(kernel, grid, block, xs, s, Wr, E, H, x, T, part,
                                   sp.split_len, fz);
    // an ordinary launch: it starts after everything before it on the stream
    // has completed (its griddepcontrol.wait then returns at once), so even
    // the weights, read before that wait, may come from the kernel before it
    kernel<<<grid, block, xs, s>>>(Wr, E, H, x, T, part, sp.split_len, fz);
    return cudaGetLastError();
  };
  if (T == 1) return go(router_kernel<1>);
  if (T <= 2) return go(router_kernel<2>);
  if (T <= 4) return go(router_kernel<4>);
  return go(router_kernel<8>);
}

cudaError_t launch_topk(const float* part, int nsplit, int T, int E, int k,
                        float* logits_out, int32_t* ids, float* w, Item* items,
                        int32_t* n_items, int32_t* sorted, cudaStream_t s) {
  return launch_after_previous(topk_kernel, dim3(T), dim3(kTopkThreads), 0, s, part, nsplit, T, E,
                               k, logits_out, ids, w, items, n_items, sorted);
}

cudaError_t launch_group(const int32_t* ids, int T, int k, int E,
                         int32_t* offs, int32_t* tok, int32_t* slot,
                         int32_t* n_union, Item* items, int32_t* n_items,
                         int32_t* sorted, int tg, uint32_t* err, cudaStream_t s,
                         int32_t* inv) {
  return launch_after_previous(group_kernel, dim3(1), dim3(1024), 0, s, ids, T, k, E, offs, tok,
                               slot, n_union, items, n_items, sorted, tg, err, inv);
}

}  // namespace dfm
