// k_phase.cu — a decode batch (T <= 8) as two phase kernels, each running
// the routed and the shared experts side by side, on disjoint sets of CTAs
// (one CTA per SM) sized so that both finish together:
//   * gate/up phase: the shared CTAs stream the shared gate/up rows at once
//     (they do not depend on the routing); the routed CTAs wait for the
//     router and run the routed gate/up. For one token every routed CTA
//     selects the experts itself from the router's partial logits (the same
//     fixed-order sums and sorting network everywhere, so every CTA gets the
//     same selection) and the first routed CTA publishes it;
//   * down phase: the routed CTAs start streaming down weights at once (the
//     selection is complete before the grid starts) and wait only for h; the
//     shared CTAs wait for the shared h.
// Both launch as programmatic dependents of the kernel before them, so the
// router -> gate/up -> down -> combine chain runs on one stream with no
// launch gaps.
#include <algorithm>

#include "bfv.cuh"
#include "mxv.cuh"
#include "select.cuh"

namespace dfm {
namespace {

constexpr int kPhaseThreads = 512;

struct SelArgs {       // one token's selection inside the gate/up phase
  const float* part;   // router partial logits [nsplit][E]; null: selected already
  int nsplit, E, k;
  int32_t* ids;        // [k] outputs, best first
  float* w;
};

// TT: the shared experts' tokens a pass (1, 2, 4 or 8); TT = 1 is one token.
template <int TT>
__global__ void __launch_bounds__(kPhaseThreads, 1)
phase_gateup_kernel(const BfvArgs sh, const MxvArgs rt_in, const SelArgs sel, int n_sh) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bars[kBfvBars > kMxvBars ? kBfvBars : kMxvBars];
  __shared__ Item sel_items[32];
  __shared__ int32_t sel_sorted[32];
  __shared__ int32_t sel_n;
  if ((int)blockIdx.x < n_sh) {
    // x is complete without a wait: the router triggers its dependents only
    // after its own wait, and each later kernel starts only after the one
    // before it has triggered
    bfv_cta<0, TT>(sh, smem, bars, blockIdx.x, n_sh, /*wait=*/false);
    return;
  }
  const int cta = blockIdx.x - n_sh, ncta = gridDim.x - n_sh;
  MxvArgs rt = rt_in;
  // the routed pipeline's barriers are set up while the router finishes
  mxv_set_up_barriers<0>(rt, bars);
  pdl_wait();  // the router (one token) or the grouping kernel
  if (TT == 1 && sel.part) {
    float sel_v = 0.f;
    int sel_e = 0;
    block_topk<kPhaseThreads / 32>(
        [&](int i) { return sum_planes<true>(sel.part + i, sel.E, sel.nsplit); },
        sel.E, reinterpret_cast<float*>(smem),
        reinterpret_cast<int*>(smem + kPhaseThreads * sizeof(float)), sel_v, sel_e);
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const bool pub = cta == 0;
      const float wt = pub ? selected_softmax(sel.k, sel_v) : 0.f;
      if (lane < sel.k) {
        // item q: expert of rank q with its one assignment q
        sel_items[lane] = Item{sel_e, lane, 1, 0};
        sel_sorted[lane] = lane;
        if (pub) {
          sel.ids[lane] = sel_e;
          sel.w[lane] = wt;
          const_cast<Item*>(rt_in.items)[lane] = Item{sel_e, lane, 1, 0};
          const_cast<int32_t*>(rt_in.sorted)[lane] = lane;
        }
      }
      if (lane == 0) {
        sel_n = sel.k;
        if (pub) *const_cast<int32_t*>(rt_in.n_items) = sel.k;
      }
      // the down phase reads the published selection as soon as it starts,
      // which is after every CTA of this grid has exited (the gate/up phase
      // triggers its dependent only implicitly)
      if (pub) __threadfence();
    }
    rt.items = sel_items;
    rt.n_items = &sel_n;
    rt.sorted = sel_sorted;
  }
  __syncthreads();  // barriers set up; the selection in shared memory
  // one token: every item is its own (the library's own selection)
  mxv_cta<0, TT == 1>(rt, smem, bars, cta, ncta, /*set_up=*/false);
}

template <int TT>
__global__ void __launch_bounds__(kPhaseThreads, 1)
phase_down_kernel(const MxvArgs rt, const BfvArgs sh, int n_rt) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bars[kBfvBars > kMxvBars ? kBfvBars : kMxvBars];
  if ((int)blockIdx.x < n_rt)
    mxv_cta<1>(rt, smem, bars, blockIdx.x, n_rt);  // rt.early: streams before h
  else
    bfv_cta<1, TT>(sh, smem, bars, blockIdx.x - n_rt, gridDim.x - n_rt, /*wait=*/true);
}

int phase_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

template <typename Kern>
cudaError_t set_smem(Kern kernel, size_t smem, size_t& configured) {
  if (configured >= smem) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) configured = smem;
  return e;
}

}  // namespace

bool phase_supported(int H, int I, int R, int E, int k) {
  const size_t gu = std::max(bfv_smem_bytes(H), mxv_smem_bytes(H, mxv_cg(0), mxv_unit(0)) +
                                                    mxv_x_bytes(H, mxv_cg(0)));
  const size_t dn = std::max(mxv_smem_bytes(I, mxv_cg(1), mxv_unit(1)), bfv_smem_bytes(R > 0 ? R : I));
  const size_t stat = (kBfvBars > kMxvBars ? kBfvBars : kMxvBars) * 8 + 1024;
  return H % 64 == 0 && I % 64 == 0 && E <= 1024 && k <= 32 && gu + stat <= 227 * 1024 &&
         dn + stat <= 227 * 1024 && gu >= kPhaseThreads * 8;
}

cudaError_t launch_phase_gateup(const uint16_t* sh_gate, const uint16_t* sh_up, int R,
                                const uint8_t* arena, size_t span_bytes, int H, int I, int k,
                                const uint16_t* x, int T, Item* items, int32_t* n_items,
                                int32_t* sorted, const float* router_part, int nsplit, int E,
                                int32_t* ids, float* w, float* hsh, float* hbuf, uint32_t* err,
                                int n_sh, const uint8_t* const* spans, bool drop,
                                cudaStream_t s) {
  const BfvArgs sh{sh_gate, sh_up, R, H, x, T, hsh, err};
  MxvArgs rt{arena, span_bytes, H, I, k, x, nullptr, items, n_items, sorted, hbuf, err, 0,
             spans};
  rt.E = E;
  rt.nassign = T * k;
  rt.max_items = std::min(T * k, E);
  if (drop) {
    rt.drop = 1;
    rt.wait_limit = kTestWaitLimit;
  }
  const SelArgs sel{T == 1 ? router_part : nullptr, nsplit, E, k, ids, w};
  // one token: the routed CTAs also keep its B fragments (mxv_x_bytes)
  const size_t smem = std::max(bfv_smem_bytes(H), mxv_smem_bytes(H, mxv_cg(0), mxv_unit(0)) +
                                                      (T == 1 ? mxv_x_bytes(H, mxv_cg(0)) : 0));
  auto go = [&](auto kernel, size_t& conf) {
    const cudaError_t e = set_smem(kernel, smem, conf);
    if (e != cudaSuccess) return e;
    return launch_after_previous(kernel, dim3(phase_sms()), dim3(kPhaseThreads), smem, s, sh, rt,
                                 sel, n_sh);
  };
  static size_t conf[4] = {0, 0, 0, 0};
  return T == 1   ? go(phase_gateup_kernel<1>, conf[0])
         : T <= 2 ? go(phase_gateup_kernel<2>, conf[1])
         : T <= 4 ? go(phase_gateup_kernel<4>, conf[2])
                  : go(phase_gateup_kernel<8>, conf[3]);
}

cudaError_t launch_phase_down(const uint8_t* arena, size_t span_bytes, int H, int I, int E,
                              int k, const Item* items, const int32_t* n_items,
                              const int32_t* sorted, const float* hbuf, float* part,
                              const uint16_t* sh_down, int R, const float* hsh, int T, float* ysh,
                              uint32_t* err, int n_sh, const uint8_t* const* spans,
                              cudaStream_t s) {
  MxvArgs rt{arena, span_bytes, H, I, 0, nullptr, hbuf, items, n_items, sorted, part, err,
             1, spans};
  rt.E = E;
  rt.nassign = T * k;
  rt.max_items = std::min(T * k, E);
  // no shared experts: no rows to stream (K only sizes the geometry)
  const BfvArgs sh{sh_down, nullptr, R > 0 ? H : 0, R > 0 ? R : I, hsh, T, ysh, err};
  const size_t smem = std::max(mxv_smem_bytes(I, mxv_cg(1), mxv_unit(1)), bfv_smem_bytes(sh.K));
  const int n_rt = phase_sms() - n_sh;
  auto go = [&](auto kernel, size_t& conf) {
    const cudaError_t e = set_smem(kernel, smem, conf);
    if (e != cudaSuccess) return e;
    return launch_after_previous(kernel, dim3(phase_sms()), dim3(kPhaseThreads), smem, s, rt, sh,
                                 n_rt);
  };
  static size_t conf[4] = {0, 0, 0, 0};
  return T == 1   ? go(phase_down_kernel<1>, conf[0])
         : T <= 2 ? go(phase_down_kernel<2>, conf[1])
         : T <= 4 ? go(phase_down_kernel<4>, conf[2])
                  : go(phase_down_kernel<8>, conf[3]);
}

}  // namespace dfm
