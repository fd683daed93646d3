// k_experts.cu — the routed-expert kernels: MXFP4 dequant-fused gate/up GEMV
// with SwiGLU epilogue, down GEMV (stand-alone launches of the per-CTA
// function in mxv.cuh), and the weighted combine.
#include <algorithm>

#include "mxv.cuh"

namespace dfm {
namespace {

template <int MODE>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) mxv_kernel(const MxvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bars[kMxvBars];
  mxv_cta<MODE>(a, smem, bars, blockIdx.x, gridDim.x);
}

// out[t][j] = residual + sum_i w[t][i] part[t k + i][j] + ysh[t][j], k <= 32.
// Every load of a thread is issued before the first FMA (one L2 round trip);
// the sum runs in slot order. The last kernel of a batch forward: its first
// thread copies the device error word, complete once the kernels before it
// are, to the host-visible mirror; with ids_out, block (0, t) also copies
// token t's ids and weights there (host memory the device writes directly).
constexpr int kCombineThreads = 128;
__device__ __forceinline__ void copy_selection(const int32_t* ids, const float* w, int k, int t,
                                               int32_t* ids_out, float* w_out) {
  if (ids_out && blockIdx.x == 0 && (int)threadIdx.x < k) {
    const size_t i = (size_t)t * k + threadIdx.x;
    ids_out[i] = ids[i];
    w_out[i] = w[i];
  }
}
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const float* __restrict__ part, const float* __restrict__ w, int k, int H,
               const float* __restrict__ ysh, const uint16_t* __restrict__ residual,
               float* __restrict__ out_f32, uint16_t* __restrict__ out_bf16, uint32_t* err,
               uint32_t* err_mirror, const int32_t* ids, int32_t* ids_out, float* w_out) {
  pdl_wait();
  if (err_mirror && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    const uint32_t e = atomicOr(err, 0u);
    if (e) *reinterpret_cast<volatile uint32_t*>(err_mirror) = e;
  }
  const int t = blockIdx.y;
  copy_selection(ids, w, k, t, ids_out, w_out);
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= H) return;
  float pv[32], wv[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (i < k) {
      pv[i] = part[((size_t)t * k + i) * H + j];
      wv[i] = w[(size_t)t * k + i];
    }
  }
  float y = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i < k) y = fmaf(wv[i], pv[i], y);
  if (ysh) y += ysh[(size_t)t * H + j];
  if (residual) y += __uint_as_float((uint32_t)residual[(size_t)t * H + j] << 16);
  if (out_f32) out_f32[(size_t)t * H + j] = y;
  if (out_bf16) out_bf16[(size_t)t * H + j] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
}

// The same for batches: each thread takes four consecutive columns with
// 16-byte loads and stores (H a multiple of 4, rows 16-byte aligned); the
// sums run in the same slot order.
__global__ void __launch_bounds__(kCombineThreads)
combine4_kernel(const float* __restrict__ part, const float* __restrict__ w, int k, int H,
                const float* __restrict__ ysh, const uint16_t* __restrict__ residual,
                float* __restrict__ out_f32, uint16_t* __restrict__ out_bf16, uint32_t* err,
                uint32_t* err_mirror, const int32_t* ids, int32_t* ids_out, float* w_out) {
  pdl_wait();
  if (blockIdx.x == 0 && blockIdx.y == 0 && err_mirror && threadIdx.x == 0) {
    const uint32_t e = atomicOr(err, 0u);
    if (e) *reinterpret_cast<volatile uint32_t*>(err_mirror) = e;
  }
  const int t = blockIdx.y;
  copy_selection(ids, w, k, t, ids_out, w_out);
  const int j = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (j >= H) return;
  // slots in groups of eight: a group's loads are issued together, the sums
  // run in slot order
  float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = 0; i0 < k; i0 += 8) {
    float4 pv[8];
    float wv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i0 + i < k) {
        pv[i] = *reinterpret_cast<const float4*>(part + ((size_t)t * k + i0 + i) * H + j);
        wv[i] = w[(size_t)t * k + i0 + i];
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i0 + i < k) {
        y.x = fmaf(wv[i], pv[i].x, y.x);
        y.y = fmaf(wv[i], pv[i].y, y.y);
        y.z = fmaf(wv[i], pv[i].z, y.z);
        y.w = fmaf(wv[i], pv[i].w, y.w);
      }
  }
  if (ysh) {
    const float4 s = *reinterpret_cast<const float4*>(ysh + (size_t)t * H + j);
    y.x += s.x;
    y.y += s.y;
    y.z += s.z;
    y.w += s.w;
  }
  if (residual) {
    const uint2 r = *reinterpret_cast<const uint2*>(residual + (size_t)t * H + j);
    y.x += __uint_as_float(r.x << 16);
    y.y += __uint_as_float(r.x & 0xFFFF0000u);
    y.z += __uint_as_float(r.y << 16);
    y.w += __uint_as_float(r.y & 0xFFFF0000u);
  }
  if (out_f32) *reinterpret_cast<float4*>(out_f32 + (size_t)t * H + j) = y;
  if (out_bf16) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(y.x)) |
                        (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.y)) << 16;
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(y.z)) |
                        (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.w)) << 16;
    *reinterpret_cast<uint2*>(out_bf16 + (size_t)t * H + j) = make_uint2(lo, hi);
  }
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

template <int MODE>
cudaError_t launch_mxv(const MxvArgs& a, int max_items, cudaStream_t s, int max_ctas) {
  const int K = MODE == 0 ? a.H : a.I;
  constexpr int CG = mxv_cg(MODE);
  const int NS = slots_per_cta(K, CG);
  const int threads = NS * mxv_wps(K, CG) * 32;
  const size_t smem = mxv_smem_bytes(K, CG, mxv_unit(MODE));
  static int configured_smem[2] = {0, 0};
  if (configured_smem[MODE] < (int)smem) {
    cudaError_t e = cudaFuncSetAttribute(mxv_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured_smem[MODE] = (int)smem;
  }
  const int tpi = MODE == 0 ? (2 * a.I) / 16 : a.H / 16;
  const long long max_tiles = (long long)max_items * tpi;
  int grid = (int)((max_tiles + NS - 1) / NS);
  if (grid > num_sms()) grid = num_sms();
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  if (grid < 1) grid = 1;
  return launch_after_previous(mxv_kernel<MODE>, dim3(grid), dim3(threads), smem, s, a);
}

}  // namespace

cudaError_t launch_gateup(const uint8_t* arena, size_t span_bytes, int H,
                          int I, int k, const uint16_t* x, const Item* items,
                          const int32_t* n_items, int max_items,
                          const int32_t* sorted, float* hbuf, int /*tg*/, int E, int nassign,
                          uint32_t* err, cudaStream_t s, int max_ctas) {
  MxvArgs a{arena, span_bytes, H, I, k, x, nullptr, items, n_items, sorted, hbuf, err, 0,
            nullptr};
  a.E = E;
  a.nassign = nassign;
  a.max_items = max_items;
  return launch_mxv<0>(a, max_items, s, max_ctas);
}

cudaError_t launch_down(const uint8_t* arena, size_t span_bytes, int H, int I,
                        const Item* items, const int32_t* n_items,
                        int max_items, const int32_t* sorted,
                        const float* hbuf, float* part, int /*tg*/, int E, int nassign,
                        uint32_t* err, cudaStream_t s, int max_ctas, bool after_gateup) {
  MxvArgs a{arena, span_bytes, H, I, 0, nullptr, hbuf, items, n_items, sorted, part, err,
            after_gateup ? 1 : 0, nullptr};
  a.E = E;
  a.nassign = nassign;
  a.max_items = max_items;
  return launch_mxv<1>(a, max_items, s, max_ctas);
}

cudaError_t launch_combine(const float* part, const float* w, int T, int k,
                           int H, const float* ysh, const uint16_t* residual,
                           float* out_f32, uint16_t* out_bf16, uint32_t* err,
                           uint32_t* err_mirror, cudaStream_t s, const int32_t* ids,
                           int32_t* ids_out, float* w_out) {
  if (ids_out && (!ids || !w_out || k > kCombineThreads)) return cudaErrorInvalidValue;
  const auto al16 = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
  if (T > 8 && H % 4 == 0 && al16(part) && (!ysh || al16(ysh)) && (!out_f32 || al16(out_f32)) &&
      (!residual || ((uintptr_t)residual & 7) == 0) && (!out_bf16 || ((uintptr_t)out_bf16 & 7) == 0)) {
    // batches: four columns a thread
    dim3 grid((H / 4 + kCombineThreads - 1) / kCombineThreads, T);
    return launch_after_previous(combine4_kernel, grid, dim3(kCombineThreads), 0, s, part, w, k,
                                 H, ysh, residual, out_f32, out_bf16, err, err_mirror, ids,
                                 ids_out, w_out);
  }
  dim3 grid((H + kCombineThreads - 1) / kCombineThreads, T);
  return launch_after_previous(combine_kernel, grid, dim3(kCombineThreads), 0, s, part, w, k, H, ysh,
                               residual, out_f32, out_bf16, err, err_mirror, ids, ids_out, w_out);
}

// Plain 16-byte copy (an input staged in host memory that the device reads
// directly, to its device buffer). An ordinary launch: the next kernel's
// programmatic wait covers this whole grid.
__global__ void __launch_bounds__(256) copy16_kernel(const uint4* __restrict__ src,
                                                     uint4* __restrict__ dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t s) {
  if (((uintptr_t)src | (uintptr_t)dst | bytes) & 15) return cudaErrorInvalidValue;
  const size_t n = bytes / 16;
  if (!n) return cudaSuccess;
  const int blocks = (int)std::min<size_t>((n + 255) / 256, 64);
  copy16_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                       n);
  return cudaGetLastError();
}

}  // namespace dfm
