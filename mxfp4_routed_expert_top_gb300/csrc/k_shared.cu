// k_shared.cu — bf16 shared-expert GEMVs (stand-alone launches of the
// per-CTA function in bfv.cuh) and RMSNorm.
#include "bfv.cuh"

namespace dfm {
namespace {

template <int MODE, int TT>
__global__ void __launch_bounds__(512, 1) bfv_kernel(const BfvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bars[kBfvBars];
  bfv_cta<MODE, TT>(a, smem, bars, blockIdx.x, gridDim.x, true);
}

int num_sms_b() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

template <int MODE, int TT>
cudaError_t launch_bfv_t(const BfvArgs& a, cudaStream_t s, int max_ctas) {
  const int NS = bfv_slots(a.K);
  const size_t smem = bfv_smem_bytes(a.K);
  static size_t configured = 0;
  if (configured < smem) {
    cudaError_t e = cudaFuncSetAttribute(bfv_kernel<MODE, TT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  const int ntiles = MODE == 0 ? a.rows / 2 : a.rows / kRows;
  int grid = (ntiles + NS - 1) / NS;
  if (grid > num_sms_b()) grid = num_sms_b();
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  bfv_kernel<MODE, TT><<<grid, NS * bfv_wps(a.K) * 32, smem, s>>>(a);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_bfv(const BfvArgs& a, cudaStream_t s, int max_ctas) {
  return a.T == 1   ? launch_bfv_t<MODE, 1>(a, s, max_ctas)
         : a.T <= 2 ? launch_bfv_t<MODE, 2>(a, s, max_ctas)
         : a.T <= 4 ? launch_bfv_t<MODE, 4>(a, s, max_ctas)
                    : launch_bfv_t<MODE, 8>(a, s, max_ctas);
}

// xn = RNE_bf16(x / sqrt(mean(x^2) + eps)); one block per token.
__global__ void __launch_bounds__(256)
rmsnorm_kernel(const uint16_t* __restrict__ x, int H, float eps,
               uint16_t* __restrict__ xn) {
  __shared__ float ws[8];
  pdl_wait();  // x comes from the preceding kernel
  pdl_launch_dependents();
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

// Read-only streaming probe: each thread keeps 16 loads of 16 bytes in flight
// (non-coherent path, no L1 allocation) and folds them into one word.
__global__ void __launch_bounds__(256) stream_read_kernel(const uint4* __restrict__ p, size_t n16,
                                                          uint32_t* __restrict__ sink) {
  constexpr int U = 16;
  uint32_t acc = 0;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (U - 1) * stride < n16; i += U * stride) {
    uint32_t v[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u)
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(v[u][0]), "=r"(v[u][1]), "=r"(v[u][2]), "=r"(v[u][3])
                   : "l"(p + i + u * stride));
#pragma unroll
    for (int u = 0; u < U; ++u) acc ^= v[u][0] ^ v[u][1] ^ v[u][2] ^ v[u][3];
  }
  for (; i < n16; i += stride) {
    const uint4 v = p[i];
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

// Expert cache fill: block (x, y) copies its share of span y from pinned host
// memory over NVLink-C2C (plain loads of the mapped pages, eight 16-byte
// loads in flight a thread) into its HBM slot; block (0, y) also points the
// span table at the slot. SM loads keep the whole copy near the link's rate
// where copy-engine copies of single spans showed a slow tail.
__global__ void __launch_bounds__(512) cache_fill_kernel(const CacheCopy* __restrict__ plan,
                                                         size_t n16,
                                                         unsigned long long* __restrict__ span_tab) {
  constexpr int U = 8;
  __shared__ CacheCopy c;
  if (threadIdx.x == 0) {
    c = plan[blockIdx.y];
    if (blockIdx.x == 0) span_tab[c.e] = (unsigned long long)(uintptr_t)c.dst;
  }
  __syncthreads();
  const uint4* __restrict__ src = static_cast<const uint4*>(c.src);
  uint4* __restrict__ dst = static_cast<uint4*>(c.dst);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (U - 1) * stride < n16; i += U * stride) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = src[i + u * stride];
#pragma unroll
    for (int u = 0; u < U; ++u) dst[i + u * stride] = v[u];
  }
  for (; i < n16; i += stride) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_cache_fill(const CacheCopy* plan, int n, size_t span_bytes,
                              unsigned long long* span_tab, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (span_bytes % 16 || n > 65535) return cudaErrorInvalidValue;
  // about four blocks an SM over all spans
  const int bx = std::max(1, (4 * num_sms_b() + n - 1) / n);
  cache_fill_kernel<<<dim3(bx, n), 512, 0, s>>>(plan, span_bytes / 16, span_tab);
  return cudaGetLastError();
}

cudaError_t launch_stream_read(const void* buf, size_t bytes, uint32_t* sink, cudaStream_t s) {
  stream_read_kernel<<<4 * num_sms_b(), 256, 0, s>>>(static_cast<const uint4*>(buf), bytes / 16,
                                                      sink);
  return cudaGetLastError();
}

cudaError_t launch_shared_gateup(const uint16_t* gate, const uint16_t* up,
                                 int R, int H, const uint16_t* x, int T,
                                 float* hsh, uint32_t* err, cudaStream_t s, int max_ctas) {
  return launch_bfv<0>(BfvArgs{gate, up, R, H, x, T, hsh, err}, s, max_ctas);
}

cudaError_t launch_shared_down(const uint16_t* down, int H, int K,
                               const float* hsh, int T, float* ysh,
                               uint32_t* err, cudaStream_t s, int max_ctas) {
  return launch_bfv<1>(BfvArgs{down, nullptr, H, K, hsh, T, ysh, err}, s, max_ctas);
}

cudaError_t launch_rmsnorm(const uint16_t* x, int T, int H, float eps,
                           uint16_t* xn, cudaStream_t s) {
  return launch_after_previous(rmsnorm_kernel, dim3(T), dim3(256), 0, s, x, H, eps, xn);
}

}  // namespace dfm
