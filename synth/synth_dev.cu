// synth_dev.cu — device-side generator of canonical expert spans.
//
// Produces exactly the bytes synth_expert_spans() produces on the host (same
// SplitMix64 counter streams, integer arithmetic only), so that 15.7 GB of
// synthetic experts per layer can be written straight into HBM. A GPU test
// checks the two implementations byte for byte. Inputs only: no part of the
// MoE layer's arithmetic lives here.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ULL;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ uint64_t at(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1) * kGolden);
}

uint64_t key_of(uint64_t seed, uint32_t cfg, uint32_t layer, uint32_t kind,
                uint64_t index) {
  uint64_t k = at(seed, 0x51A7u);
  k = at(k ^ (uint64_t)cfg, 1);
  k = at(k ^ (uint64_t)layer, 2);
  k = at(k ^ (uint64_t)kind, 3);
  k = at(k ^ index, 4);
  return k;
}

// One thread per 8 code bytes (one 64-bit store).
__global__ void fill_codes_kernel(uint64_t key, uint64_t nwords, uint8_t* dst) {
  uint64_t w = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (; w < nwords; w += stride) {
    uint64_t v = at(key, w);
    // dst + 8w is 8-byte aligned: spans and tensor offsets are multiples of 8
    reinterpret_cast<uint64_t*>(dst)[w] = v;  // little-endian byte order
  }
}

__global__ void fill_scales_kernel(uint64_t key, uint64_t n, uint8_t* dst) {
  uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (; j < n; j += stride) {
    uint64_t u32 = at(key, j) >> 32;
    dst[j] = (uint8_t)(119u + (uint32_t)((u32 * 9u) >> 32));
  }
}

}  // namespace

extern "C" {

// Fill n_exp canonical spans (experts e0 .. e0+n_exp-1) at device pointer dst.
// Requires H % 64 == 0 and I % 64 == 0 (so every tensor starts 8-byte
// aligned) and dst 8-byte aligned. Returns a cudaError_t value (0 = success).
int synth_dev_expert_spans(uint64_t seed, uint32_t cfg, uint32_t layer,
                           uint32_t e0, uint32_t n_exp, int H, int I,
                           void* dst, void* stream) {
  if (H <= 0 || I <= 0 || (H % 64) || (I % 64) || ((uintptr_t)dst & 7))
    return (int)cudaErrorInvalidValue;
  cudaStream_t s = (cudaStream_t)stream;
  const uint64_t hi = (uint64_t)H * (uint64_t)I;
  const uint64_t qn = hi / 2, sn = hi / 32;
  const uint64_t span = 3 * (qn + sn);
  uint8_t* base = (uint8_t*)dst;
  for (uint32_t n = 0; n < n_exp; ++n) {
    uint8_t* p = base + (uint64_t)n * span;
    for (int t = 0; t < 6; ++t) {
      uint64_t key = key_of(seed, cfg, layer, 16u + (uint32_t)t, e0 + n);
      if ((t & 1) == 0) {
        uint64_t nw = qn / 8;
        unsigned grid = (unsigned)((nw + 255) / 256);
        if (grid > 65535u * 4u) grid = 65535u * 4u;
        fill_codes_kernel<<<grid, 256, 0, s>>>(key, nw, p);
        p += qn;
      } else {
        unsigned grid = (unsigned)((sn + 255) / 256);
        if (grid > 65535u * 4u) grid = 65535u * 4u;
        fill_scales_kernel<<<grid, 256, 0, s>>>(key, sn, p);
        p += sn;
      }
    }
  }
  return (int)cudaGetLastError();
}

}  // extern "C"
