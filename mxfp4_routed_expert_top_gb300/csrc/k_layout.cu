// k_layout.cu — repacking canonical expert spans into the fragment layout the
// expert kernels stream (see internal.h), and back.
#include "internal.h"

namespace dfm {
namespace {

struct Canon {  // offsets of the six canonical tensors
  size_t gq, gs, uq, us, dq, ds;
};

__device__ inline Canon canon_offsets(int H, int I) {
  size_t hi = (size_t)H * I, q = hi / 2, s = hi / 32;
  return Canon{0, q, q + s, 2 * q + s, 2 * q + 2 * s, 3 * q + 2 * s};
}

// Canonical byte offset of byte `o` of a codes section of a matrix with K
// columns. Tile row rho of tile j maps to (tensor offset, row) by `gu`:
// gate/up tiles interleave 8 gate and 8 up rows; down tiles are 16 rows.
__device__ inline size_t codes_src(size_t o, int K, bool gu, const Canon& C) {
  const size_t tile = (size_t)8 * K;
  const size_t j = o / tile;
  const int rem = (int)(o - j * tile);
  const int grp = rem >> 9;            // 64-column group (8c + v)
  const int w = rem & 511;
  const int l = w >> 4, g = l >> 2, t = l & 3;
  const int s = (w >> 2) & 3, q = w & 3;
  const int rho = g + 8 * (q & 1);
  const int col = 64 * grp + 16 * s + 2 * t + 8 * (q >> 1);
  size_t base, row;
  if (gu) {
    base = rho < 8 ? C.gq : C.uq;
    row = 8 * j + (rho & 7);
  } else {
    base = C.dq;
    row = 16 * j + rho;
  }
  return base + row * (size_t)(K / 2) + (size_t)(col >> 1);
}

__device__ inline size_t scales_src(size_t o, int K, bool gu, const Canon& C) {
  const size_t tile = (size_t)K / 2;
  const size_t j = o / tile;
  const int rem = (int)(o - j * tile);
  const int c = rem >> 8;
  const int w = rem & 255;
  const int nbc = mx_nbc(K, c);
  const int g = w / (2 * nbc), i = w - g * 2 * nbc;
  const int rho = g + 8 * (i >= nbc ? 1 : 0);
  const int block = 16 * c + (i >= nbc ? i - nbc : i);
  size_t base, row;
  if (gu) {
    base = rho < 8 ? C.gs : C.us;
    row = 8 * j + (rho & 7);
  } else {
    base = C.ds;
    row = 16 * j + rho;
  }
  return base + row * (size_t)(K / 32) + (size_t)block;
}

// One thread per 16-byte unit of the device span. inverse = 0: canonical ->
// device; 1: device -> canonical.
__global__ void repack_kernel(const uint8_t* __restrict__ src,
                              uint8_t* __restrict__ dst, int n_spans, int H,
                              int I, int inverse) {
  const SpanLayout D = span_layout(H, I);
  const Canon C = canon_offsets(H, I);
  const size_t units = D.bytes / 16;
  const size_t total = units * (size_t)n_spans;
  for (size_t u = (size_t)blockIdx.x * blockDim.x + threadIdx.x; u < total;
       u += (size_t)gridDim.x * blockDim.x) {
    const size_t span = u / units;
    const size_t o0 = (u - span * units) * 16;  // offset in the device span
    const uint8_t* sbase = src + span * D.bytes;
    uint8_t* dbase = dst + span * D.bytes;
    for (int i = 0; i < 16; ++i) {
      const size_t o = o0 + i;
      size_t c;
      if (o < D.gu_scales) c = codes_src(o - D.gu_codes, H, true, C);
      else if (o < D.dn_codes) c = scales_src(o - D.gu_scales, H, true, C);
      else if (o < D.dn_scales) c = codes_src(o - D.dn_codes, I, false, C);
      else c = scales_src(o - D.dn_scales, I, false, C);
      if (!inverse) dbase[o] = sbase[c];
      else dbase[c] = sbase[o];
    }
  }
}

}  // namespace

cudaError_t launch_repack_span(const uint8_t* src, uint8_t* dst, int n_spans,
                               int H, int I, int inverse, cudaStream_t s) {
  const size_t units = span_layout(H, I).bytes / 16 * (size_t)n_spans;
  size_t grid = (units + 255) / 256;
  if (grid > 152 * 64) grid = 152 * 64;
  repack_kernel<<<(unsigned)grid, 256, 0, s>>>(src, dst, n_spans, H, I, inverse);
  return cudaGetLastError();
}

}  // namespace dfm
