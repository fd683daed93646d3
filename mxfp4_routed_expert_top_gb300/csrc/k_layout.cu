// k_layout.cu — repacking canonical expert spans into the fragment layout the
// expert kernels stream (see internal.h), and back.
#include <cuda_fp16.h>

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

// Canonical offset of byte `o` of one section (gate/up or down) of the
// device span; the section holds tiles of 16 rows x K. Tile row rho of tile
// j maps to (tensor, row) by `gu`: gate/up tiles interleave 8 gate and 8 up
// rows; down tiles are 16 consecutive rows.
__device__ inline size_t section_src(size_t o, int K, bool gu, const Canon& C) {
  const size_t tile = mx_tile_bytes(K);
  const size_t j = o / tile;
  const int rem = (int)(o - j * tile);
  const int grp = rem / kGroupBytes;
  const int w = rem - grp * kGroupBytes;
  int rho;
  bool scale;
  size_t idx;  // column byte (codes) or block (scales) within the row
  if (w < 512) {
    const int l = w >> 4, g = l >> 2, t = l & 3;
    const int s = (w >> 2) & 3, q = w & 3;
    rho = g + 8 * (q & 1);
    idx = (size_t)(64 * grp + 16 * s + 2 * t + 8 * (q >> 1)) >> 1;
    scale = false;
  } else {
    const int g = (w - 512) >> 2, i = (w - 512) & 3;
    rho = g + 8 * (i >> 1);
    idx = (size_t)(2 * grp + (i & 1));
    scale = true;
  }
  size_t base, row;
  if (gu) {
    base = rho < 8 ? (scale ? C.gs : C.gq) : (scale ? C.us : C.uq);
    row = 8 * j + (rho & 7);
  } else {
    base = scale ? C.ds : C.dq;
    row = 16 * j + rho;
  }
  const size_t row_bytes = scale ? (size_t)(K / 32) : (size_t)(K / 2);
  return base + row * row_bytes + idx;
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
      if (o < D.dn) c = section_src(o - D.gu, H, true, C);
      else c = section_src(o - D.dn, I, false, C);
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
