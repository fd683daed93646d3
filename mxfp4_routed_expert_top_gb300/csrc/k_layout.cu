// k_layout.cu — repacking canonical expert spans into the HBM layout the
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

// Decompose an offset inside a codes section into (pair, chunk, r, b).
__device__ inline void codes_coord(size_t o, int K, size_t& P, int& c, int& r,
                                   int& b) {
  P = o / (size_t)K;
  int rem = (int)(o - P * (size_t)K);
  c = rem >> 9;
  int nbc = mx_nbc(K, c);
  int w = (rem - (c << 9)) >> 4;
  r = w / nbc;
  b = w - r * nbc;
}

__device__ inline void scales_coord(size_t o, int K, size_t& G, int& c, int& r,
                                    int& b) {
  size_t gsz = (size_t)32 * mx_nb(K);
  G = o / gsz;
  int rem = (int)(o - G * gsz);
  c = rem >> 9;
  int nbc = mx_nbc(K, c);
  int w = (rem - (c << 9)) >> 4;
  r = w / nbc;
  b = w - r * nbc;
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
  for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (size_t)gridDim.x * blockDim.x) {
    const size_t span = g / units;
    const size_t o = (g - span * units) * 16;  // offset in the device span
    const uint8_t* sbase = src + span * D.bytes;
    uint8_t* dbase = dst + span * D.bytes;
    size_t coff[16];
    bool contiguous;
    if (o < D.gu_scales) {  // gate/up codes, K = H
      size_t P; int c, r, b;
      codes_coord(o - D.gu_codes, H, P, c, r, b);
      coff[0] = (r ? C.uq : C.gq) + P * (size_t)(H / 2) + (size_t)(16 * c + b) * 16;
      contiguous = true;
    } else if (o < D.dn_codes) {  // gate/up scales
      size_t G; int c, r, b;
      scales_coord(o - D.gu_scales, H, G, c, r, b);
      const int NB = mx_nb(H);
      for (int i = 0; i < 16; ++i)
        coff[i] = (r ? C.us : C.gs) + (16 * G + i) * (size_t)NB + 16 * c + b;
      contiguous = false;
    } else if (o < D.dn_scales) {  // down codes, K = I
      size_t P; int c, r, b;
      codes_coord(o - D.dn_codes, I, P, c, r, b);
      coff[0] = C.dq + (2 * P + r) * (size_t)(I / 2) + (size_t)(16 * c + b) * 16;
      contiguous = true;
    } else {  // down scales
      size_t G; int c, r, b;
      scales_coord(o - D.dn_scales, I, G, c, r, b);
      const int NB = mx_nb(I);
      for (int i = 0; i < 16; ++i)
        coff[i] = C.ds + (2 * (16 * G + i) + r) * (size_t)NB + 16 * c + b;
      contiguous = false;
    }
    if (contiguous) {
      if (!inverse)
        *reinterpret_cast<uint4*>(dbase + o) =
            *reinterpret_cast<const uint4*>(sbase + coff[0]);
      else
        *reinterpret_cast<uint4*>(dbase + coff[0]) =
            *reinterpret_cast<const uint4*>(sbase + o);
    } else {
      for (int i = 0; i < 16; ++i) {
        if (!inverse) dbase[o + i] = sbase[coff[i]];
        else dbase[coff[i]] = sbase[o + i];
      }
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
