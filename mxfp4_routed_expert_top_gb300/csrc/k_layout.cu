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



// ---------------------------------------------------------------------------
// Shared experts as f16 m16n8k16 A fragments.
//
// The shared-expert weights are bf16. The layer kernel multiplies them on the
// tensor cores in f16, which holds every bf16 value exactly once the row is
// scaled by a power of two that puts its largest magnitude in [2^14, 2^15):
// f16 normals then cover 2^28 below the row maximum (with bf16's 8-bit
// significand inside f16's 11), and smaller values keep an absolute error
// below 2^-39 of the row maximum. The scale is applied back in fp32 after
// the contraction.
//
// Tiles are 16 rows x K; k-step s of tile j is 32 lanes x 16 bytes, lane
// l = 4g + t holding {(g, 16s+2t), (g, +1)}, {(g+8, 16s+2t), +1},
// {(g, 16s+2t+8), +1}, {(g+8, 16s+2t+8), +1} as f16x2 (first column low).
// gate/up tile j: rows 0-7 = gate rows 8j..8j+7, rows 8-15 = up rows
// 8j..8j+7; down tile j: rows 16j..16j+15.
// ---------------------------------------------------------------------------
namespace {

__device__ inline float bf16_val(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

// Exponent sc of the power-of-two row scale (largest |w| in [2^14, 2^15) after
// multiplying by 2^-sc); 0 for an all-zero row.
__device__ inline int row_scale_exp(float m) {
  if (!(m > 0.f)) return 0;
  const int e = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;
  int sc = e - 14;
  return sc < -126 ? -126 : (sc > 127 ? 127 : sc);
}

// One warp per row. rows [0, Is): gate, [Is, 2Is): up, [2Is, 2Is+H): down.
__global__ void shared_row_scales(const uint16_t* __restrict__ gate,
                                  const uint16_t* __restrict__ up,
                                  const uint16_t* __restrict__ down, int down_ld,
                                  int H, int Is, float* __restrict__ gu_rs,
                                  float* __restrict__ dn_rs) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int nrows = 2 * Is + H;
  if (warp >= nrows) return;
  const uint16_t* row;
  int len;
  if (warp < Is) { row = gate + (size_t)warp * H; len = H; }
  else if (warp < 2 * Is) { row = up + (size_t)(warp - Is) * H; len = H; }
  else { row = down + (size_t)(warp - 2 * Is) * down_ld; len = Is; }
  float m = 0.f;
  for (int c = lane; c < len; c += 32) m = fmaxf(m, fabsf(bf16_val(row[c])));
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) {
    const float rs = ldexpf(1.0f, row_scale_exp(m));
    if (warp < 2 * Is) {
      const int r = warp < Is ? warp : warp - Is;
      gu_rs[(size_t)(r >> 3) * 16 + (warp < Is ? 0 : 8) + (r & 7)] = rs;
    } else {
      dn_rs[warp - 2 * Is] = rs;
    }
  }
}

__device__ inline uint32_t pack_pair(const uint16_t* p, int sc) {
  const __half2 h = __floats2half2_rn(ldexpf(bf16_val(p[0]), -sc), ldexpf(bf16_val(p[1]), -sc));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// One thread per 16-byte fragment: gate/up units first, then down units.
__global__ void shared_pack(const uint16_t* __restrict__ gate,
                            const uint16_t* __restrict__ up,
                            const uint16_t* __restrict__ down, int down_ld, int H,
                            int Is, const float* __restrict__ gu_rs,
                            const float* __restrict__ dn_rs, uint4* __restrict__ gu_out,
                            uint4* __restrict__ dn_out) {
  const size_t n_gu = (size_t)(Is / 8) * (H / 16) * 32;
  const size_t n_dn = (size_t)(H / 16) * (Is / 16) * 32;
  for (size_t u = (size_t)blockIdx.x * blockDim.x + threadIdx.x; u < n_gu + n_dn;
       u += (size_t)gridDim.x * blockDim.x) {
    const bool gu = u < n_gu;
    const size_t v = gu ? u : u - n_gu;
    const int lane = (int)(v & 31);
    const size_t tk = v >> 5;
    const int nks = gu ? H / 16 : Is / 16;
    const int j = (int)(tk / nks), ks = (int)(tk % nks);
    const int g = lane >> 2, t = lane & 3;
    const int c0 = 16 * ks + 2 * t;
    const uint16_t *r0, *r1;
    int s0, s1;
    if (gu) {
      r0 = gate + (size_t)(8 * j + g) * H;
      r1 = up + (size_t)(8 * j + g) * H;
      s0 = (int)(__float_as_uint(gu_rs[(size_t)j * 16 + g]) >> 23) - 127;
      s1 = (int)(__float_as_uint(gu_rs[(size_t)j * 16 + 8 + g]) >> 23) - 127;
    } else {
      r0 = down + (size_t)(16 * j + g) * down_ld;
      r1 = down + (size_t)(16 * j + g + 8) * down_ld;
      s0 = (int)(__float_as_uint(dn_rs[16 * j + g]) >> 23) - 127;
      s1 = (int)(__float_as_uint(dn_rs[16 * j + g + 8]) >> 23) - 127;
    }
    const uint4 o = make_uint4(pack_pair(r0 + c0, s0), pack_pair(r1 + c0, s1),
                               pack_pair(r0 + c0 + 8, s0), pack_pair(r1 + c0 + 8, s1));
    if (gu) gu_out[v] = o;
    else dn_out[v] = o;
  }
}

}  // namespace

cudaError_t launch_pack_shared(const uint16_t* gate, const uint16_t* up,
                               const uint16_t* down, int down_ld, int H, int Is,
                               uint4* gu_out, float* gu_rs, uint4* dn_out,
                               float* dn_rs, cudaStream_t s) {
  const int rows = 2 * Is + H;
  shared_row_scales<<<(rows * 32 + 255) / 256, 256, 0, s>>>(gate, up, down, down_ld, H, Is,
                                                            gu_rs, dn_rs);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t n = (size_t)(Is / 8) * (H / 16) * 32 + (size_t)(H / 16) * (Is / 16) * 32;
  size_t grid = (n + 255) / 256;
  if (grid > 152 * 32) grid = 152 * 32;
  shared_pack<<<(unsigned)grid, 256, 0, s>>>(gate, up, down, down_ld, H, Is, gu_rs, dn_rs,
                                            gu_out, dn_out);
  return cudaGetLastError();
}

}  // namespace dfm
