// internal.h — shared definitions of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dfm {

// ---------------------------------------------------------------------------
// HBM layout of an MXFP4 matrix ("pair-chunk" layout)
//
// A matrix of R rows x K columns (R % 32 == 0, K % 32 == 0) has NB = K / 32
// blocks of 32 elements per row (16 code bytes + 1 scale byte per block).
// Rows are taken in pairs P = (2P, 2P+1) and columns in chunks of up to 16
// blocks (512 elements): chunk c holds blocks 16c .. 16c + nbc(c) - 1.
//
//   codes: byte offset of (pair P, chunk c, row-in-pair r, block b, byte j)
//          = P * K + 512 c + (r * nbc(c) + b) * 16 + j
//          so one warp-wide 16-byte load per lane (lane = 16 r + b) reads the
//          whole (pair, chunk) tile as 512 contiguous bytes.
//   scales: pairs are grouped by 16 (32 rows). Byte offset of
//          (group G, chunk c, r, b, pair-in-group i)
//          = G * 32 * NB + 512 c + (r * nbc(c) + b) * 16 + i
//          so one 16-byte load gives a lane the scales of its block for all
//          16 pairs of the group.
//
// Byte j of a block keeps the canonical nibble order (element 2j in the low
// nibble). The total size equals the canonical one (K/2 + K/32 bytes a row).
// ---------------------------------------------------------------------------
__host__ __device__ inline int mx_nb(int K) { return K >> 5; }
__host__ __device__ inline int mx_nchunks(int K) { return (mx_nb(K) + 15) >> 4; }
__host__ __device__ inline int mx_nbc(int K, int c) {
  int r = mx_nb(K) - 16 * c;
  return r < 16 ? r : 16;
}

// Expert span in device layout:
//   [gate/up codes: I pairs (pair i = gate row i, up row i), K = H]
//   [gate/up scales]
//   [down codes: H/2 pairs (rows 2p, 2p+1), K = I]
//   [down scales]
struct SpanLayout {
  size_t gu_codes, gu_scales, dn_codes, dn_scales, bytes;
};
__host__ __device__ inline SpanLayout span_layout(int H, int I) {
  SpanLayout L;
  size_t hi = (size_t)H * (size_t)I;
  L.gu_codes = 0;
  L.gu_scales = hi;              // 2I rows * H/2
  L.dn_codes = hi + hi / 16;     // + 2I rows * H/32
  L.dn_scales = L.dn_codes + hi / 2;
  L.bytes = L.dn_scales + hi / 32;
  return L;
}

// Work item of the expert kernels: expert `e` applied to `cnt` (<= TG)
// assignments listed at sorted[pos .. pos + cnt).
struct Item {
  int32_t e, pos, cnt, pad;
};

constexpr int kMaxTG = 2;  // tokens per work item

enum KernelKind {
  K_ROUTER = 0, K_TOPK, K_GROUP, K_GATEUP, K_DOWN, K_COMBINE, K_SHARED_GU,
  K_SHARED_DN, K_RMSNORM, K_RESIDUAL, K_REPACK, K_OTHER, K_NKINDS
};

// Error word bits written by device-side checks.
enum : uint32_t { DEV_ERR_RANGE = 1u, DEV_ERR_TIMEOUT = 2u };

// Message returned by df_moe_last_error(NULL) on this thread.
void set_thread_error(const char* msg);

// ---- launchers (each returns cudaGetLastError()) ---------------------------
// Router K-split: partial logits of `nsplit` column ranges of `split_len`.
struct RouterSplit { int split_len, nsplit; };
inline RouterSplit router_split(int E, int H) {
  int row_blocks = (E + 7) / 8;
  int want = (2 * 152 + row_blocks - 1) / row_blocks;
  int maxs = H / 128 > 0 ? H / 128 : 1;
  if (want < 1) want = 1;
  if (want > maxs) want = maxs;
  int len = (H + want - 1) / want;
  len = (len + 127) / 128 * 128;
  return RouterSplit{len, (H + len - 1) / len};
}
cudaError_t launch_router(const float* Wr, int E, int H, const uint16_t* x,
                          int T, float* part, RouterSplit sp, cudaStream_t s);
cudaError_t launch_topk(const float* part, int nsplit, int T, int E, int k,
                        float* logits_out, int32_t* ids, float* w,
                        Item* items, int32_t* n_items, int32_t* sorted,
                        cudaStream_t s);
cudaError_t launch_group(const int32_t* ids, int T, int k, int E,
                         int32_t* offs, int32_t* tok, int32_t* slot,
                         int32_t* n_union, Item* items, int32_t* n_items,
                         int32_t* sorted, int tg, cudaStream_t s);
cudaError_t launch_gateup(const uint8_t* arena, size_t span_bytes, int H,
                          int I, int k, const uint16_t* x, const Item* items,
                          const int32_t* n_items, int max_items,
                          const int32_t* sorted, float* hbuf, int tg,
                          cudaStream_t s);
cudaError_t launch_down(const uint8_t* arena, size_t span_bytes, int H, int I,
                        const Item* items, const int32_t* n_items,
                        int max_items, const int32_t* sorted,
                        const float* hbuf, float* part, int tg,
                        cudaStream_t s);
cudaError_t launch_combine(const float* part, const float* w, int T, int k,
                           int H, const float* ysh, const uint16_t* residual,
                           float* out_f32, uint16_t* out_bf16, cudaStream_t s);
cudaError_t launch_shared_gateup(const uint16_t* gate, const uint16_t* up,
                                 int R, int H, const uint16_t* x, int T,
                                 float* hsh, cudaStream_t s);
cudaError_t launch_shared_down(const uint16_t* down, int H, int K,
                               const float* hsh, int T, float* ysh,
                               cudaStream_t s);
cudaError_t launch_rmsnorm(const uint16_t* x, int T, int H, float eps,
                           uint16_t* xn, cudaStream_t s);
cudaError_t launch_repack_span(const uint8_t* src, uint8_t* dst, int n_spans,
                               int H, int I, int inverse, cudaStream_t s);

}  // namespace dfm
