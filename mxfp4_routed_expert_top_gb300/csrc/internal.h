// internal.h — shared definitions of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dfm {

// ---------------------------------------------------------------------------
// HBM layout of an MXFP4 matrix ("fragment layout")
//
// A matrix of R rows x K columns (R % 16 == 0, K % 64 == 0) is stored as
// tiles of 16 rows x K. Inside a tile, columns go in chunks of up to 512
// (chunk c holds 64-column groups v = 0 .. nv(c)-1), and every 64-column
// group is 512 bytes: 32 lanes x 16 bytes, lane l = 4 g + t holding, for the
// four 16-column k-steps s = 0..3 of the group (k0 = 512c + 64v + 16s), the
// four bytes of an m16n8k16 A fragment:
//   byte 0: (row g,   cols k0+2t, k0+2t+1)   byte 1: (row g+8, same cols)
//   byte 2: (row g,   cols k0+2t+8, +9)      byte 3: (row g+8, same cols)
// Each byte is the canonical byte of that row (low nibble = even column).
//   codes  offset = j*8K + 512*(8c + v) + 16 l + 4 s + byte
//   scales offset = j*K/2 + 256 c + g*2*nbc(c) + i,  i < nbc(c): row g,
//                   block 16c+i; i >= nbc(c): row g+8, block 16c+i-nbc(c)
// A tile's codes (8K bytes) and scales (K/2 bytes) are each contiguous. The
// total size equals the canonical one (K/2 + K/32 bytes a row).
// ---------------------------------------------------------------------------
__host__ __device__ inline int mx_nb(int K) { return K >> 5; }
__host__ __device__ inline int mx_nchunks(int K) { return (K + 511) >> 9; }
__host__ __device__ inline int mx_nv(int K, int c) {  // 64-column groups of chunk c
  int r = (K >> 6) - 8 * c;
  return r < 8 ? r : 8;
}
__host__ __device__ inline int mx_nbc(int K, int c) { return 2 * mx_nv(K, c); }

// Expert span in device layout:
//   [gate/up codes: 2I/16 tiles, K = H; tile j rows 0-7 = gate rows 8j..8j+7,
//    rows 8-15 = up rows 8j..8j+7]
//   [gate/up scales]
//   [down codes: H/16 tiles, K = I; tile j = rows 16j..16j+15]
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

// Work items hold one expert and all of its tokens (the expert kernels walk
// them in token groups against each tile held in shared memory).
constexpr int kOneItemPerExpert = 1 << 20;

enum KernelKind {
  K_ROUTER = 0, K_TOPK, K_GROUP, K_GATEUP, K_DOWN, K_COMBINE, K_SHARED_GU,
  K_SHARED_DN, K_RMSNORM, K_RESIDUAL, K_REPACK, K_OTHER, K_NKINDS
};

// Error word bits written by device-side checks.
enum : uint32_t { DEV_ERR_RANGE = 1u, DEV_ERR_TIMEOUT = 2u };

// Message returned by df_moe_last_error(NULL) on this thread.
void set_thread_error(const char* msg);

// ---- launchers (each returns cudaGetLastError()) ---------------------------
// Router column split: `nsplit` column ranges of `split_len` (a multiple of
// 128, at most 2048) so that E * nsplit warps keep HBM busy.
struct RouterSplit { int split_len, nsplit; };
inline RouterSplit router_split(int E, int H) {
  int want = (3000 + E - 1) / E;
  const int maxs = (H + 127) / 128;
  if (want < 1) want = 1;
  if (want > maxs) want = maxs;
  int len = (H + want - 1) / want;
  len = (len + 127) / 128 * 128;
  while (len > 2048) {
    ++want;
    len = ((H + want - 1) / want + 127) / 128 * 128;
  }
  return RouterSplit{len, (H + len - 1) / len};
}
// Optional: for a single token the router's last block also selects the
// experts (saving the top-k launch); `counter` must be zero between calls.
struct RouterFuse {
  unsigned int* counter;
  int k;
  int32_t* ids;
  float* w;
  Item* items;
  int32_t* n_items;
  int32_t* sorted;
};
cudaError_t launch_router(const float* Wr, int E, int H, const uint16_t* x,
                          int T, float* part, RouterSplit sp, cudaStream_t s,
                          const RouterFuse* fuse = nullptr);
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
                          uint32_t* err, cudaStream_t s);
cudaError_t launch_down(const uint8_t* arena, size_t span_bytes, int H, int I,
                        const Item* items, const int32_t* n_items,
                        int max_items, const int32_t* sorted,
                        const float* hbuf, float* part, int tg, uint32_t* err,
                        cudaStream_t s);
cudaError_t launch_combine(const float* part, const float* w, int T, int k,
                           int H, const float* ysh, const uint16_t* residual,
                           float* out_f32, uint16_t* out_bf16, cudaStream_t s);
cudaError_t launch_shared_gateup(const uint16_t* gate, const uint16_t* up,
                                 int R, int H, const uint16_t* x, int T,
                                 float* hsh, uint32_t* err, cudaStream_t s);
cudaError_t launch_shared_down(const uint16_t* down, int H, int K,
                               const float* hsh, int T, float* ysh,
                               uint32_t* err, cudaStream_t s);
cudaError_t launch_rmsnorm(const uint16_t* x, int T, int H, float eps,
                           uint16_t* xn, cudaStream_t s);
cudaError_t launch_repack_span(const uint8_t* src, uint8_t* dst, int n_spans,
                               int H, int I, int inverse, cudaStream_t s);

}  // namespace dfm
