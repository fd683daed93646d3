// internal.h — shared definitions of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dfm {

// ---------------------------------------------------------------------------
// HBM layout of an MXFP4 matrix ("fragment layout")
//
// A matrix of R rows x K columns (R % 16 == 0, K % 64 == 0) is stored as
// tiles of 16 rows x K. A tile is K/64 groups of 544 bytes, one per 64
// columns, so one 16-byte load per lane streams a tile front to back:
//   bytes [0, 512): codes, 32 lanes x 16 bytes. Lane l = 4g + t holds, for
//     the four 16-column k-steps s of group G (k0 = 64G + 16s), the four bytes
//     of an m16n8k16 A fragment:
//       byte 0: (row g,   cols k0+2t, k0+2t+1)   byte 1: (row g+8, same cols)
//       byte 2: (row g,   cols k0+2t+8, +9)      byte 3: (row g+8, same cols)
//     each the canonical byte of that row (low nibble = even column);
//   bytes [512, 544): E8M0 scales, 8 x 4 bytes; entry g holds
//       (row g, block 2G), (row g, block 2G+1), (row g+8, block 2G),
//       (row g+8, block 2G+1).
//   codes  offset = (j*K/64 + G)*544 + 16 l + 4 s + byte
//   scales offset = (j*K/64 + G)*544 + 512 + 4 g + i
// The total size equals the canonical one (K/2 + K/32 bytes a row).
// ---------------------------------------------------------------------------
constexpr int kGroupBytes = 544;
__host__ __device__ inline int mx_ngroups(int K) { return K >> 6; }
__host__ __device__ inline size_t mx_tile_bytes(int K) {
  return (size_t)mx_ngroups(K) * kGroupBytes;
}
__host__ __device__ inline int mx_nchunks(int K) { return (K + 511) >> 9; }
__host__ __device__ inline int mx_nv(int K, int c) {  // 64-column groups of chunk c
  int r = (K >> 6) - 8 * c;
  return r < 8 ? r : 8;
}

// Expert span in device layout:
//   [gate/up: 2I/16 tiles, K = H; tile j rows 0-7 = gate rows 8j..8j+7,
//    rows 8-15 = up rows 8j..8j+7]
//   [down: H/16 tiles, K = I; tile j = rows 16j..16j+15]
struct SpanLayout {
  size_t gu, dn, bytes;
};
__host__ __device__ inline SpanLayout span_layout(int H, int I) {
  SpanLayout L;
  L.gu = 0;
  L.dn = (size_t)(2 * I / 16) * mx_tile_bytes(H);
  L.bytes = L.dn + (size_t)(H / 16) * mx_tile_bytes(I);
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
  K_SHARED_DN, K_RMSNORM, K_RESIDUAL, K_REPACK, K_OTHER, K_MX8_QUANT, K_GEMM_GU,
  K_GEMM_DN, K_CACHE_FILL, K_MX8_GU, K_MX8_DN, K_NKINDS
};

// Launches `kernel` as a programmatic dependent of the previous kernel in
// the stream: its grid may be set up, and its CTAs may start, while the
// previous kernel's last CTAs finish; the kernel itself waits for the
// previous grid's completion (griddepcontrol.wait) before reading its
// results.
template <typename... KArgs, typename... Args>
cudaError_t launch_after_previous(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, (KArgs)args...);
}

// Error word bits written by device-side checks.
enum : uint32_t { DEV_ERR_RANGE = 1u, DEV_ERR_TIMEOUT = 2u };

// Message returned by df_moe_last_error(NULL) on this thread.
void set_thread_error(const char* msg);

// ---- launchers (each returns cudaGetLastError()) ---------------------------
// max_ctas (persistent kernels): at most this many CTAs, one per SM (0: all
// SMs), so that two chains of kernels can run side by side on split SMs.
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
// after_previous: launched as a programmatic dependent of the kernel before it
// (its weights are then read before it waits for that kernel, so they must
// not be written by it); false: an ordinary launch.
cudaError_t launch_router(const float* Wr, int E, int H, const uint16_t* x,
                          int T, float* part, RouterSplit sp, cudaStream_t s,
                          const RouterFuse* fuse = nullptr, bool after_previous = true);
cudaError_t launch_topk(const float* part, int nsplit, int T, int E, int k,
                        float* logits_out, int32_t* ids, float* w,
                        Item* items, int32_t* n_items, int32_t* sorted,
                        cudaStream_t s);
// ids outside [0, E) are left out and recorded in *err (DEV_ERR_RANGE).
// inv (optional, [T*k]): the position of assignment a in expert order
// (sorted[inv[a]] = a), -1 for an assignment left out.
cudaError_t launch_group(const int32_t* ids, int T, int k, int E,
                         int32_t* offs, int32_t* tok, int32_t* slot,
                         int32_t* n_union, Item* items, int32_t* n_items,
                         int32_t* sorted, int tg, uint32_t* err, cudaStream_t s,
                         int32_t* inv = nullptr);
// E: experts of the layer, nassign: T * k (range checks of the items).
cudaError_t launch_gateup(const uint8_t* arena, size_t span_bytes, int H,
                          int I, int k, const uint16_t* x, const Item* items,
                          const int32_t* n_items, int max_items,
                          const int32_t* sorted, float* hbuf, int tg, int E, int nassign,
                          uint32_t* err, cudaStream_t s, int max_ctas = 0);
// after_gateup: the preceding kernel on `s` is the gate/up kernel of the same
// selection (so the selection is complete when this grid starts, and the
// weight stream may begin before h is).
cudaError_t launch_down(const uint8_t* arena, size_t span_bytes, int H, int I,
                        const Item* items, const int32_t* n_items,
                        int max_items, const int32_t* sorted,
                        const float* hbuf, float* part, int tg, int E, int nassign,
                        uint32_t* err, cudaStream_t s, int max_ctas = 0,
                        bool after_gateup = false);
// err_mirror (or null): the host-visible copy of the error word, written when
// the word is nonzero. ids_out / w_out (or null; k <= 128): copies of the
// selection ids [T][k] and weights w (host memory the device writes
// directly, for the host-buffer forward).
cudaError_t launch_combine(const float* part, const float* w, int T, int k,
                           int H, const float* ysh, const uint16_t* residual,
                           float* out_f32, uint16_t* out_bf16, uint32_t* err,
                           uint32_t* err_mirror, cudaStream_t s, const int32_t* ids = nullptr,
                           int32_t* ids_out = nullptr, float* w_out = nullptr);
// A 16-byte-aligned copy of `bytes` (a multiple of 16) by a small kernel,
// e.g. from host memory the device reads directly into device memory.
cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t s);
cudaError_t launch_shared_gateup(const uint16_t* gate, const uint16_t* up,
                                 int R, int H, const uint16_t* x, int T,
                                 float* hsh, uint32_t* err, cudaStream_t s,
                                 int max_ctas = 0);
cudaError_t launch_shared_down(const uint16_t* down, int H, int K,
                               const float* hsh, int T, float* ysh,
                               uint32_t* err, cudaStream_t s, int max_ctas = 0);
cudaError_t launch_rmsnorm(const uint16_t* x, int T, int H, float eps,
                           uint16_t* xn, cudaStream_t s);
// Largest decode batch: up to this many tokens a call run as decode batches
// (the phase kernels below); larger calls are batches (tcgen05 GEMMs).
constexpr int kDecodeMaxT = 8;

// Decode batches (T <= kDecodeMaxT): routed and shared experts in two phase
// kernels on every SM (k_phase.cu). The gate/up phase follows the router
// (T = 1: it selects the experts itself from the partial logits
// router_part [nsplit][E], writing ids, w, items, n_items and sorted) or the
// grouping kernel (T > 1: items, n_items, sorted are its inputs) directly on
// `s`; the down phase follows the gate/up phase directly. R = n_shared * Is
// (0: no shared experts). n_sh: CTAs (of one per SM) that run the shared
// experts, in [1, SMs - 1] (0 when R = 0); the others run the routed ones.
// spans: device [E] of span addresses (expert cache), or null for arena + e
// * span_bytes.
bool phase_supported(int H, int I, int R, int E, int k);

// Read-only streaming probe: 16-byte loads over `bytes`, one word a thread
// into sink (at least 8 * SMs * 256 words).
cudaError_t launch_stream_read(const void* buf, size_t bytes, uint32_t* sink, cudaStream_t s);
// Expert cache fill: one span copy of the plan (device-visible memory, n
// entries): `span_bytes` (a multiple of 16) from src (pinned host memory,
// mapped) to dst (an HBM slot), then span_tab[e] = dst.
struct CacheCopy {
  const void* src;
  void* dst;
  long long e;
};
cudaError_t launch_cache_fill(const CacheCopy* plan, int n, size_t span_bytes,
                              unsigned long long* span_tab, cudaStream_t s);
// drop: the test hook (one stage of the routed gate/up never filled, short
// waits), so that a bounded wait runs out.
cudaError_t launch_phase_gateup(const uint16_t* sh_gate, const uint16_t* sh_up, int R,
                                const uint8_t* arena, size_t span_bytes, int H, int I, int k,
                                const uint16_t* x, int T, Item* items, int32_t* n_items,
                                int32_t* sorted, const float* router_part, int nsplit, int E,
                                int32_t* ids, float* w, float* hsh, float* hbuf, uint32_t* err,
                                int n_sh, const uint8_t* const* spans, bool drop,
                                cudaStream_t s);
cudaError_t launch_phase_down(const uint8_t* arena, size_t span_bytes, int H, int I, int E,
                              int k, const Item* items, const int32_t* n_items,
                              const int32_t* sorted, const float* hbuf, float* part,
                              const uint16_t* sh_down, int R, const float* hsh, int T, float* ysh,
                              uint32_t* err, int n_sh, const uint8_t* const* spans,
                              cudaStream_t s);
cudaError_t launch_repack_span(const uint8_t* src, uint8_t* dst, int n_spans,
                               int H, int I, int inverse, cudaStream_t s);

// ---- routed experts of large batches on tcgen05 (k_gemm.cu) ----------------
// Grouped GEMMs over the items (one per expert, all of its tokens): the MXFP4
// weights decoded to f16 (times 2^(e - r), r a per-row reference exponent)
// straight into tensor memory, multiplied by f16 token columns on the tensor
// cores with fp32 accumulators in tensor memory. Same outputs as
// launch_gateup / launch_down with one item per expert.
bool gemm_supported(int H, int I);
// A TMA tensor map (CUtensorMap), opaque here.
struct alignas(64) ChunkMap {
  uint64_t w[16];
};
// Tensor maps of the gate/up and down tiles of an arena of E spans; false if
// the driver's encoder is unavailable or refuses the shape.
bool make_chunk_maps(const uint8_t* arena, size_t span_bytes, int H, int I, int E,
                     ChunkMap* gu, ChunkMap* dn);
// Row reference exponents: [E][2I + H] bytes, fragment row order (gate/up
// tile rows, then down rows), written by launch_row_ref for `n` spans.
size_t gemm_eref_bytes(int n_experts, int H, int I);
cudaError_t launch_row_ref(const uint8_t* spans, size_t span_bytes, int H, int I, int n,
                           uint8_t* eref, cudaStream_t s);
// B rows in expert order (R = T*k assignments, row p for sorted[p]):
// gate/up xg [R][H] f16 = x[sorted[p] / k] * 2^-s_p (exact), bsc[p] = 2^s_p;
cudaError_t launch_prep_x(const uint16_t* x, int R, int H, int k, const int32_t* sorted,
                          uint16_t* xg, float* bsc, uint32_t* err, cudaStream_t s);
// down hh [R][2][I] f16 = high and low parts of h[sorted[p]] * 2^-s_p.
cudaError_t launch_split_h(const float* h, int R, int I, const int32_t* sorted, uint16_t* hh,
                           float* bsc, uint32_t* err, cudaStream_t s);
// Tensor maps of xg ([R][H]) and hh ([2R][I]) for rows allocated for R.
bool make_b_maps(const uint16_t* xg, const uint16_t* hh, int R, int H, int I, ChunkMap* gu,
                 ChunkMap* dn);
cudaError_t launch_gemm_gateup(const ChunkMap& map, const ChunkMap& bmap, const uint8_t* arena,
                               size_t span_bytes, const uint8_t* eref, int H, int I, int k,
                               const float* bsc, const Item* items, const int32_t* n_items,
                               int max_items, const int32_t* sorted, float* hbuf, int E,
                               int nassign, uint32_t* err, cudaStream_t s);
cudaError_t launch_gemm_down(const ChunkMap& map, const ChunkMap& bmap, const uint8_t* arena,
                             size_t span_bytes, const uint8_t* eref, int H, int I, int k,
                             const float* bsc, const Item* items, const int32_t* n_items,
                             int max_items, const int32_t* sorted, float* part, int E,
                             int nassign, uint32_t* err, cudaStream_t s);

// ---- shared experts of large batches on tcgen05 (k_dense.cu) ----------------
// Tensor maps of one layer's shared-expert weights (gate, up [R][H]; down
// [H][R]; bf16) and of the h rows handed from GEMM 1 to GEMM 2 ([3 max_T][R]).
struct SharedMaps {
  ChunkMap gate, up, down, hh;
};
bool dense_supported(int H, int R);
bool make_shared_maps(const uint16_t* gate, const uint16_t* up, const uint16_t* down, int H,
                      int R, const uint16_t* hh, int max_rows, SharedMaps* out);
// h = silu(gate x) * (up x) as three bf16 parts, rows hh [T][3][R] (x: bf16
// [T][H], 16-byte aligned).
cudaError_t launch_shared_gemm_gateup(const SharedMaps& m, const uint16_t* x, int T, int H,
                                      int R, uint16_t* hh, uint32_t* err, cudaStream_t s);
// y [T][H] = down (high + middle + low).
cudaError_t launch_shared_gemm_down(const SharedMaps& m, int T, int H, int R, float* y,
                                    uint32_t* err, cudaStream_t s);

// ---- router logits of batches on tcgen05 (k_dense.cu) ------------------------
// The fp32 router weights as three bf16 parts per row ([E][3H]: high,
// middle, low, summing to the weight), written once at load; a dense bf16
// GEMM of x against them gives fp32 logits with exact products. K is split
// over CTAs to fill `sms` SMs: split s writes part[s][T][E] (summed by the
// top-k kernel). max_rows bounds splits x T (the part buffer's rows; 0: no
// bound). H: a multiple of 64.
int router_tc_splits(int E, int H, int T, int sms, size_t max_rows);
// the largest splits x T over batches of Tmin .. Tmax tokens
size_t router_tc_part_rows(int E, int H, int Tmin, int Tmax, int sms);
cudaError_t launch_router_parts(const float* w, int E, int H, uint16_t* out, cudaStream_t s);
bool make_router_map(const uint16_t* parts, int E, int H, ChunkMap* out);
// returns the number of partial planes written, -1 on a launch or encoding
// failure (x: bf16 [T][H], 16-byte aligned)
int launch_router_tc(const ChunkMap& map, const uint16_t* x, int T, int E, int H, float* part,
                     size_t max_rows, int sms, uint32_t* err, cudaStream_t s);

// ---- routed experts on block-scaled MXFP4 x E4M3 GEMMs (k_mx8.cu) ----------
// Grouped GEMMs on tcgen05.mma kind::mxf8f6f4 with the MXFP4 codes and
// scales of each 128-row tile arranged stage by stage, the activations in
// E4M3 with an E8M0 exponent per 32: one plane (the lossy MXFP8 variant: the
// activation rounded to the format) or several planes whose sum reproduces
// the activation (x: kPlanesX, h: kPlanesH; the exact path for batches).
constexpr int kPlanesX = 4, kPlanesH = 5;
bool mx8_supported(int H, int I);
// Rows of an expert-ordered activation buffer for nassign assignments of
// `planes` rows each, and the rows that a stage's 32-row scale chunk or its
// B box reads past the last one.
int mx8_rows_cap(int nassign, int planes);
// B rows a box of the batch GEMM's activation map for `planes` (the row map
// of a handle's x or h rows is made with it).
int mx8_box_rows(int planes);
// Tensor maps of the gate, up and down codes of an arena of E spans.
bool make_mx8_maps(const uint8_t* arena, size_t span_bytes, int H, int I, int E, ChunkMap* gate,
                   ChunkMap* up, ChunkMap* down);
// Tensor map of E4M3 activation rows [rows_cap][K], written as `planes`
// rows a token or assignment (its box covers one pass of the GEMM).
bool make_mx8_row_map(const uint8_t* rows, int rows_cap, int K, int planes, ChunkMap* map,
                      int box_rows = 0);
// Rounds h for the down GEMM: row n of item i is source row sorted[pos + n]
// of src (fp32 [nassign][K], 16-byte aligned), written as `planes` E4M3 rows
// (pos + n) planes + p of q ([rows_cap][K]) with their scales as row-major
// scale rows in sfp ([rows_cap][K/32]). planes: 1 or kPlanesH. With gu_part
// (kPlanesH only) the source rows are h = silu(gate) * up of the kspl parts'
// gate and up sums ([kspl][nassign][2][K], added in part order); src unused.
cudaError_t launch_mx8_rows(const float* src, int K, int planes, const Item* items,
                            const int32_t* n_items, int max_items, const int32_t* sorted,
                            int nassign, int E, uint8_t* q, int rows_cap, uint8_t* sfp,
                            uint32_t* err, cudaStream_t s, const float* gu_part = nullptr,
                            int kspl = 0);
// Rounds x (bf16 [T][K], 16-byte aligned, K <= 8192) for the gate/up GEMM:
// each token once, written to the rows of its k assignments, rows
// inv[t k + j] planes + p of q, scale rows as above. inv: the grouping's
// positions of the assignments (-1: none; null: position = assignment).
// planes: 1 or kPlanesX.
cudaError_t launch_mx8_xrows(const uint16_t* x, int K, int k, int T, const int32_t* inv,
                             int planes, uint8_t* q, int rows_cap, uint8_t* sfp, uint32_t* err,
                             cudaStream_t s);
// The GEMM's scales sf ([K/128][rows_cap][16], word q of a row the scales
// of the row 32 q later) from the row-major scale rows sfp of the first
// `rows` rows.
cudaError_t launch_mx8_scale_lines(const uint8_t* sfp, int K, int rows, int rows_cap,
                                   int planes, uint8_t* sf, cudaStream_t s);
// The rounding on plain rows: codes [rows][n], scales [rows][n/32].
cudaError_t launch_mx8_plain(const float* v, int rows, int n, uint8_t* codes, uint8_t* scales,
                             cudaStream_t s);
// Canonical spans -> the variant's span layout (inverse: back).
cudaError_t launch_mx8_layout(const uint8_t* src, uint8_t* dst, int n_spans, int H, int I,
                              size_t span_bytes, int inverse, cudaStream_t s);
// gate/up on x's planes (1 or kPlanesX). One plane: h rounded to MXFP8
// into hq/hsf (hrows_cap rows) for the down GEMM, and optionally h before
// the rounding into hbuf [nassign][I]; kPlanesX: h into hbuf (split into its
// planes by launch_mx8_rows).
cudaError_t launch_mx8_gateup(const ChunkMap& gate, const ChunkMap& up, const ChunkMap& xmap,
                              const uint8_t* arena, size_t span_bytes, int H, int I,
                              const uint8_t* xsf, int rows_cap, const Item* items,
                              const int32_t* n_items, int max_items, const int32_t* sorted,
                              int E, int nassign, float* hbuf, uint8_t* hq, uint8_t* hsf,
                              int hrows_cap, int planes, uint32_t* err, cudaStream_t s);
// down on h's planes (1 or kPlanesH): part [nassign][H].
cudaError_t launch_mx8_down(const ChunkMap& down, const ChunkMap& hmap, const uint8_t* arena,
                            size_t span_bytes, int H, int I, const uint8_t* hsf, int rows_cap,
                            const Item* items, const int32_t* n_items, int max_items,
                            const int32_t* sorted, int E, int nassign, float* part,
                            int planes, uint32_t* err, cudaStream_t s);

// One token on an exact-planes handle as two phase kernels (one CTA an SM;
// the first n_sh CTAs stream the shared experts, R > 0). Gate/up: x's planes
// at rows 4j .. 4j + 3 for every rank j (launch_mx8_xrows with k, no inv);
// each routed CTA selects the experts from the router's partial logits
// (nsplit planes) and the first publishes them (items, sorted, n_items, ids,
// w); the routed gate/up writes gate and up sums over mx8_phase_kspl(H)
// parts of K into gu_part [kspl][k][2][I] (SwiGLU by launch_mx8_rows); the
// shared CTAs write hsh. Down: h's planes at rows 5j .. 5j + 4; part [k][H]
// and ysh. Row maps: boxes of 16 rows.
int mx8_phase_kspl(int H);
bool mx8_phase_supported(int H, int I, int R);
cudaError_t launch_mx8_phase_gateup(const ChunkMap& gate, const ChunkMap& up,
                                    const ChunkMap& xmap16, const uint8_t* arena,
                                    size_t span_bytes, int H, int I, const uint8_t* xsf,
                                    int rows_cap, Item* items, int32_t* n_items,
                                    int32_t* sorted, int E, int k, const float* router_part,
                                    int nsplit, int32_t* ids, float* w, float* gu_part,
                                    const uint16_t* sh_gate, const uint16_t* sh_up, int R,
                                    const uint16_t* x, float* hsh, uint32_t* err, int n_sh,
                                    cudaStream_t s);
cudaError_t launch_mx8_phase_down(const ChunkMap& down, const ChunkMap& hmap16,
                                  const uint8_t* arena, size_t span_bytes, int H, int I,
                                  const uint8_t* hsf, int rows_cap, const Item* items,
                                  const int32_t* n_items, const int32_t* sorted, int E, int k,
                                  float* part, const uint16_t* sh_down, int R, const float* hsh,
                                  float* ysh, uint32_t* err, int n_sh, cudaStream_t s);

}  // namespace dfm
