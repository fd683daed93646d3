// abi.cu — the C ABI (include/df_moe.h): handle, weight arenas, workspace,
// loading, and the forward orchestration of the kernels.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "df_moe.h"
#include "internal.h"

using namespace dfm;

namespace {

thread_local std::string g_thread_err;

struct LayerBufs {
  uint8_t* arena = nullptr;   // E spans, device layout
  float* router = nullptr;    // [E][H]
  uint16_t* router3 = nullptr;  // [E][3H] bf16 high | middle | low (batch router on tcgen05)
  ChunkMap router_map{};        // its tensor map
  uint16_t* sh_gate = nullptr;  // [n_s*Is][H]
  uint16_t* sh_up = nullptr;    // [n_s*Is][H]
  uint16_t* sh_down = nullptr;  // [H][n_s*Is]
  uint8_t* eref = nullptr;      // [E][2I + H] row reference exponents (tcgen05 GEMMs)
  ChunkMap map_gu{}, map_dn{};  // tensor maps of the arena's tiles (tcgen05 GEMMs)
  ChunkMap mx_gate{}, mx_up{}, mx_down{};  // code tensor maps (MXFP8-activation variant)
  SharedMaps sh_maps{};         // shared experts as dense tcgen05 GEMMs (batches)
  bool sh_maps_ok = false;
  bool router_loaded = false;
  std::vector<uint8_t> shared_loaded;
  std::vector<uint8_t> expert_loaded;
  int n_experts_loaded = 0;
  // expert cache (df_moe_create_cached): every span in pinned host memory,
  // `cache_slots` of them in HBM (the arena), found through span_tab
  uint8_t* host_pool = nullptr;              // [E] spans, kernel layout (pinned, mapped)
  const uint8_t* host_pool_dev = nullptr;    // the same pages as the device sees them
  unsigned long long* span_tab = nullptr;    // device [E] span addresses (of cached experts)
  std::vector<int> slot_of, expert_of;       // expert -> slot (-1), slot -> expert (-1)
  std::vector<uint64_t> used;                // slot -> last use
};

struct Pending {
  int kind;
  cudaEvent_t a, b;
};

const char* kKindNames[K_NKINDS] = {"router", "topk", "group", "expert_gateup",
                                    "expert_down", "combine", "shared_gateup",
                                    "shared_down", "rmsnorm", "residual",
                                    "repack", "other", "mx8_quant", "gemm_gateup",
                                    "gemm_down", "cache_fill", "mx8_gateup", "mx8_down"};

}  // namespace

struct df_moe {
  df_moe_config cfg{};
  int device = 0;
  size_t span_bytes = 0;
  int R = 0;  // n_shared * shared_inter
  RouterSplit rsplit{};
  std::vector<LayerBufs> layers;
  // workspace
  float* router_part = nullptr;  // [nsplit][Tmax][E] (batches on tcgen05: [splits][T][E])
  size_t router_part_rows = 0;   // its rows (planes x tokens)
  bool router_tc = false;        // batches' router logits on tcgen05
  int router_tc_min_t = kDecodeMaxT + 1;  // from this many tokens
  float* logits = nullptr;       // [Tmax][E]
  int32_t* ids_ws = nullptr;     // [Tmax][k]
  float* w_ws = nullptr;         // [Tmax][k]
  Item* items = nullptr;         // [Tmax*k]
  int32_t* n_items = nullptr;    // [1]
  int32_t* sorted = nullptr;     // [Tmax*k]
  float* hbuf = nullptr;         // [Tmax*k][I]
  float* part = nullptr;         // [Tmax*k][H]
  float* hsh = nullptr;          // [Tmax][R]
  float* ysh = nullptr;          // [Tmax][H]
  uint16_t* xbuf[2] = {nullptr, nullptr};  // [Tmax][H] stack ping-pong
  uint16_t* xn = nullptr;        // [Tmax][H]
  uint32_t* err = nullptr;       // device error word
  // host-visible copy of the error word (pinned, mapped): the last kernel of
  // every forward writes the word there when it is nonzero
  uint32_t* err_mirror_h = nullptr;
  uint32_t* err_mirror_d = nullptr;  // the same word as the device sees it
  bool drop_next = false;            // test hook: the next forward's gate/up drops a stage
  unsigned int* counter = nullptr;  // router blocks done (zero between calls)
  // tcgen05 GEMMs for batches above the decode range
  bool gemm = false;
  uint16_t* g_xg = nullptr;      // [Tmax*k][H] f16: gate/up B rows in expert order
  uint16_t* g_hh = nullptr;      // [Tmax*k][2][I] f16: down B rows in expert order
  uint16_t* s_hh = nullptr;      // [Tmax][3][R] bf16: shared h rows (3 parts), batches
  float* g_bsc = nullptr;        // [Tmax*k] their power-of-two row scales
  ChunkMap bmap_gu{}, bmap_dn{};
  // block-scaled GEMMs on E4M3 activations: the MXFP8 variant
  // (DF_MOE_MXFP8_ACT, one plane) or exact planes (DF_MOE_PLANES); E4M3 rows
  // of x and h in expert order and their scales, stage-major
  bool mx8 = false;
  int px = 1, ph = 1;         // planes of x and of h
  int mx_xrows = 0, mx_hrows = 0;
  uint8_t* mx_xq = nullptr;   // [mx_xrows][H]
  uint8_t* mx_xsf = nullptr;  // [H/128][mx_xrows][16]
  uint8_t* mx_hq = nullptr;   // [mx_hrows][I]
  uint8_t* mx_hsf = nullptr;  // [I/128][mx_hrows][16]
  int32_t* mx_inv = nullptr;  // [Tmax*k] each assignment's position in expert order
  uint8_t* mx_xsfp = nullptr;  // [mx_xrows][H/32] row-major scales (scratch)
  uint8_t* mx_hsfp = nullptr;  // [mx_hrows][I/32]
  ChunkMap mx_xmap{}, mx_hmap{};
  // one token on exact planes: two phase kernels with the routed experts on
  // the block-scaled MMA (x's and h's planes in 16-row boxes; gate and up
  // sums over parts of K)
  bool phase_mx8 = false;
  ChunkMap mx_xmap16{}, mx_hmap16{};
  float* gu_part = nullptr;  // [kspl][k][2][I]
  bool phase = false;  // decode batches run the two phase kernels
  int sms = 0;
  cudaStream_t cap_stream = nullptr;  // CUDA-graph captures run on it
  // expert cache: HBM slots a layer (0: every expert resident in HBM)
  int cache_slots = 0;
  uint64_t cache_clock = 0;
  int64_t cache_hits = 0, cache_misses = 0, cache_bytes = 0;
  int32_t* ids_h = nullptr;  // pinned [Tmax * k]: a layer's selection on the host
  CacheCopy* fill_h = nullptr;        // pinned, mapped [Tmax * k]: a layer's fill plan
  const CacheCopy* fill_d = nullptr;  // the same as the device sees it
  std::vector<void*> host_allocs;
  // host-API device buffers
  uint16_t* hx = nullptr;
  uint16_t* hres = nullptr;
  uint16_t* hout = nullptr;
  float* hout32 = nullptr;
  int32_t* hids = nullptr;
  float* hw = nullptr;
  // host-API staging in pinned, device-mapped host memory (made on first
  // use): x, residual, out, out_f32, ids, weights, at io_off[] (host view
  // io_h, device view io_d)
  uint8_t* io_h = nullptr;
  uint8_t* io_d = nullptr;
  size_t io_off[6] = {0, 0, 0, 0, 0, 0};
  // staging for host-sourced spans
  uint8_t* staging = nullptr;
  size_t staging_spans = 0;
  std::vector<void*> allocs;
  std::string last_error;
  // timing
  bool timing = false;
  std::vector<Pending> pending;
  std::vector<cudaEvent_t> event_pool;
  double kind_ms[K_NKINDS] = {};
  int64_t kind_n[K_NKINDS] = {};
  int launches = 0;
};

namespace {

int fail(df_moe* h, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (h) h->last_error = buf;
  else g_thread_err = buf;
  return code;
}

#define CUDA_OR_FAIL(h, call)                                                  \
  do {                                                                         \
    cudaError_t e_ = (call);                                                   \
    if (e_ != cudaSuccess)                                                     \
      return fail((h), DF_MOE_ECUDA, "%s failed: %s", #call,                   \
                  cudaGetErrorString(e_));                                     \
  } while (0)

template <typename T>
int dalloc(df_moe* h, T** p, size_t n) {
  *p = nullptr;
  if (n == 0) n = 1;
  cudaError_t e = cudaMalloc((void**)p, n * sizeof(T));
  if (e != cudaSuccess) {
    *p = nullptr;
    cudaGetLastError();
    return fail(h, DF_MOE_ENOMEM, "cudaMalloc of %zu bytes failed: %s",
                n * sizeof(T), cudaGetErrorString(e));
  }
  h->allocs.push_back(*p);
  return DF_MOE_OK;
}

// Canonical spans -> the handle's device layout (inverse: back): the
// fragment layout, or for the MXFP8-activation variant the canonical codes
// with stage-major scales.
cudaError_t span_layout_copy(const df_moe* h, const uint8_t* src, uint8_t* dst, int n,
                             int inverse, cudaStream_t s) {
  const df_moe_config& c = h->cfg;
  return h->mx8 ? launch_mx8_layout(src, dst, n, c.hidden, c.inter, h->span_bytes, inverse, s)
                : launch_repack_span(src, dst, n, c.hidden, c.inter, inverse, s);
}

cudaEvent_t get_event(df_moe* h) {
  if (!h->event_pool.empty()) {
    cudaEvent_t e = h->event_pool.back();
    h->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Run one kernel launch, bracketed by events when timing is on.
template <typename F>
int run(df_moe* h, int kind, cudaStream_t s, F&& launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (h->timing) {
    a = get_event(h);
    b = get_event(h);
    cudaEventRecord(a, s);
  }
  cudaError_t e = launch();
  if (e != cudaSuccess)
    return fail(h, DF_MOE_ECUDA, "%s launch failed: %s", kKindNames[kind],
                cudaGetErrorString(e));
  if (h->timing) {
    cudaEventRecord(b, s);
    h->pending.push_back(Pending{kind, a, b});
  }
  h->launches += 1;
  return DF_MOE_OK;
}

#define RUN(h, kind, s, expr)                                   \
  do {                                                          \
    int rc_ = run((h), (kind), (s), [&]() { return (expr); });  \
    if (rc_) return rc_;                                        \
  } while (0)

int check_layer_ready(df_moe* h, int l) {
  const LayerBufs& L = h->layers[l];
  if (!L.router_loaded)
    return fail(h, DF_MOE_ESTATE, "layer %d: router not loaded", l);
  for (int s = 0; s < h->cfg.n_shared; ++s)
    if (!L.shared_loaded[s])
      return fail(h, DF_MOE_ESTATE, "layer %d: shared expert %d not loaded", l, s);
  if (L.n_experts_loaded != h->cfg.n_experts)
    return fail(h, DF_MOE_ESTATE, "layer %d: %d of %d experts loaded", l,
                L.n_experts_loaded, h->cfg.n_experts);
  return DF_MOE_OK;
}

// Router + top-k (+ grouping) of one layer. ids/w: [T][k] device.
// planes_only (one token): only the partial-logit planes; the gate/up phase
// kernel selects.
int route(df_moe* h, int l, const uint16_t* x, int T, int32_t* ids, float* w,
          cudaStream_t s, float* logits_out, int tg, bool planes_only = false) {
  const df_moe_config& c = h->cfg;
  const LayerBufs& L = h->layers[l];
  const bool direct = (T == 1 && tg == 1);
  if (direct && planes_only && !logits_out) {
    RUN(h, K_ROUTER, s, launch_router(L.router, c.n_experts, c.hidden, x, T,
                                      h->router_part, h->rsplit, s));
    return DF_MOE_OK;
  }
  if (direct && !logits_out) {
    // one token: the router's last block selects the experts and writes the
    // work items (no separate top-k launch)
    const RouterFuse fz{h->counter, c.top_k, ids, w, h->items, h->n_items, h->sorted};
    RUN(h, K_ROUTER, s, launch_router(L.router, c.n_experts, c.hidden, x, T,
                                      h->router_part, h->rsplit, s, &fz));
    return DF_MOE_OK;
  }
  int nsplit = h->rsplit.nsplit;
  if (h->router_tc && T >= h->router_tc_min_t) {
    // a batch: the logits as one GEMM on the tensor cores (the weights read
    // once for all tokens)
    int used = -1;
    RUN(h, K_ROUTER, s,
        (used = launch_router_tc(L.router_map, x, T, c.n_experts, c.hidden, h->router_part,
                                 h->router_part_rows, h->sms, h->err, s)) < 0
            ? cudaErrorLaunchFailure
            : cudaSuccess);
    nsplit = used;
  } else {
    RUN(h, K_ROUTER, s, launch_router(L.router, c.n_experts, c.hidden, x, T,
                                      h->router_part, h->rsplit, s));
  }
  RUN(h, K_TOPK, s, launch_topk(h->router_part, nsplit, T,
                                c.n_experts, c.top_k, logits_out, ids, w,
                                direct ? h->items : nullptr, h->n_items,
                                h->sorted, s));
  if (!direct)
    RUN(h, K_GROUP, s, launch_group(ids, T, c.top_k, c.n_experts, nullptr,
                                    nullptr, nullptr, nullptr, h->items,
                                    h->n_items, h->sorted, tg, h->err, s, h->mx_inv));
  return DF_MOE_OK;
}

// Routed experts of a batch grouped one item per expert (or per token at
// T = 1). Above the decode range the grouped tcgen05 GEMMs run them, unless
// the handle asks for the register-fragment kernels.
bool use_gemm(const df_moe* h, int T, int tg) {
  return h->gemm && T > kDecodeMaxT && tg == kOneItemPerExpert;
}

int expert_gateup(df_moe* h, int l, const uint16_t* x, int T, int max_items, int tg,
                  float* hbuf, cudaStream_t s, int max_ctas = 0) {
  const df_moe_config& c = h->cfg;
  const uint8_t* arena = h->layers[l].arena;
  if (h->mx8) {
    // block-scaled GEMM on E4M3 x (MXFP8, or x's planes): h rounded to MXFP8
    // for the down GEMM in its epilogue (and, when hbuf is given, h before
    // that), or, with planes, h into hbuf
    const LayerBufs& L = h->layers[l];
    // (one token selected directly: item q is assignment q, no grouping)
    RUN(h, K_MX8_QUANT, s, launch_mx8_xrows(x, c.hidden, c.top_k, T,
                                            tg == 1 ? nullptr : h->mx_inv, h->px, h->mx_xq,
                                            h->mx_xrows, h->mx_xsfp, h->err, s));
    RUN(h, K_MX8_QUANT, s, launch_mx8_scale_lines(h->mx_xsfp, c.hidden, T * c.top_k * h->px,
                                                  h->mx_xrows, h->px, h->mx_xsf, s));
    RUN(h, K_MX8_GU, s, launch_mx8_gateup(L.mx_gate, L.mx_up, h->mx_xmap, arena, h->span_bytes,
                                          c.hidden, c.inter, h->mx_xsf, h->mx_xrows, h->items,
                                          h->n_items, max_items, h->sorted, c.n_experts,
                                          T * c.top_k, hbuf, h->mx_hq, h->mx_hsf, h->mx_hrows,
                                          h->px, h->err, s));
    return DF_MOE_OK;
  }
  if (use_gemm(h, T, tg)) {
    RUN(h, K_OTHER, s, launch_prep_x(x, T * c.top_k, c.hidden, c.top_k, h->sorted, h->g_xg,
                                     h->g_bsc, h->err, s));
    RUN(h, K_GEMM_GU, s, launch_gemm_gateup(h->layers[l].map_gu, h->bmap_gu, arena,
                                            h->span_bytes, h->layers[l].eref, c.hidden, c.inter,
                                            c.top_k, h->g_bsc, h->items, h->n_items, max_items,
                                            h->sorted, hbuf, c.n_experts, T * c.top_k, h->err,
                                            s));
  } else {
    RUN(h, K_GATEUP, s, launch_gateup(arena, h->span_bytes, c.hidden, c.inter, c.top_k, x,
                                      h->items, h->n_items, max_items, h->sorted, hbuf, tg,
                                      c.n_experts, T * c.top_k, h->err, s, max_ctas));
  }
  return DF_MOE_OK;
}

int expert_down(df_moe* h, int l, const float* hbuf, int T, int max_items, int tg,
                cudaStream_t s, int max_ctas = 0, bool after_gateup = false) {
  const df_moe_config& c = h->cfg;
  const uint8_t* arena = h->layers[l].arena;
  if (h->mx8) {
    // block-scaled GEMM on E4M3 h: h (when given) rounded to MXFP8 or split
    // into its planes first; else (MXFP8) the gate/up GEMM's rounded h
    if (hbuf) {
      RUN(h, K_MX8_QUANT, s, launch_mx8_rows(hbuf, c.inter, h->ph, h->items, h->n_items,
                                             max_items, h->sorted, T * c.top_k, c.n_experts,
                                             h->mx_hq, h->mx_hrows, h->mx_hsfp, h->err, s));
      RUN(h, K_MX8_QUANT, s, launch_mx8_scale_lines(h->mx_hsfp, c.inter, T * c.top_k * h->ph,
                                                    h->mx_hrows, h->ph, h->mx_hsf, s));
    }
    RUN(h, K_MX8_DN, s, launch_mx8_down(h->layers[l].mx_down, h->mx_hmap, arena, h->span_bytes,
                                        c.hidden, c.inter, h->mx_hsf, h->mx_hrows, h->items,
                                        h->n_items, max_items, h->sorted, c.n_experts,
                                        T * c.top_k, h->part, h->ph, h->err, s));
    return DF_MOE_OK;
  }
  if (use_gemm(h, T, tg)) {
    RUN(h, K_OTHER, s, launch_split_h(hbuf, T * c.top_k, c.inter, h->sorted, h->g_hh, h->g_bsc,
                                      h->err, s));
    RUN(h, K_GEMM_DN, s, launch_gemm_down(h->layers[l].map_dn, h->bmap_dn, arena,
                                          h->span_bytes, h->layers[l].eref, c.hidden, c.inter,
                                          c.top_k, h->g_bsc, h->items, h->n_items, max_items,
                                          h->sorted, h->part, c.n_experts, T * c.top_k, h->err,
                                          s));
  } else {
    RUN(h, K_DOWN, s, launch_down(arena, h->span_bytes, c.hidden, c.inter, h->items,
                                  h->n_items, max_items, h->sorted, hbuf, h->part, tg,
                                  c.n_experts, T * c.top_k, h->err, s, max_ctas, after_gateup));
  }
  return DF_MOE_OK;
}

int shared_part(df_moe* h, int l, const uint16_t* x, int T, float* ysh,
                cudaStream_t s, int max_ctas = 0) {
  const df_moe_config& c = h->cfg;
  const LayerBufs& L = h->layers[l];
  // the dense GEMMs from 4 tokens on block-scaled handles (where the shared
  // experts do not run beside the routed ones): at 4-8 tokens the streaming
  // GEMV spends more time on its fp32 FMAs than on the weights
  const bool dense = T > kDecodeMaxT || (h->mx8 && T >= 4);
  if (dense && L.sh_maps_ok && ((uintptr_t)x & 15) == 0) {
    // a batch: two dense GEMMs on the tensor cores
    RUN(h, K_SHARED_GU, s, launch_shared_gemm_gateup(L.sh_maps, x, T, c.hidden, h->R, h->s_hh,
                                                     h->err, s));
    RUN(h, K_SHARED_DN, s, launch_shared_gemm_down(L.sh_maps, T, c.hidden, h->R, ysh, h->err, s));
    return DF_MOE_OK;
  }
  RUN(h, K_SHARED_GU, s, launch_shared_gateup(L.sh_gate, L.sh_up, h->R,
                                              c.hidden, x, T, h->hsh, h->err, s, max_ctas));
  RUN(h, K_SHARED_DN, s, launch_shared_down(L.sh_down, c.hidden, h->R, h->hsh,
                                            T, ysh, h->err, s, max_ctas));
  return DF_MOE_OK;
}

// Expert cache: brings layer l's selection (ids, on the device) into HBM
// slots. The selection comes to the host (one synchronisation); every
// selected expert not cached gets an empty slot, else the least recently
// used slot not needed now, and one fill kernel copies those experts from
// the pinned host pool into their slots and points their span-table entries
// at them (a cached expert's entry already points at its slot). Consecutive
// tokens that share experts find them cached: the last token's experts are
// the most recently used ones. This is the previous-token reuse of the Deltafin README
// ("Techniques", "I/O and streaming") and the expert LRU cache of the
// kimi-k3-in-c blog, moved from SSD -> RAM to Grace memory -> HBM. The
// blog's first trap counts a prefetched expert as a hit although its bytes
// moved, so the statistics count the bytes copied in.
int cache_plan(df_moe* h, int l, int T, const int32_t* ids, cudaStream_t s) {
  const df_moe_config& c = h->cfg;
  LayerBufs& L = h->layers[l];
  const int n = T * c.top_k;
  CUDA_OR_FAIL(h, cudaMemcpyAsync(h->ids_h, ids, n * sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  CUDA_OR_FAIL(h, cudaStreamSynchronize(s));
  const uint64_t now = ++h->cache_clock;
  std::vector<int> miss;
  int nfill = 0;
  for (int i = 0; i < n; ++i) {
    const int e = h->ids_h[i];
    if (e < 0 || e >= c.n_experts)
      return fail(h, DF_MOE_EDEVICE, "layer %d: the device selected expert %d, out of range", l,
                  e);
    const int sl = L.slot_of[e];
    if (sl >= 0) {
      if (L.used[sl] != now) {
        L.used[sl] = now;
        ++h->cache_hits;
      }
    } else if (std::find(miss.begin(), miss.end(), e) == miss.end()) {
      miss.push_back(e);
    }
  }
  for (const int e : miss) {
    int v = -1;
    for (int sl = 0; sl < h->cache_slots; ++sl) {
      if (L.used[sl] == now) continue;
      if (L.expert_of[sl] < 0) {
        v = sl;
        break;
      }
      if (v < 0 || L.used[sl] < L.used[v]) v = sl;
    }
    if (v < 0) return fail(h, DF_MOE_ESTATE, "layer %d: no free cache slot", l);
    if (L.expert_of[v] >= 0) L.slot_of[L.expert_of[v]] = -1;
    L.expert_of[v] = e;
    L.slot_of[e] = v;
    L.used[v] = now;
    // the plan buffer is free: the synchronisation above came after the
    // previous fill kernel
    h->fill_h[nfill++] = CacheCopy{L.host_pool_dev + (size_t)e * h->span_bytes,
                                   L.arena + (size_t)v * h->span_bytes, e};
  }
  if (nfill) {
    const int rc = run(h, K_CACHE_FILL, s, [&]() {
      return launch_cache_fill(h->fill_d, nfill, h->span_bytes, L.span_tab, s);
    });
    if (rc) {
      // nothing was copied: this call's experts leave their slots again
      for (int i = 0; i < nfill; ++i) {
        const int e = (int)h->fill_h[i].e;
        if (L.slot_of[e] >= 0) L.expert_of[L.slot_of[e]] = -1;
        L.slot_of[e] = -1;
      }
      return rc;
    }
    // counted once the copies are on their way: the bytes actually moved
    h->cache_misses += nfill;
    h->cache_bytes += (int64_t)nfill * (int64_t)h->span_bytes;
  }
  return DF_MOE_OK;
}

// ids_host / w_host (or null): where the combine also copies this layer's
// selection (host memory the device writes directly).
int layer_forward(df_moe* h, int l, const uint16_t* x, int T,
                  const uint16_t* residual, uint16_t* out_bf16, float* out_f32,
                  int32_t* ids, float* w, cudaStream_t s, int32_t* ids_host = nullptr,
                  float* w_host = nullptr) {
  const df_moe_config& c = h->cfg;
  const LayerBufs& L = h->layers[l];
  const int tg = T == 1 ? 1 : kOneItemPerExpert;
  const int max_items = (T == 1 && tg == 1) ? c.top_k : std::min(T * c.top_k, c.n_experts);
  const int R = c.n_shared > 0 ? h->R : 0;
  const bool phase = T <= kDecodeMaxT && h->phase;
  const bool cached = h->cache_slots > 0;
  // one token on exact planes: the routed experts on the block-scaled MMA
  const bool phase_mx8 = T == 1 && h->phase_mx8 && !cached;
  int sh_gu = 0, sh_dn = 0;
  if (phase && R > 0) {
    // CTAs for the shared experts in each phase: the split that ends both
    // sides together at the per-SM streaming rates measured on GB300 at K3
    // shape (GB/s an SM): routed MXFP4 gate/up ~32, down ~27; shared bf16
    // gate/up ~60 and down ~68 at one token, falling as the fp32 FMAs per
    // byte grow with the tokens a pass (~9 and ~11 at 8). At T = 1 the routed
    // CTAs first spend ~6 us selecting the experts.
    const double n_rt = std::min(T * c.top_k, c.n_experts);
    const double gu_rt = n_rt * 2.0 * c.inter * c.hidden * 17 / 32 / 32e3;  // us x SMs
    const double dn_rt = n_rt * (double)c.hidden * c.inter * 17 / 32 / 27e3;
    const int TT = T == 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;  // shared tokens a pass
    const double gu_sh = 2.0 * R * c.hidden * 2 / (60e3 / (1.0 + 0.81 * (TT - 1)));
    const double dn_sh = (double)R * c.hidden * 2 / (68e3 / (1.0 + 0.74 * (TT - 1)));
    auto split = [&](double sh, double rt, double rt_delay) {
      int best = 1;
      double best_t = 1e30;
      for (int n = 1; n < h->sms; ++n) {
        const double t = std::max(sh / n, rt / (h->sms - n) + rt_delay);
        if (t < best_t) { best_t = t; best = n; }
      }
      return best;
    };
    sh_gu = split(gu_sh, gu_rt, T == 1 ? 6.0 : 0.0);
    sh_dn = split(dn_sh, dn_rt, 0.0);
  }
  if (phase_mx8 && R > 0) {
    // the same balance with the block-scaled routed pipelines (~40 GB/s an
    // SM for gate/up and down) against the shared GEMV at one token
    const double n_rt = std::min(c.top_k, c.n_experts);
    const double gu_rt = n_rt * 2.0 * c.inter * c.hidden * 17 / 32 / 40e3;
    const double dn_rt = n_rt * (double)c.hidden * c.inter * 17 / 32 / 40e3;
    const double gu_sh = 2.0 * R * c.hidden * 2 / 60e3, dn_sh = (double)R * c.hidden * 2 / 68e3;
    auto split = [&](double sh, double rt, double rt_delay) {
      int best = 1;
      double best_t = 1e30;
      for (int n = 1; n < h->sms; ++n) {
        const double t = std::max(sh / n, rt / (h->sms - n) + rt_delay);
        if (t < best_t) { best_t = t; best = n; }
      }
      return best;
    };
    sh_gu = split(gu_sh, gu_rt, 6.0);
    sh_dn = split(dn_sh, dn_rt, 0.0);
  }
  if (phase_mx8) {
    // x's planes at the rows of every rank (item j reads rows 4j ..)
    RUN(h, K_MX8_QUANT, s, launch_mx8_xrows(x, c.hidden, c.top_k, 1, nullptr, h->px, h->mx_xq,
                                            h->mx_xrows, h->mx_xsfp, h->err, s));
    RUN(h, K_MX8_QUANT, s, launch_mx8_scale_lines(h->mx_xsfp, c.hidden, c.top_k * h->px,
                                                  h->mx_xrows, h->px, h->mx_xsf, s));
  }
  int rc = route(h, l, x, T, ids, w, s, nullptr, tg,
                 /*planes_only=*/(phase || phase_mx8) && !cached);
  if (rc) return rc;
  if (cached) {
    rc = cache_plan(h, l, T, ids, s);
    if (rc) return rc;
  }
  if (phase_mx8) {
    // gate/up phase (selection, routed gate/up sums, shared h), h = SwiGLU
    // of the sums as planes, down phase (routed and shared)
    RUN(h, K_MX8_GU, s, launch_mx8_phase_gateup(L.mx_gate, L.mx_up, h->mx_xmap16, L.arena,
                                                h->span_bytes, c.hidden, c.inter, h->mx_xsf,
                                                h->mx_xrows, h->items, h->n_items, h->sorted,
                                                c.n_experts, c.top_k, h->router_part,
                                                h->rsplit.nsplit, ids, w, h->gu_part, L.sh_gate,
                                                L.sh_up, R, x, h->hsh, h->err, sh_gu, s));
    RUN(h, K_MX8_QUANT, s, launch_mx8_rows(nullptr, c.inter, h->ph, h->items, h->n_items,
                                           c.top_k, h->sorted, c.top_k, c.n_experts, h->mx_hq,
                                           h->mx_hrows, h->mx_hsfp, h->err, s, h->gu_part,
                                           mx8_phase_kspl(c.hidden)));
    RUN(h, K_MX8_QUANT, s, launch_mx8_scale_lines(h->mx_hsfp, c.inter, c.top_k * h->ph,
                                                  h->mx_hrows, h->ph, h->mx_hsf, s));
    RUN(h, K_MX8_DN, s, launch_mx8_phase_down(L.mx_down, h->mx_hmap16, L.arena, h->span_bytes,
                                              c.hidden, c.inter, h->mx_hsf, h->mx_hrows,
                                              h->items, h->n_items, h->sorted, c.n_experts,
                                              c.top_k, h->part, L.sh_down, R, h->hsh, h->ysh,
                                              h->err, sh_dn, s));
  } else if (phase) {
    // decode batches: routed and shared experts together on every SM, each
    // kernel a programmatic dependent of the one before
    RUN(h, K_GATEUP, s, launch_phase_gateup(L.sh_gate, L.sh_up, R, L.arena, h->span_bytes,
                                            c.hidden, c.inter, c.top_k, x, T, h->items,
                                            h->n_items, h->sorted,
                                            cached ? nullptr : h->router_part,
                                            h->rsplit.nsplit, c.n_experts, ids, w, h->hsh,
                                            h->hbuf, h->err, sh_gu,
                                            cached ? (const uint8_t* const*)L.span_tab : nullptr,
                                            h->drop_next, s));
    h->drop_next = false;
    RUN(h, K_DOWN, s, launch_phase_down(L.arena, h->span_bytes, c.hidden, c.inter, c.n_experts,
                                        c.top_k, h->items, h->n_items, h->sorted, h->hbuf,
                                        h->part, L.sh_down, R, h->hsh, T, h->ysh, h->err, sh_dn,
                                        cached ? (const uint8_t* const*)L.span_tab : nullptr,
                                        s));
  } else {
    // batches: the shared experts, then the routed ones
    if (c.n_shared > 0) {
      rc = shared_part(h, l, x, T, h->ysh, s);
      if (rc) return rc;
    }
    // (the MXFP8 variant hands h from GEMM to GEMM already rounded)
    const bool rounded_h = h->mx8 && h->ph == 1;
    rc = expert_gateup(h, l, x, T, max_items, tg, rounded_h ? nullptr : h->hbuf, s);
    if (rc) return rc;
    rc = expert_down(h, l, rounded_h ? nullptr : h->hbuf, T, max_items, tg, s, 0,
                     /*after_gateup=*/true);
    if (rc) return rc;
  }
  RUN(h, K_COMBINE, s, launch_combine(h->part, w, T, c.top_k, c.hidden,
                                      c.n_shared > 0 ? h->ysh : nullptr,
                                      residual, out_f32, out_bf16, h->err, h->err_mirror_d, s,
                                      ids, ids_host, w_host));
  return DF_MOE_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }
bool all_aligned16(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!aligned16(p)) return false;
  return true;
}

}  // namespace

extern "C" {

const char* df_moe_last_error(const df_moe* h) {
  return h ? h->last_error.c_str() : g_thread_err.c_str();
}

size_t df_moe_span_bytes_for(int32_t H, int32_t I) {
  if (H <= 0 || I <= 0) return 0;
  return span_layout(H, I).bytes;
}

size_t df_moe_expert_span_bytes(const df_moe* h) { return h ? h->span_bytes : 0; }

void df_moe_destroy(df_moe* h) {
  if (!h) return;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(h->device);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  for (auto& p : h->pending) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  for (auto e : h->event_pool) cudaEventDestroy(e);
  for (void* p : h->allocs) cudaFree(p);
  for (void* p : h->host_allocs) cudaFreeHost(p);
  cudaSetDevice(prev);
  delete h;
}

static int create_impl(const df_moe_config* cfg, int cuda_device, int slots, df_moe** out) {
  if (!cfg || !out) return fail(nullptr, DF_MOE_EINVAL, "null argument");
  *out = nullptr;
  const df_moe_config c = *cfg;
  if (c.hidden <= 0 || c.hidden % 64 || c.hidden > 8192)
    return fail(nullptr, DF_MOE_EINVAL, "hidden must be a multiple of 64 in [64, 8192]");
  if (c.inter <= 0 || c.inter % 64 || c.inter > 8192)
    return fail(nullptr, DF_MOE_EINVAL, "inter must be a multiple of 64 in [64, 8192]");
  if (c.n_experts < 1 || c.n_experts > 1024)
    return fail(nullptr, DF_MOE_EINVAL, "n_experts must be in [1, 1024]");
  if (c.top_k < 1 || c.top_k > c.n_experts || c.top_k > 32)
    return fail(nullptr, DF_MOE_EINVAL, "top_k must be in [1, min(n_experts, 32)]");
  if (c.n_shared < 0 || c.n_shared > 8)
    return fail(nullptr, DF_MOE_EINVAL, "n_shared must be in [0, 8]");
  if (c.n_shared > 0 && (c.shared_inter <= 0 || c.shared_inter % 64 ||
                         c.n_shared * c.shared_inter > 6144))
    return fail(nullptr, DF_MOE_EINVAL,
                "shared_inter must be a multiple of 64 with n_shared*shared_inter <= 6144");
  if (c.n_layers < 1 || c.n_layers > 64)
    return fail(nullptr, DF_MOE_EINVAL, "n_layers must be in [1, 64]");
  if (c.max_tokens < 1 || c.max_tokens > 4096 || c.max_tokens * c.top_k > 65535)
    return fail(nullptr, DF_MOE_EINVAL,
                "max_tokens must be in [1, 4096] with max_tokens*top_k <= 65535");
  if (c.n_layers > 1 && !(c.flags & DF_MOE_STACK_RMSNORM_RESIDUAL))
    return fail(nullptr, DF_MOE_EINVAL, "n_layers > 1 needs DF_MOE_STACK_RMSNORM_RESIDUAL");
  if ((c.flags & ~(DF_MOE_STACK_RMSNORM_RESIDUAL | DF_MOE_PREFILL_MMA_SYNC |
                   DF_MOE_MXFP8_ACT | DF_MOE_PLANES)) != 0)
    return fail(nullptr, DF_MOE_EINVAL, "unknown flags");
  if (c.flags & (DF_MOE_MXFP8_ACT | DF_MOE_PLANES)) {
    const char* f = (c.flags & DF_MOE_MXFP8_ACT) ? "DF_MOE_MXFP8_ACT" : "DF_MOE_PLANES";
    if ((c.flags & DF_MOE_MXFP8_ACT) && (c.flags & DF_MOE_PLANES))
      return fail(nullptr, DF_MOE_EINVAL, "DF_MOE_MXFP8_ACT and DF_MOE_PLANES exclude each other");
    if (slots) return fail(nullptr, DF_MOE_EINVAL, "%s does not combine with an expert cache", f);
    if (c.flags & DF_MOE_PREFILL_MMA_SYNC)
      return fail(nullptr, DF_MOE_EINVAL, "%s does not combine with DF_MOE_PREFILL_MMA_SYNC", f);
    if (!mx8_supported(c.hidden, c.inter))
      return fail(nullptr, DF_MOE_EINVAL,
                  "%s needs hidden a multiple of 256 and inter a multiple of 128", f);
  }
  if ((c.flags & DF_MOE_STACK_RMSNORM_RESIDUAL) && !(c.rms_eps >= 0.0f))
    return fail(nullptr, DF_MOE_EINVAL, "rms_eps must be >= 0");
  if (slots) {
    if (c.max_tokens > kDecodeMaxT)
      return fail(nullptr, DF_MOE_EINVAL,
                  "an expert cache serves decode batches (max_tokens <= %d)", kDecodeMaxT);
    if (slots < std::min(c.max_tokens * c.top_k, c.n_experts) || slots > c.n_experts)
      return fail(nullptr, DF_MOE_EINVAL,
                  "cache_slots must be in [min(max_tokens*top_k, n_experts), n_experts]");
  }
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || cuda_device < 0 ||
      cuda_device >= ndev) {
    cudaGetLastError();
    return fail(nullptr, DF_MOE_EINVAL, "no CUDA device %d", cuda_device);
  }
  int prev = 0;
  cudaGetDevice(&prev);
  if (cudaSetDevice(cuda_device) != cudaSuccess)
    return fail(nullptr, DF_MOE_ECUDA, "cudaSetDevice(%d) failed", cuda_device);

  df_moe* h = new df_moe;
  h->cfg = c;
  h->device = cuda_device;
  h->cache_slots = slots;
  h->span_bytes = span_layout(c.hidden, c.inter).bytes;
  h->R = c.n_shared * c.shared_inter;
  h->rsplit = router_split(c.n_experts, c.hidden);
  cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, cuda_device);
  const size_t H = c.hidden, E = c.n_experts, k = c.top_k, I = c.inter;
  const size_t Tm = c.max_tokens, R = h->R;
  int rc = DF_MOE_OK;
  h->layers.resize(c.n_layers);
  for (int l = 0; l < c.n_layers && !rc; ++l) {
    LayerBufs& L = h->layers[l];
    L.shared_loaded.assign(c.n_shared, 0);
    L.expert_loaded.assign(c.n_experts, 0);
    rc = dalloc(h, &L.arena, (slots ? (size_t)slots : E) * h->span_bytes);
    if (!rc && slots) {
      L.slot_of.assign(E, -1);
      L.expert_of.assign(slots, -1);
      L.used.assign(slots, 0);
      rc = dalloc(h, &L.span_tab, E);
      if (!rc && cudaMemset(L.span_tab, 0, E * sizeof(unsigned long long)) != cudaSuccess)
        rc = fail(h, DF_MOE_ECUDA, "cudaMemset failed");
      void* hp = nullptr;
      if (!rc && cudaHostAlloc(&hp, E * h->span_bytes,
                               cudaHostAllocPortable | cudaHostAllocMapped) != cudaSuccess)
        rc = fail(h, DF_MOE_ENOMEM, "pinned host pool of %zu bytes failed", E * h->span_bytes);
      if (!rc) {
        h->host_allocs.push_back(hp);
        L.host_pool = static_cast<uint8_t*>(hp);
        void* dp = nullptr;
        if (cudaHostGetDevicePointer(&dp, hp, 0) != cudaSuccess)
          rc = fail(h, DF_MOE_ECUDA, "host pool not mapped into the device");
        L.host_pool_dev = static_cast<const uint8_t*>(dp);
      }
    }
    if (!rc) rc = dalloc(h, &L.router, E * H);
    if (!rc && R) rc = dalloc(h, &L.sh_gate, R * H);
    if (!rc && R) rc = dalloc(h, &L.sh_up, R * H);
    if (!rc && R) rc = dalloc(h, &L.sh_down, H * R);
  }
  // tcgen05 GEMMs: batches above the decode range, unless asked otherwise
  h->mx8 = (c.flags & (DF_MOE_MXFP8_ACT | DF_MOE_PLANES)) != 0;
  if (c.flags & DF_MOE_PLANES) {
    h->px = kPlanesX;
    h->ph = kPlanesH;
  }
  h->gemm = !slots && !h->mx8 && Tm > (size_t)kDecodeMaxT &&
            !(c.flags & DF_MOE_PREFILL_MMA_SYNC) && gemm_supported(c.hidden, c.inter);
  if (h->mx8) {
    h->mx_xrows = mx8_rows_cap((int)(Tm * k), h->px);
    h->mx_hrows = mx8_rows_cap((int)(Tm * k), h->ph);
    const size_t xrows = (size_t)h->mx_xrows, hrows = (size_t)h->mx_hrows;
    for (int l = 0; l < c.n_layers && !rc; ++l) {
      LayerBufs& L = h->layers[l];
      if (!make_mx8_maps(L.arena, h->span_bytes, c.hidden, c.inter, c.n_experts, &L.mx_gate,
                         &L.mx_up, &L.mx_down))
        rc = fail(h, DF_MOE_ECUDA, "tensor map encoding failed");
    }
    if (!rc) rc = dalloc(h, &h->mx_xq, xrows * H);
    if (!rc) rc = dalloc(h, &h->mx_xsf, H / 128 * xrows * 16);
    if (!rc) rc = dalloc(h, &h->mx_hq, hrows * I);
    if (!rc) rc = dalloc(h, &h->mx_hsf, I / 128 * hrows * 16);
    if (!rc) rc = dalloc(h, &h->mx_inv, Tm * k);
    if (!rc) rc = dalloc(h, &h->mx_xsfp, xrows * (H / 32));
    if (!rc) rc = dalloc(h, &h->mx_hsfp, hrows * (I / 32));
    if (!rc && (!make_mx8_row_map(h->mx_xq, h->mx_xrows, c.hidden, h->px, &h->mx_xmap,
                                  mx8_box_rows(h->px)) ||
                !make_mx8_row_map(h->mx_hq, h->mx_hrows, c.inter, h->ph, &h->mx_hmap,
                                  mx8_box_rows(h->ph))))
      rc = fail(h, DF_MOE_ECUDA, "tensor map encoding failed");
    h->phase_mx8 = h->px > 1 && !slots && k <= 32 && E <= 1024 &&
                   mx8_phase_supported(c.hidden, c.inter, (int)R);
    if (!rc && h->phase_mx8) {
      rc = dalloc(h, &h->gu_part, (size_t)mx8_phase_kspl(c.hidden) * k * 2 * I);
      if (!rc &&
          (!make_mx8_row_map(h->mx_xq, h->mx_xrows, c.hidden, h->px, &h->mx_xmap16, 16) ||
           !make_mx8_row_map(h->mx_hq, h->mx_hrows, c.inter, h->ph, &h->mx_hmap16, 16)))
        rc = fail(h, DF_MOE_ECUDA, "tensor map encoding failed");
    }
  }
  if (h->gemm) {
    for (int l = 0; l < c.n_layers && !rc; ++l) {
      LayerBufs& L = h->layers[l];
      rc = dalloc(h, &L.eref, gemm_eref_bytes(c.n_experts, c.hidden, c.inter));
      if (!rc && !make_chunk_maps(L.arena, h->span_bytes, c.hidden, c.inter, c.n_experts,
                                  &L.map_gu, &L.map_dn))
        rc = fail(h, DF_MOE_ECUDA, "tensor map encoding failed");
    }
    if (!rc) rc = dalloc(h, &h->g_xg, Tm * k * H);
    if (!rc) rc = dalloc(h, &h->g_hh, Tm * k * 2 * I);
    if (!rc) rc = dalloc(h, &h->g_bsc, Tm * k);
    if (!rc && !make_b_maps(h->g_xg, h->g_hh, (int)(Tm * k), c.hidden, c.inter, &h->bmap_gu,
                            &h->bmap_dn))
      rc = fail(h, DF_MOE_ECUDA, "tensor map encoding failed");
  }
  // the shared experts of batches as dense tcgen05 GEMMs (the routed
  // experts' path aside: exact GEMMs, the MXFP8 variant, or none)
  if (!rc && (h->gemm || h->mx8) && (Tm > (size_t)kDecodeMaxT || (h->mx8 && Tm >= 4)) && R &&
      dense_supported(c.hidden, (int)R)) {
    rc = dalloc(h, &h->s_hh, Tm * 3 * R);
    for (int l = 0; l < c.n_layers && !rc; ++l) {
      LayerBufs& L = h->layers[l];
      L.sh_maps_ok = make_shared_maps(L.sh_gate, L.sh_up, L.sh_down, c.hidden, (int)R, h->s_hh,
                                      (int)(3 * Tm), &L.sh_maps);
    }
  }
  // batches' router on tcgen05: the weights' bf16 parts and their map
  // (block-scaled handles run 4-8 token batches through the batch path too,
  // where the tensor-core router beats the GEMV's fp32 FMAs on x in shared
  // memory)
  h->router_tc_min_t = h->mx8 ? 4 : kDecodeMaxT + 1;
  h->router_tc = Tm >= (size_t)h->router_tc_min_t;
  for (int l = 0; l < c.n_layers && !rc && h->router_tc; ++l) {
    LayerBufs& L = h->layers[l];
    rc = dalloc(h, &L.router3, E * 3 * H);
    if (!rc && !make_router_map(L.router3, c.n_experts, c.hidden, &L.router_map))
      rc = fail(h, DF_MOE_ECUDA, "tensor map encoding failed");
  }
  h->router_part_rows = (size_t)h->rsplit.nsplit * Tm;
  if (h->router_tc)
    h->router_part_rows = std::max(h->router_part_rows,
                                   router_tc_part_rows(c.n_experts, c.hidden, h->router_tc_min_t,
                                                       (int)Tm, h->sms));
  if (!rc) rc = dalloc(h, &h->router_part, h->router_part_rows * E);
  if (!rc) rc = dalloc(h, &h->logits, Tm * E);
  if (!rc) rc = dalloc(h, &h->ids_ws, Tm * k);
  if (!rc) rc = dalloc(h, &h->w_ws, Tm * k);
  if (!rc) rc = dalloc(h, &h->items, Tm * k);
  if (!rc) rc = dalloc(h, &h->n_items, 1);
  if (!rc) rc = dalloc(h, &h->sorted, Tm * k);
  if (!rc) rc = dalloc(h, &h->hbuf, Tm * k * I);
  if (!rc) rc = dalloc(h, &h->part, Tm * k * H);
  if (!rc && R) rc = dalloc(h, &h->hsh, Tm * R);
  if (!rc) rc = dalloc(h, &h->ysh, Tm * H);
  if (!rc) rc = dalloc(h, &h->xbuf[0], Tm * H);
  if (!rc) rc = dalloc(h, &h->xbuf[1], Tm * H);
  if (!rc) rc = dalloc(h, &h->xn, Tm * H);
  if (!rc) rc = dalloc(h, &h->err, 1);
  if (!rc) rc = dalloc(h, &h->counter, 1);
  if (!rc) {
    void* hp = nullptr;
    if (cudaHostAlloc(&hp, 64, cudaHostAllocPortable | cudaHostAllocMapped) != cudaSuccess)
      rc = fail(h, DF_MOE_ENOMEM, "pinned error mirror failed");
    if (!rc) {
      h->host_allocs.push_back(hp);
      h->err_mirror_h = static_cast<uint32_t*>(hp);
      *h->err_mirror_h = 0u;
      void* dp = nullptr;
      if (cudaHostGetDevicePointer(&dp, hp, 0) != cudaSuccess)
        rc = fail(h, DF_MOE_ECUDA, "error mirror not mapped into the device");
      h->err_mirror_d = static_cast<uint32_t*>(dp);
    }
  }
  if (!rc) rc = dalloc(h, &h->hx, Tm * H);
  if (!rc) rc = dalloc(h, &h->hres, Tm * H);
  if (!rc) rc = dalloc(h, &h->hout, Tm * H);
  if (!rc) rc = dalloc(h, &h->hout32, Tm * H);
  if (!rc) rc = dalloc(h, &h->hids, (size_t)c.n_layers * Tm * k);
  if (!rc) rc = dalloc(h, &h->hw, (size_t)c.n_layers * Tm * k);
  if (!rc && slots) {
    void* hp = nullptr;
    if (cudaHostAlloc(&hp, Tm * k * sizeof(int32_t), cudaHostAllocPortable) != cudaSuccess)
      rc = fail(h, DF_MOE_ENOMEM, "pinned id buffer failed");
    else {
      h->host_allocs.push_back(hp);
      h->ids_h = static_cast<int32_t*>(hp);
    }
    hp = nullptr;
    if (!rc && cudaHostAlloc(&hp, Tm * k * sizeof(CacheCopy),
                             cudaHostAllocPortable | cudaHostAllocMapped) != cudaSuccess)
      rc = fail(h, DF_MOE_ENOMEM, "pinned fill plan failed");
    if (!rc) {
      h->host_allocs.push_back(hp);
      h->fill_h = static_cast<CacheCopy*>(hp);
      void* dp = nullptr;
      if (cudaHostGetDevicePointer(&dp, hp, 0) != cudaSuccess)
        rc = fail(h, DF_MOE_ECUDA, "fill plan not mapped into the device");
      h->fill_d = static_cast<const CacheCopy*>(dp);
    }
  }
  if (!rc) {
    // (the MXFP8 variant runs every batch through its GEMMs)
    h->phase = !h->mx8 &&
               phase_supported(H, c.inter, c.n_shared > 0 ? h->R : 0, c.n_experts, c.top_k);
    if (slots && !h->phase)
      rc = fail(h, DF_MOE_EINVAL, "an expert cache needs the decode phase kernels' shapes");
  }
  if (!rc && (cudaMemset(h->err, 0, sizeof(uint32_t)) != cudaSuccess ||
              cudaMemset(h->counter, 0, sizeof(unsigned int)) != cudaSuccess))
    rc = fail(h, DF_MOE_ECUDA, "cudaMemset failed");
  if (rc) {
    g_thread_err = h->last_error;
    df_moe_destroy(h);
    cudaSetDevice(prev);
    return rc;
  }
  cudaSetDevice(prev);
  *out = h;
  return DF_MOE_OK;
}

int df_moe_create(const df_moe_config* cfg, int cuda_device, df_moe** out) {
  return create_impl(cfg, cuda_device, 0, out);
}

int df_moe_create_cached(const df_moe_config* cfg, int cuda_device, int32_t cache_slots,
                         df_moe** out) {
  if (cache_slots < 1) return fail(nullptr, DF_MOE_EINVAL, "cache_slots must be >= 1");
  return create_impl(cfg, cuda_device, cache_slots, out);
}

int df_moe_cache_stats(const df_moe* h, int64_t* hits, int64_t* misses, int64_t* bytes_in) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  if (hits) *hits = h->cache_hits;
  if (misses) *misses = h->cache_misses;
  if (bytes_in) *bytes_in = h->cache_bytes;
  return DF_MOE_OK;
}

int df_moe_load_experts(df_moe* h, int32_t layer, const df_moe_layer_weights* w,
                        void* stream) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  if (!w) return fail(h, DF_MOE_EINVAL, "null weights");
  const df_moe_config& c = h->cfg;
  if (layer < 0 || layer >= c.n_layers)
    return fail(h, DF_MOE_ERANGE, "layer %d out of range", layer);
  cudaStream_t s = (cudaStream_t)stream;
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  LayerBufs& L = h->layers[layer];
  const cudaMemcpyKind kind = w->src_is_device ? cudaMemcpyDeviceToDevice
                                               : cudaMemcpyHostToDevice;
  const size_t H = c.hidden, Is = c.shared_inter;
  if (w->router) {
    CUDA_OR_FAIL(h, cudaMemcpyAsync(L.router, w->router,
                                    (size_t)c.n_experts * H * sizeof(float),
                                    kind, s));
    if (L.router3)
      CUDA_OR_FAIL(h, launch_router_parts(L.router, c.n_experts, c.hidden, L.router3, s));
    L.router_loaded = true;
  }
  for (int sidx = 0; sidx < c.n_shared; ++sidx) {
    const uint16_t* g = w->shared_gate ? w->shared_gate[sidx] : nullptr;
    const uint16_t* u = w->shared_up ? w->shared_up[sidx] : nullptr;
    const uint16_t* d = w->shared_down ? w->shared_down[sidx] : nullptr;
    if (!g && !u && !d) continue;
    if (!g || !u || !d)
      return fail(h, DF_MOE_EINVAL, "shared expert %d: gate, up and down go together", sidx);
    CUDA_OR_FAIL(h, cudaMemcpyAsync(L.sh_gate + sidx * Is * H, g,
                                    Is * H * sizeof(uint16_t), kind, s));
    CUDA_OR_FAIL(h, cudaMemcpyAsync(L.sh_up + sidx * Is * H, u,
                                    Is * H * sizeof(uint16_t), kind, s));
    // down_s [H][Is] becomes columns sidx*Is .. of down_cat [H][R]
    CUDA_OR_FAIL(h, cudaMemcpy2DAsync(L.sh_down + sidx * Is, h->R * sizeof(uint16_t),
                                      d, Is * sizeof(uint16_t), Is * sizeof(uint16_t),
                                      H, kind, s));
    L.shared_loaded[sidx] = 1;
  }
  if (w->expert_count > 0) {
    if (!w->experts) return fail(h, DF_MOE_EINVAL, "experts is NULL");
    if (w->expert_begin < 0 || w->expert_begin + w->expert_count > c.n_experts)
      return fail(h, DF_MOE_ERANGE, "experts [%d, %d) out of range", w->expert_begin,
                  w->expert_begin + w->expert_count);
    // without a cache the spans go to their home in the arena (with one, the
    // arena holds only slots)
    uint8_t* dst = h->cache_slots ? nullptr : L.arena + (size_t)w->expert_begin * h->span_bytes;
    if (h->cache_slots) {
      // repacked on the device in chunks of 8 spans, then kept in the pinned
      // host pool; the HBM slots fill on demand
      const size_t chunk = 8;
      if (!h->staging) {
        h->staging_spans = chunk;
        int rc = dalloc(h, &h->staging, 2 * chunk * h->span_bytes);
        if (rc) return rc;
      }
      uint8_t* packed = h->staging + chunk * h->span_bytes;
      if (w->src_is_device && !aligned16(w->experts))
        return fail(h, DF_MOE_EINVAL, "device expert spans must be 16-byte aligned");
      for (int e0 = 0; e0 < w->expert_count; e0 += (int)chunk) {
        const int n = (int)std::min<size_t>(chunk, (size_t)(w->expert_count - e0));
        const uint8_t* src = w->experts + (size_t)e0 * h->span_bytes;
        if (!w->src_is_device) {
          CUDA_OR_FAIL(h, cudaMemcpyAsync(h->staging, src, (size_t)n * h->span_bytes,
                                          cudaMemcpyHostToDevice, s));
          src = h->staging;
        }
        RUN(h, K_REPACK, s, span_layout_copy(h, src, packed, n, 0, s));
        CUDA_OR_FAIL(h, cudaMemcpyAsync(L.host_pool + (size_t)(w->expert_begin + e0) *
                                                          h->span_bytes,
                                        packed, (size_t)n * h->span_bytes,
                                        cudaMemcpyDeviceToHost, s));
      }
      CUDA_OR_FAIL(h, cudaStreamSynchronize(s));
      for (int e = w->expert_begin; e < w->expert_begin + w->expert_count; ++e) {
        // a reloaded expert leaves the cache
        const int sl = L.slot_of[e];
        if (sl >= 0) {
          L.expert_of[sl] = -1;
          L.slot_of[e] = -1;
        }
      }
    } else if (w->src_is_device) {
      if (!aligned16(w->experts))
        return fail(h, DF_MOE_EINVAL, "device expert spans must be 16-byte aligned");
      RUN(h, K_REPACK, s, span_layout_copy(h, w->experts, dst, w->expert_count, 0, s));
    } else {
      const size_t chunk = 8;
      if (!h->staging) {
        h->staging_spans = chunk;
        int rc = dalloc(h, &h->staging, chunk * h->span_bytes);
        if (rc) return rc;
      }
      for (int e0 = 0; e0 < w->expert_count; e0 += (int)chunk) {
        const int n = (int)std::min<size_t>(chunk, (size_t)(w->expert_count - e0));
        CUDA_OR_FAIL(h, cudaMemcpyAsync(h->staging,
                                        w->experts + (size_t)e0 * h->span_bytes,
                                        (size_t)n * h->span_bytes,
                                        cudaMemcpyHostToDevice, s));
        RUN(h, K_REPACK, s, span_layout_copy(h, h->staging, dst + (size_t)e0 * h->span_bytes,
                                             n, 0, s));
      }
      CUDA_OR_FAIL(h, cudaStreamSynchronize(s));
    }
    if (h->gemm)
      RUN(h, K_REPACK, s, launch_row_ref(dst, h->span_bytes, c.hidden, c.inter, w->expert_count,
                                         L.eref + (size_t)w->expert_begin *
                                                      (2 * (size_t)c.inter + c.hidden),
                                         s));
    for (int e = w->expert_begin; e < w->expert_begin + w->expert_count; ++e) {
      if (!L.expert_loaded[e]) {
        L.expert_loaded[e] = 1;
        L.n_experts_loaded += 1;
      }
    }
  }
  return DF_MOE_OK;
}

// A device-side error recorded by earlier work on `stream`: synchronises the
// stream, reads and clears the device error word and its host mirror, puts
// the router's block counter (which a call that gave up may have left
// mid-count) back to zero, and returns ETIMEOUT (a bounded wait gave up) or
// EDEVICE (a range check failed). DF_MOE_OK when the word is clear.
static int report_device_error(df_moe* h, cudaStream_t s) {
  CUDA_OR_FAIL(h, cudaStreamSynchronize(s));
  uint32_t e = 0;
  CUDA_OR_FAIL(h, cudaMemcpy(&e, h->err, 4, cudaMemcpyDeviceToHost));
  e |= *reinterpret_cast<volatile uint32_t*>(h->err_mirror_h);
  if (!e) return DF_MOE_OK;
  CUDA_OR_FAIL(h, cudaMemset(h->err, 0, 4));
  CUDA_OR_FAIL(h, cudaMemset(h->counter, 0, sizeof(unsigned int)));
  *reinterpret_cast<volatile uint32_t*>(h->err_mirror_h) = 0u;
  if (e & DEV_ERR_TIMEOUT)
    return fail(h, DF_MOE_ETIMEOUT, "a bounded device wait gave up (error word 0x%x)", e);
  return fail(h, DF_MOE_EDEVICE, "a device-side range check failed (error word 0x%x)", e);
}

// The host mirror of the error word is set: report the error (as above).
static bool mirror_set(const df_moe* h) {
  return *reinterpret_cast<volatile const uint32_t*>(h->err_mirror_h) != 0u;
}

static int forward_impl(df_moe* h, const void* x_bf16, int32_t T,
                        const void* residual_bf16, void* out_bf16, float* out_f32,
                        int32_t* ids, float* weights, uint16_t* trace_x,
                        uint16_t* trace_xn, void* stream, int32_t* ids_host = nullptr,
                        float* w_host = nullptr);

int df_moe_forward(df_moe* h, const void* x_bf16, int32_t T,
                   const void* residual_bf16, void* out_bf16, float* out_f32,
                   int32_t* ids, float* weights, void* stream) {
  return forward_impl(h, x_bf16, T, residual_bf16, out_bf16, out_f32, ids, weights,
                      nullptr, nullptr, stream);
}

int df_moe_forward_trace(df_moe* h, const void* x_bf16, int32_t T, void* out_bf16,
                         float* out_f32, int32_t* ids, float* weights, void* trace_x,
                         void* trace_xn, void* stream) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  if (!(h->cfg.flags & DF_MOE_STACK_RMSNORM_RESIDUAL))
    return fail(h, DF_MOE_EINVAL, "forward_trace needs stack mode");
  return forward_impl(h, x_bf16, T, nullptr, out_bf16, out_f32, ids, weights,
                      (uint16_t*)trace_x, (uint16_t*)trace_xn, stream);
}

static int forward_impl(df_moe* h, const void* x_bf16, int32_t T,
                        const void* residual_bf16, void* out_bf16, float* out_f32,
                        int32_t* ids, float* weights, uint16_t* trace_x,
                        uint16_t* trace_xn, void* stream, int32_t* ids_host,
                        float* w_host) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  const df_moe_config& c = h->cfg;
  h->launches = 0;
  if (!x_bf16 || !out_bf16 || !ids || !weights)
    return fail(h, DF_MOE_EINVAL, "x, out, ids and weights are required");
  if (T < 1 || T > c.max_tokens)
    return fail(h, DF_MOE_ERANGE, "T = %d outside [1, %d]", T, c.max_tokens);
  if (!aligned16(x_bf16) || !aligned16(out_bf16) ||
      (residual_bf16 && !aligned16(residual_bf16)))
    return fail(h, DF_MOE_EINVAL, "x, residual and out must be 16-byte aligned");
  const bool stack = (c.flags & DF_MOE_STACK_RMSNORM_RESIDUAL) != 0;
  if (stack && residual_bf16)
    return fail(h, DF_MOE_EINVAL, "stack mode takes no residual (x is the residual)");
  for (int l = 0; l < c.n_layers; ++l) {
    int rc = check_layer_ready(h, l);
    if (rc) return rc;
  }
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  cudaStream_t s = (cudaStream_t)stream;
  // an error that an earlier call's kernels recorded is reported now, before
  // anything is launched
  if (mirror_set(h)) return report_device_error(h, s);
  const size_t Tk = (size_t)T * c.top_k;
  if (!stack) {
    return layer_forward(h, 0, (const uint16_t*)x_bf16, T,
                         (const uint16_t*)residual_bf16, (uint16_t*)out_bf16,
                         out_f32, ids, weights, s, ids_host, w_host);
  }
  const uint16_t* cur = (const uint16_t*)x_bf16;
  const size_t TH = (size_t)T * c.hidden;
  for (int l = 0; l < c.n_layers; ++l) {
    RUN(h, K_RMSNORM, s, launch_rmsnorm(cur, T, c.hidden, c.rms_eps, h->xn, s));
    if (trace_x)
      CUDA_OR_FAIL(h, cudaMemcpyAsync(trace_x + l * TH, cur, TH * 2, cudaMemcpyDeviceToDevice, s));
    if (trace_xn)
      CUDA_OR_FAIL(h, cudaMemcpyAsync(trace_xn + l * TH, h->xn, TH * 2,
                                      cudaMemcpyDeviceToDevice, s));
    const bool last = l == c.n_layers - 1;
    uint16_t* nxt = last ? (uint16_t*)out_bf16 : h->xbuf[l & 1];
    int rc = layer_forward(h, l, h->xn, T, cur, nxt, last ? out_f32 : nullptr,
                           ids + (size_t)l * Tk, weights + (size_t)l * Tk, s,
                           ids_host ? ids_host + (size_t)l * Tk : nullptr,
                           w_host ? w_host + (size_t)l * Tk : nullptr);
    if (rc) return rc;
    cur = nxt;
  }
  return DF_MOE_OK;
}

namespace {

// Where a host-API buffer lives: pinned host memory the device reaches
// directly (its device address, 16-byte aligned), ordinary host memory, or
// memory the device owns (device or managed).
enum class Mem { pinned, host, device };
Mem classify(const void* p, void** dev) {
  cudaPointerAttributes a{};
  *dev = nullptr;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return Mem::host;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer && aligned16(a.devicePointer)) {
    *dev = a.devicePointer;
    return Mem::pinned;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return Mem::device;
  return Mem::host;
}

int ensure_io(df_moe* h) {
  if (h->io_h) return DF_MOE_OK;
  const df_moe_config& c = h->cfg;
  const size_t n = (size_t)c.max_tokens * c.hidden, nk = (size_t)c.n_layers * c.max_tokens * c.top_k;
  const size_t sz[6] = {n * 2, n * 2, n * 2, n * 4, nk * 4, nk * 4};
  size_t off = 0;
  for (int i = 0; i < 6; ++i) {
    h->io_off[i] = off;
    off += (sz[i] + 255) / 256 * 256;
  }
  void* hp = nullptr;
  if (cudaHostAlloc(&hp, off, cudaHostAllocPortable | cudaHostAllocMapped) != cudaSuccess) {
    cudaGetLastError();
    return fail(h, DF_MOE_ENOMEM, "pinned host staging of %zu bytes failed", off);
  }
  void* dp = nullptr;
  if (cudaHostGetDevicePointer(&dp, hp, 0) != cudaSuccess) {
    cudaFreeHost(hp);
    return fail(h, DF_MOE_ECUDA, "host staging not mapped into the device");
  }
  h->host_allocs.push_back(hp);
  h->io_h = static_cast<uint8_t*>(hp);
  h->io_d = static_cast<uint8_t*>(dp);
  return DF_MOE_OK;
}

}  // namespace

// Host buffers in and out. The device moves the data itself: inputs are read
// from pinned host memory (the caller's, when it is pinned and mapped, else a
// staging copy) by a small copy kernel that the router's weight stream
// overlaps; the last kernel writes the output, ids and weights straight into
// pinned host memory. Buffers in device or managed memory go through
// cudaMemcpyAsync.
int df_moe_forward_host(df_moe* h, const uint16_t* x_bf16, int32_t T,
                        const uint16_t* residual_bf16, uint16_t* out_bf16,
                        float* out_f32, int32_t* ids, float* weights,
                        void* stream) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  const df_moe_config& c = h->cfg;
  if (!x_bf16 || !out_bf16)
    return fail(h, DF_MOE_EINVAL, "x and out are required");
  if (T < 1 || T > c.max_tokens)
    return fail(h, DF_MOE_ERANGE, "T = %d outside [1, %d]", T, c.max_tokens);
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  int rc = ensure_io(h);
  if (rc) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t n = (size_t)T * c.hidden;
  const size_t nk = (size_t)c.n_layers * T * c.top_k;
  // inputs into the device buffers
  const void* in_src[2] = {x_bf16, residual_bf16};
  uint16_t* in_dst[2] = {h->hx, h->hres};
  for (int i = 0; i < 2; ++i) {
    if (!in_src[i]) continue;
    void* dev = nullptr;
    switch (classify(in_src[i], &dev)) {
      case Mem::pinned:
        RUN(h, K_OTHER, s, launch_copy16(dev, in_dst[i], n * 2, s));
        break;
      case Mem::host:
        memcpy(h->io_h + h->io_off[i], in_src[i], n * 2);
        RUN(h, K_OTHER, s, launch_copy16(h->io_d + h->io_off[i], in_dst[i], n * 2, s));
        break;
      case Mem::device:
        CUDA_OR_FAIL(h, cudaMemcpyAsync(in_dst[i], in_src[i], n * 2, cudaMemcpyDefault, s));
        break;
    }
  }
  // outputs: written by the device where it reaches them directly
  void* const user_out[4] = {out_bf16, out_f32, ids, weights};
  const size_t out_bytes[4] = {n * 2, n * 4, nk * 4, nk * 4};
  void* dev_side[4] = {h->hout, h->hout32, h->hids, h->hw};  // device buffers
  void* out_dev[4] = {nullptr, nullptr, nullptr, nullptr};   // what the kernels write
  Mem kind[4] = {Mem::device, Mem::device, Mem::device, Mem::device};
  for (int i = 0; i < 4; ++i) {
    if (!user_out[i]) continue;
    void* dev = nullptr;
    kind[i] = classify(user_out[i], &dev);
    out_dev[i] = kind[i] == Mem::pinned ? dev
                 : kind[i] == Mem::host ? h->io_d + h->io_off[2 + i]
                                        : dev_side[i];
  }
  // out and out_f32 are the forward's outputs; ids and weights stay in the
  // device buffers the later kernels read, and the combine copies them
  const bool ids_direct = ids && weights && kind[2] != Mem::device && kind[3] != Mem::device;
  rc = forward_impl(h, h->hx, T, residual_bf16 ? h->hres : nullptr,
                    out_dev[0], out_f32 ? static_cast<float*>(out_dev[1]) : nullptr, h->hids,
                    h->hw, nullptr, nullptr, stream,
                    ids_direct ? static_cast<int32_t*>(out_dev[2]) : nullptr,
                    ids_direct ? static_cast<float*>(out_dev[3]) : nullptr);
  if (rc) return rc;
  for (int i = 0; i < 4; ++i) {
    if (!user_out[i]) continue;
    const bool direct = i < 2 ? kind[i] != Mem::device : ids_direct;
    if (!direct)
      CUDA_OR_FAIL(h, cudaMemcpyAsync(user_out[i], dev_side[i], out_bytes[i], cudaMemcpyDefault,
                                      s));
  }
  CUDA_OR_FAIL(h, cudaStreamSynchronize(s));
  for (int i = 0; i < 4; ++i) {
    if (!user_out[i] || kind[i] != Mem::host) continue;
    if (i >= 2 && !ids_direct) continue;
    memcpy(user_out[i], h->io_h + h->io_off[2 + i], out_bytes[i]);
  }
  // this call's own device-side errors (published by its last kernel)
  if (mirror_set(h)) return report_device_error(h, s);
  return DF_MOE_OK;
}

int df_moe_sync(df_moe* h, void* stream) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  return report_device_error(h, (cudaStream_t)stream);
}

int df_moe_test_drop_arrival(df_moe* h) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  h->drop_next = true;
  return DF_MOE_OK;
}

// ---- single steps ----------------------------------------------------------

int df_moe_step_router(df_moe* h, int32_t layer, const void* x_bf16, int32_t T,
                       float* logits, void* stream) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  const df_moe_config& c = h->cfg;
  if (layer < 0 || layer >= c.n_layers) return fail(h, DF_MOE_ERANGE, "bad layer");
  if (T < 1 || T > c.max_tokens) return fail(h, DF_MOE_ERANGE, "bad T");
  if (!x_bf16 || !logits) return fail(h, DF_MOE_EINVAL, "null pointer");
  if (!all_aligned16({x_bf16, logits}))
    return fail(h, DF_MOE_EINVAL, "device arrays must be 16-byte aligned");
  if (!h->layers[layer].router_loaded) return fail(h, DF_MOE_ESTATE, "router not loaded");
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  cudaStream_t s = (cudaStream_t)stream;
  return route(h, layer, (const uint16_t*)x_bf16, T, h->ids_ws, h->w_ws, s,
               logits, T == 1 ? 1 : kOneItemPerExpert);
}

int df_moe_step_topk(df_moe* h, const float* logits, int32_t T, int32_t* ids,
                     float* weights, void* stream) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  const df_moe_config& c = h->cfg;
  if (T < 1 || T > c.max_tokens) return fail(h, DF_MOE_ERANGE, "bad T");
  if (!logits || !ids || !weights) return fail(h, DF_MOE_EINVAL, "null pointer");
  if (!all_aligned16({logits, ids, weights}))
    return fail(h, DF_MOE_EINVAL, "device arrays must be 16-byte aligned");
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  cudaStream_t s = (cudaStream_t)stream;
  // the top-k kernel sums nsplit partial-logit planes; one plane = logits
  RUN(h, K_TOPK, s, launch_topk(logits, 1, T, c.n_experts, c.top_k, nullptr,
                                ids, weights, nullptr, nullptr, nullptr, s));
  return DF_MOE_OK;
}

int df_moe_step_group(df_moe* h, const int32_t* ids, int32_t T, int32_t* offs,
                      int32_t* tok, int32_t* slot, int32_t* n_union,
                      void* stream) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  const df_moe_config& c = h->cfg;
  if (T < 1 || T > c.max_tokens) return fail(h, DF_MOE_ERANGE, "bad T");
  if (!ids || !offs || !tok || !slot || !n_union)
    return fail(h, DF_MOE_EINVAL, "null pointer");
  if (!all_aligned16({ids, offs, tok, slot, n_union}))
    return fail(h, DF_MOE_EINVAL, "device arrays must be 16-byte aligned");
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  cudaStream_t s = (cudaStream_t)stream;
  RUN(h, K_GROUP, s, launch_group(ids, T, c.top_k, c.n_experts, offs, tok, slot,
                                  n_union, h->items, h->n_items, h->sorted,
                                  kOneItemPerExpert, h->err, s));
  return DF_MOE_OK;
}

int df_moe_step_expert_gateup(df_moe* h, int32_t layer, const void* x_bf16,
                              int32_t T, const int32_t* ids, float* hbuf,
                              void* stream) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  const df_moe_config& c = h->cfg;
  if (layer < 0 || layer >= c.n_layers) return fail(h, DF_MOE_ERANGE, "bad layer");
  if (T < 1 || T > c.max_tokens) return fail(h, DF_MOE_ERANGE, "bad T");
  if (!x_bf16 || !ids || !hbuf) return fail(h, DF_MOE_EINVAL, "null pointer");
  if (!all_aligned16({x_bf16, ids, hbuf}))
    return fail(h, DF_MOE_EINVAL, "device arrays must be 16-byte aligned");
  if (h->layers[layer].n_experts_loaded != c.n_experts)
    return fail(h, DF_MOE_ESTATE, "experts not loaded");
  if (h->cache_slots)
    return fail(h, DF_MOE_EINVAL, "single expert steps read the resident arena: not with a cache");
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  cudaStream_t s = (cudaStream_t)stream;
  const int tg = kOneItemPerExpert;
  RUN(h, K_GROUP, s, launch_group(ids, T, c.top_k, c.n_experts, nullptr, nullptr,
                                  nullptr, nullptr, h->items, h->n_items,
                                  h->sorted, tg, h->err, s, h->mx_inv));
  return expert_gateup(h, layer, (const uint16_t*)x_bf16, T,
                       std::min(T * c.top_k, c.n_experts), tg, hbuf, s);
}

int df_moe_step_expert_down(df_moe* h, int32_t layer, const float* hbuf,
                            int32_t T, const int32_t* ids, const float* weights,
                            float* y, void* stream) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  const df_moe_config& c = h->cfg;
  if (layer < 0 || layer >= c.n_layers) return fail(h, DF_MOE_ERANGE, "bad layer");
  if (T < 1 || T > c.max_tokens) return fail(h, DF_MOE_ERANGE, "bad T");
  if (!hbuf || !ids || !weights || !y) return fail(h, DF_MOE_EINVAL, "null pointer");
  if (!all_aligned16({hbuf, ids, weights, y}))
    return fail(h, DF_MOE_EINVAL, "device arrays must be 16-byte aligned");
  if (h->layers[layer].n_experts_loaded != c.n_experts)
    return fail(h, DF_MOE_ESTATE, "experts not loaded");
  if (h->cache_slots)
    return fail(h, DF_MOE_EINVAL, "single expert steps read the resident arena: not with a cache");
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  cudaStream_t s = (cudaStream_t)stream;
  const int tg = kOneItemPerExpert;
  RUN(h, K_GROUP, s, launch_group(ids, T, c.top_k, c.n_experts, nullptr, nullptr,
                                  nullptr, nullptr, h->items, h->n_items,
                                  h->sorted, tg, h->err, s));
  const int rc = expert_down(h, layer, hbuf, T, std::min(T * c.top_k, c.n_experts), tg, s);
  if (rc) return rc;
  RUN(h, K_COMBINE, s, launch_combine(h->part, weights, T, c.top_k, c.hidden,
                                      nullptr, nullptr, y, nullptr, h->err, h->err_mirror_d, s));
  return DF_MOE_OK;
}

int df_moe_step_mxfp8(df_moe* h, const float* v, int32_t rows, int32_t n, uint8_t* codes,
                      uint8_t* scales, void* stream) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  if (!v || !codes || !scales) return fail(h, DF_MOE_EINVAL, "null pointer");
  if (rows < 0 || n < 0 || n % 32) return fail(h, DF_MOE_EINVAL, "n must be a multiple of 32");
  if (!aligned16(v)) return fail(h, DF_MOE_EINVAL, "v must be 16-byte aligned");
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  cudaStream_t s = (cudaStream_t)stream;
  RUN(h, K_MX8_QUANT, s, launch_mx8_plain(v, rows, n, codes, scales, s));
  return DF_MOE_OK;
}

int df_moe_step_shared(df_moe* h, int32_t layer, const void* x_bf16, int32_t T,
                       float* y, void* stream) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  const df_moe_config& c = h->cfg;
  if (layer < 0 || layer >= c.n_layers) return fail(h, DF_MOE_ERANGE, "bad layer");
  if (T < 1 || T > c.max_tokens) return fail(h, DF_MOE_ERANGE, "bad T");
  if (!x_bf16 || !y) return fail(h, DF_MOE_EINVAL, "null pointer");
  if (!all_aligned16({x_bf16, y}))
    return fail(h, DF_MOE_EINVAL, "device arrays must be 16-byte aligned");
  for (int sidx = 0; sidx < c.n_shared; ++sidx)
    if (!h->layers[layer].shared_loaded[sidx])
      return fail(h, DF_MOE_ESTATE, "shared expert %d not loaded", sidx);
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  cudaStream_t s = (cudaStream_t)stream;
  if (c.n_shared == 0) {
    CUDA_OR_FAIL(h, cudaMemsetAsync(y, 0, (size_t)T * c.hidden * 4, s));
    return DF_MOE_OK;
  }
  return shared_part(h, layer, (const uint16_t*)x_bf16, T, y, s);
}

int df_moe_step_rmsnorm(df_moe* h, const void* x_bf16, int32_t T, void* xn_bf16,
                        void* stream) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  const df_moe_config& c = h->cfg;
  if (T < 1 || T > c.max_tokens) return fail(h, DF_MOE_ERANGE, "bad T");
  if (!x_bf16 || !xn_bf16) return fail(h, DF_MOE_EINVAL, "null pointer");
  if (!all_aligned16({x_bf16, xn_bf16}))
    return fail(h, DF_MOE_EINVAL, "device arrays must be 16-byte aligned");
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  cudaStream_t s = (cudaStream_t)stream;
  RUN(h, K_RMSNORM, s, launch_rmsnorm((const uint16_t*)x_bf16, T, c.hidden,
                                      c.rms_eps, (uint16_t*)xn_bf16, s));
  return DF_MOE_OK;
}

int df_moe_read_expert_span(df_moe* h, int32_t layer, int32_t expert,
                            uint8_t* dst) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  const df_moe_config& c = h->cfg;
  if (layer < 0 || layer >= c.n_layers || expert < 0 || expert >= c.n_experts)
    return fail(h, DF_MOE_ERANGE, "layer/expert out of range");
  if (!dst) return fail(h, DF_MOE_EINVAL, "null dst");
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  uint8_t* tmp = nullptr;
  CUDA_OR_FAIL(h, cudaMalloc(&tmp, 2 * h->span_bytes));
  const uint8_t* src = h->layers[layer].arena + (size_t)expert * h->span_bytes;
  cudaError_t e = cudaSuccess;
  if (h->cache_slots) {  // the expert's home is the pinned host pool
    e = cudaMemcpy(tmp + h->span_bytes, h->layers[layer].host_pool +
                                            (size_t)expert * h->span_bytes,
                   h->span_bytes, cudaMemcpyHostToDevice);
    src = tmp + h->span_bytes;
  }
  if (e == cudaSuccess) e = span_layout_copy(h, src, tmp, 1, 1, nullptr);
  if (e == cudaSuccess) e = cudaMemcpy(dst, tmp, h->span_bytes, cudaMemcpyDeviceToHost);
  cudaFree(tmp);
  if (e != cudaSuccess)
    return fail(h, DF_MOE_ECUDA, "read-back failed: %s", cudaGetErrorString(e));
  return DF_MOE_OK;
}

// ---- timing ------------------------------------------------------------------

int df_moe_timing_enable(df_moe* h, int on) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  h->timing = on != 0;
  return DF_MOE_OK;
}

static int drain(df_moe* h) {
  for (auto& p : h->pending) {
    CUDA_OR_FAIL(h, cudaEventSynchronize(p.b));
    float ms = 0.f;
    CUDA_OR_FAIL(h, cudaEventElapsedTime(&ms, p.a, p.b));
    h->kind_ms[p.kind] += ms;
    h->kind_n[p.kind] += 1;
    h->event_pool.push_back(p.a);
    h->event_pool.push_back(p.b);
  }
  h->pending.clear();
  return DF_MOE_OK;
}

int df_moe_timing_reset(df_moe* h) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  int rc = drain(h);
  for (int i = 0; i < K_NKINDS; ++i) { h->kind_ms[i] = 0; h->kind_n[i] = 0; }
  return rc;
}

int df_moe_timing_get(df_moe* h, int kind, const char** name, int64_t* launches,
                      double* total_ms) {
  if (!h) return fail(nullptr, DF_MOE_EINVAL, "null handle");
  if (kind < 0 || kind >= K_NKINDS) return fail(h, DF_MOE_ERANGE, "bad kind");
  int rc = drain(h);
  if (rc) return rc;
  if (name) *name = kKindNames[kind];
  if (launches) *launches = h->kind_n[kind];
  if (total_ms) *total_ms = h->kind_ms[kind];
  return DF_MOE_OK;
}

int df_moe_last_launch_count(const df_moe* h) { return h ? h->launches : 0; }

// ---- CUDA graphs ----------------------------------------------------------

struct df_moe_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int device = 0;
  int launches = 0;
};

int df_moe_graph_create(df_moe* h, const void* x_bf16, int32_t T, const void* residual_bf16,
                        void* out_bf16, float* out_f32, int32_t* ids, float* weights,
                        df_moe_graph** out) {
  if (!h || !out) return fail(h, DF_MOE_EINVAL, "null handle or output");
  *out = nullptr;
  if (h->timing) return fail(h, DF_MOE_EINVAL, "turn timing off before capturing a graph");
  if (h->cache_slots)
    return fail(h, DF_MOE_EINVAL, "an expert cache plans each layer on the host: no graphs");
  CUDA_OR_FAIL(h, cudaSetDevice(h->device));
  if (!h->cap_stream)
    CUDA_OR_FAIL(h, cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking));
  CUDA_OR_FAIL(h, cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
  const int rc = forward_impl(h, x_bf16, T, residual_bf16, out_bf16, out_f32, ids, weights,
                              nullptr, nullptr, h->cap_stream);
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(h->cap_stream, &graph);
  if (rc) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (ec != cudaSuccess)
    return fail(h, DF_MOE_ECUDA, "graph capture failed: %s", cudaGetErrorString(ec));
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
  if (ei != cudaSuccess) {
    cudaGraphDestroy(graph);
    return fail(h, DF_MOE_ECUDA, "graph instantiation failed: %s", cudaGetErrorString(ei));
  }
  df_moe_graph* g = new df_moe_graph;
  g->graph = graph;
  g->exec = exec;
  g->device = h->device;
  g->launches = h->launches;
  *out = g;
  return DF_MOE_OK;
}

int df_moe_graph_launch(df_moe_graph* g, void* stream) {
  if (!g) return fail(nullptr, DF_MOE_EINVAL, "null graph");
  cudaError_t e = cudaSetDevice(g->device);
  if (e == cudaSuccess) e = cudaGraphLaunch(g->exec, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(nullptr, DF_MOE_ECUDA, "graph launch failed: %s", cudaGetErrorString(e));
  return DF_MOE_OK;
}

int df_moe_graph_launch_count(const df_moe_graph* g) { return g ? g->launches : 0; }

void df_moe_graph_destroy(df_moe_graph* g) {
  if (!g) return;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(g->device);
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  cudaSetDevice(prev);
  delete g;
}

int df_moe_stream_read(const void* buf, size_t bytes, uint32_t* sink, void* stream) {
  if (!buf || !sink || (bytes & 15) || ((uintptr_t)buf & 15))
    return fail(nullptr, DF_MOE_EINVAL, "buf must be 16-byte aligned, bytes a multiple of 16");
  const cudaError_t e = launch_stream_read(buf, bytes, sink, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(nullptr, DF_MOE_ECUDA, "read probe launch failed: %s", cudaGetErrorString(e));
  return DF_MOE_OK;
}

}  // extern "C"

namespace dfm {
void set_thread_error(const char* msg) { g_thread_err = msg; }
}  // namespace dfm
