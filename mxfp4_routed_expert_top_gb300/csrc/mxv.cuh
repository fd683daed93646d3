// mxv.cuh — the MXFP4 dequant-fused GEMV of the routed experts, as a
// per-CTA device function (used by the stand-alone kernels and by the decode
// phase kernels that also run the shared experts).
//
// The operation is the Deltafin README's fused MXFP4 dequant+GEMV ("Techniques
// / Compute": decode the 4-bit weights and multiply in one pass, the e8m0
// scale applied on the exponent), restated for HBM streaming on sm_103a.
//
// Why the tensor cores: at the HBM rate GB300 streams ~12.8 T MXFP4 weights/s
// against ~40 T lane-instructions/s of issue, i.e. about three instructions
// per weight for everything. A CUDA-core decode + fp32 FMA needs 3.75 (ncu),
// which makes the GEMV issue-bound. Here a warp decodes E2M1 pairs straight
// into m16n8k16 A fragments (one hardware cvt per 2 weights) and the tokens
// ride in the N = 8 columns; the contraction itself costs one warp
// instruction per 256 weights.
//
//   * A CTA holds NS "slots" = one producer warp + one consumer warp per
//     512-column chunk. A slot owns a contiguous range of tiles (16 rows x K
//     of one expert).
//   * The producer streams each tile (K/64 groups of codes + scales, one
//     contiguous block) with cp.async.bulk into a shared-memory ring
//     (mbarriers, bounded waits).
//   * Consumers: one 16-byte lds per lane = its A fragments for 4 k-steps;
//     every 32-column MX block is accumulated by two MMAs into a temporary
//     that is scaled by 2^(s-127) (per row) in fp32 and added to the result.
//   * B (x) fragments live in registers as f16. The gate/up input (bf16) is
//     scaled per (token, chunk) by a power of two that puts its largest
//     magnitude at exponent 15, so every entry within 2^32 of that maximum
//     is exact in f16 whatever the token's range. The down input h (fp32,
//     |h| up to ~1e5) is scaled the same way per (token, chunk) and split
//     into hi and lo columns (~22 bits). The scales are undone on the fp32
//     partial sums.
//   * An item (one expert and all its tokens) is processed in token groups of
//     8 (gate/up) or 4 (down) against the tile already in shared memory, so
//     each expert's weights cross HBM once per call.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "mxfrag.cuh"
#include "pipeline.cuh"

namespace dfm {


constexpr int kMaxWarps = 16;
// 64-column groups per consumer chunk: gate/up (K = H) in chunks of 512
// columns, down (K = I, a quarter to a fifth of H) in chunks of 256 so that a
// tile still spreads over several warps and a slot keeps a deep ring.
constexpr int kCGGateUp = 8, kCGDown = 4;
__host__ __device__ constexpr int mxv_cg(int mode) { return mode == 0 ? kCGGateUp : kCGDown; }
// 16-row tiles per pipeline unit (one copy, one reduction): down's tiles are a
// quarter to a fifth of gate/up's, so it takes them in pairs.
__host__ __device__ constexpr int mxv_unit(int mode) { return mode == 0 ? 1 : 2; }

// Consumer chunks of a K-long row and the groups of chunk c.
__host__ __device__ inline int mxv_nchunks(int K, int cg) { return (K + 64 * cg - 1) / (64 * cg); }
__host__ __device__ inline int mxv_nv(int K, int c, int cg) {
  const int n = mx_ngroups(K) - cg * c;
  return n < cg ? n : cg;
}
constexpr int kMaxStages = 8;
constexpr int kRedRing = 2;  // epilogue reduction ring depth
constexpr size_t kSmemBudget = 214 * 1024;

struct MxvArgs {
  const uint8_t* arena;
  size_t span_bytes;
  int H, I, k;
  const uint16_t* x;      // gate/up input, bf16 [T][H]
  const float* hin;       // down input, fp32 [T*k][I]
  const Item* items;
  const int32_t* n_items;
  const int32_t* sorted;
  float* out;             // gate/up: h [T*k][I]; down: part [T*k][H]
  uint32_t* err;
  int early;              // down only: the selection is complete at grid start
  const uint8_t* const* spans;  // [E] span addresses (expert cache), or null: arena
  // Range checks: an item whose expert is outside [0, E) or whose
  // assignments leave [0, nassign), an assignment index outside [0,
  // nassign), or more than max_items items is skipped and recorded in *err
  // (DEV_ERR_RANGE).
  int E = 0, nassign = 0, max_items = 0;
  uint32_t wait_limit = kWaitLimit;  // polls of every bounded wait
  // Test hook: the call's first unit (of whichever slot owns it) is neither
  // copied nor announced on its barrier, so its consumers' bounded wait runs
  // out.
  int drop = 0;
};

__host__ __device__ inline size_t align128(size_t v) { return (v + 127) & ~(size_t)127; }

struct SlotGeom {
  int stages;
  size_t stage_bytes, red_bytes, bytes;
};

__host__ __device__ inline SlotGeom slot_geom(int K, int NS, int cg, int u) {
  SlotGeom g;
  const int NCH = mxv_nchunks(K, cg);
  g.stage_bytes = (size_t)u * mx_tile_bytes(K);
  g.red_bytes = (size_t)kRedRing * NCH * u * 32 * 16;
  const size_t fixed = g.red_bytes;
  const size_t per_slot = kSmemBudget / NS;
  int st = (int)((per_slot > fixed ? per_slot - fixed : 0) / g.stage_bytes);
  g.stages = st < 2 ? 2 : (st > kMaxStages ? kMaxStages : st);
  g.bytes = align128((size_t)g.stages * g.stage_bytes + fixed);
  return g;
}

// A slot is its chunk warps, a producer warp and, where the CTA has a warp
// to spare for it (the same number of slots either way), a reducer warp.
__host__ __device__ inline bool mxv_own_reducer(int K, int cg) {
  const int NCH = mxv_nchunks(K, cg);
  return kMaxWarps / (NCH + 2) >= 1 && kMaxWarps / (NCH + 2) == kMaxWarps / (NCH + 1);
}
__host__ __device__ inline int mxv_wps(int K, int cg) {
  return mxv_nchunks(K, cg) + (mxv_own_reducer(K, cg) ? 2 : 1);
}
__host__ __device__ inline int slots_per_cta(int K, int cg) {
  const int ns = kMaxWarps / mxv_wps(K, cg);
  return ns > 0 ? ns : 1;
}

constexpr int kMxvBarsPerSlot = 2 * kMaxStages + 2 * kRedRing;
constexpr int kMxvBars = kMaxWarps / 2 * kMxvBarsPerSlot;  // at most 8 slots

// Dynamic shared memory of one CTA for contraction length K.
__host__ __device__ inline size_t mxv_smem_bytes(int K, int cg, int u) {
  const int NS = slots_per_cta(K, cg);
  return (size_t)NS * slot_geom(K, NS, cg, u).bytes;
}
// The one-token gate/up path also keeps the token's B fragments in shared
// memory (after the slots): per chunk, per pair of k-steps, per lane t4 of
// B row 0, 16 bytes; then 16 zero bytes that the other rows read.
__host__ __device__ inline size_t mxv_x_bytes(int K, int cg) {
  return (size_t)mxv_nchunks(K, cg) * (2 * cg) * 4 * 16 + 16;
}

// MODE 0: gate/up (K = H, 8 tokens per group), MODE 1: down (K = I, 4 tokens
// per group, columns 2t / 2t+1 = hi / lo part of token t).
// Initialises the mbarriers of every slot of the CTA (one thread each slot).
template <int MODE>
__device__ __forceinline__ void mxv_set_up_barriers(const MxvArgs& a, uint64_t* bars) {
  constexpr int CG = mxv_cg(MODE);
  const int K = MODE == 0 ? a.H : a.I;
  const int NCH = mxv_nchunks(K, CG);
  const int wps = mxv_wps(K, CG);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = slots_per_cta(K, CG);
  const int s = warp / wps, role = warp - s * wps;
  if (s < NS && role == NCH && lane == 0) {
    const int S = slot_geom(K, NS, CG, mxv_unit(MODE)).stages;
    uint64_t* full = bars + (size_t)s * kMxvBarsPerSlot;
    uint64_t* empty = full + kMaxStages;
    uint64_t* rfull = empty + kMaxStages;
    uint64_t* rempty = rfull + kRedRing;
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NCH);
    }
    for (int i = 0; i < kRedRing; ++i) {
      mbar_init(&rfull[i], NCH);
      mbar_init(&rempty[i], 1);
    }
    fence_barrier_init();  // the initialising thread's inits, to the async proxy
  }
}

// One CTA's share of the work: slot s of the CTA takes the s-th of the
// CTA's NS ranges of the ncta * NS equal ranges of tiles. `smem` holds the
// slots' rings and reduction entries (mxv_smem_bytes), `bars` their
// mbarriers (kMxvBars). Warps beyond the CTA's NS slots only take part in the
// barrier set-up. With `set_up` false the caller has already run
// mxv_set_up_barriers, a __syncthreads and the wait for the preceding grid.
// ONE (gate/up of a single token whose selection the CTA made itself): every
// item is that token's, so its B fragments are loaded once before the loop,
// the items need no range check, and only the token's D column is summed.
template <int MODE, bool ONE = false>
__device__ __forceinline__ void mxv_cta(const MxvArgs& a, uint8_t* smem, uint64_t* bars,
                                        int cta, int ncta, bool set_up = true) {
  static_assert(!ONE || MODE == 0, "the one-token path is gate/up only");
  constexpr int GT = MODE == 0 ? 8 : 4;  // tokens per group
  constexpr int CG = mxv_cg(MODE);
  constexpr int U = mxv_unit(MODE);
  const int K = MODE == 0 ? a.H : a.I;
  const int NCH = mxv_nchunks(K, CG);
  const bool own_reducer = mxv_own_reducer(K, CG);
  const int wps = mxv_wps(K, CG);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = slots_per_cta(K, CG);
  const int s = warp / wps, role = warp - s * wps;
  const SlotGeom geo = slot_geom(K, NS, CG, U);
  const int S = geo.stages;
  uint8_t* base = smem + (size_t)s * geo.bytes;
  uint8_t* ring = base;
  float* red = reinterpret_cast<float*>(base + (size_t)S * geo.stage_bytes);
  uint64_t* full = bars + (size_t)s * kMxvBarsPerSlot;
  uint64_t* empty = full + kMaxStages;
  uint64_t* rfull = empty + kMaxStages;   // reduction entry written by all chunks
  uint64_t* rempty = rfull + kRedRing;    // reduction entry summed and freed

  if (set_up) {
    mxv_set_up_barriers<MODE>(a, bars);
    __syncthreads();
  }

  // Gate/up needs the selection and x of the preceding kernels. Down's
  // weight stream needs only the selection; launched right after the gate/up
  // kernel (`early`), the selection is complete before this grid starts (the
  // gate/up grid published it before triggering this launch), so the
  // producer streams weights while the gate/up grid drains and only the
  // consumers wait, for h. Reads made before the wait bypass L1. The
  // selection may also sit in shared memory (items, n_items, sorted), for a
  // caller that computed it in the CTA (not with `early`).
  const bool early = MODE == 1 && a.early;
  if (!early && set_up) pdl_wait();
  // Down: every CTA is resident (one wave), so the next kernel (the
  // combine) may be set up now and start on each SM as this one's CTA
  // leaves. Gate/up triggers only implicitly, when its CTAs exit: launched
  // onto SMs that gate/up left early, down's weight streams competed for HBM
  // with the gate/up stragglers on the critical path. Measured on GB300 at
  // batch 1 that cost 1.6 us a step on average and pushed p90 from 103 to
  // 109 us.
  if (MODE == 1) pdl_launch_dependents();
  if (s >= NS) return;
  const SpanLayout L = span_layout(a.H, a.I);
  const int tpi = (MODE == 0 ? (2 * a.I) / 16 : a.H / 16) / U;  // units per item
  int n_items = early ? __ldcg(a.n_items) : *a.n_items;
  if (n_items < 0 || n_items > a.max_items) {
    if (threadIdx.x == 0) atomicOr(a.err, DEV_ERR_RANGE);
    n_items = n_items < 0 ? 0 : a.max_items;
  }
  const int ntiles = n_items * tpi;
  // an item the kernels can run: its expert exists and its assignments lie
  // in the sorted list (the producer and the consumers skip the others alike)
  auto item_ok = [&](const Item& it) {
    return ONE || ((unsigned)it.e < (unsigned)a.E && it.cnt >= 1 && it.pos >= 0 &&
                   it.pos + it.cnt <= a.nassign);
  };
  const long long nslots = (long long)ncta * NS;
  const long long gs = (long long)cta * NS + s;
  const int t_begin = (int)(ntiles * gs / nslots);
  const int t_end = (int)(ntiles * (gs + 1) / nslots);
  const size_t sec_off = MODE == 0 ? L.gu : L.dn;
  const uint32_t tile_bytes = (uint32_t)mx_tile_bytes(K);
  const uint32_t unit_bytes = U * tile_bytes;

  if (role == NCH) {
    // ---------------- producer: one elected lane ----------------
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      bool ok = true;
      int cur_item = -1;
      bool cur_ok = false;
      const uint8_t* span = nullptr;
      // per stage: armed at least once (bit) and the parity of its last
      // armed phase (bit), for the final wait on the copies in flight
      uint32_t armed = 0u, last_par = 0u;
      for (int t = t_begin; t < t_end; ++t) {
        const int item = t / tpi, j = t - item * tpi;
        if (item != cur_item) {
          cur_item = item;
          Item it;
          if (early) {
            const int4 v = __ldcg(reinterpret_cast<const int4*>(a.items + item));
            it = Item{v.x, v.y, v.z, v.w};
          } else {
            it = a.items[item];
          }
          cur_ok = item_ok(it);
          if (!cur_ok) {
            atomicOr(a.err, DEV_ERR_RANGE);
          } else {
            span = a.spans ? reinterpret_cast<const uint8_t*>(__ldcg(
                                 reinterpret_cast<const unsigned long long*>(a.spans) + it.e))
                           : a.arena + (size_t)it.e * a.span_bytes;
          }
        }
        if (!cur_ok) continue;
        if (!mbar_wait(&empty[stage], phase ^ 1, a.wait_limit)) { ok = false; break; }
        if (a.drop && t == 0) {
          // test hook: this stage is never filled
        } else {
          uint8_t* dst = ring + (size_t)stage * geo.stage_bytes;
          mbar_arrive_expect_tx(&full[stage], unit_bytes);
          bulk_g2s(dst, span + sec_off + (size_t)j * unit_bytes, unit_bytes,
                   &full[stage], pol);
          armed |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
        }
        if (++stage == (uint32_t)S) { stage = 0; phase ^= 1; }
      }
      if (!ok) atomicOr(a.err, DEV_ERR_TIMEOUT);
      // Every copy this lane issued must land before the CTA may exit: wait
      // (bounded) for the last armed phase of each stage.
      for (int i = 0; i < S; ++i)
        if (armed >> i & 1u) (void)mbar_wait(&full[i], last_par >> i & 1u, a.wait_limit);
    }
    return;
  }

  // ------- consumers: warp `role` = chunk c (or the reducer, NCH + 1) -------
  if (early) pdl_wait();
  const bool reducer = role == NCH + 1;
  const int c = role;
  const int g = lane >> 2, t4 = lane & 3;
  const int nv = mxv_nv(K, c, CG);
  uint32_t stage = 0, phase = 0;
  int cur_item = -1, loaded_grp = -1, loaded_tok = -2;
  Item it{0, 0, 0, 0};
  int a_lane = -1;     // sorted[pos + lane] of the current item (cnt <= 32)
  uint32_t bx[4 * CG][2];  // B fragments, 2 registers per k-step of the chunk
  float csc = 1.f;     // down: 2^s of this lane's token (column pair)
  // gate/up: 2^s of the group's eight tokens (B rows g), one row per warp
  __shared__ float xsc[kMaxWarps][8];
  int n_epi = 0;
  bool ok = true;

  // assignment of token `ti` of the current item (all lanes must call)
  auto assignment = [&](int ti) -> int {
    const int v = __shfl_sync(0xffffffffu, a_lane, ti & 31);
    if (ti >= it.cnt) return -1;
    if (it.cnt <= 32) return v;
    const int w = a.sorted[it.pos + ti];
    if ((unsigned)w >= (unsigned)a.nassign) {
      atomicOr(a.err, DEV_ERR_RANGE);
      return -1;
    }
    return w;
  };

  bool cur_ok = false;
  // gate/up B fragments of token `tok` (-1: none) for this warp's chunk, as
  // f16 of x * 2^-s, s putting the largest magnitude of the token's chunk at
  // exponent 15: bf16's 8-bit significands are then exact in f16 down to
  // 2^32 below the maximum, and smaller entries keep an absolute error below
  // 2^-40 of it. A NaN or inf maximum (exponent field 255) keeps s = 112, so
  // non-finite stays non-finite. Every lane must call; 2^s goes to xsc.
  auto load_x = [&](int tok) {
    // pass 1: the raw bf16 pairs and the largest |x| of the chunk (the four
    // lanes t4 = 0..3 of row g hold it all)
    uint32_t mbits = 0u;
#pragma unroll
    for (int ks = 0; ks < 4 * CG; ++ks) {
      uint32_t v0 = 0u, v1 = 0u;
      if (tok >= 0 && ks < 4 * nv) {
        const uint16_t* xp = a.x + (size_t)tok * a.H + 64 * CG * c + 16 * ks + 2 * t4;
        v0 = *reinterpret_cast<const uint32_t*>(xp);
        v1 = *reinterpret_cast<const uint32_t*>(xp + 8);
      }
      bx[ks][0] = v0;
      bx[ks][1] = v1;
      mbits = max(mbits, max(max(v0 & 0x7FFFu, (v0 >> 16) & 0x7FFFu),
                             max(v1 & 0x7FFFu, (v1 >> 16) & 0x7FFFu)));
    }
    mbits = max(mbits, __shfl_xor_sync(0xffffffffu, mbits, 1));
    mbits = max(mbits, __shfl_xor_sync(0xffffffffu, mbits, 2));
    // pass 2: scale and convert in place
    int sh = 0;
    if (mbits != 0u) sh = min(max((int)(mbits >> 7) - 127 - 15, -120), 112);
    const float dn = pow2i(-sh);
#pragma unroll
    for (int ks = 0; ks < 4 * CG; ++ks) {
      const uint32_t w0 = bx[ks][0], w1 = bx[ks][1];
      bx[ks][0] = f2_to_h2(__uint_as_float(w0 << 16) * dn, __uint_as_float(w0 & 0xFFFF0000u) * dn);
      bx[ks][1] = f2_to_h2(__uint_as_float(w1 << 16) * dn, __uint_as_float(w1 & 0xFFFF0000u) * dn);
    }
    // 2^s of token g, kept in shared memory (not in registers across the
    // loop, where the B fragments fill the register file)
    if (t4 == 0) xsc[warp][g] = pow2i(sh);
    __syncwarp();
  };
  // one token: its B fragments for this chunk go to shared memory once
  // (B row 0 only; the other rows read zeros), and the loop reads them back
  // per k-step pair, which leaves the register file to the decode pipeline
  uint4* const xs = reinterpret_cast<uint4*>(smem + (size_t)NS * geo.bytes);
  const uint4* xsl = xs + (g == 0 ? (size_t)c * (2 * CG) * 4 + t4
                                  : (size_t)mxv_nchunks(K, CG) * (2 * CG) * 4);
  const int xstride = g == 0 ? 4 : 0;
  if (ONE && !reducer) {
    load_x(g == 0 ? 0 : -1);  // every item is token 0's
    if (g == 0) {
#pragma unroll
      for (int pp = 0; pp < 2 * CG; ++pp)
        xs[(size_t)(c * (2 * CG) + pp) * 4 + t4] =
            make_uint4(bx[2 * pp][0], bx[2 * pp][1], bx[2 * pp + 1][0], bx[2 * pp + 1][1]);
    }
    if (c == 0 && lane == 0) xs[(size_t)mxv_nchunks(K, CG) * (2 * CG) * 4] = make_uint4(0, 0, 0, 0);
    __syncwarp();
  }

  for (int t = t_begin; t < t_end && ok; ++t) {
    const int item = t / tpi, j = t - item * tpi;
    if (item != cur_item) {
      cur_item = item;
      it = a.items[item];
      cur_ok = item_ok(it);
      a_lane = cur_ok && lane < it.cnt ? a.sorted[it.pos + lane] : -1;
      if ((unsigned)a_lane >= (unsigned)a.nassign && a_lane != -1) {
        atomicOr(a.err, DEV_ERR_RANGE);
        a_lane = -1;
      }
    }
    if (!cur_ok) continue;  // skipped by the producer too
    if (!reducer) {
      ok = mbar_wait(&full[stage], phase, a.wait_limit);
      if (!ok) break;
    }
    const uint8_t* tile = ring + (size_t)stage * geo.stage_bytes;

    for (int grp = 0; grp < it.cnt && ok; grp += GT) {
      float acc[U][4];
#pragma unroll
      for (int st = 0; st < U; ++st) acc[st][0] = acc[st][1] = acc[st][2] = acc[st][3] = 0.f;
      if (!reducer) {
        // ---- B fragments of this token group (reloaded only when they change)
        if (item != loaded_grp >> 16 || grp != (loaded_grp & 0xFFFF)) {
          if (MODE == 0) {
            if (!ONE) {
              const int aa = assignment(grp + g);
              const int tok = aa >= 0 ? aa / a.k : -1;
              if (__any_sync(0xffffffffu, tok != loaded_tok)) {
                loaded_tok = tok;
                load_x(tok);
              }
            }
          } else {
            const int aa = assignment(grp + (g >> 1));
            const float* hrow = aa >= 0 ? a.hin + (size_t)aa * a.I + 64 * CG * c + 2 * t4 : nullptr;
            // pass 1: largest |h| of the token's chunk (the four lanes t4 = 0..3
            // of a row g hold it all between them)
            float m = 0.f;
            if (hrow) {
              for (int ks = 0; ks < 4 * nv; ++ks) {
                const float2 p0 = *reinterpret_cast<const float2*>(hrow + 16 * ks);
                const float2 p1 = *reinterpret_cast<const float2*>(hrow + 16 * ks + 8);
                m = fmaxf(m, fmaxf(fmaxf(fabsf(p0.x), fabsf(p0.y)),
                                   fmaxf(fabsf(p1.x), fabsf(p1.y))));
              }
            }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            int sh = 0;
            if (m > 0.f) {
              const int e = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;
              sh = min(max(e - 14, -112), 112);
            }
            const float dn = pow2i(-sh);
            const bool lo = (g & 1) != 0;
            // pass 2: scaled f16 hi (even g) or lo (odd g) parts
  #pragma unroll
            for (int ks = 0; ks < 4 * CG; ++ks) {
              uint32_t r[2] = {0u, 0u};
              if (hrow && ks < 4 * nv) {
  #pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  const float2 p = *reinterpret_cast<const float2*>(hrow + 16 * ks + 8 * hh);
                  const float v0 = p.x * dn, v1 = p.y * dn;
                  const __half2 hi = __floats2half2_rn(v0, v1);
                  if (!lo) {
                    r[hh] = *reinterpret_cast<const uint32_t*>(&hi);
                  } else {
                    const float2 f = __half22float2(hi);
                    r[hh] = f2_to_h2(v0 - f.x, v1 - f.y);
                  }
                }
              }
              bx[ks][0] = r[0];
              bx[ks][1] = r[1];
            }
            // this lane's D columns 2t4, 2t4+1 belong to token t4 (rows g = 2 t4)
            csc = __shfl_sync(0xffffffffu, pow2i(sh), 4 * (2 * t4));
          }
          loaded_grp = (item << 16) | grp;
        }

        // ---- the unit's tiles (16 rows x this chunk each) against the group
        const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int st = 0; st < U; ++st) {
#pragma unroll
          for (int v = 0; v < CG; ++v) {
            if (v < nv) {
              const uint8_t* grp_p = tile + st * tile_bytes + kGroupBytes * (CG * c + v);
              const uint4 q = lds128(grp_p + 16 * lane);
              const uint32_t w[4] = {q.x, q.y, q.z, q.w};
              // scales: (row g, block 0), (row g, block 1), (row g+8, 0), (row g+8, 1)
              const uint32_t sc = lds_u32(grp_p + 512 + 4 * g);
#pragma unroll
              for (int hb = 0; hb < 2; ++hb) {  // the two 32-column blocks of v
                uint32_t a0[4], a1[4];
                decode_word(w[2 * hb], a0);
                decode_word(w[2 * hb + 1], a1);
                float d[4];
                if (ONE) {
                  const uint4 bb = lds128(xsl + (size_t)(2 * v + hb) * xstride);
                  mma16816(d, a0, bb.x, bb.y, zero);
                  mma16816(d, a1, bb.z, bb.w, d);
                } else {
                  mma16816(d, a0, bx[4 * v + 2 * hb][0], bx[4 * v + 2 * hb][1], zero);
                  mma16816(d, a1, bx[4 * v + 2 * hb + 1][0], bx[4 * v + 2 * hb + 1][1], d);
                }
                const float sg = __uint_as_float(((sc >> (8 * hb)) & 0xFFu) << 23);
                const float sg8 = __uint_as_float(((sc >> (16 + 8 * hb)) & 0xFFu) << 23);
                acc[st][0] = fmaf(d[0], sg, acc[st][0]);
                if (!ONE) acc[st][1] = fmaf(d[1], sg, acc[st][1]);
                acc[st][2] = fmaf(d[2], sg8, acc[st][2]);
                if (!ONE) acc[st][3] = fmaf(d[3], sg8, acc[st][3]);
              }
            }
          }
        }
        if (grp + GT >= it.cnt) {  // last use of this unit: release the stage
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[stage]);
        }
        if (MODE == 1) {
          // y rows g, g+8 of token t4 = (hi + lo) * 2^s
#pragma unroll
          for (int st = 0; st < U; ++st) {
            acc[st][0] = (acc[st][0] + acc[st][1]) * csc;
            acc[st][2] = (acc[st][2] + acc[st][3]) * csc;
          }
        } else {
          // undo the scales of this lane's D columns 2t4, 2t4+1 (tokens
          // 2t4, 2t4+1 of the group)
          const float2 cs = lds_f2(&xsc[warp][2 * t4]);
#pragma unroll
          for (int st = 0; st < U; ++st) {
            acc[st][0] *= cs.x;
            acc[st][1] *= cs.y;
            acc[st][2] *= cs.x;
            acc[st][3] *= cs.y;
          }
        }
      }

      // ---- cross-chunk reduction through a ring of shared-memory entries:
      // every chunk warp writes its partial; the reducer (a warp of its own
      // where the CTA has one to spare, else the chunk warps in turn) sums
      // the entry in chunk order, writes the rows and frees the entry
      const int r = n_epi % kRedRing, u = n_epi / kRedRing;
      float4* rb = reinterpret_cast<float4*>(red) + (size_t)r * NCH * U * 32;  // [c][st][lane]
      if (!reducer) {
        if (u >= 1 && !mbar_wait(&rempty[r], (u - 1) & 1, a.wait_limit)) { ok = false; break; }
#pragma unroll
        for (int st = 0; st < U; ++st)
          rb[(c * U + st) * 32 + lane] = make_float4(acc[st][0], acc[st][1], acc[st][2], acc[st][3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&rfull[r]);
      }
      if (reducer || (!own_reducer && c == n_epi % NCH)) {
        if (!mbar_wait(&rfull[r], u & 1, a.wait_limit)) { ok = false; break; }
#pragma unroll
        for (int st = 0; st < U; ++st) {
          float4 sum = rb[st * 32 + lane];
          for (int cc = 1; cc < NCH; ++cc) {
            const float4 v4 = rb[(cc * U + st) * 32 + lane];
            sum.x += v4.x; sum.y += v4.y; sum.z += v4.z; sum.w += v4.w;
          }
          const int tl = U * j + st;  // tile of the item
          if (MODE == 0) {
            // columns 2t4, 2t4+1 = tokens grp+2t4, grp+2t4+1; rows g (gate)
            // and g+8 (up) of intermediate index 8 tl + g
            const int a0i = assignment(grp + 2 * t4), a1i = assignment(grp + 2 * t4 + 1);
            if (a0i >= 0) a.out[(size_t)a0i * a.I + 8 * tl + g] = silu_f(sum.x) * sum.z;
            if (a1i >= 0) a.out[(size_t)a1i * a.I + 8 * tl + g] = silu_f(sum.y) * sum.w;
          } else {
            const int ai = assignment(grp + t4);
            if (ai >= 0) {
              a.out[(size_t)ai * a.H + 16 * tl + g] = sum.x;
              a.out[(size_t)ai * a.H + 16 * tl + g + 8] = sum.z;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty[r]);
      }
      ++n_epi;
    }
    if (!reducer && ++stage == (uint32_t)S) { stage = 0; phase ^= 1; }
  }
  // A failed (timed-out) wait: record it and leave; every other wait of the
  // CTA is bounded too, so the rest of the slot ends on its own.
  if (!ok) atomicOr(a.err, DEV_ERR_TIMEOUT);
}

}  // namespace dfm
