// bfv.cuh — the streaming bf16 GEMV of the shared experts, as a per-CTA
// device function (used by the stand-alone kernels and by the decode phase
// kernels that also run the routed experts).
//
// The shared experts run for every token next to the routed ones ("add the
// two shared experts", Deltafin analysis §5.1). Their n_shared gate/up
// matrices are concatenated along rows and their down matrices along
// columns, so the shared part is one SwiGLU FFN of intermediate n_shared*Is.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"
#include "mxfrag.cuh"
#include "pipeline.cuh"

namespace dfm {

constexpr int kColsPerWarp = 1024;  // 4 x 256 columns, 8 bf16 per lane
constexpr int kIt = kColsPerWarp / 256;
constexpr int kTT = 8;              // tokens per pass

__device__ __forceinline__ void bf16x8_to_f32(uint4 q, float (&f)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// Streaming bf16 GEMV. Persistent CTAs of NS slots; a slot is one producer
// warp plus NW consumer warps, warp w owning columns [1024 w, 1024 w + 1024).
// A tile is 4 weight rows: gate rows i, i+1 and up rows i, i+1 (MODE 0, the
// SwiGLU pair) or down rows r..r+3 (MODE 1). The producer streams tiles with
// cp.async.bulk into a shared-memory ring; consumers read 16 bytes (8 bf16)
// per lane per step and accumulate in fp32 against x held in registers.
// Partials meet through a small ring of shared-memory entries whose
// finalizer role rotates over the consumer warps (mbarrier handoffs, bounded
// waits).
// ---------------------------------------------------------------------------
constexpr int kRows = 4;
constexpr int kRing = 4;
constexpr int kMaxStagesB = 8;
constexpr size_t kBudget = 200 * 1024;

struct BfvArgs {
  const uint16_t* w0;  // MODE 0: gate [R][K]; MODE 1: down [H][K]
  const uint16_t* w1;  // MODE 0: up [R][K]
  int rows, K;         // MODE 0: R (intermediates); MODE 1: H
  const void* x;       // MODE 0: bf16 [T][K]; MODE 1: fp32 [T][K]
  int T;
  float* out;          // MODE 0: hsh [T][R]; MODE 1: ysh [T][H]
  uint32_t* err;
};

__host__ __device__ inline int bfv_warps(int K) {
  const int w = (K + kColsPerWarp - 1) / kColsPerWarp;
  return w < 1 ? 1 : (w > 8 ? 8 : w);
}
struct BfvGeom {
  int stages;
  size_t stage_bytes, red_bytes, bytes;
};
__host__ __device__ inline BfvGeom bfv_geom(int K, int NS);
// slots per CTA for wps warps a slot: as many as the warp limit allows while
// the CTA's shared memory (at least two stages a slot) stays within 220 KB
__host__ __device__ inline int bfv_slots_for(int K, int wps) {
  int ns = 16 / wps;
  if (ns < 1) ns = 1;
  while (ns > 1 && (size_t)ns * bfv_geom(K, ns).bytes > 220 * 1024) --ns;
  return ns;
}
// A slot is its consumer warps, a producer warp and, where the CTA has a warp
// to spare for it (the same number of slots either way), a reducer warp.
__host__ __device__ inline bool bfv_own_reducer(int K) {
  const int NW = bfv_warps(K);
  return bfv_slots_for(K, NW + 2) == bfv_slots_for(K, NW + 1);
}
__host__ __device__ inline int bfv_wps(int K) {
  return bfv_warps(K) + (bfv_own_reducer(K) ? 2 : 1);
}
__host__ __device__ inline int bfv_slots(int K) { return bfv_slots_for(K, bfv_wps(K)); }
__host__ __device__ inline BfvGeom bfv_geom(int K, int NS) {
  BfvGeom g;
  const int NW = bfv_warps(K);
  g.stage_bytes = (size_t)kRows * K * 2;
  g.red_bytes = (size_t)kRing * NW * kRows * kTT * 4;
  const size_t fixed = g.red_bytes;
  const size_t per = kBudget / NS;
  int st = (int)((per > fixed ? per - fixed : 0) / g.stage_bytes);
  g.stages = st < 2 ? 2 : (st > kMaxStagesB ? kMaxStagesB : st);
  g.bytes = ((size_t)g.stages * g.stage_bytes + fixed + 127) & ~(size_t)127;
  return g;
}

constexpr int kBfvBarsPerSlot = 2 * kMaxStagesB + 2 * kRing;
constexpr int kBfvBars = 8 * kBfvBarsPerSlot;  // at most 8 slots

// Dynamic shared memory of one CTA for contraction length K.
__host__ __device__ inline size_t bfv_smem_bytes(int K) {
  const int NS = bfv_slots(K);
  return (size_t)NS * bfv_geom(K, NS).bytes;
}

// One CTA's share of the work (NS slots of the CTA over ncta * NS equal
// ranges of tiles). `smem` holds the rings and reduction entries
// (bfv_smem_bytes), `bars` the mbarriers (kBfvBars). With `wait` the inputs
// come from the preceding grid (programmatic dependent launch); without it
// they must have been complete when the grid started. Inputs are read
// through L2 only.
// TT: tokens a pass (1, 2, 4 or 8); with TT = 1 the one token's x stays in
// registers across tiles.
template <int MODE, int TT>
__device__ __forceinline__ void bfv_cta(const BfvArgs& a, uint8_t* smem, uint64_t* bars,
                                        int cta, int ncta, bool wait) {
  const int NW = bfv_warps(a.K);
  const bool own_reducer = bfv_own_reducer(a.K);
  const int wps = bfv_wps(a.K);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = bfv_slots(a.K);
  const int s = warp / wps, role = warp - s * wps;
  const BfvGeom geo = bfv_geom(a.K, NS);
  const int S = geo.stages;
  uint8_t* base = smem + (size_t)s * geo.bytes;
  float* red = reinterpret_cast<float*>(base + (size_t)S * geo.stage_bytes);
  uint64_t* full = bars + (size_t)s * kBfvBarsPerSlot;
  uint64_t* empty = full + kMaxStagesB;
  uint64_t* rfull = empty + kMaxStagesB;
  uint64_t* rempty = rfull + kRing;
  if (s < NS && role == NW && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NW);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&rfull[i], NW);
      mbar_init(&rempty[i], 1);
    }
    fence_barrier_init();  // the initialising thread's inits, to the async proxy
  }
  __syncthreads();
  if (wait) pdl_wait();
  if (s >= NS) return;

  const int ntiles = MODE == 0 ? a.rows / 2 : a.rows / kRows;
  const long long nslots = (long long)ncta * NS;
  const long long gs = (long long)cta * NS + s;
  const int t_begin = (int)(ntiles * gs / nslots);
  const int t_end = (int)(ntiles * (gs + 1) / nslots);
  if (t_begin >= t_end) return;  // no tiles for this slot (or no rows at all)
  const uint32_t row_bytes = (uint32_t)a.K * 2;

  if (role == NW) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      bool ok = true;
      for (int t = t_begin; t < t_end; ++t) {
        if (!mbar_wait(&empty[stage], phase ^ 1)) { ok = false; break; }
        uint8_t* dst = base + (size_t)stage * geo.stage_bytes;
        mbar_arrive_expect_tx(&full[stage], kRows * row_bytes);
        if (MODE == 0) {
          const size_t i0 = (size_t)2 * t;
          bulk_g2s(dst, a.w0 + i0 * a.K, 2 * row_bytes, &full[stage], pol);
          bulk_g2s(dst + 2 * row_bytes, a.w1 + i0 * a.K, 2 * row_bytes, &full[stage], pol);
        } else {
          bulk_g2s(dst, a.w0 + (size_t)kRows * t * a.K, kRows * row_bytes, &full[stage], pol);
        }
        ++issued;
        if (++stage == (uint32_t)S) { stage = 0; phase ^= 1; }
      }
      if (!ok) atomicOr(a.err, DEV_ERR_TIMEOUT);
      for (int i = 0; i < S && i < issued; ++i) {
        const int n = (issued - i + S - 1) / S;
        (void)mbar_wait(&full[i], (uint32_t)((n - 1) & 1));
      }
    }
    return;
  }

  // consumers: warp `role` owns columns [1024 role, +1024); role NW + 1 is
  // the reducer
  const bool reducer = role == NW + 1;
  const int w = role;
  const int c0 = w * kColsPerWarp + 8 * lane;
  constexpr bool ONE = TT == 1;
  float xr[kIt][8];  // x of the single token (ONE), kept across tiles
#pragma unroll
  for (int i = 0; i < kIt; ++i) {
#pragma unroll
    for (int q = 0; q < 8; ++q) xr[i][q] = 0.f;
    if (ONE && c0 + 256 * i < a.K) {
      if (MODE == 0) {
        bf16x8_to_f32(__ldcg(reinterpret_cast<const uint4*>(
                          static_cast<const uint16_t*>(a.x) + c0 + 256 * i)), xr[i]);
      } else {
        const float* xp = static_cast<const float*>(a.x) + c0 + 256 * i;
        const float4 p = __ldcg(reinterpret_cast<const float4*>(xp));
        const float4 q = __ldcg(reinterpret_cast<const float4*>(xp + 4));
        xr[i][0] = p.x; xr[i][1] = p.y; xr[i][2] = p.z; xr[i][3] = p.w;
        xr[i][4] = q.x; xr[i][5] = q.y; xr[i][6] = q.z; xr[i][7] = q.w;
      }
    }
  }
  uint32_t stage = 0, phase = 0;
  int n_epi = 0;
  bool ok = true;
  for (int t = t_begin; t < t_end && ok; ++t) {
    if (!reducer) {
      ok = mbar_wait(&full[stage], phase);
      if (!ok) break;
    }
    const uint16_t* tile = reinterpret_cast<const uint16_t*>(base + (size_t)stage * geo.stage_bytes);
    const int groups = ONE ? 1 : (a.T + TT - 1) / TT;
    for (int gi = 0; gi < groups && ok; ++gi) {
      const int t0 = gi * TT;
      const int tt = ONE ? 1 : min(TT, a.T - t0);
      const int ri = n_epi % kRing, u = n_epi / kRing;
      float* rb = red + (size_t)ri * NW * kRows * kTT;
      if (!reducer) {
        float acc[kRows][TT];
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
          for (int q = 0; q < TT; ++q) acc[r][q] = 0.f;
#pragma unroll
        for (int i = 0; i < kIt; ++i) {
          if (c0 + 256 * i >= a.K) continue;
          float xf[TT][8];
          if (ONE) {
#pragma unroll
            for (int q = 0; q < 8; ++q) xf[0][q] = xr[i][q];
          } else {
#pragma unroll
            for (int tk = 0; tk < TT; ++tk) {
#pragma unroll
              for (int q = 0; q < 8; ++q) xf[tk][q] = 0.f;
              if (tk < tt) {
                if (MODE == 0) {
                  bf16x8_to_f32(__ldcg(reinterpret_cast<const uint4*>(
                                    static_cast<const uint16_t*>(a.x) + (size_t)(t0 + tk) * a.K +
                                    c0 + 256 * i)), xf[tk]);
                } else {
                  const float* xp = static_cast<const float*>(a.x) + (size_t)(t0 + tk) * a.K +
                                    c0 + 256 * i;
                  const float4 p = __ldcg(reinterpret_cast<const float4*>(xp));
                  const float4 q = __ldcg(reinterpret_cast<const float4*>(xp + 4));
                  xf[tk][0] = p.x; xf[tk][1] = p.y; xf[tk][2] = p.z; xf[tk][3] = p.w;
                  xf[tk][4] = q.x; xf[tk][5] = q.y; xf[tk][6] = q.z; xf[tk][7] = q.w;
                }
              }
            }
          }
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            float wf[8];
            bf16x8_to_f32(lds128(tile + (size_t)r * a.K + c0 + 256 * i), wf);
#pragma unroll
            for (int tk = 0; tk < TT; ++tk)
#pragma unroll
              for (int q = 0; q < 8; ++q) acc[r][tk] = fmaf(wf[q], xf[tk][q], acc[r][tk]);
          }
        }
        if (gi == groups - 1) {  // last read of this tile: release the stage
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[stage]);
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
          for (int q = 0; q < TT; ++q) acc[r][q] = warp_sum(acc[r][q]);

        // partials of (row, token) through the reduction ring
        if (u >= 1 && !mbar_wait(&rempty[ri], (u - 1) & 1)) { ok = false; break; }
        if (lane == 0) {
#pragma unroll
          for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int q = 0; q < TT; ++q) rb[(w * kRows + r) * kTT + q] = acc[r][q];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rfull[ri]);
      }
      if (reducer || (!own_reducer && w == n_epi % NW)) {
        if (!mbar_wait(&rfull[ri], u & 1)) { ok = false; break; }
        float v = 0.f;
        const int r = lane / kTT, q = lane % kTT;
        if (lane < kRows * kTT && q < tt)
          for (int ww = 0; ww < NW; ++ww) v += rb[(ww * kRows + r) * kTT + q];
        if (MODE == 0) {
          // rows 0,1 = gate of intermediates 2t, 2t+1; rows 2,3 = up
          const float up = __shfl_down_sync(0xffffffffu, v, 2 * kTT);
          if (lane < 2 * kTT && q < tt)
            a.out[(size_t)(t0 + q) * a.rows + 2 * t + r] = silu_f(v) * up;
        } else {
          if (lane < kRows * kTT && q < tt)
            a.out[(size_t)(t0 + q) * a.rows + kRows * t + r] = v;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty[ri]);
      }
      ++n_epi;
    }
    if (!reducer && ++stage == (uint32_t)S) { stage = 0; phase ^= 1; }
  }
  if (!ok) atomicOr(a.err, DEV_ERR_TIMEOUT);
}

}  // namespace dfm
