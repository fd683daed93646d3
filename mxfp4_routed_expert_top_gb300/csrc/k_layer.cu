// k_layer.cu — one MoE layer for a decode batch (T <= 8 tokens) as a single
// persistent cooperative kernel.
//
// What it computes is the layer of the Deltafin analysis ("§5.1 MoE block":
// router scores all experts, the top 16 are applied as SwiGLU FFNs, their
// outputs are weighted by a softmax over the selected logits and summed, the
// shared experts are added) with the weights in MXFP4 as in the Deltafin
// README ("Techniques / Compute": 4-bit E2M1 values with an e8m0 scale per 32
// weights, decoded and multiplied in one pass).
//
// Why one kernel: at batch 1 the layer moves 438.6 MB, 65 us at HBM speed,
// split over a chain of dependent steps. As separate launches every step pays
// its own ramp-up, tail and launch gap (together about a third of the time).
// Here all warps of the GPU work through one queue of units in dependency
// order, so the next step's weights are streaming while the previous step's
// last units finish, and the HBM stays busy from the first router row to the
// last down tile.
//
// Units (all are one warp; `ld` = direct 16-byte loads, 8 groups in flight):
//   RT  router: logits of one expert over a K slice, fp32 FMA
//   TK  top-k of one token: sum of the slices, selection, softmax; the last
//       TK groups the T*k assignments into per-expert items
//   SG  shared gate/up: 16 rows x K slice of one shared expert, f16 MMA
//   RG  routed gate/up: 16 rows x K slice of one selected expert, MXFP4
//   SD  shared down: 16 output rows of one shared expert
//   RD  routed down: 16 output rows of one selected expert
// Results pass between units as follows:
//   * split-K partials: the last slice to finish (ticket) sums all slices in
//     slice order and applies SwiGLU;
//   * the last gate/up tile of an expert (ticket) converts its h into the
//     down GEMV's B fragments (f16 hi + lo, scaled per token by a power of
//     two) and raises the expert's flag (the call's epoch);
//   * the last down unit of each 16-row block (ticket) does the weighted
//     combine, adds the shared experts and the residual, and writes out.
// Every sum has a fixed order, so results do not depend on timing. Waits
// poll with a time and iteration limit and report DEV_ERR_TIMEOUT. The
// launch is cooperative, so every warp the queue can wait on is resident.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "internal.h"
#include "mxfrag.cuh"
#include "pipeline.cuh"

namespace dfm {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kStageBytes = 4 * kGroupBytes;  // 4 MXFP4 groups; f16 and fp32 use 2048
constexpr int kMaxStages = 4;
constexpr int kMaxSlices = 8;  // K slices of a gate/up tile (host caps ks_gu, ks_sg)
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;
constexpr uint32_t kWaitPolls = 1u << 22;
constexpr unsigned FULL = 0xffffffffu;

__host__ __device__ inline size_t align128(size_t v) { return (v + 127) & ~(size_t)127; }

// Shared memory per CTA: x as f16 B fragments (H/64 x T x 128 bytes), x as
// bf16 for the router (T x H x 2 bytes, when it fits beside rings of at least
// 3 stages; else the router reads x from global memory), then each warp's
// ring with as many stages (<= kMaxStages) as fit. The dynamic budget leaves
// room below the 227 KB per-block limit for the static unit table.
constexpr int kSmemLimit = 224 * 1024;
constexpr long long kRingPerStage = (long long)kWarps * (kStageBytes + 8);
__host__ __device__ inline size_t layer_xf_bytes(int H, int T) {
  return align128((size_t)(H >> 6) * T * 128);
}
__host__ __device__ inline size_t layer_xr_bytes(int H, int T) {
  const size_t xr = align128((size_t)T * H * 2);
  return (long long)(kSmemLimit - layer_xf_bytes(H, T) - xr) >= 3 * kRingPerStage ? xr : 0;
}
__host__ __device__ inline int layer_stages(int H, int T) {
  const long long s =
      ((long long)kSmemLimit - (long long)layer_xf_bytes(H, T) - (long long)layer_xr_bytes(H, T)) /
      kRingPerStage;
  return (int)(s > kMaxStages ? kMaxStages : s);
}


__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Bounded wait (all lanes) for *f == epoch; every lane's last poll is an
// acquire that saw the value. false: timed out (recorded in err).
__device__ bool wait_flag(const uint32_t* f, uint32_t epoch, uint32_t* err) {
  uint64_t t0 = 0;
  for (uint32_t it = 0; it < kWaitPolls; ++it) {
    const uint32_t v = ld_acquire(f);
    if (__all_sync(FULL, v == epoch)) return true;
    if (it == 0) t0 = globaltimer();
    const int late = (it & 31) == 31 && globaltimer() - t0 > kWaitNs;
    if (__shfl_sync(FULL, late, 0)) break;
    __nanosleep(128);
  }
  if ((threadIdx.x & 31) == 0) atomicOr(err, DEV_ERR_TIMEOUT);
  __syncwarp();
  return false;
}

// Takes a ticket: returns its previous value (all lanes). The increment is a
// release for every lane's earlier writes (the warp barrier orders them
// before lane 0's atomic) and an acquire for the lanes' later reads. The
// caller that gets the last value resets the ticket.
__device__ __forceinline__ uint32_t take_ticket(uint32_t* t) {
  __syncwarp();
  uint32_t old = 0;
  if ((threadIdx.x & 31) == 0)
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
  old = __shfl_sync(FULL, old, 0);
  __syncwarp();
  return old;
}

// Publishes every lane's earlier writes under flag f = epoch.
__device__ __forceinline__ void raise_flag(uint32_t* f, uint32_t epoch) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) st_release(f, epoch);
}

// Monotone map of a float to an unsigned integer (a < b <=> key(a) < key(b)
// for non-NaN values).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
  return v > bv || (v == bv && e < be);
}

struct Ctx {
  const LayerKernelArgs* a;
  uint32_t xa;  // shared address of x as B fragments, k-steps 0-1 of each group
  uint32_t xb;  // k-steps 2-3
  uint32_t xr;  // shared address of x as bf16 [T][H] for the router, or 0
  int lane, g, t4;
  bool items_seen;
  int n_items;
  // this warp's ring of bulk copies: S stages of kStageBytes, one mbarrier
  // each; stage sequence numbers `head` (issued) and `tail` (consumed)
  uint32_t rbuf, rbar;
  int S;
  uint32_t head, tail;
  // the next unit, claimed when the current one starts (lane 0 holds the
  // claim), and how far its weights have been prefetched: nstate 0 = not
  // resolved yet, 1 = streaming (nissued stages issued), 2 = nothing to
  // prefetch. `pre` = stages of the current unit issued before it started.
  uint32_t claim;
  int nstate, nissued, pre;
  const volatile int* ub;  // unit ranges (shared memory)
  void* nsrc;              // this warp's slot for the next unit's source (shared memory)
};

__device__ __forceinline__ uint32_t* sw(const LayerKernelArgs& a, size_t off) {
  return a.sync + off;
}

// ---------------------------------------------------------------------------
// Per-warp streaming through shared memory.
//
// Lane 0 of a warp issues bulk copies (cp.async.bulk, completing on the
// stage's mbarrier) of a unit's weights, which are one contiguous range, in
// chunks of at most kStageBytes, keeping S stages in flight; the warp
// consumes them in order. Each SM thus holds up to 16 x S x 2 KB of loads in
// flight without spending registers on them, and a warp busy with an
// epilogue or a wait does not idle the SM's memory pipe.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 lds128a(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32a(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void ring_issue(Ctx& c, const void* src, uint32_t bytes) {
  const uint32_t slot = c.head % (uint32_t)c.S;
  if (c.lane == 0) {
    const uint32_t bar = c.rbar + 8u * slot;
    const uint32_t dst = c.rbuf + (uint32_t)kStageBytes * slot;
    // the warp's reads of this stage (generic proxy) precede the copy's writes
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(l2_evict_first_policy())
        : "memory");
  }
  ++c.head;
}

// A stage gathered from 4 row tiles: group G of each (`src` = tile 0's group,
// tiles `stride` bytes apart), 4 x kGroupBytes.
__device__ __forceinline__ void ring_issue4(Ctx& c, const uint8_t* src, size_t stride) {
  const uint32_t slot = c.head % (uint32_t)c.S;
  if (c.lane == 0) {
    const uint32_t bar = c.rbar + 8u * slot;
    const uint32_t dst = c.rbuf + (uint32_t)kStageBytes * slot;
    const uint64_t pol = l2_evict_first_policy();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(4u * kGroupBytes)
                 : "memory");
#pragma unroll
    for (int r = 0; r < 4; ++r)
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
          "[%0], [%1], %2, [%3], %4;" ::"r"(dst + (uint32_t)(r * kGroupBytes)),
          "l"(src + r * stride), "r"((uint32_t)kGroupBytes), "r"(bar), "l"(pol)
          : "memory");
  }
  ++c.head;
}

// Bounded wait for stage `n` (all lanes); returns its shared address, or 0
// after a timeout (recorded).
__device__ __forceinline__ uint32_t ring_wait(Ctx& c, uint32_t n) {
  const uint32_t slot = n % (uint32_t)c.S, parity = (n / (uint32_t)c.S) & 1u;
  const uint32_t bar = c.rbar + 8u * slot;
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (__all_sync(FULL, ok != 0)) return c.rbuf + (uint32_t)kStageBytes * slot;
  }
  if (c.lane == 0) atomicOr(c.a->err, DEV_ERR_TIMEOUT);
  return 0;
}

// Before leaving after an error: let every copy still in flight land.
__device__ void ring_drain(Ctx& c) {
  for (uint32_t n = c.tail; n != c.head; ++n) (void)ring_wait(c, n);
  c.tail = c.head;
}

// What a unit streams. kind 1: `bytes` contiguous bytes from p in stages of
// `chunk` (the last may be shorter); kind 2: stage i gathers group i of 4 row
// tiles (p + i * 544 + r * stride, r < 4); kind 0: nothing.
struct Src {
  const uint8_t* p;
  size_t stride;
  uint32_t bytes, chunk;
  int kind, nst;
};

__device__ __forceinline__ Src src_contig(const void* p, uint32_t bytes, uint32_t chunk) {
  return Src{reinterpret_cast<const uint8_t*>(p), 0, bytes, chunk, 1,
             (int)((bytes + chunk - 1) / chunk)};
}
__device__ __forceinline__ Src src_quad(const uint8_t* p, size_t stride, int ngroups) {
  return Src{p, stride, 0, 0, 2, ngroups};
}
__device__ __forceinline__ Src src_none() { return Src{nullptr, 0, 0, 0, 0, 0}; }

__device__ __forceinline__ void issue_src(Ctx& c, const Src& s, int i) {
  if (s.kind == 2)
    ring_issue4(c, s.p + (size_t)i * kGroupBytes, s.stride);
  else
    ring_issue(c, s.p + (size_t)i * s.chunk, min(s.chunk, s.bytes - (uint32_t)i * s.chunk));
}

// Source of unit u (defined with the units); 0 when it cannot be known yet
// (a routed unit before the routing is published) and !wait.
__device__ int unit_src(Ctx& c, int u, Src& s, bool wait);

// One step of prefetching the next unit: resolve it once, then issue one of
// its stages if the ring has room.
__device__ __forceinline__ void prefetch_step(Ctx& c) {
  if (c.nstate == 2) return;
  Src* ns = reinterpret_cast<Src*>(c.nsrc);
  if (c.nstate == 0) {
    const int un = (int)__shfl_sync(FULL, c.claim, 0);
    Src s;
    if (!unit_src(c, un, s, false)) return;  // retried at the next step
    if (c.lane == 0) *ns = s;
    __syncwarp();
    c.nstate = s.nst > 0 ? 1 : 2;
    c.nissued = 0;
    if (c.nstate == 2) return;
  }
  const Src s = *ns;
  if (c.nissued < s.nst && (int)(c.head - c.tail) < c.S) {
    issue_src(c, s, c.nissued);
    ++c.nissued;
  }
}

// Streams the stages of s through the ring; f(st, addr) is called for stage
// st with its shared address. The first c.pre stages may already be in the
// ring (prefetched). Once every stage of s is issued, freed slots go to the
// next unit's first stages. false: a wait timed out.
template <class F>
__device__ __forceinline__ bool run_stream(Ctx& c, const Src& s, F&& f, bool prefetch = true) {
  int issued = c.pre;
  c.pre = 0;
  while (issued < s.nst && (int)(c.head - c.tail) < c.S) issue_src(c, s, issued++);
#pragma unroll 1
  for (int st = 0; st < s.nst; ++st) {
    const uint32_t sa = ring_wait(c, c.tail);
    if (!sa) return false;
    f(st, sa);
    __syncwarp();
    ++c.tail;
    if (issued < s.nst) issue_src(c, s, issued++);
    else if (prefetch) prefetch_step(c);
  }
  return true;
}

// acc += 16 rows x 64 columns of MXFP4 (codes q, scales sc) times B. bA holds
// the B registers of k-steps 0 and 1, bB of k-steps 2 and 3.
template <int NCG>
__device__ __forceinline__ void mx_group(uint4 q, uint32_t sc, const uint4 (&bA)[NCG],
                                         const uint4 (&bB)[NCG], float (&acc)[NCG][4]) {
  const float s0 = e8m0_byte(sc, 0), s1 = e8m0_byte(sc, 1);   // row g
  const float u0 = e8m0_byte(sc, 2), u1 = e8m0_byte(sc, 3);   // row g+8
  uint32_t a0[4], a1[4], a2[4], a3[4];
  decode_word(q.x, a0);
  decode_word(q.y, a1);
  decode_word(q.z, a2);
  decode_word(q.w, a3);
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int cg = 0; cg < NCG; ++cg) {
    float d[4];
    mma16816(d, a0, bA[cg].x, bA[cg].y, zero);  // block 2G
    mma16816(d, a1, bA[cg].z, bA[cg].w, d);
    acc[cg][0] = fmaf(d[0], s0, acc[cg][0]);
    acc[cg][1] = fmaf(d[1], s0, acc[cg][1]);
    acc[cg][2] = fmaf(d[2], u0, acc[cg][2]);
    acc[cg][3] = fmaf(d[3], u0, acc[cg][3]);
    mma16816(d, a2, bB[cg].x, bB[cg].y, zero);  // block 2G+1
    mma16816(d, a3, bB[cg].z, bB[cg].w, d);
    acc[cg][0] = fmaf(d[0], s1, acc[cg][0]);
    acc[cg][1] = fmaf(d[1], s1, acc[cg][1]);
    acc[cg][2] = fmaf(d[2], u1, acc[cg][2]);
    acc[cg][3] = fmaf(d[3], u1, acc[cg][3]);
  }
}

// x as B fragments of group G (global group index) for token `tok` (zero
// for tok < 0).
__device__ __forceinline__ void x_frag(const Ctx& c, int G, int tok, uint4& bA, uint4& bB) {
  bA = make_uint4(0, 0, 0, 0);
  bB = make_uint4(0, 0, 0, 0);
  if (tok >= 0) {
    const uint32_t off = (uint32_t)((G * c.a->T + tok) * 4 + c.t4) * 16u;
    bA = lds128a(c.xa + off);
    bB = lds128a(c.xb + off);
  }
}

// Down input fragments of group G, column group cg, from hfd (global, L2).
__device__ __forceinline__ void h_frag(const Ctx& c, const uint4* hfd, int cg, int G,
                                       uint4& bA, uint4& bB) {
  const size_t o = ((size_t)(cg * c.a->hf_groups + G) * 2) * 32 + c.lane;
  bA = __ldcg(hfd + o);
  bB = __ldcg(hfd + o + 32);
}

// ---------------------------------------------------------------------------
// h -> down B fragments (the last gate/up tile of an expert).
// Column n of the down MMA (lane g = n) is token slot c = 4 cg + n/2 of the
// item, the high (n even) or low (n odd) f16 part of h * 2^-s(c); s(c) puts
// the slot's largest |h| just under 2^15.
// ---------------------------------------------------------------------------
__device__ __noinline__ void make_down_input(const Ctx c, int d, int K, int cnt, const float* rows0,
                                const int32_t* sorted_pos, int row_ld, uint32_t epoch) {
  const LayerKernelArgs& a = *c.a;
  float dnv = 1.f;
  if (c.lane < cnt) {
    uint32_t* hm = sw(a, a.sl.hmax) + (size_t)d * kLayerMaxT + c.lane;
    const float m = __uint_as_float(__ldcg(hm));
    int sh = 0;
    if (m > 0.f) {
      const int e = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;
      sh = min(max(e - 14, -100), 100);
    }
    a.hsc[(size_t)d * kLayerMaxT + c.lane] = pow2i(sh);
    dnv = pow2i(-sh);
    *hm = 0u;  // ready for the next call
  }
  const int NG = K >> 6;
  const int ncg = (cnt + 3) >> 2;
  const bool lo = (c.g & 1) != 0;
  for (int cg = 0; cg < ncg; ++cg) {
    const int slot = 4 * cg + (c.g >> 1);
    const float dn = __shfl_sync(FULL, dnv, slot & 31);
    const float* hrow = nullptr;
    if (slot < cnt)
      hrow = sorted_pos ? rows0 + (size_t)__ldcg(sorted_pos + slot) * row_ld
                        : rows0 + (size_t)slot * row_ld;
    uint4* out = a.hf + ((size_t)(d * 2 + cg) * a.hf_groups) * 2 * 32;
    for (int G0 = 0; G0 < NG; G0 += 4) {
      float2 p[4][8];
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        const int G = G0 + gg;
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // i = 2 ks + half
          p[gg][i] = make_float2(0.f, 0.f);
          if (hrow && G < NG)
            p[gg][i] = __ldcg(reinterpret_cast<const float2*>(
                hrow + 64 * G + 16 * (i >> 1) + 8 * (i & 1) + 2 * c.t4));
        }
      }
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        const int G = G0 + gg;
        if (G < NG) {
          uint32_t wv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float v0 = p[gg][i].x * dn, v1 = p[gg][i].y * dn;
            const __half2 hi = __floats2half2_rn(v0, v1);
            if (!lo) {
              wv[i] = *reinterpret_cast<const uint32_t*>(&hi);
            } else {
              const float2 f = __half22float2(hi);
              wv[i] = f2_to_h2(v0 - f.x, v1 - f.y);
            }
          }
          out[((size_t)G * 2 + 0) * 32 + c.lane] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          out[((size_t)G * 2 + 1) * 32 + c.lane] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
        }
      }
    }
  }
  raise_flag(sw(a, a.sl.f_hp) + d, epoch);
}

// Rows 64q..64q+63 of every token: residual + sum_i w_i (sum over the K
// parts of expert i's down GEMV) + shared experts, in fixed order.
// Row layout of `part`: routed expert i of token t, K part h: h*T*k + t*k + i;
// shared expert s, token t: ks_dn*T*k + s*T + t.
__device__ __noinline__ void combine_rows(const Ctx c, int qb) {
  const LayerKernelArgs& a = *c.a;
  const int H = a.H, k = a.k, T = a.T;
  const size_t Tk = (size_t)T * k;
  for (int t = 0; t < T; ++t) {
    float wv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) wv[i] = i < k ? __ldcg(a.w + (size_t)t * k + i) : 0.f;
    for (int half = 0; half < 2; ++half) {
      const int row = 64 * qb + 32 * half + c.lane;
      float p0[32], p1[32];  // every load of the row in flight at once
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        p0[i] = i < k ? __ldcg(a.part + ((size_t)t * k + i) * H + row) : 0.f;
        p1[i] = (i < k && a.ks_dn > 1) ? __ldcg(a.part + (Tk + (size_t)t * k + i) * H + row) : 0.f;
      }
      float y = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < k) y = fmaf(wv[i], a.ks_dn > 1 ? p0[i] + p1[i] : p0[i], y);
      for (int s = 0; s < a.n_shared; ++s)
        y += __ldcg(a.part + ((size_t)a.ks_dn * Tk + (size_t)s * T + t) * H + row);
      if (a.residual) y += __uint_as_float((uint32_t)a.residual[(size_t)t * H + row] << 16);
      if (a.out_f32) a.out_f32[(size_t)t * H + row] = y;
      if (a.out_bf16)
        a.out_bf16[(size_t)t * H + row] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
    }
  }
}

// A down unit wrote its rows of block qb (64 rows): the last of the
// n_items * ks_dn routed and 4 * n_shared shared writers combines the block.
__device__ void rows_done(const Ctx& c, int qb) {
  const LayerKernelArgs& a = *c.a;
  uint32_t* t = sw(a, a.sl.t_rows) + qb;
  const uint32_t old = take_ticket(t);
  if (old == (uint32_t)(c.n_items * a.ks_dn + 4 * a.n_shared) - 1u) {
    if (c.lane == 0) *t = 0u;
    combine_rows(c, qb);
  }
}

// Whether the routing (items, n_items) is published; with wait = false a
// single poll. With wait = true false means a timeout (recorded).
__device__ bool items_ready(Ctx& c, bool wait) {
  if (c.items_seen) return true;
  const LayerKernelArgs& a = *c.a;
  const uint32_t* f = sw(a, a.sl.f_items);
  if (wait) {
    if (!wait_flag(f, a.epoch, a.err)) return false;
  } else if (!__all_sync(FULL, ld_acquire(f) == a.epoch)) {
    return false;
  }
  c.n_items = __ldcg(a.n_items);
  c.items_seen = true;
  return true;
}

__device__ __forceinline__ bool ensure_items(Ctx& c) { return items_ready(c, true); }

__device__ __forceinline__ Item load_item(const LayerKernelArgs& a, int i) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(a.items + i));
  return Item{v.x, v.y, v.z, v.w};
}

// Largest |h| of token columns 2t4, 2t4+1 over the 8 rows of the tile, merged
// into the down item's per-slot maxima.
__device__ void note_hmax(const Ctx& c, int d, int cnt, float h0, float h1) {
  float m0 = fabsf(h0), m1 = fabsf(h1);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    m0 = fmaxf(m0, __shfl_xor_sync(FULL, m0, o));
    m1 = fmaxf(m1, __shfl_xor_sync(FULL, m1, o));
  }
  if (c.g == 0) {
    uint32_t* hm = sw(*c.a, c.a->sl.hmax) + (size_t)d * kLayerMaxT;
    if (2 * c.t4 < cnt) atomicMax(hm + 2 * c.t4, __float_as_uint(m0));
    if (2 * c.t4 + 1 < cnt) atomicMax(hm + 2 * c.t4 + 1, __float_as_uint(m1));
  }
}

// ---------------------------------------------------------------------------
// Unit sources. Each unit streams one Src; the same functions serve the unit
// itself and the prefetch of the next unit, so both see the same bytes.
// ---------------------------------------------------------------------------

__device__ __forceinline__ Src src_router(const LayerKernelArgs& a, int u) {
  const int e = u / a.ks_rt, q = u - e * a.ks_rt;
  const int n64 = a.H >> 6;
  const int c0 = (q * n64 / a.ks_rt) * 64, c1 = ((q + 1) * n64 / a.ks_rt) * 64;
  return c1 > c0 ? src_contig(a.Wr + (size_t)e * a.H + c0, (uint32_t)(c1 - c0) * 4u, 2048u)
                 : src_none();
}

__device__ __forceinline__ Src src_shared_gateup(const LayerKernelArgs& a, int u) {
  const int q = u % a.ks_sg, tj = u / a.ks_sg;
  const int NG = a.H >> 6;
  const int G0 = q * NG / a.ks_sg, G1 = (q + 1) * NG / a.ks_sg;
  return src_contig(a.sh_gu + ((size_t)tj * (a.H >> 4) + 4 * G0) * 32,
                    (uint32_t)(G1 - G0) * 2048u, 2048u);
}

__device__ __forceinline__ Src src_routed_gateup(const LayerKernelArgs& a, int u, int e) {
  const int quads = (a.I >> 3) >> 2;
  const int q = u % a.ks_gu, jq = (u / a.ks_gu) % quads;
  const int NG = a.H >> 6;
  const int G0 = q * NG / a.ks_gu, G1 = (q + 1) * NG / a.ks_gu;
  const size_t tb = mx_tile_bytes(a.H);
  return src_quad(a.arena + (size_t)e * a.span_bytes + (size_t)(4 * jq) * tb +
                      (size_t)G0 * kGroupBytes,
                  tb, G1 - G0);
}

__device__ __forceinline__ Src src_shared_down(const LayerKernelArgs& a, int u) {
  const int rows_t = a.H >> 4;
  const int j = u / a.n_shared, s = u - j * a.n_shared;
  const int NK = a.Is >> 4;
  return src_contig(a.sh_dn + ((size_t)s * rows_t + j) * NK * 32, (uint32_t)NK * 512u, 2048u);
}

__device__ __forceinline__ Src src_routed_down(const LayerKernelArgs& a, int u, int e) {
  const int per = (a.H >> 6) * a.ks_dn;
  const int rem = u % per;
  const int qb = rem / a.ks_dn, h = rem - qb * a.ks_dn;
  const int NG = a.I >> 6;
  const int G0 = h * NG / a.ks_dn, G1 = (h + 1) * NG / a.ks_dn;
  const size_t tb = mx_tile_bytes(a.I);
  const SpanLayout L = span_layout(a.H, a.I);
  return src_quad(a.arena + (size_t)e * a.span_bytes + L.dn + (size_t)(4 * qb) * tb +
                      (size_t)G0 * kGroupBytes,
                  tb, G1 - G0);
}

__device__ bool items_ready(Ctx& c, bool wait);
__device__ __forceinline__ Item load_item(const LayerKernelArgs& a, int i);

__device__ int unit_src(Ctx& c, int u, Src& s, bool wait) {
  const LayerKernelArgs& a = *c.a;
  const volatile int* b = c.ub;
  if (u >= b[5]) { s = src_none(); return 1; }
  if (u < b[0]) { s = src_router(a, u); return 1; }
  if (u < b[2]) { s = src_shared_gateup(a, u - b[1]); return 1; }
  if (u >= b[3] && u < b[4]) { s = src_shared_down(a, u - b[3]); return 1; }
  if (!items_ready(c, wait)) return 0;
  int i;
  if (u < b[3]) {
    const int quads = (a.I >> 3) >> 2;
    i = (u - b[2]) / a.ks_gu / quads;
  } else {
    i = (u - b[4]) / ((a.H >> 6) * a.ks_dn);
  }
  if (i >= c.n_items) { s = src_none(); return 1; }
  const Item it = load_item(a, i);
  s = u < b[3] ? src_routed_gateup(a, u - b[2], it.e) : src_routed_down(a, u - b[4], it.e);
  return 1;
}

// ---------------------------------------------------------------------------
// Units
// ---------------------------------------------------------------------------

__device__ __noinline__ void route_block(const Ctx c, int blk);

__device__ bool unit_router(Ctx& c, int u) {
  const LayerKernelArgs& a = *c.a;
  const int e = u / a.ks_rt, q = u - e * a.ks_rt;
  const int H = a.H, T = a.T;
  const int n64 = H >> 6;  // slice bounds on 64-column steps (16-byte aligned)
  const int c0 = (q * n64 / a.ks_rt) * 64, c1 = ((q + 1) * n64 / a.ks_rt) * 64;
  float acc[kLayerMaxT];
#pragma unroll
  for (int t = 0; t < kLayerMaxT; ++t) acc[t] = 0.f;
  if (c1 > c0) {
    const bool ok = run_stream(
        c, src_router(a, u), [&](int st, uint32_t sa) {
          const int col0 = c0 + 512 * st;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int f = c.lane + 32 * j;  // float4 index within the chunk
            if (col0 + 4 * f < c1) {
              const uint4 wv = lds128a(sa + 16u * f);
#pragma unroll
              for (int t = 0; t < kLayerMaxT; ++t) {
                if (t < T) {
                  uint2 xv;
                  if (c.xr) {
                    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                                 : "=r"(xv.x), "=r"(xv.y)
                                 : "r"(c.xr + 2u * (uint32_t)(t * H + col0 + 4 * f)));
                  } else {
                    xv = *reinterpret_cast<const uint2*>(a.x + (size_t)t * H + col0 + 4 * f);
                  }
                  acc[t] = fmaf(__uint_as_float(wv.x), bf16_lo(xv.x), acc[t]);
                  acc[t] = fmaf(__uint_as_float(wv.y), bf16_hi(xv.x), acc[t]);
                  acc[t] = fmaf(__uint_as_float(wv.z), bf16_lo(xv.y), acc[t]);
                  acc[t] = fmaf(__uint_as_float(wv.w), bf16_hi(xv.y), acc[t]);
                }
              }
            }
          }
        });
    if (!ok) return false;
  }
#pragma unroll
  for (int t = 0; t < kLayerMaxT; ++t) {
    if (t < T) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
      if (c.lane == 0) a.logit_part[((size_t)q * T + t) * a.E + e] = v;
    }
  }
  // the last unit of the expert's block of 32 selects the block's best
  const int blk = e / kRouterBlock;
  const int nb_e = min(kRouterBlock, a.E - blk * kRouterBlock);
  uint32_t* tb = sw(a, a.sl.t_rtb) + blk;
  if (take_ticket(tb) == (uint32_t)(nb_e * a.ks_rt) - 1u) {
    if (c.lane == 0) *tb = 0u;
    route_block(c, blk);
  }
  return true;
}

// Groups the T*k assignments (a = t*k + i) by expert: items in ascending
// expert id, assignments of an item in ascending a. One warp, n <= 256.
__device__ __noinline__ void group_items(const Ctx c) {
  const LayerKernelArgs& a = *c.a;
  const int n = a.T * a.k;
  const int nm = (n + 31) >> 5;
  int ea[8], rank[8], cnt[8], itm[8];
  bool first[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int x = c.lane + 32 * m;
    ea[m] = (m < nm && x < n) ? __ldcg(a.ids + x) : 0x7fffffff;
    rank[m] = 0;
    cnt[m] = 0;
    itm[m] = 0;
    first[m] = true;
  }
#pragma unroll
  for (int mb = 0; mb < 8; ++mb) {
    if (mb < nm) {
      for (int bl = 0; bl < 32; ++bl) {
        const int b = 32 * mb + bl;
        if (b >= n) break;
        const int eb = __shfl_sync(FULL, ea[mb], bl);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int x = c.lane + 32 * m;
          if (eb < ea[m] || (eb == ea[m] && b < x)) ++rank[m];
          if (eb == ea[m]) {
            ++cnt[m];
            if (b < x) first[m] = false;
          }
        }
      }
    }
  }
  int nfirst = 0;
#pragma unroll
  for (int mb = 0; mb < 8; ++mb) {
    if (mb < nm) {
      for (int bl = 0; bl < 32; ++bl) {
        const int b = 32 * mb + bl;
        if (b >= n) break;
        const int eb = __shfl_sync(FULL, ea[mb], bl);
        const bool fb = __shfl_sync(FULL, (int)first[mb], bl) != 0;
        if (fb) {
          ++nfirst;
#pragma unroll
          for (int m = 0; m < 8; ++m)
            if (eb < ea[m]) ++itm[m];
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int x = c.lane + 32 * m;
    if (m < nm && x < n) {
      a.sorted[rank[m]] = x;
      if (first[m]) a.items[itm[m]] = Item{ea[m], rank[m], cnt[m], 0};
    }
  }
  if (c.lane == 0) *a.n_items = nfirst;
}

// Routing, in two steps. The last router unit of each block of 32 experts
// sums the block's logits (its K slices in slice order) and sorts them, best
// first (higher logit, then lower id), with a bitonic network across the
// lanes; the block's top min(k, 32) go to `cand`. The last block merges the
// sorted lists of all blocks (one per lane, read from this warp's idle ring
// buffer), so the selection equals a full sort of the logits. Weights are a
// softmax over the k selected logits.

// Bitonic sort of one (value, id) per lane across the warp: lane 0 ends with
// the best.
__device__ __forceinline__ void warp_sort_desc(float& v, int& e) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float ov = __shfl_xor_sync(FULL, v, stride);
      const int oe = __shfl_xor_sync(FULL, e, stride);
      const bool want_better = ((lane & stride) == 0) == ((lane & size) == 0 || size == 32);
      const bool other_better = better(ov, oe, v, e);
      if (want_better == other_better && (ov != v || oe != e)) {
        v = ov;
        e = oe;
      }
    }
  }
}

__device__ __noinline__ void route_final(const Ctx c);

__device__ __noinline__ void route_block(const Ctx c, int blk) {
  const LayerKernelArgs& a = *c.a;
  const int E = a.E, T = a.T;
  const int e = blk * kRouterBlock + c.lane;
  const int nblk = (E + kRouterBlock - 1) / kRouterBlock;
  for (int t = 0; t < T; ++t) {
    float p[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      p[q] = (e < E && q < a.ks_rt) ? __ldcg(a.logit_part + ((size_t)q * T + t) * E + e) : 0.f;
    float v = -INFINITY;
    int id = 0x7fffffff;
    if (e < E) {
      v = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < a.ks_rt) v += p[q];
      id = e;
    }
    warp_sort_desc(v, id);
    if (c.lane < a.k) a.cand[((size_t)t * nblk + blk) * kRouterBlock + c.lane] =
        make_float2(v, __int_as_float(id));
  }
  uint32_t* tk = sw(a, a.sl.t_rt);
  if (take_ticket(tk) == (uint32_t)nblk - 1u) {
    if (c.lane == 0) *tk = 0u;
    route_final(c);
  }
}

__device__ __noinline__ void route_final(const Ctx c) {
  const LayerKernelArgs& a = *c.a;
  const int E = a.E, k = a.k, T = a.T;
  const int nblk = (E + kRouterBlock - 1) / kRouterBlock;
  const int mine = c.lane < nblk ? min(k, min(kRouterBlock, E - c.lane * kRouterBlock)) : 0;
  // lane b's sorted list in shared memory (this warp's ring buffer is idle;
  // layer_kernel_supports checks that 32 lists of k entries fit)
  const uint32_t lst = c.rbuf + (uint32_t)(c.lane * k) * 8u;
  for (int t = 0; t < T; ++t) {
    for (int r0 = 0; r0 < mine; r0 += 16) {
      float2 cv[16];  // loads in flight before the stores
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (r0 + r < mine) cv[r] = __ldcg(a.cand + ((size_t)t * nblk + c.lane) * kRouterBlock + r0 + r);
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (r0 + r < mine)
          asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(lst + 8u * (r0 + r)),
                       "f"(cv[r].x), "f"(cv[r].y)
                       : "memory");
    }
    __syncwarp();
    int head = 0;
    float hv = -INFINITY;
    int he = 0x7fffffff;
    auto load_head = [&]() {
      hv = -INFINITY;
      he = 0x7fffffff;
      if (head < mine) {
        float x, y;
        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(x), "=f"(y) : "r"(lst + 8u * head));
        hv = x;
        he = __float_as_int(y);
      }
    };
    load_head();
    float sel_v = -INFINITY;
    int sel_e = 0x7fffffff;
    for (int r = 0; r < k; ++r) {
      // best head: largest logit (as an order-preserving integer key), then
      // the lowest id among equal logits
      const uint32_t key = order_key(hv);
      const uint32_t kmax = __reduce_max_sync(FULL, key);
      const int be = (int)__reduce_min_sync(FULL, key == kmax ? (uint32_t)he : 0x7fffffffu);
      const float bv = __shfl_sync(FULL, hv, __ffs(__ballot_sync(FULL, key == kmax && he == be)) - 1);
      if (c.lane == r) {
        sel_v = bv;
        sel_e = be;
      }
      if (be == he) {  // this lane's head was taken (ids are unique)
        ++head;
        load_head();
      }
    }
    __syncwarp();
    // softmax over the selected logits (the largest is rank 0)
    const float vmax = __shfl_sync(FULL, sel_v, 0);
    const float ex = c.lane < k ? expf(sel_v - vmax) : 0.f;
    float z = ex;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) z += __shfl_xor_sync(FULL, z, o);
    if (c.lane < k) {
      a.ids[(size_t)t * k + c.lane] = sel_e;
      a.w[(size_t)t * k + c.lane] = ex / z;
      if (T == 1) {
        a.items[c.lane] = Item{sel_e, c.lane, 1, 0};
        a.sorted[c.lane] = c.lane;
      }
    }
  }
  if (T == 1) {
    if (c.lane == 0) *a.n_items = k;
  } else {
    __syncwarp();
    group_items(c);
  }
  raise_flag(sw(a, a.sl.f_items), a.epoch);
}

// Last K slice of shared gate/up tile j of shared expert s: sums the slices'
// partials in slice order, applies the row scales and SwiGLU, writes h; the
// expert's last finished tile converts its h for the down GEMV.
__device__ __noinline__ void finish_sg_tile(const Ctx c, const float4* P, int q, float4 own,
                                            int s, int j) {
  const LayerKernelArgs& a = *c.a;
  const int T = a.T, tiles = a.Is >> 3;
  const int tj = s * tiles + j;
  float4 pv[kMaxSlices];
#pragma unroll
  for (int qq = 0; qq < kMaxSlices; ++qq)
    if (qq < a.ks_sg && qq != q) pv[qq] = __ldcg(P + (size_t)qq * 32 + c.lane);
  float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int qq = 0; qq < kMaxSlices; ++qq) {
    if (qq < a.ks_sg) {
      const float4 v = qq == q ? own : pv[qq];
      sum.x += v.x;
      sum.y += v.y;
      sum.z += v.z;
      sum.w += v.w;
    }
  }
  const float rg = a.sh_gu_rs[(size_t)tj * 16 + c.g];
  const float ru = a.sh_gu_rs[(size_t)tj * 16 + c.g + 8];
  const int c0 = 2 * c.t4, c1 = c0 + 1;
  float h0 = 0.f, h1 = 0.f;
  if (c0 < T) {
    h0 = silu_f(sum.x * rg) * (sum.z * ru);
    a.hsh32[((size_t)s * T + c0) * a.Is + 8 * j + c.g] = h0;
  }
  if (c1 < T) {
    h1 = silu_f(sum.y * rg) * (sum.w * ru);
    a.hsh32[((size_t)s * T + c1) * a.Is + 8 * j + c.g] = h1;
  }
  const int d = a.max_items + s;
  note_hmax(c, d, T, h0, h1);
  uint32_t* ti = sw(a, a.sl.t_item) + d;
  if (take_ticket(ti) == (uint32_t)tiles - 1u) {
    if (c.lane == 0) *ti = 0u;
    make_down_input(c, d, a.Is, T, a.hsh32 + (size_t)s * T * a.Is, nullptr, a.Is, a.epoch);
  }
}

__device__ bool unit_shared_gateup(Ctx& c, int u) {
  const LayerKernelArgs& a = *c.a;
  const int tiles = a.Is >> 3;
  const int q = u % a.ks_sg, tj = u / a.ks_sg;  // tj = s * tiles + j
  const int s = tj / tiles, j = tj - s * tiles;
  const int H = a.H, T = a.T, NG = H >> 6;
  const int G0 = q * NG / a.ks_sg;
  const int tok = c.g < T ? c.g : -1;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  // one chunk = the 4 k-steps of one group
  const bool ok = run_stream(c, src_shared_gateup(a, u), [&](int st, uint32_t sa) {
                           uint4 bA, bB;
                           x_frag(c, G0 + st, tok, bA, bB);
                           const uint32_t b[8] = {bA.x, bA.y, bA.z, bA.w,
                                                  bB.x, bB.y, bB.z, bB.w};
#pragma unroll
                           for (int kk = 0; kk < 4; ++kk) {
                             const uint4 q4 = lds128a(sa + 512u * kk + 16u * c.lane);
                             const uint32_t af[4] = {q4.x, q4.y, q4.z, q4.w};
                             mma16816(acc, af, b[2 * kk], b[2 * kk + 1], acc);
                           }
                         });
  if (!ok) return false;
  float4* P = a.sg_part + (size_t)tj * a.ks_sg * 32;
  __stcg(P + (size_t)q * 32 + c.lane, make_float4(acc[0], acc[1], acc[2], acc[3]));
  uint32_t* tk = sw(a, a.sl.t_sg) + tj;
  if (take_ticket(tk) != (uint32_t)a.ks_sg - 1u) return true;
  if (c.lane == 0) *tk = 0u;
  finish_sg_tile(c, P, q, make_float4(acc[0], acc[1], acc[2], acc[3]), s, j);
  return true;
}


// Last K slice of gate/up tile j of item i: sums the slices' partials in
// slice order (its own from registers), applies SwiGLU, writes h and notes
// the per-token maxima.
__device__ __noinline__ void finish_gu_tile(const Ctx c, const float4* P, int q, float4 own,
                                            int i, const Item it, int j) {
  const LayerKernelArgs& a = *c.a;
  float4 pv[kMaxSlices];
#pragma unroll
  for (int qq = 0; qq < kMaxSlices; ++qq)
    if (qq < a.ks_gu && qq != q) pv[qq] = __ldcg(P + (size_t)qq * 32 + c.lane);
  float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int qq = 0; qq < kMaxSlices; ++qq) {
    if (qq < a.ks_gu) {
      const float4 v = qq == q ? own : pv[qq];
      sum.x += v.x;
      sum.y += v.y;
      sum.z += v.z;
      sum.w += v.w;
    }
  }
  const int c0 = 2 * c.t4, c1 = c0 + 1;
  float h0 = 0.f, h1 = 0.f;
  if (c0 < it.cnt) {
    h0 = silu_f(sum.x) * sum.z;
    a.h32[(size_t)__ldcg(a.sorted + it.pos + c0) * a.I + 8 * j + c.g] = h0;
  }
  if (c1 < it.cnt) {
    h1 = silu_f(sum.y) * sum.w;
    a.h32[(size_t)__ldcg(a.sorted + it.pos + c1) * a.I + 8 * j + c.g] = h1;
  }
  note_hmax(c, i, it.cnt, h0, h1);
}

// Routed gate/up: 4 row tiles (tile quad jq of item i) x K slice q. Each
// group's B (x) is loaded once for the 4 tiles. A tile's K slices are summed,
// in slice order, by the slice that finishes last, which then applies SwiGLU;
// the expert's last finished tile converts its h for the down GEMV.
__device__ bool unit_routed_gateup(Ctx& c, int u) {
  const LayerKernelArgs& a = *c.a;
  if (!ensure_items(c)) return false;
  const int tiles = a.I >> 3, quads = tiles >> 2;
  const int q = u % a.ks_gu, iq = u / a.ks_gu;  // iq = i * quads + jq
  const int i = iq / quads, jq = iq - i * quads;
  if (i >= c.n_items) return true;
  const Item it = load_item(a, i);
  const int H = a.H, NG = H >> 6;
  const int G0 = q * NG / a.ks_gu, G1 = (q + 1) * NG / a.ks_gu;
  const size_t tb = mx_tile_bytes(H);
  const uint8_t* base = a.arena + (size_t)it.e * a.span_bytes + (size_t)(4 * jq) * tb;
  const int tok = c.g < it.cnt ? __ldcg(a.sorted + it.pos + c.g) / a.k : -1;
  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int v = 0; v < 4; ++v) acc[r][v] = 0.f;
  const bool ok = run_stream(c, src_quad(base + (size_t)G0 * kGroupBytes, tb, G1 - G0),
                             [&](int st, uint32_t sa) {
    const int G = G0 + st;
    uint4 bA[1], bB[1];
    x_frag(c, G, tok, bA[0], bB[0]);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t ga = sa + (uint32_t)(kGroupBytes * r);
      const uint4 q4 = lds128a(ga + 16u * c.lane);
      const uint32_t sc = lds32a(ga + 512u + 4u * c.g);
      float ar[1][4] = {{acc[r][0], acc[r][1], acc[r][2], acc[r][3]}};
      mx_group<1>(q4, sc, bA, bB, ar);
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[r][v] = ar[0][v];
    }
  });
  if (!ok) return false;
  // K-slice partials of the 4 tiles; lanes 0..3 take the 4 tickets at once
  const int tj0 = i * tiles + 4 * jq;
  float4* P = a.gu_part + (size_t)tj0 * a.ks_gu * 32;
#pragma unroll
  for (int r = 0; r < 4; ++r)
    __stcg(P + ((size_t)r * a.ks_gu + q) * 32 + c.lane,
           make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]));
  __syncwarp();
  uint32_t old = 0;
  if (c.lane < 4)
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(sw(a, a.sl.t_gu) + tj0 + c.lane)
                 : "memory");
  const unsigned last = __ballot_sync(FULL, c.lane < 4 && old == (uint32_t)a.ks_gu - 1u) & 0xFu;
  if (!last) return true;
  if (c.lane < 4 && ((last >> c.lane) & 1u)) sw(a, a.sl.t_gu)[tj0 + c.lane] = 0u;
  __syncwarp();
  int n_done = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    if ((last >> r) & 1u) {
      ++n_done;
      finish_gu_tile(c, P + (size_t)r * a.ks_gu * 32, q,
                     make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]), i, it,
                     4 * jq + r);
    }
  }
  // tiles of this expert finished here: the last one converts its h
  __syncwarp();
  uint32_t* ti = sw(a, a.sl.t_item) + i;
  uint32_t prev = 0;
  if (c.lane == 0)
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(prev)
                 : "l"(ti), "r"((uint32_t)n_done)
                 : "memory");
  prev = __shfl_sync(FULL, prev, 0);
  __syncwarp();
  if (prev + (uint32_t)n_done == (uint32_t)tiles) {
    if (c.lane == 0) *ti = 0u;
    make_down_input(c, i, a.I, it.cnt, a.h32, a.sorted + it.pos, a.I, a.epoch);
  }
  return true;
}

// Writes rows g and g+8 of down tile j for the token slots of column group cg
// (K part `half` of a routed expert, or a shared expert when sorted_pos is
// null: part row shared_base + slot).
__device__ __forceinline__ void store_down(const Ctx& c, int d, int cg, int cnt, int j,
                                           const float (&acc)[4], float rs0, float rs1,
                                           const int32_t* sorted_pos, size_t shared_base,
                                           int half) {
  const LayerKernelArgs& a = *c.a;
  const int slot = 4 * cg + c.t4;
  if (slot >= cnt) return;
  const float sc = __ldcg(a.hsc + (size_t)d * kLayerMaxT + slot);
  const size_t row = sorted_pos ? (size_t)half * a.T * a.k + (size_t)__ldcg(sorted_pos + slot)
                                : shared_base + slot;
  float* p = a.part + row * a.H + 16 * j + c.g;
  p[0] = (acc[0] + acc[1]) * sc * rs0;
  p[8] = (acc[2] + acc[3]) * sc * rs1;
}

// Down GEMVs. B (the item's h fragments, in L2) is prefetched one chunk of
// 4 groups ahead in a register ring indexed by the group's position in the
// chunk.

// MXFP4 down: 4 row tiles x groups [G0, G1); B for group G+D is requested
// while group G is computed.
template <int NCG>
__device__ bool down_mx4(Ctx& c, const uint8_t* base, size_t stride, int G0, int G1,
                         const uint4* hfd, float (&acc)[4][NCG][4], bool prefetch = true) {
  constexpr int D = 2;  // groups of B requested ahead
  uint4 rbA[D][NCG], rbB[D][NCG];
#pragma unroll
  for (int d = 0; d < D; ++d)
#pragma unroll
    for (int cg = 0; cg < NCG; ++cg)
      if (G0 + d < G1) h_frag(c, hfd, cg, G0 + d, rbA[d][cg], rbB[d][cg]);
  // ring slot of group G is (G - G0) % D; rotate the registers instead of
  // indexing them with a run-time slot
  return run_stream(c, src_quad(base + (size_t)G0 * kGroupBytes, stride, G1 - G0),
                    [&](int st, uint32_t sa) {
    const int G = G0 + st;
    uint4 bA[NCG], bB[NCG];
#pragma unroll
    for (int cg = 0; cg < NCG; ++cg) {
      bA[cg] = rbA[0][cg];
      bB[cg] = rbB[0][cg];
#pragma unroll
      for (int d = 0; d + 1 < D; ++d) {
        rbA[d][cg] = rbA[d + 1][cg];
        rbB[d][cg] = rbB[d + 1][cg];
      }
      if (G + D < G1) h_frag(c, hfd, cg, G + D, rbA[D - 1][cg], rbB[D - 1][cg]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t ga = sa + (uint32_t)(kGroupBytes * r);
      const uint4 q4 = lds128a(ga + 16u * c.lane);
      const uint32_t sc = lds32a(ga + 512u + 4u * c.g);
      mx_group<NCG>(q4, sc, bA, bB, acc[r]);
    }
  }, prefetch);
}

// f16 tile of NK k-steps (NK % 4 == 0); chunk st = group st, whose B was
// loaded one chunk earlier.
template <int NCG>
__device__ bool down_f16(Ctx& c, const uint4* A, int NK, const uint4* hfd,
                         float (&acc)[NCG][4]) {
  const int NG = NK >> 2;
  uint4 nA[NCG], nB[NCG];
#pragma unroll
  for (int cg = 0; cg < NCG; ++cg) h_frag(c, hfd, cg, 0, nA[cg], nB[cg]);
  return run_stream(c, src_contig(A, (uint32_t)NK * 512u, 2048u),
                [&](int st, uint32_t sa) {
                  uint32_t b[NCG][8];
#pragma unroll
                  for (int cg = 0; cg < NCG; ++cg) {
                    b[cg][0] = nA[cg].x; b[cg][1] = nA[cg].y; b[cg][2] = nA[cg].z; b[cg][3] = nA[cg].w;
                    b[cg][4] = nB[cg].x; b[cg][5] = nB[cg].y; b[cg][6] = nB[cg].z; b[cg][7] = nB[cg].w;
                    if (st + 1 < NG) h_frag(c, hfd, cg, st + 1, nA[cg], nB[cg]);
                  }
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk) {
                    const uint4 q4 = lds128a(sa + 512u * kk + 16u * c.lane);
                    const uint32_t af[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                    for (int cg = 0; cg < NCG; ++cg)
                      mma16816(acc[cg], af, b[cg][2 * kk], b[cg][2 * kk + 1], acc[cg]);
                  }
                });
}

__device__ bool unit_shared_down(Ctx& c, int u) {
  const LayerKernelArgs& a = *c.a;
  if (!ensure_items(c)) return false;
  const int rows_t = a.H >> 4;
  const int j = u / a.n_shared, s = u - j * a.n_shared;
  const int d = a.max_items + s;
  if (!wait_flag(sw(a, a.sl.f_hp) + d, a.epoch, a.err)) return false;
  const int NK = a.Is >> 4;
  const uint4* A = a.sh_dn + ((size_t)s * rows_t + j) * NK * 32;
  const uint4* hfd = a.hf + (size_t)d * 2 * a.hf_groups * 2 * 32;
  const float rs0 = a.sh_dn_rs[(size_t)s * a.H + 16 * j + c.g];
  const float rs1 = a.sh_dn_rs[(size_t)s * a.H + 16 * j + c.g + 8];
  const size_t base = (size_t)a.ks_dn * a.T * a.k + (size_t)s * a.T;
  if (a.T <= 4) {
    float acc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
    if (!down_f16<1>(c, A, NK, hfd, acc)) return false;
    store_down(c, d, 0, a.T, j, acc[0], rs0, rs1, nullptr, base, 0);
  } else {
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (!down_f16<2>(c, A, NK, hfd, acc)) return false;
    store_down(c, d, 0, a.T, j, acc[0], rs0, rs1, nullptr, base, 0);
    store_down(c, d, 1, a.T, j, acc[1], rs0, rs1, nullptr, base, 0);
  }
  rows_done(c, j >> 2);
  return true;
}

// Items with 5..8 tokens (two column groups; only for T > 4), kept out of
// line so that their registers do not weigh on the common path.
// Works on a copy of the warp's context and returns the ring position it
// reached (tail; head equals tail after a completed stream), or ~0u after a
// timeout.
__device__ __noinline__ uint32_t routed_down_wide(Ctx c, const uint8_t* base, size_t tb, int G0,
                                                  int G1, const uint4* hfd, int i, const Item it,
                                                  int qb, int h) {
  float acc[4][2][4] = {};
  if (!down_mx4<2>(c, base, tb, G0, G1, hfd, acc, false)) {
    ring_drain(c);
    return ~0u;
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    store_down(c, i, 0, it.cnt, 4 * qb + r, acc[r][0], 1.f, 1.f, c.a->sorted + it.pos, 0, h);
    store_down(c, i, 1, it.cnt, 4 * qb + r, acc[r][1], 1.f, 1.f, c.a->sorted + it.pos, 0, h);
  }
  return c.tail;
}

// Routed down: row block qb (4 row tiles) of item i, K part h.
__device__ bool unit_routed_down(Ctx& c, int u) {
  const LayerKernelArgs& a = *c.a;
  if (!ensure_items(c)) return false;
  // expert-major: an expert's down units follow its gate/up units, whose
  // last tile converts h just before
  const int per = (a.H >> 6) * a.ks_dn;
  const int i = u / per, rem = u - i * per;
  const int qb = rem / a.ks_dn, h = rem - qb * a.ks_dn;
  if (i >= c.n_items) return true;
  if (!wait_flag(sw(a, a.sl.f_hp) + i, a.epoch, a.err)) return false;
  const Item it = load_item(a, i);
  const SpanLayout L = span_layout(a.H, a.I);
  const size_t tb = mx_tile_bytes(a.I);
  const uint8_t* base = a.arena + (size_t)it.e * a.span_bytes + L.dn + (size_t)(4 * qb) * tb;
  const uint4* hfd = a.hf + (size_t)i * 2 * a.hf_groups * 2 * 32;
  const int NG = a.I >> 6;
  const int G0 = h * NG / a.ks_dn, G1 = (h + 1) * NG / a.ks_dn;
  if (it.cnt <= 4) {
    float acc[4][1][4] = {};
    if (!down_mx4<1>(c, base, tb, G0, G1, hfd, acc)) return false;
#pragma unroll
    for (int r = 0; r < 4; ++r)
      store_down(c, i, 0, it.cnt, 4 * qb + r, acc[r][0], 1.f, 1.f, a.sorted + it.pos, 0, h);
  } else {
    const uint32_t pos = routed_down_wide(c, base, tb, G0, G1, hfd, i, it, qb, h);
    if (pos == ~0u) return false;  // its copies were drained
    c.head = c.tail = pos;
  }
  rows_done(c, qb);
  return true;
}

// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kThreads, 1) layer_kernel(const __grid_constant__ LayerKernelArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.H, T = a.T, NG = H >> 6;
  const int S = layer_stages(H, T);
  uint4* xfA = reinterpret_cast<uint4*>(smem);
  uint4* xfB = xfA + (size_t)NG * T * 4;
  uint8_t* xr = smem + layer_xf_bytes(H, T);  // bf16 x for the router (if it fits)
  const bool have_xr = layer_xr_bytes(H, T) != 0;
  uint8_t* rings = xr + layer_xr_bytes(H, T);
  uint64_t* bars = reinterpret_cast<uint64_t*>(rings + (size_t)kWarps * S * kStageBytes);
  const int warp = threadIdx.x >> 5;

  // x as f16 B fragments: entry (G, tok, t4) of xfA holds, for k-steps 0 and
  // 1 of group G, {b0, b1} = x[tok] at columns (64G + 16s + 2t4, +1) and
  // (64G + 16s + 8 + 2t4, +1); xfB the same for k-steps 2 and 3.
  const int nent = NG * T * 4;
  for (int idx = threadIdx.x; idx < 2 * nent; idx += blockDim.x) {
    const int half = idx >= nent ? 1 : 0;
    const int e = idx - half * nent;
    const int t4 = e & 3, tok = (e >> 2) % T, G = (e >> 2) / T;
    const uint16_t* xr = a.x + (size_t)tok * H + 64 * G + 32 * half + 2 * t4;
    uint32_t wv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // i = 2 (k-step within half) + (b0/b1)
      const uint32_t p = *reinterpret_cast<const uint32_t*>(xr + 16 * (i >> 1) + 8 * (i & 1));
      wv[i] = f2_to_h2(bf16_lo(p), bf16_hi(p));
    }
    (half ? xfB : xfA)[e] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
  if (have_xr)
    for (int idx = threadIdx.x; idx < T * H / 8; idx += blockDim.x)
      reinterpret_cast<uint4*>(xr)[idx] = reinterpret_cast<const uint4*>(a.x)[idx];
  __shared__ int unit_bounds[6];
  __shared__ Src next_src[kWarps];
  if (threadIdx.x == 0) {
    const int tiles_r = a.I >> 3, tiles_s = a.Is >> 3, rows_t = H >> 4;
    unit_bounds[0] = a.E * a.ks_rt;
    unit_bounds[1] = unit_bounds[0];  // (no separate top-k units)
    unit_bounds[2] = unit_bounds[1] + a.n_shared * tiles_s * a.ks_sg;
    unit_bounds[3] = unit_bounds[2] + a.max_items * (tiles_r / 4) * a.ks_gu;
    unit_bounds[4] = unit_bounds[3] + a.n_shared * rows_t;
    unit_bounds[5] = unit_bounds[4] + (rows_t / 4) * a.max_items * a.ks_dn;
  }
  if ((threadIdx.x & 31) == 0)
    for (int i = 0; i < S; ++i) mbar_init(&bars[warp * S + i], 1);
  fence_barrier_init();
  __syncthreads();

  Ctx c;
  c.a = &a;
  c.xa = smem_u32(xfA);
  c.xb = smem_u32(xfB);
  c.xr = have_xr ? smem_u32(xr) : 0u;
  c.lane = threadIdx.x & 31;
  c.g = c.lane >> 2;
  c.t4 = c.lane & 3;
  c.items_seen = false;
  c.n_items = 0;
  c.rbuf = smem_u32(rings + (size_t)warp * S * kStageBytes);
  c.rbar = smem_u32(&bars[warp * S]);
  c.S = S;
  c.head = 0;
  c.tail = 0;
  c.claim = 0;
  c.nstate = 2;
  c.nissued = 0;
  c.pre = 0;
  c.ub = unit_bounds;
  c.nsrc = &next_src[warp];

  uint32_t* queue = sw(a, a.sl.queue);
  // unit ranges of the queue: [0, b[0]) router, then shared gate/up
  // [b[1], b[2]), routed gate/up, shared down, routed down (b[5] = total).
  // Read from shared memory on every dispatch so they hold no registers
  // across the units.
  const volatile int* b = unit_bounds;
  // Units are claimed one at a time: a claim made ahead would hold a unit
  // whose inputs may be far from ready while the queue moves on.
  bool ok = true;
  if (c.lane == 0) c.claim = atomicAdd(queue, 1u);
  int u = (int)__shfl_sync(FULL, c.claim, 0);
  c.pre = 0;
  for (;;) {
    if (u >= b[5]) break;
    // Units are claimed one at a time. (A unit claimed ahead, to prefetch its
    // weights, pulls later units out of the queue early; measured, the waits
    // this causes on the hand-off chains cost more than the prefetch gains.)
    const bool ahead = false;
    if (ahead && c.lane == 0) c.claim = atomicAdd(queue, 1u);
    c.nstate = ahead ? 0 : 2;
    c.nissued = 0;
    if (u < b[0]) ok = unit_router(c, u);
    else if (u < b[2]) ok = unit_shared_gateup(c, u - b[1]);
    else if (u < b[3]) ok = unit_routed_gateup(c, u - b[2]);
    else if (u < b[4]) ok = unit_shared_down(c, u - b[3]);
    else ok = unit_routed_down(c, u - b[4]);
    if (!ok) break;
    if (!ahead && c.lane == 0) c.claim = atomicAdd(queue, 1u);
    u = (int)__shfl_sync(FULL, c.claim, 0);
    c.pre = c.nstate == 1 ? c.nissued : 0;
  }
  if (!ok) {  // error recorded; the host resets the sync block
    ring_drain(c);
    return;
  }
  // The last warp out resets the queue for the next call.
  if (c.lane == 0) {
    uint32_t* ex = sw(a, a.sl.exit);
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(ex) : "memory");
    if (old == gridDim.x * (blockDim.x >> 5) - 1u) {
      *queue = 0u;
      *ex = 0u;
    }
  }
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

}  // namespace

bool layer_kernel_supports(int H, int T, int k, int E) {
  const int S = layer_stages(H, T);
  const int nblk = (E + kRouterBlock - 1) / kRouterBlock;
  return T >= 1 && T <= kLayerMaxT && S >= 2 && nblk <= 32 &&
         (size_t)nblk * k * 8 <= (size_t)S * kStageBytes;
}

size_t layer_kernel_smem(int H, int T) {
  return layer_xf_bytes(H, T) + layer_xr_bytes(H, T) + (size_t)layer_stages(H, T) * kRingPerStage;
}

int layer_kernel_grid() {
  static int grid = -1;
  if (grid < 0) {
    if (cudaFuncSetAttribute(layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemLimit) != cudaSuccess) {
      cudaGetLastError();
      grid = 0;
      return grid;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, layer_kernel, kThreads,
                                                      kSmemLimit) != cudaSuccess) {
      cudaGetLastError();
      per_sm = 0;
    }
    grid = per_sm > 0 ? per_sm * sm_count() : 0;
  }
  return grid;
}

cudaError_t launch_layer(const LayerKernelArgs& a, cudaStream_t s) {
  const int grid = layer_kernel_grid();
  if (grid <= 0) return cudaErrorCooperativeLaunchTooLarge;
  if (layer_stages(a.H, a.T) < 2) return cudaErrorInvalidValue;
  void* args[] = {const_cast<LayerKernelArgs*>(&a)};
  return cudaLaunchCooperativeKernel((const void*)layer_kernel, dim3(grid), dim3(kThreads),
                                     args, layer_kernel_smem(a.H, a.T), s);
}

}  // namespace dfm
