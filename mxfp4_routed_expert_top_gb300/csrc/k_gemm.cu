// k_gemm.cu — the routed experts of a large batch (prefill) as grouped,
// block-scaled MXFP4 GEMMs on the 5th-generation tensor cores.
//
// The same layer step as the decode GEMVs: the Deltafin README's fused
// MXFP4 dequant + matmul ("Techniques / Compute": E2M1 weights with an E8M0
// scale per 32, decoded and multiplied in one pass), with the tokens that
// chose an expert gathered as the MMA's N dimension, so that every expert's
// weights cross HBM once however many tokens use them.
//
// Numerics. tcgen05.mma kind::f16 multiplies f16 A and B exactly and
// accumulates in fp32. A is the decoded weight E2M1(q) * 2^(e - r), with r a
// per-row reference exponent computed at load time (the row's largest block
// exponent minus 13), so every block within 26 octaves of the row's largest
// is exact in f16; the row factor 2^(r - 127) is applied to the fp32
// accumulator. B is x (gate/up) or the down input h, in f16 with a power of
// two per row (x: exact for bf16; h: a high and a low f16 part in two
// columns, |h - hi - lo| <= 2^-22 |h|), removed again in the epilogue. The B
// rows are first written in expert order (one per assignment, grouped as the
// items list them), so that a block's columns are consecutive rows: one
// TMA tile per chunk.
//
// One persistent CTA per SM, 832 threads in roles; a unit is one expert x one
// M tile of 128 weight rows (8 of the 16-row fragment tiles: 64 gate + 64 up
// rows, or 128 down rows) x all of the expert's tokens, in blocks of at most
// 32 columns (32 tokens for gate/up, 16 for down: hi and lo columns):
//   warp 20     streams each 64-column chunk of the unit's 8 tiles
//               (8 x 544 B, one 4-d TMA tensor copy) into a ring of raw
//               stages;
//   warp 21     loads the B tile of the chunk (32 rows x 64 f16, one 2-d TMA
//               copy in the 128-byte swizzle layout) into a ring of
//               shared-memory stages;
//   warps 4-19  four groups of four warps; group g takes the chunks n with
//               n % 4 == g. Each warp decodes two tiles (the 32 tensor
//               memory lanes it may write): E2M1 -> f16 (cvt), times the
//               block's 2^(e - r) (mul.f16x2), stored straight into tensor
//               memory (tcgen05.st .16x128b: the register fragment of the
//               16-row tile lands in its 16 lanes, K along the columns), so
//               the A operand never touches shared memory;
//   warps 22-25 one per decoder group: issues the group's tcgen05.mma (A from
//               tensor memory, B from shared memory, M = 128, N = 16 or 32,
//               K = 16) into the group's own fp32 accumulator, one of two in
//               tensor memory per group (one issuing thread per accumulator
//               keeps its MMAs in order);
//   warps 0-3   read a finished block (tcgen05.ld, one row per thread), sum
//               the groups' accumulators and write h = silu(gate) * up, or the
//               down rows per token, while the next block accumulates in the
//               other buffers.
// Barrier waits and fences cost a few hundred cycles of latency each; four
// MMA warps overlap them, where a single one would serialise them.
// Asynchronous instructions are issued by one elected lane of a converged
// warp.
// Every wait is bounded; on a timeout the CTA records it, lets its copies
// and MMAs land, frees its tensor memory and leaves.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "internal.h"
#include "mxfrag.cuh"
#include "pipeline.cuh"
#include "umma.cuh"

namespace dfm {
namespace {

constexpr int kEpiWarps = 4;                   // warps 0-3
constexpr int kDecWarp0 = 4, kDecWarps = 16;   // warps 4-19
constexpr int kDecGroups = 4;                  // groups of 4 warps, every fourth chunk
constexpr int kGroupWarps = kDecWarps / kDecGroups;
constexpr int kRawWarp = 20, kBWarp = 21, kMmaWarp0 = 22;  // MMA warps 22-25
constexpr int kThr = 26 * 32;
constexpr int kM = 128;                        // weight rows per unit
constexpr int kTilesPerM = kM / 16;
constexpr int kCG = 2;                         // 64-column groups per chunk
constexpr int kCodeBytes = kTilesPerM * kCG * kGroupBytes;  // 8704: one 128-column chunk
constexpr int kRefBytes = kM;                  // reference exponents of the rows
constexpr int kRawBytes = kCodeBytes + kRefBytes;
constexpr int kRaw = 16;                       // raw chunks in flight
constexpr int kA = 4;                          // A stages (tensor memory)
constexpr int kSB = 8;                         // B stages (shared memory)
constexpr int kNMax = 32;                      // MMA N at most (B rows of a block)
constexpr int kBHalf = kNMax * 64 * 2;         // one TMA box: 32 rows x 64 f16
constexpr int kBBytes = kCG * kBHalf;          // B stage: 32 rows x 128 f16
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;                // per group two accumulators of kNMax columns
constexpr uint32_t kACol = 2 * kDecGroups * kNMax;  // kA A stages of 32 kCG columns
constexpr uint32_t kAStageCols = 32 * kCG;

static_assert(kACol + kAStageCols * kA <= kTmemCols, "tensor memory");
static_assert(kRawBytes % 16 == 0, "bulk copies need 16-byte aligned stages");

struct GemmArgs {
  ChunkMap map;         // 4-d tensor map of the expert tiles (gate/up or down)
  ChunkMap bmap;        // 2-d tensor map of the B rows in expert order
  const uint8_t* arena;
  size_t span_bytes;
  const uint8_t* eref;  // [E][2I + H] row reference exponents, fragment row order
  int H, I, k;
  const float* bsc;     // [T*k] 2^s of the B row(s) of each sorted assignment
  const Item* items;
  const int32_t* n_items;
  const int32_t* sorted;
  int max_items;
  float* out;           // gate/up: h [T*k][I]; down: part [T*k][H]
  uint32_t* err;
  // range checks: an item whose expert is outside [0, E) or whose
  // assignments leave [0, nassign) is skipped by every role alike, an
  // assignment index outside [0, nassign) is not written, and either is
  // recorded in *err (DEV_ERR_RANGE)
  int E, nassign;
};

struct Smem {
  uint64_t raw_full[kRaw], raw_empty[kRaw];
  uint64_t a_full[kA], a_free[kA];    // A stage decoded / read by its MMAs
  uint64_t b_full[kSB], b_free[kSB];  // B stage loaded / read by its MMAs
  uint64_t acc_full[2];   // every chunk of a block committed (one arrival per chunk)
  // Epilogue warps that have finished reading a block, summed over blocks.
  // A counter, not a barrier: the four MMA warps run at their own pace, and a
  // warp that is two blocks ahead of the epilogue would read a barrier's
  // parity as the phase before last.
  uint32_t epi_done;
  uint32_t tmem;
  int err;
};

constexpr size_t kBRingOffset = ((size_t)kRaw * kRawBytes + 1023) / 1024 * 1024;
constexpr size_t gemm_smem_bytes() {
  return kBRingOffset + (size_t)kSB * kBBytes + sizeof(Smem);
}
static_assert(gemm_smem_bytes() <= 227 * 1024, "shared memory");

// The sequence every role walks: for each of the CTA's units (expert item,
// M tile), each block of the item's tokens, the K/64 chunks.
struct Walk {
  int j;          // unit index of this CTA (u = blockIdx.x + j * gridDim.x)
  int item, mt;
  int tb, ntb;    // token block of the unit
  int c;          // chunk
  bool done;
};

template <int MODE>
__device__ __forceinline__ int walk_nc(const GemmArgs& a) {
  return (MODE == 0 ? a.H : a.I) / (64 * kCG);
}
template <int MODE>
__device__ __forceinline__ int walk_mt(const GemmArgs& a) { return MODE == 0 ? a.I / 64 : a.H / kM; }
template <int MODE>
__device__ __forceinline__ int block_tokens() { return MODE == 0 ? kNMax : kNMax / 2; }

template <int MODE>
__device__ void walk_seek(const GemmArgs& a, int n_items, Walk& w) {
  const int MT = walk_mt<MODE>(a);
  const int units = a.max_items * MT;
  for (;; ++w.j) {
    const int u = blockIdx.x + w.j * (int)gridDim.x;
    if (u >= units) {
      w.done = true;
      return;
    }
    w.item = u / MT;
    w.mt = u - w.item * MT;
    if (w.item >= n_items) {
      w.done = true;  // items are dense: none beyond n_items
      return;
    }
    const Item it = a.items[w.item];
    if ((unsigned)it.e >= (unsigned)a.E || it.pos < 0 || it.cnt < 0 ||
        it.pos + it.cnt > a.nassign) {
      if ((threadIdx.x & 31) == 0) atomicOr(a.err, DEV_ERR_RANGE);
      continue;
    }
    const int cnt = it.cnt;
    if (cnt <= 0) continue;
    w.ntb = (cnt + block_tokens<MODE>() - 1) / block_tokens<MODE>();
    w.tb = 0;
    w.c = 0;
    w.done = false;
    return;
  }
}

template <int MODE>
__device__ void walk_start(const GemmArgs& a, int n_items, Walk& w) {
  w.j = 0;
  w.done = false;
  walk_seek<MODE>(a, n_items, w);
}

template <int MODE>
__device__ void walk_next_block(const GemmArgs& a, int n_items, Walk& w) {
  w.c = 0;
  if (++w.tb < w.ntb) return;
  ++w.j;
  walk_seek<MODE>(a, n_items, w);
}

template <int MODE>
__device__ void walk_next(const GemmArgs& a, int n_items, Walk& w) {
  if (++w.c < walk_nc<MODE>(a)) return;
  walk_next_block<MODE>(a, n_items, w);
}

// Columns of a token block: rows of B (tokens for gate/up; hi and lo
// columns of each token for down), and the MMA N (a multiple of 16).
template <int MODE>
__device__ __forceinline__ int block_rows(const Item& it, int tb) {
  const int nb = min(block_tokens<MODE>(), it.cnt - tb * block_tokens<MODE>());
  return MODE == 0 ? nb : 2 * nb;
}
__device__ __forceinline__ int mma_n(int rows) { return (rows + 15) & ~15; }

// Bounded wait that sleeps between polls: for the warps off the critical
// path, whose polling would otherwise crowd the shared-memory pipe that the
// MMA warp's own barrier operations go through.
constexpr uint32_t kSleepWaitLimit = 1u << 22;
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  for (uint32_t i = 0; i < kSleepWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    __nanosleep(ns);
  }
  return false;
}

// Bounded wait until a shared counter reaches `target` (acquire).
__device__ __forceinline__ bool wait_count(const uint32_t* ctr, uint32_t target) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(ctr)) : "memory");
    if (v >= target) return true;
  }
  return false;
}

// A value the compiler can treat as warp-uniform (lane 0's), for the
// operands of instructions that take uniform registers.
__device__ __forceinline__ uint32_t uni(uint32_t v) { return __shfl_sync(0xffffffffu, v, 0); }
__device__ __forceinline__ uint64_t uni64(uint64_t v) {
  return ((uint64_t)uni((uint32_t)(v >> 32)) << 32) | uni((uint32_t)v);
}

__device__ __forceinline__ void set_err(Smem* sm) { *(volatile int*)&sm->err = 1; }
__device__ __forceinline__ bool has_err(Smem* sm) { return *(volatile int*)&sm->err != 0; }

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// The MMAs of one chunk (K = 64: four K = 16 steps) and the commits that
// follow them, issued by one elected lane of a converged warp in one
// straight-line block: A at tensor memory column a (+8 per step), B from the
// descriptor bd (+bstep per step), accumulating into d unless `fresh`;
// commits to the A stage, the B stage and the block barriers (none when
// a_free is 0). A commit tracks the issuing thread's own MMAs, so every
// chunk commits to the block barrier (one arrival per chunk).
__device__ __forceinline__ void mma_chunk(uint32_t d, uint32_t a, uint64_t bd, uint64_t bstep,
                                          uint32_t idesc, uint32_t fresh, uint32_t a_free,
                                          uint32_t b_free, uint32_t acc) {
  asm volatile(
      "{\n\t"
      ".reg .pred e, p0, pt, pc;\n\t"
      ".reg .b32 r, a1, a2, a3;\n\t"
      ".reg .b64 b1, b2, b3;\n\t"
      "elect.sync r|e, 0xffffffff;\n\t"
      "setp.eq.u32 p0, %5, 0;\n\t"
      "setp.eq.u32 pt, %5, %5;\n\t"
      "add.u32 a1, %1, 8;\n\t"
      "add.u32 a2, %1, 16;\n\t"
      "add.u32 a3, %1, 24;\n\t"
      "add.u64 b1, %2, %3;\n\t"
      "add.u64 b2, b1, %3;\n\t"
      "add.u64 b3, b2, %3;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %4, pt;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %4, pt;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %4, pt;\n\t"
      "setp.ne.and.u32 pc, %6, 0, e;\n\t"
      "@pc tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t"
      "@pc tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t"
      "@pc tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%8];\n\t"
      "}" ::"r"(d),
      "r"(a), "l"(bd), "l"(bstep), "r"(idesc), "r"(fresh), "r"(a_free), "r"(b_free), "r"(acc)
      : "memory");
}

// 2^d as an f16 pair, d = e - r for an E8M0 byte e and a reference r;
// NaN for e = 255 (the E8M0 NaN of OCP MX v1.0), 0 below the f16 range.
__device__ __forceinline__ uint32_t pow2_h2(uint32_t e, uint32_t r) {
  int d = (int)e - (int)r;
  d = max(-40, min(d, 15));
  const float f = e == 255u ? __uint_as_float(0x7FC00000u) : __uint_as_float((uint32_t)(d + 127) << 23);
  const __half2 h = __float2half2_rn(f);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ---------------------------------------------------------------------------
// Roles
// ---------------------------------------------------------------------------

template <int MODE>
__device__ void role_raw(const GemmArgs& a, int n_items, Smem* sm, uint8_t* raw, int lane) {
  // the whole warp walks; lane 0 issues one tensor copy per chunk (8 tiles x
  // 544 B), kRaw chunks ahead of the decoders
  const uint64_t pol = l2_evict_first_policy();
  const size_t eref_row = (size_t)2 * a.I + a.H;
  Walk w;
  walk_start<MODE>(a, n_items, w);
  uint32_t n = 0;
  int e = 0, e_item = -1;
  while (!w.done) {
    const uint32_t rs = n % kRaw;
    bool ok = n < (uint32_t)kRaw || mbar_wait_sleep(&sm->raw_empty[rs], ((n / kRaw) - 1) & 1, 128);
    ok = __all_sync(0xffffffffu, ok) && !has_err(sm);
    if (!ok) {
      set_err(sm);
      break;
    }
    if (w.item != e_item) {
      e_item = w.item;
      e = a.items[w.item].e;
    }
    {
      const uint32_t dst = smem_u32(raw + (size_t)rs * kRawBytes);
      const uint32_t bar = smem_u32(&sm->raw_full[rs]);
      // the reference exponents ride with the first chunk of a block that
      // each decoder group sees (chunks 0 and 1)
      const uint32_t ref = w.c < kDecGroups ? 1u : 0u;
      const uint8_t* rsrc = a.eref + (size_t)e * eref_row + (MODE == 0 ? 0 : 2 * (size_t)a.I) +
                            (size_t)kM * w.mt;
      // one elected lane: expect the bytes, then the tensor copy (and the
      // reference exponents)
      asm volatile(
          "{\n\t"
          ".reg .pred e, pr;\n\t"
          ".reg .b32 r, nb;\n\t"
          "elect.sync r|e, 0xffffffff;\n\t"
          "setp.ne.and.u32 pr, %8, 0, e;\n\t"
          "selp.u32 nb, %10, %11, pr;\n\t"
          "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%6], nb;\n\t"
          "@e cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;\n\t"
          "@pr cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
          " [%12], [%9], %13, [%6], %7;\n\t"
          "}" ::"r"(uni(dst)),
          "l"(&a.map), "r"(0), "r"(uni(kCG * w.c)), "r"(uni(kTilesPerM * w.mt)), "r"(uni(e)),
          "r"(uni(bar)), "l"(pol), "r"(uni(ref)), "l"(uni64((uint64_t)rsrc)),
          "r"((uint32_t)(kCodeBytes + kRefBytes)), "r"((uint32_t)kCodeBytes),
          "r"(uni(dst + (uint32_t)kCodeBytes)), "r"((uint32_t)kRefBytes)
          : "memory");
    }
    ++n;
    walk_next<MODE>(a, n_items, w);
  }
  // let every copy in flight land (the last fill of each slot)
  if (lane == 0) {
    const uint32_t first = n > (uint32_t)kRaw ? n - kRaw : 0;
    for (uint32_t m = first; m < n; ++m) (void)mbar_wait(&sm->raw_full[m % kRaw], (m / kRaw) & 1);
  }
}

// One tile's 16 code bytes of this lane -> 16 registers of f16 pairs in the
// order of tcgen05.st .16x128b.x8: per k-step, (g, k), (g+8, k), (g, k+8),
// (g+8, k+8).
__device__ __forceinline__ void load_tile(uint32_t tile_s, int lane, uint32_t (&cw)[4],
                                          uint32_t& sc) {
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(cw[0]), "=r"(cw[1]), "=r"(cw[2]), "=r"(cw[3])
               : "r"(tile_s + 16u * lane));
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sc) : "r"(tile_s + 512u + 4u * (lane >> 2)));
}

__device__ __forceinline__ void decode_tile(const uint32_t (&cw)[4], uint32_t sc, uint32_t rg,
                                            uint32_t rg8, uint32_t (&v)[16]) {
  // scale entry g: (row g, block 2G), (row g, 2G+1), (row g+8, 2G), (row g+8, 2G+1)
  uint32_t f0, f1, f80, f81;
  const int d0 = (int)(sc & 0xFF) - (int)rg, d1 = (int)((sc >> 8) & 0xFF) - (int)rg;
  const int d2 = (int)((sc >> 16) & 0xFF) - (int)rg8, d3 = (int)(sc >> 24) - (int)rg8;
  if (min(min(d0, d1), min(d2, d3)) >= -14 && __vcmpeq4(sc, 0xFFFFFFFFu) == 0) {
    // 2^d as a normal f16, both halves: exponent field d + 15 (d <= 13 by
    // the choice of r)
    f0 = (uint32_t)(d0 + 15) * 0x04000400u;
    f1 = (uint32_t)(d1 + 15) * 0x04000400u;
    f80 = (uint32_t)(d2 + 15) * 0x04000400u;
    f81 = (uint32_t)(d3 + 15) * 0x04000400u;
  } else {  // NaN scales, or blocks far below the row's largest
    f0 = pow2_h2(sc & 0xFF, rg);
    f1 = pow2_h2((sc >> 8) & 0xFF, rg);
    f80 = pow2_h2((sc >> 16) & 0xFF, rg8);
    f81 = pow2_h2(sc >> 24, rg8);
  }
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    uint32_t hv[4];
    decode_word(cw[ks], hv);
    const uint32_t fg = ks < 2 ? f0 : f1, fg8 = ks < 2 ? f80 : f81;
    v[4 * ks + 0] = hmul2(hv[0], fg);
    v[4 * ks + 1] = hmul2(hv[1], fg8);
    v[4 * ks + 2] = hmul2(hv[2], fg);
    v[4 * ks + 3] = hmul2(hv[3], fg8);
  }
}

__device__ __forceinline__ void tmem_st_16x128b_x8(uint32_t ta, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(ta),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

template <int MODE>
__device__ void role_decode(const GemmArgs& a, int n_items, Smem* sm, const uint8_t* raw,
                            uint32_t tmem, int warp, int lane) {
  const int q = warp & 3;                            // tensor memory lanes 32q..32q+31
  const int grp = (warp - kDecWarp0) / kGroupWarps;  // chunks n with n % kDecGroups == grp
  const int g = lane >> 2;
  const int NC = walk_nc<MODE>(a);
  Walk w;
  walk_start<MODE>(a, n_items, w);
  uint32_t nb0 = 0;               // global index of the block's chunk 0
  uint32_t rf[4] = {0, 0, 0, 0};  // reference exponents: rows g, g+8 of tiles 2q, 2q+1
  bool ok = true;
  while (!w.done && ok) {
    // this group's chunks of the block: n = nb0 + c with n % kDecGroups == grp
    for (int c = (grp - (int)(nb0 % kDecGroups) + kDecGroups) % kDecGroups; c < NC; c += kDecGroups) {
      const uint32_t n = nb0 + c;
      const uint32_t rs = n % kRaw, s = n % kA;
      ok = mbar_wait(&sm->raw_full[rs], (n / kRaw) & 1);
      if (ok && n >= (uint32_t)kA) ok = mbar_wait(&sm->a_free[s], ((n / kA) - 1) & 1);
      ok = __all_sync(0xffffffffu, ok) && !has_err(sm);
      if (!ok) break;
      const uint8_t* base = raw + (size_t)rs * kRawBytes;
      if (c < kDecGroups) {
        rf[0] = base[kCodeBytes + 32 * q + g];
        rf[1] = base[kCodeBytes + 32 * q + g + 8];
        rf[2] = base[kCodeBytes + 32 * q + 16 + g];
        rf[3] = base[kCodeBytes + 32 * q + 16 + g + 8];
      }
      // stage layout [tile][group][544 B]; tile 2q -> lanes 32q.., 2q+1 -> 32q+16..
      const uint32_t t0 = smem_u32(base) + (uint32_t)(2 * q * kCG * kGroupBytes);
      const uint32_t t1 = t0 + (uint32_t)(kCG * kGroupBytes);
      uint32_t cw[kCG][2][4], sc[kCG][2];
#pragma unroll
      for (int j = 0; j < kCG; ++j) {
        load_tile(t0 + (uint32_t)(j * kGroupBytes), lane, cw[j][0], sc[j][0]);
        load_tile(t1 + (uint32_t)(j * kGroupBytes), lane, cw[j][1], sc[j][1]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->raw_empty[rs]);
      const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + kACol + kAStageCols * s;
#pragma unroll
      for (int j = 0; j < kCG; ++j) {
        uint32_t v0[16], v1[16];
        decode_tile(cw[j][0], sc[j][0], rf[0], rf[1], v0);
        decode_tile(cw[j][1], sc[j][1], rf[2], rf[3], v1);
        tmem_st_16x128b_x8(ta + 32u * j, v0);
        tmem_st_16x128b_x8(ta + (16u << 16) + 32u * j, v1);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->a_full[s]);
    }
    nb0 += NC;
    walk_next_block<MODE>(a, n_items, w);
  }
  if (!ok) set_err(sm);
}

// The MMA warp of decoder group grp: the group's chunks in order, into the
// group's accumulators.
template <int MODE>
__device__ void role_mma(const GemmArgs& a, int n_items, Smem* sm, const uint8_t* bring,
                         uint32_t tmem, int grp) {
  const int NC = walk_nc<MODE>(a);
  Walk w;
  walk_start<MODE>(a, n_items, w);
  uint32_t nb0 = 0, blk = 0;
  int last = -1;  // the last chunk whose MMAs this warp issued
  bool ok = true;
  while (!w.done && ok) {
    const uint32_t idesc = umma::idesc_f16_f32(kM, mma_n(block_rows<MODE>(a.items[w.item], w.tb)));
    for (int c = (grp - (int)(nb0 % kDecGroups) + kDecGroups) % kDecGroups; c < NC; c += kDecGroups) {
      const uint32_t n = nb0 + c;
      const uint32_t s = n % kA, sbi = n % kSB, ab = blk & 1;
      const uint32_t fresh = c < kDecGroups ? 1u : 0u;  // the group's first chunk of the block
      ok = mbar_wait(&sm->a_full[s], (n / kA) & 1) && mbar_wait(&sm->b_full[sbi], (n / kSB) & 1);
      if (ok && fresh && blk >= 2) ok = wait_count(&sm->epi_done, kEpiWarps * (blk - 1));
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = uni(tmem + kAccCol + (uint32_t)kNMax * (2 * grp + ab));
      const uint32_t at = uni(tmem + kACol + kAStageCols * s);
      const uint64_t bd = uni64(umma::smem_desc_sw128(smem_u32(bring + (size_t)sbi * kBBytes)));
      // group 0: fresh on the group's first chunk; group 1 always accumulates
      mma_chunk(d, at, bd, 32 >> 4, uni(idesc), uni(fresh), 0u, 0u, 0u);
      mma_chunk(d, at + 32u, bd + (uint64_t)(kBHalf >> 4), 32 >> 4, uni(idesc), 0u,
                uni(smem_u32(&sm->a_free[s])), uni(smem_u32(&sm->b_free[sbi])),
                uni(smem_u32(&sm->acc_full[ab])));
      last = (int)n;
    }
    nb0 += NC;
    ++blk;
    walk_next_block<MODE>(a, n_items, w);
  }
  if (!ok) set_err(sm);
  // the MMAs must land before the tensor memory is released (a commit tracks
  // all of the issuing thread's earlier MMAs)
  if (last >= 0) (void)mbar_wait(&sm->a_free[last % kA], ((uint32_t)last / kA) & 1);
}

// The B warp: one tensor copy per chunk, the block's 32 consecutive rows in
// expert order (rows past the block belong to the next item or lie past the
// end, where the copy fills zeros; their columns are never read back).
template <int MODE>
__device__ void role_b(const GemmArgs& a, int n_items, Smem* sm, uint8_t* bring, int lane) {
  const int NC = walk_nc<MODE>(a);
  Walk w;
  walk_start<MODE>(a, n_items, w);
  uint32_t n = 0;
  bool ok = true;
  while (!w.done && ok) {
    const Item it = a.items[w.item];
    const int row0 = (MODE == 0 ? 1 : 2) * (it.pos + w.tb * block_tokens<MODE>());
    for (int c = 0; c < NC; ++c) {
      const uint32_t s = n % kSB;
      if (n >= (uint32_t)kSB) {
        const bool got =
            __all_sync(0xffffffffu, mbar_wait_sleep(&sm->b_free[s], ((n / kSB) - 1) & 1, 128));
        if (!got || has_err(sm)) {
          set_err(sm);
          ok = false;
          break;
        }
      }
      asm volatile(
          "{\n\t"
          ".reg .pred e;\n\t"
          ".reg .b32 r;\n\t"
          "elect.sync r|e, 0xffffffff;\n\t"
          "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%4], %5;\n\t"
          "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%2, %3}], [%4];\n\t"
          "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          " [%6], [%1, {%7, %3}], [%4];\n\t"
          "}" ::"r"(uni(smem_u32(bring + (size_t)s * kBBytes))),
          "l"(&a.bmap), "r"(uni(128 * c)), "r"(uni(row0)), "r"(uni(smem_u32(&sm->b_full[s]))),
          "r"((uint32_t)kBBytes), "r"(uni(smem_u32(bring + (size_t)s * kBBytes + kBHalf))),
          "r"(uni(128 * c + 64))
          : "memory");
      ++n;
    }
    if (ok) walk_next_block<MODE>(a, n_items, w);
  }
  // let every copy in flight land (the last fill of each stage)
  if (lane == 0) {
    const uint32_t first = n > (uint32_t)kSB ? n - kSB : 0;
    for (uint32_t m = first; m < n; ++m) (void)mbar_wait(&sm->b_full[m % kSB], (m / kSB) & 1);
  }
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t ta, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(ta));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int MODE>
__device__ void role_epilogue(const GemmArgs& a, int n_items, Smem* sm, uint32_t tmem, int warp,
                              int lane) {
  const int m = 32 * warp + lane;  // accumulator row = tensor memory lane
  const size_t eref_row = (size_t)2 * a.I + a.H;
  const int NC = walk_nc<MODE>(a);
  Walk w;
  walk_start<MODE>(a, n_items, w);
  uint32_t blk = 0;
  while (!w.done) {
    const Item it = a.items[w.item];
    const int rows = block_rows<MODE>(it, w.tb), N = mma_n(rows);
    const int n0 = w.tb * block_tokens<MODE>();
    // per-column data: lane j holds the assignment and the B row scale of the
    // block's token j (sorted position it.pos + n0 + j)
    const int nt = MODE == 0 ? rows : rows / 2;  // tokens in the block (<= 32)
    int asg0 = 0;
    float sc0 = 0.f;
    if (lane < nt) {
      asg0 = a.sorted[it.pos + n0 + lane];
      sc0 = a.bsc[it.pos + n0 + lane];
      if ((unsigned)asg0 >= (unsigned)a.nassign) {
        atomicOr(a.err, DEV_ERR_RANGE);
        asg0 = -1;
      }
    }
    const uint32_t e_ref = a.eref[(size_t)it.e * eref_row + (MODE == 0 ? 0 : 2 * (size_t)a.I) +
                                  (size_t)kM * w.mt + m];
    const float rowfac = __uint_as_float(e_ref ? (e_ref << 23) : 0x00400000u);  // 2^(r - 127)
    const uint32_t ab = blk & 1;
    const bool got = __all_sync(0xffffffffu, mbar_wait_sleep(&sm->acc_full[ab], (blk / 2) & 1, 256));
    if (!got || has_err(sm)) {
      set_err(sm);
      break;
    }
    tc_fence_after();
    // the groups that hold chunks of this block (all four unless K < 256):
    // chunk c of block blk went to group (blk * NC + c) % 4
    uint32_t gmask = 0;
    for (int c = 0; c < NC && c < kDecGroups; ++c) gmask |= 1u << ((blk * NC + c) % kDecGroups);
    const uint32_t d = tmem + ((uint32_t)(32 * warp) << 16) + kAccCol + (uint32_t)kNMax * ab;
    for (int c0 = 0; c0 < N; c0 += 16) {
      uint32_t r[16];
      float acc[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = 0.f;
      for (int gg = 0; gg < kDecGroups; ++gg) {
        if (!(gmask >> gg & 1)) continue;
        tmem_ld_32x32b_x16(d + (uint32_t)(2 * kNMax * gg + c0), r);
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] += __uint_as_float(r[i]);
      }
      if (MODE == 0) {
        // rows 16t + rho: gate row rho < 8 pairs with up row rho + 8 (lane ^ 8)
        const int rho = m & 15;
        const int irow = 64 * w.mt + 8 * (m >> 4) + rho;  // intermediate index
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = c0 + i;
          const int asg = __shfl_sync(0xffffffffu, asg0, col);
          const float xs = __shfl_sync(0xffffffffu, sc0, col);
          const float v = acc[i] * rowfac * xs;
          const float up = __shfl_xor_sync(0xffffffffu, v, 8);
          if (rho < 8 && col < rows && asg >= 0) a.out[(size_t)asg * a.I + irow] = silu_f(v) * up;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const int tok = (c0 + i) >> 1;  // columns 2 tok (hi), 2 tok + 1 (lo)
          const int asg = __shfl_sync(0xffffffffu, asg0, tok);
          const float hs = __shfl_sync(0xffffffffu, sc0, tok);
          if (tok < nt && asg >= 0)
            a.out[(size_t)asg * a.H + (size_t)kM * w.mt + m] =
                (acc[i] + acc[i + 1]) * rowfac * hs;
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0)  // this warp's reads of the block are done
      asm volatile("red.release.cta.shared::cta.add.u32 [%0], 1;" ::"r"(smem_u32(&sm->epi_done))
                   : "memory");
    ++blk;
    walk_next_block<MODE>(a, n_items, w);
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThr, 1) gemm_kernel(const __grid_constant__ GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* raw = smem;
  uint8_t* bring = smem + kBRingOffset;  // 1024-aligned: the 128-byte swizzle
  Smem* sm = reinterpret_cast<Smem*>(bring + (size_t)kSB * kBBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm->tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < kRaw; ++i) {
      mbar_init(&sm->raw_full[i], 1);
      mbar_init(&sm->raw_empty[i], kGroupWarps);
    }
    for (int i = 0; i < kA; ++i) {
      mbar_init(&sm->a_full[i], kGroupWarps);
      mbar_init(&sm->a_free[i], 1);
    }
    for (int i = 0; i < kSB; ++i) {
      mbar_init(&sm->b_full[i], 1);
      mbar_init(&sm->b_free[i], 1);
    }
    for (int i = 0; i < 2; ++i)
      mbar_init(&sm->acc_full[i], (uint32_t)walk_nc<MODE>(a));  // one commit per chunk
    sm->epi_done = 0;
    sm->err = 0;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&sm->tmem);

  pdl_wait();  // items and the B sources come from the preceding kernels
  int n_items = *a.n_items;
  if (n_items < 0 || n_items > a.max_items) {
    if (threadIdx.x == 0) atomicOr(a.err, DEV_ERR_RANGE);
    n_items = n_items < 0 ? 0 : a.max_items;
  }
  if (warp < kEpiWarps) {
    role_epilogue<MODE>(a, n_items, sm, tmem, warp, lane);
  } else if (warp < kDecWarp0 + kDecWarps) {
    role_decode<MODE>(a, n_items, sm, raw, tmem, warp, lane);
  } else if (warp == kRawWarp) {
    role_raw<MODE>(a, n_items, sm, raw, lane);
  } else if (warp == kBWarp) {
    role_b<MODE>(a, n_items, sm, bring, lane);
  } else {
    role_mma<MODE>(a, n_items, sm, bring, tmem, warp - kMmaWarp0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && has_err(sm)) atomicOr(a.err, DEV_ERR_TIMEOUT);
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

// ---------------------------------------------------------------------------
// B sources: rows in f16 with a power-of-two scale per row
// ---------------------------------------------------------------------------

// s = floor(log2(mx)) - 14, so that the row's largest magnitude lands in
// [2^14, 2^15) (f16 holds up to 65504); 0 for zero or non-finite rows;
// clamped to [-112, 112] so that 2^s and 2^-s are normal floats.
__device__ __forceinline__ int row_shift(float mx) {
  const uint32_t eb = (__float_as_uint(mx) >> 23) & 0xFF;
  if (mx == 0.f || eb == 0xFF) return 0;
  return max(-112, min((int)eb - 127 - 14, 112));
}

__device__ float block_max_abs(float v, float* red) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) red[0] = v;
  }
  __syncthreads();
  const float r = red[0];
  __syncthreads();
  return r;
}

// Gate/up B rows in expert order: row p = x[sorted[p] / k] * 2^-s (f16,
// exact for bf16 x), bsc[p] = 2^s, s from the token's largest |x|.
__global__ void __launch_bounds__(256) prep_x_kernel(const uint16_t* x, int H, int k,
                                                     const int32_t* sorted, __half* xg,
                                                     float* bsc, uint32_t* err) {
  __shared__ float red[32];
  const int p = blockIdx.x;
  int a = sorted[p];
  if ((unsigned)a >= gridDim.x) {  // R = T * k assignments
    if (threadIdx.x == 0) atomicOr(err, DEV_ERR_RANGE);
    a = 0;
  }
  const uint16_t* xr = x + (size_t)(a / k) * H;
  float mx = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x)
    mx = fmaxf(mx, fabsf(__uint_as_float((uint32_t)xr[i] << 16)));
  mx = block_max_abs(mx, red);
  const int sh = row_shift(mx);
  const float inv = __uint_as_float((uint32_t)(127 - sh) << 23);
  for (int i = threadIdx.x; i < H; i += blockDim.x)
    xg[(size_t)p * H + i] = __float2half_rn(__uint_as_float((uint32_t)xr[i] << 16) * inv);
  if (threadIdx.x == 0) bsc[p] = __uint_as_float((uint32_t)(127 + sh) << 23);
}

// Down B rows in expert order: rows 2p, 2p + 1 = high and low f16 parts of
// h[sorted[p]] * 2^-s, bsc[p] = 2^s.
__global__ void __launch_bounds__(256) split_h_kernel(const float* h, int I,
                                                      const int32_t* sorted, __half* hh,
                                                      float* bsc, uint32_t* err) {
  __shared__ float red[32];
  const int p = blockIdx.x;
  int a = sorted[p];
  if ((unsigned)a >= gridDim.x) {  // R = T * k assignments
    if (threadIdx.x == 0) atomicOr(err, DEV_ERR_RANGE);
    a = 0;
  }
  const float* hr = h + (size_t)a * I;
  float mx = 0.f;
  for (int i = threadIdx.x; i < I; i += blockDim.x) mx = fmaxf(mx, fabsf(hr[i]));
  mx = block_max_abs(mx, red);
  const int sh = row_shift(mx);
  const float inv = __uint_as_float((uint32_t)(127 - sh) << 23);
  __half* hi = hh + (size_t)p * 2 * I;
  for (int i = threadIdx.x; i < I; i += blockDim.x) {
    const float v = hr[i] * inv;
    const __half q = __float2half_rn(v);
    hi[i] = q;
    hi[I + i] = __float2half_rn(v - __half2float(q));
  }
  if (threadIdx.x == 0) bsc[p] = __uint_as_float((uint32_t)(127 + sh) << 23);
}

// Reference exponent of every fragment row of `n` spans: the largest E8M0
// byte of the row other than 255, minus 13, at least 0.
__global__ void __launch_bounds__(256) row_ref_kernel(const uint8_t* arena, size_t span_bytes,
                                                      int H, int I, int n, uint8_t* eref) {
  const int rows_per = 2 * I + H;
  const long long total = (long long)n * rows_per;
  const SpanLayout L = span_layout(H, I);
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int e = (int)(idx / rows_per);
    const int fr = (int)(idx - (long long)e * rows_per);  // fragment row in the span
    const bool gu = fr < 2 * I;
    const int K = gu ? H : I;
    const int tile = (gu ? fr : fr - 2 * I) >> 4, rho = fr & 15;
    const uint8_t* t = arena + (size_t)e * span_bytes + (gu ? L.gu : L.dn) +
                       (size_t)tile * mx_tile_bytes(K);
    const int off = 512 + 4 * (rho & 7) + (rho >> 3) * 2;
    int mx = -1;
    for (int G = 0; G < mx_ngroups(K); ++G) {
      const uint8_t* p = t + (size_t)G * kGroupBytes + off;
      const int e0 = p[0], e1 = p[1];
      if (e0 != 255) mx = max(mx, e0);
      if (e1 != 255) mx = max(mx, e1);
    }
    eref[idx] = (uint8_t)max(mx - 13, 0);
  }
}

int sm_count_g() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

template <int MODE>
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s) {
  static bool configured = false;
  const size_t smem = gemm_smem_bytes();
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int MT = MODE == 0 ? a.I / 64 : a.H / kM;
  const long long units = (long long)a.max_items * MT;
  int grid = sm_count_g();
  if (units < grid) grid = (int)(units > 0 ? units : 1);
  gemm_kernel<MODE><<<grid, kThr, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool gemm_supported(int H, int I) {
  return H % kM == 0 && H % (64 * kCG) == 0 && I % (64 * kCG) == 0 && I % 64 == 0 && H >= kM;
}

// The tiles of one matrix kind of every expert as a 4-d tensor of u32:
// (136 words of a 544-byte group, K/64 groups, tiles of the expert, expert),
// so that one box (136, 1, 8, 1) is the chunk of 8 tiles a unit needs.
namespace {
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return encode;
}
}  // namespace

bool make_chunk_maps(const uint8_t* arena, size_t span_bytes, int H, int I, int E,
                     ChunkMap* gu, ChunkMap* dn) {
  static_assert(sizeof(ChunkMap) == sizeof(CUtensorMap), "tensor map size");
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return false;
  const SpanLayout L = span_layout(H, I);
  for (int mode = 0; mode < 2; ++mode) {
    const int K = mode == 0 ? H : I, tiles = mode == 0 ? 2 * I / 16 : H / 16;
    const cuuint64_t dims[4] = {kGroupBytes / 4, (cuuint64_t)(K / 64), (cuuint64_t)tiles,
                                (cuuint64_t)E};
    const cuuint64_t strides[3] = {kGroupBytes, mx_tile_bytes(K), span_bytes};
    const cuuint32_t box[4] = {kGroupBytes / 4, kCG, kTilesPerM, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    void* base = const_cast<uint8_t*>(arena + (mode == 0 ? L.gu : L.dn));
    CUtensorMap* m = reinterpret_cast<CUtensorMap*>(mode == 0 ? gu : dn);
    if (encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, base, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

size_t gemm_eref_bytes(int n_experts, int H, int I) {
  return (size_t)n_experts * (2 * (size_t)I + H);
}

cudaError_t launch_row_ref(const uint8_t* arena, size_t span_bytes, int H, int I, int n,
                           uint8_t* eref, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const long long total = (long long)n * (2 * I + H);
  const int grid = (int)std::min<long long>((total + 255) / 256, 4096);
  row_ref_kernel<<<grid, 256, 0, s>>>(arena, span_bytes, H, I, n, eref);
  return cudaGetLastError();
}

cudaError_t launch_prep_x(const uint16_t* x, int R, int H, int k, const int32_t* sorted,
                          uint16_t* xg, float* bsc, uint32_t* err, cudaStream_t s) {
  prep_x_kernel<<<R, 256, 0, s>>>(x, H, k, sorted, reinterpret_cast<__half*>(xg), bsc, err);
  return cudaGetLastError();
}

cudaError_t launch_split_h(const float* h, int R, int I, const int32_t* sorted, uint16_t* hh,
                           float* bsc, uint32_t* err, cudaStream_t s) {
  split_h_kernel<<<R, 256, 0, s>>>(h, I, sorted, reinterpret_cast<__half*>(hh), bsc, err);
  return cudaGetLastError();
}

// 2-d maps of the expert-ordered B rows: gate/up [R][H] and down [2R][I]
// f16, boxes of 64 columns x kNMax rows in the 128-byte swizzle layout.
bool make_b_maps(const uint16_t* xg, const uint16_t* hh, int R, int H, int I, ChunkMap* gu,
                 ChunkMap* dn) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return false;
  for (int mode = 0; mode < 2; ++mode) {
    const int K = mode == 0 ? H : I;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)(mode == 0 ? R : 2 * R)};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, kNMax};
    const cuuint32_t es[2] = {1, 1};
    void* base = const_cast<uint16_t*>(mode == 0 ? xg : hh);
    CUtensorMap* m = reinterpret_cast<CUtensorMap*>(mode == 0 ? gu : dn);
    if (encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

cudaError_t launch_gemm_gateup(const ChunkMap& map, const ChunkMap& bmap, const uint8_t* arena,
                               size_t span_bytes, const uint8_t* eref, int H, int I, int k,
                               const float* bsc, const Item* items, const int32_t* n_items,
                               int max_items, const int32_t* sorted, float* hbuf, int E,
                               int nassign, uint32_t* err, cudaStream_t s) {
  GemmArgs a{map, bmap, arena, span_bytes, eref, H, I, k, bsc,
             items, n_items, sorted, max_items, hbuf, err, E, nassign};
  return launch_gemm<0>(a, s);
}

cudaError_t launch_gemm_down(const ChunkMap& map, const ChunkMap& bmap, const uint8_t* arena,
                             size_t span_bytes, const uint8_t* eref, int H, int I, int k,
                             const float* bsc, const Item* items, const int32_t* n_items,
                             int max_items, const int32_t* sorted, float* part, int E,
                             int nassign, uint32_t* err, cudaStream_t s) {
  GemmArgs a{map, bmap, arena, span_bytes, eref, H, I, k, bsc,
             items, n_items, sorted, max_items, part, err, E, nassign};
  return launch_gemm<1>(a, s);
}

}  // namespace dfm
