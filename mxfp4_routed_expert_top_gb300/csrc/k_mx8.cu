// k_mx8.cu — the routed experts with MXFP8 activations (the lossy variant):
// grouped GEMMs on tcgen05.mma kind::mxf8f6f4 with hardware block scales.
//
// Kimi K3 is trained quantisation-aware with MXFP4 weights and MXFP8
// activations (Deltafin analysis, section 2.1); the pages' reference runs
// keep the numerics exact and list the lossy switches apart (section 9.2).
// Here the activations entering the routed experts (x for gate/up, h for
// down) are rounded to MXFP8 — OCP microscaling blocks of 32 along the
// contraction, E4M3 elements sharing one E8M0 exponent — and the tensor core
// multiplies the E2M1 weights by the E4M3 activations, applying both blocks'
// exponents itself. Products are exact and the sums are fp32, so the only
// loss is the rounding of the activations to the format.
//
// Weights: MXFP4 codes (low nibble first), arranged at load time so that
// each 128-row tile's 128-column stage is 8 KB of contiguous rows of 64
// bytes ([tile][stage][row][64 bytes]: the stream of a unit is sequential),
// read by TMA as 16U4_ALIGN16B, which puts every 16 codes in the first 8
// bytes of a 16-byte group of shared memory: the operand layout of
// kind::mxf8f6f4 for a 4-bit type (a byte of space per element, so a K = 32
// step is 32 bytes, as for the 8-bit B).
// Scales reach tensor memory by tcgen05.cp .32x128b.warpx4, issued by the MMA
// thread just before the stage's MMAs (the tensor pipe keeps them in order):
// it copies 32 rows of 16 bytes to the 32 lanes of every lane quarter, and
// the MMA reads row r (A) or token n (B) at lane r mod 32 of its quarter,
// column base + r/32 (n/32), byte = the K step. So a stage's scales are a
// 512-byte chunk holding the word of row r at 16 (r mod 32) + 4 (r / 32):
//   weights: arranged so at load time, per 128-row tile and 128-column stage
//            (one bulk copy per operand and stage);
//   activations: rows of 16 bytes whose word j is the scale word of row
//            + 32 j, so that the 32 rows from any first row are that chunk
//            (stage-major: [K/128][rows][16 bytes]).
// Activation rows: E4M3, in expert order (row p for sorted position p).
//
// Two persistent CTAs per SM, 192 threads in roles; a unit is one item x its
// 128-row operands (gate/up: 128 gate and the same 128 up rows, two MMAs a K
// step into two accumulators, so that each thread of the epilogue holds both
// values of its h row; down: one 128-row tile), x the item's tokens in passes
// (the MMA's N a multiple of 16), the contraction in stages of 128 columns:
//   warp 4     TMA: a stage's A operands (one 128-row box each), its B rows
//              (a pass in one or two boxes) and its scale chunks (bulk
//              copies), on a ring of shared-memory stages;
//   warp 5     per stage: the scale copies to tensor memory, the MMAs (M =
//              128, K = 32) into one of 3 (gate/up) or 4 (down) accumulator
//              sets in turn, the commits;
//   warps 0-3  the epilogue of a finished pass, one TMEM lane (one row) a
//              thread: gate/up: h = silu(gate) * up, rounded to MXFP8 per 32
//              rows (one warp a block) for the down GEMM; down: the rows of
//              each assignment's output.
// Every wait is bounded; after a timeout every role leaves its loop, the
// copies and MMAs in flight land, and the CTA frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "bfv.cuh"
#include "internal.h"
#include "pipeline.cuh"
#include "select.cuh"
#include "umma.cuh"

namespace dfm {
namespace {

constexpr int kThr = 192;
constexpr int kTmaWarp = 4, kMmaWarp = 5;
constexpr int kM = 128, kHalfRows = 64;
constexpr int kKS = 128;                  // contraction columns a stage
constexpr int kABytes = kM * kKS;         // 16384: one A operand (a byte a code)
constexpr int kATx = kM * kKS / 2;       // 8192: an A operand's codes as copied (packed)
constexpr int kSfBytes = 512;            // a stage's scale chunk (an operand's, or the tokens')
constexpr int kSfRowBytes = 16;           // an activation row's scale words
constexpr uint32_t kTmemCols = 512;  // an SM's tensor memory
// B rows a TMA box: a whole pass of exact planes (16 tokens x P planes) in
// one box, 32 rows for one plane (passes of 32 or 64 rows). A box may run
// past the pass into the next item's rows (or past the buffer: zero fill);
// the MMA columns there are never read.
__host__ __device__ constexpr int box_rows(int planes) { return planes > 1 ? 16 * planes : 32; }

// CTAs an SM runs of each GEMM: two, each with half the shared and tensor
// memory, so that one CTA's pass and unit boundaries (accumulator hand-over,
// ring ramp) overlap the other's streaming. Measured at batch 512 against one
// CTA an SM: MXFP8 gate/up and down 9-11% faster, exact planes 6% (gate/up)
// and 7% (down) faster.
__host__ __device__ constexpr int ctas_per_sm(int mode, int planes) {
  (void)mode;
  (void)planes;
  return 2;
}

// Per GEMM, token tile KN (tokens a pass at most) and planes P: one
// 128-row A operand a stage (gate/up: 64 gate rows and the same 64 up rows,
// so that one MMA gives both values of 64 h rows; down: a 128-row tile), the
// stages that fit in the CTA's share of shared memory beside the gate/up
// epilogue's exchange buffers, the accumulator sets that fit in its share of
// tensor memory beside the stages' scales, and the layout of one stage in
// shared memory and of the tensor memory columns. Gate/up stages hold the
// two 128-row tiles' raw scale chunks; the MMA warp assembles the operand's
// chunk from their halves in place of the first. (Units of the full 128 gate and 128 up
// rows, two accumulators, left one accumulator set a CTA with two CTAs an
// SM; one 128-row down tile a unit measured 7% faster than pairs of tiles.)
template <int MODE, int KN, int P>
struct Geo {
  static constexpr int CPS = ctas_per_sm(MODE, P);
  static constexpr uint32_t TmemCols = kTmemCols / CPS;
  static constexpr int RawSf = MODE == 0 ? 2 : 1;  // raw A scale chunks a stage
  static constexpr int BR = KN < box_rows(P) ? KN : box_rows(P);  // B rows a box
  static constexpr int BBytes = KN * kKS;
  static constexpr int StageBytes = kABytes + BBytes + RawSf * kSfBytes + kSfBytes;
  // gate/up: the up rows' values handed to the gate rows, two buffers of 64
  // rows x XW floats (one pass's tokens, 32 at a time for one plane)
  static constexpr int XW = (P == 1 ? 32 : KN / P) + 1;
  static constexpr size_t XBytes = MODE == 0 ? 2 * 64 * XW * 4 : 0;
  static constexpr int S0 = (int)(((CPS == 1 ? 226 * 1024 : 111 * 1024) - XBytes) / StageBytes);
  static constexpr int S = S0 > 12 ? 12 : S0;
  static constexpr size_t offA = 0;
  static constexpr size_t offB = offA + (size_t)S * kABytes;
  static constexpr size_t offSfRaw = offB + (size_t)S * BBytes;
  static constexpr size_t offSfb = offSfRaw + (size_t)S * RawSf * kSfBytes;
  static constexpr size_t offX = offSfb + (size_t)S * kSfBytes;
  static constexpr size_t offBars = offX + XBytes;
  static constexpr uint32_t accCols = KN;      // one accumulator set
  static constexpr uint32_t sfStride = 4 + 4;  // per stage 4 A, 4 B scale columns
  static constexpr int NACC0 = (int)((TmemCols - S * sfStride) / accCols);
  static constexpr int NACC = NACC0 > 4 ? 4 : NACC0;  // accumulator sets (MMA runs ahead)
  static constexpr uint32_t sfCol = NACC * accCols;
};

template <int S, int NACC>
struct Bars {
  uint64_t full[S], empty[S];
  uint64_t accf[NACC], acce[NACC], fin;
  uint64_t xfull[2], xempty[2];  // gate/up: the exchange buffers written / read
  uint32_t tmem;
  int err;
};
template <int MODE, int KN, int P>
constexpr size_t smem_bytes() {
  using G = Geo<MODE, KN, P>;
  return G::offBars + sizeof(Bars<G::S, G::NACC>);
}
// Fits: the CTAs of an SM in its shared memory, at least two stages, one
// accumulator set (two where one CTA runs on an SM), the scale columns.
template <int MODE, int KN, int P>
constexpr bool geo_ok() {
  using G = Geo<MODE, KN, P>;
  return smem_bytes<MODE, KN, P>() <= (G::CPS == 1 ? 227 * 1024 : 112 * 1024) && G::S >= 2 &&
         G::NACC >= (G::CPS == 1 ? 2 : 1) && G::sfCol + G::sfStride * G::S <= G::TmemCols &&
         G::offB % 1024 == 0 && G::BBytes % 1024 == 0;
}
static_assert(geo_ok<0, 32, 1>() && geo_ok<0, 64, 1>() && geo_ok<1, 32, 1>() &&
                  geo_ok<1, 64, 1>() && geo_ok<0, 64, kPlanesX>() && geo_ok<1, 80, kPlanesH>(),
              "shared or tensor memory");

struct Mx8Args {
  ChunkMap amap0, amap1;  // gate/up: gate and up codes; down: down codes
  ChunkMap bmap;          // activation rows [rows_cap][K] E4M3
  const uint8_t* arena;
  size_t span_bytes;
  size_t sfa0, sfa1;      // span offsets of the A operands' scale sections
  int K, MT;              // contraction; M tiles an item
  int I, H;
  const uint8_t* bsf;     // activation scales [K/128][rows_cap][16]
  int rows_cap;
  const Item* items;
  const int32_t* n_items;
  const int32_t* sorted;
  int max_items, E, nassign;
  float* hbuf;            // gate/up: optional [nassign][I] h before rounding
  uint8_t* hq;            // gate/up: [hrows_cap][I] E4M3 rows of h (expert order)
  uint8_t* hsf;           // gate/up: [I/128][hrows_cap][16] their scales
  int hrows_cap;          // gate/up: rows of hq
  float* part;            // down: [nassign][H]
  uint32_t* err;
  // gate/up of one token beside the shared experts: each unit covers
  // 1/kspl of K and writes its gate and up sums, before SwiGLU, to
  // gu_part [kspl][nassign][2][I] (kspl 0 or 1: whole K, h out)
  int kspl;
  float* gu_part;
};

// ---------------------------------------------------------------------------
// MXFP8 rounding (OCP microscaling, E4M3 elements, E8M0 per 32)
// ---------------------------------------------------------------------------

// 2^e for e in [-127, 127] (2^-127 is a subnormal float).
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __int_as_float((e + 127) << 23) : __int_as_float(0x00400000);
}

// The block's shared exponent: floor(log2(amax)) - 8 (8 is E4M3's largest
// exponent), clamped to E8M0's [-127, 127]; -127 for an all-zero block.
__device__ __forceinline__ int mx8_shared_exp(float amax) {
  if (amax == 0.f) return -127;
  return max(-127, min(127, ilogbf(amax) - 8));
}

// E4M3 code -> its value (exact).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(code | code << 8)));
  return __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFFu)));
}

// E4M3 code of v, nearest with ties to even, |v| beyond 448 saturating.
__device__ __forceinline__ uint32_t e4m3_rn_sat(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(v));
  return r & 0xFFu;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Places a row's scales take in the stage-major, row-interleaved layout of
// an activation buffer of `planes` rows a token or assignment: word q of row
// R holds the scales of row R + 32 q, and a GEMM pass reads words q <
// ceil(pass rows / 32) of the 32 rows from its first (the other words reach
// no MMA column). Passes hold at most 16 P rows of planes, 64 of one plane.
__host__ __device__ constexpr int scale_places(int planes) {
  return planes > 1 ? (16 * planes + 31) / 32 : 2;
}

// Writes the scale byte of block j (along K) of activation row `row` into
// that layout: stage j/4, byte j mod 4 of word q of row row - 32 q, q <
// places.
__device__ __forceinline__ void put_scale(uint8_t* sf, int rows_cap, int row, int j, uint8_t v,
                                          int places) {
  const size_t ks = (size_t)(j >> 2);
  for (int q = 0; q < places; ++q)
    if (row - 32 * q >= 0) sf[((ks * rows_cap + row - 32 * q) * 4 + q) * 4 + (j & 3)] = v;
}

// ---------------------------------------------------------------------------
// tensor memory, MMA and copy helpers
// ---------------------------------------------------------------------------

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
__device__ __forceinline__ void mma_mx(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}" ::"r"(d),
      "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
// Weight tiles (read once a call): evict-first in L2, so that the streamed
// weights do not push out the activation rows every M tile re-reads.
// Coordinates (element, row in the tile, stage, tile, expert).
__device__ __forceinline__ void tma5d_stream(void* dst, const ChunkMap* m, int r, int ks, int tile,
                                             int e, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(dst)),
      "l"(m), "r"(0), "r"(r), "r"(ks), "r"(tile), "r"(e), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, const void* src) {
  const uint64_t d = umma::smem_desc(smem_u32(src), 128, 128);
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}
__device__ __forceinline__ void tma2d(void* dst, const ChunkMap* m, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(m), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_plain(void* dst, const void* src, uint32_t bytes,
                                           uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: gives up after ~200 ms (and records it in *err), or soon
// after another role of the CTA has given up.
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;
__device__ __forceinline__ bool wait_or_give_up(uint64_t* bar, uint32_t parity, int* err) {
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (*(volatile int*)err) return false;
      if (global_ns() - t0 > kWaitNs) {
        *(volatile int*)err = 1;
        return false;
      }
    }
  }
}
// The same for all lanes of a warp, which then agree.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* err) {
  const bool ok = wait_or_give_up(bar, parity, err);
  return __all_sync(0xffffffffu, ok);
}
// Bounded wait that records nothing (teardown).
__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity) && global_ns() - t0 < kWaitNs) {
  }
}

// The sequence every role walks: the pipeline's units (u = vcta + j *
// nvcta), each one's passes of at most KN tokens, each pass's stages
// [kb, ke) (all of K, or the unit's part of it).
struct Unit {
  bool ok;
  int e, mt, pos, cnt, ks, kb, ke;
};
__device__ __forceinline__ int kspl_of(const Mx8Args& a) { return a.kspl > 1 ? a.kspl : 1; }
// Only the one-token phase kernels (token tile 16) split K; the batch GEMM's
// instantiations compile without it.
constexpr int kSplitKN = 16;
template <int P, bool SPLIT>
__device__ __forceinline__ Unit unit_at(const Mx8Args& a, const Item* items, int u) {
  Unit w;
  int item;
  if constexpr (SPLIT) {
    const int ksp = kspl_of(a), per_item = a.MT * ksp;
    item = u / per_item;
    const int rem = u - item * per_item;
    w.mt = rem / ksp;
    w.ks = rem - w.mt * ksp;
    const int nks = a.K / kKS;
    w.kb = nks * w.ks / ksp;
    w.ke = nks * (w.ks + 1) / ksp;
  } else {
    item = u / a.MT;
    w.mt = u - item * a.MT;
    w.ks = 0;
    w.kb = 0;
    w.ke = a.K / kKS;
    items = a.items;
  }
  const Item it = items[item];
  w.e = it.e;
  w.pos = it.pos;
  w.cnt = it.cnt;
  w.ok = (unsigned)it.e < (unsigned)a.E && it.cnt >= 1 && it.pos >= 0 &&
         it.pos + it.cnt <= a.nassign &&
         (it.pos + it.cnt) * P + (box_rows(P) > 32 ? box_rows(P) : 32) <= a.rows_cap;
  return w;
}

// ---------------------------------------------------------------------------
// roles
// ---------------------------------------------------------------------------

// Where one pipeline (a TMA warp, an MMA warp, four epilogue warps) of the
// one-token phase kernels works: its index among the grid's pipelines and the
// selection it reads (a copy in shared memory at gate/up). The batch GEMM's
// roles walk their units from the block index instead: a start and stride
// read from here cost its gate/up 3%.
struct Pipe {
  int vcta, nvcta;
  const Item* items;
  const int32_t* sorted;
};

template <int MODE, int KN, int P>
__device__ void role_tma(const Mx8Args& a, int n_units, uint8_t* smem,
                         Bars<Geo<MODE, KN, P>::S, Geo<MODE, KN, P>::NACC>* b, const Pipe& c) {
  using G = Geo<MODE, KN, P>;
  const int nks = a.K / kKS;
  uint32_t g = 0;
  uint32_t armed = 0u, last_par = 0u;
  bool ok = true;
  const uint64_t pol = l2_evict_first_policy();
  // (the batch GEMM: one pipeline a CTA, its units blockIdx.x + j gridDim.x)
  const int u0 = KN == kSplitKN ? c.vcta : (int)blockIdx.x;
  const int du = KN == kSplitKN ? c.nvcta : (int)gridDim.x;
  for (int u = u0; u < n_units && ok; u += du) {
    const Unit w = unit_at<P, KN == kSplitKN>(a, c.items, u);
    if (!w.ok) continue;
    const uint8_t* span = a.arena + (size_t)w.e * a.span_bytes;
    for (int tb = 0; tb < w.cnt && ok; tb += KN / P) {
      const int nr = min(KN / P, w.cnt - tb) * P;  // B rows of the pass (tokens x planes)
      constexpr int BR = G::BR;
      static_assert(KN % BR == 0, "B boxes of a pass");
      const int nb = (nr + BR - 1) / BR;
      const int row = (w.pos + tb) * P;
      const int kb = KN == kSplitKN ? w.kb : 0, ke = KN == kSplitKN ? w.ke : nks;
      for (int ks = kb; ks < ke; ++ks, ++g) {
        const uint32_t s = g % G::S, ph = (g / G::S) & 1u;
        if (!wait_or_give_up(&b->empty[s], ph ^ 1u, &b->err)) { ok = false; break; }
        uint64_t* full = &b->full[s];
        mbar_arrive_expect_tx(full, kATx + G::RawSf * kSfBytes + nb * BR * kKS + kSfBytes);
        uint8_t* as = smem + G::offA + (size_t)s * kABytes;
        uint8_t* raw = smem + G::offSfRaw + (size_t)s * G::RawSf * kSfBytes;
        if (MODE == 0) {
          // 64 gate rows into operand rows 0-63, the same 64 up rows into
          // rows 64-127; both 128-row tiles' scale chunks
          const int tile = w.mt >> 1, r0 = kHalfRows * (w.mt & 1);
          tma5d_stream(as, &a.amap0, r0, ks, tile, w.e, full, pol);
          tma5d_stream(as + kABytes / 2, &a.amap1, r0, ks, tile, w.e, full, pol);
          bulk_g2s(raw, span + a.sfa0 + ((size_t)tile * nks + ks) * kSfBytes, kSfBytes, full,
                   pol);
          bulk_g2s(raw + kSfBytes, span + a.sfa1 + ((size_t)tile * nks + ks) * kSfBytes,
                   kSfBytes, full, pol);
        } else {
          tma5d_stream(as, &a.amap0, 0, ks, w.mt, w.e, full, pol);
          bulk_g2s(raw, span + a.sfa0 + ((size_t)w.mt * nks + ks) * kSfBytes, kSfBytes, full,
                   pol);
        }
        uint8_t* bs = smem + G::offB + (size_t)s * G::BBytes;
        for (int i = 0; i < nb; ++i)
          tma2d(bs + i * BR * kKS, &a.bmap, ks * kKS, row + BR * i, full);
        bulk_plain(smem + G::offSfb + (size_t)s * kSfBytes,
                   a.bsf + ((size_t)ks * a.rows_cap + row) * kSfRowBytes, kSfBytes, full);
        armed |= 1u << s;
        last_par = (last_par & ~(1u << s)) | (ph << s);
      }
    }
  }
  // the copies in flight land before the CTA may leave
  for (int s = 0; s < G::S; ++s)
    if (armed >> s & 1u) drain(&b->full[s], last_par >> s & 1u);
}

// The whole MMA warp walks the stages (its lanes assemble a gate/up stage's
// A scale chunk); lane 0 issues the tensor-core work.
template <int MODE, int KN, int P>
__device__ void role_mma(const Mx8Args& a, int n_units, uint8_t* smem,
                         Bars<Geo<MODE, KN, P>::S, Geo<MODE, KN, P>::NACC>* b, uint32_t tmem,
                         const Pipe& c, int lane) {
  using G = Geo<MODE, KN, P>;
  const int nks = a.K / kKS;
  uint32_t g = 0, pc = 0;
  bool ok = true;
  // (the batch GEMM: one pipeline a CTA, its units blockIdx.x + j gridDim.x)
  const int u0 = KN == kSplitKN ? c.vcta : (int)blockIdx.x;
  const int du = KN == kSplitKN ? c.nvcta : (int)gridDim.x;
  for (int u = u0; u < n_units && ok; u += du) {
    const Unit w = unit_at<P, KN == kSplitKN>(a, c.items, u);
    if (!w.ok) continue;
    for (int tb = 0; tb < w.cnt && ok; tb += KN / P, ++pc) {
      const int N = (min(KN / P, w.cnt - tb) * P + 15) & ~15;
      const uint32_t acc = pc % G::NACC;
      if (!warp_wait(&b->acce[acc], ((pc / G::NACC) & 1u) ^ 1u, &b->err)) { ok = false; break; }
      tc_fence_after();
      const int kb = KN == kSplitKN ? w.kb : 0, ke = KN == kSplitKN ? w.ke : nks;
      for (int ks = kb; ks < ke; ++ks, ++g) {
        const uint32_t s = g % G::S, ph = (g / G::S) & 1u;
        if (!warp_wait(&b->full[s], ph, &b->err)) { ok = false; break; }
        tc_fence_after();
        const uint8_t* raw = smem + G::offSfRaw + (size_t)s * G::RawSf * kSfBytes;
        const uint8_t* sfa = raw;
        if (MODE == 0) {
          // the operand's scale chunk: line i = the words of rows i and 32 + i
          // of the 64 gate rows (words 2h, 2h + 1 of the gate tile's line i,
          // h the tile half), then those of the 64 up rows
          // (in place of the gate chunk: lane i alone reads and writes line i)
          uint8_t* asm_sf = smem + G::offSfRaw + (size_t)s * G::RawSf * kSfBytes;
          const int h = w.mt & 1;
          const uint2 gw = *reinterpret_cast<const uint2*>(raw + 16 * lane + 8 * h);
          const uint2 uw = *reinterpret_cast<const uint2*>(raw + kSfBytes + 16 * lane + 8 * h);
          *reinterpret_cast<uint4*>(asm_sf + 16 * lane) = make_uint4(gw.x, gw.y, uw.x, uw.y);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          sfa = asm_sf;
        }
        if (lane == 0) {
          const uint32_t bs = smem_u32(smem + G::offB + (size_t)s * G::BBytes);
          const uint32_t as = smem_u32(smem + G::offA + (size_t)s * kABytes);
          const uint32_t col = tmem + G::sfCol + G::sfStride * s;
          // the stage's scales into tensor memory, ahead of its MMAs
          tc_cp_sf(col, sfa);
          tc_cp_sf(col + 4, smem + G::offSfb + (size_t)s * kSfBytes);
#pragma unroll
          for (int kk = 0; kk < kKS / 32; ++kk) {
            const uint32_t idesc = umma::idesc_mxf8f6f4_e2m1_e4m3(kM, N, kk, kk);
            mma_mx(tmem + acc * G::accCols, umma::smem_desc_sw128(as + 32 * kk),
                   umma::smem_desc_sw128(bs + 32 * kk), idesc, col, col + 4,
                   ks != kb || kk != 0);
          }
          tc_commit(&b->empty[s]);
        }
        __syncwarp();
      }
      if (ok && lane == 0) tc_commit(&b->accf[acc]);
    }
  }
  // every MMA issued completes before the tensor memory is freed
  if (lane == 0) {
    tc_commit(&b->fin);
    drain(&b->fin, 0);
  }
}

__device__ __forceinline__ void tmem_ld32(uint32_t addr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
      "%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
      "[%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(addr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t addr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(addr));
}

// KN consecutive accumulator columns of this warp's lanes (x32 loads, then
// an x16 for a remainder of 16); the caller waits.
template <int KN>
__device__ __forceinline__ void tmem_ld_cols(uint32_t addr, uint32_t (&v)[KN]) {
#pragma unroll
  for (int c = 0; c + 32 <= KN; c += 32)
    tmem_ld32(addr + c, *reinterpret_cast<uint32_t(*)[32]>(v + c));
  if constexpr (KN % 32 == 16) tmem_ld16(addr + KN - 16, v + KN - 16);
}

// `warp`: the warp's tensor memory lane quarter (its index mod 4).
template <int MODE, int KN, int P>
__device__ void role_epilogue(const Mx8Args& a, int n_units, uint8_t* smem,
                              Bars<Geo<MODE, KN, P>::S, Geo<MODE, KN, P>::NACC>* b,
                              uint32_t tmem, const Pipe& c, int warp, int lane) {
  using G = Geo<MODE, KN, P>;
  constexpr int TPP = KN / P;  // tokens a pass
  const int L = 32 * warp + lane;
  const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
  // gate/up: tensor memory lanes 0-63 hold the unit's 64 gate rows (warps 0,
  // 1), lanes 64-127 the same rows of up (warps 2, 3), which hand their
  // values to the gate warps through the exchange buffers
  const bool upw = MODE == 0 && warp >= 2;
  float* const xbuf = reinterpret_cast<float*>(smem + G::offX);
  uint32_t pc = 0, xk = 0;
  bool ok = true;
  // one hand-over of n values a row (up warps: give vals; gate warps: the
  // up values land in vals); false when a bounded wait gave up
  auto exchange = [&](float* vals, int n) -> bool {
    float* buf = xbuf + (size_t)(xk & 1u) * 64 * G::XW;
    bool fine = true;
    if (upw) {
      if (xk >= 2) fine = warp_wait(&b->xempty[xk & 1u], ((xk >> 1) - 1u) & 1u, &b->err);
      if (fine) {
#pragma unroll
        for (int i = 0; i < n; ++i) buf[(L - 64) * G::XW + i] = vals[i];
        __syncwarp();
        if (lane == 0) mbar_arrive(&b->xfull[xk & 1u]);
      }
    } else {
      fine = warp_wait(&b->xfull[xk & 1u], (xk >> 1) & 1u, &b->err);
      if (fine) {
#pragma unroll
        for (int i = 0; i < n; ++i) vals[i] = buf[L * G::XW + i];
        __syncwarp();
        if (lane == 0) mbar_arrive(&b->xempty[xk & 1u]);
      }
    }
    ++xk;
    return fine;
  };
  const bool split = KN == kSplitKN && kspl_of(a) > 1;
  // (the batch GEMM: one pipeline a CTA, its units blockIdx.x + j gridDim.x)
  const int u0 = KN == kSplitKN ? c.vcta : (int)blockIdx.x;
  const int du = KN == kSplitKN ? c.nvcta : (int)gridDim.x;
  for (int u = u0; u < n_units && ok; u += du) {
    const Unit w = unit_at<P, KN == kSplitKN>(a, c.items, u);
    if (!w.ok) {
      if (L == 0) atomicOr(a.err, DEV_ERR_RANGE);
      continue;
    }
    // this thread's row: gate/up, the h row of a gate warp's thread; down,
    // the output row
    const int r = MODE == 0 ? kHalfRows * w.mt + L : kM * w.mt + L;
    for (int tb = 0; tb < w.cnt && ok; tb += TPP, ++pc) {
      const int nv = min(TPP, w.cnt - tb);
      const uint32_t acc = pc % G::NACC;
      if (!warp_wait(&b->accf[acc], (pc / G::NACC) & 1u, &b->err)) { ok = false; break; }
      tc_fence_after();
      if constexpr (P == 1) {
        // (one plane: whole K only)
        for (int c0 = 0; c0 < nv; c0 += 32) {
          const int nc = min(32, nv - c0);
          // the chunk's assignment indices, one a lane, fetched together
          const int my_a = lane < nc ? a.sorted[w.pos + tb + c0 + lane] : -1;
          uint32_t v[32];
          tmem_ld32(lane_addr + acc * G::accCols + c0, v);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          if (MODE == 1) {
#pragma unroll
            for (int n = 0; n < 32; ++n) {
              if (n >= nc) break;
              const int aa = __shfl_sync(0xffffffffu, my_a, n);
              if ((unsigned)aa < (unsigned)a.nassign) {
                a.part[(size_t)aa * a.H + r] = __uint_as_float(v[n]);
              } else if (lane == 0) {
                atomicOr(a.err, DEV_ERR_RANGE);
              }
            }
          } else {
            float f[32];
#pragma unroll
            for (int n = 0; n < 32; ++n) f[n] = __uint_as_float(v[n]);
            if (!exchange(f, 32)) { ok = false; break; }
            if (!upw) {
              const int blk = 2 * w.mt + warp;  // MXFP8 block of h along I
#pragma unroll
              for (int n = 0; n < 32; ++n) {
                if (n >= nc) break;
                const float gt = __uint_as_float(v[n]);
                const float hv = gt / (1.f + expf(-gt)) * f[n];  // silu(gate) * up
                const int aa = __shfl_sync(0xffffffffu, my_a, n);
                if (a.hbuf && (unsigned)aa < (unsigned)a.nassign)
                  a.hbuf[(size_t)aa * a.I + r] = hv;
                const int sh = mx8_shared_exp(warp_max(fabsf(hv)));
                const int row = w.pos + tb + c0 + n;
                a.hq[(size_t)row * a.I + r] = (uint8_t)e4m3_rn_sat(hv * pow2f(-sh));
                if (lane == 0)
                  put_scale(a.hsf, a.hrows_cap, row, blk, (uint8_t)(sh + 127), scale_places(1));
              }
            }
          }
        }
        if (!ok) break;
      } else {
        // planes: token n's value is the sum of its P columns, in plane order
        static_assert(KN % 16 == 0 && KN <= 96 && TPP <= 32, "plane pass columns");
        const int my_a = lane < nv ? (KN == kSplitKN ? c.sorted : a.sorted)[w.pos + tb + lane] : -1;
        uint32_t v[KN];
        float gs[TPP];
        tmem_ld_cols<KN>(lane_addr + acc * G::accCols, v);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int n = 0; n < TPP; ++n) {
          float t = __uint_as_float(v[n * P]);
#pragma unroll
          for (int q = 1; q < P; ++q) t += __uint_as_float(v[n * P + q]);
          gs[n] = t;
        }
        float us[TPP];
        if (MODE == 0 && split) {
          // a part of K: every row's sum as it stands (gate rows from warps
          // 0, 1; up rows from warps 2, 3), SwiGLU after the parts are added
          const int rr = kHalfRows * w.mt + (L & (kHalfRows - 1));
#pragma unroll
          for (int n = 0; n < TPP; ++n) {
            if (n >= nv) break;
            const int aa = __shfl_sync(0xffffffffu, my_a, n);
            if ((unsigned)aa < (unsigned)a.nassign)
              a.gu_part[(((size_t)w.ks * a.nassign + aa) * 2 + (upw ? 1 : 0)) * a.I + rr] = gs[n];
            else if (lane == 0)
              atomicOr(a.err, DEV_ERR_RANGE);
          }
        } else if (MODE == 0) {
#pragma unroll
          for (int n = 0; n < TPP; ++n) us[n] = gs[n];
          if (!exchange(us, TPP)) { ok = false; break; }
        }
        if (!upw && !(MODE == 0 && split)) {
#pragma unroll
          for (int n = 0; n < TPP; ++n) {
            if (n >= nv) break;
            const int aa = __shfl_sync(0xffffffffu, my_a, n);
            if ((unsigned)aa < (unsigned)a.nassign) {
              if (MODE == 0) {
                const float gt = gs[n];
                a.hbuf[(size_t)aa * a.I + r] = gt / (1.f + expf(-gt)) * us[n];  // silu(gate) * up
              } else {
                a.part[(size_t)aa * a.H + r] = gs[n];
              }
            } else if (lane == 0) {
              atomicOr(a.err, DEV_ERR_RANGE);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b->acce[acc]);
    }
  }
}

template <int MODE, int KN, int P>
__global__ void __launch_bounds__(kThr, ctas_per_sm(MODE, P)) mx8_gemm_kernel(const __grid_constant__ Mx8Args a) {
  using G = Geo<MODE, KN, P>;
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars<G::S, G::NACC>* b = reinterpret_cast<Bars<G::S, G::NACC>*>(smem + G::offBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&b->tmem)),
                 "r"(G::TmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < G::S; ++i) {
      mbar_init(&b->full[i], 1);
      mbar_init(&b->empty[i], 1);
    }
    for (int i = 0; i < G::NACC; ++i) {
      mbar_init(&b->accf[i], 1);
      mbar_init(&b->acce[i], 4);
    }
    mbar_init(&b->fin, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b->xfull[i], 2);
      mbar_init(&b->xempty[i], 2);
    }
    b->err = 0;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&b->tmem);
  int n_items = *a.n_items;
  if (n_items < 0 || n_items > a.max_items) {
    if (threadIdx.x == 0) atomicOr(a.err, DEV_ERR_RANGE);
    n_items = n_items < 0 ? 0 : a.max_items;
  }
  const int n_units = n_items * a.MT;  // (whole K)
  const Pipe c{(int)blockIdx.x, (int)gridDim.x, a.items, a.sorted};
  if (warp < 4) {
    role_epilogue<MODE, KN, P>(a, n_units, smem, b, tmem, c, warp, lane);
  } else if (warp == kTmaWarp) {
    if (lane == 0) role_tma<MODE, KN, P>(a, n_units, smem, b, c);
  } else if (warp == kMmaWarp) {
    role_mma<MODE, KN, P>(a, n_units, smem, b, tmem, c, lane);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && b->err) atomicOr(a.err, DEV_ERR_TIMEOUT);
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(G::TmemCols)
                 : "memory");
}

// ---------------------------------------------------------------------------
// One token on a block-scaled handle, beside the shared experts
// ---------------------------------------------------------------------------

// One token's selection inside a kernel that runs its experts: the router's
// partial logits and where the selection goes.
struct SelArgs {
  const float* part;   // router partial logits [nsplit][E]; null: selected already
  int nsplit, E, k;
  int32_t* ids;        // [k] outputs, best first
  float* w;
};

// The token's top k by the whole CTA (NW warps), from the logits summed in
// plane order. Every CTA that calls gets the same selection (same sums, same
// network). Item q is the expert of rank q with its one assignment q: the
// items and the sorted list go to shared memory (sel_items, sel_sorted,
// *sel_n); with `pub` also the ids and softmax weights and the items,
// sorted list and count to global memory, followed by a fence. `scratch`:
// NW * 32 floats and as many ints. Every thread calls; on return the shared
// copies are complete after a __syncthreads.
template <int NW>
__device__ void select_one_token(const SelArgs& sel, uint8_t* scratch, Item* sel_items,
                                 int32_t* sel_sorted, int32_t* sel_n, Item* g_items,
                                 int32_t* g_sorted, int32_t* g_n, bool pub) {
  float sel_v = 0.f;
  int sel_e = 0;
  block_topk<NW>([&](int i) { return sum_planes<true>(sel.part + i, sel.E, sel.nsplit); },
                 sel.E, reinterpret_cast<float*>(scratch),
                 reinterpret_cast<int*>(scratch + NW * 32 * sizeof(float)), sel_v, sel_e);
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const float wt = pub ? selected_softmax(sel.k, sel_v) : 0.f;
    if (lane < sel.k) {
      sel_items[lane] = Item{sel_e, lane, 1, 0};
      sel_sorted[lane] = lane;
      if (pub) {
        sel.ids[lane] = sel_e;
        sel.w[lane] = wt;
        g_items[lane] = Item{sel_e, lane, 1, 0};
        g_sorted[lane] = lane;
      }
    }
    if (lane == 0) {
      *sel_n = sel.k;
      if (pub) *g_n = sel.k;
    }
    if (pub) __threadfence();
  }
}

constexpr int kPhThr = 512;
constexpr int kPhKN = kSplitKN;  // B rows a pass: the token's planes (4 of x, 5 of h), MMA N 16
template <int MODE>
struct PhGeo {
  static constexpr int P = MODE == 0 ? kPlanesX : kPlanesH;
  using G = Geo<MODE, kPhKN, P>;
  // a pipeline's share of the CTA's shared memory (the batch GEMM's layout
  // for two CTAs an SM), a multiple of 1024 bytes
  static constexpr size_t Bytes = (smem_bytes<MODE, kPhKN, P>() + 1023) & ~(size_t)1023;
};
static_assert(geo_ok<0, kPhKN, kPlanesX>() && geo_ok<1, kPhKN, kPlanesH>(), "phase pipelines");

// A decode step of one token as two phase kernels whose routed experts run
// on the block-scaled MMA: the CTAs below n_sh stream the shared experts
// (the bf16 GEMV), every other CTA runs two pipelines of the batch GEMM
// (warps 0-5 and 6-11, each with half the CTA's shared and tensor memory, as
// two CTAs an SM do in the batch GEMM) over the 16 selected experts. Gate/up
// (MODE 0): each routed CTA selects the experts itself from the router's
// partial logits (the first one publishes them), and each unit covers 1/kspl
// of K and writes its gate and up sums (SwiGLU follows once the parts are
// added, in mx8_rows_kernel). Down (MODE 1): the selection comes from the
// gate/up phase, h's planes from the kernels between. The K split evens out
// the load: 16 experts x 24 half-tiles are too few units for the routed CTAs.
template <int MODE>
__global__ void __launch_bounds__(kPhThr, 1)
    mx8_phase_kernel(const __grid_constant__ Mx8Args a, const BfvArgs sh, const SelArgs sel,
                     int n_sh) {
  constexpr int P = PhGeo<MODE>::P;
  using G = typename PhGeo<MODE>::G;
  using Bs = Bars<G::S, G::NACC>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t bfv_bars[kBfvBars];
  __shared__ Item sel_items[32];
  __shared__ int32_t sel_sorted[32];
  __shared__ int32_t sel_n;
  if ((int)blockIdx.x < n_sh) {
    // gate/up: x is complete when the grid starts; down: the shared h is
    // the gate/up phase's
    bfv_cta<MODE, 1>(sh, smem, bfv_bars, blockIdx.x, n_sh, /*wait=*/MODE == 1);
    return;
  }
  const int cta = blockIdx.x - n_sh, ncta = gridDim.x - n_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pipe = warp / 6, role = warp - 6 * pipe;  // warps 12-15 only help select
  Bs* const b0 = reinterpret_cast<Bs*>(smem + G::offBars);
  // set-up while the preceding kernel finishes: the SM's tensor memory (half
  // of it to each pipeline) and each pipeline's barriers
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&b0->tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (lane == 0 && role == 5 && pipe < 2) {
    Bs* b = reinterpret_cast<Bs*>(smem + pipe * PhGeo<MODE>::Bytes + G::offBars);
    for (int i = 0; i < G::S; ++i) {
      mbar_init(&b->full[i], 1);
      mbar_init(&b->empty[i], 1);
    }
    for (int i = 0; i < G::NACC; ++i) {
      mbar_init(&b->accf[i], 1);
      mbar_init(&b->acce[i], 4);
    }
    mbar_init(&b->fin, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b->xfull[i], 2);
      mbar_init(&b->xempty[i], 2);
    }
    b->err = 0;
    fence_barrier_init();
  }
  pdl_wait();  // gate/up: the router's partial logits; down: h's planes
  const Item* items = a.items;
  const int32_t* sorted = a.sorted;
  int n_items;
  if (MODE == 0) {
    select_one_token<kPhThr / 32>(sel, smem, sel_items, sel_sorted, &sel_n,
                                  const_cast<Item*>(a.items), const_cast<int32_t*>(a.sorted),
                                  const_cast<int32_t*>(a.n_items), cta == 0);
    // (the selection's scratch is stage memory the copies fill next)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    items = sel_items;
    sorted = sel_sorted;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (MODE == 0) {
    n_items = sel_n;
  } else {
    n_items = __ldcg(a.n_items);
    if (n_items < 0 || n_items > a.max_items) {
      if (threadIdx.x == 0) atomicOr(a.err, DEV_ERR_RANGE);
      n_items = n_items < 0 ? 0 : a.max_items;
    }
  }
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&b0->tmem);
  const int n_units = n_items * a.MT * kspl_of(a);
  if (pipe < 2) {
    uint8_t* const ps = smem + pipe * PhGeo<MODE>::Bytes;
    Bs* const pb = reinterpret_cast<Bs*>(ps + G::offBars);
    const uint32_t pt = tmem + pipe * (kTmemCols / 2);
    const Pipe c{2 * cta + pipe, 2 * ncta, items, sorted};
    if (role < 4) {
      role_epilogue<MODE, kPhKN, P>(a, n_units, ps, pb, pt, c, warp & 3, lane);
    } else if (role == 4) {
      if (lane == 0) role_tma<MODE, kPhKN, P>(a, n_units, ps, pb, c);
    } else {
      role_mma<MODE, kPhKN, P>(a, n_units, ps, pb, pt, c, lane);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const Bs* b1 = reinterpret_cast<const Bs*>(smem + PhGeo<MODE>::Bytes + G::offBars);
    if (b0->err || b1->err) atomicOr(a.err, DEV_ERR_TIMEOUT);
  }
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

// One 32-element block as P planes (P = 1: its MXFP8 rounding): plane p's
// codes (8 words, element 4 m + c in byte c of word m) and its shared
// exponent. Plane p is the MXFP8 rounding of what the planes before it left,
// each with its own block exponent, and the remainder is exact in fp32 at
// every step (the value minus its rounding), so the planes' sum reproduces
// the block up to the last remainder.
template <int P>
__device__ __forceinline__ void block_planes(float (&v)[32], uint32_t (&wq)[P][8], int (&sh)[P]) {
#pragma unroll
  for (int pl = 0; pl < P; ++pl) {
    float amax = 0.f;
#pragma unroll
    for (int m = 0; m < 32; ++m) amax = fmaxf(amax, fabsf(v[m]));
    sh[pl] = mx8_shared_exp(amax);
    const float sc = pow2f(-sh[pl]), back = pow2f(sh[pl]);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      uint32_t word = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t code = e4m3_rn_sat(v[4 * m + c] * sc);
        word |= code << (8 * c);
        if (P > 1) v[4 * m + c] -= e4m3_value(code) * back;
      }
      wq[pl][m] = word;
    }
  }
}

// A stage's four scale bytes of each plane (blocks 4 ks .. 4 ks + 3, held
// by lanes 4 g .. 4 g + 3) as one word, in the group's first lane. Every lane
// of the warp calls.
template <int P>
__device__ __forceinline__ void stage_words(const int (&sh)[P], uint32_t (&sw)[P]) {
#pragma unroll
  for (int pl = 0; pl < P; ++pl) {
    const uint32_t b0 = (uint32_t)(sh[pl] + 127);
    sw[pl] = b0 | __shfl_down_sync(0xffffffffu, b0, 1) << 8 |
             __shfl_down_sync(0xffffffffu, b0, 2) << 16 |
             __shfl_down_sync(0xffffffffu, b0, 3) << 24;
  }
}

// Writes block j of the P rows row0 .. row0 + P - 1: the codes into q
// [rows][K], and (the group's first lane) the stage words into the row-major
// scale rows sfp [rows][K/32] (a warp's words are one contiguous piece of a
// row; mx8_scale_lines_kernel then builds the GEMM's layout from them).
template <int P>
__device__ __forceinline__ void store_planes(uint8_t* q, uint8_t* sfp, int K, int row0, int j,
                                             int lane, const uint32_t (&wq)[P][8],
                                             const uint32_t (&sw)[P]) {
#pragma unroll
  for (int pl = 0; pl < P; ++pl) {
    const int row = row0 + pl;
    uint4* d = reinterpret_cast<uint4*>(q + (size_t)row * K + 32 * j);
    d[0] = make_uint4(wq[pl][0], wq[pl][1], wq[pl][2], wq[pl][3]);
    d[1] = make_uint4(wq[pl][4], wq[pl][5], wq[pl][6], wq[pl][7]);
    if ((lane & 3) == 0)
      *reinterpret_cast<uint32_t*>(sfp + (size_t)row * (K / 32) + j) = sw[pl];
  }
}

// The GEMM's stage-major, row-interleaved scale lines from row-major scale
// rows: line (ks, R) = the stage-ks words of rows R, R + 32, ... (the first
// `places` of them; the rest zero), one 16-byte store a thread, consecutive
// threads consecutive lines. Rows at or past `rows` (never written) read as
// zero words.
__global__ void __launch_bounds__(256) mx8_scale_lines_kernel(const uint8_t* __restrict__ sfp,
                                                              int nb, int rows, int lines,
                                                              int rows_cap, int places,
                                                              uint8_t* __restrict__ sf) {
  const long long n = (long long)lines * (nb / 4);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int ks = (int)(i / lines), R = (int)(i - (long long)ks * lines);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = R + 32 * q;
      w[q] = q < places && r < rows
                 ? __ldg(reinterpret_cast<const uint32_t*>(sfp + (size_t)r * nb + 4 * ks))
                 : 0u;
    }
    *reinterpret_cast<uint4*>(sf + ((size_t)ks * rows_cap + R) * 16) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// fp32 rows (h given by the caller) for the block-scaled down GEMM: block =
// item, thread = one (row, 32-column block) pair of the item. Row n of item
// i is source row sorted[pos + n] (an assignment); its P planes go to q rows
// (pos + n) P + p.
// With gu_part (gate and up sums over kspl parts of K, [kspl][nassign][2][K])
// the rows are h = SwiGLU of the parts' sums, added in part order.
template <int P>
__global__ void __launch_bounds__(256) mx8_rows_kernel(const float* src, int K, const Item* items,
                                                       const int32_t* n_items, int max_items,
                                                       const int32_t* sorted, int nassign, int E,
                                                       uint8_t* q, uint8_t* sfp, int rows_cap,
                                                       uint32_t* err, const float* gu_part,
                                                       int kspl) {
  const int i = blockIdx.x;
  int ni = *n_items;
  if (ni > max_items) ni = max_items;
  if (i >= ni) return;
  const Item it = items[i];
  if ((unsigned)it.e >= (unsigned)E || it.cnt < 1 || it.pos < 0 || it.pos + it.cnt > nassign ||
      (it.pos + it.cnt) * P + 32 > rows_cap) {
    if (threadIdx.x == 0) atomicOr(err, DEV_ERR_RANGE);
    return;
  }
  const int nblk = K / 32;  // a multiple of 4: the four blocks of a stage sit in 4 lanes
  const int lane = threadIdx.x & 31;
  // the item's (row, block) pairs, spread over the block's threads; every
  // lane of a warp runs the same iterations (the scale words are gathered
  // across lanes), lanes past the last pair only shuffle
  const int total = it.cnt * nblk;
  for (int t0 = threadIdx.x - lane; t0 < total; t0 += blockDim.x) {
    const int t = t0 + lane;
    const int n = (t < total ? t : 0) / nblk, j = (t < total ? t : 0) - n * nblk;
    const int aa = sorted[it.pos + n];
    const bool bad = (unsigned)aa >= (unsigned)nassign;
    if (bad && t < total && j == 0) atomicOr(err, DEV_ERR_RANGE);
    const bool live = t < total && !bad;
    float v[32];
    if (live && gu_part) {
      float gs[32], us[32];
#pragma unroll
      for (int m = 0; m < 32; ++m) gs[m] = us[m] = 0.f;
      for (int ks = 0; ks < kspl; ++ks) {
        const float4* pg =
            reinterpret_cast<const float4*>(gu_part + ((size_t)ks * nassign + aa) * 2 * K + 32 * j);
        const float4* pu = pg + K / 4;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 f = pg[c], g = pu[c];
          gs[4 * c] += f.x;
          gs[4 * c + 1] += f.y;
          gs[4 * c + 2] += f.z;
          gs[4 * c + 3] += f.w;
          us[4 * c] += g.x;
          us[4 * c + 1] += g.y;
          us[4 * c + 2] += g.z;
          us[4 * c + 3] += g.w;
        }
      }
#pragma unroll
      for (int m = 0; m < 32; ++m) v[m] = gs[m] / (1.f + expf(-gs[m])) * us[m];  // silu(gate) * up
    } else if (live) {
      const float4* p = reinterpret_cast<const float4*>(src + (size_t)aa * K + 32 * j);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 f = p[c];
        v[4 * c] = f.x;
        v[4 * c + 1] = f.y;
        v[4 * c + 2] = f.z;
        v[4 * c + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int m = 0; m < 32; ++m) v[m] = 0.f;
    }
    uint32_t wq[P][8];
    int sh[P];
    block_planes<P>(v, wq, sh);
    uint32_t sw[P];
    stage_words<P>(sh, sw);
    if (live) store_planes<P>(q, sfp, K, (it.pos + n) * P, j, lane, wq, sw);
  }
}

// x (bf16 [T][K]) for the block-scaled gate/up GEMM, one token a CTA: its P
// planes (P = 1: its MXFP8 rounding) computed once and written to the rows
// of each of its k assignments in expert order, q rows inv[t k + j] P + p (an
// assignment left out of the grouping, inv = -1, gets none; no inv: the
// position is the assignment). Thread j of column group y: 32-column block
// 128 y + j.
template <int P>
__global__ void __launch_bounds__(128) mx8_xrows_kernel(const uint16_t* __restrict__ x, int K,
                                                        int k, const int32_t* __restrict__ inv,
                                                        int nassign, uint8_t* q, uint8_t* sfp,
                                                        int rows_cap, uint32_t* err) {
  __shared__ int dst[32];  // the token's positions in expert order (k <= 32)
  const int t = blockIdx.x;
  if ((int)threadIdx.x < k) {
    int p = inv ? inv[t * k + threadIdx.x] : t * k + threadIdx.x;
    if (p >= nassign || (p >= 0 && (p + 1) * P + max(32, box_rows(P)) > rows_cap)) {
      atomicOr(err, DEV_ERR_RANGE);
      p = -1;
    }
    dst[threadIdx.x] = p;
  }
  __syncthreads();
  const int nblk = K / 32;
  const int j = 128 * blockIdx.y + threadIdx.x, lane = threadIdx.x & 31;
  if ((j & ~31) >= nblk) return;  // a whole warp past the row
  const bool live = j < nblk;
  float v[32];
  if (live) {
    const uint4* p = reinterpret_cast<const uint4*>(x + (size_t)t * K + 32 * j);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 u = p[c];
      const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        v[8 * c + 2 * m] = __uint_as_float(wd[m] << 16);
        v[8 * c + 2 * m + 1] = __uint_as_float(wd[m] & 0xFFFF0000u);
      }
    }
  } else {
#pragma unroll
    for (int m = 0; m < 32; ++m) v[m] = 0.f;
  }
  uint32_t wq[P][8];
  int sh[P];
  block_planes<P>(v, wq, sh);
  uint32_t sw[P];
  stage_words<P>(sh, sw);
  if (!live) return;
  for (int i = 0; i < k; ++i) {
    const int p = dst[i];
    if (p >= 0) store_planes<P>(q, sfp, K, p * P, j, lane, wq, sw);
  }
}

// The same rounding on plain rows (the format's own layout): codes [rows][n],
// scales [rows][n/32]; one thread a block.
__global__ void mx8_plain_kernel(const float* v, int rows, int n, uint8_t* codes,
                                 uint8_t* scales) {
  const int nb = n / 32;
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (long long)rows * nb) return;
  const float* p = v + t * 32;
  float amax = 0.f;
  for (int m = 0; m < 32; ++m) amax = fmaxf(amax, fabsf(p[m]));
  const int sh = mx8_shared_exp(amax);
  const float sc = pow2f(-sh);
  for (int m = 0; m < 32; ++m) codes[t * 32 + m] = (uint8_t)e4m3_rn_sat(p[m] * sc);
  scales[t] = (uint8_t)(sh + 127);
}

// Canonical span <-> MXFP8-path span: the three code sections go to
// [tile][stage][row][64 bytes], the three scale sections to 512-byte chunks
// per tile and stage (or back, `inverse`). One thread a byte.
__global__ void mx8_layout_kernel(const uint8_t* src, uint8_t* dst, int n_spans, int H, int I,
                                  size_t span, int inverse) {
  const size_t q = (size_t)H * I / 2, sb = (size_t)H * I / 32;
  const size_t off_q[3] = {0, q + sb, 2 * q + 2 * sb};
  const size_t off_s[3] = {q, 2 * q + sb, 3 * q + 2 * sb};
  const int Ks[3] = {H, H, I};
  const size_t total = (size_t)n_spans * span;
  for (size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (size_t)gridDim.x * blockDim.x) {
    const size_t sp = t / span, o = t - sp * span;
    size_t canon = o, dev = o;
    for (int m = 0; m < 3; ++m) {
      if (o >= off_q[m] && o < off_q[m] + q) {
        // codes: [tile][stage][row][64 bytes]
        const size_t r0 = o - off_q[m];
        const int K = Ks[m], rb = K / 2, nks = K / kKS;
        const int r = (int)(r0 / rb), c = (int)(r0 - (size_t)r * rb);
        dev = off_q[m] + (((size_t)(r / kM) * nks + c / (kKS / 2)) * kM + r % kM) * (kKS / 2) +
              c % (kKS / 2);
        break;
      }
      if (o >= off_s[m] && o < off_s[m] + sb) {
        const size_t r0 = o - off_s[m];
        const int K = Ks[m], nb = K / 32, nks = K / kKS;
        const int r = (int)(r0 / nb), kb = (int)(r0 - (size_t)r * nb);
        const int rr = r % kM;  // row in its 128-row tile: word at 16 (rr mod 32) + 4 (rr / 32)
        dev = off_s[m] + ((size_t)(r / kM) * nks + kb / 4) * kSfBytes + 16 * (rr % 32) +
              4 * (rr / 32) + (kb & 3);
        canon = o;
        break;
      }
    }
    if (!inverse)
      dst[sp * span + dev] = src[sp * span + canon];
    else
      dst[sp * span + canon] = src[sp * span + dev];
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (!enc) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return enc;
}

int sms_mx8() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

template <int MODE, int KN, int P>
cudaError_t launch_mx8_kn(const Mx8Args& a, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    const cudaError_t e =
        cudaFuncSetAttribute(mx8_gemm_kernel<MODE, KN, P>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_bytes<MODE, KN, P>());
    if (e != cudaSuccess) return e;
    configured = true;
  }
  Mx8Args b = a;
  b.MT = MODE == 0 ? b.I / kHalfRows : b.H / kM;  // gate/up: 64-row halves; down: tiles
  const long long units = (long long)b.max_items * b.MT;
  int grid = ctas_per_sm(MODE, P) * sms_mx8();
  if (units < grid) grid = (int)(units > 0 ? units : 1);
  mx8_gemm_kernel<MODE, KN, P><<<grid, kThr, smem_bytes<MODE, KN, P>(), s>>>(b);
  return cudaGetLastError();
}

// MXFP8 (planes = 1): the token tile is 32 when the items average up to 24
// tokens (a smaller B slot leaves room for more stages, i.e. more weight
// bytes in flight), else 64 (fewer passes over each expert's weights).
// Planes: 16 tokens a pass (64 B rows of x's 4 planes, 80 of h's 5; 12
// tokens of h, N 64, leave three accumulator sets instead of two but measured
// 14% slower at batch 512: items of 13-16 tokens take a second pass over
// their weights).
template <int MODE>
cudaError_t launch_mx8(const Mx8Args& a, int planes, cudaStream_t s) {
  if (planes > 1) {
    constexpr int P = MODE == 0 ? kPlanesX : kPlanesH;
    if (planes != P) return cudaErrorInvalidValue;
    return launch_mx8_kn<MODE, 16 * P, P>(a, s);
  }
  return a.nassign <= 24LL * a.max_items ? launch_mx8_kn<MODE, 32, 1>(a, s)
                                         : launch_mx8_kn<MODE, 64, 1>(a, s);
}

}  // namespace

bool mx8_supported(int H, int I) { return H % (2 * kM) == 0 && I % kKS == 0; }

int mx8_box_rows(int planes) { return box_rows(planes); }

int mx8_rows_cap(int nassign, int planes) {
  // a stage's token scales are read as 32 rows from the pass's first, its
  // B rows as box_rows(planes) rows: neither runs past the buffer
  return nassign * planes + std::max(32, box_rows(planes));
}

bool make_mx8_maps(const uint8_t* arena, size_t span_bytes, int H, int I, int E, ChunkMap* gate,
                   ChunkMap* up, ChunkMap* down) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  const size_t q = (size_t)H * I / 2, sb = (size_t)H * I / 32;
  const size_t offs[3] = {0, q + sb, 2 * (q + sb)};
  ChunkMap* maps[3] = {gate, up, down};
  for (int m = 0; m < 3; ++m) {
    const int K = m < 2 ? H : I, rows = m < 2 ? I : H;
    // (128 codes = 64 bytes, 128 rows, K/128 stages, rows/128 tiles, E experts)
    const cuuint64_t dims[5] = {(cuuint64_t)kKS, (cuuint64_t)kM, (cuuint64_t)(K / kKS),
                                (cuuint64_t)(rows / kM), (cuuint64_t)E};
    const cuuint64_t strides[4] = {(cuuint64_t)kKS / 2, (cuuint64_t)kM * kKS / 2,
                                   (cuuint64_t)K / kKS * kM * kKS / 2, (cuuint64_t)span_bytes};
    // gate/up: 64-row halves of a tile (a unit's gate or up rows); down: tiles
    const cuuint32_t box[5] = {kKS, (cuuint32_t)(m < 2 ? kHalfRows : kM), 1, 1, 1};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (enc(reinterpret_cast<CUtensorMap*>(maps[m]), CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 5,
            const_cast<uint8_t*>(arena + offs[m]), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

bool make_mx8_row_map(const uint8_t* rows_buf, int rows_cap, int K, int planes, ChunkMap* map,
                      int box_r) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows_cap};
  const cuuint64_t strides[1] = {(cuuint64_t)K};
  const cuuint32_t box[2] = {kKS, (cuuint32_t)(box_r > 0 ? box_r : box_rows(planes))};
  const cuuint32_t es[2] = {1, 1};
  return enc(reinterpret_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
             const_cast<uint8_t*>(rows_buf), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_mx8_scale_lines(const uint8_t* sfp, int K, int rows, int rows_cap,
                                   int planes, uint8_t* sf, cudaStream_t s) {
  // a pass reads the 32 lines from its first row, which is below `rows`
  const int lines = std::min(rows_cap, rows + 32);
  const long long n = (long long)lines * (K / 128);
  const int blocks = (int)std::min<long long>((n + 255) / 256, 4096);
  mx8_scale_lines_kernel<<<blocks, 256, 0, s>>>(sfp, K / 32, rows, lines, rows_cap,
                                                scale_places(planes), sf);
  return cudaGetLastError();
}

cudaError_t launch_mx8_rows(const float* src, int K, int planes, const Item* items,
                            const int32_t* n_items, int max_items, const int32_t* sorted,
                            int nassign, int E, uint8_t* q, int rows_cap, uint8_t* sfp,
                            uint32_t* err, cudaStream_t s, const float* gu_part, int kspl) {
  if (max_items <= 0) return cudaSuccess;
  if (gu_part && (planes == 1 || kspl < 1)) return cudaErrorInvalidValue;
  auto go = [&](auto kernel) {
    kernel<<<max_items, 256, 0, s>>>(src, K, items, n_items, max_items, sorted, nassign, E, q,
                                     sfp, rows_cap, err, gu_part, kspl);
    return cudaGetLastError();
  };
  if (planes == 1) return go(mx8_rows_kernel<1>);
  if (planes == kPlanesH) return go(mx8_rows_kernel<kPlanesH>);
  return cudaErrorInvalidValue;
}

cudaError_t launch_mx8_xrows(const uint16_t* x, int K, int k, int T, const int32_t* inv,
                             int planes, uint8_t* q, int rows_cap, uint8_t* sfp, uint32_t* err,
                             cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (K % 128 || k > 32) return cudaErrorInvalidValue;
  const dim3 grid(T, (K / 32 + 127) / 128);
  auto go = [&](auto kernel) {
    kernel<<<grid, 128, 0, s>>>(x, K, k, inv, T * k, q, sfp, rows_cap, err);
    return cudaGetLastError();
  };
  if (planes == 1) return go(mx8_xrows_kernel<1>);
  if (planes == kPlanesX) return go(mx8_xrows_kernel<kPlanesX>);
  return cudaErrorInvalidValue;
}

cudaError_t launch_mx8_plain(const float* v, int rows, int n, uint8_t* codes, uint8_t* scales,
                             cudaStream_t s) {
  const long long blocks = (long long)rows * (n / 32);
  if (blocks <= 0) return cudaSuccess;
  mx8_plain_kernel<<<(unsigned)((blocks + 255) / 256), 256, 0, s>>>(v, rows, n, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_mx8_layout(const uint8_t* src, uint8_t* dst, int n_spans, int H, int I,
                              size_t span_bytes, int inverse, cudaStream_t s) {
  if (n_spans <= 0) return cudaSuccess;
  const size_t total = (size_t)n_spans * span_bytes;
  const int grid = (int)std::min<size_t>((total + 255) / 256, 8192);
  mx8_layout_kernel<<<grid, 256, 0, s>>>(src, dst, n_spans, H, I, span_bytes, inverse);
  return cudaGetLastError();
}

cudaError_t launch_mx8_gateup(const ChunkMap& gate, const ChunkMap& up, const ChunkMap& xmap,
                              const uint8_t* arena, size_t span_bytes, int H, int I,
                              const uint8_t* xsf, int rows_cap, const Item* items,
                              const int32_t* n_items, int max_items, const int32_t* sorted,
                              int E, int nassign, float* hbuf, uint8_t* hq, uint8_t* hsf,
                              int hrows_cap, int planes, uint32_t* err, cudaStream_t s) {
  // one plane: h rounded to MXFP8 (hq); planes: h as fp32 rows (hbuf)
  if (planes == 1 ? !hq : !hbuf) return cudaErrorInvalidValue;
  const size_t q = (size_t)H * I / 2, sb = (size_t)H * I / 32;
  Mx8Args a{};
  a.amap0 = gate;
  a.amap1 = up;
  a.bmap = xmap;
  a.arena = arena;
  a.span_bytes = span_bytes;
  a.sfa0 = q;
  a.sfa1 = 2 * q + sb;
  a.K = H;
  a.MT = I / kHalfRows;  // (set per geometry at launch)
  a.I = I;
  a.H = H;
  a.bsf = xsf;
  a.rows_cap = rows_cap;
  a.items = items;
  a.n_items = n_items;
  a.sorted = sorted;
  a.max_items = max_items;
  a.E = E;
  a.nassign = nassign;
  a.hbuf = hbuf;
  a.hq = hq;
  a.hsf = hsf;
  a.hrows_cap = hrows_cap;
  a.err = err;
  return launch_mx8<0>(a, planes, s);
}

cudaError_t launch_mx8_down(const ChunkMap& down, const ChunkMap& hmap, const uint8_t* arena,
                            size_t span_bytes, int H, int I, const uint8_t* hsf, int rows_cap,
                            const Item* items, const int32_t* n_items, int max_items,
                            const int32_t* sorted, int E, int nassign, float* part,
                            int planes, uint32_t* err, cudaStream_t s) {
  const size_t q = (size_t)H * I / 2, sb = (size_t)H * I / 32;
  Mx8Args a{};
  a.amap0 = down;
  a.amap1 = down;
  a.bmap = hmap;
  a.arena = arena;
  a.span_bytes = span_bytes;
  a.sfa0 = 3 * q + 2 * sb;
  a.sfa1 = a.sfa0;
  a.K = I;
  a.MT = H / kM;  // (set per geometry at launch)
  a.I = I;
  a.H = H;
  a.bsf = hsf;
  a.rows_cap = rows_cap;
  a.items = items;
  a.n_items = n_items;
  a.sorted = sorted;
  a.max_items = max_items;
  a.E = E;
  a.nassign = nassign;
  a.part = part;
  a.err = err;
  return launch_mx8<1>(a, planes, s);
}

namespace {

template <int MODE>
cudaError_t launch_phase_mx8(const Mx8Args& a, const BfvArgs& sh, const SelArgs& sel, int n_sh,
                             cudaStream_t s) {
  const int sms = sms_mx8();
  if (n_sh < 0 || n_sh >= sms || (n_sh > 0 && sh.rows <= 0)) return cudaErrorInvalidValue;
  const size_t smem =
      std::max(2 * PhGeo<MODE>::Bytes, n_sh > 0 ? bfv_smem_bytes(sh.K) : (size_t)0);
  static size_t configured = 0;
  if (configured < smem) {
    const cudaError_t e = cudaFuncSetAttribute(
        mx8_phase_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  return launch_after_previous(mx8_phase_kernel<MODE>, dim3(sms), dim3(kPhThr), smem, s, a, sh,
                               sel, n_sh);
}

}  // namespace

int mx8_phase_kspl(int H) {
  // parts of K a gate/up unit: 16 x (I/64) half-tiles are too few units for
  // ~230 routed pipelines; eight parts give each ~13
  const int nks = H / kKS;
  return std::max(1, std::min(8, nks));
}

bool mx8_phase_supported(int H, int I, int R) {
  return mx8_supported(H, I) && I % kHalfRows == 0 && (R == 0 || bfv_smem_bytes(H) <= 220 * 1024);
}

cudaError_t launch_mx8_phase_gateup(const ChunkMap& gate, const ChunkMap& up,
                                    const ChunkMap& xmap16, const uint8_t* arena,
                                    size_t span_bytes, int H, int I, const uint8_t* xsf,
                                    int rows_cap, Item* items, int32_t* n_items,
                                    int32_t* sorted, int E, int k, const float* router_part,
                                    int nsplit, int32_t* ids, float* w, float* gu_part,
                                    const uint16_t* sh_gate, const uint16_t* sh_up, int R,
                                    const uint16_t* x, float* hsh, uint32_t* err, int n_sh,
                                    cudaStream_t s) {
  if (!router_part || !gu_part || k > 32 || (R > 0 && !hsh)) return cudaErrorInvalidValue;
  const size_t q = (size_t)H * I / 2, sb = (size_t)H * I / 32;
  Mx8Args a{};
  a.amap0 = gate;
  a.amap1 = up;
  a.bmap = xmap16;
  a.arena = arena;
  a.span_bytes = span_bytes;
  a.sfa0 = q;
  a.sfa1 = 2 * q + sb;
  a.K = H;
  a.MT = I / kHalfRows;
  a.I = I;
  a.H = H;
  a.bsf = xsf;
  a.rows_cap = rows_cap;
  a.items = items;
  a.n_items = n_items;
  a.sorted = sorted;
  a.max_items = k;
  a.E = E;
  a.nassign = k;
  a.err = err;
  a.kspl = mx8_phase_kspl(H);
  a.gu_part = gu_part;
  const BfvArgs sh{sh_gate, sh_up, R, H, x, 1, hsh, err};
  const SelArgs sel{router_part, nsplit, E, k, ids, w};
  return launch_phase_mx8<0>(a, sh, sel, R > 0 ? n_sh : 0, s);
}

cudaError_t launch_mx8_phase_down(const ChunkMap& down, const ChunkMap& hmap16,
                                  const uint8_t* arena, size_t span_bytes, int H, int I,
                                  const uint8_t* hsf, int rows_cap, const Item* items,
                                  const int32_t* n_items, const int32_t* sorted, int E, int k,
                                  float* part, const uint16_t* sh_down, int R, const float* hsh,
                                  float* ysh, uint32_t* err, int n_sh, cudaStream_t s) {
  if (k > 32 || (R > 0 && (!hsh || !ysh))) return cudaErrorInvalidValue;
  const size_t q = (size_t)H * I / 2, sb = (size_t)H * I / 32;
  Mx8Args a{};
  a.amap0 = down;
  a.amap1 = down;
  a.bmap = hmap16;
  a.arena = arena;
  a.span_bytes = span_bytes;
  a.sfa0 = 3 * q + 2 * sb;
  a.sfa1 = a.sfa0;
  a.K = I;
  a.MT = H / kM;
  a.I = I;
  a.H = H;
  a.bsf = hsf;
  a.rows_cap = rows_cap;
  a.items = items;
  a.n_items = n_items;
  a.sorted = sorted;
  a.max_items = k;
  a.E = E;
  a.nassign = k;
  a.part = part;
  a.err = err;
  const BfvArgs sh{sh_down, nullptr, R > 0 ? H : 0, R > 0 ? R : I, hsh, 1, ysh, err};
  const SelArgs sel{nullptr, 0, E, k, nullptr, nullptr};
  return launch_phase_mx8<1>(a, sh, sel, R > 0 ? n_sh : 0, s);
}

}  // namespace dfm
