// k_experts.cu — the routed-expert kernels: MXFP4 dequant-fused gate/up GEMV
// with SwiGLU epilogue, down GEMV, and the weighted combine.
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
//   * Persistent CTAs; a CTA holds NS "slots" = one producer warp + one
//     consumer warp per 512-column chunk. A slot owns a contiguous range of
//     tiles (16 rows x K of one expert).
//   * The producer streams each tile (K/64 groups of codes + scales, one
//     contiguous block) with cp.async.bulk into a shared-memory ring
//     (mbarriers, bounded waits).
//   * Consumers: one 16-byte lds per lane = its A fragments for 4 k-steps;
//     every 32-column MX block is accumulated by two MMAs into a temporary
//     that is scaled by 2^(s-127) (per row) in fp32 and added to the result.
//   * B (x) fragments live in registers as f16: the gate/up input is bf16,
//     exact in f16 except |x| < 2^-17 (error <= 2^-25). The down input h
//     (fp32, |h| up to ~1e5) is scaled per (token, chunk) by a power of two
//     into f16 range and split into hi and lo columns (~22 bits).
//   * An item (one expert and all its tokens) is processed in token groups of
//     8 (gate/up) or 4 (down) against the tile already in shared memory, so
//     each expert's weights cross HBM once per call.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "mxfrag.cuh"
#include "pipeline.cuh"

namespace dfm {
namespace {

constexpr int kMaxWarps = 16;
constexpr int kMaxStages = 8;
constexpr int kRedRing = 4;  // epilogue reduction ring depth
constexpr size_t kSmemBudget = 200 * 1024;

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
};

__host__ __device__ inline size_t align128(size_t v) { return (v + 127) & ~(size_t)127; }

struct SlotGeom {
  int stages;
  size_t stage_bytes, red_bytes, bytes;
};

__host__ __device__ inline SlotGeom slot_geom(int K, int NS) {
  SlotGeom g;
  const int NCH = mx_nchunks(K);
  g.stage_bytes = mx_tile_bytes(K);
  g.red_bytes = (size_t)kRedRing * NCH * 32 * 16;
  const size_t fixed = g.red_bytes + (2 * kMaxStages + 2 * kRedRing) * 8;
  const size_t per_slot = kSmemBudget / NS;
  int st = (int)((per_slot > fixed ? per_slot - fixed : 0) / g.stage_bytes);
  g.stages = st < 2 ? 2 : (st > kMaxStages ? kMaxStages : st);
  g.bytes = align128((size_t)g.stages * g.stage_bytes + fixed);
  return g;
}

__host__ __device__ inline int slots_per_cta(int K) {
  const int NCH = mx_nchunks(K);
  const int ns = kMaxWarps / (NCH + 1);
  return ns > 0 ? ns : 1;
}

// MODE 0: gate/up (K = H, 8 tokens per group), MODE 1: down (K = I, 4 tokens
// per group, columns 2t / 2t+1 = hi / lo part of token t).
template <int MODE>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) mxv_kernel(const MxvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int GT = MODE == 0 ? 8 : 4;  // tokens per group
  const int K = MODE == 0 ? a.H : a.I;
  const int NCH = mx_nchunks(K);
  const int wps = NCH + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = (blockDim.x >> 5) / wps;
  const int s = warp / wps, role = warp - s * wps;
  const SlotGeom geo = slot_geom(K, NS);
  const int S = geo.stages;
  uint8_t* base = smem + (size_t)s * geo.bytes;
  uint8_t* ring = base;
  float* red = reinterpret_cast<float*>(base + (size_t)S * geo.stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(
      reinterpret_cast<uint8_t*>(red) + geo.red_bytes);
  uint64_t* empty = full + kMaxStages;
  uint64_t* rfull = empty + kMaxStages;   // reduction entry written by all chunks
  uint64_t* rempty = rfull + kRedRing;    // reduction entry read by its finalizer

  if (role == NCH && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NCH);
    }
    for (int i = 0; i < kRedRing; ++i) {
      mbar_init(&rfull[i], NCH);
      mbar_init(&rempty[i], 1);
    }
  }
  fence_barrier_init();
  __syncthreads();

  pdl_wait();  // items, x and h come from the preceding kernels
  // every CTA is resident (one wave): the next kernel may be set up now and
  // start on each SM as this one's CTA leaves
  pdl_launch_dependents();
  const SpanLayout L = span_layout(a.H, a.I);
  const int tpi = MODE == 0 ? (2 * a.I) / 16 : a.H / 16;  // tiles per item
  const int ntiles = *a.n_items * tpi;
  const long long nslots = (long long)gridDim.x * NS;
  const long long gs = (long long)blockIdx.x * NS + s;
  const int t_begin = (int)(ntiles * gs / nslots);
  const int t_end = (int)(ntiles * (gs + 1) / nslots);
  const size_t sec_off = MODE == 0 ? L.gu : L.dn;
  const uint32_t tile_bytes = (uint32_t)mx_tile_bytes(K);

  if (role == NCH) {
    // ---------------- producer: one elected lane ----------------
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      bool ok = true;
      int cur_item = -1;
      const uint8_t* span = nullptr;
      for (int t = t_begin; t < t_end; ++t) {
        const int item = t / tpi, j = t - item * tpi;
        if (item != cur_item) {
          cur_item = item;
          span = a.arena + (size_t)a.items[item].e * a.span_bytes;
        }
        if (!mbar_wait(&empty[stage], phase ^ 1)) { ok = false; break; }
        uint8_t* dst = ring + (size_t)stage * geo.stage_bytes;
        mbar_arrive_expect_tx(&full[stage], tile_bytes);
        bulk_g2s(dst, span + sec_off + (size_t)j * tile_bytes, tile_bytes,
                 &full[stage], pol);
        ++issued;
        if (++stage == (uint32_t)S) { stage = 0; phase ^= 1; }
      }
      if (!ok) atomicOr(a.err, DEV_ERR_TIMEOUT);
      // Every copy this lane issued must land before the CTA may exit: wait
      // (bounded) for the last armed phase of each stage.
      for (int i = 0; i < S && i < issued; ++i) {
        const int n = (issued - i + S - 1) / S;
        (void)mbar_wait(&full[i], (uint32_t)((n - 1) & 1));
      }
    }
    return;
  }

  // ---------------- consumers: warp `role` = chunk c ----------------
  const int c = role;
  const int g = lane >> 2, t4 = lane & 3;
  const int nv = mx_nv(K, c);
  uint32_t stage = 0, phase = 0;
  int cur_item = -1, loaded_grp = -1, loaded_tok = -2;
  Item it{0, 0, 0, 0};
  int a_lane = -1;     // sorted[pos + lane] of the current item (cnt <= 32)
  uint32_t bx[32][2];  // B fragments, 2 registers per k-step of the chunk
  float csc = 1.f;     // down: 2^s of this lane's token (column pair)
  int n_epi = 0;
  bool ok = true;

  // assignment of token `ti` of the current item (all lanes must call)
  auto assignment = [&](int ti) -> int {
    const int v = __shfl_sync(0xffffffffu, a_lane, ti & 31);
    if (ti >= it.cnt) return -1;
    return it.cnt <= 32 ? v : a.sorted[it.pos + ti];
  };

  for (int t = t_begin; t < t_end && ok; ++t) {
    const int item = t / tpi, j = t - item * tpi;
    if (item != cur_item) {
      cur_item = item;
      it = a.items[item];
      a_lane = lane < it.cnt ? a.sorted[it.pos + lane] : -1;
    }
    ok = mbar_wait(&full[stage], phase);
    if (!ok) break;
    const uint8_t* tile = ring + (size_t)stage * geo.stage_bytes;

    for (int grp = 0; grp < it.cnt && ok; grp += GT) {
      // ---- B fragments of this token group (reloaded only when they change)
      if (item != loaded_grp >> 16 || grp != (loaded_grp & 0xFFFF)) {
        if (MODE == 0) {
          const int aa = assignment(grp + g);
          const int tok = aa >= 0 ? aa / a.k : -1;
          if (tok != loaded_tok) {
            loaded_tok = tok;
#pragma unroll
            for (int ks = 0; ks < 32; ++ks) {
              uint32_t v0 = 0u, v1 = 0u;
              if (tok >= 0 && ks < 4 * nv) {
                const uint16_t* xp = a.x + (size_t)tok * a.H + 512 * c + 16 * ks + 2 * t4;
                const uint32_t w0 = *reinterpret_cast<const uint32_t*>(xp);
                const uint32_t w1 = *reinterpret_cast<const uint32_t*>(xp + 8);
                v0 = f2_to_h2(__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xFFFF0000u));
                v1 = f2_to_h2(__uint_as_float(w1 << 16), __uint_as_float(w1 & 0xFFFF0000u));
              }
              bx[ks][0] = v0;
              bx[ks][1] = v1;
            }
          }
        } else {
          const int aa = assignment(grp + (g >> 1));
          const float* hrow = aa >= 0 ? a.hin + (size_t)aa * a.I + 512 * c + 2 * t4 : nullptr;
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
            sh = min(max(e - 14, -100), 100);
          }
          const float dn = pow2i(-sh);
          const bool lo = (g & 1) != 0;
          // pass 2: scaled f16 hi (even g) or lo (odd g) parts
#pragma unroll
          for (int ks = 0; ks < 32; ++ks) {
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

      // ---- the tile (16 rows x this chunk) against the group
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        if (v < nv) {
          const uint8_t* grp_p = tile + kGroupBytes * (8 * c + v);
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
            mma16816(d, a0, bx[4 * v + 2 * hb][0], bx[4 * v + 2 * hb][1], zero);
            mma16816(d, a1, bx[4 * v + 2 * hb + 1][0], bx[4 * v + 2 * hb + 1][1], d);
            const float sg = __uint_as_float(((sc >> (8 * hb)) & 0xFFu) << 23);
            const float sg8 = __uint_as_float(((sc >> (16 + 8 * hb)) & 0xFFu) << 23);
            acc[0] = fmaf(d[0], sg, acc[0]);
            acc[1] = fmaf(d[1], sg, acc[1]);
            acc[2] = fmaf(d[2], sg8, acc[2]);
            acc[3] = fmaf(d[3], sg8, acc[3]);
          }
        }
      }
      if (grp + GT >= it.cnt) {  // last use of this tile: release the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
      }
      if (MODE == 1) {
        // y rows g, g+8 of token t4 = (hi + lo) * 2^s
        acc[0] = (acc[0] + acc[1]) * csc;
        acc[2] = (acc[2] + acc[3]) * csc;
      }

      // ---- cross-chunk reduction through a ring of shared-memory entries;
      // the finalizer role rotates over the chunk warps
      const int r = n_epi % kRedRing, u = n_epi / kRedRing;
      if (u >= 1 && !mbar_wait(&rempty[r], (u - 1) & 1)) { ok = false; break; }
      float4* rb = reinterpret_cast<float4*>(red) + (size_t)r * NCH * 32;
      rb[c * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&rfull[r]);
      if (c == n_epi % NCH) {
        if (!mbar_wait(&rfull[r], u & 1)) { ok = false; break; }
        float4 sum = rb[lane];
        for (int cc = 1; cc < NCH; ++cc) {
          const float4 v4 = rb[cc * 32 + lane];
          sum.x += v4.x; sum.y += v4.y; sum.z += v4.z; sum.w += v4.w;
        }
        if (MODE == 0) {
          // columns 2t4, 2t4+1 = tokens grp+2t4, grp+2t4+1; rows g (gate) and
          // g+8 (up) of intermediate index 8j + g
          const int a0i = assignment(grp + 2 * t4), a1i = assignment(grp + 2 * t4 + 1);
          if (a0i >= 0) a.out[(size_t)a0i * a.I + 8 * j + g] = silu_f(sum.x) * sum.z;
          if (a1i >= 0) a.out[(size_t)a1i * a.I + 8 * j + g] = silu_f(sum.y) * sum.w;
        } else {
          const int ai = assignment(grp + t4);
          if (ai >= 0) {
            a.out[(size_t)ai * a.H + 16 * j + g] = sum.x;
            a.out[(size_t)ai * a.H + 16 * j + g + 8] = sum.z;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty[r]);
      }
      ++n_epi;
    }
    if (++stage == (uint32_t)S) { stage = 0; phase ^= 1; }
  }
  // A failed (timed-out) wait: record it and leave; every other wait of the
  // CTA is bounded too, so the rest of the slot ends on its own.
  if (!ok) atomicOr(a.err, DEV_ERR_TIMEOUT);
}

// out[t][j] = residual + sum_i w[t][i] part[t k + i][j] + ysh[t][j]
__global__ void combine_kernel(const float* __restrict__ part,
                               const float* __restrict__ w, int k, int H,
                               const float* __restrict__ ysh,
                               const uint16_t* __restrict__ residual,
                               float* __restrict__ out_f32,
                               uint16_t* __restrict__ out_bf16) {
  pdl_wait();
  const int t = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= H) return;
  float y = 0.f;
  for (int i = 0; i < k; ++i)
    y = fmaf(w[(size_t)t * k + i], part[((size_t)t * k + i) * H + j], y);
  if (ysh) y += ysh[(size_t)t * H + j];
  if (residual) y += __uint_as_float((uint32_t)residual[(size_t)t * H + j] << 16);
  if (out_f32) out_f32[(size_t)t * H + j] = y;
  if (out_bf16) out_bf16[(size_t)t * H + j] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
}

int num_sms() {
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
cudaError_t launch_mxv(const MxvArgs& a, int max_items, cudaStream_t s, int max_ctas) {
  const int K = MODE == 0 ? a.H : a.I;
  const int NCH = mx_nchunks(K);
  const int NS = slots_per_cta(K);
  const int threads = NS * (NCH + 1) * 32;
  const SlotGeom geo = slot_geom(K, NS);
  const size_t smem = (size_t)NS * geo.bytes;
  static int configured_smem[2] = {0, 0};
  if (configured_smem[MODE] < (int)smem) {
    cudaError_t e = cudaFuncSetAttribute(mxv_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured_smem[MODE] = (int)smem;
  }
  const int tpi = MODE == 0 ? (2 * a.I) / 16 : a.H / 16;
  const long long max_tiles = (long long)max_items * tpi;
  int grid = (int)((max_tiles + NS - 1) / NS);
  if (grid > num_sms()) grid = num_sms();
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  if (grid < 1) grid = 1;
  return launch_after_previous(mxv_kernel<MODE>, dim3(grid), dim3(threads), smem, s, a);
}

}  // namespace

cudaError_t launch_gateup(const uint8_t* arena, size_t span_bytes, int H,
                          int I, int k, const uint16_t* x, const Item* items,
                          const int32_t* n_items, int max_items,
                          const int32_t* sorted, float* hbuf, int /*tg*/,
                          uint32_t* err, cudaStream_t s, int max_ctas) {
  MxvArgs a{arena, span_bytes, H, I, k, x, nullptr, items, n_items, sorted, hbuf, err};
  return launch_mxv<0>(a, max_items, s, max_ctas);
}

cudaError_t launch_down(const uint8_t* arena, size_t span_bytes, int H, int I,
                        const Item* items, const int32_t* n_items,
                        int max_items, const int32_t* sorted,
                        const float* hbuf, float* part, int /*tg*/, uint32_t* err,
                        cudaStream_t s, int max_ctas) {
  MxvArgs a{arena, span_bytes, H, I, 0, nullptr, hbuf, items, n_items, sorted, part, err};
  return launch_mxv<1>(a, max_items, s, max_ctas);
}

cudaError_t launch_combine(const float* part, const float* w, int T, int k,
                           int H, const float* ysh, const uint16_t* residual,
                           float* out_f32, uint16_t* out_bf16, cudaStream_t s) {
  dim3 grid((H + 255) / 256, T);
  return launch_after_previous(combine_kernel, grid, dim3(256), 0, s, part, w, k, H, ysh,
                               residual, out_f32, out_bf16);
}

}  // namespace dfm
