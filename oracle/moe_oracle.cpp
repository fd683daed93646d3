// moe_oracle.cpp — CPU reference of the MXFP4 routed-expert MoE layer.
//
// TEST INFRASTRUCTURE (see moe_oracle.h). Plain loops, double accumulation,
// no blocking or reordering beyond the definitions. OpenMP only splits
// independent output elements across threads; every output element is
// accumulated by one thread in a fixed order, so results do not depend on
// the thread count.
#include "moe_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <utility>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// E2M1 magnitudes for the three low bits of a code; bit 3 is the sign.
// The value set {0, 0.5, 1, 1.5, 2, 3, 4, 6} is the FP4 (E2M1) element type
// of the OCP microscaling formats that the pages' experts use
// (kimi-k3-in-c blog, "先把账算明白": 4-bit values, one shared 8-bit exponent
// per 32 elements; Deltafin README credits ml_dtypes as its e2m1 reference).
const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

inline uint8_t nibble(const uint8_t* q_row, int c) {
  // element 2m in the low nibble of byte m, element 2m+1 in the high nibble
  uint8_t b = q_row[c >> 1];
  return (c & 1) ? (uint8_t)(b >> 4) : (uint8_t)(b & 15);
}

}  // namespace

extern "C" {

double orc_e2m1_value(uint8_t code) {
  double m = kE2M1[code & 7];
  return (code & 8) ? -m : m;
}

double orc_e8m0_value(uint8_t e) {
  if (e == 255) return NAN;
  return std::ldexp(1.0, (int)e - 127);
}

double orc_bf16_to_f64(uint16_t b) {
  uint32_t bits = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return (double)f;
}

uint16_t orc_f64_to_bf16(double v) {
  if (std::isnan(v)) return 0x7FC0;
  uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  double a = std::fabs(v);
  if (a == 0.0) return sign;
  if (std::isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e;
  std::frexp(a, &e);                         // a in [2^(e-1), 2^e)
  int qexp = (e - 1 >= -126) ? (e - 8) : -133;  // spacing of bf16 values near a
  double r = std::nearbyint(std::ldexp(a, -qexp));  // ties to even
  double rv = std::ldexp(r, qexp);
  if (rv > 0x1.FEp127) return (uint16_t)(sign | 0x7F80);  // overflow to inf
  float f = (float)rv;                       // exact: <= 8 significant bits
  uint32_t bits;
  std::memcpy(&bits, &f, 4);
  return (uint16_t)(sign | (bits >> 16));
}

size_t orc_span_bytes(int H, int I) {
  size_t hi = (size_t)H * (size_t)I;
  return 3 * (hi / 2 + hi / 32);
}

void orc_span_offsets(int H, int I, size_t off[6]) {
  // gate_q [I][H/2], gate_s [I][H/32], up_q, up_s, down_q [H][I/2],
  // down_s [H][I/32]: the six tensors of one expert, contiguous (Deltafin
  // README, "I/O and streaming": an expert's six tensors are one range).
  size_t hi = (size_t)H * (size_t)I;
  size_t q = hi / 2, s = hi / 32;
  off[0] = 0;
  off[1] = q;
  off[2] = q + s;
  off[3] = 2 * q + s;
  off[4] = 2 * q + 2 * s;
  off[5] = 3 * q + 2 * s;
}

void orc_mx_dequant(const uint8_t* q, const uint8_t* s, int rows, int cols,
                    double* W) {
  for (int r = 0; r < rows; ++r) {
    const uint8_t* qr = q + (size_t)r * (cols / 2);
    const uint8_t* sr = s + (size_t)r * (cols / 32);
    for (int c = 0; c < cols; ++c)
      W[(size_t)r * cols + c] =
          orc_e2m1_value(nibble(qr, c)) * orc_e8m0_value(sr[c / 32]);
  }
}

void orc_mx_gemv(const uint8_t* q, const uint8_t* s, int rows, int cols,
                 const double* x, double* y) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    const uint8_t* qr = q + (size_t)r * (cols / 2);
    const uint8_t* sr = s + (size_t)r * (cols / 32);
    double acc = 0.0;
    for (int c = 0; c < cols; ++c)
      acc += orc_e2m1_value(nibble(qr, c)) * orc_e8m0_value(sr[c / 32]) * x[c];
    y[r] = acc;
  }
}

void orc_router_logits(const float* Wr, int E, int H, const uint16_t* x_bf16,
                       int T, double* logits) {
  std::vector<double> x((size_t)H);
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < H; ++j) x[j] = orc_bf16_to_f64(x_bf16[(size_t)t * H + j]);
#pragma omp parallel for schedule(static)
    for (int e = 0; e < E; ++e) {
      const float* w = Wr + (size_t)e * H;
      double acc = 0.0;
      for (int j = 0; j < H; ++j) acc += (double)w[j] * x[j];
      logits[(size_t)t * E + e] = acc;
    }
  }
}

void orc_topk_softmax(const double* logits, int T, int E, int k, int32_t* ids,
                      double* w) {
  std::vector<std::pair<double, int>> v((size_t)E);
  for (int t = 0; t < T; ++t) {
    const double* l = logits + (size_t)t * E;
    for (int e = 0; e < E; ++e) v[e] = {l[e], e};
    std::sort(v.begin(), v.end(),
              [](const std::pair<double, int>& a, const std::pair<double, int>& b) {
                if (a.first != b.first) return a.first > b.first;
                return a.second < b.second;
              });
    double lmax = v[0].first, z = 0.0;
    for (int i = 0; i < k; ++i) z += std::exp(v[i].first - lmax);
    for (int i = 0; i < k; ++i) {
      ids[(size_t)t * k + i] = v[i].second;
      w[(size_t)t * k + i] = std::exp(v[i].first - lmax) / z;
    }
  }
}

double orc_silu(double g) { return g / (1.0 + std::exp(-g)); }

void orc_expert_gateup(const uint8_t* span, int H, int I, const double* x,
                       double* h) {
  size_t off[6];
  orc_span_offsets(H, I, off);
  std::vector<double> g((size_t)I), u((size_t)I);
  orc_mx_gemv(span + off[0], span + off[1], I, H, x, g.data());
  orc_mx_gemv(span + off[2], span + off[3], I, H, x, u.data());
  for (int r = 0; r < I; ++r) h[r] = orc_silu(g[r]) * u[r];
}

void orc_expert_down(const uint8_t* span, int H, int I, const double* h,
                     double* y) {
  size_t off[6];
  orc_span_offsets(H, I, off);
  orc_mx_gemv(span + off[4], span + off[5], H, I, h, y);
}

void orc_expert_ffn(const uint8_t* span, int H, int I, const double* x,
                    double* y) {
  std::vector<double> h((size_t)I);
  orc_expert_gateup(span, H, I, x, h.data());
  orc_expert_down(span, H, I, h.data(), y);
}

static void bf16_gemv(const uint16_t* W, int rows, int cols, const double* x,
                      double* y) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    const uint16_t* wr = W + (size_t)r * cols;
    double acc = 0.0;
    for (int c = 0; c < cols; ++c) acc += orc_bf16_to_f64(wr[c]) * x[c];
    y[r] = acc;
  }
}

void orc_shared_ffn(const uint16_t* gate, const uint16_t* up,
                    const uint16_t* down, int H, int Is, const double* x,
                    double* y) {
  std::vector<double> g((size_t)Is), u((size_t)Is), h((size_t)Is);
  bf16_gemv(gate, Is, H, x, g.data());
  bf16_gemv(up, Is, H, x, u.data());
  for (int r = 0; r < Is; ++r) h[r] = orc_silu(g[r]) * u[r];
  bf16_gemv(down, H, Is, h.data(), y);
}

int orc_group(const int32_t* ids, int T, int k, int E, int32_t* offs,
              int32_t* tok, int32_t* slot) {
  std::vector<int32_t> count((size_t)E, 0);
  for (int a = 0; a < T * k; ++a) count[ids[a]] += 1;
  offs[0] = 0;
  int distinct = 0;
  for (int e = 0; e < E; ++e) {
    offs[e + 1] = offs[e] + count[e];
    distinct += count[e] > 0;
  }
  std::vector<int32_t> fill(offs, offs + E);
  for (int a = 0; a < T * k; ++a) {  // ascending a keeps each segment ordered
    int p = fill[ids[a]]++;
    tok[p] = a / k;
    slot[p] = a % k;
  }
  return distinct;
}

void orc_rmsnorm_bf16(const uint16_t* x, int T, int H, double eps,
                      uint16_t* xn) {
  for (int t = 0; t < T; ++t) {
    const uint16_t* xr = x + (size_t)t * H;
    double ss = 0.0;
    for (int j = 0; j < H; ++j) {
      double v = orc_bf16_to_f64(xr[j]);
      ss += v * v;
    }
    double denom = std::sqrt(ss / (double)H + eps);
    for (int j = 0; j < H; ++j)
      xn[(size_t)t * H + j] = orc_f64_to_bf16(orc_bf16_to_f64(xr[j]) / denom);
  }
}

// ---- MXFP8 (OCP microscaling, E4M3 elements) ----------------------------
// The element type is FP8 E4M3 as the OCP 8-bit floating point format
// defines it: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, subnormals
// at exponent field 0, no infinities, and S.1111.111 the only NaN; the largest
// finite magnitude is 1.75 * 2^8 = 448. The block scale is E8M0 (2^(e-127)).
// The conversion of a block follows the OCP MX specification's recipe: the
// shared exponent is floor(log2(max|v|)) minus the element type's largest
// exponent (8 for E4M3), and each element is v / 2^shared rounded to the
// element type.

double orc_e4m3_value(uint8_t code) {
  const int sgn = code >> 7, ex = (code >> 3) & 15, man = code & 7;
  if (ex == 15 && man == 7) return NAN;
  const double mag = ex == 0 ? std::ldexp((double)man, -9)              // 2^-6 * m/8
                             : std::ldexp(1.0 + man / 8.0, ex - 7);
  return sgn ? -mag : mag;
}

uint8_t orc_e4m3_from_f64(double v) {
  const uint8_t sgn = std::signbit(v) ? 0x80 : 0x00;
  double a = std::fabs(v);
  if (a >= 448.0) return (uint8_t)(sgn | 0x7E);  // saturate: 1.110 * 2^8
  // spacing of E4M3 values near a: 2^(e - 3) for a in [2^e, 2^(e+1)),
  // e >= -6; the subnormal spacing 2^-9 below 2^-6
  int e = -7;
  if (a >= std::ldexp(1.0, -6)) {
    std::frexp(a, &e);  // a in [2^(e-1), 2^e)
    e -= 1;
  }
  const int q = e >= -6 ? e - 3 : -9;
  const double r = std::nearbyint(std::ldexp(a, -q));  // ties to even
  const double rv = std::ldexp(r, q);
  if (rv > 448.0) return (uint8_t)(sgn | 0x7E);
  // encode rv exactly
  if (rv < std::ldexp(1.0, -6)) return (uint8_t)(sgn | (uint8_t)std::ldexp(rv, 9));
  int re;
  const double fr = std::frexp(rv, &re);  // rv = fr * 2^re, fr in [0.5, 1)
  const int ex = re - 1 + 7;
  const int man = (int)std::ldexp(fr * 2.0 - 1.0, 3);
  return (uint8_t)(sgn | (ex << 3) | man);
}

uint8_t orc_mxfp8_block(const double* v, uint8_t* codes) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[i]));
  int shared = -127;
  if (amax > 0.0) {
    int e;
    std::frexp(amax, &e);  // amax in [2^(e-1), 2^e): floor(log2) = e - 1
    shared = std::min(127, std::max(-127, e - 1 - 8));
  }
  for (int i = 0; i < 32; ++i) codes[i] = orc_e4m3_from_f64(std::ldexp(v[i], -shared));
  return (uint8_t)(shared + 127);
}

void orc_mxfp8_quantize(const double* v, int rows, int n, uint8_t* codes,
                        uint8_t* scales) {
  for (int r = 0; r < rows; ++r)
    for (int b = 0; b < n / 32; ++b)
      scales[(size_t)r * (n / 32) + b] =
          orc_mxfp8_block(v + (size_t)r * n + 32 * b, codes + (size_t)r * n + 32 * b);
}

void orc_mxfp8_dequant(const uint8_t* codes, const uint8_t* scales, int rows,
                       int n, double* v) {
  for (int r = 0; r < rows; ++r)
    for (int i = 0; i < n; ++i)
      v[(size_t)r * n + i] = orc_e4m3_value(codes[(size_t)r * n + i]) *
                             orc_e8m0_value(scales[(size_t)r * (n / 32) + i / 32]);
}

int orc_moe_layer(const orc_layer* L, const uint16_t* x, int T,
                  const uint16_t* residual, double* out, int32_t* ids,
                  double* w, double* logits_out, double* routed_out,
                  double* shared_out) {
  const int H = L->H, E = L->E, k = L->k, I = L->I;
  std::vector<double> logits((size_t)T * E);
  orc_router_logits(L->router, E, H, x, T, logits.data());
  orc_topk_softmax(logits.data(), T, E, k, ids, w);
  if (logits_out) std::copy(logits.begin(), logits.end(), logits_out);

  // fetch each needed expert once, from this thread
  std::map<int, const uint8_t*> spans;
  for (int a = 0; a < T * k; ++a) {
    int e = ids[a];
    if (spans.count(e)) continue;
    const uint8_t* p = L->get_span(L->ctx, L->layer, e);
    if (!p) return -1;
    spans[e] = p;
  }

  std::vector<double> xd((size_t)H), y((size_t)H), routed((size_t)H),
      shared((size_t)H);
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < H; ++j) xd[j] = orc_bf16_to_f64(x[(size_t)t * H + j]);
    std::fill(routed.begin(), routed.end(), 0.0);
    for (int i = 0; i < k; ++i) {
      int e = ids[(size_t)t * k + i];
      double wi = w[(size_t)t * k + i];
      orc_expert_ffn(spans[e], H, I, xd.data(), y.data());
      for (int j = 0; j < H; ++j) routed[j] += wi * y[j];
    }
    std::fill(shared.begin(), shared.end(), 0.0);
    for (int s = 0; s < L->n_shared; ++s) {
      orc_shared_ffn(L->shared_gate[s], L->shared_up[s], L->shared_down[s], H,
                     L->Is, xd.data(), y.data());
      for (int j = 0; j < H; ++j) shared[j] += y[j];
    }
    for (int j = 0; j < H; ++j) {
      double r = residual ? orc_bf16_to_f64(residual[(size_t)t * H + j]) : 0.0;
      out[(size_t)t * H + j] = r + (routed[j] + shared[j]);
      if (routed_out) routed_out[(size_t)t * H + j] = routed[j];
      if (shared_out) shared_out[(size_t)t * H + j] = shared[j];
    }
  }
  return 0;
}

int orc_moe_stack(const orc_layer* layers, int nl, const uint16_t* x, int T,
                  double eps, uint16_t* x_out, double* last_f64, int32_t* ids,
                  double* w, double* logits) {
  const int H = layers[0].H, k = layers[0].k, E = layers[0].E;
  std::vector<uint16_t> cur(x, x + (size_t)T * H), xn((size_t)T * H);
  std::vector<double> out((size_t)T * H);
  for (int l = 0; l < nl; ++l) {
    orc_rmsnorm_bf16(cur.data(), T, H, eps, xn.data());
    int rc = orc_moe_layer(&layers[l], xn.data(), T, cur.data(), out.data(),
                           ids + (size_t)l * T * k, w + (size_t)l * T * k,
                           logits ? logits + (size_t)l * T * E : nullptr,
                           nullptr, nullptr);
    if (rc) return rc;
    for (size_t j = 0; j < out.size(); ++j) cur[j] = orc_f64_to_bf16(out[j]);
  }
  std::copy(cur.begin(), cur.end(), x_out);
  if (last_f64) std::copy(out.begin(), out.end(), last_f64);
  return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

}  // extern "C"
