/*
 * moe_oracle.h — CPU reference of the MXFP4 routed-expert MoE layer.
 *
 * TEST INFRASTRUCTURE. This is the plain, slow, obviously correct oracle that
 * the CUDA library is checked against. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the library never does. It shares
 * no code with the CUDA path. All floating-point arithmetic is in double;
 * bf16 and fp32 inputs are widened exactly.
 *
 * What it computes (one MoE layer of a Kimi-K3-shaped model at decode):
 *   - Router: logit[t][e] = sum_j Wr[e][j] * x[t][j], then the top k of E
 *     experts ("the router picks 16 of 896"; Deltafin analysis §5.1,
 *     Deltafin README "How it works").
 *   - Weights over the selected experts: softmax of their logits.
 *   - Each selected expert: SwiGLU FFN y = Wd (silu(Wg x) * (Wu x)) with
 *     MXFP4 weights W[r][c] = E2M1(q[r][c]) * 2^(s[r][c/32] - 127)
 *     ("4-bit mantissa plus one 8-bit exponent shared by 32 elements",
 *     kimi-k3-in-c blog, "先把账算明白"; the fused dequant+GEMV of the
 *     Deltafin README, "Techniques / Compute").
 *   - Output: residual + sum_i w_i y_i + sum_s shared_s(x) ("add the two
 *     shared experts", Deltafin analysis §5.1).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 * low nibble = even element; 32-element blocks along the input dimension;
 * SwiGLU as silu(gate) * up; shared experts unweighted; ids in descending
 * logit order with ties to the lower id.
 *
 * Parity pins: every function is pinned by the CPU tests against the pages'
 * printed byte arithmetic, ml_dtypes' E2M1 decode, closed forms, library
 * routines (numpy matmul / sort) and brute force on tiny inputs.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- formats ---------------------------------------------------------- */
double orc_e2m1_value(uint8_t code);      /* explicit 16-entry table       */
double orc_e8m0_value(uint8_t e);         /* 2^(e-127); e = 255 -> NaN      */
double orc_bf16_to_f64(uint16_t b);       /* exact widening                 */
uint16_t orc_f64_to_bf16(double v);       /* round to nearest, ties to even */
size_t orc_span_bytes(int H, int I);      /* 3 * H * I * 17 / 32            */
/* offsets of gate_q, gate_s, up_q, up_s, down_q, down_s within a span */
void orc_span_offsets(int H, int I, size_t off[6]);

/* ---- MXFP4 matrices (q: [rows][cols/2], s: [rows][cols/32]) ------------ */
void orc_mx_dequant(const uint8_t* q, const uint8_t* s, int rows, int cols,
                    double* W /* [rows][cols] */);
/* fused decode-and-accumulate: y[r] = sum_c W[r][c] x[c] */
void orc_mx_gemv(const uint8_t* q, const uint8_t* s, int rows, int cols,
                 const double* x, double* y);

/* ---- steps -------------------------------------------------------------- */
void orc_router_logits(const float* Wr, int E, int H, const uint16_t* x_bf16,
                       int T, double* logits /* [T][E] */);
/* ids in descending logit order, ties to the lower id; w = softmax over the
 * k selected logits. */
void orc_topk_softmax(const double* logits, int T, int E, int k,
                      int32_t* ids /* [T][k] */, double* w /* [T][k] */);
double orc_silu(double g);
/* h[r] = silu((Wg x)[r]) * (Wu x)[r], r < I */
void orc_expert_gateup(const uint8_t* span, int H, int I, const double* x,
                       double* h);
/* y[o] = sum_r Wd[o][r] h[r], o < H */
void orc_expert_down(const uint8_t* span, int H, int I, const double* h,
                     double* y);
void orc_expert_ffn(const uint8_t* span, int H, int I, const double* x,
                    double* y);
/* bf16 shared expert: y = Wd (silu(Wg x) * (Wu x)) */
void orc_shared_ffn(const uint16_t* gate, const uint16_t* up,
                    const uint16_t* down, int H, int Is, const double* x,
                    double* y);
/* counting sort of the T*k assignments a = t*k + j by expert id:
 * offs[e]..offs[e+1] is expert e's segment, ordered by a; tok/slot give
 * (t, j) of each entry. Returns the number of distinct experts. */
int orc_group(const int32_t* ids, int T, int k, int E, int32_t* offs,
              int32_t* tok, int32_t* slot);
/* y = x / sqrt(mean(x^2) + eps), unit gain, in double; result rounded to
 * bf16 (the input the next layer sees) */
void orc_rmsnorm_bf16(const uint16_t* x, int T, int H, double eps,
                      uint16_t* xn);

/* ---- MXFP8 activations (the lossy variant) ------------------------------
 * Kimi K3 is trained quantisation-aware with MXFP4 weights and MXFP8
 * activations (Deltafin analysis, section 2.1). The activation format is the
 * OCP microscaling one: blocks of 32 elements along the contraction, each an
 * FP8 E4M3 value, sharing one E8M0 exponent. */
double orc_e4m3_value(uint8_t code);   /* bias 7, no inf; 0x7F / 0xFF NaN  */
/* Nearest E4M3 code of v, ties to even, |v| above 448 saturating to 448
 * (E4M3 has no inf); v finite. */
uint8_t orc_e4m3_from_f64(double v);
/* One block: X = 2^(floor(log2(max|v|)) - 8), exponent clamped to
 * [-127, 127] (an all-zero block takes 2^-127); codes[i] =
 * e4m3(v[i] / X), scale = the E8M0 code of X. v finite. Returns the scale. */
uint8_t orc_mxfp8_block(const double* v, uint8_t* codes);
/* Rows of n elements (n % 32 == 0): codes [rows][n], scales [rows][n/32]. */
void orc_mxfp8_quantize(const double* v, int rows, int n, uint8_t* codes,
                        uint8_t* scales);
/* The dequantised values: codes[i] * 2^(scale - 127). */
void orc_mxfp8_dequant(const uint8_t* codes, const uint8_t* scales, int rows,
                       int n, double* v);

/* ---- whole layer / stack ------------------------------------------------ */
/* Expert spans are fetched on demand, once per needed expert, from the
 * calling thread: get_span(ctx, layer, expert) returns a canonical span. */
typedef const uint8_t* (*orc_get_span_fn)(void* ctx, int layer, int expert);

typedef struct {
  int H, E, k, I, n_shared, Is;
  const float* router;                 /* [E][H]                         */
  const uint16_t* const* shared_gate;  /* n_shared pointers, [Is][H] bf16 */
  const uint16_t* const* shared_up;    /* [Is][H]                        */
  const uint16_t* const* shared_down;  /* [H][Is]                        */
  orc_get_span_fn get_span;
  void* ctx;
  int layer;
} orc_layer;

/* out[t][:] = (residual ? residual[t] : 0) + routed + shared, in double.
 * Optional outputs: logits [T][E], routed [T][H], shared_y [T][H].
 * Returns 0, or -1 if get_span returned NULL. */
int orc_moe_layer(const orc_layer* L, const uint16_t* x, int T,
                  const uint16_t* residual, double* out, int32_t* ids,
                  double* w, double* logits, double* routed, double* shared_y);

/* Stack of nl layers: per layer xn = bf16(rmsnorm(x)); x = bf16(x + MoE(xn)).
 * x_out = final bf16 x; last_f64 = x + MoE(xn) of the last layer before
 * rounding; ids/w are [nl][T][k]; logits (nullable) [nl][T][E]. */
int orc_moe_stack(const orc_layer* layers, int nl, const uint16_t* x, int T,
                  double eps, uint16_t* x_out, double* last_f64, int32_t* ids,
                  double* w, double* logits);

int orc_num_threads(void);
void orc_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
