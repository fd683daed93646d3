/*
 * synth.h — seeded synthetic inputs for the MXFP4 routed-expert MoE layer.
 *
 * This module produces INPUTS only: random bytes, integers and normally
 * distributed numbers. It holds none of the layer's arithmetic (no decode,
 * no GEMV, no routing). Both the CPU oracle and the CUDA path are fed from it.
 *
 * Generator: SplitMix64 used as a counter-based function. For a stream key K,
 * the i-th 64-bit output is
 *     at(K, i) = mix64(K + (i + 1) * 0x9E3779B97F4A7C15)
 * where mix64 is the SplitMix64 output finaliser (Steele, Lea & Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014; constants as
 * in Vigna's public-domain splitmix64.c). Every element of every tensor is a
 * pure function of (seed, config id, layer, tensor kind, index, element), so
 * any slice — one expert span out of 896 — can be produced on its own, on the
 * host or on the device, with bit-identical results.
 *
 * Distributions (the workload recipe):
 *   - E2M1 codes: uniform over all 16 codes; packed byte j of a code tensor is
 *     byte (j % 8) (little-endian) of at(K, j / 8), i.e. two uniform nibbles.
 *   - E8M0 scales: 119 + floor(9 * u32 / 2^32) with u32 = at(K, j) >> 32, i.e.
 *     uniform over the 9 exponents {119..127} = scales 2^-8 .. 2^0.
 *   - Normal values: Box–Muller on two uniforms, computed in double with only
 *     IEEE basic operations (+ - * / sqrt) and this module's own log and cos
 *     series, compiled without FMA contraction, so that x86-64 and aarch64
 *     produce the same bits. fp32 = RNE of the double; bf16 = RNE of that fp32.
 */
#ifndef SYNTH_H
#define SYNTH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Tensor kinds (part of the stream key). */
enum {
  SYNTH_KIND_ROUTER = 1,       /* fp32 [E][H] ~ N(0, 1/H)              */
  SYNTH_KIND_SHARED_GATE = 2,  /* bf16 [Is][H] ~ N(0, 0.02^2)          */
  SYNTH_KIND_SHARED_UP = 3,    /* bf16 [Is][H]                         */
  SYNTH_KIND_SHARED_DOWN = 4,  /* bf16 [H][Is]                         */
  SYNTH_KIND_X = 5,            /* bf16 [H] per token ~ N(0, 1)         */
  SYNTH_KIND_RESIDUAL = 6,     /* bf16 [H] per token ~ N(0, 1)         */
  SYNTH_KIND_X_STREAM = 7,     /* fp64 innovations of a token stream   */
  SYNTH_KIND_EXPERT_BASE = 16  /* + tensor id 0..5 of an expert span   */
};

/* Expert span tensors in canonical order. */
enum {
  SYNTH_T_GATE_Q = 0, SYNTH_T_GATE_S = 1, SYNTH_T_UP_Q = 2,
  SYNTH_T_UP_S = 3, SYNTH_T_DOWN_Q = 4, SYNTH_T_DOWN_S = 5
};

uint64_t synth_mix64(uint64_t z);
uint64_t synth_at(uint64_t key, uint64_t i);
uint64_t synth_key(uint64_t seed, uint32_t cfg, uint32_t layer, uint32_t kind,
                   uint64_t index);

/* Byte size of one canonical expert span:
 *   gate_q [I][H/2] | gate_s [I][H/32] | up_q [I][H/2] | up_s [I][H/32] |
 *   down_q [H][I/2] | down_s [H][I/32]                                    */
size_t synth_span_bytes(int H, int I);

/* Fill n_exp consecutive canonical spans (experts e0 .. e0+n_exp-1). */
void synth_expert_spans(uint64_t seed, uint32_t cfg, uint32_t layer,
                        uint32_t e0, uint32_t n_exp, int H, int I,
                        uint8_t* dst);

/* Normal samples: element i of the stream keyed by `key`, for i in
 * [first, first + n). */
void synth_normal_f64(uint64_t key, uint64_t first, uint64_t n, double sigma,
                      double* dst);
void synth_normal_f32(uint64_t key, uint64_t first, uint64_t n, double sigma,
                      float* dst);
void synth_normal_bf16(uint64_t key, uint64_t first, uint64_t n, double sigma,
                       uint16_t* dst);

/* Uniform 64-bit words (for tests of the generator itself). */
void synth_words(uint64_t key, uint64_t first, uint64_t n, uint64_t* dst);

int synth_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
