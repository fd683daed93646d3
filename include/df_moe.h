/*
 * df_moe.h — C ABI of the GB300 MXFP4 routed-expert MoE layer (sm_103a).
 *
 * The operation is the decode-time sparse Mixture-of-Experts layer of a
 * Kimi-K3-shaped model, as the pages walk through one token (Deltafin
 * analysis "Kimi K3極限部署技術解析", §5.1; Deltafin README, "How it works"):
 * the router scores E experts and picks the top k (896 and 16 in K3), each
 * picked expert runs a SwiGLU FFN whose weights are MXFP4, the expert outputs
 * are weighted and summed, and the shared experts are added.
 *
 *   logits[t][e] = sum_j Wr[e][j] x[t][j]                     (fp32)
 *   ids[t]       = top-k of logits[t], descending, ties -> lower id
 *   w[t][i]      = softmax over the k selected logits
 *   y[t]         = sum_i w[t][i] Wd_e (silu(Wg_e x) * (Wu_e x)),  e = ids[t][i]
 *                + sum_s Wd_s (silu(Wg_s x) * (Wu_s x))          (shared, bf16)
 *   out[t]       = residual[t] + y[t]
 *
 * MXFP4 (kimi-k3-in-c blog "2.78T 模型塞进 8GB 内存…", section 先把账算明白):
 * W[r][c] = E2M1(q[r][c]) * 2^(s[r][c/32] - 127), 4-bit codes with one 8-bit
 * exponent per 32 elements along the input dimension, 0.53125 B/weight.
 *
 * Conventions of every call:
 *   - Pointers marked "device" are CUDA device pointers on the handle's
 *     device; "host" pointers are ordinary host memory (pinned is faster).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is
 *     enqueued asynchronously on it unless the call says otherwise.
 *   - Every call returns DF_MOE_OK (0) or a negative DF_MOE_E* code; the
 *     message is available from df_moe_last_error(handle) (or, for calls that
 *     fail before a handle exists, df_moe_last_error(NULL), thread-local).
 *   - bf16 tensors are passed as 16-bit words (uint16_t / void*).
 *   - The library owns all weight storage and its workspace. The caller owns
 *     every input and output buffer.
 *   - No call is safe to run concurrently with another call on the same
 *     handle (they share workspace).
 */
#ifndef DF_MOE_H
#define DF_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DF_MOE_API __attribute__((visibility("default")))
#else
#define DF_MOE_API
#endif

#define DF_MOE_OK 0
#define DF_MOE_EINVAL (-1)   /* invalid argument                              */
#define DF_MOE_ENOMEM (-2)   /* device or host allocation failed              */
#define DF_MOE_ECUDA (-3)    /* a CUDA runtime call failed                    */
#define DF_MOE_ESTATE (-4)   /* forward before every weight was loaded        */
#define DF_MOE_ERANGE (-5)   /* T > max_tokens, index out of range            */
#define DF_MOE_ETIMEOUT (-6) /* a bounded device-side wait gave up            */
#define DF_MOE_EDEVICE (-7)  /* a device-side check recorded an error         */

/* Stack mode: before every layer x is RMS-normalised (unit gain, rms_eps) and
 * rounded to bf16; after it the layer output is added to x and rounded to
 * bf16. `out` is the final x. */
#define DF_MOE_STACK_RMSNORM_RESIDUAL 1u
/* Flag bit 2u is reserved: create rejects it as an unknown flag. */
/* Batches above the decode range (T > 8) run the routed experts on the
 * register-fragment (mma.sync) kernels of the decode chain instead of the
 * default grouped GEMMs on the 5th-generation tensor cores (tcgen05, fp32
 * accumulators in tensor memory). For comparison; same results within the
 * stated tolerances. */
#define DF_MOE_PREFILL_MMA_SYNC 4u
/* The lossy MXFP8-activation variant: the inputs of the routed experts (x
 * into gate/up, h into down) are rounded to MXFP8 — blocks of 32 along the
 * contraction, E4M3 elements sharing an E8M0 exponent, the exponent
 * floor(log2 max|v|) - 8, elements rounded to nearest even and saturated at
 * 448 — and the experts run as grouped GEMMs on the 5th-generation tensor
 * cores' block-scaled MXFP4 x MXFP8 MMA. Kimi K3 is trained with MXFP8
 * activations (Deltafin analysis, section 2.1); the pages' reference runs
 * keep activations exact, and so does every handle without this flag. The
 * router and the shared experts stay exact. Needs hidden a multiple of 256
 * and inter a multiple of 128; not with an expert cache or
 * DF_MOE_PREFILL_MMA_SYNC. */
#define DF_MOE_MXFP8_ACT 8u
/* The same block-scaled tensor-core GEMMs on exact activations: x and h
 * enter them as sums of E4M3 planes (x: 4, h: 5), each plane the MXFP8
 * rounding of what the planes before it left, so that the sum reproduces the
 * activation to fp32 precision; the results are the exact path's, within its
 * tolerances. Meant for batches (prefill): on such a handle decode calls run
 * these GEMMs too (one token: two phase kernels that run them beside the
 * shared experts, the gate/up sums taken over eight parts of K), slower than
 * the default decode kernels below 4 tokens. Same shape rules as
 * DF_MOE_MXFP8_ACT, and not together with it. */
#define DF_MOE_PLANES 16u

typedef struct df_moe df_moe; /* opaque, library-owned */

typedef struct {
  int32_t hidden;       /* H: multiple of 64                                   */
  int32_t n_experts;    /* E: routed experts per layer, 1..1024                */
  int32_t top_k;        /* k: experts per token, 1..min(E, 32)                 */
  int32_t inter;        /* I: routed-expert intermediate, multiple of 64       */
  int32_t n_shared;     /* shared experts per layer (0..8)                     */
  int32_t shared_inter; /* Is: shared intermediate, multiple of 64             */
  int32_t n_layers;     /* L >= 1                                              */
  int32_t max_tokens;   /* largest T a forward call may use (1..4096)          */
  float rms_eps;        /* stack mode only                                     */
  uint32_t flags;       /* DF_MOE_STACK_RMSNORM_RESIDUAL | DF_MOE_PREFILL_MMA_SYNC |
                           DF_MOE_MXFP8_ACT | DF_MOE_PLANES */
} df_moe_config;

/* Weights of one layer, any subset per call (NULL / 0 = leave unchanged). */
typedef struct {
  /* fp32 [E][H] row-major. */
  const float* router;
  /* expert_count canonical spans back to back, one per expert, expert ids
   * expert_begin .. expert_begin + expert_count - 1. A span is the six
   * tensors of one expert, contiguous (Deltafin README, "Techniques / I/O and
   * streaming": an expert's six tensors are one contiguous range):
   *   gate_q [I][H/2] | gate_s [I][H/32] | up_q [I][H/2] | up_s [I][H/32] |
   *   down_q [H][I/2] | down_s [H][I/32]
   * q bytes hold element 2m in the low nibble and 2m+1 in the high nibble;
   * s bytes are E8M0 exponents of 32 consecutive elements along the input
   * dimension. The span is 3*H*I*17/32 bytes (17,547,264 at K3 shape). */
  const uint8_t* experts;
  int32_t expert_begin;
  int32_t expert_count;
  /* n_shared pointers each, bf16: gate [Is][H], up [Is][H], down [H][Is]. */
  const uint16_t* const* shared_gate;
  const uint16_t* const* shared_up;
  const uint16_t* const* shared_down;
  /* 1: every pointer above is device memory; 0: host memory. The pointer
   * arrays themselves are always host memory. */
  int32_t src_is_device;
} df_moe_layer_weights;

/* Allocates the weight arenas (one expert-major arena of E spans per layer,
 * router and shared weights) and the workspace on `cuda_device`.
 * Errors: EINVAL (bad config), ENOMEM, ECUDA. */
DF_MOE_API int df_moe_create(const df_moe_config* cfg, int cuda_device, df_moe** out);

/* Expert cache (models larger than HBM): as df_moe_create, but every
 * layer's experts live in pinned host memory (the Grace side, reached over
 * NVLink-C2C) and only `cache_slots` of them a layer in HBM. Each forward
 * layer brings its selection to the host (one synchronisation: forward is
 * synchronous on its stream), gives the selected experts that are not
 * cached free or least recently used slots, copies them in with one fill
 * kernel (SM loads of the mapped host pool) and runs the decode kernels on
 * the slots. A call whose experts are all cached copies nothing.
 * Consecutive tokens that reuse experts find them cached (the Deltafin
 * README, "Techniques", and the kimi-k3-in-c blog's expert LRU cache stream
 * experts from SSD with the same reuse). The library owns the pinned pool
 * (n_layers * n_experts spans) and frees it in df_moe_destroy; load_experts
 * fills it. Limits: max_tokens <= 8,
 * min(max_tokens*top_k, n_experts) <= cache_slots <= n_experts; no graphs
 * and no single expert steps on such a handle. Errors as df_moe_create
 * (ENOMEM also when the pinned pool cannot be allocated). */
DF_MOE_API int df_moe_create_cached(const df_moe_config* cfg, int cuda_device,
                                    int32_t cache_slots, df_moe** out);
/* Since creation: selected experts found cached, experts copied in, and the
 * bytes copied from host to HBM. Zeros for a handle without a cache. */
DF_MOE_API int df_moe_cache_stats(const df_moe* h, int64_t* hits, int64_t* misses,
                                  int64_t* bytes_in);

/* Frees everything. NULL-safe. The caller must not have work in flight. */
DF_MOE_API void df_moe_destroy(df_moe* h);

/* Message of the last failing call on h (or of this thread when h is NULL).
 * Valid until the next call on the same handle/thread. */
DF_MOE_API const char* df_moe_last_error(const df_moe* h);

/* Bytes of one expert span for this handle's shape / for (H, I). */
DF_MOE_API size_t df_moe_expert_span_bytes(const df_moe* h);
DF_MOE_API size_t df_moe_span_bytes_for(int32_t hidden, int32_t inter);

/* Copies the given weights of `layer` into the library's arenas, repacking
 * expert spans into the kernels' HBM layout (still one contiguous span of the
 * same size per expert). Host sources are staged through a bounded pinned
 * buffer; the call returns after the host buffers have been consumed.
 * Device sources may be freed after `stream` has synchronised.
 * Errors: EINVAL, ERANGE (layer or expert range), ECUDA. */
DF_MOE_API int df_moe_load_experts(df_moe* h, int32_t layer,
                        const df_moe_layer_weights* w, void* stream);

/* One forward pass over T tokens (1 <= T <= max_tokens), asynchronous.
 *   x_bf16        device [T][H] bf16
 *   residual_bf16 device [T][H] bf16 or NULL (single-layer mode only)
 *   out_bf16      device [T][H] bf16 (RNE of the fp32 result)
 *   out_f32       device [T][H] fp32 or NULL: the fp32 result before rounding
 *   ids           device [L][T][k] int32, descending logit order
 *   weights       device [L][T][k] fp32, softmax over the selected logits
 * Errors: EINVAL, ERANGE (T), ESTATE (weights not loaded), ECUDA, and the
 * error recorded by the device-side checks of an earlier call: ETIMEOUT (a
 * bounded wait gave up) or EDEVICE (an index out of range was skipped). The
 * last kernel of every call copies the device error word to a host-visible
 * word when it is nonzero; a call that finds that word set synchronises
 * `stream`, clears the error, returns it and launches nothing (results of
 * the call that recorded it are not to be trusted). A call after that runs
 * normally. */
DF_MOE_API int df_moe_forward(df_moe* h, const void* x_bf16, int32_t T,
                   const void* residual_bf16, void* out_bf16, float* out_f32,
                   int32_t* ids, float* weights, void* stream);

/* Stack mode: the same forward pass, also recording every layer's inputs as
 * the device computed them, for checking a layer against a reference on
 * exactly those inputs.
 *   trace_x   device [L][T][H] bf16 or NULL: x entering layer l (the residual)
 *   trace_xn  device [L][T][H] bf16 or NULL: its RMS-normalised form, the
 *             input of layer l's router and experts
 * Errors as df_moe_forward; EINVAL outside stack mode. */
DF_MOE_API int df_moe_forward_trace(df_moe* h, const void* x_bf16, int32_t T,
                         void* out_bf16, float* out_f32, int32_t* ids,
                         float* weights, void* trace_x, void* trace_xn,
                         void* stream);

/* Same, with HOST buffers: moves x (and residual) to the device, runs the
 * forward, brings the results back and synchronises `stream` before
 * returning. The device moves the data itself: a small copy kernel reads the
 * inputs from pinned host memory (the caller's buffer when it is pinned and
 * mapped with a 16-byte-aligned device address, else a pinned staging copy
 * the handle makes on first use), and the last kernel writes the output,
 * ids and weights into pinned host memory (the caller's, or the staging,
 * copied out after the synchronisation). Pinned caller buffers save the
 * staging copies. Buffers in device or managed memory are also accepted
 * (moved with cudaMemcpyAsync). out_f32, residual, ids and weights may be
 * NULL. Errors as df_moe_forward, ENOMEM if the staging cannot be made, and
 * ETIMEOUT / EDEVICE recorded by this call's own kernels (checked after the
 * synchronisation; the error is then cleared). */
DF_MOE_API int df_moe_forward_host(df_moe* h, const uint16_t* x_bf16, int32_t T,
                        const uint16_t* residual_bf16, uint16_t* out_bf16,
                        float* out_f32, int32_t* ids, float* weights,
                        void* stream);

/* Synchronises `stream` and reports (and clears) any device-side error
 * word: ETIMEOUT if a bounded wait gave up, EDEVICE if a range check failed,
 * DF_MOE_OK otherwise. */
DF_MOE_API int df_moe_sync(df_moe* h, void* stream);

/* Test hook for the failure path (no GPU fault involved): the next forward
 * call's gate/up phase (decode batches, T <= 8) leaves one stage of one
 * routed-expert pipeline unfilled and unannounced, and its bounded waits use
 * a short limit (2^12 polls). The waiting warps give up, record a timeout in
 * the device error word and leave; every other wait of the call is bounded
 * too, so the call ends. That call's results are wrong and the error is
 * reported as ETIMEOUT by df_moe_sync, by df_moe_forward_host after its
 * synchronisation, or by the next forward. One-shot. Errors: EINVAL (null). */
DF_MOE_API int df_moe_test_drop_arrival(df_moe* h);

/* ---- CUDA graphs -----------------------------------------------------------
 * A forward pass captured once into a CUDA graph and replayed: one launch a
 * step instead of one per kernel, the programmatic dependencies between the
 * kernels kept as graph edges. The graph is bound to the buffers given here;
 * between launches the caller changes the CONTENTS of x (and residual), not
 * the pointers. Arguments as df_moe_forward; the capture runs on a stream of
 * the handle's own, so `stream` may be any stream (the legacy default one
 * included) and nothing is enqueued on it.
 * Not with timing on (EINVAL). The graph holds no
 * reference to the handle's host state: destroy it before the handle. */
typedef struct df_moe_graph df_moe_graph; /* opaque */
DF_MOE_API int df_moe_graph_create(df_moe* h, const void* x_bf16, int32_t T,
                                   const void* residual_bf16, void* out_bf16, float* out_f32,
                                   int32_t* ids, float* weights, df_moe_graph** out);
/* Enqueues one replay on `stream`. Errors: EINVAL (null graph), ECUDA. */
DF_MOE_API int df_moe_graph_launch(df_moe_graph* g, void* stream);
/* Kernel launches in one replay. */
DF_MOE_API int df_moe_graph_launch_count(const df_moe_graph* g);
/* NULL-safe. */
DF_MOE_API void df_moe_graph_destroy(df_moe_graph* g);

/* ---- read bandwidth probe --------------------------------------------------
 * Streams `bytes` (a multiple of 16, buf 16-byte aligned) of device memory
 * with 16-byte loads into one word per thread of `sink` (device, at least
 * 152 * 8 * 256 words): the read-only streaming rate the layer's kernels are
 * measured against beside the copy peak. Errors: EINVAL, ECUDA. */
DF_MOE_API int df_moe_stream_read(const void* buf, size_t bytes, uint32_t* sink, void* stream);

/* ---- single steps (the rows of the hot path, for per-step checks) ---------
 * Each runs one step of the forward on its own, with the same kernels. Every
 * device array argument of the steps below (x, logits, ids, weights, hbuf,
 * y, xn, and group's outputs) must be 16-byte aligned, as the kernels read
 * and write them with vector accesses and tensor maps; a misaligned one is
 * EINVAL before anything is launched. */

/* logits device [T][E] fp32 of layer `layer`. */
DF_MOE_API int df_moe_step_router(df_moe* h, int32_t layer, const void* x_bf16, int32_t T,
                       float* logits, void* stream);
/* ids device [T][k], weights device [T][k] from logits device [T][E]. */
DF_MOE_API int df_moe_step_topk(df_moe* h, const float* logits, int32_t T, int32_t* ids,
                     float* weights, void* stream);
/* Counting sort of the T*k assignments a = t*k + j by expert: offs device
 * [E+1]; tok, slot device [T*k] (segment of expert e ordered by a);
 * n_union device [1] = number of distinct experts. */
DF_MOE_API int df_moe_step_group(df_moe* h, const int32_t* ids, int32_t T, int32_t* offs,
                      int32_t* tok, int32_t* slot, int32_t* n_union,
                      void* stream);
/* hbuf device [T*k][I] fp32: silu(Wg x) * (Wu x) of expert ids[t][j] at row
 * t*k + j. */
DF_MOE_API int df_moe_step_expert_gateup(df_moe* h, int32_t layer, const void* x_bf16,
                              int32_t T, const int32_t* ids, float* hbuf,
                              void* stream);
/* y device [T][H] fp32 = sum_j weights[t][j] Wd_{ids[t][j]} hbuf[t*k + j]. */
DF_MOE_API int df_moe_step_expert_down(df_moe* h, int32_t layer, const float* hbuf,
                            int32_t T, const int32_t* ids,
                            const float* weights, float* y, void* stream);
/* With DF_MOE_MXFP8_ACT the two expert steps take MXFP8 activations: gate/up
 * rounds x first (hbuf is h before its own rounding), down rounds hbuf first.
 * The rounding alone, with the same kernels' routine: v device [rows][n] fp32
 * (n a multiple of 32, 16-byte aligned) -> codes device [rows][n] E4M3 bytes,
 * scales device [rows][n/32] E8M0 bytes. Any handle. Errors: EINVAL. */
DF_MOE_API int df_moe_step_mxfp8(df_moe* h, const float* v, int32_t rows, int32_t n,
                                 uint8_t* codes, uint8_t* scales, void* stream);
/* y device [T][H] fp32 = sum over shared experts. */
DF_MOE_API int df_moe_step_shared(df_moe* h, int32_t layer, const void* x_bf16, int32_t T,
                       float* y, void* stream);
/* xn device [T][H] bf16 = RNE(x / sqrt(mean(x^2) + rms_eps)). */
DF_MOE_API int df_moe_step_rmsnorm(df_moe* h, const void* x_bf16, int32_t T, void* xn_bf16,
                        void* stream);

/* Reads expert `expert` of `layer` back from the device layout into canonical
 * span order (dst: host, df_moe_expert_span_bytes bytes). Synchronous. */
DF_MOE_API int df_moe_read_expert_span(df_moe* h, int32_t layer, int32_t expert,
                            uint8_t* dst);

/* ---- measurement ---------------------------------------------------------
 * With timing on, every kernel launch of forward is bracketed by CUDA events
 * on its stream; df_moe_timing_get returns, per kernel kind, the launches and
 * the summed device time since the last reset. */
#define DF_MOE_KERNEL_KINDS 18
DF_MOE_API int df_moe_timing_enable(df_moe* h, int on);
DF_MOE_API int df_moe_timing_reset(df_moe* h);
DF_MOE_API int df_moe_timing_get(df_moe* h, int kind, const char** name,
                      int64_t* launches, double* total_ms);
/* Kernels launched by the last forward call. */
DF_MOE_API int df_moe_last_launch_count(const df_moe* h);

/* ---- routing without any allocation ---------------------------------------
 * No counterpart in the pages: an addition for callers that must not
 * allocate device memory, such as a serving engine that has already divided
 * all of HBM among its own pools, or a decode loop that cannot afford the
 * device-wide synchronisation a cudaMalloc/cudaFree may cause. It needs no
 * handle.
 *
 * Router GEMV + top-k + softmax over the selected logits (the same kernels
 * and the same results as df_moe_step_router followed by df_moe_step_topk),
 * with the partial-logit scratch in a fixed 1 MiB array of device memory that
 * is part of the library: every GPU that loads the library holds it until the
 * process exits. The call allocates nothing (no cudaMalloc/cudaFree, no
 * allocating library routine).
 *   router  device [E][H] fp32      x_bf16  device [T][H] bf16; both 16-byte aligned
 *           (EINVAL otherwise, checked before anything is launched)
 *   ids     device [T][k] int32     weights device [T][k] fp32
 * Limits: H a multiple of 32 up to 8192, 1 <= E <= 1024, 1 <= k <=
 * min(E, 32), and the scratch must hold nsplit*T*E floats (262,144 floats;
 * nsplit is the router's column split, 4 at H = 7168 and E = 896, so T <= 73
 * there). Larger calls fail with DF_MOE_ERANGE and a message from
 * df_moe_last_error(NULL); nothing is launched then.
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it for the life of the process; make that
 * first call before any stream capture. A device reset (cudaDeviceReset)
 * would leave the cached address stale: this entry point does not support
 * calls after one. The router kernel is an ordinary launch on `stream`, so
 * inputs written by the caller's kernels earlier on that stream are seen. All calls share the one array: calls that overlap on the GPU (on
 * different streams, or from different threads) race and must be ordered by
 * the caller. Nothing in it needs clearing between calls: each call writes
 * every scratch element it later reads. */
DF_MOE_API int df_moe_route_noalloc(const float* router, int32_t E, int32_t H,
                                    const void* x_bf16, int32_t T, int32_t k,
                                    int32_t* ids, float* weights, void* stream);

#ifdef __cplusplus
}
#endif
#endif
