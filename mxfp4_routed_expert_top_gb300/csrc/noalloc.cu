// noalloc.cu — routing (router GEMV + top-k) that allocates nothing.
//
// For callers that may not allocate device memory (an engine that owns all
// of HBM through its own pools, or a decode loop that must not hit the
// device-wide synchronisation an allocation can cause). The partial-logit
// scratch lives in a file-scope device array instead of the handle's
// workspace; the kernels are the library's own router and top-k kernels.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "df_moe.h"
#include "internal.h"

namespace {

constexpr size_t kScratchFloats = 262144;  // 1 MiB of partial logits
static __device__ __align__(256) float g_route_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_addr[kMaxDevices] = {};  // device address, per device

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  dfm::set_thread_error(buf);
  return code;
}

// The array's name is only a host-side stand-in; the kernels need its device
// address, looked up once per device with that device current.
int scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DF_MOE_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(DF_MOE_ERANGE, "device %d not supported", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess || !p)
      return fail(DF_MOE_ECUDA, "cudaGetSymbolAddress of the routing scratch: %s",
                  cudaGetErrorString(e));
    g_scratch_addr[dev] = (float*)p;
  }
  *out = g_scratch_addr[dev];
  return DF_MOE_OK;
}

}  // namespace

extern "C" DF_MOE_API int df_moe_route_noalloc(const float* router, int32_t E,
                                               int32_t H, const void* x_bf16,
                                               int32_t T, int32_t k, int32_t* ids,
                                               float* weights, void* stream) {
  if (!router || !x_bf16 || !ids || !weights)
    return fail(DF_MOE_EINVAL, "router, x, ids and weights are required");
  if ((uintptr_t)x_bf16 & 15) return fail(DF_MOE_EINVAL, "x must be 16-byte aligned");
  // the router kernel reads the weights with 16-byte loads
  if ((uintptr_t)router & 15) return fail(DF_MOE_EINVAL, "router must be 16-byte aligned");
  if (H <= 0 || H % 32 || H > 8192)
    return fail(DF_MOE_EINVAL, "H must be a multiple of 32 in [32, 8192]");
  if (E < 1 || E > 1024) return fail(DF_MOE_EINVAL, "E must be in [1, 1024]");
  if (k < 1 || k > E || k > 32) return fail(DF_MOE_EINVAL, "k must be in [1, min(E, 32)]");
  if (T < 1) return fail(DF_MOE_ERANGE, "T = %d: at least one token is needed", T);
  const dfm::RouterSplit sp = dfm::router_split(E, H);
  const size_t need = (size_t)sp.nsplit * (size_t)T * (size_t)E;
  if (need > kScratchFloats)
    return fail(DF_MOE_ERANGE,
                "T = %d needs %zu floats of routing scratch (%d column splits x T x E); "
                "the fixed scratch holds %zu",
                T, need, sp.nsplit, kScratchFloats);
  float* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  // an ordinary launch, not a programmatic dependent: here the router
  // weights are the caller's, and the caller's kernel just before this call
  // may have written them
  cudaError_t e = dfm::launch_router(router, E, H, (const uint16_t*)x_bf16, T,
                                     scratch, sp, s, nullptr, /*after_previous=*/false);
  if (e != cudaSuccess)
    return fail(DF_MOE_ECUDA, "router launch: %s", cudaGetErrorString(e));
  e = dfm::launch_topk(scratch, sp.nsplit, T, E, k, nullptr, ids, weights,
                       nullptr, nullptr, nullptr, s);
  if (e != cudaSuccess)
    return fail(DF_MOE_ECUDA, "top-k launch: %s", cudaGetErrorString(e));
  return DF_MOE_OK;
}
