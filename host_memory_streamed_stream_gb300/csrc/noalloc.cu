// RMSNorm backward that allocates nothing: its scratch lives in a fixed device array
// inside the library instead of a caller-supplied buffer.
//
// Why: some callers cannot allocate device memory at the point where they need this
// kernel. Examples are code running under a memory manager that owns the whole device
// (a framework's caching allocator or a fixed memory budget), and code paths where the
// implicit device-wide synchronisation of cudaMalloc/cudaFree is not allowed. Such a
// caller passes only its inputs and outputs.
//
// The scratch is a file-scope __device__ array of kNoAllocPartialFloats floats (9.5 MiB);
// every GPU that loads the library holds it until the process exits. In host code the
// array's name is only a host-side stand-in, so the kernel is given the device address
// obtained with cudaGetSymbolAddress, once per device, with that device current. The
// first call on a device does that set-up; that first call should come before any
// stream capture. All calls share the one array and it keeps the last call's contents:
// every element that is read is first written by the same call, so nothing needs
// clearing, but calls that overlap on the GPU (different streams, or different host
// threads) race on the array and must be serialised by the caller.
#include <mutex>
#include <string>

#include "kernels.h"
#include "mt.h"
#include "mt_kernels.h"

namespace {

constexpr int kNoAllocMaxDevices = 64;
constexpr long long kNoAllocPartialFloats = 304LL * 8192LL;  // rmsnorm_bwd_parts(T) * h <= this

static __device__ __align__(256) float g_noalloc_partial[kNoAllocPartialFloats];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kNoAllocMaxDevices] = {};

}  // namespace

void mt_set_global_error(const std::string& m);  // message for mt_last_error(NULL)
extern const char* const kRmsBwdAlignMsg;          // the alignment rule, worded once (capi_kernels.cu)

namespace {
int noalloc_fail(int code, const std::string& m) {
  mt_set_global_error(m);
  return code;
}
}  // namespace

extern "C" int mtk_rmsnorm_bwd_noalloc(const void* dy, const void* x, const void* gamma, const void* rstd,
                                       const void* dres, void* dx, void* dx_bf16, void* dgamma, int T, int h,
                                       void* stream) {
  if (!dy || !x || !gamma || !rstd || !dx || !dgamma || T <= 0 || h <= 0)
    return noalloc_fail(MT_EINVAL, "null pointer or non-positive size");
  if (!mt::rmsnorm_bwd_aligned(static_cast<const float*>(dy), static_cast<const float*>(x),
                               static_cast<const mt::bf16*>(gamma), static_cast<const float*>(dres),
                               static_cast<const float*>(dx), static_cast<const mt::bf16*>(dx_bf16), nullptr))
    return noalloc_fail(MT_EINVAL, kRmsBwdAlignMsg);
  const long long need = static_cast<long long>(mt::rmsnorm_bwd_parts(T)) * h;
  if (need > kNoAllocPartialFloats)
    return noalloc_fail(MT_EINVAL, "mtk_rmsnorm_bwd_noalloc: min(T, 304) * h = " + std::to_string(need) +
                                       " floats exceeds the fixed scratch of " +
                                       std::to_string(kNoAllocPartialFloats) + " floats");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return noalloc_fail(MT_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return noalloc_fail(MT_EINVAL, "device index out of range");
  float* partial = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_partial);
      if (e != cudaSuccess || !p)
        return noalloc_fail(MT_ECUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
      g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    partial = g_noalloc_ptr[dev];
  }
  e = mt::rmsnorm_bwd(static_cast<const float*>(dy), static_cast<const float*>(x),
                      static_cast<const mt::bf16*>(gamma), static_cast<const float*>(rstd),
                      static_cast<const float*>(dres), static_cast<float*>(dx), static_cast<mt::bf16*>(dx_bf16),
                      partial, static_cast<mt::bf16*>(dgamma), T, h, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return noalloc_fail(e == cudaErrorInvalidValue ? MT_EINVAL : MT_ECUDA, cudaGetErrorString(e));
  return MT_OK;
}
