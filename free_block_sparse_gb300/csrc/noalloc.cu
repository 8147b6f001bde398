// Mask prediction for callers that cannot allocate device memory.
//
// Some callers of this library are not allowed to call cudaMalloc: plug-ins loaded into a host
// application whose own allocator has already reserved the device memory it is willing to
// give out, and latency-critical loops in which the device synchronisation that cudaMalloc
// and cudaFree can cause is not acceptable.  sparge_predict_mask_noalloc serves them: it runs
// the same two kernels as sparge_predict_mask, but their scratch (pooled means and
// similarities) lives in a fixed array in this file instead of a caller-provided workspace.
#include <cstdio>
#include <mutex>

#include "../../include/sparge.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB, held by every GPU that loads the library
constexpr int kMaxDevices = 64;

// Stage-1 scratch shared by every call of sparge_predict_mask_noalloc on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};  // the context each address was looked up in

// cuCtxGetCurrent through the runtime's driver entry point (no link-time dependency on libcuda).
typedef CUresult (*ctx_get_fn_t)(CUcontext *);
ctx_get_fn_t ctx_get_fn() {
  static ctx_get_fn_t fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r) == cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<ctx_get_fn_t>(p);
  });
  return fn;
}

}  // namespace

extern "C" int sparge_predict_mask_noalloc(const sparge_tensor *q, const sparge_tensor *k, float topk, float theta,
                                           int is_causal, uint8_t *mask, sparge_stream_t stream) {
  sparge::View qv, kv;
  int rc = sparge::validate_predict_args(q, k, topk, theta, &qv, &kv);
  if (rc) return rc;
  const size_t need = sparge::predict_ws_bytes(qv.B, qv.H, kv.H, qv.N, kv.N, qv.d);
  if (need > kScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg), "shape needs %zu bytes of scratch; the allocation-free call holds %zu", need,
             kScratchBytes);
    return sparge::report_error(SPARGE_ERR_UNSUPPORTED, msg);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return sparge::report_error(SPARGE_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return sparge::report_error(SPARGE_ERR_UNSUPPORTED, "device ordinal too large");
  // the device's current context: a new one (after cudaDeviceReset, say) holds a new copy of the array
  CUcontext ctx = nullptr;
  ctx_get_fn_t get = ctx_get_fn();
  if (!get || get(&ctx) != CUDA_SUCCESS || !ctx)
    return sparge::report_error(SPARGE_ERR_CUDA, "no current CUDA context for the allocation-free call");
  void *scratch = nullptr;
  {
    // First call on a device (or in a new context of it): look up the device address of the
    // array with that device current.
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return sparge::report_error(SPARGE_ERR_CUDA, cudaGetErrorString(e));
      g_scratch_addr[dev] = p;
      g_scratch_ctx[dev] = ctx;
    }
    scratch = g_scratch_addr[dev];
  }
  // Nothing in the scratch has to start at zero: every value the kernels read is written earlier
  // in the same call, except the padding columns of the pooled keys, whose products are discarded.
  return sparge::run_predict(qv, kv, topk, theta, is_causal, mask, scratch, kScratchBytes,
                             reinterpret_cast<cudaStream_t>(stream));
}
