// noalloc.cu -- jfa_bwd_noalloc: the jagged backward with its scratch memory
// in a fixed static device array instead of a caller-provided workspace.
//
// Who needs this: callers that cannot obtain device memory at the point of
// the call, for example a plug-in running inside a framework that owns every
// byte of device memory through its own pool and has nothing to lend for
// scratch, or a latency-critical path that must not call cudaMalloc (which
// may synchronise the whole device). They still pass their inputs and
// outputs; only the scratch (the status block and the fp32 dQ accumulator
// that jfa_bwd keeps in its workspace) moves here.
//
// The array lives in this translation unit alone, so its module (and the
// memory) is only loaded when this entry point is first used under lazy
// module loading; with eager loading every device gets it when the library
// is loaded. Either way each device that has it keeps it until the process
// exits.
#include <cuda_runtime.h>

#include <mutex>

#include "host_common.h"
#include "jfa.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB per device
constexpr size_t kStatusBytes = 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. The name of the
// array is only a host-side handle; the address has to be looked up once per
// device with that device current.
jfa_status scratch_for_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return jfa::fail(JFA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return jfa::fail(JFA_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return jfa::fail(JFA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return JFA_OK;
}

}  // namespace

extern "C" jfa_status jfa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                      const float *lse, const void *dout, const void *offsets,
                                      jfa_index_t idx, int64_t B, int64_t T, int H, int D,
                                      float scale, const int32_t *d_sm_ptr,
                                      const int32_t *d_tiles, int num_sms, void *dq, void *dk,
                                      void *dv, jfa_stream_t stream) {
  if (H < 1 || D < 1 || T < 0) return jfa::fail(JFA_ERR_INVALID_ARG, "bad sizes");
  const size_t need = jfa_workspace_size(JFA_OP_BWD, T, H, D);
  if (need > kScratchBytes)
    return jfa::fail(JFA_ERR_WORKSPACE,
                     "jfa_bwd_noalloc: T*H*D = %lld needs %zu bytes of scratch, more than its "
                     "fixed %zu-byte static buffer (T*H*D <= %zu); use jfa_bwd with a workspace",
                     (long long)(T * H * D), need, kScratchBytes,
                     (kScratchBytes - kStatusBytes) / sizeof(float));
  void *scratch = nullptr;
  jfa_status st = scratch_for_current_device(&scratch);
  if (st != JFA_OK) return st;
  // The status block must start at zero; jfa_bwd clears the accumulator itself.
  cudaError_t e = cudaMemsetAsync(scratch, 0, kStatusBytes, (cudaStream_t)stream);
  if (e != cudaSuccess) return jfa::fail(JFA_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
  return jfa_bwd(q, k, v, o, lse, dout, offsets, idx, B, T, H, D, scale, d_sm_ptr, d_tiles,
                 num_sms, dq, dk, dv, scratch, kScratchBytes, stream);
}
