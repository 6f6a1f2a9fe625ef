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

#include "host_common.h"
#include "jfa.h"

namespace {

using jfa::kStatusBytes;

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array in the current device's context. In
// host code the array's name is only a handle, so the address is looked up
// with the device current. It is looked up at every call (a host-side query,
// no allocation) rather than cached, so it stays right after a
// cudaDeviceReset, which reloads the module and the array with it.
jfa_status scratch_for_current_device(void **out) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p)
    return jfa::fail(JFA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
  *out = p;
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
  // The status block needs no clearing here: the array starts at zero, a
  // kernel only writes its error words when a wait gives up (they then stay
  // set until jfa_noalloc_check_status reads and clears them), and the
  // backward's closing cast resets the cleared-accumulator count, so jfa_bwd
  // always clears the accumulator itself.
  return jfa_bwd(q, k, v, o, lse, dout, offsets, idx, B, T, H, D, scale, d_sm_ptr, d_tiles,
                 num_sms, dq, dk, dv, scratch, kScratchBytes, stream);
}

extern "C" jfa_status jfa_noalloc_check_status(jfa_stream_t stream) {
  void *scratch = nullptr;
  jfa_status st = scratch_for_current_device(&scratch);
  if (st != JFA_OK) return st;
  return jfa::read_status_block(scratch, stream);
}
