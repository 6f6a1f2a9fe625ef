// selftest.cu -- jfa_selftest_wait_timeout: exercises the bounded-wait
// failure path on the GPU without any fault. One thread waits on an mbarrier
// phase that nothing completes, with the caller's time limit; the wait gives
// up, records the timeout (error code, wait site, block) in the workspace
// status block like any kernel of the library, and the kernel returns.
#include <cuda_runtime.h>

#include "host_common.h"
#include "jfa.h"
#include "sm103.cuh"

namespace {

using jfa::kStatusBytes;
constexpr int kSite = 99;  // the wait site reported by this probe

__global__ void wait_timeout_probe(uint32_t *status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    jfa::dev::mbar_init(&bar, 1);  // one arrival completes phase 0; none ever comes
    abort_flag = 0;
    jfa::dev::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const jfa::dev::WaitCtl ctl{status, &abort_flag, timeout_ns};
    (void)jfa::dev::mbar_wait(&bar, 0, ctl, kSite);
  }
}

}  // namespace

extern "C" jfa_status jfa_selftest_wait_timeout(void *workspace, size_t ws_bytes,
                                                uint64_t timeout_ns, jfa_stream_t stream) {
  if (!workspace || ws_bytes < kStatusBytes)
    return jfa::fail(JFA_ERR_WORKSPACE, "workspace missing or smaller than %zu bytes", kStatusBytes);
  if (timeout_ns < 1000 || timeout_ns > 1000000000ull)
    return jfa::fail(JFA_ERR_INVALID_ARG, "timeout_ns must be in [1 us, 1 s]");
  wait_timeout_probe<<<1, 32, 0, (cudaStream_t)stream>>>(static_cast<uint32_t *>(workspace),
                                                         timeout_ns);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return jfa::fail(JFA_ERR_CUDA, "probe launch: %s", cudaGetErrorString(e));
  return JFA_OK;
}
