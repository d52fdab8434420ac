// Diagnostics: exercises the bounded-wait path that every kernel of the library uses.
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/tts.h"
#include "ptx.cuh"

namespace {

// Waits on an mbarrier phase that nothing ever completes. The bounded wait gives up
// after its time limit, sets the timeout bit in *status and the kernel returns, so the
// CUDA context stays usable.
__global__ void wait_timeout_kernel(uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  tts::mbar_init(tts::smem_u32(&bar), 1);
  tts::fence_mbar_init();
  tts::mbar_wait(tts::smem_u32(&bar), 0, &abort_flag, status);
}

}  // namespace

extern "C" tts_status tts_debug_wait_timeout(uint32_t* dev_status, void* stream) {
  if (dev_status == nullptr) return TTS_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status);
  return cudaGetLastError() == cudaSuccess ? TTS_OK : TTS_ERR_CUDA;
}
