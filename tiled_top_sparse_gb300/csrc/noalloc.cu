// Allocation-free variant of dense attention with fp32 inputs.
//
// tts_attn_fwd_varlen with fp32 q/k/v needs device scratch to hold the bf16
// copies of its inputs, and asks its caller for that scratch as a workspace.
// Some callers cannot provide one: code running where another runtime has
// reserved the device's whole memory pool, or a serving loop that must not
// allocate once it has started (allocation can block and fragments memory).
// For them this entry point uses a fixed scratch array that lives in the
// library's own device memory (kNoAllocScratchBytes, reserved on every GPU that
// loads the library, until the process exits) and calls no allocator at all.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/tts.h"

namespace {

constexpr size_t kNoAllocScratchBytes = TTS_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Device-side scratch. In host code this name is only a stand-in for the
// symbol, never a device address: the address is looked up per device below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
// Per device: the context the address was looked up in, and the address. A device
// reset (or a released and re-created primary context) loads the module again, and
// the array may then sit at another address; a new context triggers a new lookup.
struct ScratchSlot {
  unsigned long long ctx_id = 0;  // the driver's unique context id (never reused)
  void* ptr = nullptr;
};
ScratchSlot g_slot[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

void* driver_fn(const char* name) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return f;
}

// Unique id of the calling thread's current context; 0 when none is current.
CUresult current_ctx_id(unsigned long long* id) {
  static const CtxGetCurrentFn get = reinterpret_cast<CtxGetCurrentFn>(driver_fn("cuCtxGetCurrent"));
  static const CtxGetIdFn get_id = reinterpret_cast<CtxGetIdFn>(driver_fn("cuCtxGetId"));
  *id = 0;
  if (get == nullptr || get_id == nullptr) return CUDA_ERROR_NOT_SUPPORTED;
  CUcontext ctx = nullptr;
  CUresult r = get(&ctx);
  if (r != CUDA_SUCCESS || ctx == nullptr) return r;
  return get_id(ctx, id);
}

// Device address of the scratch array in the current context of the current device;
// looked up once per (device, context), with that device current, and cached.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long id = 0;
  if (current_ctx_id(&id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchSlot& s = g_slot[dev];
  if (id == 0 || s.ptr == nullptr || s.ctx_id != id) {
    // The lookup also makes the device's primary context current when no context is.
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (current_ctx_id(&id) != CUDA_SUCCESS || id == 0) return cudaErrorDeviceUninitialized;
    s.ctx_id = id;
    s.ptr = p;
  }
  *out = s.ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" tts_status tts_attn_fwd_varlen_f32_noalloc(
    const float* q, const float* k, const float* v, int64_t total_q, int64_t total_k,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch, int32_t max_seqlen_q,
    int32_t max_seqlen_k, int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim,
    int32_t causal, float scale, float* out, float* lse, uint32_t* dev_status, void* stream) {
  if (total_q < 0 || total_k < 0 || num_heads_q < 1 || num_heads_kv < 1 || head_dim < 1)
    return TTS_ERR_INVALID_ARG;
  const size_t need = tts_attn_workspace_bytes(total_q, total_k, num_heads_q, num_heads_kv,
                                               head_dim, TTS_F32);
  if (need > kNoAllocScratchBytes) return TTS_ERR_WORKSPACE;  // inputs too large for the array
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return TTS_ERR_CUDA;
  return tts_attn_fwd_varlen(q, k, v, TTS_F32, total_q, total_k, cu_seqlens_q, cu_seqlens_k,
                             batch, max_seqlen_q, max_seqlen_k, num_heads_q, num_heads_kv,
                             head_dim, causal, scale, out, lse, scratch, kNoAllocScratchBytes,
                             dev_status, stream);
}
