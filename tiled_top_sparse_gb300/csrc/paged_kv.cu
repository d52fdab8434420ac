// Paged KV cache write: the path that fills the cache the sparse attention reads.
//
// "推理引擎的蝴蝶效应 -- 从V32 模型的输出不一致说起" (section 实验方法和结果) reads the
// KV cache through pagetable_1 and rules out its write path before blaming the index
// order; "从 SGLang Kernel源码到 GPU Trace" (section 2.2) names the page-table-managed
// cache (PagedKVCache). Token t of the call belongs to request req_ids[t] (or request t)
// and sits at logical position positions[t] of that request's sequence; its row goes to
// kv_cache[page_tables[req, pos / page_size], pos % page_size, :]. One warp moves one
// row in 16-byte pieces; a token whose request, position or page is out of range is
// skipped and reported in the status word.
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace tts {
namespace {

__global__ void __launch_bounds__(256) paged_kv_write_kernel(
    const uint4* __restrict__ kv_new, int64_t ntok, int pieces, const int32_t* __restrict__ req_ids,
    const int32_t* __restrict__ positions, const int32_t* __restrict__ page_tables, int max_pages,
    int nreq, uint4* __restrict__ kv_cache, int num_pages, int page_size, uint32_t* status) {
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= ntok) return;
  const int64_t r = req_ids != nullptr ? req_ids[t] : t;
  const int64_t pos = positions[t];
  bool ok = r >= 0 && r < nreq && pos >= 0 && pos < (int64_t)max_pages * page_size;
  int64_t pg = -1;
  if (ok) {
    pg = page_tables[r * max_pages + pos / page_size];
    ok = pg >= 0 && pg < num_pages;
  }
  if (!ok) {
    if (lane == 0 && status != nullptr) atomicOr(status, kDevIndexRange);
    return;
  }
  uint4* dst = kv_cache + (pg * page_size + pos % page_size) * pieces;
  const uint4* src = kv_new + t * pieces;
  for (int c = lane; c < pieces; c += 32) dst[c] = __ldg(src + c);
}

}  // namespace

cudaError_t launch_paged_kv_write(const void* kv_new, int64_t ntok, int32_t dim,
                                  const int32_t* req_ids, const int32_t* positions,
                                  const int32_t* page_tables, int32_t max_pages, int32_t nreq,
                                  void* kv_cache, int32_t num_pages, int32_t page_size,
                                  uint32_t* dev_status, cudaStream_t stream) {
  const int pieces = dim * 2 / 16;  // bf16 row in 16-byte pieces (dim % 8 == 0)
  const int64_t threads = ntok * 32;
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  paged_kv_write_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      static_cast<const uint4*>(kv_new), ntok, pieces, req_ids, positions, page_tables,
      max_pages, nreq, static_cast<uint4*>(kv_cache), num_pages, page_size, dev_status);
  return cudaGetLastError();
}

}  // namespace tts
