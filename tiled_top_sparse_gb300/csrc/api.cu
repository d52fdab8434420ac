// C ABI of libtts.so: host-side argument validation, workspace carving and
// launches. Every check that needs only host values happens here, before any
// work is enqueued; values that live on the device are checked in the kernels.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/tts.h"
#include "internal.h"
#include "ptx.cuh"

namespace tts {

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank,
                           void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                           const uint32_t* box, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t bx[5], es[5];
  for (uint32_t i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  return g_encode(map, dtype, rank, base, d, s, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace tts

using namespace tts;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline tts_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return TTS_OK;
  if (e == cudaErrorInvalidValue) return TTS_ERR_INVALID_ARG;
  return TTS_ERR_CUDA;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
constexpr size_t kCounterBytes = 256;  // attention workspace: work-item counter

}  // namespace

extern "C" {

const char* tts_status_string(int status) {
  switch (status) {
    case TTS_OK: return "ok";
    case TTS_ERR_INVALID_ARG: return "invalid argument";
    case TTS_ERR_UNSUPPORTED: return "unsupported shape or option";
    case TTS_ERR_CUDA: return "CUDA error";
    case TTS_ERR_INDEX_RANGE: return "device reported an out-of-range index (entry skipped)";
    case TTS_ERR_DEVICE_TIMEOUT: return "device reported an expired bounded wait";
    case TTS_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int tts_status_from_device(uint32_t dev_status) {
  if (dev_status & TTS_DEV_TIMEOUT) return TTS_ERR_DEVICE_TIMEOUT;
  if (dev_status & TTS_DEV_BAD_ARG) return TTS_ERR_INVALID_ARG;
  if (dev_status & TTS_DEV_INDEX_RANGE) return TTS_ERR_INDEX_RANGE;
  return TTS_OK;
}

int tts_version(void) { return 100; }

size_t tts_attn_workspace_bytes(int64_t total_q, int64_t total_k, int32_t num_heads_q,
                                int32_t num_heads_kv, int32_t head_dim, tts_dtype in_dtype) {
  if (total_q < 0 || total_k < 0 || num_heads_q < 1 || num_heads_kv < 1 || head_dim < 1) return 0;
  // 256 bytes for the work-item counter of the persistent kernel, then (fp32 inputs)
  // the bf16 copies of q, k and v.
  if (in_dtype != TTS_F32) return kCounterBytes;
  const size_t nq = (size_t)total_q * num_heads_q * head_dim * 2;
  const size_t nk = (size_t)total_k * num_heads_kv * head_dim * 2;
  return kCounterBytes + align_up(nq, 256) + 2 * align_up(nk, 256);
}

tts_status tts_attn_fwd_varlen(const void* q, const void* k, const void* v, tts_dtype in_dtype,
                               int64_t total_q, int64_t total_k, const int32_t* cu_seqlens_q,
                               const int32_t* cu_seqlens_k, int32_t batch, int32_t max_seqlen_q,
                               int32_t max_seqlen_k, int32_t num_heads_q, int32_t num_heads_kv,
                               int32_t head_dim, int32_t causal, float scale, float* out,
                               float* lse, void* workspace, size_t workspace_bytes,
                               uint32_t* dev_status, void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || cu_seqlens_q == nullptr ||
      cu_seqlens_k == nullptr || out == nullptr)
    return TTS_ERR_INVALID_ARG;
  if (in_dtype != TTS_BF16 && in_dtype != TTS_F32) return TTS_ERR_INVALID_ARG;
  if (batch < 1 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
      num_heads_q < 1 || num_heads_kv < 1 || head_dim < 1)
    return TTS_ERR_INVALID_ARG;
  if (num_heads_q % num_heads_kv != 0) return TTS_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return TTS_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return TTS_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 80 && head_dim != 128) return TTS_ERR_UNSUPPORTED;
  if (total_q > 0x7FFFFF00LL || total_k > 0x7FFFFF00LL) return TTS_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return TTS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (total_q == 0 || max_seqlen_q == 0) return TTS_OK;  // nothing to compute

  const size_t need =
      tts_attn_workspace_bytes(total_q, total_k, num_heads_q, num_heads_kv, head_dim, in_dtype);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return TTS_ERR_WORKSPACE;
  AttnArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.work_counter = static_cast<uint32_t*>(workspace);
  if (in_dtype == TTS_F32) {
    uint8_t* w = static_cast<uint8_t*>(workspace) + kCounterBytes;
    const int64_t nq = total_q * num_heads_q * head_dim;
    const int64_t nk = total_k * num_heads_kv * head_dim;
    void* qb = w;
    void* kb = w + align_up((size_t)nq * 2, 256);
    void* vb = static_cast<uint8_t*>(kb) + align_up((size_t)nk * 2, 256);
    cudaError_t e = launch_f32_to_bf16(static_cast<const float*>(q), qb, nq, st);
    if (e == cudaSuccess) e = launch_f32_to_bf16(static_cast<const float*>(k), kb, nk, st);
    if (e == cudaSuccess) e = launch_f32_to_bf16(static_cast<const float*>(v), vb, nk, st);
    if (e != cudaSuccess) return TTS_ERR_CUDA;
    a.q = qb;
    a.k = kb;
    a.v = vb;
  }
  a.total_q = total_q;
  a.total_k = total_k;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.batch = batch;
  a.max_seqlen_q = max_seqlen_q;
  a.max_seqlen_k = max_seqlen_k;
  a.hq = num_heads_q;
  a.hkv = num_heads_kv;
  a.d = head_dim;
  a.causal = causal;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  a.dev_status = dev_status;
  int drv = 0;
  cudaError_t e = launch_attn_fwd(a, &drv, st);
  if (drv != 0) return TTS_ERR_CUDA;
  return from_cuda(e);
}

tts_status tts_topk_select(const float* logits, int64_t row_stride, int32_t rows,
                           const int32_t* row_starts, const int32_t* row_lens, int32_t k,
                           int32_t* idx, uint32_t* dev_status, void* stream) {
  if (logits == nullptr || row_starts == nullptr || row_lens == nullptr || idx == nullptr)
    return TTS_ERR_INVALID_ARG;
  if (rows < 0 || row_stride < 1 || k < 1) return TTS_ERR_INVALID_ARG;
  if (k > 4096 || row_stride > 16384) return TTS_ERR_UNSUPPORTED;
  if (rows == 0) return TTS_OK;
  return from_cuda(launch_topk_select(logits, row_stride, rows, row_starts, row_lens, k, idx,
                                      dev_status, static_cast<cudaStream_t>(stream)));
}

size_t tts_topk_long_workspace_bytes(int32_t rows, int64_t row_stride, int32_t k) {
  if (rows <= 0 || row_stride < 1 || k < 1 || k > 4096 || row_stride > (int64_t(1) << 30))
    return 0;
  return topk_long_workspace_bytes(rows, row_stride, k);
}

tts_status tts_topk_select_long(const float* logits, int64_t row_stride, int32_t rows,
                                const int32_t* row_starts, const int32_t* row_lens, int32_t k,
                                int32_t* idx, void* workspace, size_t workspace_bytes,
                                uint32_t* dev_status, void* stream) {
  if (logits == nullptr || row_starts == nullptr || row_lens == nullptr || idx == nullptr)
    return TTS_ERR_INVALID_ARG;
  if (rows < 0 || row_stride < 1 || k < 1) return TTS_ERR_INVALID_ARG;
  if (k > 4096 || row_stride > (int64_t(1) << 30)) return TTS_ERR_UNSUPPORTED;
  if (rows == 0) return TTS_OK;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 15) != 0 ||
      workspace_bytes < topk_long_workspace_bytes(rows, row_stride, k))
    return TTS_ERR_INVALID_ARG;
  return from_cuda(launch_topk_long(logits, row_stride, rows, row_starts, row_lens, k, idx,
                                    workspace, dev_status, static_cast<cudaStream_t>(stream)));
}

size_t tts_sparse_workspace_bytes(int32_t nq) {
  if (nq <= 0) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();  // no device: report no split
    return 0;
  }
  return sparse_split_workspace_bytes(nq, sms);
}

tts_status tts_sparse_attn_paged(const void* q, int32_t nq, int32_t num_heads, int32_t dqk,
                                 int32_t dv, const void* kv_cache, int32_t num_pages,
                                 int32_t page_size, const int32_t* page_table,
                                 int32_t num_logical_pages, int32_t kv_len, const int32_t* idx,
                                 int32_t topk, float scale, float* out, float* lse,
                                 void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                 void* stream) {
  if (q == nullptr || kv_cache == nullptr || page_table == nullptr || idx == nullptr ||
      out == nullptr)
    return TTS_ERR_INVALID_ARG;
  if (workspace != nullptr && !aligned16(workspace)) return TTS_ERR_INVALID_ARG;
  if (nq < 0 || num_heads < 1 || dqk < 1 || dv < 1 || dv > dqk || num_pages < 1 ||
      page_size < 1 || num_logical_pages < 0 || kv_len < 0 || topk < 1)
    return TTS_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return TTS_ERR_INVALID_ARG;
  if ((int64_t)num_pages * page_size > 0x7FFFFF00LL) return TTS_ERR_UNSUPPORTED;
  if (num_heads != 128 || dqk != 576 || dv != 512 || topk > 2048) return TTS_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out)) return TTS_ERR_INVALID_ARG;
  if (nq == 0) return TTS_OK;
  SparseArgs a;
  a.q = q;
  a.kv_cache = kv_cache;
  a.page_table = page_table;
  a.idx = idx;
  a.nq = nq;
  a.heads = num_heads;
  a.dqk = dqk;
  a.dv = dv;
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.num_logical_pages = num_logical_pages;
  a.kv_len = kv_len;
  a.topk = topk;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  a.workspace = workspace;
  a.workspace_bytes = workspace == nullptr ? 0 : workspace_bytes;
  a.dev_status = dev_status;
  int drv = 0;
  cudaError_t e = launch_sparse_attn(a, &drv, static_cast<cudaStream_t>(stream));
  if (drv != 0) return TTS_ERR_CUDA;
  return from_cuda(e);
}

tts_status tts_sparse_attn_decode(const void* q, int32_t nreq, int32_t num_heads, int32_t dqk,
                                  int32_t dv, const void* kv_cache, int32_t num_pages,
                                  int32_t page_size, const int32_t* page_tables,
                                  int32_t max_pages, const int32_t* kv_lens, const int32_t* idx,
                                  int32_t topk, float scale, float* out, float* lse,
                                  void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                  void* stream) {
  if (q == nullptr || kv_cache == nullptr || page_tables == nullptr || kv_lens == nullptr ||
      idx == nullptr || out == nullptr)
    return TTS_ERR_INVALID_ARG;
  if (workspace != nullptr && !aligned16(workspace)) return TTS_ERR_INVALID_ARG;
  if (nreq < 0 || num_heads < 1 || dqk < 1 || dv < 1 || dv > dqk || num_pages < 1 ||
      page_size < 1 || max_pages < 1 || topk < 1)
    return TTS_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return TTS_ERR_INVALID_ARG;
  if ((int64_t)num_pages * page_size > 0x7FFFFF00LL ||
      (int64_t)max_pages * page_size > 0x7FFFFF00LL)
    return TTS_ERR_UNSUPPORTED;
  if (num_heads != 128 || dqk != 576 || dv != 512 || topk > 2048) return TTS_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out)) return TTS_ERR_INVALID_ARG;
  if (nreq == 0) return TTS_OK;
  SparseArgs a;
  a.q = q;
  a.kv_cache = kv_cache;
  a.page_table = page_tables;
  a.kv_lens = kv_lens;
  a.pt_stride = max_pages;
  a.idx = idx;
  a.nq = nreq;
  a.heads = num_heads;
  a.dqk = dqk;
  a.dv = dv;
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.num_logical_pages = max_pages;
  a.kv_len = 0;
  a.topk = topk;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  a.workspace = workspace;
  a.workspace_bytes = workspace == nullptr ? 0 : workspace_bytes;
  a.dev_status = dev_status;
  int drv = 0;
  cudaError_t e = launch_sparse_attn(a, &drv, static_cast<cudaStream_t>(stream));
  if (drv != 0) return TTS_ERR_CUDA;
  return from_cuda(e);
}

tts_status tts_paged_kv_write(const void* kv_new, int64_t ntok, int32_t dim,
                              const int32_t* req_ids, const int32_t* positions,
                              const int32_t* page_tables, int32_t max_pages, int32_t nreq,
                              void* kv_cache, int32_t num_pages, int32_t page_size,
                              uint32_t* dev_status, void* stream) {
  if (kv_new == nullptr || positions == nullptr || page_tables == nullptr || kv_cache == nullptr)
    return TTS_ERR_INVALID_ARG;
  if (ntok < 0 || dim < 8 || dim % 8 != 0 || max_pages < 1 || nreq < 1 || num_pages < 1 ||
      page_size < 1)
    return TTS_ERR_INVALID_ARG;
  if (!aligned16(kv_new) || !aligned16(kv_cache)) return TTS_ERR_INVALID_ARG;
  if (ntok == 0) return TTS_OK;
  return from_cuda(launch_paged_kv_write(kv_new, ntok, dim, req_ids, positions, page_tables,
                                         max_pages, nreq, kv_cache, num_pages, page_size,
                                         dev_status, static_cast<cudaStream_t>(stream)));
}

tts_status tts_quantize_fp8_prefill(const void* q, int64_t total_q, int32_t num_heads_q,
                                   const void* k, int64_t total_k, int32_t num_heads_kv,
                                   int32_t head_dim, void* q8, float* q_scale, void* k8,
                                   float* k_scale, void* stream) {
  if (total_q < 0 || total_k < 0 || num_heads_q < 1 || num_heads_kv < 1 ||
      num_heads_kv > 4096 || head_dim < 4 || head_dim % 4 != 0)
    return TTS_ERR_INVALID_ARG;
  if (k_scale == nullptr || !aligned16(k_scale)) return TTS_ERR_INVALID_ARG;
  if (total_q > 0 && (q == nullptr || q8 == nullptr || q_scale == nullptr || !aligned16(q) ||
                      !aligned16(q8) || !aligned16(q_scale)))
    return TTS_ERR_INVALID_ARG;
  if (total_k > 0 && (k == nullptr || k8 == nullptr || !aligned16(k) || !aligned16(k8)))
    return TTS_ERR_INVALID_ARG;
  return from_cuda(launch_quant_fp8_prefill(q, total_q, num_heads_q, k, total_k, num_heads_kv,
                                            head_dim, q8, q_scale, k8, k_scale,
                                            static_cast<cudaStream_t>(stream)));
}

tts_status tts_attn_fwd_varlen_fp8(const void* q8, const float* q_scale, const void* k8,
                                   const float* k_scale, const void* v, int64_t total_q,
                                   int64_t total_k, const int32_t* cu_seqlens_q,
                                   const int32_t* cu_seqlens_k, int32_t batch,
                                   int32_t max_seqlen_q, int32_t max_seqlen_k,
                                   int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim,
                                   int32_t causal, float scale, float* out, float* lse,
                                   void* workspace, size_t workspace_bytes,
                                   uint32_t* dev_status, void* stream) {
  if (q8 == nullptr || q_scale == nullptr || k8 == nullptr || k_scale == nullptr ||
      v == nullptr || cu_seqlens_q == nullptr || cu_seqlens_k == nullptr || out == nullptr)
    return TTS_ERR_INVALID_ARG;
  if (batch < 1 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
      num_heads_q < 1 || num_heads_kv < 1 || head_dim < 1)
    return TTS_ERR_INVALID_ARG;
  if (num_heads_q % num_heads_kv != 0) return TTS_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return TTS_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return TTS_ERR_INVALID_ARG;
  if (head_dim != 128) return TTS_ERR_UNSUPPORTED;
  if (total_q > 0x7FFFFF00LL || total_k > 0x7FFFFF00LL) return TTS_ERR_UNSUPPORTED;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v) || !aligned16(out))
    return TTS_ERR_INVALID_ARG;
  if (total_q == 0 || max_seqlen_q == 0) return TTS_OK;  // nothing to compute
  if (workspace == nullptr || workspace_bytes < kCounterBytes || !aligned16(workspace))
    return TTS_ERR_WORKSPACE;
  AttnArgs a;
  a.q = q8;
  a.k = k8;
  a.v = v;
  a.fp8 = true;
  a.q_scale = q_scale;
  a.k_scale = k_scale;
  a.work_counter = static_cast<uint32_t*>(workspace);
  a.total_q = total_q;
  a.total_k = total_k;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.batch = batch;
  a.max_seqlen_q = max_seqlen_q;
  a.max_seqlen_k = max_seqlen_k;
  a.hq = num_heads_q;
  a.hkv = num_heads_kv;
  a.d = head_dim;
  a.causal = causal;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  a.dev_status = dev_status;
  int drv = 0;
  cudaError_t e = launch_attn_fwd(a, &drv, static_cast<cudaStream_t>(stream));
  if (drv != 0) return TTS_ERR_CUDA;
  return from_cuda(e);
}

tts_status tts_rope_cache(int32_t max_pos, int32_t rot_dim, float base, float* cos_sin,
                          void* stream) {
  if (cos_sin == nullptr || !aligned16(cos_sin)) return TTS_ERR_INVALID_ARG;
  if (max_pos < 1 || rot_dim < 2 || rot_dim % 2 != 0) return TTS_ERR_INVALID_ARG;
  if (!(base > 1.f) || !std::isfinite(base)) return TTS_ERR_INVALID_ARG;
  return from_cuda(launch_rope_cache(max_pos, rot_dim, static_cast<double>(base), cos_sin,
                                     static_cast<cudaStream_t>(stream)));
}

tts_status tts_qkv_rope(const void* x, int64_t n, int32_t hidden, const void* w,
                        const float* bias, const int32_t* positions, const float* cos_sin,
                        int32_t max_pos, int32_t num_heads, int32_t head_dim, void* q, void* k,
                        void* v, uint32_t* dev_status, void* stream) {
  if (n < 0 || n > 0x7FFFFFFFLL || hidden < 8 || hidden % 8 != 0 || max_pos < 1 ||
      num_heads < 1 || head_dim < 2)
    return TTS_ERR_INVALID_ARG;
  const int hpt = qkv_heads_per_tile(head_dim);
  if (hpt == 0 || (3LL * num_heads) % hpt != 0) return TTS_ERR_UNSUPPORTED;
  if ((int64_t)num_heads * head_dim > 0x7FFFFFFFLL / 3) return TTS_ERR_UNSUPPORTED;
  if (n == 0) return TTS_OK;  // empty tensors may come with null data pointers
  if (x == nullptr || w == nullptr || positions == nullptr || cos_sin == nullptr ||
      q == nullptr || k == nullptr || v == nullptr)
    return TTS_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      !aligned16(cos_sin) || (bias != nullptr && !aligned16(bias)))
    return TTS_ERR_INVALID_ARG;
  QkvArgs a;
  a.x = x;
  a.w = w;
  a.bias = bias;
  a.positions = positions;
  a.cos_sin = cos_sin;
  a.n = n;
  a.hidden = hidden;
  a.heads = num_heads;
  a.head_dim = head_dim;
  a.max_pos = max_pos;
  a.q = q;
  a.k = k;
  a.v = v;
  a.dev_status = dev_status;
  int drv = 0;
  cudaError_t e = launch_qkv_rope(a, &drv, static_cast<cudaStream_t>(stream));
  if (drv != 0) return TTS_ERR_CUDA;
  return from_cuda(e);
}

}  // extern "C"
