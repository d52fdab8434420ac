// Internal launch interface between the C ABI layer and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tts {

// ---- top-k
size_t topk_smem_bytes(int64_t row_stride, int k);
cudaError_t launch_topk_select(const float* logits, int64_t row_stride, int32_t rows,
                               const int32_t* row_starts, const int32_t* row_lens, int32_t k,
                               int32_t* idx, uint32_t* dev_status, cudaStream_t stream);
size_t topk_long_workspace_bytes(int32_t rows, int64_t row_stride, int32_t k);
cudaError_t launch_topk_long(const float* logits, int64_t row_stride, int32_t rows,
                             const int32_t* row_starts, const int32_t* row_lens, int32_t k,
                             int32_t* idx, void* workspace, uint32_t* dev_status,
                             cudaStream_t stream);

// ---- paged KV cache write
cudaError_t launch_paged_kv_write(const void* kv_new, int64_t ntok, int32_t dim,
                                  const int32_t* req_ids, const int32_t* positions,
                                  const int32_t* page_tables, int32_t max_pages, int32_t nreq,
                                  void* kv_cache, int32_t num_pages, int32_t page_size,
                                  uint32_t* dev_status, cudaStream_t stream);

// ---- dense attention
struct AttnArgs {
  const void* q;  // bf16
  const void* k;
  const void* v;
  int64_t total_q, total_k;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int batch, max_seqlen_q, max_seqlen_k, hq, hkv, d, causal;
  float scale;
  float* out;
  float* lse;
  uint32_t* dev_status;
  uint32_t* work_counter;  // device scratch word (the launch zeroes it on the stream)
  bool fp8 = false;        // q, k are e4m3 codes with the scales below (head_dim 128)
  const float* q_scale = nullptr;  // [total_q, hq]
  const float* k_scale = nullptr;  // [hkv]
};
// Returns cudaSuccess or the first error; *drv_err receives a CUresult from tensor-map encoding.
cudaError_t launch_attn_fwd(const AttnArgs& a, int* drv_err, cudaStream_t stream);
cudaError_t launch_f32_to_bf16(const float* in, void* out, int64_t n, cudaStream_t stream);
// e4m3 block quantization of the prefill's q (per token and head) and k (per KV head).
cudaError_t launch_quant_fp8_prefill(const void* q, int64_t total_q, int hq, const void* k,
                                     int64_t total_k, int hkv, int d, void* q8, float* q_scale,
                                     void* k8, float* k_scale, cudaStream_t stream);

// ---- sparse attention
struct SparseArgs {
  const void* q;         // bf16 [nq, H, dqk]
  const void* kv_cache;  // bf16 [pages, page_size, dqk]
  const int32_t* page_table;
  const int32_t* kv_lens = nullptr;  // decode: per-query lengths (else kv_len for all)
  int pt_stride = 0;                 // decode: page-table row stride (else one shared table)
  const int32_t* idx;
  int nq, heads, dqk, dv, num_pages, page_size, num_logical_pages, kv_len, topk;
  float scale;
  float* out;
  float* lse;
  void* workspace;  // optional: enables the split of the last, partial wave
  size_t workspace_bytes;
  uint32_t* dev_status;
};
cudaError_t launch_sparse_attn(const SparseArgs& a, int* drv_err, cudaStream_t stream);
// Workspace bytes with which launch_sparse_attn splits the last wave of nq queries on a
// device with `sms` SMs (0: no split for this shape).
size_t sparse_split_workspace_bytes(int nq, int sms);

// ---- vision QKV projection + RoPE
struct QkvArgs {
  const void* x;  // bf16 [n, hidden]
  const void* w;  // bf16 [3 * heads * head_dim, hidden]
  const float* bias;
  const int32_t* positions;
  const float* cos_sin;  // [max_pos, head_dim / 2, 2]
  int64_t n;
  int hidden, heads, head_dim, max_pos;
  void* q;
  void* k;
  void* v;
  uint32_t* dev_status;
};
// Heads per output tile for head_dim (0: head_dim not built).
int qkv_heads_per_tile(int head_dim);
cudaError_t launch_qkv_rope(const QkvArgs& a, int* drv_err, cudaStream_t stream);
cudaError_t launch_rope_cache(int max_pos, int rot_dim, double base, float* cos_sin,
                              cudaStream_t stream);

// ---- tensor maps (driver entry point fetched through the runtime)
CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank,
                           void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                           const uint32_t* box, CUtensorMapSwizzle swizzle);

}  // namespace tts
