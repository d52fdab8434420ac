/*
 * tts.h -- C ABI of libtts.so: tiled dense attention, deterministic top-k
 * selection and permutation-invariant paged sparse attention for sm_103a.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named as device pointers must point to device memory of the
 *   current CUDA device; sizes and scalars are host values. The caller owns
 *   all memory. The library allocates nothing and keeps no state between
 *   calls except cached driver entry points and, per device, the number of
 *   CTA pairs tts_qkv_rope can keep resident (queried on its first call) and
 *   the largest shared-memory limit tts_topk_select has set on its kernels
 *   (a launch refused after a context reset sets it again).
 *   One exception: tts_attn_fwd_varlen_f32_noalloc (end of this file) uses a
 *   fixed TTS_NOALLOC_SCRATCH_BYTES array of device memory that the library
 *   itself holds on every GPU that loads it, and caches that array's address
 *   per device and context.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *   entry point only enqueues work on that stream; none synchronises.
 * - Host-side argument errors return a non-OK status and enqueue nothing.
 *   A launch failure returns TTS_ERR_CUDA. Errors are never swallowed.
 * - Values only the device can see (cu_seqlens, index lists, page tables,
 *   top-k windows) are checked by the kernels: a bad entry is skipped (never
 *   dereferenced) and a TTS_DEV_* bit is OR-ed into *dev_status when
 *   dev_status is not NULL. Kernels never trap. A bounded wait that expires
 *   sets TTS_DEV_TIMEOUT and the kernel returns early (its output is then
 *   undefined). tts_status_from_device() turns a read-back word into a status.
 * - No float atomics are used anywhere: for fixed inputs every output is
 *   bitwise reproducible run to run.
 */
#ifndef TTS_H_
#define TTS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TTS_OK = 0,
  TTS_ERR_INVALID_ARG = 1,    /* null pointer, negative size, misaligned pointer, ... */
  TTS_ERR_UNSUPPORTED = 2,    /* legal but not built (head_dim, head count, sizes) */
  TTS_ERR_CUDA = 3,           /* a CUDA runtime / driver call or a launch failed */
  TTS_ERR_INDEX_RANGE = 4,    /* device reported an out-of-range entry (skipped) */
  TTS_ERR_DEVICE_TIMEOUT = 5, /* device reported an expired bounded wait */
  TTS_ERR_WORKSPACE = 6       /* workspace missing or smaller than required */
} tts_status;

typedef enum { TTS_BF16 = 0, TTS_F32 = 1 } tts_dtype;

/* Bits a kernel ORs into *dev_status. */
#define TTS_DEV_INDEX_RANGE 0x1u
#define TTS_DEV_TIMEOUT 0x2u
#define TTS_DEV_BAD_ARG 0x4u

const char* tts_status_string(int status);
/* Map a dev_status word read back to the host onto a status (timeout wins). */
int tts_status_from_device(uint32_t dev_status);
/* Library version, major * 10000 + minor * 100 + patch. */
int tts_version(void);

/*
 * Dense attention forward over packed variable-length sequences.
 *
 * Follows the piece-wise attention of "DeepSeek V4.1 上 4×RTX 3090：视觉链路的两个坑
 * 和修复" (section 三: S = Q_blk K^T, row softmax, P V, rows mapped back to the
 * global rows of the block) and the varlen batch of "从 SGLang Kernel源码到 GPU
 * Trace" (section 2.2: cu_seqlens_q / cu_seqlens_k; keys beyond a sequence's
 * length are skipped, section 3.2), with FP32 softmax statistics and FP32
 * accumulation ("AMD MI250部署DeepSeek-V4-Flash", sections 3.1 and 4.1) and the
 * causal mask applied as -inf (section 3.3).
 *
 * For sequence b (tokens cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q, and
 * cu_seqlens_k[b] .. of k / v), query row i, head h, KV head g = h / (Hq/Hkv):
 *   s_j = scale * q[i,h,:] . k[j,g,:]   for visible j: j < Lk and, if causal,
 *                                       j <= i + (Lk - Lq)  (bottom-right)
 *   out[i,h,:] = sum_j softmax(s)_j v[j,g,:]      lse[i,h] = ln sum_j e^{s_j}
 * A row with no visible key gets out = 0, lse = -inf.
 *
 * q    device, [total_q, num_heads_q, head_dim], row-major, in_dtype
 * k, v device, [total_k, num_heads_kv, head_dim], row-major, in_dtype
 *      TTS_F32 inputs are rounded to bf16 (nearest-even) on the device first;
 *      the MMAs always take bf16 operands and accumulate in fp32.
 * cu_seqlens_q, cu_seqlens_k  device int32 [batch + 1], non-decreasing from 0,
 *      last entry <= total_q / total_k (checked on the device: TTS_DEV_BAD_ARG,
 *      offending sequences are skipped).
 * max_seqlen_q, max_seqlen_k  host upper bounds of the sequence lengths (they
 *      size the grid; a longer sequence is flagged TTS_DEV_BAD_ARG and skipped).
 * head_dim   64, 80 or 128.    num_heads_q % num_heads_kv == 0.
 * out  device fp32 [total_q, num_heads_q, head_dim]; lse device fp32
 *      [total_q, num_heads_q] (may be NULL). Rows of q not covered by any
 *      sequence are left untouched.
 * workspace  device scratch of at least tts_attn_workspace_bytes(...) bytes
 *      (16-byte aligned), owned by the caller and not used after the stream
 *      reaches the end of this call: 256 bytes for the persistent kernel's
 *      work-item counter (zeroed on the stream by the call itself), plus the
 *      bf16 copies of q, k and v when in_dtype is TTS_F32. Concurrent calls
 *      need separate workspaces. Missing or smaller: TTS_ERR_WORKSPACE.
 * q, k, v must be 16-byte aligned.
 */
size_t tts_attn_workspace_bytes(int64_t total_q, int64_t total_k, int32_t num_heads_q,
                                int32_t num_heads_kv, int32_t head_dim, tts_dtype in_dtype);

tts_status tts_attn_fwd_varlen(const void* q, const void* k, const void* v, tts_dtype in_dtype,
                               int64_t total_q, int64_t total_k, const int32_t* cu_seqlens_q,
                               const int32_t* cu_seqlens_k, int32_t batch, int32_t max_seqlen_q,
                               int32_t max_seqlen_k, int32_t num_heads_q, int32_t num_heads_kv,
                               int32_t head_dim, int32_t causal, float scale, float* out,
                               float* lse, void* workspace, size_t workspace_bytes,
                               uint32_t* dev_status, void* stream);

/*
 * Deterministic top-k selection over per-row indexer logits.
 *
 * Follows "推理引擎的蝴蝶效应 -- 从V32 模型的输出不一致说起" (section 实验方法和
 * 结果: logits (323, 2590) with row_starts / row_lens give top-k indices
 * (323, 2048); a stable sort replaces the unstable top-k) and the fixed
 * tie-break rule of "AMD MI250部署DeepSeek-V4-Flash" (section 4.2).
 *
 * Row r's window is logits[r * row_stride + row_starts[r] .. + row_lens[r]).
 * idx[r, 0 .. min(k, len)) = window positions (relative to row_starts[r])
 * ordered by value descending, equal values by ascending position (lower
 * index wins); remaining slots are -1. Values compare as floats (-0 == +0).
 * NaN logits are not supported (their rank is unspecified).
 * A window that does not fit in the row sets TTS_DEV_INDEX_RANGE and yields
 * an all -1 row.
 *
 * logits   device fp32 [rows, row_stride]
 * row_starts, row_lens  device int32 [rows]
 * idx      device int32 [rows, k]
 * Limits: 1 <= k <= 4096, 1 <= row_stride <= 16384 (TTS_ERR_UNSUPPORTED otherwise).
 */
tts_status tts_topk_select(const float* logits, int64_t row_stride, int32_t rows,
                           const int32_t* row_starts, const int32_t* row_lens, int32_t k,
                           int32_t* idx, uint32_t* dev_status, void* stream);

/*
 * Top-k over long rows: the same result as tts_topk_select (same definition,
 * tie rule and output layout, see above) for rows of any length up to 2^30,
 * such as the long-context indexer rows of "从 SGLang Kernel源码到 GPU Trace"
 * (section 2.2). Sample-select in three launches: per row, a threshold key from a
 * sample of the window (1/32 of it at most); one pass over the window, split over
 * many CTAs, that keeps every value at or above the threshold (integer atomics
 * only); per row, the k largest kept values placed in (value, position) order by
 * value buckets ranked inside (a radix select and a sort for rows piling up on a
 * few values). A row the sample misjudges (fewer than min(k, len) kept,
 * or more than 16384, e.g. a row piling up on one value) is instead finished
 * exactly by one CTA straight from the window (radix select, ties ranked by
 * position): correct for every input, but a few passes over the row at one SM's
 * bandwidth. The result is deterministic.
 *
 * workspace  device scratch of at least tts_topk_long_workspace_bytes(rows,
 *            row_stride, k) bytes, 16-byte aligned, owned by the caller and
 *            not shared by two calls in flight; its contents are overwritten
 *            (the call zeroes what it needs on the stream first).
 * Limits: 1 <= k <= 4096, 1 <= row_stride <= 2^30 (TTS_ERR_UNSUPPORTED
 * otherwise); a too small or misaligned workspace is TTS_ERR_INVALID_ARG.
 * Errors in row_starts / row_lens behave as in tts_topk_select.
 */
size_t tts_topk_long_workspace_bytes(int32_t rows, int64_t row_stride, int32_t k);
tts_status tts_topk_select_long(const float* logits, int64_t row_stride, int32_t rows,
                                const int32_t* row_starts, const int32_t* row_lens, int32_t k,
                                int32_t* idx, void* workspace, size_t workspace_bytes,
                                uint32_t* dev_status, void* stream);

/*
 * Sparse attention over a paged KV cache, invariant to the order of the index list.
 *
 * Follows "推理引擎的蝴蝶效应 -- 从V32 模型的输出不一致说起" (section 实验方法和
 * 结果: the KV rows are fetched through pagetable_1 and sorting the index list
 * makes outputs identical; section 进一步探索, equations 1-2: the online-softmax
 * merge whose rounding depends on block order). The kernel sorts each query's
 * index list ascending before attending, so any permutation of idx[n, :] gives
 * bitwise identical out / lse.
 *
 * For query n and head h: the valid entries i of idx[n, :] (0 <= i < kv_len,
 * page_table[i / page_size] in [0, num_pages)), sorted ascending, duplicates
 * kept; row_i = kv_cache[page_table[i / page_size], i % page_size, :];
 *   s_i = scale * q[n,h,:] . row_i[0:dqk]
 *   out[n,h,:] = sum_i softmax(s)_i row_i[0:dv]     lse[n,h] = ln sum_i e^{s_i}
 * Entries equal to -1 are empty slots. Other invalid entries are skipped and set
 * TTS_DEV_INDEX_RANGE. A query with no valid entry gets out = 0, lse = -inf.
 *
 * q          device bf16 [nq, num_heads, dqk]
 * kv_cache   device bf16 [num_pages, page_size, dqk]  (V = the first dv columns)
 * page_table device int32 [num_logical_pages]
 * idx        device int32 [nq, topk]
 * out        device fp32 [nq, num_heads, dv];  lse device fp32 [nq, num_heads] or NULL
 * workspace  device scratch, optional (NULL / 0 bytes: not used). With at least
 *            tts_sparse_workspace_bytes(nq) bytes: (1) a first launch writes every
 *            query's canonical list (validated, sorted, resolved to physical rows) into
 *            the workspace, so the attention CTAs start gathering at once instead of
 *            sorting first (same lists, same results bit for bit); (2) the (query,
 *            V half) units of the last, partial wave of CTAs each run as 2 to 16 CTAs
 *            (as many as fit that wave) over consecutive tiles of the sorted list, and
 *            their unnormalised results are merged in part order (the online-softmax
 *            merge) by the last of them to finish, or, beyond 4 parts, by a merge
 *            launch of one CTA per (unit, 16 heads). The result stays deterministic and
 *            order-invariant; split units round differently from unsplit ones. Owned by
 *            the caller; calls that may overlap on the GPU need separate workspaces.
 * Built shape: num_heads = 128, dqk = 576, dv = 512, 1 <= topk <= 2048,
 * page_size >= 1 (TTS_ERR_UNSUPPORTED otherwise). q, kv_cache, out and workspace
 * 16-byte aligned.
 */
tts_status tts_sparse_attn_paged(const void* q, int32_t nq, int32_t num_heads, int32_t dqk,
                                 int32_t dv, const void* kv_cache, int32_t num_pages,
                                 int32_t page_size, const int32_t* page_table,
                                 int32_t num_logical_pages, int32_t kv_len, const int32_t* idx,
                                 int32_t topk, float scale, float* out, float* lse,
                                 void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                 void* stream);

/*
 * Decode-shaped sparse attention: one query per request, each request with its own
 * page table and length, in one call. The same computation as tts_sparse_attn_paged
 * (see above: sorted index list, so bitwise invariant under index permutations),
 * with query n reading its KV rows through page_tables[n, :] and its own kv_lens[n]:
 * the per-request page tables of the paged cache in "从 SGLang Kernel源码到 GPU
 * Trace" (section 2.2, PagedKVCache) under the sparse attention and index rule of
 * "推理引擎的蝴蝶效应" (sections 实验方法和结果, 进一步探索). With few requests, the
 * workspace lets every (request, V half) unit run as up to 16 CTAs over consecutive
 * tiles of its sorted list, merged in part order (split-KV with a fixed-order combine).
 *
 * q           device bf16 [nreq, num_heads, dqk]
 * kv_cache    device bf16 [num_pages, page_size, dqk], shared by all requests
 * page_tables device int32 [nreq, max_pages]; entry g of row n = physical page of
 *             request n's logical page g
 * kv_lens     device int32 [nreq]; a negative length reads as 0 and is reported
 * idx         device int32 [nreq, topk], logical positions in the request's sequence
 * out, lse, workspace, dev_status, errors and built shape: as tts_sparse_attn_paged
 * (the workspace size is tts_sparse_workspace_bytes(nreq)); max_pages >= 1.
 */
tts_status tts_sparse_attn_decode(const void* q, int32_t nreq, int32_t num_heads, int32_t dqk,
                                  int32_t dv, const void* kv_cache, int32_t num_pages,
                                  int32_t page_size, const int32_t* page_tables,
                                  int32_t max_pages, const int32_t* kv_lens, const int32_t* idx,
                                  int32_t topk, float scale, float* out, float* lse,
                                  void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                  void* stream);

/*
 * Paged KV cache write: the write path of the cache read above ("推理引擎的蝴蝶效应",
 * section 实验方法和结果, where the cache is reached through pagetable_1 and its write
 * path is ruled out; "从 SGLang Kernel源码到 GPU Trace", section 2.2, PagedKVCache).
 * Token t (of ntok) belongs to request req_ids[t] (req_ids NULL: request t) at logical
 * position positions[t]; its row kv_new[t, :] is copied to
 *   kv_cache[page_tables[req, pos / page_size], pos % page_size, :].
 * A token whose request is outside [0, nreq), whose position is outside
 * [0, max_pages * page_size) or whose page entry is outside [0, num_pages) is skipped
 * and sets TTS_DEV_INDEX_RANGE. Two tokens of one call with the same destination: the
 * row left there is one of theirs, which one is unspecified.
 *
 * kv_new      device bf16 [ntok, dim], dim a multiple of 8
 * req_ids     device int32 [ntok] or NULL;  positions device int32 [ntok]
 * page_tables device int32 [nreq, max_pages]
 * kv_cache    device bf16 [num_pages, page_size, dim]
 * kv_new and kv_cache 16-byte aligned; nothing is allocated.
 */
tts_status tts_paged_kv_write(const void* kv_new, int64_t ntok, int32_t dim,
                              const int32_t* req_ids, const int32_t* positions,
                              const int32_t* page_tables, int32_t max_pages, int32_t nreq,
                              void* kv_cache, int32_t num_pages, int32_t page_size,
                              uint32_t* dev_status, void* stream);

/*
 * Workspace bytes for nq queries on the current device (0 for nq <= 0 or without a
 * device): the partial results of the split last wave (when the shape splits; at most
 * about 132 KB per SM), then, from the next 256-byte boundary, the canonical lists
 * (4 bytes per query rounded up to 256, plus nq * 2048 * 4 bytes).
 */
size_t tts_sparse_workspace_bytes(int32_t nq);

/*
 * FP8 (e4m3) block quantization of the prefill's q and k, for tts_attn_fwd_varlen_fp8.
 *
 * "从 SGLang Kernel源码到 GPU Trace" (section 3.2) runs part of the prefill in FP8; "AMD
 * MI250部署DeepSeek-V4-Flash" allows FP8 matmul inputs with FP32 accumulation (section
 * 4.1) and quantizes by blocks (section 5.3). The pages fix neither the format nor the
 * blocks; the reading taken: e4m3 (largest finite value 448), one block per (token,
 * head) row of q and one block per KV head of k (all its tokens), scale = max|x| / 448
 * in fp32 (1 for an all-zero block), code = e4m3(x / scale) with the division in fp32
 * and the conversion to nearest, ties to even, saturating at +-448.
 *
 * q        device bf16 [total_q, num_heads_q, head_dim]
 * k        device bf16 [total_k, num_heads_kv, head_dim]
 * q8, k8   device e4m3 codes, one byte per value, same layouts, written
 * q_scale  device fp32 [total_q, num_heads_q], written
 * k_scale  device fp32 [num_heads_kv], written (it also holds the per-head maxima
 *          between the launches this call enqueues)
 * head_dim a multiple of 4; num_heads_kv <= 4096; all pointers 16-byte aligned; a
 * zero-sized q (or k) may come with null pointers for its tensors. Deterministic: the
 * per-head maxima are reduced with integer atomics on the bits of |x|.
 */
tts_status tts_quantize_fp8_prefill(const void* q, int64_t total_q, int32_t num_heads_q,
                                   const void* k, int64_t total_k, int32_t num_heads_kv,
                                   int32_t head_dim, void* q8, float* q_scale, void* k8,
                                   float* k_scale, void* stream);

/*
 * Dense attention forward with FP8 (e4m3) q and k in the S = Q K^T product.
 *
 * As tts_attn_fwd_varlen (same sequences, masks, layouts of v / out / lse, workspace of
 * tts_attn_workspace_bytes(..., TTS_BF16) bytes, device checks and errors), except that
 * q and k arrive as e4m3 codes with the scales of tts_quantize_fp8_prefill, and the
 * scores are
 *   s_j = scale * q_scale[i, h] * k_scale[g] * sum_t q8[i,h,t] k8[j,g,t]
 * computed by e4m3 x e4m3 tensor-core products accumulated in fp32. The softmax
 * statistics stay fp32 and P V stays bf16 x bf16 with fp32 accumulation, as the
 * precision table of "AMD MI250部署DeepSeek-V4-Flash" (section 4.1) keeps the softmax
 * path and P V. head_dim must be 128 (else TTS_ERR_UNSUPPORTED).
 *
 * q8      device e4m3 [total_q, num_heads_q, 128]     q_scale device fp32 [total_q, num_heads_q]
 * k8      device e4m3 [total_k, num_heads_kv, 128]    k_scale device fp32 [num_heads_kv]
 * v       device bf16 [total_k, num_heads_kv, 128]
 */
tts_status tts_attn_fwd_varlen_fp8(const void* q8, const float* q_scale, const void* k8,
                                   const float* k_scale, const void* v, int64_t total_q,
                                   int64_t total_k, const int32_t* cu_seqlens_q,
                                   const int32_t* cu_seqlens_k, int32_t batch,
                                   int32_t max_seqlen_q, int32_t max_seqlen_k,
                                   int32_t num_heads_q, int32_t num_heads_kv, int32_t head_dim,
                                   int32_t causal, float scale, float* out, float* lse,
                                   void* workspace, size_t workspace_bytes,
                                   uint32_t* dev_status, void* stream);

/*
 * cos/sin table of rotary position embedding, built once and read by tts_qkv_rope.
 *
 * The position-indexed table of "从 SGLang Kernel源码到 GPU Trace" (section 3.3: cos
 * and sin of every position up to the longest sequence, computed ahead of the
 * prefill instead of inside it). For position p < max_pos and pair j < rot_dim / 2:
 *   cos_sin[(p * rot_dim/2 + j) * 2 + 0] = cos(p * base^(-2j / rot_dim))
 *   cos_sin[(p * rot_dim/2 + j) * 2 + 1] = sin(p * base^(-2j / rot_dim))
 * The angle and its cosine / sine are evaluated in double precision and rounded to
 * fp32 once.
 *
 * cos_sin  device fp32 [max_pos, rot_dim / 2, 2], 16-byte aligned, written.
 * max_pos >= 1, rot_dim even and >= 2, base > 1 and finite; otherwise
 * TTS_ERR_INVALID_ARG and nothing is enqueued.
 */
tts_status tts_rope_cache(int32_t max_pos, int32_t rot_dim, float base, float* cos_sin,
                          void* stream);

/*
 * Vision-encoder QKV projection fused with rotary position embedding.
 *
 * The qkv + RoPE step of the vision encoder in "DeepSeek V4.1 上 4×RTX 3090：视觉链路
 * 的两个坑和修复" (坑 1, checked block by block against a CPU reference), reading its
 * cos/sin from the table of tts_rope_cache ("从 SGLang Kernel源码到 GPU Trace",
 * section 3.3). For token t, with y = W x[t] + bias (y has 3 * H * d entries: the H
 * q heads, then the H k heads, then the H v heads, d each):
 *   q[t,h,j]       = y_q[j] c - y_q[j + d/2] s      for j < d/2,
 *   q[t,h,j + d/2] = y_q[j] s + y_q[j + d/2] c      (c, s) = cos_sin[positions[t], j]
 * and the same for k; v[t,h,:] = y_v. The pages do not fix the RoPE variant; this
 * is one-dimensional rotate-half RoPE on the full head (pairs j, j + d/2).
 * The products run on the tensor cores with bf16 operands and an fp32 accumulator;
 * bias and rotation are applied in fp32; results are rounded to bf16 (nearest even).
 *
 * x          device bf16 [n, hidden], row-major
 * w          device bf16 [3 * num_heads * head_dim, hidden], row-major (the weight
 *            of a linear layer: one row per output feature)
 * bias       device fp32 [3 * num_heads * head_dim], or NULL for none
 * positions  device int32 [n]; an entry outside [0, max_pos) is skipped: that token's
 *            q and k are written as zeros and TTS_DEV_INDEX_RANGE is set
 * cos_sin    device fp32 [max_pos, head_dim / 2, 2] as written by tts_rope_cache
 *            (rot_dim = head_dim)
 * q, k, v    device bf16 [n, num_heads, head_dim], written
 * head_dim in {64, 80, 128}; 3 * num_heads must be a multiple of the heads per output
 * tile (3 for head_dim 80, 4 for 64, 2 for 128): otherwise TTS_ERR_UNSUPPORTED.
 * hidden >= 8 and a multiple of 8; x, w, q, k, v, bias and cos_sin 16-byte aligned;
 * n <= 2^31 - 1; otherwise TTS_ERR_INVALID_ARG. n = 0 enqueues nothing and accepts
 * null data pointers (after the size checks above). Nothing is
 * allocated; every output element is written by exactly one thread, so the result is
 * bitwise reproducible.
 */
tts_status tts_qkv_rope(const void* x, int64_t n, int32_t hidden, const void* w,
                        const float* bias, const int32_t* positions, const float* cos_sin,
                        int32_t max_pos, int32_t num_heads, int32_t head_dim, void* q, void* k,
                        void* v, uint32_t* dev_status, void* stream);

/*
 * Diagnostics (no counterpart in the pages): launches one thread that waits on a
 * barrier phase nothing completes. The wait is bounded like every wait in the library:
 * after about one second it ORs TTS_DEV_TIMEOUT into *dev_status (device pointer,
 * required) and the kernel returns, leaving the CUDA context usable. Used by the
 * test-suite to check the timeout path without faulting or hanging the GPU.
 */
tts_status tts_debug_wait_timeout(uint32_t* dev_status, void* stream);

/*
 * Allocation-free variant of tts_attn_fwd_varlen for fp32 q / k / v.
 *
 * This entry point has no counterpart in the pages; it exists for callers that
 * cannot allocate device memory when they call: for example code running while
 * another runtime has reserved the device's whole memory pool, or a serving loop
 * that forbids allocation after start-up. The fp32 path needs scratch for the bf16
 * copies of its inputs; here that scratch is a fixed array inside the library
 * (TTS_NOALLOC_SCRATCH_BYTES of device memory, reserved on every GPU that loads the
 * library until the process exits), so the call takes no workspace argument and
 * calls no allocator. Everything else -- arguments, layouts, results, errors -- is
 * as for tts_attn_fwd_varlen with in_dtype = TTS_F32.
 *
 * - The call needs tts_attn_workspace_bytes(total_q, total_k, num_heads_q,
 *   num_heads_kv, head_dim, TTS_F32) bytes of the array: 256 bytes for the work
 *   counter, plus the bf16 copies, 2 * total_q * num_heads_q * head_dim bytes for q
 *   and 2 * total_k * num_heads_kv * head_dim bytes each for k and v, every copy
 *   rounded up to a multiple of 256. Inputs that need more than
 *   TTS_NOALLOC_SCRATCH_BYTES are rejected with TTS_ERR_WORKSPACE before any work
 *   is enqueued.
 * - The first call on a device looks up the array's device address on that device
 *   (which must be current) and caches it per context, so a new context (after a
 *   device reset, say) looks it up again; make that first call before capturing a
 *   stream into a CUDA graph.
 * - Every call on a device shares the one array, which keeps the last call's
 *   contents; nothing in it needs to start at zero, because each call overwrites
 *   every byte it reads. Calls that overlap on the GPU (e.g. on two streams at
 *   once) race on the array and give undefined results: serialise them.
 */
#define TTS_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

tts_status tts_attn_fwd_varlen_f32_noalloc(const float* q, const float* k, const float* v,
                                           int64_t total_q, int64_t total_k,
                                           const int32_t* cu_seqlens_q,
                                           const int32_t* cu_seqlens_k, int32_t batch,
                                           int32_t max_seqlen_q, int32_t max_seqlen_k,
                                           int32_t num_heads_q, int32_t num_heads_kv,
                                           int32_t head_dim, int32_t causal, float scale,
                                           float* out, float* lse, uint32_t* dev_status,
                                           void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TTS_H_ */
