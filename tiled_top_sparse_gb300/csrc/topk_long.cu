// Deterministic top-k over long rows (windows far beyond one CTA's shared memory).
//
// Same definition as the short-row kernel (the stable-sort fix of "推理引擎的蝴蝶效应",
// section 实验方法和结果, with the lower-index-wins tie rule of "AMD MI250部署
// DeepSeek-V4-Flash", 4.2): the k window positions with the largest values, ordered by
// value descending and, among equal values, by ascending position. It serves windows as
// long as the long-context indexer rows of "从 SGLang Kernel源码到 GPU Trace"
// (section 2.2), where one row no longer fits a CTA.
//
// Each row is cut into chunks of kChunk values, one CTA per (row, chunk). Values map to
// order-preserving 32-bit keys (-0 folded onto +0). Launches, in stream order:
//   1. four histogram passes over the key's four bytes (MSB first). Pass p counts, per
//      chunk, the keys whose higher bytes equal the digits already chosen (per-warp
//      shared histograms, summed per CTA) and adds the counts to the row's histogram
//      with integer atomics. Every CTA of pass p first re-derives the chosen digits from
//      the earlier histograms (the same scan on the same integers, so all CTAs agree).
//      After the last pass the key T of rank k is known, and so is how many keys equal
//      to T are still needed (need_ties). The last pass also keeps each chunk's own
//      histogram, which counts that chunk's keys == T.
//   2. collect: each chunk CTA picks its keys > T and its first m keys == T by position,
//      m = need_ties minus the ties of the earlier chunks (from the kept chunk
//      histograms), clamped to [0, its own ties]; only the chunk where the cut falls
//      ranks its ties (a block scan), every other one takes all or none of them. The
//      picks gather in shared memory and go out behind one atomic per CTA: exactly
//      min(k, len) (key, position) pairs per row, as 64-bit composites
//      key << 32 | ~position, in any slot order.
//   3. sort: one CTA per row sorts the composites descending (bitonic network). The
//      composites are unique, so the result depends on the input alone.
// No float arithmetic decides anything and no CTA waits for another: the order of the
// atomics only changes slot order, which the final sort removes.
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace tts {
namespace {

constexpr int kLThreads = 512;
constexpr int kLWarps = kLThreads / 32;
constexpr int kChunk = 16384;                  // window values per CTA
constexpr int kUnroll = 8;                     // loads in flight per thread
constexpr int kBins = 256;                     // one byte of the key per pass
constexpr int kPasses = 4;
__host__ __device__ constexpr int shift_of(int pass) { return 24 - 8 * pass; }

// Per-row workspace (ints): h [4][256], count [4], chunk histograms [G][256], then the
// candidates (uint64) [k].
struct RowWs {
  int* h[kPasses];
  int* count;
  int* chunk_h;
  uint64_t* cand;
};
__host__ __device__ __forceinline__ int64_t row_ints(int g) {
  return (int64_t)kBins * kPasses + 4 + (int64_t)g * kBins;
}
__host__ __device__ __forceinline__ int64_t row_stride_ints(int g, int k) {
  return (row_ints(g) + 2 * (int64_t)k + 3) & ~int64_t(3);  // keeps the candidates 16-B aligned
}
__device__ __forceinline__ RowWs row_ws(int* ws, int64_t row, int g, int k) {
  int* b = ws + row * row_stride_ints(g, k);
  RowWs w;
  for (int p = 0; p < kPasses; ++p) w.h[p] = b + p * kBins;
  w.count = b + kPasses * kBins;
  w.chunk_h = w.count + 4;
  w.cand = reinterpret_cast<uint64_t*>(b + ((row_ints(g) + 1) & ~int64_t(1)));
  return w;
}

__device__ __forceinline__ uint32_t key_of(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7FFFFFFFu) == 0) u = 0;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread; *total = the block's sum.
__device__ __forceinline__ int scan_excl(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = (lane < kLWarps) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kLWarps) warp_tot[lane] = t;
  }
  __syncthreads();
  const int before = (warp > 0) ? warp_tot[warp - 1] : 0;
  *total = warp_tot[kLWarps - 1];
  __syncthreads();
  return before + x - v;
}

// The digit d of a descending histogram walk at which `remaining` is reached:
// count(bins > d) < remaining <= count(bins >= d). Thread t owns bins 255-8t down to
// 248-8t. Returns d; *above = count(bins > d). Block-collective.
__device__ int pick_digit(const int* hist, int remaining, int* warp_tot, int* s_pick,
                          int* above) {
  const int t = threadIdx.x;
  int c[8], s = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int b = kBins - 1 - 8 * t - q;
    c[q] = (8 * t < kBins) ? __ldcg(hist + b) : 0;
    s += c[q];
  }
  int tot;
  int run = scan_excl(s, warp_tot, &tot);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (run < remaining && remaining <= run + c[q]) {
      s_pick[0] = kBins - 1 - 8 * t - q;
      s_pick[1] = run;
    }
    run += c[q];
  }
  __syncthreads();
  const int d = s_pick[0];
  *above = s_pick[1];
  __syncthreads();
  return d;
}

struct Sel {
  uint32_t prefix, mask;
  int remaining;
};
// The digits chosen by passes [0, upto): block-collective, identical in every CTA.
__device__ Sel chosen(const RowWs& w, int k, int upto, int* warp_tot, int* s_pick) {
  Sel s{0u, 0u, k};
  for (int q = 0; q < upto; ++q) {
    int above;
    const int d = pick_digit(w.h[q], s.remaining, warp_tot, s_pick, &above);
    s.remaining -= above;
    s.prefix |= static_cast<uint32_t>(d) << shift_of(q);
    s.mask |= static_cast<uint32_t>(kBins - 1) << shift_of(q);
  }
  return s;
}

__device__ __forceinline__ bool window_ok(int64_t st, int64_t len, int64_t row_stride) {
  return st >= 0 && len >= 0 && st + len <= row_stride;
}

__global__ void __launch_bounds__(kLThreads) topk_long_hist_kernel(
    const float* __restrict__ logits, int64_t row_stride, const int32_t* __restrict__ row_starts,
    const int32_t* __restrict__ row_lens, int k, int g, int pass, int* ws, uint32_t* status) {
  __shared__ int whist[kLWarps][kBins];  // one histogram per warp: atomics stay in-warp
  __shared__ int warp_tot[kLWarps];
  __shared__ int s_pick[2];
  const int64_t row = blockIdx.x / g;
  const int chunk = blockIdx.x % g;
  const int64_t st = row_starts[row], len = row_lens[row];
  if (!window_ok(st, len, row_stride)) {
    if (pass == 0 && chunk == 0 && threadIdx.x == 0 && status != nullptr)
      atomicOr(status, kDevIndexRange);
    return;
  }
  if (len <= k) return;  // every value of the window is taken
  const RowWs w = row_ws(ws, row, g, k);
  const Sel sel = chosen(w, k, pass, warp_tot, s_pick);
  const int shift = shift_of(pass);
  for (int b = threadIdx.x; b < kLWarps * kBins; b += kLThreads) (&whist[0][0])[b] = 0;
  __syncthreads();
  int* const my = whist[threadIdx.x >> 5];
  const int64_t c0 = (int64_t)chunk * kChunk;
  const int64_t c1 = (c0 + kChunk < len) ? c0 + kChunk : len;
  const float* src = logits + row * row_stride + st;
  for (int64_t j0 = c0; j0 < c1; j0 += kLThreads * kUnroll) {
    float v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = j0 + u * kLThreads + threadIdx.x;
      v[u] = (j < c1) ? __ldg(src + j) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = j0 + u * kLThreads + threadIdx.x;
      const uint32_t key = key_of(v[u]);
      const bool active = j < c1 && (key & sel.mask) == sel.prefix;
      const uint32_t dgt = (key >> shift) & (kBins - 1);
      const uint32_t act = __ballot_sync(0xFFFFFFFFu, active);
      if (active) {  // one shared atomic per distinct digit in the warp
        const uint32_t peers = __match_any_sync(act, dgt);
        if ((__ffs(peers) - 1) == (threadIdx.x & 31)) atomicAdd(&my[dgt], __popc(peers));
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < kBins) {
    int v = 0;
#pragma unroll
    for (int q = 0; q < kLWarps; ++q) v += whist[q][threadIdx.x];
    if (v != 0) atomicAdd(w.h[pass] + threadIdx.x, v);
    if (pass == kPasses - 1) w.chunk_h[(int64_t)chunk * kBins + threadIdx.x] = v;
  }
}

__global__ void __launch_bounds__(kLThreads) topk_long_collect_kernel(
    const float* __restrict__ logits, int64_t row_stride, const int32_t* __restrict__ row_starts,
    const int32_t* __restrict__ row_lens, int k, int g, int* ws, uint32_t* status) {
  extern __shared__ __align__(16) uint64_t picks[];  // [k]: this chunk's picks
  __shared__ int warp_tot[kLWarps];
  __shared__ int s_pick[2];
  __shared__ int s_n, s_base;
  const int64_t row = blockIdx.x / g;
  const int chunk = blockIdx.x % g;
  const int64_t st = row_starts[row], len = row_lens[row];
  if (!window_ok(st, len, row_stride)) return;
  const int64_t c0 = (int64_t)chunk * kChunk;
  if (c0 >= len) return;
  const int64_t c1 = (c0 + kChunk < len) ? c0 + kChunk : len;
  const RowWs w = row_ws(ws, row, g, k);
  const bool all = len <= k;
  uint32_t T = 0;
  int m = 0, n_eq = 0;  // this chunk takes its first m keys == T (of n_eq)
  if (!all) {
    const Sel sel = chosen(w, k, kPasses, warp_tot, s_pick);
    T = sel.prefix;
    const int lo = T & (kBins - 1);
    int part = 0;  // ties (keys == T) in the chunks before this one
    for (int c = threadIdx.x; c < chunk; c += kLThreads)
      part += __ldcg(w.chunk_h + (int64_t)c * kBins + lo);
    int before;
    scan_excl(part, warp_tot, &before);
    n_eq = __ldcg(w.chunk_h + (int64_t)chunk * kBins + lo);
    m = sel.remaining - before;  // need_ties - earlier ties
    m = m < 0 ? 0 : (m > n_eq ? n_eq : m);
  }
  if (threadIdx.x == 0) s_n = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const float* src = logits + row * row_stride + st;
  auto put = [&](bool pick, uint32_t key, int64_t j) {  // warp-aggregated slot in `picks`
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, pick);
    int base = 0;
    if (lane == 0 && b != 0) base = atomicAdd(&s_n, __popc(b));
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    if (pick) {
      const int slot = base + __popc(b & ((1u << lane) - 1u));
      if (slot < k)
        picks[slot] = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~j);
      else if (status != nullptr)
        atomicOr(status, kDevBadArg);  // never: a row has exactly min(k, len) picks
    }
  };
  if (all || m == 0 || m == n_eq) {
    const bool take_eq = all || m > 0;
    for (int64_t j0 = c0; j0 < c1; j0 += kLThreads * kUnroll) {
      float v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t j = j0 + u * kLThreads + threadIdx.x;
        v[u] = (j < c1) ? __ldg(src + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t j = j0 + u * kLThreads + threadIdx.x;
        const uint32_t key = key_of(v[u]);
        put(j < c1 && (all || key > T || (take_eq && key == T)), key, j);
      }
    }
  } else {
    // The chunk where the cut falls: rank its ties by position. Each warp owns a
    // contiguous slice of the chunk; a first sweep counts the slice's ties, a block scan
    // turns the counts into each slice's first rank, a second sweep picks.
    constexpr int kSlice = kChunk / kLWarps;
    const int warp = threadIdx.x >> 5;
    const int64_t s0 = c0 + (int64_t)warp * kSlice;
    const int64_t s1 = (s0 + kSlice < c1) ? s0 + kSlice : c1;
    int mine = 0;
    for (int64_t j0 = s0; j0 < s1; j0 += 32) {
      const int64_t j = j0 + lane;
      mine += __popc(__ballot_sync(0xFFFFFFFFu, j < s1 && key_of(__ldg(src + j)) == T));
    }
    int tot;
    int rank = scan_excl(lane == 0 ? mine : 0, warp_tot, &tot);
    rank = __shfl_sync(0xFFFFFFFFu, rank, 0);  // ties before this warp's slice
    for (int64_t j0 = s0; j0 < s1; j0 += 32) {
      const int64_t j = j0 + lane;
      const uint32_t key = (j < s1) ? key_of(__ldg(src + j)) : 0u;
      const bool eq = j < s1 && key == T;
      const uint32_t e = __ballot_sync(0xFFFFFFFFu, eq);
      const int r = rank + __popc(e & ((1u << lane) - 1u));
      put(j < s1 && (key > T || (eq && r < m)), key, j);
      rank += __popc(e);
    }
  }
  __syncthreads();
  const int n = s_n < k ? s_n : k;
  if (threadIdx.x == 0) s_base = n > 0 ? atomicAdd(w.count, n) : 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kLThreads) {
    if (s_base + i < k)
      w.cand[s_base + i] = picks[i];
    else if (status != nullptr)
      atomicOr(status, kDevBadArg);
  }
}

__global__ void __launch_bounds__(kLThreads) topk_long_sort_kernel(
    const int64_t row_stride, const int32_t* __restrict__ row_starts,
    const int32_t* __restrict__ row_lens, int k, int g, int sort_n, int* ws,
    int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) uint64_t sel[];  // [sort_n]
  const int64_t row = blockIdx.x;
  const int64_t st = row_starts[row], len = row_lens[row];
  int32_t* out = idx + row * (int64_t)k;
  const bool ok = window_ok(st, len, row_stride);
  const int take = ok ? (int)(len < k ? len : k) : 0;
  const RowWs w = row_ws(ws, row, g, k);
  for (int j = threadIdx.x; j < sort_n; j += kLThreads)
    sel[j] = (j < take) ? __ldcg(w.cand + j) : 0ull;  // padding sorts last
  __syncthreads();
  for (int size = 2; size <= sort_n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (sort_n >> 1); i += kLThreads) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = sel[lo], b = sel[hi];
        if ((a < b) == desc) {
          sel[lo] = b;
          sel[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int j = threadIdx.x; j < k; j += kLThreads)
    out[j] = (j < take) ? static_cast<int32_t>(~static_cast<uint32_t>(sel[j] & 0xFFFFFFFFull)) : -1;
}

int chunks_of(int64_t row_stride) { return (int)((row_stride + kChunk - 1) / kChunk); }

}  // namespace

size_t topk_long_workspace_bytes(int32_t rows, int64_t row_stride, int32_t k) {
  if (rows <= 0 || row_stride < 1 || k < 1) return 0;
  return (size_t)rows * (size_t)row_stride_ints(chunks_of(row_stride), k) * sizeof(int);
}

cudaError_t launch_topk_long(const float* logits, int64_t row_stride, int32_t rows,
                             const int32_t* row_starts, const int32_t* row_lens, int32_t k,
                             int32_t* idx, void* workspace, uint32_t* dev_status,
                             cudaStream_t stream) {
  const int g = chunks_of(row_stride);
  const int64_t blocks = (int64_t)rows * g;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  int* ws = static_cast<int*>(workspace);
  // Histograms, counters and chunk histograms start at zero (candidates need no reset).
  const int64_t per_row = row_stride_ints(g, k);
  cudaError_t e = cudaSuccess;
  if (per_row * rows * (int64_t)sizeof(int) > 0)
    e = cudaMemsetAsync(ws, 0, (size_t)per_row * rows * sizeof(int), stream);
  if (e != cudaSuccess) return e;
  for (int pass = 0; pass < kPasses; ++pass) {
    topk_long_hist_kernel<<<(unsigned)blocks, kLThreads, 0, stream>>>(
        logits, row_stride, row_starts, row_lens, k, g, pass, ws, dev_status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  topk_long_collect_kernel<<<(unsigned)blocks, kLThreads, (size_t)k * sizeof(uint64_t), stream>>>(
      logits, row_stride, row_starts, row_lens, k, g, ws, dev_status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int sort_n = 2;
  while (sort_n < k) sort_n <<= 1;
  const size_t smem = (size_t)sort_n * sizeof(uint64_t);
  e = cudaFuncSetAttribute(topk_long_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  topk_long_sort_kernel<<<rows, kLThreads, smem, stream>>>(row_stride, row_starts, row_lens, k,
                                                            g, sort_n, ws, idx);
  return cudaGetLastError();
}

}  // namespace tts
