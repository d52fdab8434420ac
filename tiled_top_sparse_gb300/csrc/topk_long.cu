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
// order-preserving 32-bit keys (-0 folded onto +0); a key and its position travel as the
// 64-bit composite key << 32 | ~position, which orders exactly as the definition does
// (key descending, then position ascending) and is unique. Launches, in stream order:
//   1. pass 0: histogram of the keys' top byte, per chunk (kept) and per row (integer
//      atomics). The row's histogram fixes the top byte d0 of the k-th key.
//   2. compact: keys whose top byte is above d0 are picks (fewer than k of them); keys
//      whose top byte is d0 are the candidates, copied as composites into a per-row list
//      in position order (each chunk's offset comes from the kept chunk histograms, each
//      warp's from a block scan). Only these two launches read the rows.
//   3. passes 1-3 over the candidates: histograms of the next three bytes among the
//      candidates matching the digits chosen so far. Every CTA re-derives those digits
//      from the earlier histograms (the same scan on the same integers, so all CTAs
//      agree). After pass 3 the key T of rank k is known, and so is how many candidates
//      equal to T are still needed; pass 3 keeps each chunk's own histogram too.
//   4. collect: each candidate chunk picks its keys > T and its first m keys == T in
//      list (= position) order, m = the ties still needed minus those of the earlier
//      chunks, clamped to its own count; only the chunk where the cut falls ranks ties.
//   5. sort: one CTA per row sorts its k composites descending (bitonic network).
// No float arithmetic decides anything and no CTA waits for another; atomics only
// change the slot order of the picks, which the final sort removes.
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

// Per-row workspace: ints h [4][256], count [4], chunk histograms of pass 0 and of
// pass 3 [G][256] each (zeroed per call); then the picks (uint64) [k] and the candidate
// list (uint64) [row_stride].
struct RowWs {
  int* h[kPasses];
  int* count;
  int* chunk_h0;
  int* chunk_h3;
  uint64_t* cand;
  uint64_t* list;
};
__host__ __device__ __forceinline__ int64_t zeroed_bytes(int g) {
  return (((int64_t)kBins * kPasses + 4 + 2 * (int64_t)g * kBins) * 4 + 15) & ~int64_t(15);
}
__host__ __device__ __forceinline__ int64_t row_bytes(int g, int k, int64_t row_stride) {
  return zeroed_bytes(g) + 8 * ((int64_t)k + (k & 1)) + 8 * (row_stride + (row_stride & 1));
}
__device__ __forceinline__ RowWs row_ws(uint8_t* ws, int64_t row, int g, int k,
                                        int64_t row_stride) {
  uint8_t* b = ws + row * row_bytes(g, k, row_stride);
  int* bi = reinterpret_cast<int*>(b);
  RowWs w;
  for (int p = 0; p < kPasses; ++p) w.h[p] = bi + p * kBins;
  w.count = bi + kPasses * kBins;
  w.chunk_h0 = w.count + 4;
  w.chunk_h3 = w.chunk_h0 + (int64_t)g * kBins;
  w.cand = reinterpret_cast<uint64_t*>(b + zeroed_bytes(g));
  w.list = w.cand + k + (k & 1);
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

// Where a CTA's keys come from: the row itself (pass 0, compact) or the row's candidate
// list (passes 1-3, collect). Both give (key, composite) for an index of the range.
struct RowSrc {
  const float* x;  // the window, or nullptr for the list
  const uint64_t* list;
  __device__ __forceinline__ uint64_t get(int64_t j) const {
    if (x != nullptr) {
      const uint32_t key = key_of(__ldg(x + j));
      return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~j);
    }
    return __ldcg(list + j);
  }
};

// Per (row, chunk) setup shared by the kernels. Returns false for an invalid window. The
// chunks cut the window; over the candidate list the kernel sets the range itself
// (in_list) once it knows the list's length.
struct Job {
  int64_t row, c0, c1;
  int chunk;
  bool all;  // len <= k: every value of the window is a pick
  RowWs w;
  RowSrc src;
};
template <bool kList>
__device__ __forceinline__ bool setup(Job& jb, const float* logits, int64_t row_stride,
                                      const int32_t* row_starts, const int32_t* row_lens,
                                      int k, int g, uint8_t* ws) {
  jb.row = blockIdx.x / g;
  jb.chunk = blockIdx.x % g;
  const int64_t st = row_starts[jb.row], len = row_lens[jb.row];
  if (!window_ok(st, len, row_stride)) return false;
  jb.all = len <= k;
  jb.w = row_ws(ws, jb.row, g, k, row_stride);
  jb.src.x = kList ? nullptr : logits + jb.row * row_stride + st;
  jb.src.list = jb.w.list;
  jb.c0 = (int64_t)jb.chunk * kChunk;
  jb.c1 = (jb.c0 + kChunk < len) ? jb.c0 + kChunk : len;
  return true;
}
// Over the candidate list: its length, which the compact launch records in count[1].
__device__ __forceinline__ void in_list(Job& jb) {
  const int64_t n = __ldcg(jb.w.count + 1);
  jb.c1 = (jb.c0 + kChunk < n) ? jb.c0 + kChunk : n;
}

// Histogram of key byte `pass` over the CTA's range, among keys matching the digits
// chosen by the earlier passes; added to the row's histogram, and kept per chunk for
// passes 0 and 3.
template <bool kList>
__global__ void __launch_bounds__(kLThreads) topk_long_hist_kernel(
    const float* __restrict__ logits, int64_t row_stride, const int32_t* __restrict__ row_starts,
    const int32_t* __restrict__ row_lens, int k, int g, int pass, uint8_t* ws,
    uint32_t* status) {
  __shared__ int whist[kLWarps][kBins];  // one histogram per warp: atomics stay in-warp
  __shared__ int warp_tot[kLWarps];
  __shared__ int s_pick[2];
  Job jb;
  if (!setup<kList>(jb, logits, row_stride, row_starts, row_lens, k, g, ws)) {
    if (!kList && blockIdx.x % g == 0 && threadIdx.x == 0 && status != nullptr) {
      const int64_t r = blockIdx.x / g, st = row_starts[r], len = row_lens[r];
      if (!window_ok(st, len, row_stride)) atomicOr(status, kDevIndexRange);
    }
    return;
  }
  if (jb.all) return;
  if (kList) {
    in_list(jb);
    if (jb.c0 >= jb.c1) return;  // beyond the list (its chunk histograms stay zero)
  }
  const Sel sel = chosen(jb.w, k, pass, warp_tot, s_pick);
  const int shift = shift_of(pass);
  for (int b = threadIdx.x; b < kLWarps * kBins; b += kLThreads) (&whist[0][0])[b] = 0;
  __syncthreads();
  int* const my = whist[threadIdx.x >> 5];
  for (int64_t j0 = jb.c0; j0 < jb.c1; j0 += kLThreads * kUnroll) {
    uint32_t v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = j0 + u * kLThreads + threadIdx.x;
      if (kList)
        v[u] = (j < jb.c1) ? static_cast<uint32_t>(__ldcg(jb.src.list + j) >> 32) : 0u;
      else
        v[u] = (j < jb.c1) ? key_of(__ldg(jb.src.x + j)) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = j0 + u * kLThreads + threadIdx.x;
      const uint32_t key = v[u];
      const bool active = j < jb.c1 && (key & sel.mask) == sel.prefix;
      if (active) atomicAdd(&my[(key >> shift) & (kBins - 1)], 1);  // this warp's own bins
    }
  }
  __syncthreads();
  if (threadIdx.x < kBins) {
    int v = 0;
#pragma unroll
    for (int q = 0; q < kLWarps; ++q) v += whist[q][threadIdx.x];
    if (v != 0) atomicAdd(jb.w.h[pass] + threadIdx.x, v);
    int* keep = pass == 0 ? jb.w.chunk_h0 : (pass == kPasses - 1 ? jb.w.chunk_h3 : nullptr);
    if (keep != nullptr) keep[(int64_t)jb.chunk * kBins + threadIdx.x] = v;
  }
}

// Picks gathered in shared memory (warp-aggregated slots), then sent to the row's pick
// array behind one atomic per CTA.
struct PickBuf {
  uint64_t* s;
  int* s_n;
  int k;
  uint32_t* status;
  __device__ __forceinline__ void put(bool pick, uint64_t comp) const {
    const int lane = threadIdx.x & 31;
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, pick);
    int base = 0;
    if (lane == 0 && b != 0) base = atomicAdd(s_n, __popc(b));
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    if (pick) {
      const int slot = base + __popc(b & ((1u << lane) - 1u));
      if (slot < k)
        s[slot] = comp;
      else if (status != nullptr)
        atomicOr(status, kDevBadArg);  // never: a row has exactly min(k, len) picks
    }
  }
};
__device__ __forceinline__ void flush_picks(const PickBuf& pb, const RowWs& w, int* s_base) {
  __syncthreads();
  const int n = *pb.s_n < pb.k ? *pb.s_n : pb.k;
  if (threadIdx.x == 0) *s_base = n > 0 ? atomicAdd(w.count, n) : 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kLThreads) {
    if (*s_base + i < pb.k)
      w.cand[*s_base + i] = pb.s[i];
    else if (pb.status != nullptr)
      atomicOr(pb.status, kDevBadArg);
  }
}

// Keys with a top byte above the k-th key's are picks; those with its top byte go to the
// candidate list, in position order.
__global__ void __launch_bounds__(kLThreads) topk_long_compact_kernel(
    const float* __restrict__ logits, int64_t row_stride, const int32_t* __restrict__ row_starts,
    const int32_t* __restrict__ row_lens, int k, int g, uint8_t* ws, uint32_t* status) {
  extern __shared__ __align__(16) uint64_t picks[];  // [k]
  __shared__ int warp_tot[kLWarps];
  __shared__ int s_pick[2];
  __shared__ int s_n, s_base;
  Job jb;
  if (!setup<false>(jb, logits, row_stride, row_starts, row_lens, k, g, ws)) return;
  if (jb.c0 >= jb.c1) return;
  if (threadIdx.x == 0) s_n = 0;
  __syncthreads();
  const PickBuf pb{picks, &s_n, k, status};
  if (jb.all) {
    for (int64_t j0 = jb.c0; j0 < jb.c1; j0 += kLThreads) {
      const int64_t j = j0 + threadIdx.x;
      pb.put(j < jb.c1, j < jb.c1 ? jb.src.get(j) : 0ull);
    }
    flush_picks(pb, jb.w, &s_base);
    return;
  }
  const Sel sel = chosen(jb.w, k, 1, warp_tot, s_pick);
  const uint32_t d0 = sel.prefix >> 24;
  if (jb.chunk == 0 && threadIdx.x == 0) jb.w.count[1] = __ldcg(jb.w.h[0] + d0);
  int part = 0;  // candidates in the chunks before this one
  for (int c = threadIdx.x; c < jb.chunk; c += kLThreads)
    part += __ldcg(jb.w.chunk_h0 + (int64_t)c * kBins + d0);
  int base;
  scan_excl(part, warp_tot, &base);
  // each warp owns a contiguous slice: count its candidates, scan, then write them
  constexpr int kSlice = kChunk / kLWarps;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t s0 = jb.c0 + (int64_t)warp * kSlice;
  const int64_t s1 = (s0 + kSlice < jb.c1) ? s0 + kSlice : jb.c1;
  const float* x = jb.src.x;
  int mine = 0;
  for (int64_t j0 = s0; j0 < s1; j0 += 32 * kUnroll) {
    float v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = j0 + 32 * u + lane;
      v[u] = (j < s1) ? __ldg(x + j) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = j0 + 32 * u + lane;
      mine += __popc(__ballot_sync(0xFFFFFFFFu, j < s1 && (key_of(v[u]) >> 24) == d0));
    }
  }
  int tot;
  int at = scan_excl(lane == 0 ? mine : 0, warp_tot, &tot);
  at = base + __shfl_sync(0xFFFFFFFFu, at, 0);
  for (int64_t j0 = s0; j0 < s1; j0 += 32 * kUnroll) {
    float v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = j0 + 32 * u + lane;
      v[u] = (j < s1) ? __ldg(x + j) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = j0 + 32 * u + lane;
      const uint32_t key = key_of(v[u]);
      const uint64_t comp = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~j);
      const uint32_t top = key >> 24;
      const bool cand = j < s1 && top == d0;
      const uint32_t b = __ballot_sync(0xFFFFFFFFu, cand);
      if (cand) jb.w.list[at + __popc(b & ((1u << lane) - 1u))] = comp;
      at += __popc(b);
      pb.put(j < s1 && top > d0, comp);
    }
  }
  flush_picks(pb, jb.w, &s_base);
}

// Candidates > T, and the first m candidates == T of this chunk (list order = position
// order), are picks.
__global__ void __launch_bounds__(kLThreads) topk_long_collect_kernel(
    const float* __restrict__ logits, int64_t row_stride, const int32_t* __restrict__ row_starts,
    const int32_t* __restrict__ row_lens, int k, int g, uint8_t* ws, uint32_t* status) {
  extern __shared__ __align__(16) uint64_t picks[];  // [k]
  __shared__ int warp_tot[kLWarps];
  __shared__ int s_pick[2];
  __shared__ int s_n, s_base;
  Job jb;
  if (!setup<true>(jb, logits, row_stride, row_starts, row_lens, k, g, ws) || jb.all) return;
  in_list(jb);
  if (jb.c0 >= jb.c1) return;
  const Sel sel = chosen(jb.w, k, kPasses, warp_tot, s_pick);
  const uint32_t T = sel.prefix;
  const int lo = T & (kBins - 1);
  int part = 0;  // ties (keys == T) in the chunks before this one
  for (int c = threadIdx.x; c < jb.chunk; c += kLThreads)
    part += __ldcg(jb.w.chunk_h3 + (int64_t)c * kBins + lo);
  int before;
  scan_excl(part, warp_tot, &before);
  const int n_eq = __ldcg(jb.w.chunk_h3 + (int64_t)jb.chunk * kBins + lo);
  int m = sel.remaining - before;
  m = m < 0 ? 0 : (m > n_eq ? n_eq : m);
  if (threadIdx.x == 0) s_n = 0;
  __syncthreads();
  const PickBuf pb{picks, &s_n, k, status};
  if (m == 0 || m == n_eq) {
    const bool take_eq = m > 0;
    for (int64_t j0 = jb.c0; j0 < jb.c1; j0 += kLThreads * kUnroll) {
      uint64_t v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t j = j0 + u * kLThreads + threadIdx.x;
        v[u] = (j < jb.c1) ? jb.src.get(j) : 0ull;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t j = j0 + u * kLThreads + threadIdx.x;
        const uint32_t key = static_cast<uint32_t>(v[u] >> 32);
        pb.put(j < jb.c1 && (key > T || (take_eq && key == T)), v[u]);
      }
    }
  } else {  // the chunk where the cut falls: per-warp slices ranked by one block scan
    constexpr int kSlice = kChunk / kLWarps;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t s0 = jb.c0 + (int64_t)warp * kSlice;
    const int64_t s1 = (s0 + kSlice < jb.c1) ? s0 + kSlice : jb.c1;
    int mine = 0;
    for (int64_t j0 = s0; j0 < s1; j0 += 32) {
      const int64_t j = j0 + lane;
      const bool eq = j < s1 && static_cast<uint32_t>(jb.src.get(j) >> 32) == T;
      mine += __popc(__ballot_sync(0xFFFFFFFFu, eq));
    }
    int tot;
    int rank = scan_excl(lane == 0 ? mine : 0, warp_tot, &tot);
    rank = __shfl_sync(0xFFFFFFFFu, rank, 0);  // ties before this warp's slice
    for (int64_t j0 = s0; j0 < s1; j0 += 32) {
      const int64_t j = j0 + lane;
      const uint64_t comp = (j < s1) ? jb.src.get(j) : 0ull;
      const uint32_t key = static_cast<uint32_t>(comp >> 32);
      const bool eq = j < s1 && key == T;
      const uint32_t e = __ballot_sync(0xFFFFFFFFu, eq);
      const int r = rank + __popc(e & ((1u << lane) - 1u));
      pb.put(j < s1 && (key > T || (eq && r < m)), comp);
      rank += __popc(e);
    }
  }
  flush_picks(pb, jb.w, &s_base);
}

constexpr int kSortThreads = 1024;  // one compare-exchange per thread and stage at k = 2048
__global__ void __launch_bounds__(kSortThreads) topk_long_sort_kernel(
    const int64_t row_stride, const int32_t* __restrict__ row_starts,
    const int32_t* __restrict__ row_lens, int k, int g, int sort_n, uint8_t* ws,
    int32_t* __restrict__ idx) {
  extern __shared__ __align__(16) uint64_t sel[];  // [sort_n]
  const int64_t row = blockIdx.x;
  const int64_t st = row_starts[row], len = row_lens[row];
  int32_t* out = idx + row * (int64_t)k;
  const bool ok = window_ok(st, len, row_stride);
  const int take = ok ? (int)(len < k ? len : k) : 0;
  const RowWs w = row_ws(ws, row, g, k, row_stride);
  for (int j = threadIdx.x; j < sort_n; j += kSortThreads)
    sel[j] = (j < take) ? __ldcg(w.cand + j) : 0ull;  // padding sorts last
  __syncthreads();
  for (int size = 2; size <= sort_n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (sort_n >> 1); i += kSortThreads) {
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
  for (int j = threadIdx.x; j < k; j += kSortThreads)
    out[j] = (j < take) ? static_cast<int32_t>(~static_cast<uint32_t>(sel[j] & 0xFFFFFFFFull)) : -1;
}

int chunks_of(int64_t row_stride) { return (int)((row_stride + kChunk - 1) / kChunk); }

}  // namespace

size_t topk_long_workspace_bytes(int32_t rows, int64_t row_stride, int32_t k) {
  if (rows <= 0 || row_stride < 1 || k < 1) return 0;
  return (size_t)rows * (size_t)row_bytes(chunks_of(row_stride), k, row_stride);
}

cudaError_t launch_topk_long(const float* logits, int64_t row_stride, int32_t rows,
                             const int32_t* row_starts, const int32_t* row_lens, int32_t k,
                             int32_t* idx, void* workspace, uint32_t* dev_status,
                             cudaStream_t stream) {
  const int g = chunks_of(row_stride);
  const int64_t blocks = (int64_t)rows * g;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // Histograms, counters and chunk histograms start at zero (the rest needs no reset).
  cudaError_t e = cudaMemset2DAsync(ws, (size_t)row_bytes(g, k, row_stride), 0,
                                    (size_t)zeroed_bytes(g), (size_t)rows, stream);
  if (e != cudaSuccess) return e;
  const size_t pick_smem = (size_t)k * sizeof(uint64_t);
  topk_long_hist_kernel<false><<<(unsigned)blocks, kLThreads, 0, stream>>>(
      logits, row_stride, row_starts, row_lens, k, g, 0, ws, dev_status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  topk_long_compact_kernel<<<(unsigned)blocks, kLThreads, pick_smem, stream>>>(
      logits, row_stride, row_starts, row_lens, k, g, ws, dev_status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  for (int pass = 1; pass < kPasses; ++pass) {
    topk_long_hist_kernel<true><<<(unsigned)blocks, kLThreads, 0, stream>>>(
        logits, row_stride, row_starts, row_lens, k, g, pass, ws, dev_status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  topk_long_collect_kernel<<<(unsigned)blocks, kLThreads, pick_smem, stream>>>(
      logits, row_stride, row_starts, row_lens, k, g, ws, dev_status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int sort_n = 2;
  while (sort_n < k) sort_n <<= 1;
  const size_t smem = (size_t)sort_n * sizeof(uint64_t);
  e = cudaFuncSetAttribute(topk_long_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  topk_long_sort_kernel<<<rows, kSortThreads, smem, stream>>>(row_stride, row_starts, row_lens, k,
                                                            g, sort_n, ws, idx);
  return cudaGetLastError();
}

}  // namespace tts
