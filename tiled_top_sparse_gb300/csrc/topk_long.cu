// Deterministic top-k over long rows (windows far beyond one CTA's shared memory).
//
// Same definition as the short-row kernel (the stable-sort fix of "推理引擎的蝴蝶效应",
// section 实验方法和结果, with the lower-index-wins tie rule of "AMD MI250部署
// DeepSeek-V4-Flash", 4.2): the k window positions with the largest values, ordered by
// value descending and, among equal values, by ascending position. It serves windows as
// long as the long-context indexer rows of "从 SGLang Kernel源码到 GPU Trace"
// (section 2.2), where one row no longer fits a CTA.
//
// Values map to order-preserving 32-bit keys (-0 folded onto +0); a key and its position
// travel as the 64-bit composite key << 32 | ~position, which orders exactly as the
// definition does (key descending, then position ascending) and is unique. Sample-select,
// two launches in stream order (after a reset of each row's header):
//   1. compact: one CTA per (row, chunk). Every CTA of a row first reads the same
//      32-value blocks spread evenly over the window (4096 values at most), histograms
//      their keys' top 12 bits and takes as threshold t the lower bound of the bucket
//      where the sample's count from the top reaches its share of 1.5 * min(k, len) +
//      256 values (windows of up to kCap values take t = 0), so all CTAs of a row agree
//      on t without waiting for one another. It then streams its chunk once and appends
//      every value with key >= t to the row's candidate array (gathered per CTA in
//      shared memory, placed by one integer atomic per CTA: the order in the array is
//      arbitrary, its contents are not).
//   2. finish: one CTA per row. If the candidates number at least min(k, len) and fit
//      the array, every selected composite is among them (at least min(k, len) keys are
//      >= t, so the min(k, len)-th largest key is too). They are ranked by buckets: a
//      counting pass over their keys, a scan, and each member of a bucket that starts
//      before min(k, len) placed at its bucket's start plus the number of larger
//      composites in its bucket (a row piling up on a few values takes an MSB-first
//      radix select over the composites and a bitonic sort instead). Else (the sample
//      misjudged the row) the CTA finds the picks exactly on its own: a radix select
//      over the window's keys, a collect that ranks ties by position, and the sort.
// Either way the result is fully determined by the input, and no CTA waits for another.
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace tts {
namespace {

constexpr int kCap = 16384;           // candidates kept per row
constexpr int kLThreads = 512;        // sample and compact CTAs
constexpr int kLWarps = kLThreads / 32;
constexpr int kChunkQuantum = 4096;   // compact chunks are multiples of this many values
constexpr int kUnroll = 8;            // loads in flight per thread (scalar path)
constexpr int kUnroll4 = 4;           // float4 loads in flight per thread (vector path)
constexpr int kSampleBlocks = 128;    // 32-value sample blocks per row, at most
constexpr int kSampleBits = 12;       // key bits of the sample histogram
static_assert(kSampleBlocks * 32 % 512 == 0, "whole rounds of samples per thread");
constexpr int kFinishThreads = 1024;
constexpr int kMaxTake = 4096;        // k <= 4096
constexpr int kFWarps = kFinishThreads / 32;

// Per-row workspace: header {threshold key, candidate count, 2 spare} then kCap
// composites.
constexpr int64_t kRowBytes = 16 + 8 * (int64_t)kCap;
__host__ __device__ __forceinline__ uint32_t* row_head(uint8_t* ws, int64_t row) {
  return reinterpret_cast<uint32_t*>(ws + row * kRowBytes);
}
__host__ __device__ __forceinline__ uint64_t* row_cand(uint8_t* ws, int64_t row) {
  return reinterpret_cast<uint64_t*>(ws + row * kRowBytes + 16);
}

__device__ __forceinline__ uint32_t key_of(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7FFFFFFFu) == 0) u = 0;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint64_t comp_of(uint32_t key, int64_t pos) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(pos));
}
__device__ __forceinline__ bool window_ok(int64_t st, int64_t len, int64_t row_stride) {
  return st >= 0 && len >= 0 && st + len <= row_stride;
}

// Block-wide exclusive scan of one int per thread (NW warps); *total = the block's sum.
template <int NW>
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
    int t = (lane < NW) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < NW) warp_tot[lane] = t;
  }
  __syncthreads();
  const int before = (warp > 0) ? warp_tot[warp - 1] : 0;
  *total = warp_tot[NW - 1];
  __syncthreads();
  return before + x - v;
}

// ---------------------------------------------------------------------------- 1. sample
// The row's threshold key from its sample (block-collective; every CTA of a row computes
// the same value from the same values): the lower bound of the 12-bit key bucket where
// the sample's count from the top reaches its share of 1.5 * take + 256 values.
// Windows are at most 2^30 long, so 32-bit arithmetic holds every quantity here.
__device__ uint32_t sample_threshold(const float* __restrict__ x, uint32_t len, uint32_t take,
                                     uint32_t* hist, int* warp_tot, uint32_t* s_t) {
  uint32_t nb = len / 32;
  if (nb > kSampleBlocks) nb = kSampleBlocks;
  const uint32_t stride = len / nb;  // >= 32
  const uint32_t ns = 32 * nb;       // <= 4096
  // ceil((1.5 take + 256) ns / len): the product is below 6400 * 4096 < 2^32.
  uint32_t want = ((3 * take / 2 + 256) * ns + len - 1) / len;
  if (want > ns) want = ns;
  for (int b = threadIdx.x; b < (1 << kSampleBits); b += kLThreads) hist[b] = 0u;
  if (threadIdx.x == 0) *s_t = 0u;  // sample too small to reach `want`: every key
  __syncthreads();
  // Every sample load goes out before any is used (one round trip, not one per sample).
  constexpr int kPerThread = kSampleBlocks * 32 / kLThreads;
  float sv[kPerThread];
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const uint32_t s = u * kLThreads + threadIdx.x;  // (s >> 5) * stride + 31 < len
    sv[u] = (s < ns) ? __ldg(x + ((s >> 5) * stride + (s & 31))) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const uint32_t s = u * kLThreads + threadIdx.x;
    if (s < ns) atomicAdd(&hist[key_of(sv[u]) >> (32 - kSampleBits)], 1u);
  }
  __syncthreads();
  // Descending walk: thread t owns buckets 4095 - 8t down to 4088 - 8t.
  constexpr int kPer = (1 << kSampleBits) / kLThreads;
  uint32_t c[kPer];
  int sum = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    c[q] = hist[(1 << kSampleBits) - 1 - kPer * threadIdx.x - q];
    sum += (int)c[q];
  }
  int tot;
  int run = scan_excl<kLWarps>(sum, warp_tot, &tot);
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    if (run < (int)want && (int)want <= run + (int)c[q])
      *s_t = (uint32_t)((1 << kSampleBits) - 1 - kPer * (int)threadIdx.x - q) << (32 - kSampleBits);
    run += (int)c[q];
  }
  __syncthreads();
  return *s_t;
}

// ---------------------------------------------------------------------------- 2. compact
// One CTA per (row, chunk): the row's threshold (windows of up to kCap values: every
// key), then one pass over the chunk. The CTA gathers its candidates in shared memory,
// reserves their place in the row's array with one atomic, and copies them there; a CTA
// with more than kLocal candidates adds kCap + 1 to the count instead, which sends its
// row to the exact path.
constexpr int kLocal = 3072;
__global__ void __launch_bounds__(kLThreads, 3) topk_long_compact_kernel(
    const float* __restrict__ logits, int64_t row_stride, const int32_t* __restrict__ row_starts,
    const int32_t* __restrict__ row_lens, int k, int g, int64_t chunk_len, uint8_t* ws) {
  __shared__ uint2 local[kLocal];  // candidates: (value bits, window position)
  __shared__ uint32_t hist[1 << kSampleBits];
  __shared__ int warp_tot[kLWarps];
  __shared__ uint32_t s_n, s_base, s_t;
  const int64_t row = blockIdx.x / g;
  const int chunk = blockIdx.x % g;
  const int64_t st = row_starts[row], len = row_lens[row];
  if (!window_ok(st, len, row_stride)) return;
  const int64_t c0 = (int64_t)chunk * chunk_len;
  const int64_t c1 = (c0 + chunk_len < len) ? c0 + chunk_len : len;
  if (c0 >= c1) return;
  uint32_t* head = row_head(ws, row);
  uint64_t* cand = row_cand(ws, row);
  const float* x = logits + row * row_stride + st;
  const int64_t take = len < k ? len : k;
  const uint32_t t =
      len <= kCap ? 0u : sample_threshold(x, (uint32_t)len, (uint32_t)take, hist, warp_tot, &s_t);
  if (threadIdx.x == 0) s_n = 0u;
  __syncthreads();
  // key(x) >= t  <=>  x >= the float whose key is t (keys order as the floats do, -0 and
  // +0 alike), so each value costs one float comparison. A warp whose lanes hold no
  // candidate moves on after one ballot; otherwise each lane with candidates takes a
  // slot per candidate (a few per cent of the values) and keeps its bits and position;
  // keys and composites are formed once per candidate, on the copy out. t = 0 takes
  // every value.
  const bool all = t == 0u;
  const float tf = __uint_as_float((t & 0x80000000u) ? (t & 0x7FFFFFFFu) : ~t);
  auto put = [&](float v, int64_t j) {  // every value taken: slots follow the positions
    const uint32_t slot = all ? (uint32_t)(j - c0) : atomicAdd(&s_n, 1u);
    if (slot < (uint32_t)kLocal) local[slot] = make_uint2(__float_as_uint(v), (uint32_t)j);
  };
  auto take4 = [&](float4 v, int64_t j, int valid) {  // valid: how many of the 4 are in
    const float m = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    const bool any = valid > 0 && (all || m >= tf);
    if (__ballot_sync(0xFFFFFFFFu, any) == 0u) return;  // warp-uniform
    if (any) {
      if (all || v.x >= tf) put(v.x, j);
      if (valid > 1 && (all || v.y >= tf)) put(v.y, j + 1);
      if (valid > 2 && (all || v.z >= tf)) put(v.z, j + 2);
      if (valid > 3 && (all || v.w >= tf)) put(v.w, j + 3);
    }
  };
  // Whole rounds of loads without bounds checks, then a checked last round. Vector loads
  // when the chunk starts on a 16-byte boundary (the whole CTA agrees).
  if ((reinterpret_cast<uintptr_t>(x + c0) & 15) == 0) {
    constexpr int64_t kStep = 4 * kLThreads * kUnroll4;
    int64_t j0 = c0;
    for (; j0 + kStep <= c1; j0 += kStep) {
      const float4* x4 = reinterpret_cast<const float4*>(x + j0) + threadIdx.x;
      float4 v[kUnroll4];
#pragma unroll
      for (int u = 0; u < kUnroll4; ++u) v[u] = __ldg(x4 + u * kLThreads);
#pragma unroll
      for (int u = 0; u < kUnroll4; ++u) take4(v[u], j0 + 4 * (u * kLThreads + threadIdx.x), 4);
    }
    for (; j0 < c1; j0 += kStep) {
      float4 v[kUnroll4];
#pragma unroll
      for (int u = 0; u < kUnroll4; ++u) {
        const int64_t j = j0 + 4 * (u * kLThreads + threadIdx.x);
        v[u] = (j + 3 < c1) ? __ldg(reinterpret_cast<const float4*>(x + j))
                            : make_float4(j < c1 ? __ldg(x + j) : 0.f,
                                          j + 1 < c1 ? __ldg(x + j + 1) : 0.f,
                                          j + 2 < c1 ? __ldg(x + j + 2) : 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kUnroll4; ++u) {
        const int64_t j = j0 + 4 * (u * kLThreads + threadIdx.x);
        const int64_t in = c1 - j;
        take4(v[u], j, in <= 0 ? 0 : (in >= 4 ? 4 : (int)in));
      }
    }
  } else {
    constexpr int64_t kStep = kLThreads * kUnroll;
    auto take1 = [&](float v, int64_t j, bool ok) {
      const bool c = ok && (all || v >= tf);
      if (__ballot_sync(0xFFFFFFFFu, c) == 0u) return;  // warp-uniform
      if (c) put(v, j);
    };
    int64_t j0 = c0;
    for (; j0 + kStep <= c1; j0 += kStep) {
      float v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u] = __ldg(x + j0 + u * kLThreads + threadIdx.x);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) take1(v[u], j0 + u * kLThreads + threadIdx.x, true);
    }
    for (; j0 < c1; j0 += kStep) {
      float v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t j = j0 + u * kLThreads + threadIdx.x;
        v[u] = (j < c1) ? __ldg(x + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t j = j0 + u * kLThreads + threadIdx.x;
        take1(v[u], j, j < c1);
      }
    }
  }
  if (all && threadIdx.x == 0) s_n = (uint32_t)(c1 - c0);
  __syncthreads();
  const uint32_t n = s_n;
  if (n == 0) return;
  if (threadIdx.x == 0)
    s_base = atomicAdd(head + 1, n <= (uint32_t)kLocal ? n : (uint32_t)kCap + 1u);
  __syncthreads();
  if (n > (uint32_t)kLocal) return;
  const uint32_t base = s_base;
  for (uint32_t i = threadIdx.x; i < n; i += kLThreads)
    if (base + i < (uint32_t)kCap) {
      const uint2 c = local[i];
      cand[base + i] = comp_of(key_of(__uint_as_float(c.x)), c.y);
    }
}

// ---------------------------------------------------------------------------- 3. finish
// Bucket-rank selection of the candidates (the way the one-CTA kernel ranks short
// windows): the candidates' keys are mapped linearly onto kFBuckets buckets in
// descending key order; a counting pass and a scan place every bucket, the buckets that
// start before `take` are filled (atomic cursors: any order inside a bucket), and each
// member's output place is its bucket's start plus the number of larger composites in
// its bucket. A bucket holds at least a value's ties (up to ~90 copies of one bf16 value
// among the picks of a normal row); when the keys take fewer than 256 values, each value
// gets 16 buckets, one per sixteenth of the window in position order, so the
// comparisons stay few. A selectable bucket of more than kFMaxBucket members sends the
// row to the radix select and bitonic sort.
constexpr int kFBuckets = 4096;
constexpr int kFBucketBits = 12;
constexpr uint32_t kFMaxBucket = 512;
constexpr int kFSlots = kMaxTake + kFMaxBucket;  // selectable members, at most
static_assert(kFBuckets == 4 * kFinishThreads, "one uint4 of counters per thread");
// Shared memory after the kCap candidates: per bucket its count / start | end, the
// insertion cursors, then the placed members' composites and their buckets' words. The
// radix path's picks (kMaxTake composites) reuse the same bytes.
constexpr size_t kFRegion = 4 * kFBuckets * 2 + (8 + 4) * (size_t)kFSlots;
static_assert(kFRegion >= 8 * (size_t)kMaxTake, "the picks fit the bucket region");
constexpr size_t kFinishSmem = 8 * (size_t)kCap + kFRegion;

// Bitonic sort, descending, of the n = E * kFinishThreads composites in buf (E = 2 or 4),
// whose result it writes to out as positions (the first `take`, then -1 up to k). Thread
// t holds elements t E .. t E + E - 1 in registers. Compare-exchanges between elements of
// one thread are register swaps, between threads of one warp shuffles; only strides of
// 32 E or more go through shared memory (double-buffered in buf and spare: one barrier
// per such stage). The network is the textbook one: for size = 2, 4, .., n and stride =
// size / 2, .., 1, the element e and its partner e ^ stride are put in descending order
// when e & size is 0 and in ascending order otherwise.
template <int E>
__device__ void sort_desc_out(uint64_t* buf, uint64_t* spare, int take, int k,
                              int32_t* __restrict__ out) {
  constexpr int n = E * kFinishThreads;
  const int lane = threadIdx.x & 31;
  const int e0 = threadIdx.x * E;
  uint64_t v[E];
#pragma unroll
  for (int i = 0; i < E; ++i) v[i] = buf[e0 + i];
  uint64_t* bufs[2] = {spare, buf};
  int which = 0;
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32 * E) {  // partner in another warp: through shared memory
        uint64_t* b = bufs[which];
        which ^= 1;
#pragma unroll
        for (int i = 0; i < E; ++i) b[e0 + i] = v[i];
        __syncthreads();
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const int e = e0 + i;
          const uint64_t p = b[e ^ stride];
          const bool desc = (e & size) == 0, lo = (e & stride) == 0;
          v[i] = (desc == lo) ? (v[i] > p ? v[i] : p) : (v[i] < p ? v[i] : p);
        }
      } else if (stride >= E) {  // partner in another lane of this warp
        const int lm = stride / E;
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const int e = e0 + i;
          const uint64_t p = __shfl_xor_sync(0xFFFFFFFFu, v[i], lm);
          const bool desc = (e & size) == 0, lo = (e & stride) == 0;
          v[i] = (desc == lo) ? (v[i] > p ? v[i] : p) : (v[i] < p ? v[i] : p);
        }
      } else {  // partner in this thread
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const int j = i ^ stride;
          if (j > i) {
            const bool desc = ((e0 + i) & size) == 0;
            const uint64_t a = v[i], c = v[j];
            if ((a < c) == desc) {
              v[i] = c;
              v[j] = a;
            }
          }
        }
      }
    }
  }
  (void)lane;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int e = e0 + i;
    if (e < k)
      out[e] = (e < take) ? static_cast<int32_t>(~static_cast<uint32_t>(v[i] & 0xFFFFFFFFull)) : -1;
  }
  for (int e = n + threadIdx.x; e < k; e += kFinishThreads) out[e] = -1;
}

// Exact selection by one CTA straight from the window: MSB-first radix select (4 x 8
// bits) of the key of rank `take`, then the picks -- every key above it, and the first
// ties in position order (block scans) -- into sel[0, take). Returns nothing; sel holds
// the picks in arbitrary order.
__device__ void select_exact(const float* __restrict__ x, int64_t len, int take, uint64_t* sel,
                             int* hist, int* warp_tot, int* s_digit, int* s_above, int* s_n) {
  uint32_t prefix = 0, mask = 0;
  int remaining = take;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int b = threadIdx.x; b < 256; b += kFinishThreads) hist[b] = 0;
    __syncthreads();
    for (int64_t j = threadIdx.x; j < len; j += kFinishThreads) {
      const uint32_t key = key_of(__ldg(x + j));
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFFu], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {  // lane l owns bins 255 - 8l .. 248 - 8l (descending)
      const int l = threadIdx.x;
      int c[8], s = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        c[q] = hist[255 - 8 * l - q];
        s += c[q];
      }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (l >= o) incl += y;
      }
      int above = incl - s;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (above < remaining && remaining <= above + c[q]) {
          *s_digit = 255 - 8 * l - q;
          *s_above = above;
        }
        above += c[q];
      }
    }
    __syncthreads();
    remaining -= *s_above;
    prefix |= static_cast<uint32_t>(*s_digit) << shift;
    mask |= 0xFFu << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;  // take - remaining keys are > T; `remaining` ties needed
  if (threadIdx.x == 0) *s_n = 0;
  __syncthreads();
  int ties_before = 0;
  for (int64_t j0 = 0; j0 < len; j0 += kFinishThreads) {
    const int64_t j = j0 + threadIdx.x;
    const uint32_t key = (j < len) ? key_of(__ldg(x + j)) : 0u;
    const bool gt = j < len && key > T;
    const bool eq = j < len && key == T;
    int tot;
    const int rank = ties_before + scan_excl<kFWarps>(eq ? 1 : 0, warp_tot, &tot);
    if (gt || (eq && rank < remaining)) {
      const int slot = atomicAdd(s_n, 1);
      if (slot < take) sel[slot] = comp_of(key, j);
    }
    ties_before += tot;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kFinishThreads) topk_long_finish_kernel(
    const float* __restrict__ logits, int64_t row_stride, const int32_t* __restrict__ row_starts,
    const int32_t* __restrict__ row_lens, int k, uint8_t* ws, int32_t* __restrict__ idx,
    uint32_t* status) {
  extern __shared__ __align__(16) uint64_t sel[];  // [kCap] candidates, then kFRegion bytes
  __shared__ int hist[256];
  __shared__ int warp_tot[kFWarps];
  __shared__ int s_digit, s_above, s_n;
  __shared__ unsigned long long s_or, s_and;
  __shared__ uint32_t s_kmin, s_kmax, s_maxc, s_ranked;
  __shared__ uint32_t s_wsum[kFWarps];
  const int64_t row = blockIdx.x;
  const int64_t st = row_starts[row], len = row_lens[row];
  int32_t* out = idx + row * (int64_t)k;
  if (!window_ok(st, len, row_stride)) {
    if (threadIdx.x == 0 && status != nullptr) atomicOr(status, kDevIndexRange);
    for (int j = threadIdx.x; j < k; j += kFinishThreads) out[j] = -1;
    return;
  }
  const int take = (int)(len < k ? len : k);
  const int64_t cnt = (int64_t)__ldcg(row_head(ws, row) + 1);
  uint64_t* const picks = sel + kCap;  // [kMaxTake]: the selected composites, to sort
  // The candidates decide the row unless they are too few (the sample misjudged the
  // row) or too many for the array.
  const bool exact = !(cnt >= take && cnt <= kCap);
  if (!exact) {
    const int n = (int)cnt;
    const uint64_t* cand = row_cand(ws, row);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t* const se = reinterpret_cast<uint32_t*>(sel + kCap);        // [kFBuckets]
    uint32_t* const cur = se + kFBuckets;                                 // [kFBuckets]
    uint64_t* const slot_c = reinterpret_cast<uint64_t*>(cur + kFBuckets);  // [kFSlots]
    uint32_t* const slot_w = reinterpret_cast<uint32_t*>(slot_c + kFSlots);  // [kFSlots]
    // Load, with a census of the bits (OR / AND) so that bytes on which every candidate
    // agrees need no radix pass, and the keys' range for the buckets.
    reinterpret_cast<uint4*>(se)[tid] = make_uint4(0u, 0u, 0u, 0u);
    unsigned long long c_or = 0ull, c_and = ~0ull;
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    for (int j = tid; j < n; j += kFinishThreads) {
      const uint64_t c = __ldcg(cand + j);
      sel[j] = c;
      c_or |= c;
      c_and &= c;
      kmin = min(kmin, static_cast<uint32_t>(c >> 32));
      kmax = max(kmax, static_cast<uint32_t>(c >> 32));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      c_or |= __shfl_xor_sync(0xFFFFFFFFu, c_or, o);
      c_and &= __shfl_xor_sync(0xFFFFFFFFu, c_and, o);
    }
    kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
    kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
    if (tid == 0) {
      s_or = 0ull;
      s_and = ~0ull;
      s_kmin = 0xFFFFFFFFu;
      s_kmax = 0u;
      s_maxc = 0u;
      s_ranked = static_cast<uint32_t>(n);
    }
    __syncthreads();
    if (lane == 0) {
      atomicOr(&s_or, c_or);
      atomicAnd(&s_and, c_and);
      atomicMin(&s_kmin, kmin);
      atomicMax(&s_kmax, kmax);
    }
    __syncthreads();
    // Bucket order is (key descending, position ascending) order. Keys are mapped
    // linearly: bucket (kmax - key) >> sh. When the keys take fewer than 256 distinct
    // values (all candidates share the key's low tz bits, and the span holds fewer than
    // 256 steps of 2^tz), every key gets 16 buckets of its own, one per sixteenth of the
    // window in position order, which splits the ties of one value (the many copies of a
    // bf16 value among a normal row's picks) into groups ranked separately.
    const uint32_t bmax = s_kmax, span = bmax - s_kmin;
    const uint32_t kvary = static_cast<uint32_t>((s_or ^ s_and) >> 32);
    const int tz = kvary != 0u ? __ffs(kvary) - 1 : 0;
    const bool split = (span >> tz) < (uint32_t)(kFBuckets / 16);  // uniform
    const int sh = split ? tz : max(0, (32 - __clz(span)) - kFBucketBits);
    const int psh = max(0, (32 - __clz(static_cast<uint32_t>(len - 1))) - 4);
    auto bucket_of = [&](uint64_t c) -> uint32_t {
      const uint32_t kb = (bmax - static_cast<uint32_t>(c >> 32)) >> sh;
      return split ? (kb << 4) | ((~static_cast<uint32_t>(c)) >> psh) : kb;
    };
    for (int j = tid; j < n; j += kFinishThreads) atomicAdd(&se[bucket_of(sel[j])], 1u);
    __syncthreads();
    {  // exclusive scan: thread tid owns buckets 4 tid .. 4 tid + 3; counts < 2^16
      const uint4 c4 = reinterpret_cast<const uint4*>(se)[tid];
      const uint32_t w[4] = {c4.x, c4.y, c4.z, c4.w};
      const uint32_t tot = w[0] + w[1] + w[2] + w[3];
      uint32_t x = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) s_wsum[warp] = x;
      __syncthreads();
      uint32_t run = x - tot + __reduce_add_sync(0xFFFFFFFFu, lane < warp ? s_wsum[lane] : 0u);
      const uint32_t tk = static_cast<uint32_t>(take);
      uint32_t o[4], mx = 0u;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t e = run + w[q];
        o[q] = run | (e << 16);
        if (run < tk) mx = max(mx, w[q]);  // only buckets that start before take count
        if (run < tk && tk <= e) s_ranked = e;
        run = e;
      }
      mx = __reduce_max_sync(0xFFFFFFFFu, mx);
      if (lane == 0) atomicMax(&s_maxc, mx);
      const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
      reinterpret_cast<uint4*>(se)[tid] = ov;
      reinterpret_cast<uint4*>(cur)[tid] = ov;
    }
    __syncthreads();
    if (s_maxc <= kFMaxBucket) {  // uniform
      const uint32_t ranked = s_ranked;  // <= take + kFMaxBucket
      for (int j = tid; j < n; j += kFinishThreads) {
        const uint64_t c = sel[j];
        const uint32_t b = bucket_of(c);
        const uint32_t bw = se[b];
        if ((bw & 0xFFFFu) < static_cast<uint32_t>(take)) {
          const uint32_t slot = atomicAdd(&cur[b], 1u) & 0xFFFFu;
          slot_c[slot] = c;
          slot_w[slot] = bw;
        }
      }
      __syncthreads();
      // Rank in bucket order: thread t takes slots t, t + kFinishThreads, ...
      for (uint32_t j = tid; j < ranked; j += kFinishThreads) {
        const uint64_t me = slot_c[j];
        const uint32_t bw = slot_w[j], s0 = bw & 0xFFFFu;
        uint32_t rank = 0;
        const uint64_t* const end = slot_c + (bw >> 16);
#pragma unroll 1
        for (const uint64_t* m = slot_c + s0; m < end; ++m) rank += *m > me ? 1u : 0u;
        const uint32_t dst = s0 + rank;
        if (dst < static_cast<uint32_t>(take))
          out[dst] = static_cast<int32_t>(~static_cast<uint32_t>(me & 0xFFFFFFFFull));
      }
      for (int e = take + tid; e < k; e += kFinishThreads) out[e] = -1;
      return;
    } else {
      const uint64_t varying = s_or ^ s_and, common = s_and;
      // The take-th largest composite C among the candidates (they are unique): an
      // MSB-first radix select over the 64 bits, then every composite >= C is a pick.
      uint64_t prefix = 0, mask = 0;
      int remaining = take;
      for (int pass = 0; pass < 8 && n > take; ++pass) {
        const int shift = 56 - 8 * pass;
        if (((varying >> shift) & 0xFFu) == 0) {  // the same byte in every candidate
          prefix |= common & (0xFFull << shift);
          mask |= 0xFFull << shift;
          continue;
        }
        for (int b = threadIdx.x; b < 256; b += kFinishThreads) hist[b] = 0;
        __syncthreads();
        for (int j = threadIdx.x; j < n; j += kFinishThreads) {
          const uint64_t c = sel[j];
          if ((c & mask) == prefix) atomicAdd(&hist[(int)((c >> shift) & 0xFFu)], 1);
        }
        __syncthreads();
        if (threadIdx.x < 32) {  // lane l owns bins 255 - 8l .. 248 - 8l (descending)
          const int l = threadIdx.x;
          int c[8], sum = 0;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            c[q] = hist[255 - 8 * l - q];
            sum += c[q];
          }
          int incl = sum;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (l >= o) incl += y;
          }
          int above = incl - sum;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (above < remaining && remaining <= above + c[q]) {
              s_digit = 255 - 8 * l - q;
              s_above = above;
            }
            above += c[q];
          }
        }
        __syncthreads();
        remaining -= s_above;
        prefix |= static_cast<uint64_t>(s_digit) << shift;
        mask |= 0xFFull << shift;
        __syncthreads();
      }
      const uint64_t C = (n > take) ? prefix : 0ull;  // n == take: every candidate
      if (threadIdx.x == 0) s_n = 0;
      __syncthreads();
      for (int j = threadIdx.x; j < n; j += kFinishThreads) {
        const uint64_t c = sel[j];
        if (c >= C) {
          const int slot = atomicAdd(&s_n, 1);
          if (slot < take) picks[slot] = c;
        }
      }
    }
  } else {  // the sample misjudged this row: select exactly from the window itself
    select_exact(logits + row * row_stride + st, len, take, picks, hist, warp_tot, &s_digit,
                 &s_above, &s_n);
  }
  // Sort the picks (padding with 0, which sorts last) and write their positions.
  const int sort_n = take <= 2 * kFinishThreads ? 2 * kFinishThreads : 4 * kFinishThreads;
  for (int j = take + threadIdx.x; j < sort_n; j += kFinishThreads) picks[j] = 0ull;
  __syncthreads();
  if (sort_n == 2 * kFinishThreads)
    sort_desc_out<2>(picks, sel, take, k, out);
  else
    sort_desc_out<4>(picks, sel, take, k, out);
}

// Chunk length (a multiple of kChunkQuantum) such that rows x chunks about fills the
// device with three compact CTAs per SM.
int64_t chunk_len_for(int64_t row_stride, int32_t rows, int sms) {
  int64_t want = (int64_t)(3 * (sms > 0 ? sms : 1)) / (rows > 0 ? rows : 1);
  if (want < 1) want = 1;
  int64_t len = (row_stride + want - 1) / want;
  len = (len + kChunkQuantum - 1) / kChunkQuantum * kChunkQuantum;
  return len;
}

}  // namespace

size_t topk_long_workspace_bytes(int32_t rows, int64_t row_stride, int32_t k) {
  if (rows <= 0 || row_stride < 1 || k < 1) return 0;
  return (size_t)rows * (size_t)kRowBytes;
}

cudaError_t launch_topk_long(const float* logits, int64_t row_stride, int32_t rows,
                             const int32_t* row_starts, const int32_t* row_lens, int32_t k,
                             int32_t* idx, void* workspace, uint32_t* dev_status,
                             cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t ea = cudaGetDevice(&dev);
  if (ea == cudaSuccess) ea = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ea != cudaSuccess) return ea;
  const int64_t chunk_len = chunk_len_for(row_stride, rows, sms);
  const int64_t g64 = (row_stride + chunk_len - 1) / chunk_len;
  const int64_t blocks = (int64_t)rows * g64;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const int g = (int)g64;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // Each row's header (threshold, candidate count) starts at zero.
  cudaError_t e = cudaMemset2DAsync(ws, (size_t)kRowBytes, 0, 16, (size_t)rows, stream);
  if (e != cudaSuccess) return e;
  topk_long_compact_kernel<<<(unsigned)blocks, kLThreads, 0, stream>>>(
      logits, row_stride, row_starts, row_lens, k, g, chunk_len, ws);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = kFinishSmem;
  e = cudaFuncSetAttribute(topk_long_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  topk_long_finish_kernel<<<rows, kFinishThreads, smem, stream>>>(
      logits, row_stride, row_starts, row_lens, k, ws, idx, dev_status);
  return cudaGetLastError();
}

}  // namespace tts
