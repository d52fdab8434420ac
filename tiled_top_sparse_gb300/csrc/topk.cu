// Deterministic top-k selection: one CTA per row.
//
// Definition (the stable-sort fix of "推理引擎的蝴蝶效应", section 实验方法和结果,
// with the lower-index-wins tie rule of "AMD MI250部署DeepSeek-V4-Flash", 4.2):
// the k window positions with the largest values, ordered by value descending
// and, among equal values, by ascending position.
//
// Windows of up to 4096 values (the indexer's rows are 2590 long) take the bucket-rank
// path: a counting pass places value buckets (a linear map of each sign half's keys
// onto 2048 buckets) at their final offsets, and each selectable element is ranked
// inside its bucket by comparing unique (key, position) composites. A window whose
// values pile up on few keys (a bucket of more than 128 values) takes a stable LSD
// radix sort of the whole window on the inverted key instead (passes of 8 bits;
// stability keeps equal values in ascending position). Both give the same result.
// Longer windows take the select-then-sort path:
//  1. map each float of the window to an order-preserving 32-bit key
//     (-0 folded onto +0, so equal floats get equal keys);
//  2. MSB-first radix select over 4 x 8-bit digits finds the key T of rank k
//     and how many elements equal to T are still needed;
//  3. compact the selected set: every key > T, plus the lowest-position keys == T
//     (positions ranked by a block-wide scan, so the choice never depends on
//     thread timing);
//  4. sort the selected (key, position) pairs as one 64-bit composite
//     (key << 32 | ~position) descending with a bitonic network. Composites are
//     unique, so the result is fully determined by the input.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace tts {
namespace {

constexpr int kTopkThreads = 512;
constexpr int kWarps = kTopkThreads / 32;
// The one-CTA paths hold E values per thread, so they sort windows of up to
// kTopkThreads * E values: E = 6 where rows are at most 3072 long (less shared memory:
// four CTAs per SM), E = 8 up to 4096 (three).
template <int E>
constexpr int sort_max() {
  return kTopkThreads * E;
}
// Shared memory of the radix path: two key/position buffers and per-warp digit counters.
template <int E>
constexpr size_t radix_smem() {
  return 2 * sort_max<E>() * (4 + 2) + kWarps * 256 * 4;
}

__device__ __forceinline__ uint32_t ordered_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7FFFFFFFu) == 0) u = 0;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread; returns the exclusive prefix,
// writes the block total to *total. Uses `warp_tot` (kWarps ints) in smem.
__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = (lane < kWarps) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kWarps) warp_tot[lane] = t;  // inclusive warp totals
  }
  __syncthreads();
  const int before = (warp > 0) ? warp_tot[warp - 1] : 0;
  *total = warp_tot[kWarps - 1];
  __syncthreads();
  return before + x - v;
}

// Stable LSD radix sort of a window of n <= kSortMax keys, descending (the sort runs
// ascending on ~key), carrying 16-bit positions; writes the first k positions to out.
// Element order inside a pass: warp w owns indices [w * 32E, (w + 1) * 32E), step s
// of lane l holds index w * 32E + 32 s + l, so ranks computed warp by warp and step
// by step preserve the input order of equal digits.
template <int P>
__device__ __forceinline__ void radix_topk(const float* __restrict__ src, int n, int k,
                                          int32_t* __restrict__ out, uint8_t* smem) {
  constexpr int kSortPerThread = P;
  constexpr int kSortMax = sort_max<P>();
  uint32_t* const key_buf = reinterpret_cast<uint32_t*>(smem);              // [2][kSortMax]
  uint16_t* const pos_buf = reinterpret_cast<uint16_t*>(smem + 8 * kSortMax);  // [2][kSortMax]
  uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + 12 * kSortMax);  // [kWarps][256]
  __shared__ uint32_t digit_base[256];
  __shared__ int warp_tot[kWarps];
  __shared__ uint32_t s_or[2], s_and[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = (n + kTopkThreads - 1) / kTopkThreads;  // steps per warp (<= P)
  const int wbase = warp * 32 * E;
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t* wcnt = cnt + warp * 256;
  // Passes that cannot change the order are skipped. Digit p < 3 of a key is a
  // function of the sign alone when digit p of the raw float bits (-0 as +0) is the
  // same across the window; the sign sits in digit 3, so keys that agree on the passes
  // that run agree on such digits too, and the stable sort is unchanged without them.
  // Digit 3 is skipped only if it is itself constant (then the pass is the identity).
  if (tid < 2) {
    s_or[tid] = 0u;
    s_and[tid] = 0xFFFFFFFFu;
  }
  uint32_t key[kSortPerThread];
  uint32_t k_or = 0u, k_and = 0xFFFFFFFFu, r_or = 0u, r_and = 0xFFFFFFFFu;
#pragma unroll
  for (int st = 0; st < kSortPerThread; ++st) {
    const int idx = wbase + 32 * st + lane;
    key[st] = 0u;
    if (st < E && idx < n) {
      uint32_t u = __float_as_uint(__ldg(src + idx));
      if ((u & 0x7FFFFFFFu) == 0) u = 0;
      key[st] = ~((u & 0x80000000u) ? ~u : (u | 0x80000000u));
      k_or |= key[st];
      k_and &= key[st];
      r_or |= u;
      r_and &= u;
    }
  }
  k_or = __reduce_or_sync(0xFFFFFFFFu, k_or);
  k_and = __reduce_and_sync(0xFFFFFFFFu, k_and);
  r_or = __reduce_or_sync(0xFFFFFFFFu, r_or);
  r_and = __reduce_and_sync(0xFFFFFFFFu, r_and);
  __syncthreads();
  if (lane == 0) {
    atomicOr(&s_or[0], k_or);
    atomicAnd(&s_and[0], k_and);
    atomicOr(&s_or[1], r_or);
    atomicAnd(&s_and[1], r_and);
  }
  __syncthreads();
  const uint32_t key_var = s_or[0] ^ s_and[0], raw_var = s_or[1] ^ s_and[1];
  int in = 0;             // buffer holding the current order
  bool from_regs = true;  // no pass has run yet: keys in registers, positions = indices
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 8 * pass;
    if (((key_var >> shift) & 0xFFu) == 0u ||
        (pass < 3 && ((raw_var >> shift) & 0xFFu) == 0u))
      continue;
    for (int d = lane; d < 256; d += 32) wcnt[d] = 0u;
    __syncwarp();
    // Per element: its key, and (position << 16 | rank within its digit and warp); the
    // digit is recomputed from the key. Both fit 16 bits (n <= 4096).
    uint32_t pr[kSortPerThread];
#pragma unroll
    for (int st = 0; st < kSortPerThread; ++st) {
      if (st < E) {
        const int idx = wbase + 32 * st + lane;
        const bool present = idx < n;
        uint32_t pos = 0;
        if (present) {
          if (from_regs) {
            pos = static_cast<uint32_t>(idx);
          } else {
            key[st] = key_buf[in * kSortMax + idx];
            pos = pos_buf[in * kSortMax + idx];
          }
        }
        const uint32_t dig = (key[st] >> shift) & 0xFFu;
        const uint32_t act = __ballot_sync(0xFFFFFFFFu, present);
        pr[st] = 0xFFFFFFFFu;  // absent
        if (present) {
          const uint32_t peers = __match_any_sync(act, dig);
          const uint32_t c0 = wcnt[dig];
          pr[st] = (pos << 16) | (c0 + __popc(peers & lt_mask));
          __syncwarp(act);
          if ((__ffs(peers) - 1) == lane) wcnt[dig] = c0 + __popc(peers);
        }
        __syncwarp();
      }
    }
    __syncthreads();
    // Per digit: exclusive prefix over warps (in place) and the digit's total.
    uint32_t total = 0;
    if (tid < 256) {
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t c = cnt[w * 256 + tid];
        cnt[w * 256 + tid] = total;
        total += c;
      }
    }
    int all;
    const int before = block_excl_scan(tid < 256 ? (int)total : 0, warp_tot, &all);
    if (tid < 256) digit_base[tid] = (uint32_t)before;
    __syncthreads();
#pragma unroll
    for (int st = 0; st < kSortPerThread; ++st) {
      if (st < E && pr[st] != 0xFFFFFFFFu) {
        const uint32_t dig = (key[st] >> shift) & 0xFFu;
        const uint32_t dst = digit_base[dig] + wcnt[dig] + (pr[st] & 0xFFFFu);
        key_buf[(in ^ 1) * kSortMax + dst] = key[st];
        pos_buf[(in ^ 1) * kSortMax + dst] = static_cast<uint16_t>(pr[st] >> 16);
      }
    }
    __syncthreads();
    in ^= 1;
    from_regs = false;
  }
  // No pass ran: every key is equal and the order is the positions'.
  for (int j = tid; j < k; j += kTopkThreads)
    out[j] = (j < n) ? (from_regs ? j : (int32_t)pos_buf[in * kSortMax + j]) : -1;
}

// Bucket-rank path for windows of up to kSortMax values.
//
// Every value gets the sort key skey = ~ordered_key (ascending skey = descending value,
// -0 folded onto +0). The keys of each sign half (skey < 2^31: values >= +0; skey >= 2^31:
// negative values) are mapped linearly onto kHalfBuckets buckets between the half's
// smallest and largest key, so bucket order is key order, and a counting pass places
// every bucket at its final offset. The counting pass's atomic also hands each element a
// slot inside its bucket (in no particular order). Inside a bucket the elements are
// ranked by the unique composite (key offset inside the bucket << 12 | position), which
// orders exactly as (value descending, position ascending); a bucket spans at most 2^19
// key codes (a half's span is below 2^31, divided into 2^12 buckets) and positions need
// 12 bits, so the composite fits 31 bits. The rank of an element is the number of
// smaller composites in its bucket, found by comparing against every member: cheap
// while buckets hold a handful of values, which is the case unless the window's values
// pile up on a few keys. Returns false, having written nothing, when some bucket holds
// more than kMaxBucket values; the caller then takes the radix path, which gives the
// same result. Buckets that start at or beyond k are never ranked: none of their
// values is selected.
constexpr int kHalfBits = 11;
constexpr int kHalfBuckets = 1 << kHalfBits;
constexpr int kBuckets = 2 * kHalfBuckets;
constexpr uint32_t kMaxBucket = 128;
constexpr int kThreadBuckets = kBuckets / kTopkThreads;  // buckets per thread in the scan
static_assert(kThreadBuckets * kTopkThreads == kBuckets && kThreadBuckets % 4 == 0,
              "the scan gives every thread whole uint4s of counters");
// Shared memory: one word per bucket (its count, then its start | end << 16), and per
// selectable slot the composite with its bucket's word.
template <int E>
constexpr size_t bucket_smem() {
  return 4 * kBuckets + 8 * sort_max<E>();
}

// value(st, i) gives element st of this thread (window position i = st * kTopkThreads +
// tid).
template <int E, class Value>
__device__ __forceinline__ bool bucket_topk(Value value, int n, int k, int32_t* __restrict__ out,
                                            uint8_t* smem) {
  constexpr int kSortPerThread = E;
  static_assert(sort_max<E>() <= 4096, "positions must fit the composite's 12 bits");
  uint32_t* const se = reinterpret_cast<uint32_t*>(smem);              // [kBuckets]
  uint2* const slots = reinterpret_cast<uint2*>(smem + 4 * kBuckets);  // [kSortMax]
  // Per warp: min / max skey of the non-negative half, then of the negative half.
  __shared__ uint4 s_wrng[kWarps];
  __shared__ uint32_t s_maxc, s_ranked;
  __shared__ uint32_t s_wsum[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_maxc = 0u;
    s_ranked = static_cast<uint32_t>(n);
  }
#pragma unroll
  for (int q = 0; q < kThreadBuckets / 4; ++q)
    reinterpret_cast<uint4*>(se)[q * kTopkThreads + tid] = make_uint4(0u, 0u, 0u, 0u);
  // Element st of thread tid is window position st * kTopkThreads + tid (coalesced). A
  // warp whose first position of step st lies past the window stops there (warp-uniform).
  uint32_t sk[kSortPerThread];
  uint32_t pmin = 0xFFFFFFFFu, pmax = 0u, nmin = 0xFFFFFFFFu, nmax = 0u;
#pragma unroll
  for (int st = 0; st < kSortPerThread; ++st) {
    if (st * kTopkThreads + warp * 32 >= n) break;
    const int i = st * kTopkThreads + tid;
    sk[st] = 0u;
    if (i < n) {
      uint32_t u = __float_as_uint(value(st, i));
      if ((u & 0x7FFFFFFFu) == 0) u = 0;
      const uint32_t s = (u & 0x80000000u) ? u : ~(u | 0x80000000u);  // ~ordered_key
      sk[st] = s;
      if (s < 0x80000000u) {
        pmin = min(pmin, s);
        pmax = max(pmax, s);
      } else {
        nmin = min(nmin, s);
        nmax = max(nmax, s);
      }
    }
  }
  pmin = __reduce_min_sync(0xFFFFFFFFu, pmin);
  pmax = __reduce_max_sync(0xFFFFFFFFu, pmax);
  nmin = __reduce_min_sync(0xFFFFFFFFu, nmin);
  nmax = __reduce_max_sync(0xFFFFFFFFu, nmax);
  if (lane == 0) s_wrng[warp] = make_uint4(pmin, pmax, nmin, nmax);
  __syncthreads();  // also: the bucket counters are zeroed
  {  // every warp reduces the warps' ranges itself (lane w reads warp w's)
    const uint4 r = lane < kWarps ? s_wrng[lane] : make_uint4(0xFFFFFFFFu, 0u, 0xFFFFFFFFu, 0u);
    pmin = __reduce_min_sync(0xFFFFFFFFu, r.x);
    pmax = __reduce_max_sync(0xFFFFFFFFu, r.y);
    nmin = __reduce_min_sync(0xFFFFFFFFu, r.z);
    nmax = __reduce_max_sync(0xFFFFFFFFu, r.w);
  }
  // Per half: its smallest key and the shift that maps its span onto kHalfBuckets buckets.
  // A half's span is below 2^31, so the shift is at most 20 and the composite (offset
  // inside the bucket << 12 | position) fits 32 bits.
  const uint32_t base0 = pmin, base1 = nmin;
  const uint32_t span0 = pmax - base0, span1 = nmax - base1;  // garbage if empty
  const int sh0 = max(0, (32 - __clz(span0)) - kHalfBits);
  const int sh1 = max(0, (32 - __clz(span1)) - kHalfBits);
  const uint32_t low0 = (1u << sh0) - 1u, low1 = (1u << sh1) - 1u;
  // Per element: bucket << 16 | its slot inside the bucket (the count before it), or ~0.
  uint32_t bs[kSortPerThread];
#pragma unroll
  for (int st = 0; st < kSortPerThread; ++st) {
    if (st * kTopkThreads + warp * 32 >= n) break;
    const int i = st * kTopkThreads + tid;
    bs[st] = 0xFFFFFFFFu;
    if (i < n) {
      const uint32_t s = sk[st];
      const bool neg = s >= 0x80000000u;
      const uint32_t off = s - (neg ? base1 : base0);
      const int sh = neg ? sh1 : sh0;
      const uint32_t b = (neg ? kHalfBuckets : 0) + (off >> sh);
      sk[st] = ((off & (neg ? low1 : low0)) << 12) | static_cast<uint32_t>(i);  // composite
      bs[st] = (b << 16) | atomicAdd(&se[b], 1u);
    }
  }
  __syncthreads();
  // Exclusive prefix over the buckets in ascending order: thread tid owns buckets
  // [kThreadBuckets tid, kThreadBuckets (tid + 1)). Counts and offsets stay below 2^16.
  // Each bucket's word becomes start | end << 16. The thread whose bucket holds output
  // place k - 1 records where that bucket ends: every slot before it is ranked, nothing
  // after it is selected.
  {
    uint4* const mine4 = reinterpret_cast<uint4*>(se) + tid * (kThreadBuckets / 4);
    uint32_t w[kThreadBuckets];
#pragma unroll
    for (int q = 0; q < kThreadBuckets / 4; ++q) {
      const uint4 c = mine4[q];
      w[4 * q] = c.x;
      w[4 * q + 1] = c.y;
      w[4 * q + 2] = c.z;
      w[4 * q + 3] = c.w;
    }
    uint32_t tot = 0u, mx = 0u;
#pragma unroll
    for (int j = 0; j < kThreadBuckets; ++j) {
      tot += w[j];
      mx = max(mx, w[j]);
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    uint32_t x = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_wsum[warp] = x;
    if (lane == 0) atomicMax(&s_maxc, mx);
    __syncthreads();
    uint32_t run = x - tot + __reduce_add_sync(0xFFFFFFFFu, lane < warp ? s_wsum[lane] : 0u);
    const uint32_t kk = static_cast<uint32_t>(k);
    const bool mine = run < kk && kk <= run + tot;  // place k - 1 lies in these buckets
    uint32_t o[kThreadBuckets];
#pragma unroll
    for (int j = 0; j < kThreadBuckets; ++j) {
      const uint32_t e = run + w[j];
      o[j] = run | (e << 16);
      if (mine && run < kk && kk <= e) s_ranked = e;
      run = e;
    }
#pragma unroll
    for (int q = 0; q < kThreadBuckets / 4; ++q)
      mine4[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
  }
  __syncthreads();
  if (s_maxc > kMaxBucket) return false;  // uniform: every thread reads the same word
  const uint32_t ranked = s_ranked;        // slots [0, ranked) hold the selectable buckets
  // Place the composites of buckets that start before k, each with its bucket's word.
#pragma unroll
  for (int st = 0; st < kSortPerThread; ++st) {
    if (st * kTopkThreads + warp * 32 >= n) break;
    const uint32_t v = bs[st];
    if (v != 0xFFFFFFFFu) {
      const uint32_t bw = se[v >> 16];
      const uint32_t s0 = bw & 0xFFFFu;
      if (s0 < static_cast<uint32_t>(k)) slots[s0 + (v & 0xFFFFu)] = make_uint2(sk[st], bw);
    }
  }
  __syncthreads();
  // Rank in bucket order: thread tid takes slots tid, tid + 512, ...; neighbouring lanes
  // hold neighbouring slots, mostly of the same bucket, so their loads of the bucket's
  // members coincide, and their places (the bucket's start plus the number of smaller
  // composites in it) fall in the same few output lines.
  for (uint32_t j = tid; j < ranked; j += kTopkThreads) {
    const uint2 me = slots[j];
    const uint32_t s0 = me.y & 0xFFFFu;
    uint32_t rank = 0;
    const uint2* const end = slots + (me.y >> 16);
#pragma unroll 1  // buckets hold a few values: an unrolled loop costs more than it saves
    for (const uint2* m = slots + s0; m < end; ++m) rank += m->x < me.x ? 1u : 0u;
    const uint32_t dst = s0 + rank;
    if (dst < static_cast<uint32_t>(k)) out[dst] = static_cast<int32_t>(me.x & 0xFFFu);
  }
  for (int j = n + tid; j < k; j += kTopkThreads) out[j] = -1;
  return true;
}

// Four CTAs per SM for E = 6 (<= 32 registers a thread), three for E = 8 (<= 40).
template <int E>
__global__ void __launch_bounds__(kTopkThreads, E <= 6 ? 4 : 3) topk_select_kernel(
    const float* __restrict__ logits, int64_t row_stride, const int32_t* __restrict__ row_starts,
    const int32_t* __restrict__ row_lens, int k, int sort_n, int32_t* __restrict__ idx,
    uint32_t* dev_status) {
  constexpr int kSortPerThread = E;
  constexpr int kSortMax = sort_max<E>();
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t* sel = reinterpret_cast<uint64_t*>(smem);                      // [sort_n]
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + 8 * (size_t)sort_n);  // [row_stride]
  __shared__ int hist[256];
  __shared__ int warp_tot[kWarps];
  __shared__ int s_digit, s_above, s_nsel;

  const int tid = threadIdx.x;
  const int64_t r = blockIdx.x;
  int32_t* out = idx + r * (int64_t)k;
  // Windows usually start at the row's beginning: the row's first values are loaded
  // while its bounds are read, saving a dependent round trip (used only if st == 0).
  float pre[kSortPerThread];
  const int pre_n = static_cast<int>(row_stride < kSortMax ? row_stride : kSortMax);
  const float* row = logits + r * row_stride;
#pragma unroll
  for (int e = 0; e < kSortPerThread; ++e) {
    pre[e] = 0.f;
    if (e * kTopkThreads + (tid & ~31) >= pre_n) continue;  // warp-uniform
    const int i = e * kTopkThreads + tid;
    if (i < pre_n) pre[e] = __ldg(row + i);
  }
  const int64_t st = row_starts[r];
  const int64_t len = row_lens[r];
  if (st < 0 || len < 0 || st + len > row_stride) {
    if (tid == 0 && dev_status != nullptr) atomicOr(dev_status, kDevIndexRange);
    for (int j = tid; j < k; j += kTopkThreads) out[j] = -1;
    return;
  }
  const int n = static_cast<int>(len);
  const float* src = logits + r * row_stride + st;
  if (n <= kSortMax) {
    const bool have_pre = st == 0;
    auto value = [&](int e, int i) { return have_pre ? pre[e] : __ldg(src + i); };
    if (!bucket_topk<E>(value, n, k, out, smem)) {
      __syncthreads();  // the radix path reuses the shared memory
      radix_topk<E>(src, n, k, out, smem);
    }
    return;
  }
  for (int j = tid; j < n; j += kTopkThreads) keys[j] = ordered_key(__ldg(src + j));
  __syncthreads();

  const int take = n < k ? n : k;
  if (n > k) {
    // ---- radix select: find the key of rank k (1-based, descending) ----
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int b = tid; b < 256; b += kTopkThreads) hist[b] = 0;
      __syncthreads();
      for (int j0 = 0; j0 < n; j0 += kTopkThreads) {
        const int j = j0 + tid;
        bool active = false;
        uint32_t dgt = 0;
        if (j < n) {
          const uint32_t key = keys[j];
          active = (key & mask) == prefix;
          dgt = (key >> shift) & 0xFFu;
        }
        const uint32_t act = __ballot_sync(0xFFFFFFFFu, active);
        if (active) {
          const uint32_t peers = __match_any_sync(act, dgt);
          if ((__ffs(peers) - 1) == (tid & 31)) atomicAdd(&hist[dgt], __popc(peers));
        }
      }
      __syncthreads();
      if (tid < 32) {
        // lane l owns bins 255-8l .. 248-8l (descending)
        int c[8], s = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          c[t] = hist[255 - 8 * tid - t];
          s += c[t];
        }
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (tid >= o) incl += y;
        }
        int above = incl - s;  // count in bins strictly above this lane's first bin
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (above < remaining && remaining <= above + c[t]) {
            s_digit = 255 - 8 * tid - t;
            s_above = above;
          }
          above += c[t];
        }
      }
      __syncthreads();
      remaining -= s_above;
      prefix |= static_cast<uint32_t>(s_digit) << shift;
      mask |= 0xFFu << shift;
      __syncthreads();
    }
    const uint32_t T = prefix;
    const int need_ties = remaining;  // 1 <= need_ties; k - need_ties keys are > T
    // ---- compaction: keys > T in any slot order, ties by ascending position ----
    if (tid == 0) s_nsel = 0;
    __syncthreads();
    int ties_before = 0;
    for (int j0 = 0; j0 < n; j0 += kTopkThreads) {
      const int j = j0 + tid;
      const uint32_t key = (j < n) ? keys[j] : 0u;
      const bool gt = (j < n) && key > T;
      const bool eq = (j < n) && key == T;
      int tot;
      const int rank = ties_before + block_excl_scan(eq ? 1 : 0, warp_tot, &tot);
      const bool pick = gt || (eq && rank < need_ties);
      if (pick) {
        const int slot = atomicAdd(&s_nsel, 1);
        sel[slot] = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~j);
      }
      ties_before += tot;
    }
  } else {
    for (int j = tid; j < n; j += kTopkThreads)
      sel[j] = (static_cast<uint64_t>(keys[j]) << 32) | static_cast<uint32_t>(~j);
  }
  for (int j = take + tid; j < sort_n; j += kTopkThreads) sel[j] = 0ull;  // sorts last
  __syncthreads();

  // ---- bitonic sort, descending ----
  for (int size = 2; size <= sort_n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < (sort_n >> 1); i += kTopkThreads) {
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
  for (int j = tid; j < k; j += kTopkThreads)
    out[j] = (j < take) ? static_cast<int32_t>(~static_cast<uint32_t>(sel[j] & 0xFFFFFFFFull)) : -1;
}

}  // namespace

// Rows of at most sort_max<6>() values take the E = 6 kernel, all others E = 8.
static bool short_rows(int64_t row_stride) { return row_stride <= sort_max<6>(); }

template <int E>
static size_t smem_bytes(int64_t row_stride, int k) {
  const int64_t cap = row_stride < k ? row_stride : k;
  int sort_n = 2;
  while (sort_n < cap) sort_n <<= 1;
  size_t smem = 8 * (size_t)sort_n + 4 * (size_t)row_stride;  // the select path
  if (row_stride <= sort_max<E>()) smem = 0;                  // never taken
  if (smem < radix_smem<E>()) smem = radix_smem<E>();
  if (smem < bucket_smem<E>()) smem = bucket_smem<E>();
  return smem;
}

size_t topk_smem_bytes(int64_t row_stride, int k) {
  return short_rows(row_stride) ? smem_bytes<6>(row_stride, k) : smem_bytes<8>(row_stride, k);
}

template <int E>
static cudaError_t launch(const float* logits, int64_t row_stride, int32_t rows,
                          const int32_t* row_starts, const int32_t* row_lens, int32_t k,
                          int32_t* idx, uint32_t* dev_status, cudaStream_t stream) {
  const int64_t cap = row_stride < k ? row_stride : k;
  int sort_n = 2;
  while (sort_n < cap) sort_n <<= 1;
  const size_t smem = smem_bytes<E>(row_stride, k);
  // The shared-memory limit is a per-device attribute of the kernel; raise it only when
  // a call needs more than a previous call on this device set (races only repeat it).
  static std::atomic<int> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || configured[dev].load(std::memory_order_relaxed) < (int)smem) {
    e = cudaFuncSetAttribute(topk_select_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store((int)smem, std::memory_order_relaxed);
  }
  topk_select_kernel<E><<<rows, kTopkThreads, smem, stream>>>(logits, row_stride, row_starts,
                                                               row_lens, k, sort_n, idx,
                                                               dev_status);
  e = cudaGetLastError();
  if (e == cudaErrorInvalidValue) {
    // A new context (after a device reset, say) starts from the default limit: set it
    // and launch once more (the refused launch ran nothing).
    e = cudaFuncSetAttribute(topk_select_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    topk_select_kernel<E><<<rows, kTopkThreads, smem, stream>>>(logits, row_stride, row_starts,
                                                                 row_lens, k, sort_n, idx,
                                                                 dev_status);
    e = cudaGetLastError();
  }
  return e;
}

cudaError_t launch_topk_select(const float* logits, int64_t row_stride, int32_t rows,
                               const int32_t* row_starts, const int32_t* row_lens, int32_t k,
                               int32_t* idx, uint32_t* dev_status, cudaStream_t stream) {
  return short_rows(row_stride)
             ? launch<6>(logits, row_stride, rows, row_starts, row_lens, k, idx, dev_status,
                         stream)
             : launch<8>(logits, row_stride, rows, row_starts, row_lens, k, idx, dev_status,
                         stream);
}

}  // namespace tts
