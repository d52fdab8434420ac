// Sparse attention through a paged KV cache, invariant to the order of the index list.
//
// What it computes ("推理引擎的蝴蝶效应 -- 从V32 模型的输出不一致说起", sections
// 实验方法和结果 and 进一步探索): for query n and head h, softmax attention over the
// KV rows selected by idx[n, :], each fetched through the page table
// (row = kv_cache[page_table[i / page_size], i % page_size]); K = the row's 576
// values, V = its first 512. The write-up shows that feeding the same index set
// in a different order changes bf16 outputs, because the online-softmax merge
// (its equations 1-2) rounds differently per block order, and that sorting the
// indices restores identical results. This kernel therefore sorts each query's
// list ascending first; tiles are then visited in that canonical order with no
// atomics, so any permutation of idx[n, :] gives bitwise identical out / lse.
//
// Layout of the work (one CTA = one query n and one half r of the 512 V columns):
//   * the 128 heads form the MMA M dimension; the KV tile is 64 gathered rows;
//   * TMEM (512 columns): Q_lo [0,128) = the 4 Q slabs (64 columns each) whose
//     columns are also this CTA's V columns, held as the A operand of TS MMAs;
//     S double buffer [128,192) [192,256); O half [256,512);
//   * shared memory: the other 5 Q slabs (80 KB), and two stages of the gathered
//     tile split into its 5 K-only slabs (40 KB) and 4 V slabs (32 KB); Q_lo passes
//     through the (still idle) V stages on its way into TMEM;
//   * warps 0-3 gather the K-only slabs (16-byte cp.async into the 128-byte-swizzled
//     layout the MMA reads), warps 4-7 the V slabs (TMA tile::gather4, four rows per
//     copy, same layout), warp 8 issues MMAs, warps 12-15 run the softmax (one head
//     per thread); all 16 warps write the output (TMA stores of staged boxes).
// Both CTAs of a query compute all of S (each over the 9 slabs in its own fixed
// order, so their roundings may differ) and accumulate O for their 256 V columns:
// the S work is done twice so that no partial scores move between SMs. The (query,
// half) units of the last, partial wave of CTAs can run as 2-16 parts over
// consecutive tiles of the sorted list, merged in part order (by the last part to
// finish, or for more than four parts by a merge launch).
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace tts {
namespace {

constexpr int kThreads = 512;
constexpr int kHeads = 128;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kTileN = 64;                  // gathered KV rows per tile
constexpr int kSlabBytes = kTileN * 128;    // one 64-column slab of a tile: 8 KB
constexpr int kQSlabBytes = kHeads * 128;   // one 64-column slab of Q: 16 KB
constexpr int kKOnly = 5, kVSlabs = 4;
constexpr int kQhiBytes = kKOnly * kQSlabBytes;      // 80 KB
constexpr int kKStage = kKOnly * kSlabBytes;         // 40 KB
constexpr int kVStage = kVSlabs * kSlabBytes;        // 32 KB
constexpr int kSmemBytes = kQhiBytes + 2 * kKStage + 2 * kVStage + 1024;
constexpr int kMaxTopk = 2048;
constexpr int kMaxTiles = kMaxTopk / kTileN;         // 32
constexpr int kCountCap = 16384;  // kv_len up to this uses a counting sort
constexpr int kScratchInts = 2 * kKStage / 4;  // sort scratch: the K stages (80 KB)
constexpr int kMaxParts = 16;
// Units split into at most this many parts are merged by their last part to finish;
// wider splits (small batches) leave the merge to a launch of its own, spread over many
// CTAs, since one CTA reading every part's partial O would take longer than the split
// saves.
constexpr int kKernelMergeParts = 4;
// One partial result: O [128 heads][256 columns], then m [128] and l [128].
constexpr int kSlotFloats = kHeads * 256 + 2 * kHeads;
static_assert(kMaxTopk <= 4 * kThreads, "one round of four index loads per thread");
static_assert(kCountCap + kMaxTopk <= kScratchInts, "counts and the sorted list fit");

struct SparseParams {
  const uint16_t* q;  // bf16 bits [nq, 128, 576]
  const uint16_t* kv;  // bf16 bits [pages * page_size, 576]
  const int32_t* page_table;  // row n of the tables starts at page_table + n * pt_stride
  const int32_t* kv_lens;     // per query (decode), or nullptr: kv_len for every query
  int pt_stride;              // 0: one table shared by all queries
  const int32_t* idx;
  float* out;
  float* lse;
  uint32_t* dev_status;
  int nq, num_pages, page_size, num_logical_pages, kv_len, topk, sort_n;
  int page_shift;  // log2(page_size) when it is a power of two, else -1
  float scale, scale_log2;
  // Split of the last, partial wave: CTAs [0, n_main) are whole units (query, V half);
  // each later unit runs as `parts` CTAs over consecutive tile ranges, whose partial
  // results (unnormalised O, m, l) go to `partial` and are merged by the last finisher.
  int n_main, parts;
  float* partial;  // [tail units][parts][kSlotFloats]
  uint32_t* done;  // [tail units], zero at launch
  // Canonical lists made by the sort launch (nullptr: the attention kernel sorts):
  // query n's physical rows at sorted_rows + n * kMaxTopk, their count sorted_cnt[n].
  int32_t* sorted_rows;
  int32_t* sorted_cnt;
};

// One TMA copy of four whole rows (tile::gather4): 64 columns of each of rows r0..r3 of a
// 2-D tensor map whose box is {64, 1}, landing as four consecutive 128-byte rows of the
// map's swizzled layout at dst.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int x, int r0, int r1, int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}

// The merge of a split unit's parts (unnormalised O, m, l of each part, in the slots of
// `slot0`), in part order:
//   out = sum_p w_p O_p / sum_p w_p l_p,  w_p = 2^((m_p - M) * scale * log2 e),
//   M = max_p m_p  (the online-softmax merge, with a fixed order).
// merge_weights: head h's weights w_p / L into s_w[p * ld + hw] (and its lse, written by
// the unit of the first V half).
template <int P>
__device__ __forceinline__ void merge_weights(const SparseParams& p, const float* slot0,
                                              int nparts, int h, int n, int r, float* s_w,
                                              int ld, int hw = -1) {
  if (hw < 0) hw = h;
  float mp[P], w[P];
  float M = -INFINITY;
#pragma unroll
  for (int pp = 0; pp < P; ++pp)
    if (pp < nparts) {
      mp[pp] = __ldcg(slot0 + pp * kSlotFloats + kHeads * 256 + h);
      M = fmaxf(M, mp[pp]);
    }
  float L = 0.f;
#pragma unroll
  for (int pp = 0; pp < P; ++pp)
    if (pp < nparts) {
      w[pp] = (mp[pp] == -INFINITY) ? 0.f : ex2_approx((mp[pp] - M) * p.scale_log2);
      L += __ldcg(slot0 + pp * kSlotFloats + kHeads * 256 + kHeads + h) * w[pp];
    }
  const float inv_L = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
  for (int pp = 0; pp < P; ++pp)
    if (pp < nparts) s_w[pp * ld + hw] = w[pp] * inv_L;
  if (r == 0 && p.lse != nullptr)
    p.lse[(int64_t)n * kHeads + h] =
        (L > 0.f) ? M * p.scale + log2f(L) * 0.69314718055994531f : -INFINITY;
}
// merge_row_chunk: columns 4 c4 .. 4 c4 + 3 of head h's 256 (weights at row hw of s_w).
template <int P>
__device__ __forceinline__ void merge_row_chunk(const float* slot0, int nparts, const float* s_w,
                                                int ld, int h, int hw, int c4, float* obase) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int pp = 0; pp < P; ++pp)
    if (pp < nparts) {
      const float4 v =
          __ldcg(reinterpret_cast<const float4*>(slot0 + pp * kSlotFloats + h * 256) + c4);
      const float wq = s_w[pp * ld + hw];
      acc.x = fmaf(v.x, wq, acc.x);
      acc.y = fmaf(v.y, wq, acc.y);
      acc.z = fmaf(v.z, wq, acc.z);
      acc.w = fmaf(v.w, wq, acc.w);
    }
  *reinterpret_cast<float4*>(obase + (int64_t)h * kDv + 4 * c4) = acc;
}

__device__ __forceinline__ int kslab_of(int r, int i) {  // i-th K-only slab (global id)
  return r == 0 ? 4 + i : (i < 4 ? i : 8);
}

// Canonical order of query n's index list: entries validated (-1 and out-of-range
// entries dropped, the latter reported), sorted ascending (duplicates kept) and resolved
// through the page table to physical KV rows. Needs all kThreads threads; scratch holds
// counts [kv_len] (counting sort, kv_len <= kCountCap), a copy of the page table when it
// fits, then the sorted list, which *rows points at on return. *s_cnt must be zero on
// entry (shared); returns the number of valid entries.
__device__ __forceinline__ int canonical_rows(const SparseParams& p, int n, int32_t* scratch,
                                              int scratch_ints, int* s_cnt, int* s_wsum,
                                              const int32_t** rows) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t* idx_row = p.idx + (int64_t)n * p.topk;
  const int32_t* const ptab = p.page_table + (int64_t)n * p.pt_stride;
  int kv_len = p.kv_len;
  if (p.kv_lens != nullptr) {
    kv_len = p.kv_lens[n];
    if (kv_len < 0) {  // every entry of this query is then out of range
      if (tid == 0 && p.dev_status != nullptr) atomicOr(p.dev_status, kDevIndexRange);
      kv_len = 0;
    }
  }
  const bool by_count = kv_len <= kCountCap;
  const int n_scan = by_count ? p.topk : p.sort_n;
  const int n_counts = by_count ? kv_len : 0;
  const int nlp = p.num_logical_pages;
  const bool pt_cached = n_counts + nlp + n_scan <= scratch_ints;
  int32_t* counts = scratch;
  int32_t* pt = counts + n_counts;
  int32_t* sorted = pt + (pt_cached ? nlp : 0);
  // The index loads go out first; their round trip overlaps the zeroing and the
  // page-table copy.
  int32_t iv[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int j = u * kThreads + tid;
    iv[u] = (j < p.topk) ? idx_row[j] : -1;
  }
  for (int v = tid; v < n_counts; v += kThreads) counts[v] = 0;
  if (pt_cached)
    for (int g = tid; g < nlp; g += kThreads) pt[g] = ptab[g];
  __syncthreads();
  auto page_of = [&](int g) -> int32_t { return pt_cached ? pt[g] : ptab[g]; };
  // logical position -> (logical page, offset); shifts for power-of-two page sizes
  auto lpage = [&](int v) { return p.page_shift >= 0 ? v >> p.page_shift : v / p.page_size; };
  auto row_of = [&](int v) -> int32_t {
    const int g = lpage(v);
    return page_of(g) * p.page_size + (v - g * p.page_size);
  };
  int my_valid = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int j = u * kThreads + tid;
    if (j >= n_scan) continue;
    const int32_t i = iv[u];
    int key = 0x7FFFFFFF;
    if (i != -1 && j < p.topk) {
      const bool in = i >= 0 && i < kv_len && lpage(i) < nlp;
      const int32_t pg = in ? page_of(lpage(i)) : -1;
      if (pg >= 0 && pg < p.num_pages) {
        key = i;
        ++my_valid;
      } else if (p.dev_status != nullptr) {
        atomicOr(p.dev_status, kDevIndexRange);
      }
    }
    if (by_count) {
      if (key != 0x7FFFFFFF) atomicAdd(&counts[key], 1);  // integer: order-independent
    } else {
      sorted[j] = key;
    }
  }
  if (my_valid) atomicAdd(s_cnt, my_valid);
  __syncthreads();
  if (by_count) {
    // Counting sort: thread t owns a contiguous range of positions; an exclusive scan
    // of the per-range totals gives where each range's entries start.
    const int per = (kv_len + kThreads - 1) / kThreads;
    const int v0 = tid * per, v1 = min(kv_len, v0 + per);
    int tot = 0;
    for (int v = v0; v < v1; ++v) tot += counts[v];
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += s_wsum[w];
    int pos = before + incl - tot;
    // The sorted list holds physical KV rows (page-table resolved) in logical order.
    for (int v = v0; v < v1; ++v) {
      const int c = counts[v];
      if (c == 0) continue;
      const int32_t row = row_of(v);
      for (int k = 0; k < c; ++k) sorted[pos++] = row;
    }
  } else {
    for (int size = 2; size <= p.sort_n; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < (p.sort_n >> 1); i += kThreads) {
          const int lo = 2 * i - (i & (stride - 1));
          const int hi = lo + stride;
          const bool asc = (lo & size) == 0;
          const int a = sorted[lo], b = sorted[hi];
          if ((a > b) == asc) {
            sorted[lo] = b;
            sorted[hi] = a;
          }
        }
        __syncthreads();
      }
    }
  }
  __syncthreads();
  const int cnt = *s_cnt;
  if (!by_count) {  // the bitonic path sorted logical positions: resolve them now
    for (int pos = tid; pos < cnt; pos += kThreads) {
      const int32_t v = sorted[pos];
      sorted[pos] = row_of(v);
    }
    __syncthreads();
  }
  *rows = sorted;
  return cnt;
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ CUtensorMap kvmap,
                       const __grid_constant__ CUtensorMap outmap, const SparseParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_qhi, bar_qlo_smem, bar_qlo, bar_kfull[2], bar_vfull[2], bar_kempty[2],
      bar_vempty[2], bar_s[2], bar_p[2], bar_o, bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_cnt;
  __shared__ int s_wsum[kThreads / 32];
  __shared__ float s_inv_l[kHeads];
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int u = blockIdx.x, part = 0, nparts = 1;
  if (u >= p.n_main) {
    const int k = u - p.n_main;
    u = p.n_main + k / p.parts;
    part = k % p.parts;
    nparts = p.parts;
  }
  const int n = u >> 1, r = u & 1;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQhi = sb;
  const uint32_t sK0 = sb + kQhiBytes;
  const uint32_t sV0 = sK0 + 2 * kKStage;

  if (tid == 0) {
    s_abort = 0;
    s_cnt = 0;
    mbar_init(smem_u32(&bar_qhi), 1);
    mbar_init(smem_u32(&bar_qlo_smem), 1);
    mbar_init(smem_u32(&bar_qlo), 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_kfull[i]), 128);
      mbar_init(smem_u32(&bar_vfull[i]), 4);  // one expect-tx arrival per V warp
      mbar_init(smem_u32(&bar_kempty[i]), 1);
      mbar_init(smem_u32(&bar_vempty[i]), 1);
      mbar_init(smem_u32(&bar_s[i]), 1);
      mbar_init(smem_u32(&bar_p[i]), 128);
    }
    mbar_init(smem_u32(&bar_o), 1);
    mbar_init(smem_u32(&bar_drain), 1);
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(&s_tmem), 512);
    tmem_relinquish();
  }
  __syncthreads();
  // All of Q by TMA, issued before the sort: the 5 slabs that stay in shared memory,
  // and the 4 Q_lo slabs into the V stages (idle until Q_lo has moved on into TMEM).
  if (tid == 0) {
    prefetch_tmap(&qmap);
    prefetch_tmap(&kvmap);
    mbar_arrive_expect_tx(smem_u32(&bar_qhi), kQhiBytes);
    for (int i = 0; i < kKOnly; ++i)
      tma_load_3d(sQhi + i * kQSlabBytes, &qmap, smem_u32(&bar_qhi), 64 * kslab_of(r, i), 0, n);
    mbar_arrive_expect_tx(smem_u32(&bar_qlo_smem), kVSlabs * kQSlabBytes);
    for (int i = 0; i < kVSlabs; ++i)
      tma_load_3d(sV0 + i * kQSlabBytes, &qmap, smem_u32(&bar_qlo_smem), 64 * (4 * r + i), 0, n);
  }

  // ---- canonical order: the query's index list validated, sorted ascending and
  // resolved to physical rows -- by the sort launch (in the workspace) or here (in the
  // still unused K stages) ----
  const int32_t* sorted;
  int cnt;
  if (p.sorted_rows != nullptr) {
    sorted = p.sorted_rows + (int64_t)n * kMaxTopk;
    cnt = p.sorted_cnt[n];
  } else {
    cnt = canonical_rows(p, n, reinterpret_cast<int32_t*>(smem + kQhiBytes), kScratchInts, &s_cnt,
                         s_wsum, &sorted);
  }
  const int n_tiles = (cnt + kTileN - 1) / kTileN;
  // This CTA's tiles of the sorted list (all of them unless the unit is split).
  const int t_begin = part * n_tiles / nparts;
  const int nt = (part + 1) * n_tiles / nparts - t_begin;
  // Producer warp w keeps, in registers, the physical rows of entries 16 * (w & 3) ..
  // +15 of every tile: lane l holds entry l & 15 of the even tiles (l < 16) or of the
  // odd tiles (l >= 16), oldest first, and drops the front one once that tile is issued.
  // Entries past the list (last tile only) take the last listed row, so every copy
  // stays in range; the softmax gives them zero weight.
  const int32_t fill_row = cnt > 0 ? sorted[cnt - 1] : 0;
  int32_t rows_q[kMaxTiles / 2];
  if (warp < 8) {
    const int e = 16 * (warp & 3) + (lane & 15);
#pragma unroll
    for (int k = 0; k < kMaxTiles / 2; ++k) {
      const int pos = (t_begin + 2 * k + (lane >> 4)) * kTileN + e;
      rows_q[k] = pos < cnt ? sorted[pos] : fill_row;
    }
  }
  tc_fence_before();
  __syncthreads();  // sort scratch is free from here on
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;

  if (warp < 8) {
    // ------------------------------------------------------------ Q_lo -> TMEM, gather
    bool go = true;
    if (warp < 4) {
      // Q_lo: from the V stages (landed by TMA, 128-byte-swizzled rows) into TMEM.
      const int h = tid;  // warp w covers TMEM lanes 32w..32w+31
      const bool okq = __all_sync(
          0xFFFFFFFFu, mbar_wait(smem_u32(&bar_qlo_smem), 0, abort_flag, p.dev_status));
      if (okq) {
        const uint8_t* qrow = smem + kQhiBytes + 2 * kKStage + h * 128;
#pragma unroll 1
        for (int i = 0; i < kVSlabs; ++i) {
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 x =
                *reinterpret_cast<const uint4*>(qrow + i * kQSlabBytes + ((c ^ (h & 7)) << 4));
            v[4 * c] = x.x;
            v[4 * c + 1] = x.y;
            v[4 * c + 2] = x.z;
            v[4 * c + 3] = x.w;
          }
          tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + i * 32, v);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_qlo));  // also: the V stages are free for gathering
    } else {
      go = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bar_qlo), 0, abort_flag, p.dev_status));
    }
    const bool kside = warp < 4;
    // Producer warp w of a role copies entries 16*(w&3) .. +15 of the tile. K side: lane
    // l copies the 16-byte chunk (l & 7) of entry 16*(w&3) + 4*rr + (l >> 3), rr = 0..3,
    // so one warp instruction moves four whole 128-byte row segments. V side: lanes 0..3
    // each issue one four-row TMA gather per slab. Row offsets come from the lane that
    // owns the entry (rows_q), by shuffle.
    const int e_base = 16 * (warp & 3);
    const int chunk = lane & 7;
    for (int j = 0; go && j < nt; ++j) {
      const int st = j & 1;
      if (j >= 2) {  // the decision is warp-wide: the shuffles below need every lane
        const uint32_t eb = smem_u32(kside ? &bar_kempty[st] : &bar_vempty[st]);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(eb, ((j >> 1) - 1) & 1, abort_flag, p.dev_status)))
          break;
      }
      const int32_t mine = rows_q[0];
      const int src = (j & 1) * 16;  // the lanes that hold this tile's rows
      if ((lane >> 4) == (j & 1)) {
#pragma unroll
        for (int k = 0; k + 1 < kMaxTiles / 2; ++k) rows_q[k] = rows_q[k + 1];
      }
      const uint32_t stage = kside ? sK0 + st * kKStage : sV0 + st * kVStage;
      if (!kside) {
        const uint32_t fb = smem_u32(&bar_vfull[st]);
        const int gi = lane & 3;
        const int32_t r0 = __shfl_sync(0xFFFFFFFFu, mine, src + 4 * gi);
        const int32_t r1 = __shfl_sync(0xFFFFFFFFu, mine, src + 4 * gi + 1);
        const int32_t r2 = __shfl_sync(0xFFFFFFFFu, mine, src + 4 * gi + 2);
        const int32_t r3 = __shfl_sync(0xFFFFFFFFu, mine, src + 4 * gi + 3);
        if (lane == 0) mbar_arrive_expect_tx(fb, 16 * kVSlabs * 128);
        __syncwarp();
        if (lane < 4) {
          const uint32_t dst = stage + (e_base + 4 * gi) * 128;
#pragma unroll
          for (int i = 0; i < kVSlabs; ++i)
            tma_gather4(dst + i * kSlabBytes, &kvmap, fb, 64 * (4 * r + i), r0, r1, r2, r3);
        }
        continue;
      }
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int el = rr * 4 + (lane >> 3);  // entry within this warp's 16
        const int32_t row = __shfl_sync(0xFFFFFFFFu, mine, src + el);
        const int e = e_base + el;
        const uint16_t* src_row = p.kv + (int64_t)row * kDqk + chunk * 8;
        const uint32_t dst = stage + e * 128 + ((chunk ^ (e & 7)) << 4);
#pragma unroll
        for (int i = 0; i < kKOnly; ++i)
          cp_async_16(dst + i * kSlabBytes, src_row + kslab_of(r, i) * 64, 16);
      }
      // Arrive when this thread's copies have landed, without waiting for them here: the
      // next tile's copies go out while these are in flight (the MMA warp orders the
      // landed data for the tensor core with a proxy fence after its wait).
      cp_async_arrive_noinc(smem_u32(&bar_kfull[st]));
    }
    cp_async_wait_all();  // nothing may still be landing when the CTA exits
    if (!kside && lane == 0)  // nor any copy-engine gather
      for (int j = (nt > 2 ? nt - 2 : 0); j < nt; ++j)
        mbar_wait(smem_u32(&bar_vfull[j & 1]), (j >> 1) & 1, nullptr, p.dev_status);
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop converged; the elected lane issues.
    if (nt > 0) {
      const uint32_t e = elect_one();
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kTileN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 256, 0, 1);
      const uint32_t S_t[2] = {tmem + 128, tmem + 192};
      const uint32_t O_t = tmem + 256;
      const uint64_t dq = smem_desc(sQhi, 16, 1024, kSw128);
      const uint64_t dk[2] = {smem_desc(sK0, 16, 1024, kSw128),
                              smem_desc(sK0 + kKStage, 16, 1024, kSw128)};
      const uint64_t dvk[2] = {smem_desc(sV0, 16, 1024, kSw128),
                               smem_desc(sV0 + kVStage, 16, 1024, kSw128)};
      const uint64_t dvn[2] = {smem_desc(sV0, kSlabBytes, 1024, kSw128),
                               smem_desc(sV0 + kVStage, kSlabBytes, 1024, kSw128)};
      bool ok = warp_wait(smem_u32(&bar_qhi), 0, abort_flag, p.dev_status) &&
                warp_wait(smem_u32(&bar_qlo), 0, abort_flag, p.dev_status);
      // S(t) = Q K^T for tile t into S buffer t&1, in two parts with a fixed order:
      // the K-only slabs (Q from shared memory), then the V slabs (Q from TMEM).
      auto issue_s_k = [&](int t) -> bool {
        const int st = t & 1;
        if (!warp_wait(smem_u32(&bar_kfull[st]), (t >> 1) & 1, abort_flag, p.dev_status))
          return false;
        fence_proxy_async_smem();  // gathered rows (generic proxy) -> tensor core reads
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < kKOnly; ++i)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ss_elect(S_t[st], dq + ((i * kQSlabBytes + ks * 32) >> 4),
                         dk[st] + ((i * kSlabBytes + ks * 32) >> 4), idesc_s, (i | ks) != 0, e);
        mma_commit_elect(smem_u32(&bar_kempty[st]), e);
        return true;
      };
      auto issue_s_v = [&](int t) -> bool {
        const int st = t & 1;
        if (!warp_wait(smem_u32(&bar_vfull[st]), (t >> 1) & 1, abort_flag, p.dev_status))
          return false;
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < kVSlabs; ++i)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ts_elect(S_t[st], tmem + i * 32 + ks * 8,
                         dvk[st] + ((i * kSlabBytes + ks * 32) >> 4), idesc_s, 1, e);
        mma_commit_elect(smem_u32(&bar_s[st]), e);
        return true;
      };
      // Issue order: PV(t), S_v(t+1), S_k(t+2). The V slabs of tile t+1 were gathered
      // while S_v(t), S_k(t+1) and PV(t) ran; softmax(t+1) overlaps S_k(t+2).
      if (ok) {
        tc_fence_after();
        ok = issue_s_k(0) && issue_s_v(0) && (nt < 2 || issue_s_k(1));
      }
      for (int j = 0; ok && j < nt; ++j) {
        const int st = j & 1;
        if (!warp_wait(smem_u32(&bar_p[st]), (j >> 1) & 1, abort_flag, p.dev_status)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kTileN / 16; ++ks)
          mma_ts_elect(O_t, S_t[st] + ks * 8, dvn[st] + ((ks * 2048) >> 4), idesc_pv,
                       (j > 0 || ks > 0) ? 1u : 0u, e);
        mma_commit_elect(smem_u32(&bar_vempty[st]), e);
        if (j + 1 == nt) mma_commit_elect(smem_u32(&bar_o), e);
        if (j + 1 < nt && !issue_s_v(j + 1)) break;
        if (j + 2 < nt && !issue_s_k(j + 2)) break;
      }
      mma_commit_elect(smem_u32(&bar_drain), e);
      mbar_wait(smem_u32(&bar_drain), 0, nullptr, p.dev_status);
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ softmax / epilogue
    const int h = ((warp & 3) << 5) + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = p.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int st = j & 1;
      const uint32_t S_row = tmem + 128 + st * 64 + lane_off;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bar_s[st]), (j >> 1) & 1, abort_flag,
                                              p.dev_status));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[64];
      const float pm0 = tmem_ld32_max(S_row, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      const float pm1 = tmem_ld32_max(S_row + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld_wait();
      float* s = reinterpret_cast<float*>(sr);
      const int valid = cnt - (t_begin + j) * kTileN;  // entries of this tile that exist
      float tile_max = fmaxf(pm0, pm1);
      if (valid < kTileN) {  // entries past the list must not count in the max
#pragma unroll
        for (int cc = 0; cc < kTileN; ++cc)
          if (cc >= valid) s[cc] = -INFINITY;
        tile_max = row_max<kTileN>(s);
      }
      const float m_new = fmaxf(m_ref, tile_max);
      const bool resc = (m_new - m_ref) * c > 8.0f;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx((m_ref - m_new) * c);
        l *= alpha;
        m_ref = m_new;
      }
      const float neg_mc = (m_ref == -INFINITY) ? 0.f : -m_ref * c;
      l += exp2_pack_sum<kTileN>(sr, c, neg_mc);  // P as bf16 pairs over sr[0..31]
      tmem_st32(S_row, *reinterpret_cast<const uint32_t(*)[32]>(&sr[0]));
      if (j > 0 && __any_sync(0xFFFFFFFFu, resc)) {
        // O holds every PV up to tile j-1: PV(j-1) was issued before S_v(j), whose
        // completion this thread has observed (one commit covers all earlier MMAs).
        const uint32_t O_row = tmem + 256 + lane_off;
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(O_row + c0, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(O_row + c0, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_p[st]));
    }
    if (ok && nt > 0)
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bar_o), 0, abort_flag, p.dev_status));
    if (nparts == 1) {
      s_inv_l[h] = (l > 0.f) ? 1.f / l : 0.f;
      if (ok && r == 0 && p.lse != nullptr)
        p.lse[(int64_t)n * kHeads + h] =
            (l > 0.f) ? m_ref * p.scale + log2f(l) * 0.69314718055994531f : -INFINITY;
    } else {  // a part: O stays unnormalised; m and l go next to it
      s_inv_l[h] = 1.f;
      float* ml = p.partial + (int64_t)((u - p.n_main) * nparts + part) * kSlotFloats +
                  kHeads * 256;
      ml[h] = m_ref;
      ml[kHeads + h] = l;
    }
  }

  // The Q copies must have landed before the CTA may exit (they are otherwise only
  // waited for by roles that may have given up early).
  if (tid == 0) {
    mbar_wait(smem_u32(&bar_qhi), 0, nullptr, p.dev_status);
    mbar_wait(smem_u32(&bar_qlo_smem), 0, nullptr, p.dev_status);
  }
  tc_fence_before();
  __syncthreads();  // O is complete (bar_o) and every gather has landed
  tc_fence_after();

  // ---- epilogue: out = O / l (or a part's O, to its slot), by all 16 warps ----
  // Warp w reads TMEM lanes 32(w&3)..+31 (its heads) and columns 64(w>>2)..+63 of the
  // O half, 32 columns at a time, into an 8 KB slice of the idle gather stages laid out
  // as two 128-byte-swizzled 32 x 32 boxes; whole rows go out by TMA stores (a part's
  // O goes to its slot with plain stores, four heads per instruction).
  const bool fine = *abort_flag == 0;  // stable: every role has finished
  if (fine) {
    const int hq = warp & 3;
    const uint32_t O_row = tmem + 256 + (static_cast<uint32_t>(hq * 32) << 16);
    const float inv_l = s_inv_l[hq * 32 + lane];
    float* slot = p.partial + (int64_t)((u - p.n_main) * nparts + part) * kSlotFloats +
                  hq * 32 * 256;
#pragma unroll 1
    for (int ci = 0; ci < 2; ++ci) {
      const int c0 = (warp >> 2) * 64 + 32 * ci;
      float4* stage = reinterpret_cast<float4*>(smem + kQhiBytes + warp * 8192 + ci * 4096);
      uint32_t o[32];
      if (nt > 0) {
        tmem_ld32(O_row + c0, o);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q)
        stage[lane * 8 + (q ^ (lane & 7))] =
            make_float4(__uint_as_float(o[4 * q]) * inv_l, __uint_as_float(o[4 * q + 1]) * inv_l,
                        __uint_as_float(o[4 * q + 2]) * inv_l,
                        __uint_as_float(o[4 * q + 3]) * inv_l);
      if (nparts == 1) {
        fence_proxy_async_smem();  // the staged rows, for the copy engine
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&outmap, smem_u32(stage), 256 * r + c0, hq * 32, n);
          bulk_commit();
        }
      } else {
        __syncwarp();
#pragma unroll
        for (int rr = 0; rr < 32; rr += 4) {
          const int hh = rr + (lane >> 3), q = lane & 7;
          *reinterpret_cast<float4*>(slot + (int64_t)hh * 256 + c0 + 4 * q) =
              stage[hh * 8 + (q ^ (hh & 7))];
        }
      }
    }
    if (nparts == 1 && lane == 0) bulk_wait_read_all();  // the slices stay until read
  }
  if (nparts > 1 && nparts <= kKernelMergeParts && fine) {
    // The last part of the unit to finish merges all parts in part order:
    //   out = sum_p w_p O_p / sum_p w_p l_p,  w_p = 2^((m_p - M) * scale * log2 e),
    //   M = max_p m_p  (the online-softmax merge, with a fixed order).
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&p.done[u - p.n_main], 1u) == (uint32_t)(nparts - 1);
    __syncthreads();
    if (s_last) {
      __threadfence();
      const float* slot0 = p.partial + (int64_t)(u - p.n_main) * nparts * kSlotFloats;
      // merge weights [part][head], in the idle gather stages (the staging is done)
      float* s_w = reinterpret_cast<float*>(smem + kQhiBytes);
      if (tid < kHeads)
        merge_weights<kKernelMergeParts>(p, slot0, nparts, tid, n, r, s_w, kHeads);
      __syncthreads();
      float* obase = p.out + (int64_t)n * kHeads * kDv + 256 * r;
      for (int i = tid; i < kHeads * 64; i += kThreads)
        merge_row_chunk<kKernelMergeParts>(slot0, nparts, s_w, kHeads, i >> 6, i >> 6,
                                           i & 63, obase);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The merge of units split into more than kKernelMergeParts parts: one CTA per (split
// unit, 16 heads), after the attention launch, with the in-kernel merge's arithmetic.
constexpr int kMergeHeads = 16;
constexpr int kMergeThreads = 256;
__global__ void __launch_bounds__(kMergeThreads) sparse_merge_kernel(const SparseParams p) {
  __shared__ float s_w[kMaxParts * kMergeHeads];
  const int k = blockIdx.x / (kHeads / kMergeHeads);
  const int h0 = (blockIdx.x % (kHeads / kMergeHeads)) * kMergeHeads;
  const int u = p.n_main + k, n = u >> 1, r = u & 1;
  const float* slot0 = p.partial + (int64_t)k * p.parts * kSlotFloats;
  if (threadIdx.x < kMergeHeads)
    merge_weights<kMaxParts>(p, slot0, p.parts, h0 + threadIdx.x, n, r, s_w, kMergeHeads,
                             threadIdx.x);
  __syncthreads();
  float* obase = p.out + (int64_t)n * kHeads * kDv + 256 * r;
  for (int i = threadIdx.x; i < kMergeHeads * 64; i += kMergeThreads)
    merge_row_chunk<kMaxParts>(slot0, p.parts, s_w, kMergeHeads, h0 + (i >> 6), i >> 6, i & 63,
                               obase);
}

// The canonical lists of every query ahead of the attention launch, one CTA per query,
// so that the attention CTAs start gathering at once instead of sorting first.
__global__ void __launch_bounds__(kThreads)
    sparse_sort_kernel(const SparseParams p, int scratch_ints) {
  extern __shared__ int32_t scratch[];
  __shared__ int s_cnt;
  __shared__ int s_wsum[kThreads / 32];
  const int n = blockIdx.x;
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  const int32_t* rows;
  const int cnt = canonical_rows(p, n, scratch, scratch_ints, &s_cnt, s_wsum, &rows);
  int32_t* dst = p.sorted_rows + (int64_t)n * kMaxTopk;
  for (int i = threadIdx.x; i < cnt; i += kThreads) dst[i] = rows[i];
  if (threadIdx.x == 0) p.sorted_cnt[n] = cnt;
}

// The split of the last wave: with U = 2 nq units on `sms` SMs, the U mod sms units of
// the partial wave run as `parts` CTAs each, as many as still fit in one wave (at most
// kMaxParts); a small batch (decode with few requests) so fills the SMs.
struct SplitPlan {
  int tail = 0, parts = 1;
  size_t done_bytes = 0, bytes = 0;
};
SplitPlan plan_split(int nq, int sms) {
  SplitPlan s;
  const int units = 2 * nq;
  const int tail = sms > 0 ? units % sms : 0;
  if (tail == 0) return s;
  int parts = sms / tail;
  if (parts > kMaxParts) parts = kMaxParts;
  if (parts < 2) return s;
  s.tail = tail;
  s.parts = parts;
  s.done_bytes = ((size_t)tail * 4 + 255) / 256 * 256;
  s.bytes = s.done_bytes + (size_t)tail * parts * kSlotFloats * sizeof(float);
  return s;
}

}  // namespace

// Workspace layout: the split region (when the shape splits), then from the next 256-byte
// boundary the canonical lists: counts [nq] (rounded up to 256 bytes), rows [nq][kMaxTopk].
size_t sorted_lists_bytes(int nq) {
  return ((size_t)nq * 4 + 255) / 256 * 256 + (size_t)nq * kMaxTopk * 4;
}

size_t sparse_split_workspace_bytes(int nq, int sms) {
  return (plan_split(nq, sms).bytes + 255) / 256 * 256 + sorted_lists_bytes(nq);
}

cudaError_t launch_sparse_attn(const SparseArgs& a, int* drv_err, cudaStream_t stream) {
  if (a.heads != kHeads || a.dqk != kDqk || a.dv != kDv || a.topk > kMaxTopk)
    return cudaErrorNotSupported;
  CUtensorMap qmap;
  const uint64_t dims[3] = {(uint64_t)kDqk, (uint64_t)kHeads, (uint64_t)a.nq};
  const uint64_t strides[2] = {(uint64_t)kDqk * 2, (uint64_t)kHeads * kDqk * 2};
  const uint32_t box[3] = {64, kHeads, 1};
  CUresult rr = encode_tensor_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                                  const_cast<void*>(a.q), dims, strides, box,
                                  CU_TENSOR_MAP_SWIZZLE_128B);
  if (rr != CUDA_SUCCESS) {
    *drv_err = (int)rr;
    return cudaErrorInvalidValue;
  }
  // The cache as rows of 576 values for the four-row gathers (box: 64 columns x 1 row).
  CUtensorMap kvmap;
  const uint64_t kv_dims[2] = {(uint64_t)kDqk, (uint64_t)a.num_pages * a.page_size};
  const uint64_t kv_strides[1] = {(uint64_t)kDqk * 2};
  const uint32_t kv_box[2] = {64, 1};
  rr = encode_tensor_map(&kvmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                         const_cast<void*>(a.kv_cache), kv_dims, kv_strides, kv_box,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  if (rr != CUDA_SUCCESS) {
    *drv_err = (int)rr;
    return cudaErrorInvalidValue;
  }
  // The output as 32 x 32 fp32 boxes (32 columns = 128 bytes, 32 heads) for TMA stores.
  CUtensorMap outmap;
  const uint64_t o_dims[3] = {(uint64_t)kDv, (uint64_t)kHeads, (uint64_t)a.nq};
  const uint64_t o_strides[2] = {(uint64_t)kDv * 4, (uint64_t)kHeads * kDv * 4};
  const uint32_t o_box[3] = {32, 32, 1};
  rr = encode_tensor_map(&outmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.out, o_dims, o_strides,
                         o_box, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rr != CUDA_SUCCESS) {
    *drv_err = (int)rr;
    return cudaErrorInvalidValue;
  }
  SparseParams p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.kv = static_cast<const uint16_t*>(a.kv_cache);
  p.page_table = a.page_table;
  p.kv_lens = a.kv_lens;
  p.pt_stride = a.pt_stride;
  p.idx = a.idx;
  p.out = a.out;
  p.lse = a.lse;
  p.dev_status = a.dev_status;
  p.nq = a.nq;
  p.num_pages = a.num_pages;
  p.page_size = a.page_size;
  p.page_shift = -1;
  for (int sh = 0; sh < 31; ++sh)
    if ((1 << sh) == a.page_size) p.page_shift = sh;
  p.num_logical_pages = a.num_logical_pages;
  p.kv_len = a.kv_len;
  p.topk = a.topk;
  int sort_n = 64;
  while (sort_n < a.topk) sort_n <<= 1;
  p.sort_n = sort_n;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  const int units = 2 * a.nq;
  p.n_main = units;
  p.parts = 1;
  p.partial = nullptr;
  p.done = nullptr;
  p.sorted_rows = nullptr;
  p.sorted_cnt = nullptr;
  int grid = units;
  if (a.workspace != nullptr) {
    int dev = 0, sms = 0;
    cudaError_t ea = cudaGetDevice(&dev);
    if (ea == cudaSuccess) ea = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (ea != cudaSuccess) return ea;
    const SplitPlan sp = plan_split(a.nq, sms);
    const size_t lists_at = (sp.bytes + 255) / 256 * 256;
    if (a.workspace_bytes >= lists_at + sorted_lists_bytes(a.nq)) {
      // The canonical lists first, by a launch of their own (one CTA per query).
      p.sorted_cnt = reinterpret_cast<int32_t*>(static_cast<char*>(a.workspace) + lists_at);
      p.sorted_rows = reinterpret_cast<int32_t*>(static_cast<char*>(a.workspace) + lists_at +
                                                 ((size_t)a.nq * 4 + 255) / 256 * 256);
      // Scratch: counts (counting sort), the page table when it fits, the list; with one
      // length for every query its need is known here, else the largest.
      int scratch_ints = kScratchInts;
      if (a.kv_lens == nullptr) {
        const int n_counts = a.kv_len <= kCountCap ? a.kv_len : 0;
        const int n_scan = a.kv_len <= kCountCap ? a.topk : sort_n;
        const int want = n_counts + a.num_logical_pages + n_scan;
        scratch_ints = want < kScratchInts ? want : kScratchInts;
        if (scratch_ints < n_counts + n_scan) scratch_ints = n_counts + n_scan;
      }
      const size_t sort_smem = (size_t)scratch_ints * 4;
      ea = cudaFuncSetAttribute(sparse_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sort_smem);
      if (ea != cudaSuccess) return ea;
      sparse_sort_kernel<<<a.nq, kThreads, sort_smem, stream>>>(p, scratch_ints);
      ea = cudaGetLastError();
      if (ea != cudaSuccess) return ea;
    }
    if (sp.parts > 1 && a.workspace_bytes >= sp.bytes) {
      p.done = static_cast<uint32_t*>(a.workspace);
      p.partial = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + sp.done_bytes);
      p.n_main = units - sp.tail;
      p.parts = sp.parts;
      grid = p.n_main + sp.tail * sp.parts;
      if (sp.parts <= kKernelMergeParts) {  // the last part to finish merges
        ea = cudaMemsetAsync(p.done, 0, (size_t)sp.tail * 4, stream);
        if (ea != cudaSuccess) return ea;
      }
    }
  }
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  sparse_attn_kernel<<<grid, kThreads, kSmemBytes, stream>>>(qmap, kvmap, outmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.parts <= kKernelMergeParts) return e;
  const int tail = (grid - p.n_main) / p.parts;
  sparse_merge_kernel<<<tail * (kHeads / kMergeHeads), kMergeThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace tts
