// Dense attention forward (non-causal vision and varlen causal GQA prefill).
//
// What it computes: for every query row, softmax(scale * q K^T) V over the
// visible keys, plus lse = ln sum exp(scale * q k) -- the S-gemm / softmax /
// PV-gemm pieces of "DeepSeek V4.1 上 4×RTX 3090" (section 三), over the
// cu_seqlens batches of "从 SGLang Kernel源码到 GPU Trace" (section 2.2, keys past
// a sequence's length skipped as in section 3.2), FP32 statistics and FP32
// accumulation as in "AMD MI250部署DeepSeek-V4-Flash" (3.1, 4.1), causal mask
// as -inf (3.3), and the online-softmax merge of "推理引擎的蝴蝶效应" (进一步探索,
// equations 1-2) applied tile after tile in a fixed order.
//
// How: one persistent CTA per SM takes work items -- (sequence, 256-row query
// pair, head), heaviest first -- from a global counter in the caller's workspace:
//   warp 0        TMA producer: picks the items, then per item K/V 128-row tiles
//                 into a ring and the two Q tiles (the next item's loads overlap
//                 the current item's last tiles and epilogue)
//   warp 1        TMEM allocator + tcgen05 MMA issuer (the whole warp runs the
//                 issue loop converged; one elected lane issues)
//   warps 4..7    softmax warpgroup 0 (query rows 0..127 of the pair)
//   warps 8..11   softmax warpgroup 1 (query rows 128..255)
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [384,384+D).
// S = Q K^T lands in TMEM; each softmax thread owns one row (TMEM lane), keeps
// the running max / sum in fp32 registers, writes P as bf16 pairs over the first
// 64 columns of its S region, and the MMA warp issues O += P V with P read
// straight from TMEM. The two warpgroups ping-pong so the tensor core works
// on one tile's MMAs while the other tile's softmax runs.
// The running max is only moved (and O rescaled) when it grows by more than
// 2^8 in the exp2 domain; otherwise P uses the older max, which bounds P by
// 256 and is exact in real arithmetic (the final O / l cancels the offset).
// No S or P matrix ever touches global memory, so there is no piece buffer
// to index (the q0*N overflow of the vision write-up cannot happen here).
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace tts {
namespace {

constexpr int kAttnThreads = 384;
constexpr int kBlockM = 128;  // query rows per softmax warpgroup
constexpr int kBlockN = 128;  // keys per K/V tile

// Instruction descriptor for kind::f8f6f4 with e4m3 A and B (format code 0), fp32 D,
// both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
// D[tmem] (+)= A[smem] * B[smem], e4m3 operands, from the elected lane of a converged warp.
__device__ __forceinline__ void mma_ss_f8_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate,
                                                uint32_t pred) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
      : "memory");
}

// F8: q and k are e4m3 (one byte per value) and S = Q K^T runs as kind::f8f6f4 MMAs;
// V, P and O stay bf16 / fp32. Built for D = 128 only.
template <int D, bool F8 = false>
struct AttnCfg {
  static constexpr int kQKCols = F8 ? 128 : 64;  // q / k values per 128-byte row
  static constexpr int kMainBoxes = D / kQKCols;  // SW128 boxes of q / k
  static constexpr int kTail = F8 ? 0 : D % 64;   // 0 or 16 (SW32 box)
  static constexpr int kBoxBytes = kBlockN * 128;  // one SW128 box of 128 rows
  static constexpr int kTailBytes = kBlockN * 32;  // one SW32 box of 128 rows
  static constexpr int kTileBytes = kMainBoxes * kBoxBytes + (kTail ? kTailBytes : 0);
  // V for d=80 is loaded as three 32-column SW64 boxes (d 80..95 zero-filled by the
  // tensor map's bounds) so that one N=96 MMA per K step covers it; d=64/128 reuse the
  // K/Q layout.
  static constexpr int kVBoxes = kTail ? 3 : D / 64;
  static constexpr int kVBoxBytes = kTail ? kBlockN * 64 : kBoxBytes;
  static constexpr int kVTileBytes = kVBoxes * kVBoxBytes;
  static constexpr int kPvN = kTail ? 96 : D;
  static constexpr int kStages = (D <= 80 || F8) ? 3 : 2;
  static constexpr int kStageBytes = 8 * 4096;  // output staging, 4 KB per softmax warp
  static constexpr int kSmemBytes =
      (2 + kStages) * kTileBytes + kStages * kVTileBytes + kStageBytes + 1024;
  static_assert(kTail == 0 || kTail == 16, "head_dim must be 64, 80 or 128");
  static_assert(!F8 || D == 128, "the e4m3 q / k path is built for head_dim 128");
};

struct AttnMaps {
  CUtensorMap q, k, v;           // SW128 boxes {64, 1, 128} (q / k e4m3: {128, 1, 128})
  CUtensorMap q_t, k_t;          // SW32 boxes {16, 1, 128} for the d=64..79 tail
  CUtensorMap v_t;               // d=80: SW64 boxes {32, 1, 128} for all of V
};

struct AttnParams {
  const int32_t* cu_q;
  const int32_t* cu_k;
  uint32_t* work_counter;  // items handed out so far (zeroed before the launch)
  int n_items;
  float* out;
  float* lse;
  uint32_t* dev_status;
  int64_t total_q, total_k;
  int batch, max_seqlen_q, max_seqlen_k, hq, hkv, causal, pairs_max;
  float scale, scale_log2;
  const float* q_scale;  // e4m3 path: [total_q, hq] per (token, head)
  const float* k_scale;  // e4m3 path: [hkv] per KV head
};

// Load one 128-row tile (all boxes) of a [tokens, heads, D] tensor (F8: of e4m3 q / k).
template <int D, bool F8 = false>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* main,
                                          const CUtensorMap* tail, uint32_t bar, int head,
                                          int token) {
  using C = AttnCfg<D, F8>;
#pragma unroll
  for (int b = 0; b < C::kMainBoxes; ++b)
    tma_load_3d(dst + b * C::kBoxBytes, main, bar, b * C::kQKCols, head, token);
  if constexpr (C::kTail != 0)
    tma_load_3d(dst + C::kMainBoxes * C::kBoxBytes, tail, bar, C::kMainBoxes * 64, head, token);
}

// S[tmem] = Q[smem] K[smem]^T over the D-deep contraction. q_d / k_d are the
// descriptors of the tiles' first box; every other K step is a constant offset
// (the 14-bit start-address field never carries: shared addresses are < 256 KB).
// e: the elected lane of the converged issuing warp.
// F8: e4m3 x e4m3 -> fp32, K = 32 per MMA, so the same 32-byte steps cover the row.
template <int D, bool F8 = false>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t q_d, uint64_t k_d,
                                         uint64_t q_tail_d, uint64_t k_tail_d, uint32_t e) {
  using C = AttnCfg<D, F8>;
  constexpr uint32_t idesc =
      F8 ? idesc_e4m3_f32(128, kBlockN) : idesc_bf16_f32(128, kBlockN, 0, 0);
#pragma unroll
  for (int ks = 0; ks < C::kMainBoxes * 4; ++ks) {
    const uint32_t off = ((ks / 4) * C::kBoxBytes + (ks % 4) * 32) >> 4;
    if constexpr (F8)
      mma_ss_f8_elect(d_tmem, q_d + off, k_d + off, idesc, ks > 0, e);
    else
      mma_ss_elect(d_tmem, q_d + off, k_d + off, idesc, ks > 0, e);
  }
  if constexpr (C::kTail != 0) mma_ss_elect(d_tmem, q_tail_d, k_tail_d, idesc, 1, e);
}

// O[tmem] (+)= P[tmem] V[smem]; V is MN-major (d contiguous). v_d describes the
// first V box (SW128 boxes for d=64/128, SW64 boxes for d=80).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_d,
                                         uint32_t accumulate, uint32_t e) {
  using C = AttnCfg<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(128, C::kPvN, 0, 1);
  constexpr uint32_t kStep = C::kTail ? 16 * 64 : 16 * 128;  // 16 key rows of one box
#pragma unroll
  for (int ks = 0; ks < kBlockN / 16; ++ks)
    mma_ts_elect(o_tmem, p_tmem + ks * 8, v_d + ((ks * kStep) >> 4), idesc,
                 (ks > 0) ? 1u : accumulate, e);
}


// One work item = (256-row query pair, sequence, head); `it` enumerates them with
// the heaviest (latest, causal) pairs of every sequence first. Every role decodes
// an item the same way. Returns false for items with nothing to compute and for
// sequences whose cu_seqlens entries are invalid.
struct Item {
  int64_t q_start, k_start, Lq, Lk, q_lo;
  int h, g, n_tiles;  // n_tiles: K/V tiles streamed = max(n0, n1)
  int n0, n1;         // tiles each warpgroup needs (0: no rows, or no visible key)
};
__device__ __forceinline__ bool decode_item(const AttnParams& p, int it, Item& w, bool* bad) {
  const int h = it % p.hq;
  const int t = it / p.hq;
  const int b = t % p.batch;
  const int pr = p.pairs_max - 1 - t / p.batch;
  const int64_t q_start = p.cu_q[b], k_start = p.cu_k[b];
  const int64_t q_end = p.cu_q[b + 1], k_end = p.cu_k[b + 1];
  const int64_t Lq = q_end - q_start, Lk = k_end - k_start;
  *bad = false;
  if (q_start < 0 || k_start < 0 || Lq < 0 || Lk < 0 || q_end > p.total_q || k_end > p.total_k ||
      Lq > p.max_seqlen_q || Lk > p.max_seqlen_k) {
    *bad = (pr == 0 && h == 0);  // report each bad sequence once
    return false;
  }
  // First query row of the pair (within the sequence). With an odd number of 128-row
  // query tiles the pairs start one tile early, so the tile without a partner is tile 0
  // (the cheapest under a causal mask: one key tile) and the first warpgroup of pair 0
  // has no rows.
  const int64_t n_qt = (Lq + kBlockM - 1) / kBlockM;
  const int64_t q_lo = (int64_t)pr * 2 * kBlockM - ((n_qt & 1) ? kBlockM : 0);
  if (q_lo >= Lq) return false;
  // Keys each warpgroup's rows can see: all of them, or (causal) up to its last row's
  // diagonal; none for a warpgroup without rows (the odd last tile of a sequence).
  auto keys_for = [&](int64_t r_first, int64_t r_end) -> int64_t {
    if (r_first >= Lq || r_end <= 0) return 0;
    if (!p.causal) return Lk;
    const int64_t lim = (r_end < Lq ? r_end : Lq) - 1 + (Lk - Lq) + 1;
    return lim < 0 ? 0 : (lim < Lk ? lim : Lk);
  };
  const int64_t kv_end0 = keys_for(q_lo, q_lo + kBlockM);
  const int64_t kv_end1 = keys_for(q_lo + kBlockM, q_lo + 2 * kBlockM);
  const int64_t kv_end = kv_end0 > kv_end1 ? kv_end0 : kv_end1;
  w.q_start = q_start;
  w.k_start = k_start;
  w.Lq = Lq;
  w.Lk = Lk;
  w.q_lo = q_lo;
  w.h = h;
  w.g = h / (p.hq / p.hkv);
  w.n_tiles = (int)((kv_end + kBlockN - 1) / kBlockN);
  w.n0 = (int)((kv_end0 + kBlockN - 1) / kBlockN);
  w.n1 = (int)((kv_end1 + kBlockN - 1) / kBlockN);
  return true;
}

// Persistent: one CTA per SM takes items from a global counter until none are left.
// Per CTA, items flow through a two-slot ring (producer -> MMA warp + softmax warps);
// barrier phases run on counters that continue across items: gt = K/V tiles so far
// (ring slots, S / P phases), nq = items with at least one tile (Q, O phases).
template <int D, bool F8 = false>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_kernel(const __grid_constant__ AttnMaps maps, const AttnParams p) {
  using C = AttnCfg<D, F8>;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  // bar_k / bar_v: K and V of a tile landed. With three stages (d <= 80) the V load
  // has time to land before the S MMA that first needs the tile, so both share bar_k
  // and the MMA warp waits once per tile; with two stages (d = 128) V gets its own
  // barrier so S(j+1) does not wait for V(j+1), and K's slot is released (bar_k_empty)
  // as soon as both S MMAs of its tile are done, a PV pair before V's slot
  // (bar_kv_empty), so the next K load starts that much earlier.
  constexpr bool kOneKV = NS >= 3;
  __shared__ __align__(8) uint64_t bar_item_full[2], bar_item_empty[2], bar_q[2], bar_q_empty[2],
      bar_k[NS], bar_v[NS], bar_k_empty[NS], bar_kv_empty[NS], bar_s[2], bar_p[2], bar_o[2],
      bar_drain;
  __shared__ int s_item[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ[2] = {s_base, s_base + C::kTileBytes};
  auto sK = [&](int st) { return s_base + (2 + st) * C::kTileBytes; };
  auto sV = [&](int st) {
    return s_base + (2 + NS) * C::kTileBytes + st * C::kVTileBytes;
  };
  // Output staging: 4 KB per softmax warp, after the K/V ring.
  uint8_t* stage_base = smem + (2 + NS) * C::kTileBytes + NS * C::kVTileBytes;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_item_full[i]), 1);
      mbar_init(smem_u32(&bar_item_empty[i]), 1 + 8);  // MMA warp + 8 softmax warps
      mbar_init(smem_u32(&bar_q[i]), 1);
      mbar_init(smem_u32(&bar_q_empty[i]), 1);
      mbar_init(smem_u32(&bar_s[i]), 1);
      mbar_init(smem_u32(&bar_p[i]), kBlockM);
      mbar_init(smem_u32(&bar_o[i]), 1);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bar_k[i]), 1);
      mbar_init(smem_u32(&bar_v[i]), 1);
      mbar_init(smem_u32(&bar_k_empty[i]), 1);
      mbar_init(smem_u32(&bar_kv_empty[i]), 1);
    }
    mbar_init(smem_u32(&bar_drain), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  volatile int* item_slot = s_item;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&maps.q);
      prefetch_tmap(&maps.k);
      prefetch_tmap(&maps.v);
      int ni = 0, nq = 0, gt = 0;
      int last_k[NS], last_v[NS];  // latest tile armed on each ring slot (-1: none)
      for (int i = 0; i < NS; ++i) last_k[i] = last_v[i] = -1;
      int q_armed[2] = {0, 0};  // per Q tile: items whose Q copy was started
      // Start the K (and V) copies of ring tile gj = item tile j.
      auto load_k = [&](int gj, const Item& w, int j) -> bool {
        const int st = gj % NS;
        const uint32_t empty_ph = ((gj / NS) - 1) & 1;
        if (gj >= NS && !mbar_wait(smem_u32(kOneKV ? &bar_kv_empty[st] : &bar_k_empty[st]),
                                   empty_ph, abort_flag, p.dev_status))
          return false;
        const int tok = (int)(w.k_start + (int64_t)j * kBlockN);
        const uint32_t bk = smem_u32(&bar_k[st]);
        mbar_arrive_expect_tx(bk, kOneKV ? C::kTileBytes + C::kVTileBytes : C::kTileBytes);
        load_tile<D, F8>(sK(st), &maps.k, &maps.k_t, bk, w.g, tok);
        last_k[st] = gj;
        return true;
      };
      auto load_v = [&](int gj, const Item& w, int j) -> bool {
        const int st = gj % NS;
        const uint32_t bv = smem_u32(kOneKV ? &bar_k[st] : &bar_v[st]);
        if (!kOneKV) {
          if (gj >= NS && !mbar_wait(smem_u32(&bar_kv_empty[st]), ((gj / NS) - 1) & 1, abort_flag,
                                     p.dev_status))
            return false;
          mbar_arrive_expect_tx(bv, C::kVTileBytes);
        }
        const int tok = (int)(w.k_start + (int64_t)j * kBlockN);
        if constexpr (C::kTail != 0) {
#pragma unroll
          for (int b = 0; b < C::kVBoxes; ++b)
            tma_load_3d(sV(st) + b * C::kVBoxBytes, &maps.v_t, bv, b * 32, w.g, tok);
        } else {
          load_tile<D>(sV(st), &maps.v, &maps.v, bv, w.g, tok);
        }
        last_v[st] = gj;
        return true;
      };
      bool ok = true;
      while (ok) {
        Item w;
        int it;
        for (;;) {  // next item with work (bad sequences are reported here, once)
          it = (int)atomicAdd(p.work_counter, 1u);
          if (it >= p.n_items) {
            it = -1;
            break;
          }
          bool bad;
          if (decode_item(p, it, w, &bad)) break;
          if (bad && p.dev_status) atomicOr(p.dev_status, kDevBadArg);
        }
        const int slot = ni & 1;
        if (ni >= 2 &&
            !mbar_wait(smem_u32(&bar_item_empty[slot]), ((ni >> 1) - 1) & 1, abort_flag,
                       p.dev_status))
          break;
        item_slot[slot] = it;
        mbar_arrive(smem_u32(&bar_item_full[slot]));  // release: the slot write is visible
        ++ni;
        if (it < 0) break;
        const int n = w.n_tiles;
        if (n == 0) continue;
        // The first ring tiles go first (their slots free up while the previous item
        // finishes); Q waits for the previous item's last S MMAs; the remaining tiles
        // need slots that this item's own MMAs free, so they come after Q.
        const int pre = n < NS ? n : NS;
        for (int j = 0; ok && j < pre; ++j) ok = load_k(gt + j, w, j) && load_v(gt + j, w, j);
        for (int wq = 0; ok && wq < 2; ++wq) {
          if (nq >= 1 && !mbar_wait(smem_u32(&bar_q_empty[wq]), (nq - 1) & 1, abort_flag,
                                    p.dev_status)) {
            ok = false;
            break;
          }
          const uint32_t bq = smem_u32(&bar_q[wq]);
          mbar_arrive_expect_tx(bq, C::kTileBytes);
          load_tile<D, F8>(sQ[wq], &maps.q, &maps.q_t, bq, w.h,
                       (int)(w.q_start + w.q_lo + wq * kBlockM));
          q_armed[wq] = nq + 1;
        }
        for (int j = pre; ok && j < n; ++j) ok = load_k(gt + j, w, j) && load_v(gt + j, w, j);
        gt += n;
        ++nq;
      }
      if (*abort_flag) {
        // Best-effort drain of copies still in flight before the CTA can exit: each
        // barrier's latest armed phase is the only one that can still be pending.
        for (int wq = 0; wq < 2; ++wq)
          if (q_armed[wq] > 0)
            mbar_wait(smem_u32(&bar_q[wq]), (q_armed[wq] - 1) & 1, nullptr, nullptr);
        for (int st = 0; st < NS; ++st) {
          if (last_k[st] >= 0)
            mbar_wait(smem_u32(&bar_k[st]), (last_k[st] / NS) & 1, nullptr, nullptr);
          if (!kOneKV && last_v[st] >= 0)
            mbar_wait(smem_u32(&bar_v[st]), (last_v[st] / NS) & 1, nullptr, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t e = elect_one();
    const uint32_t S_t[2] = {tmem, tmem + 128};
    const uint32_t O_t[2] = {tmem + 256, tmem + 384};
    constexpr uint32_t kTailOff = C::kMainBoxes * C::kBoxBytes;
    uint64_t qd[2], qtd[2], kd[NS], ktd[NS], vd[NS];
    for (int w = 0; w < 2; ++w) {
      qd[w] = smem_desc(sQ[w], 16, 1024, kSw128);
      qtd[w] = smem_desc(sQ[w] + kTailOff, 16, 256, kSw32);
    }
    for (int i = 0; i < NS; ++i) {
      kd[i] = smem_desc(sK(i), 16, 1024, kSw128);
      ktd[i] = smem_desc(sK(i) + kTailOff, 16, 256, kSw32);
      vd[i] = C::kTail ? smem_desc(sV(i), C::kVBoxBytes, 512, kSw64)
                       : smem_desc(sV(i), C::kBoxBytes, 1024, kSw128);
    }
    // gt: K/V tiles so far (ring phases); g0 / g1: tiles of each warpgroup so far (S and P
    // phases); nq: items with tiles (Q phases).
    int ni = 0, nq = 0, gt = 0, g0 = 0, g1 = 0;
    bool ok = true;
    while (ok) {
      const int slot = ni & 1;
      if (!warp_wait(smem_u32(&bar_item_full[slot]), (ni >> 1) & 1, abort_flag, p.dev_status))
        break;
      const int it = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_item_empty[slot]));
      ++ni;
      if (it < 0) break;
      Item w;
      bool bad;
      decode_item(p, it, w, &bad);
      const int n = w.n_tiles, n0 = w.n0, n1 = w.n1;
      if (n == 0) continue;
      const int st0 = gt % NS;
      ok = warp_wait(smem_u32(&bar_q[0]), nq & 1, abort_flag, p.dev_status) &&
           warp_wait(smem_u32(&bar_k[st0]), (gt / NS) & 1, abort_flag, p.dev_status);
      if (!ok) break;
      tc_fence_after();
      if (n0 > 0) {
        issue_qk<D, F8>(S_t[0], qd[0], kd[st0], qtd[0], ktd[st0], e);
        mma_commit_elect(smem_u32(&bar_s[0]), e);
      }
      if (n0 <= 1) mma_commit_elect(smem_u32(&bar_q_empty[0]), e);
      ok = warp_wait(smem_u32(&bar_q[1]), nq & 1, abort_flag, p.dev_status);
      if (!ok) break;
      tc_fence_after();
      if (n1 > 0) {
        issue_qk<D, F8>(S_t[1], qd[1], kd[st0], qtd[1], ktd[st0], e);
        mma_commit_elect(smem_u32(&bar_s[1]), e);
      }
      if (!kOneKV) mma_commit_elect(smem_u32(&bar_k_empty[st0]), e);
      if (n1 <= 1) mma_commit_elect(smem_u32(&bar_q_empty[1]), e);
      // Order on the tensor core: PV0(j) S0(j+1) PV1(j) S1(j+1), each warpgroup only for
      // the tiles its rows can see (its fully masked tiles are never computed). First the
      // tiles after which both warpgroups still have one (the straight-line body), then
      // the last one or two, where a warpgroup may stop or sit out.
      const int nb = n0 < n1 ? n0 : n1;
      int j = 0;
      for (; j + 1 < nb; ++j) {
        const int gj = gt + j;
        const int st = gj % NS;
        const int st1 = (gj + 1) % NS;
        if (!kOneKV && !warp_wait(smem_u32(&bar_v[st]), (gj / NS) & 1, abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        if (!warp_wait(smem_u32(&bar_p[0]), (g0 + j) & 1, abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv<D>(O_t[0], S_t[0], vd[st], j > 0, e);
        if (!warp_wait(smem_u32(&bar_k[st1]), ((gj + 1) / NS) & 1, abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_qk<D, F8>(S_t[0], qd[0], kd[st1], qtd[0], ktd[st1], e);
        mma_commit_elect(smem_u32(&bar_s[0]), e);
        if (j + 2 == n0) mma_commit_elect(smem_u32(&bar_q_empty[0]), e);
        if (!warp_wait(smem_u32(&bar_p[1]), (g1 + j) & 1, abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv<D>(O_t[1], S_t[1], vd[st], j > 0, e);
        mma_commit_elect(smem_u32(&bar_kv_empty[st]), e);
        issue_qk<D, F8>(S_t[1], qd[1], kd[st1], qtd[1], ktd[st1], e);
        mma_commit_elect(smem_u32(&bar_s[1]), e);
        if (!kOneKV) mma_commit_elect(smem_u32(&bar_k_empty[st1]), e);
        if (j + 2 == n1) mma_commit_elect(smem_u32(&bar_q_empty[1]), e);
      }
      for (; ok && j < n; ++j) {
        const int gj = gt + j;
        const int st = gj % NS;
        const int st1 = (gj + 1) % NS;
        const bool act0 = j < n0, act1 = j < n1;
        const bool more0 = j + 1 < n0, more1 = j + 1 < n1;
        if (!kOneKV && !warp_wait(smem_u32(&bar_v[st]), (gj / NS) & 1, abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        // warpgroup 0
        if (act0) {
          if (!warp_wait(smem_u32(&bar_p[0]), (g0 + j) & 1, abort_flag, p.dev_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv<D>(O_t[0], S_t[0], vd[st], j > 0, e);
          if (more0) {
            if (!warp_wait(smem_u32(&bar_k[st1]), ((gj + 1) / NS) & 1, abort_flag,
                           p.dev_status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_qk<D, F8>(S_t[0], qd[0], kd[st1], qtd[0], ktd[st1], e);
            mma_commit_elect(smem_u32(&bar_s[0]), e);
            if (!kOneKV && !more1) mma_commit_elect(smem_u32(&bar_k_empty[st1]), e);
            if (j + 2 == n0) mma_commit_elect(smem_u32(&bar_q_empty[0]), e);
          } else {
            mma_commit_elect(smem_u32(&bar_o[0]), e);
          }
        }
        // warpgroup 1
        if (act1) {
          if (!warp_wait(smem_u32(&bar_p[1]), (g1 + j) & 1, abort_flag, p.dev_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv<D>(O_t[1], S_t[1], vd[st], j > 0, e);
        }
        mma_commit_elect(smem_u32(&bar_kv_empty[st]), e);  // every PV of this tile issued
        if (act1) {
          if (more1) {
            if (!more0 && !warp_wait(smem_u32(&bar_k[st1]), ((gj + 1) / NS) & 1, abort_flag,
                                     p.dev_status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_qk<D, F8>(S_t[1], qd[1], kd[st1], qtd[1], ktd[st1], e);
            mma_commit_elect(smem_u32(&bar_s[1]), e);
            if (!kOneKV) mma_commit_elect(smem_u32(&bar_k_empty[st1]), e);
            if (j + 2 == n1) mma_commit_elect(smem_u32(&bar_q_empty[1]), e);
          } else {
            mma_commit_elect(smem_u32(&bar_o[1]), e);
          }
        }
      }
      gt += n;
      g0 += n0;
      g1 += n1;
      ++nq;
    }
    // Drain: every MMA issued by this warp is complete before TMEM is freed.
    mma_commit_elect(smem_u32(&bar_drain), e);
    mbar_wait(smem_u32(&bar_drain), 0, nullptr, p.dev_status);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / epilogue
    const int wg = (warp - 4) >> 2;            // 0 or 1
    const int row = ((warp & 3) << 5) + lane;  // TMEM lane == row within the tile
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t S_row = tmem + wg * 128 + lane_off;
    const uint32_t O_row = tmem + 256 + wg * 128 + lane_off;
    float4* stage = reinterpret_cast<float4*>(stage_base + (warp - 4) * 4096);
    int ni = 0, nq = 0, gt = 0;
    bool ok = true;
    while (ok) {
      const int slot = ni & 1;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bar_item_full[slot]), (ni >> 1) & 1,
                                              abort_flag, p.dev_status));
      if (!ok) break;
      const int it = item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_item_empty[slot]));
      ++ni;
      if (it < 0) break;
      Item w;
      bool bad;
      decode_item(p, it, w, &bad);
      const int n_tiles = wg == 0 ? w.n0 : w.n1;  // tiles this warpgroup's rows can see
      const int64_t Lq = w.Lq, Lk = w.Lk;
      const int64_t i = w.q_lo + wg * kBlockM + row;  // query row within the sequence
      int64_t limit = Lk;                            // keys [0, limit) visible to this row
      if (p.causal) {
        const int64_t lim = i + (Lk - Lq) + 1;
        limit = lim < limit ? lim : limit;
      }
      // exp2-domain factor and natural scale of this row's scores; the e4m3 path folds
      // in the row's q scale and the KV head's k scale (S is a product of codes).
      float c = p.scale_log2, sc = p.scale;
      if constexpr (F8) {
        const float f =
            ((i >= 0 && i < Lq) ? p.q_scale[(w.q_start + i) * p.hq + w.h] : 1.f) * p.k_scale[w.g];
        c *= f;
        sc *= f;
      }
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < n_tiles; ++j) {
        const int gj = gt + j;
        // tcgen05.ld/st are warp-collective: leave the loop as a whole warp.
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bar_s[wg]), gj & 1, abort_flag,
                                                p.dev_status));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[128];
        float part_max[4];  // TMEM returns each 32-column chunk's max with the data
  #pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          part_max[q4] =
              tmem_ld32_max(S_row + q4 * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[q4 * 32]));
        tmem_ld_wait();
        float* s = reinterpret_cast<float*>(sr);
        const int64_t kv0 = (int64_t)j * kBlockN;
        float tile_max = fmaxf(fmax3(part_max[0], part_max[1], part_max[2]), part_max[3]);
        if (kv0 + kBlockN > limit) {  // masked columns must not count in the max
          const int64_t lim = limit - kv0;
  #pragma unroll
          for (int cc = 0; cc < 128; ++cc)
            if (cc >= lim) s[cc] = -INFINITY;
          tile_max = row_max<128>(s);
        }
        const float m_new = fmaxf(m_ref, tile_max);
        const bool resc = (m_new - m_ref) * c > 8.0f;  // false for -inf - -inf (NaN)
        float alpha = 1.f;
        if (resc) {
          alpha = ex2_approx((m_ref - m_new) * c);  // 0 when m_ref = -inf
          l *= alpha;
          m_ref = m_new;
        }
        const float neg_mc = (m_ref == -INFINITY) ? 0.f : -m_ref * c;
        // P packed as bf16 pairs in place (over sr[0..63], or sr[0..31] and sr[64..95]).
        if constexpr (D >= 128) {
          // Two halves: the first half of P goes to TMEM while the second is computed
          // (and fewer values stay live, which at d = 128 removes most spills).
          const float l_a = exp2_pack_sum<64>(sr, c, neg_mc);
          tmem_st32(S_row, *reinterpret_cast<const uint32_t(*)[32]>(&sr[0]));
          const float l_b = exp2_pack_sum<64>(sr + 64, c, neg_mc);
          tmem_st32(S_row + 32, *reinterpret_cast<const uint32_t(*)[32]>(&sr[64]));
          l += l_a + l_b;
        } else {
          l += exp2_pack_sum<128>(sr, c, neg_mc);
  #pragma unroll
          for (int q4 = 0; q4 < 2; ++q4)
            tmem_st32(S_row + q4 * 32, *reinterpret_cast<const uint32_t(*)[32]>(&sr[q4 * 32]));
        }
        // Rescale O (its previous PV finished: it was issued before this tile's S MMA,
        // whose completion this thread observed).
        if (j > 0 && __any_sync(0xFFFFFFFFu, resc)) {
  #pragma unroll
          for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t o[16];
            tmem_ld16(O_row + c0, o);
            tmem_ld_wait();
  #pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(O_row + c0, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&bar_p[wg]));
      }
      // ---- epilogue: out = O / l, lse = m * scale + ln l ----
      if (ok && n_tiles > 0)
        ok = __all_sync(0xFFFFFFFFu,
                        mbar_wait(smem_u32(&bar_o[wg]), nq & 1, abort_flag, p.dev_status));
      if (!ok) break;
      tc_fence_after();
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      // Rows leave TMEM one per thread; this warp's 4 KB staging slice turns them into
      // whole 128-byte row segments, so each store instruction writes full lines.
      const int64_t row0 = w.q_lo + wg * kBlockM + (warp & 3) * 32;  // this warp's first row
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        constexpr int kW = 32;
        const int cw = (D - c0 < kW) ? D - c0 : kW;  // 32, or 16 for the d = 80 tail
        uint32_t o[32];
        if (n_tiles > 0) {
          if (cw == 32) {
            tmem_ld32(O_row + c0, o);
          } else {
            tmem_ld16(O_row + c0, *reinterpret_cast<uint32_t(*)[16]>(&o[0]));
          }
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) o[q] = 0u;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < cw / 4)
            stage[lane * 8 + (q ^ (lane & 7))] = make_float4(
                __uint_as_float(o[4 * q]) * inv_l, __uint_as_float(o[4 * q + 1]) * inv_l,
                __uint_as_float(o[4 * q + 2]) * inv_l, __uint_as_float(o[4 * q + 3]) * inv_l);
        __syncwarp();
        const int lpr = cw / 4;  // lanes per row segment
        for (int rr = 0; rr < 32; rr += 32 / lpr) {
          const int r = rr + lane / lpr, q = lane % lpr;
          const float4 v = stage[r * 8 + (q ^ (r & 7))];
          const int64_t ii = row0 + r;
          if (ii >= 0 && ii < Lq)
            *reinterpret_cast<float4*>(p.out + ((w.q_start + ii) * p.hq + w.h) * (int64_t)D +
                                       c0 + 4 * q) = v;
        }
        __syncwarp();
      }
      if (i >= 0 && i < Lq && p.lse != nullptr)
        p.lse[(w.q_start + i) * p.hq + w.h] =
            (l > 0.f) ? m_ref * sc + log2f(l) * 0.69314718055994531f : -INFINITY;
      gt += n_tiles;
      if (n_tiles > 0) ++nq;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

__global__ void f32_to_bf16_kernel(const float4* __restrict__ in, uint2* __restrict__ out,
                                   int64_t n4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = in[i];
    out[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

template <int D, bool F8 = false>
cudaError_t launch_d(const AttnArgs& a, int* drv_err, cudaStream_t stream) {
  using C = AttnCfg<D, F8>;
  AttnMaps maps;
  // es: bytes per value (2: bf16, 1: e4m3 q / k)
  auto make = [&](CUtensorMap* m, const void* base, int64_t tokens, int heads, uint32_t box0,
                  CUtensorMapSwizzle sw, int es = 2) -> bool {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)heads, (uint64_t)tokens};
    const uint64_t strides[2] = {(uint64_t)D * es, (uint64_t)heads * D * es};
    const uint32_t box[3] = {box0, 1, (uint32_t)kBlockN};
    CUresult r = encode_tensor_map(
        m, es == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
        const_cast<void*>(base), dims, strides, box, sw);
    if (r != CUDA_SUCCESS) {
      *drv_err = (int)r;
      return false;
    }
    return true;
  };
  const int64_t tq = a.total_q > 0 ? a.total_q : 1, tk = a.total_k > 0 ? a.total_k : 1;
  constexpr int qk_es = F8 ? 1 : 2;
  if (!make(&maps.q, a.q, tq, a.hq, C::kQKCols, CU_TENSOR_MAP_SWIZZLE_128B, qk_es) ||
      !make(&maps.k, a.k, tk, a.hkv, C::kQKCols, CU_TENSOR_MAP_SWIZZLE_128B, qk_es) ||
      !make(&maps.v, a.v, tk, a.hkv, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if constexpr (C::kTail != 0) {
    if (!make(&maps.q_t, a.q, tq, a.hq, 16, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make(&maps.k_t, a.k, tk, a.hkv, 16, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make(&maps.v_t, a.v, tk, a.hkv, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  } else {
    maps.q_t = maps.q;
    maps.k_t = maps.k;
    maps.v_t = maps.v;
  }
  AttnParams p;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.out = a.out;
  p.lse = a.lse;
  p.dev_status = a.dev_status;
  p.total_q = a.total_q;
  p.total_k = a.total_k;
  p.batch = a.batch;
  p.max_seqlen_q = a.max_seqlen_q;
  p.max_seqlen_k = a.max_seqlen_k;
  p.hq = a.hq;
  p.hkv = a.hkv;
  p.causal = a.causal;
  p.pairs_max = (a.max_seqlen_q + 2 * kBlockM - 1) / (2 * kBlockM);
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.q_scale = a.q_scale;
  p.k_scale = a.k_scale;
  const int64_t items = (int64_t)a.batch * p.pairs_max * a.hq;
  if (items == 0) return cudaSuccess;
  if (items > 0x7FFFFFFF || a.work_counter == nullptr) return cudaErrorInvalidConfiguration;
  p.work_counter = a.work_counter;
  p.n_items = (int)items;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // One persistent CTA per SM (the kernel's shared memory and TMEM allow one).
  const int grid = (int)(items < sms ? items : sms);
  e = cudaFuncSetAttribute(attn_fwd_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(a.work_counter, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<D, F8><<<grid, kAttnThreads, C::kSmemBytes, stream>>>(maps, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnArgs& a, int* drv_err, cudaStream_t stream) {
  switch (a.d) {
    case 64: return a.fp8 ? cudaErrorInvalidValue : launch_d<64>(a, drv_err, stream);
    case 80: return a.fp8 ? cudaErrorInvalidValue : launch_d<80>(a, drv_err, stream);
    case 128: return a.fp8 ? launch_d<128, true>(a, drv_err, stream)
                           : launch_d<128>(a, drv_err, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_f32_to_bf16(const float* in, void* out, int64_t n, cudaStream_t stream) {
  // n is a multiple of 4 (head_dim is), pointers 16 / 8-byte aligned.
  const int64_t n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  int blocks = (int)((n4 + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  f32_to_bf16_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(in),
                                                  reinterpret_cast<uint2*>(out), n4);
  return cudaGetLastError();
}

}  // namespace tts
