// Vision-encoder QKV projection fused with rotary position embedding, and the
// position-indexed cos/sin table it reads.
//
// What it computes ("DeepSeek V4.1 上 4×RTX 3090", 坑 1: the qkv + RoPE step of the
// vision encoder; "从 SGLang Kernel源码到 GPU Trace", section 3.3: cos/sin of every
// position precomputed once into a small cached table that the projection kernel
// reads): y = x W^T + bias for every token, split into q, k and v heads; every q
// and k head is turned pair by pair, pairs (j, j + d/2) by the angle
// pos * base^(-2j/d); v is written as projected. The pages leave the RoPE variant
// open; this one-dimensional rotate-half form is the reading taken.
//
// How: a persistent tcgen05 GEMM on CTA pairs (a cluster of two CTAs on two SMs).
// A pair computes a 256-token x BN tile with M = 256 MMAs (cta_group::2): each CTA
// stages its own 128 rows of x and half of the tile's BN rows of W, and the tensor
// cores of both SMs read both W halves, so every staged byte feeds twice the work
// of a one-SM tile. BN is whole heads (3 heads of 80, 4 of 64 or 2 of 128), so a
// row's rotation partner is always in the same thread's accumulator row and the
// rotation happens in the epilogue, between TMEM and the store -- y never goes to
// global memory unrotated, and no two threads ever write the same output element
// (the race of the vision write-up has no place to happen).
//   warp 0      TMA producer (both CTAs): x box 64 x 128 and W box 64 x BN/2,
//               128-byte swizzle, into a six-stage ring
//   warp 1      TMEM (512 columns, allocated by the pair together). Leader CTA:
//               MMA issuer -- waits until both CTAs' copies of a stage have landed,
//               D[tmem] += x W^T (kind::f16, bf16 operands, fp32 accumulators in
//               both SMs' TMEM), commits to the stage's empty barrier of both CTAs;
//               two accumulators (columns 0 / 256) so one tile's epilogue overlaps
//               the next tile's MMAs. The peer's copies count their bytes on the
//               leader's stage barrier directly (TMA with cta_group::2).
//   warps 2..5  epilogue (both CTAs), one token row per thread (TMEM lane = warp % 4):
//               + bias, rotation in fp32, bf16 rounding (nearest even), staged per
//               head in a 32-row shared-memory buffer per warp and written by TMA
//               stores (rows past the last token are clipped by the tensor map);
//               the accumulator is handed back to the leader's MMA warp by local /
//               remote arrives.
// Pair tiles go to pairs round-robin; every wait is bounded.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace tts {
namespace {

constexpr int kQkvThreads = 192;
constexpr int kBM = 128;  // tokens per CTA (256 per CTA pair)
constexpr int kBK = 64;   // hidden columns per stage (one 128-byte swizzle row)

template <int D>
struct QkvCfg {
  static constexpr int kHpt = (D == 80) ? 3 : 256 / D;  // heads per tile
  static constexpr int kBN = kHpt * D;                  // MMA N: 240 / 256 / 256
  static constexpr int kBNh = kBN / 2;                  // W rows staged by each CTA
  static constexpr int kStages = 6;
  static constexpr int kABytes = kBM * 128;
  static constexpr int kBBytes = kBNh * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kOutBytes = 32 * D * 2;  // one head of one warp's 32 rows, bf16
  static constexpr int kSmemBytes = kStages * kStageBytes + 4 * kOutBytes + 1024;
  static_assert(kBN % 16 == 0 && kBN <= 256 && kBNh % 8 == 0, "MMA N");
  static_assert(kStageBytes % 1024 == 0 && kABytes % 1024 == 0, "swizzle atoms");
  static_assert(kSmemBytes + 256 + kBN * 4 <= 232448, "shared memory");
};

struct QkvMaps {
  CUtensorMap x;       // {hidden, n} bf16, box {64, 128}, 128-byte swizzle
  CUtensorMap w;       // {hidden, 3 H D} bf16, box {64, BN/2}, 128-byte swizzle
  CUtensorMap out[3];  // q, k, v: {H D, n} bf16, box {D, 32}, no swizzle
};

struct QkvParams {
  const float* bias;      // [3 H D] or null
  const int32_t* pos;     // [n]
  const float2* cos_sin;  // [max_pos, D/2] (cos, sin)
  uint32_t* dev_status;
  int n, heads, max_pos, tiles_n, n_tiles, k_steps;  // n_tiles: 256-token pair tiles
};

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, uint32_t src, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
}
// Wait until no bulk group of this thread is still reading shared memory.
__device__ __forceinline__ void bulk_wait_read_0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// TMA tile load into this CTA's shared memory whose completion (bytes) is counted on an
// mbarrier of either CTA of the pair (`bar` a shared::cluster address, from mapa).
__device__ __forceinline__ void tma_load_2d_to_pair_bar(uint32_t dst, const CUtensorMap* m,
                                                        uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// ---- tcgen05 on a CTA pair (every tcgen05 instruction of the kernel uses cta_group::2)
// Allocation and release are collective: one warp of each CTA of the pair issues them.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D[tmem of both CTAs] (+)= A[smem of both CTAs: 128 rows each] * B[smem of both CTAs:
// N/2 rows each]^T, issued by the elected lane of the leader CTA's converged warp.
__device__ __forceinline__ void mma_pair_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate,
                                               uint32_t pred) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
      : "memory");
}
// Arrive once on the barrier at this shared-memory offset in every CTA of `mask` when
// all tcgen05 operations issued so far by this thread are complete.
__device__ __forceinline__ void commit_pair_mc_elect(uint32_t bar, uint16_t mask, uint32_t pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
      "@q tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(bar),
      "h"(mask), "r"(pred)
      : "memory");
}
// Barrier over every thread of both CTAs (release / acquire at cluster scope). The
// non-.aligned form, so lanes that reach it apart are fine.
__device__ __forceinline__ void pair_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Bounded wait with cluster-scope acquire, warp-collective (the result is the warp's AND).
__device__ __forceinline__ bool warp_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort,
                                             uint32_t* status) {
  const bool ok = mbar_wait<true>(bar, parity, abort, status);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Bounded wait that polls without suspending (cluster-scope acquire): for the producer
// and MMA warps, whose wake-up latency after a phase completes is on the tensor
// core's critical path. The clock is read once every 256 polls.
__device__ __forceinline__ bool mbar_peek_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool spin_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort,
                                             uint32_t* status) {
  if (mbar_peek_cl(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_peek_cl(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        if (status != nullptr) atomicOr(status, kDevTimeout);
        *abort = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool warp_spin_cl(uint32_t bar, uint32_t parity, volatile int* abort,
                                             uint32_t* status) {
  const bool ok = spin_wait_cl(bar, parity, abort, status);
  return __all_sync(0xFFFFFFFFu, ok);
}

template <int D>
__global__ void __launch_bounds__(kQkvThreads, 1)
    qkv_rope_kernel(const __grid_constant__ QkvMaps maps, const QkvParams p) {
  using C = QkvCfg<D>;
  constexpr int NS = C::kStages;
  constexpr int H2 = D / 2;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[NS], bar_empty[NS], bar_acc_full[2],
      bar_acc_empty[2], bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float4 s_bias[C::kBN / 4];  // the current tile's bias (epilogue)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();  // 0: leader (issues the MMAs), 1: peer
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  auto sA = [&](int st) { return s_base + st * C::kStageBytes; };
  auto sB = [&](int st) { return s_base + st * C::kStageBytes + C::kABytes; };
  uint8_t* out_base = smem + NS * C::kStageBytes;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bar_full[i]), 1);        // leader: both CTAs' copies of a stage
      mbar_init(smem_u32(&bar_empty[i]), 1);       // the leader's commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_acc_full[i]), 1);    // the leader's commit
      mbar_init(smem_u32(&bar_acc_empty[i]), 8);   // leader: 4 epilogue warps per CTA
    }
    mbar_init(smem_u32(&bar_drain), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&s_tmem), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  pair_sync();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&maps.x);
      prefetch_tmap(&maps.w);
      // Both CTAs' copies of a stage count on the leader's full barrier, which the
      // leader arms with the pair's bytes; the peer's copies land there directly.
      const uint32_t full0 = mapa_shared(smem_u32(&bar_full[0]), 0);
      int g = 0;  // stages filled so far (ring position and phase)
      bool ok = true;
      for (int t = pair; ok && t < p.n_tiles; t += n_pairs) {
        const int tm = t / p.tiles_n, tn = t % p.tiles_n;
        const int arow = tm * 2 * kBM + static_cast<int>(rank) * kBM;
        const int brow = tn * C::kBN + static_cast<int>(rank) * C::kBNh;
        for (int ks = 0; ks < p.k_steps; ++ks, ++g) {
          const int st = g % NS;
          if (g >= NS && !spin_wait_cl(smem_u32(&bar_empty[st]), ((g / NS) - 1) & 1,
                                       abort_flag, p.dev_status)) {
            ok = false;
            break;
          }
          if (rank == 0) {
            const uint32_t bf = smem_u32(&bar_full[st]);
            mbar_arrive_expect_tx(bf, 2 * C::kStageBytes);
            tma_load_2d(sA(st), &maps.x, bf, ks * kBK, arow);
            tma_load_2d(sB(st), &maps.w, bf, ks * kBK, brow);
          } else {
            const uint32_t bf = full0 + st * 8;
            tma_load_2d_to_pair_bar(sA(st), &maps.x, bf, ks * kBK, arow);
            tma_load_2d_to_pair_bar(sB(st), &maps.w, bf, ks * kBK, brow);
          }
        }
      }
      if (!ok && rank == 0) {
        // Best-effort drain: the latest armed phase of each stage is the only one
        // that can still have copies (of either CTA) in flight.
        for (int j = g - 1; j >= 0 && j >= g - NS; --j)
          mbar_wait(smem_u32(&bar_full[j % NS]), (j / NS) & 1, nullptr, nullptr);
      }
    }
  } else if (warp == 1 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer (leader)
    const uint32_t e = elect_one();
    constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, C::kBN, 0, 0);
    int g = 0, i = 0;
    bool ok = true;
    for (int t = pair; ok && t < p.n_tiles; t += n_pairs, ++i) {
      const int a = i & 1;
      if (i >= 2 && !warp_spin_cl(smem_u32(&bar_acc_empty[a]), ((i >> 1) - 1) & 1, abort_flag,
                                  p.dev_status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + a * 256;
      for (int ks = 0; ks < p.k_steps; ++ks, ++g) {
        const int st = g % NS;
        const uint32_t ph = (g / NS) & 1;
        if (!warp_spin_cl(smem_u32(&bar_full[st]), ph, abort_flag, p.dev_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = smem_desc(sA(st), 16, 1024, kSw128);
        const uint64_t bd = smem_desc(sB(st), 16, 1024, kSw128);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)  // 32-byte steps inside the swizzle row
          mma_pair_elect(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (ks | kk) != 0, e);
        commit_pair_mc_elect(smem_u32(&bar_empty[st]), 0x3, e);
      }
      if (!ok) break;
      commit_pair_mc_elect(smem_u32(&bar_acc_full[a]), 0x3, e);
    }
    // Every MMA issued by this warp completes before the pair frees TMEM.
    commit_pair_mc_elect(smem_u32(&bar_drain), 0x1, e);
    mbar_wait(smem_u32(&bar_drain), 0, nullptr, p.dev_status);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;  // TMEM lane quarter = rows q4*32 .. q4*32+31 of this CTA
    const int et = tid - 64;  // 0 .. 127 over the four epilogue warps
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    uint8_t* obuf = out_base + (warp - 2) * C::kOutBytes;  // this warp's staging buffer
    const uint32_t acc_empty0 = mapa_shared(smem_u32(&bar_acc_empty[0]), 0);  // leader's
    bool ok = true;
    int i = 0;
    // Every epilogue warp runs every iteration (both named barriers included), also
    // after a wait gave up, so the barriers always see all 128 threads.
    for (int t = pair; t < p.n_tiles; t += n_pairs, ++i) {
      const int a = i & 1;
      const int tm = t / p.tiles_n, tn = t % p.tiles_n;
      const int row0 = tm * 2 * kBM + static_cast<int>(rank) * kBM + q4 * 32;  // warp's first
      const int row = row0 + lane;
      // A warp whose 32 rows all lie past the last token only frees the accumulator.
      const bool live = row0 < p.n;
      const int hh0 = tn * C::kHpt;  // first head column of the tile, in [0, 3H)
      const bool any_rot = hh0 < 2 * p.heads;
      // The tile's bias (BN values) goes to shared memory and the token's cos/sin row to
      // registers while the MMAs of the tile still run.
      named_barrier_sync(1, 128);  // every warp is done with the previous tile's bias
      for (int c = et; c < C::kBN / 4; c += 128)
        s_bias[c] = p.bias ? __ldg(reinterpret_cast<const float4*>(
                                       p.bias + static_cast<int64_t>(hh0) * D) + c)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      // Position of this thread's token; a position outside the table is reported,
      // and that token's q and k are written as zeros.
      int pos = 0;
      bool pos_ok = true;
      if (ok && live && row < p.n && any_rot) {
        pos = p.pos[row];
        pos_ok = pos >= 0 && pos < p.max_pos;
        if (!pos_ok) {
          if (p.dev_status) atomicOr(p.dev_status, kDevIndexRange);
          pos = 0;
        }
      }
      const float4* cs4 =
          reinterpret_cast<const float4*>(p.cos_sin + static_cast<int64_t>(pos) * H2);
      // d <= 80: the token's cos/sin row (d/2 pairs) is kept in registers for the tile.
      constexpr bool kCsRegs = D <= 80;
      float4 csr[kCsRegs ? H2 / 2 : 1];
      if constexpr (kCsRegs) {
        if (ok && live && any_rot) {
#pragma unroll
          for (int u = 0; u < H2 / 2; ++u) csr[u] = __ldg(cs4 + u);
        }
      }
      named_barrier_sync(1, 128);  // the bias is in shared memory
      ok = ok && warp_wait_cl(smem_u32(&bar_acc_full[a]), (i >> 1) & 1, abort_flag,
                              p.dev_status);
      if (!ok) continue;
      tc_fence_after();
#pragma unroll 1
      for (int hl = 0; hl < C::kHpt; ++hl) {
        const int hh = hh0 + hl;
        const int part = hh / p.heads, head = hh - part * p.heads;
        const bool rot = part < 2;
        const float4* b4 = s_bias + hl * (D / 4);
        const uint32_t tcol = lane_base + a * 256 + hl * D;
        uint8_t* myrow = obuf + lane * (D * 2);
        if (live) {
          uint4 packed[D / 8];  // the head's D bf16 results, written after the wait below
          uint32_t r[D];  // the head's D accumulator columns of this row, one round trip
#pragma unroll
          for (int c = 0; c < D; c += 8)
            tmem_ld8(tcol + c, *reinterpret_cast<uint32_t(*)[8]>(&r[c]));
          tmem_ld_wait();
#pragma unroll
          for (int j0 = 0; j0 < H2; j0 += 8) {
            float ylo[8], yhi[8];
            const float4 b0 = b4[j0 / 4], b1 = b4[j0 / 4 + 1];
            const float4 c0 = b4[(H2 + j0) / 4], c1 = b4[(H2 + j0) / 4 + 1];
            const float bl[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
            const float bh[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              ylo[u] = __uint_as_float(r[j0 + u]) + bl[u];
              yhi[u] = __uint_as_float(r[H2 + j0 + u]) + bh[u];
            }
            if (rot) {
              float cs[16];  // (cos, sin) of pairs j0 .. j0+7
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float4 v = kCsRegs ? csr[(j0 / 2 + u) % (kCsRegs ? H2 / 2 : 1)]
                                         : __ldg(cs4 + j0 / 2 + u);
                cs[4 * u] = v.x;
                cs[4 * u + 1] = v.y;
                cs[4 * u + 2] = v.z;
                cs[4 * u + 3] = v.w;
              }
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const float c = pos_ok ? cs[2 * u] : 0.f, s = pos_ok ? cs[2 * u + 1] : 0.f;
                const float a0 = ylo[u], b0 = yhi[u];
                ylo[u] = fmaf(a0, c, -b0 * s);
                yhi[u] = fmaf(a0, s, b0 * c);
              }
            }
            uint4 plo, phi;
            plo.x = pack_bf16x2(ylo[0], ylo[1]);
            plo.y = pack_bf16x2(ylo[2], ylo[3]);
            plo.z = pack_bf16x2(ylo[4], ylo[5]);
            plo.w = pack_bf16x2(ylo[6], ylo[7]);
            phi.x = pack_bf16x2(yhi[0], yhi[1]);
            phi.y = pack_bf16x2(yhi[2], yhi[3]);
            phi.z = pack_bf16x2(yhi[4], yhi[5]);
            phi.w = pack_bf16x2(yhi[6], yhi[7]);
            packed[j0 / 8] = plo;
            packed[(H2 + j0) / 8] = phi;
          }
          // The previous head's store must be done reading the staging buffer; it was
          // issued before this head's TMEM loads and arithmetic, which hide most of it.
          if (lane == 0) bulk_wait_read_0();
          __syncwarp();
#pragma unroll
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(myrow)[c] = packed[c];
        }
        if (hl == C::kHpt - 1) {
          // Every TMEM read of this accumulator is done: hand it back to the leader.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (rank == 0)
              mbar_arrive(smem_u32(&bar_acc_empty[a]));
            else
              mbar_arrive_remote(acc_empty0 + a * 8);
          }
        }
        if (live) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&maps.out[part], smem_u32(obuf), head * D, row0);
            bulk_commit();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_read_all();  // staging stays until every store has read it
  }

  // Neither CTA leaves (or frees TMEM) while its peer may still read its shared memory,
  // arrive on its barriers or read TMEM.
  tc_fence_before();
  __syncwarp();
  pair_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// Co-resident CTA pairs of qkv_rope_kernel<D> on the current device (cached per device).
template <int D>
int max_pairs(int dev, const cudaLaunchConfig_t& cfg) {
  // Host threads may make their first calls at the same time: every thread that finds
  // the slot empty computes the same value, and the slot is read and written atomically.
  static std::atomic<int> cache[64];
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, qkv_rope_kernel<D>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    n = sms / 2 > 0 ? sms / 2 : 1;
  }
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int D>
cudaError_t launch_qkv_d(const QkvArgs& a, int* drv_err, cudaStream_t stream) {
  using C = QkvCfg<D>;
  QkvMaps maps;
  const uint64_t n = static_cast<uint64_t>(a.n);
  const uint64_t hidden = static_cast<uint64_t>(a.hidden);
  const uint64_t cols = 3ull * a.heads * D;
  auto make = [&](CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box0,
                  uint32_t box1, CUtensorMapSwizzle sw) -> bool {
    const uint64_t dims[2] = {inner, outer};
    const uint64_t strides[1] = {inner * 2};
    const uint32_t box[2] = {box0, box1};
    CUresult r = encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                   const_cast<void*>(base), dims, strides, box, sw);
    if (r != CUDA_SUCCESS) {
      *drv_err = static_cast<int>(r);
      return false;
    }
    return true;
  };
  if (!make(&maps.x, a.x, hidden, n, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make(&maps.w, a.w, hidden, cols, kBK, C::kBNh, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make(&maps.out[0], a.q, (uint64_t)a.heads * D, n, D, 32, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make(&maps.out[1], a.k, (uint64_t)a.heads * D, n, D, 32, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make(&maps.out[2], a.v, (uint64_t)a.heads * D, n, D, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  QkvParams p;
  p.bias = a.bias;
  p.pos = a.positions;
  p.cos_sin = reinterpret_cast<const float2*>(a.cos_sin);
  p.dev_status = a.dev_status;
  p.n = static_cast<int>(a.n);
  p.heads = a.heads;
  p.max_pos = a.max_pos;
  p.tiles_n = static_cast<int>(cols / C::kBN);
  const int64_t tiles_m = (a.n + 2 * kBM - 1) / (2 * kBM);
  const int64_t n_tiles = tiles_m * p.tiles_n;
  if (n_tiles > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  p.n_tiles = static_cast<int>(n_tiles);
  p.k_steps = (a.hidden + kBK - 1) / kBK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(qkv_rope_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kQkvThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2, 1, 1);
  const int pairs_max = max_pairs<D>(dev, cfg);
  const int pairs = static_cast<int>(n_tiles < pairs_max ? n_tiles : pairs_max);
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  e = cudaLaunchKernelEx(&cfg, qkv_rope_kernel<D>, maps, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The cos/sin table: pair j of position p turns by p * base^(-2j/rot_dim). The angle
// and its sine and cosine are taken in double precision and rounded to fp32 once.
__global__ void rope_cache_kernel(float2* __restrict__ out, int max_pos, int rot_dim,
                                  double base) {
  const int half = rot_dim / 2;
  const int64_t total = static_cast<int64_t>(max_pos) * half;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(i / half), j = static_cast<int>(i % half);
    const double inv_freq = pow(base, -2.0 * j / rot_dim);
    double s, c;
    sincos(static_cast<double>(pos) * inv_freq, &s, &c);
    out[i] = make_float2(static_cast<float>(c), static_cast<float>(s));
  }
}

}  // namespace

int qkv_heads_per_tile(int head_dim) {
  switch (head_dim) {
    case 64: return QkvCfg<64>::kHpt;
    case 80: return QkvCfg<80>::kHpt;
    case 128: return QkvCfg<128>::kHpt;
    default: return 0;
  }
}

cudaError_t launch_qkv_rope(const QkvArgs& a, int* drv_err, cudaStream_t stream) {
  switch (a.head_dim) {
    case 64: return launch_qkv_d<64>(a, drv_err, stream);
    case 80: return launch_qkv_d<80>(a, drv_err, stream);
    case 128: return launch_qkv_d<128>(a, drv_err, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rope_cache(int max_pos, int rot_dim, double base, float* cos_sin,
                              cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(max_pos) * (rot_dim / 2);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  rope_cache_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
      reinterpret_cast<float2*>(cos_sin), max_pos, rot_dim, base);
  return cudaGetLastError();
}

}  // namespace tts
