// FP8 (e4m3) block quantization of the prefill's q and k, the input side of the FP8
// QK^T product ("从 SGLang Kernel源码到 GPU Trace", section 3.2: part of the prefill
// runs in FP8; "AMD MI250部署DeepSeek-V4-Flash", section 4.1: matmul inputs may be FP8
// with FP32 accumulation, section 5.3: FP8 by block quantization).
//
// q [Tq, Hq, d] bf16: one block per (token, head) row of d values.
// k [Tk, Hkv, d] bf16: one block per KV head, over every token.
// scale = (block's max |x|) / 448 in fp32 (1 for an all-zero block); code =
// e4m3(x / scale): the division in fp32 (IEEE, round to nearest), the conversion to
// nearest with ties to even, saturating at +-448.
//
// k's per-head maximum is reduced with integer atomicMax on the bits of |x| (for
// non-negative floats the bit patterns order like the values), so the result does
// not depend on the order of the atomics. The k_scale array holds those bits until
// the last launch turns them into scales.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace tts {
namespace {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t x0 = __nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3);
  const uint32_t x1 = __nv_cvt_float_to_fp8(b, __NV_SATFINITE, __NV_E4M3);
  const uint32_t x2 = __nv_cvt_float_to_fp8(c, __NV_SATFINITE, __NV_E4M3);
  const uint32_t x3 = __nv_cvt_float_to_fp8(d, __NV_SATFINITE, __NV_E4M3);
  return x0 | (x1 << 8) | (x2 << 16) | (x3 << 24);
}

__device__ __forceinline__ float4 load_bf16x4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
}

// One warp per row of d values (d a multiple of 4): row maximum, its scale, the codes.
// Without head_amax the row's own scale is computed and written to row_scale; with it
// the scale comes from the per-head maximum bits in head_amax[row % heads].
__global__ void quant_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int d,
                                  uint8_t* __restrict__ codes, float* __restrict__ row_scale,
                                  const uint32_t* __restrict__ head_amax, int heads) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5);
       r < rows; r += warps) {
    const __nv_bfloat16* xr = x + r * d;
    float s;
    if (head_amax == nullptr) {
      float amax = 0.f;
      for (int c = lane * 4; c < d; c += 128) {
        const float4 v = load_bf16x4(xr + c);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      s = amax > 0.f ? amax / 448.0f : 1.0f;
      if (lane == 0) row_scale[r] = s;
    } else {
      const float amax = __uint_as_float(head_amax[r % heads]);
      s = amax > 0.f ? amax / 448.0f : 1.0f;
    }
    for (int c = lane * 4; c < d; c += 128) {
      const float4 v = load_bf16x4(xr + c);
      *reinterpret_cast<uint32_t*>(codes + r * d + c) = e4m3x4(v.x / s, v.y / s, v.z / s, v.w / s);
    }
  }
}

// d = 128: half a warp per row (8 values, 16 bytes per lane), four rows per half-warp
// loaded before any arithmetic, so a warp keeps 2 KB of loads in flight (the one-warp-
// per-row loop above keeps 256 bytes). The same scales and codes as quant_rows_kernel.
constexpr int kFastRows = 4;
__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    f[2 * i] = __low2float(b);
    f[2 * i + 1] = __high2float(b);
  }
}
__global__ void quant_rows128_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                     uint8_t* __restrict__ codes, float* __restrict__ row_scale,
                                     const uint32_t* __restrict__ head_amax, int heads) {
  const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t warp_id = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5);
  // The loop bound is the warp's (both halves run every iteration, so the shuffles
  // always see all 32 lanes); rows past the end are masked.
  for (int64_t wb = warp_id * 2 * kFastRows; wb < rows; wb += nwarps * 2 * kFastRows) {
    const int64_t rb = wb + half * kFastRows;
    uint4 u[kFastRows];
#pragma unroll
    for (int j = 0; j < kFastRows; ++j) {
      const int64_t r = rb + j;
      u[j] = r < rows ? *reinterpret_cast<const uint4*>(x + r * 128 + hl * 8)
                      : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kFastRows; ++j) {
      const int64_t r = rb + j;
      float f[8];
      bf16x8_to_f32(u[j], f);
      float s;
      if (head_amax == nullptr) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        s = amax > 0.f ? amax / 448.0f : 1.0f;
        if (hl == 0 && r < rows) row_scale[r] = s;
      } else {
        const float amax = r < rows ? __uint_as_float(head_amax[r % heads]) : 0.f;
        s = amax > 0.f ? amax / 448.0f : 1.0f;
      }
      if (r < rows)
        *reinterpret_cast<uint2*>(codes + r * 128 + hl * 8) =
            make_uint2(e4m3x4(f[0] / s, f[1] / s, f[2] / s, f[3] / s),
                       e4m3x4(f[4] / s, f[5] / s, f[6] / s, f[7] / s));
    }
  }
}

// Per-head max |x| of k [rows = tokens * heads, d]: each block reduces its rows per
// head in shared memory, then one integer atomicMax per head and block.
__global__ void head_amax_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int d,
                                 int heads, uint32_t* __restrict__ head_amax) {
  extern __shared__ uint32_t s_amax[];  // [heads]
  for (int h = threadIdx.x; h < heads; h += blockDim.x) s_amax[h] = 0u;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5);
       r < rows; r += warps) {
    const __nv_bfloat16* xr = x + r * d;
    float amax = 0.f;
    for (int c = lane * 4; c < d; c += 128) {
      const float4 v = load_bf16x4(xr + c);
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (lane == 0) atomicMax(&s_amax[r % heads], __float_as_uint(amax));
  }
  __syncthreads();
  for (int h = threadIdx.x; h < heads; h += blockDim.x)
    if (s_amax[h] != 0u) atomicMax(&head_amax[h], s_amax[h]);
}

// d = 128: the same per-head maxima with half a warp per row and four rows per half-warp
// in flight (the layout of quant_rows128_kernel).
__global__ void head_amax128_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                    int heads, uint32_t* __restrict__ head_amax) {
  extern __shared__ uint32_t s_amax[];  // [heads]
  for (int h = threadIdx.x; h < heads; h += blockDim.x) s_amax[h] = 0u;
  __syncthreads();
  const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t warp_id = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5);
  for (int64_t wb = warp_id * 2 * kFastRows; wb < rows; wb += nwarps * 2 * kFastRows) {
    const int64_t rb = wb + half * kFastRows;
    uint4 u[kFastRows];
#pragma unroll
    for (int j = 0; j < kFastRows; ++j) {
      const int64_t r = rb + j;
      u[j] = r < rows ? *reinterpret_cast<const uint4*>(x + r * 128 + hl * 8)
                      : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kFastRows; ++j) {
      float f[8];
      bf16x8_to_f32(u[j], f);
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      const int64_t r = rb + j;
      if (hl == 0 && r < rows) atomicMax(&s_amax[r % heads], __float_as_uint(amax));
    }
  }
  __syncthreads();
  for (int h = threadIdx.x; h < heads; h += blockDim.x)
    if (s_amax[h] != 0u) atomicMax(&head_amax[h], s_amax[h]);
}

// The per-head maximum bits become the per-head scales.
__global__ void head_scale_kernel(float* k_scale, int heads) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h < heads) {
    const float amax = __uint_as_float(reinterpret_cast<const uint32_t*>(k_scale)[h]);
    k_scale[h] = amax > 0.f ? amax / 448.0f : 1.0f;
  }
}

int row_blocks(int64_t rows) {
  int64_t b = (rows + (kQuantThreads / 32) - 1) / (kQuantThreads / 32);
  if (b > 152 * 8) b = 152 * 8;
  return static_cast<int>(b < 1 ? 1 : b);
}
int row128_blocks(int64_t rows) {
  const int64_t per_block = (kQuantThreads / 32) * 2 * kFastRows;  // rows per block and pass
  int64_t b = (rows + per_block - 1) / per_block;
  if (b > 152 * 8) b = 152 * 8;
  return static_cast<int>(b < 1 ? 1 : b);
}

cudaError_t quant_rows(const void* x, int64_t rows, int d, void* codes, float* row_scale,
                       const uint32_t* head_amax, int heads, cudaStream_t stream) {
  if (d == 128)
    quant_rows128_kernel<<<row128_blocks(rows), kQuantThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(x), rows, static_cast<uint8_t*>(codes), row_scale,
        head_amax, heads);
  else
    quant_rows_kernel<<<row_blocks(rows), kQuantThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(x), rows, d, static_cast<uint8_t*>(codes), row_scale,
        head_amax, heads);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_fp8_prefill(const void* q, int64_t total_q, int hq, const void* k,
                                     int64_t total_k, int hkv, int d, void* q8, float* q_scale,
                                     void* k8, float* k_scale, cudaStream_t stream) {
  const int64_t qrows = total_q * hq, krows = total_k * hkv;
  if (qrows > 0) {
    const cudaError_t e = quant_rows(q, qrows, d, q8, q_scale, nullptr, 1, stream);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaMemsetAsync(k_scale, 0, sizeof(float) * hkv, stream);
  if (e != cudaSuccess) return e;
  uint32_t* amax = reinterpret_cast<uint32_t*>(k_scale);
  if (krows > 0) {
    if (d == 128)
      head_amax128_kernel<<<row128_blocks(krows), kQuantThreads, sizeof(uint32_t) * hkv,
                            stream>>>(static_cast<const __nv_bfloat16*>(k), krows, hkv, amax);
    else
      head_amax_kernel<<<row_blocks(krows), kQuantThreads, sizeof(uint32_t) * hkv, stream>>>(
          static_cast<const __nv_bfloat16*>(k), krows, d, hkv, amax);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = quant_rows(k, krows, d, k8, nullptr, amax, hkv, stream);
    if (e != cudaSuccess) return e;
  }
  head_scale_kernel<<<(hkv + 127) / 128, 128, 0, stream>>>(k_scale, hkv);
  return cudaGetLastError();
}

}  // namespace tts
