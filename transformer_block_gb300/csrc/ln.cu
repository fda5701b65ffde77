// ln.cu — LayerNorm of the token rows (the single LN shared by both branches of the
// parallel block, MegaScale reading notes, section 1.1, eq. (4)).
//
// Each thread keeps its share of the row in registers as vectors of 8 elements (one
// 128-bit load of bf16, or two of fp32 for the fp32 residual stream of a stack), so x is
// read from HBM once. The mean and then the centred variance are reduced in fp32, and the
// normalised, affine-mapped row is written back as bf16 or fp16 (round to nearest even).
// HBM-bound: one read and one write of the row. Three shapes of work:
//   * rows up to 4096 bf16 (2048 fp32) elements: one warp per row, 8 rows per CTA,
//     reductions by warp shuffles only (layernorm_rows_kernel, 1 warp per row);
//   * up to 16384 bf16 (8192 fp32): four warps per row, 2 rows per CTA, the warps' partial
//     sums through shared memory (layernorm_rows_kernel, 4 warps per row); each thread
//     holds only as many vectors as the row needs (4, 6, 8, 12 or 16), and with 12 or fewer
//     three CTAs fit per SM, so more rows are in flight on the few-row workloads;
//   * longer fp32 rows: one 256-thread CTA per row, CTA-wide reductions
//     (layernorm_kernel). The FP8 variant (layernorm_e4m3_kernel) uses this shape for all
//     rows.
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace pb {
namespace {

constexpr int THREADS = 256;
// vectors of 8 elements per thread in the one-CTA-per-row kernels (rows up to kLnMaxH)
constexpr int MAXV = kLnMaxH / (8 * THREADS);

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < THREADS / 32; ++w) s += red[w];
  __syncthreads();
  return s;
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float m = 0.f;
#pragma unroll
  for (int w = 0; w < THREADS / 32; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  return m;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* row, int idx, float (&f)[8]) {
  const uint4 u = reinterpret_cast<const uint4*>(row)[idx];
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
    f[2 * e] = p.x;
    f[2 * e + 1] = p.y;
  }
}

__device__ __forceinline__ void load8(const float* row, int idx, float (&f)[8]) {
  const float4 a = reinterpret_cast<const float4*>(row)[2 * idx];
  const float4 b = reinterpret_cast<const float4*>(row)[2 * idx + 1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if (F16) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// RMS: RMSNorm, x / sqrt(mean x^2 + eps) * gamma (no centring, no beta).
template <typename TIn, bool F16, bool RMS>
__global__ void __launch_bounds__(THREADS) layernorm_kernel(const TIn* __restrict__ x,
                                                            const __nv_bfloat16* __restrict__ gamma,
                                                            const __nv_bfloat16* __restrict__ beta,
                                                            uint4* __restrict__ out, int H,
                                                            float eps, int* status) {
  __shared__ float red[THREADS / 32];
  const int nv = H / 8;
  const int64_t row = blockIdx.x;
  const TIn* xr = x + row * H;
  float v[MAXV][8];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
      load8(xr, idx, v[i]);
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += v[i][e];
    }
  }
  const float mean = RMS ? 0.f : block_sum(sum, red) / float(H);
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sq += (v[i][e] - mean) * (v[i][e] - mean);
    }
  }
  const float var = block_sum(sq, red) / float(H);
  const float rstd = rsqrtf(var + eps);
  uint4* orow = out + row * nv;
  bool out_of_range = false;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
      float g[8], b[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, o[8];
      load8(gamma, idx, g);
      if (!RMS) load8(beta, idx, b);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        o[e] = (v[i][e] - mean) * rstd * g[e] + b[e];
        if (F16) out_of_range |= !(fabsf(o[e]) <= kF16Max);
      }
      uint4 u;
      u.x = pack2<F16>(o[0], o[1]);
      u.y = pack2<F16>(o[2], o[3]);
      u.z = pack2<F16>(o[4], o[5]);
      u.w = pack2<F16>(o[6], o[7]);
      orow[idx] = u;
    }
  }
  if (F16 && out_of_range && status != nullptr) atomicCAS(status, 0, kStatusRange);
}

// Rows that fit the registers of one or four warps: the mean and the variance need only
// warp shuffles (and, for four warps, one exchange through shared memory), and each SM
// keeps many rows' loads in flight. Thread t of a row holds vectors t, t + 32 WPR, ...
// (VPL of them) of 8 elements as loaded (bf16 stays packed) and converts them on each of
// the three passes.
template <typename TIn>
struct RowVec;
template <>
struct RowVec<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* row, int idx) {
    u = reinterpret_cast<const uint4*>(row)[idx];
  }
  // A bf16 is the top half of its fp32 value. The shifts are volatile so that each pass
  // converts again instead of the compiler keeping all fp32 values live (spills).
  __device__ __forceinline__ void get(float (&f)[8]) const {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t lo, hi;
      asm volatile("shl.b32 %0, %1, 16;" : "=r"(lo) : "r"(w[e]));
      asm volatile("and.b32 %0, %1, 0xffff0000;" : "=r"(hi) : "r"(w[e]));
      f[2 * e] = __uint_as_float(lo);
      f[2 * e + 1] = __uint_as_float(hi);
    }
  }
};
template <>
struct RowVec<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* row, int idx) {
    a = reinterpret_cast<const float4*>(row)[2 * idx];
    b = reinterpret_cast<const float4*>(row)[2 * idx + 1];
  }
  __device__ __forceinline__ void get(float (&f)[8]) const {
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the WPR warps of one row: warp shuffles, then (WPR > 1) the warps' partial sums
// through shared memory behind the row's own named barrier. `slot` separates the two
// reductions of a row, so no slot is written twice.
template <int WPR>
__device__ __forceinline__ float row_sum(float v, float* red, int slot) {
  v = warp_sum(v);
  if (WPR == 1) return v;
  const int warp = threadIdx.x >> 5, grp = warp / WPR;
  if ((threadIdx.x & 31) == 0) red[slot * (THREADS / 32) + warp] = v;
  named_barrier(1 + grp, 32 * WPR);
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < WPR; ++w) s += red[slot * (THREADS / 32) + grp * WPR + w];
  return s;
}

// WPR warps per row (1 or 4), THREADS / (32 WPR) rows per CTA. Every thread of a row's
// warps takes the same branches around the named barriers (the early exit depends only on
// the row).
template <typename TIn, bool F16, bool RMS, int VPL, int WPR>
__global__ void __launch_bounds__(THREADS, (WPR == 4 && VPL <= 12) ? 3 : 2) layernorm_rows_kernel(
    const TIn* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
    const __nv_bfloat16* __restrict__ beta, uint4* __restrict__ out, int64_t rows, int H,
    float eps, int* status) {
  __shared__ float red[2 * (THREADS / 32)];
  constexpr int RT = 32 * WPR;  // threads per row
  const int t = int(threadIdx.x) % RT;
  const int64_t row = int64_t(blockIdx.x) * (THREADS / RT) + int(threadIdx.x) / RT;
  if (row >= rows) return;
  const int nv = H / 8;
  const TIn* xr = x + row * H;
  RowVec<TIn> v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int idx = t + RT * i;
    if (idx < nv) v[i].load(xr, idx);
  }
  float sum = 0.f;
  if (!RMS) {
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      if (t + RT * i < nv) {
        float f[8];
        v[i].get(f);
#pragma unroll
        for (int e = 0; e < 8; ++e) sum += f[e];
      }
    }
  }
  const float mean = RMS ? 0.f : row_sum<WPR>(sum, red, 0) / float(H);
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    if (t + RT * i < nv) {
      float f[8];
      v[i].get(f);
#pragma unroll
      for (int e = 0; e < 8; ++e) sq += (f[e] - mean) * (f[e] - mean);
    }
  }
  const float rstd = rsqrtf(row_sum<WPR>(sq, red, 1) / float(H) + eps);
  uint4* orow = out + row * nv;
  bool out_of_range = false;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int idx = t + RT * i;
    if (idx < nv) {
      float f[8], g[8], b[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, o[8];
      v[i].get(f);
      load8(gamma, idx, g);
      if (!RMS) load8(beta, idx, b);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        o[e] = (f[e] - mean) * rstd * g[e] + b[e];
        if (F16) out_of_range |= !(fabsf(o[e]) <= kF16Max);
      }
      uint4 u;
      u.x = pack2<F16>(o[0], o[1]);
      u.y = pack2<F16>(o[2], o[3]);
      u.z = pack2<F16>(o[4], o[5]);
      u.w = pack2<F16>(o[6], o[7]);
      orow[idx] = u;
    }
  }
  if (F16 && out_of_range && status != nullptr) atomicCAS(status, 0, kStatusRange);
}

// LayerNorm / RMSNorm straight to FP8 E4M3 (the FP8 GEMM operand): the normalised row is
// computed in fp32 as above, its largest magnitude reduced across the CTA, and each value
// written as E4M3(o * 448 / amax), the row's scale amax / 448 to scales[row] (per-row
// current scaling, the steps of quant.cu).
template <typename TIn, bool RMS>
__global__ void __launch_bounds__(THREADS) layernorm_e4m3_kernel(
    const TIn* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
    const __nv_bfloat16* __restrict__ beta, uint2* __restrict__ out, float* __restrict__ scales,
    int H, float eps) {
  __shared__ float red[THREADS / 32];
  const int nv = H / 8;
  const int64_t row = blockIdx.x;
  const TIn* xr = x + row * H;
  float v[MAXV][8];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
      load8(xr, idx, v[i]);
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += v[i][e];
    }
  }
  const float mean = RMS ? 0.f : block_sum(sum, red) / float(H);
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sq += (v[i][e] - mean) * (v[i][e] - mean);
    }
  }
  const float rstd = rsqrtf(block_sum(sq, red) / float(H) + eps);
  // the normalised values replace x in registers
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
      float g[8], b[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      load8(gamma, idx, g);
      if (!RMS) load8(beta, idx, b);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[i][e] = (v[i][e] - mean) * rstd * g[e] + b[e];
        amax = fmaxf(amax, fabsf(v[i][e]));
      }
    }
  }
  amax = block_max(amax, red);
  const float inv = amax > 0.f ? 448.f / amax : 0.f;
  if (threadIdx.x == 0) scales[row] = amax / 448.f;
  uint2* orow = out + row * nv;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) orow[idx] = quant8_e4m3(v[i], inv);
  }
}

template <typename TIn, bool F16, int VPL, int WPR>
cudaError_t launch_rows(int64_t rows, int H, const void* x, const __nv_bfloat16* gamma,
                        const __nv_bfloat16* beta, float eps, void* out, int* status,
                        cudaStream_t stream) {
  constexpr int RPC = THREADS / (32 * WPR);  // rows per CTA
  const int64_t grid = (rows + RPC - 1) / RPC;
  if (beta == nullptr)
    layernorm_rows_kernel<TIn, F16, true, VPL, WPR><<<unsigned(grid), THREADS, 0, stream>>>(
        static_cast<const TIn*>(x), gamma, beta, static_cast<uint4*>(out), rows, H, eps, status);
  else
    layernorm_rows_kernel<TIn, F16, false, VPL, WPR><<<unsigned(grid), THREADS, 0, stream>>>(
        static_cast<const TIn*>(x), gamma, beta, static_cast<uint4*>(out), rows, H, eps, status);
  return cudaGetLastError();
}

// Vectors of 8 elements a thread of layernorm_rows_kernel may hold: 16 packed bf16 vectors
// (64 registers) or 8 fp32 vectors; so one warp covers rows up to 4096 bf16 / 2048 fp32
// elements and four warps up to 16384 / 8192.
template <typename TIn>
constexpr int kRowMaxVpl = sizeof(TIn) == 2 ? 16 : 8;

template <typename TIn, bool F16>
cudaError_t launch_t(int64_t rows, int H, const void* x, const __nv_bfloat16* gamma,
                     const __nv_bfloat16* beta, float eps, void* out, int* status,
                     cudaStream_t stream) {
  const int nv = H / 8;
  const int vpl1 = (nv + 31) / 32, vpl4 = (nv + 127) / 128;
  if (vpl1 <= kRowMaxVpl<TIn>) {
    if (vpl1 <= 1) return launch_rows<TIn, F16, 1, 1>(rows, H, x, gamma, beta, eps, out, status, stream);
    if (vpl1 <= 2) return launch_rows<TIn, F16, 2, 1>(rows, H, x, gamma, beta, eps, out, status, stream);
    if (vpl1 <= 4) return launch_rows<TIn, F16, 4, 1>(rows, H, x, gamma, beta, eps, out, status, stream);
    if (vpl1 <= 8) return launch_rows<TIn, F16, 8, 1>(rows, H, x, gamma, beta, eps, out, status, stream);
    if constexpr (kRowMaxVpl<TIn> >= 16)
      return launch_rows<TIn, F16, 16, 1>(rows, H, x, gamma, beta, eps, out, status, stream);
  }
  if (vpl4 <= kRowMaxVpl<TIn>) {
    // as few vector registers as the row needs: fewer registers, more rows in flight per SM
    if (vpl4 <= 4) return launch_rows<TIn, F16, 4, 4>(rows, H, x, gamma, beta, eps, out, status, stream);
    if (vpl4 <= 6) return launch_rows<TIn, F16, 6, 4>(rows, H, x, gamma, beta, eps, out, status, stream);
    if (vpl4 <= 8) return launch_rows<TIn, F16, 8, 4>(rows, H, x, gamma, beta, eps, out, status, stream);
    if constexpr (kRowMaxVpl<TIn> >= 16) {
      if (vpl4 <= 12)
        return launch_rows<TIn, F16, 12, 4>(rows, H, x, gamma, beta, eps, out, status, stream);
      return launch_rows<TIn, F16, 16, 4>(rows, H, x, gamma, beta, eps, out, status, stream);
    }
  }
  if (beta == nullptr)
    layernorm_kernel<TIn, F16, true><<<unsigned(rows), THREADS, 0, stream>>>(
        static_cast<const TIn*>(x), gamma, beta, static_cast<uint4*>(out), H, eps, status);
  else
    layernorm_kernel<TIn, F16, false><<<unsigned(rows), THREADS, 0, stream>>>(
        static_cast<const TIn*>(x), gamma, beta, static_cast<uint4*>(out), H, eps, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_layernorm(int64_t rows, int H, const void* x, bool x_f32,
                             const __nv_bfloat16* gamma, const __nv_bfloat16* beta, float eps,
                             void* out, bool out_f16, int* status, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (H <= 0 || H % 8 != 0 || H > kLnMaxH || rows > 0x7fffffff) return cudaErrorInvalidValue;
  if (x_f32)
    return out_f16 ? launch_t<float, true>(rows, H, x, gamma, beta, eps, out, status, stream)
                   : launch_t<float, false>(rows, H, x, gamma, beta, eps, out, status, stream);
  return out_f16
             ? launch_t<__nv_bfloat16, true>(rows, H, x, gamma, beta, eps, out, status, stream)
             : launch_t<__nv_bfloat16, false>(rows, H, x, gamma, beta, eps, out, status, stream);
}

cudaError_t launch_layernorm_e4m3(int64_t rows, int H, const void* x, bool x_f32,
                                  const __nv_bfloat16* gamma, const __nv_bfloat16* beta,
                                  float eps, uint8_t* out, float* scales, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (H <= 0 || H % 8 != 0 || H > kLnMaxH || rows > 0x7fffffff) return cudaErrorInvalidValue;
  uint2* o = reinterpret_cast<uint2*>(out);
  const unsigned g = unsigned(rows);
  if (x_f32) {
    if (beta == nullptr)
      layernorm_e4m3_kernel<float, true><<<g, THREADS, 0, stream>>>(
          static_cast<const float*>(x), gamma, beta, o, scales, H, eps);
    else
      layernorm_e4m3_kernel<float, false><<<g, THREADS, 0, stream>>>(
          static_cast<const float*>(x), gamma, beta, o, scales, H, eps);
  } else {
    if (beta == nullptr)
      layernorm_e4m3_kernel<__nv_bfloat16, true><<<g, THREADS, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(x), gamma, beta, o, scales, H, eps);
    else
      layernorm_e4m3_kernel<__nv_bfloat16, false><<<g, THREADS, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(x), gamma, beta, o, scales, H, eps);
  }
  return cudaGetLastError();
}

}  // namespace pb
