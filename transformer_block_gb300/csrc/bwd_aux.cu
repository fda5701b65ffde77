// bwd_aux.cu — the memory-bound steps of the block's backward pass around its GEMMs and
// attention kernel:
//   * delta_i = dO_i . O_i per query and head (the softmax backward's row term);
//   * the fp32 dq accumulator to bf16 dq (scaled by 1/sqrt(dh)) in the dz operand;
//   * the normalisation backward (LayerNorm or RMSNorm) with the residual gradient added:
//     dx = dy + rstd (g - mean g - xhat mean(g xhat)), g = dxn * gamma;
//   * the parameter and bias gradients as column sums over the tokens, in a fixed order
//     (partial sums over kColBlocks row blocks, then one pass over the blocks), so they
//     are the same bits on every run.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace pb {
namespace {

constexpr int THREADS = 256;

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
    f[2 * e] = v.x;
    f[2 * e + 1] = v.y;
  }
}

// One warp per (token, head): dh / 32 consecutive elements per lane.
__global__ void attn_delta_kernel(const __nv_bfloat16* __restrict__ dO,
                                  const __nv_bfloat16* __restrict__ O, int64_t o_ld, int B, int S,
                                  int nh, int dh, float* __restrict__ delta, int64_t lse_ld) {
  const int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t T = int64_t(B) * S;
  if (w >= T * nh) return;
  const int64_t t = w / nh;
  const int head = int(w % nh);
  const int H = nh * dh;
  const __nv_bfloat16* a = dO + t * H + head * dh;
  const __nv_bfloat16* o = O + t * o_ld + head * dh;
  float acc = 0.f;
  for (int d = lane * 2; d < dh; d += 64) {
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(a + d));
    const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(o + d));
    acc += x.x * y.x + x.y * y.y;
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) {
    const int64_t b = t / S, i = t % S;
    delta[(b * nh + head) * lse_ld + i] = acc;
  }
}

__global__ void dq_to_bf16_kernel(const float* __restrict__ dq, int64_t T, int H, float scale,
                                  __nv_bfloat16* __restrict__ dz, int64_t ldz) {
  const int64_t nv = int64_t(H) / 8;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < T * nv;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t t = i / nv, c = (i % nv) * 8;
    const float4 a = *reinterpret_cast<const float4*>(dq + t * H + c);
    const float4 b = *reinterpret_cast<const float4*>(dq + t * H + c + 4);
    *reinterpret_cast<uint4*>(dz + t * ldz + c) =
        make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                   pack_bf16x2(b.x * scale, b.y * scale), pack_bf16x2(b.z * scale, b.w * scale));
  }
}

// A bf16 is the top half of its fp32 value. The shifts are volatile so that each pass
// converts the packed row again instead of the compiler keeping all fp32 values live.
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
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

// Sum over the WPR warps of one row: warp shuffles, then (WPR > 1) the warps' partial sums
// through shared memory behind the row's own named barrier; `slot` keeps the four
// reductions of a row apart, so no slot is written twice.
template <int WPR>
__device__ __forceinline__ float row_sum(float v, float* red, int slot) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (WPR == 1) return v;
  const int warp = threadIdx.x >> 5, grp = warp / WPR;
  if ((threadIdx.x & 31) == 0) red[slot * (THREADS / 32) + warp] = v;
  named_barrier(1 + grp, 32 * WPR);
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < WPR; ++w) s += red[slot * (THREADS / 32) + grp * WPR + w];
  return s;
}

// WPR warps per row (1 or 4), THREADS / (32 WPR) rows per CTA; thread t of a row holds
// the row's x vectors t, t + 32 WPR, ... packed in registers and reads dxn, gamma and dy
// in the passes that need them (dxn twice: the second read hits in cache). The
// statistics follow the forward kernel: fp32, two passes. Every thread of a row's warps
// takes the same branches around the named barriers.
template <bool RMS, int VPL, int WPR>
__global__ void __launch_bounds__(THREADS, 2) norm_bwd_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
    const float* __restrict__ dxn, const __nv_bfloat16* __restrict__ dy, int64_t T, int H,
    float eps, __nv_bfloat16* __restrict__ dx, float2* __restrict__ stats) {
  __shared__ float red[4 * (THREADS / 32)];
  constexpr int RT = 32 * WPR;  // threads per row
  const int t = int(threadIdx.x) % RT;
  const int64_t row = int64_t(blockIdx.x) * (THREADS / RT) + int(threadIdx.x) / RT;
  if (row >= T) return;
  const int nv = H / 8;
  uint4 xv[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int idx = t + RT * i;
    if (idx < nv) xv[i] = *reinterpret_cast<const uint4*>(x + row * H + idx * 8);
  }
  float sum = 0.f;
  if (!RMS) {
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (t + RT * i < nv) {
        float f[8];
        unpack8(xv[i], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) sum += f[e];
      }
  }
  const float mu = RMS ? 0.f : row_sum<WPR>(sum, red, 0) / float(H);
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (t + RT * i < nv) {
      float f[8];
      unpack8(xv[i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) sq += (f[e] - mu) * (f[e] - mu);
    }
  const float rstd = rsqrtf(row_sum<WPR>(sq, red, 1) / float(H) + eps);
  // g = dxn * gamma; sums of g and of g * xhat
  float sg = 0.f, sgx = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int idx = t + RT * i;
    if (idx < nv) {
      float f[8], gm[8];
      unpack8(xv[i], f);
      load8(gamma + idx * 8, gm);
      const float4 d0 = *reinterpret_cast<const float4*>(dxn + row * H + idx * 8);
      const float4 d1 = *reinterpret_cast<const float4*>(dxn + row * H + idx * 8 + 4);
      const float d[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float g = d[e] * gm[e];
        sg += g;
        sgx += g * (f[e] - mu) * rstd;
      }
    }
  }
  const float mean_g = RMS ? 0.f : row_sum<WPR>(sg, red, 2) / float(H);
  const float mean_gx = row_sum<WPR>(sgx, red, 3) / float(H);
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int idx = t + RT * i;
    if (idx < nv) {
      float f[8], gm[8], r[8];
      unpack8(xv[i], f);
      load8(gamma + idx * 8, gm);
      load8(dy + row * H + idx * 8, r);
      const float4 d0 = *reinterpret_cast<const float4*>(dxn + row * H + idx * 8);
      const float4 d1 = *reinterpret_cast<const float4*>(dxn + row * H + idx * 8 + 4);
      const float d[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e)
        r[e] += rstd * (d[e] * gm[e] - mean_g - (f[e] - mu) * rstd * mean_gx);
      *reinterpret_cast<uint4*>(dx + row * H + idx * 8) =
          make_uint4(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]), pack_bf16x2(r[4], r[5]),
                     pack_bf16x2(r[6], r[7]));
    }
  }
  if (t == 0) stats[row] = make_float2(mu, rstd);
}

template <bool RMS, int VPL, int WPR>
void launch_norm_rows(int64_t T, int H, const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                      const float* dxn, const __nv_bfloat16* dy, float eps, __nv_bfloat16* dx,
                      float2* stats, cudaStream_t stream) {
  constexpr int RPC = THREADS / (32 * WPR);  // rows per CTA
  const int64_t grid = (T + RPC - 1) / RPC;
  norm_bwd_kernel<RMS, VPL, WPR><<<unsigned(grid), THREADS, 0, stream>>>(x, gamma, dxn, dy, T,
                                                                          H, eps, dx, stats);
}

template <bool RMS>
void launch_norm_bwd_t(int64_t T, int H, const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                       const float* dxn, const __nv_bfloat16* dy, float eps,
                       __nv_bfloat16* dx, float2* stats, cudaStream_t stream) {
  // one warp per row up to 4096 elements (16 packed vectors per lane), else four warps
  // (up to 16384 = kLnMaxH)
  const int nv = H / 8;
  const int vpl1 = (nv + 31) / 32, vpl4 = (nv + 127) / 128;
  if (vpl1 <= 1) return launch_norm_rows<RMS, 1, 1>(T, H, x, gamma, dxn, dy, eps, dx, stats, stream);
  if (vpl1 <= 2) return launch_norm_rows<RMS, 2, 1>(T, H, x, gamma, dxn, dy, eps, dx, stats, stream);
  if (vpl1 <= 4) return launch_norm_rows<RMS, 4, 1>(T, H, x, gamma, dxn, dy, eps, dx, stats, stream);
  if (vpl1 <= 8) return launch_norm_rows<RMS, 8, 1>(T, H, x, gamma, dxn, dy, eps, dx, stats, stream);
  if (vpl1 <= 16) return launch_norm_rows<RMS, 16, 1>(T, H, x, gamma, dxn, dy, eps, dx, stats, stream);
  if (vpl4 <= 8) return launch_norm_rows<RMS, 8, 4>(T, H, x, gamma, dxn, dy, eps, dx, stats, stream);
  return launch_norm_rows<RMS, 16, 4>(T, H, x, gamma, dxn, dy, eps, dx, stats, stream);
}

// Partial column sums over row block blockIdx.y: one column per thread (coalesced rows).
__global__ void norm_param_partial_kernel(const __nv_bfloat16* __restrict__ x,
                                          const float* __restrict__ dxn,
                                          const float2* __restrict__ stats, int64_t T, int H,
                                          float* __restrict__ partials) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= H) return;
  const int64_t per = (T + kColBlocks - 1) / kColBlocks;
  const int64_t r0 = int64_t(blockIdx.y) * per;
  const int64_t r1 = r0 + per < T ? r0 + per : T;
  float sg = 0.f, sb = 0.f;
  for (int64_t r = r0; r < r1; ++r) {
    const float2 st = stats[r];
    const float d = dxn[r * H + c];
    sg += d * (__bfloat162float(x[r * H + c]) - st.x) * st.y;
    sb += d;
  }
  partials[int64_t(blockIdx.y) * H + c] = sg;
  partials[int64_t(kColBlocks + blockIdx.y) * H + c] = sb;
}

__global__ void norm_param_reduce_kernel(const float* __restrict__ partials, int H,
                                         float* __restrict__ dgamma, float* __restrict__ dbeta,
                                         bool accumulate) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= H) return;
  float sg = 0.f, sb = 0.f;
  for (int k = 0; k < kColBlocks; ++k) {
    sg += partials[int64_t(k) * H + c];
    sb += partials[int64_t(kColBlocks + k) * H + c];
  }
  dgamma[c] = accumulate ? dgamma[c] + sg : sg;
  if (dbeta != nullptr) dbeta[c] = accumulate ? dbeta[c] + sb : sb;
}

__global__ void col_partial_kernel(const __nv_bfloat16* __restrict__ m, int64_t rows, int64_t N,
                                   int64_t ld, float* __restrict__ partials) {
  const int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= N) return;
  const int64_t per = (rows + kColBlocks - 1) / kColBlocks;
  const int64_t r0 = int64_t(blockIdx.y) * per;
  const int64_t r1 = r0 + per < rows ? r0 + per : rows;
  float s = 0.f;
  for (int64_t r = r0; r < r1; ++r) s += __bfloat162float(m[r * ld + c]);
  partials[int64_t(blockIdx.y) * N + c] = s;
}

// The same partial sums, 8 columns per thread from 16-byte loads (a warp reads 512
// contiguous bytes of a row) and 4 rows in flight; each column still adds its rows in
// increasing order, so the sums are the same bits as col_partial_kernel's. Needs N and ld
// multiples of 8 and m 16-byte aligned.
__global__ void col_partial8_kernel(const __nv_bfloat16* __restrict__ m, int64_t rows,
                                    int64_t N, int64_t ld, float* __restrict__ partials) {
  const int64_t c0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
  if (c0 >= N) return;
  const int64_t per = (rows + kColBlocks - 1) / kColBlocks;
  const int64_t r0 = int64_t(blockIdx.y) * per;
  const int64_t r1 = r0 + per < rows ? r0 + per : rows;
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int64_t r = r0;
  for (; r + 4 <= r1; r += 4) {
    uint4 u[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) u[q] = *reinterpret_cast<const uint4*>(m + (r + q) * ld + c0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float f[8];
      load8(reinterpret_cast<const __nv_bfloat16*>(&u[q]), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) s[e] += f[e];
    }
  }
  for (; r < r1; ++r) {
    float f[8];
    load8(m + r * ld + c0, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) s[e] += f[e];
  }
  float4* dst = reinterpret_cast<float4*>(partials + int64_t(blockIdx.y) * N + c0);
  dst[0] = make_float4(s[0], s[1], s[2], s[3]);
  dst[1] = make_float4(s[4], s[5], s[6], s[7]);
}

__global__ void col_reduce_kernel(const float* __restrict__ partials, int64_t N, float* out0,
                                  float* out1, int64_t split, int64_t glu_F, bool accumulate) {
  const int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= N) return;
  float s = 0.f;
  for (int k = 0; k < kColBlocks; ++k) s += partials[int64_t(k) * N + c];
  float* dst;
  if (c < split) {
    dst = out0 ? out0 + c : nullptr;
  } else {
    int64_t j = c - split;
    if (glu_F > 0) {
      const int64_t t = j / 32, i = j % 32;
      j = i < 16 ? 16 * t + i : glu_F + 16 * t + (i - 16);
    }
    dst = out1 ? out1 + j : nullptr;
  }
  if (dst != nullptr) *dst = accumulate ? *dst + s : s;
}

}  // namespace

cudaError_t launch_attn_delta(const __nv_bfloat16* dO, const __nv_bfloat16* O, int64_t o_ld,
                              int B, int S, int nh, int dh, float* delta, int64_t lse_ld,
                              cudaStream_t stream) {
  const int64_t warps = int64_t(B) * S * nh;
  if (warps <= 0) return cudaSuccess;
  if (dh % 64 != 0) return cudaErrorInvalidValue;
  const int64_t blocks = (warps * 32 + THREADS - 1) / THREADS;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  attn_delta_kernel<<<unsigned(blocks), THREADS, 0, stream>>>(dO, O, o_ld, B, S, nh, dh, delta,
                                                               lse_ld);
  return cudaGetLastError();
}

cudaError_t launch_dq_to_bf16(const float* dq_acc, int64_t T, int H, float scale,
                              __nv_bfloat16* dz, int64_t ldz, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  if (H % 8 != 0 || ldz % 8 != 0) return cudaErrorInvalidValue;
  dq_to_bf16_kernel<<<1024, THREADS, 0, stream>>>(dq_acc, T, H, scale, dz, ldz);
  return cudaGetLastError();
}

cudaError_t launch_norm_bwd(int64_t T, int H, const __nv_bfloat16* x,
                            const __nv_bfloat16* gamma, const float* dxn,
                            const __nv_bfloat16* dy, float eps, bool rms, __nv_bfloat16* dx,
                            float2* stats, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  if (H <= 0 || H % 8 != 0 || H > kLnMaxH || T > 0x7fffffff) return cudaErrorInvalidValue;
  if (rms)
    launch_norm_bwd_t<true>(T, H, x, gamma, dxn, dy, eps, dx, stats, stream);
  else
    launch_norm_bwd_t<false>(T, H, x, gamma, dxn, dy, eps, dx, stats, stream);
  return cudaGetLastError();
}

cudaError_t launch_norm_param_grads(int64_t T, int H, const __nv_bfloat16* x, const float* dxn,
                                    const float2* stats, float* partials, float* dgamma,
                                    float* dbeta, bool accumulate, cudaStream_t stream) {
  if (H <= 0) return cudaSuccess;
  const unsigned gx = unsigned((H + THREADS - 1) / THREADS);
  norm_param_partial_kernel<<<dim3(gx, kColBlocks), THREADS, 0, stream>>>(x, dxn, stats, T, H,
                                                                          partials);
  norm_param_reduce_kernel<<<gx, THREADS, 0, stream>>>(partials, H, dgamma, dbeta, accumulate);
  return cudaGetLastError();
}

cudaError_t launch_col_sums(const __nv_bfloat16* m, int64_t rows, int64_t N, int64_t ld,
                            float* partials, float* out0, float* out1, int64_t split,
                            int64_t glu_F, bool accumulate, cudaStream_t stream) {
  if (N <= 0) return cudaSuccess;
  if (glu_F > 0 && ((N - split) != 2 * glu_F || glu_F % 16 != 0)) return cudaErrorInvalidValue;
  const int64_t gx = (N + THREADS - 1) / THREADS;
  if (gx > 0x7fffffff) return cudaErrorInvalidValue;
  if (N % 8 == 0 && ld % 8 == 0 && (reinterpret_cast<uintptr_t>(m) & 15) == 0) {
    const int64_t gx8 = (N / 8 + THREADS - 1) / THREADS;
    col_partial8_kernel<<<dim3(unsigned(gx8), kColBlocks), THREADS, 0, stream>>>(m, rows, N,
                                                                                 ld, partials);
  } else {
    col_partial_kernel<<<dim3(unsigned(gx), kColBlocks), THREADS, 0, stream>>>(m, rows, N, ld,
                                                                               partials);
  }
  col_reduce_kernel<<<unsigned(gx), THREADS, 0, stream>>>(partials, N, out0, out1, split, glu_F,
                                                          accumulate);
  return cudaGetLastError();
}

}  // namespace pb
