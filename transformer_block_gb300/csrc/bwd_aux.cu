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
constexpr int MAXV = kLnMaxH / (8 * THREADS);  // vectors of 8 per thread and row

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

// One CTA per row. The statistics follow the forward kernel: fp32, two passes.
template <bool RMS>
__global__ void __launch_bounds__(THREADS) norm_bwd_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
    const float* __restrict__ dxn, const __nv_bfloat16* __restrict__ dy, int H, float eps,
    __nv_bfloat16* __restrict__ dx, float2* __restrict__ stats) {
  __shared__ float red[THREADS / 32];
  const int64_t row = blockIdx.x;
  const int nv = H / 8;
  const __nv_bfloat16* xr = x + row * H;
  float v[MAXV][8];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
      load8(xr + idx * 8, v[i]);
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += v[i][e];
    }
  }
  const float mu = RMS ? 0.f : block_sum(sum, red) / float(H);
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sq += (v[i][e] - mu) * (v[i][e] - mu);
    }
  }
  const float rstd = rsqrtf(block_sum(sq, red) / float(H) + eps);
  // v becomes xhat; g = dxn * gamma
  float g[MAXV][8];
  float sg = 0.f, sgx = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
      float gm[8];
      load8(gamma + idx * 8, gm);
      const float4 d0 = *reinterpret_cast<const float4*>(dxn + row * H + idx * 8);
      const float4 d1 = *reinterpret_cast<const float4*>(dxn + row * H + idx * 8 + 4);
      const float d[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[i][e] = (v[i][e] - mu) * rstd;
        g[i][e] = d[e] * gm[e];
        sg += g[i][e];
        sgx += g[i][e] * v[i][e];
      }
    }
  }
  const float mean_g = RMS ? 0.f : block_sum(sg, red) / float(H);
  const float mean_gx = block_sum(sgx, red) / float(H);
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
      float r[8];
      load8(dy + row * H + idx * 8, r);
#pragma unroll
      for (int e = 0; e < 8; ++e) r[e] += rstd * (g[i][e] - mean_g - v[i][e] * mean_gx);
      *reinterpret_cast<uint4*>(dx + row * H + idx * 8) =
          make_uint4(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]), pack_bf16x2(r[4], r[5]),
                     pack_bf16x2(r[6], r[7]));
    }
  }
  if (threadIdx.x == 0) stats[row] = make_float2(mu, rstd);
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
    norm_bwd_kernel<true><<<unsigned(T), THREADS, 0, stream>>>(x, gamma, dxn, dy, H, eps, dx,
                                                               stats);
  else
    norm_bwd_kernel<false><<<unsigned(T), THREADS, 0, stream>>>(x, gamma, dxn, dy, H, eps, dx,
                                                                stats);
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
  col_partial_kernel<<<dim3(unsigned(gx), kColBlocks), THREADS, 0, stream>>>(m, rows, N, ld,
                                                                             partials);
  col_reduce_kernel<<<unsigned(gx), THREADS, 0, stream>>>(partials, N, out0, out1, split, glu_F,
                                                          accumulate);
  return cudaGetLastError();
}

}  // namespace pb
