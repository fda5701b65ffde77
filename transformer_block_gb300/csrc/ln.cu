// ln.cu — LayerNorm of the token rows (the single LN shared by both branches of the
// parallel block, MegaScale reading notes, section 1.1, eq. (4)).
//
// One 128-thread CTA per row. Each thread keeps its share of the row in registers as
// 128-bit vectors (8 bf16), so x is read from HBM once; the mean and then the centred
// variance are reduced across the CTA in fp32 (warp shuffles, then 4 partial sums in
// shared memory); the normalised, affine-mapped row is written back as bf16 (round to
// nearest even). HBM-bound: 2 bytes read + 2 bytes written per element.
#include "kernels.h"

namespace pb {
namespace {

constexpr int THREADS = 128;
constexpr int MAXV = kLnMaxH / (8 * THREADS);  // 16 vectors per thread

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const float s = red[0] + red[1] + red[2] + red[3];
  __syncthreads();
  return s;
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
    f[2 * e] = p.x;
    f[2 * e + 1] = p.y;
  }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(THREADS) layernorm_kernel(const uint4* __restrict__ x,
                                                            const uint4* __restrict__ gamma,
                                                            const uint4* __restrict__ beta,
                                                            uint4* __restrict__ out, int H,
                                                            float eps) {
  __shared__ float red[4];
  const int nv = H / 8;
  const int64_t row = blockIdx.x;
  const uint4* xr = x + row * nv;
  uint4 v[MAXV];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
      v[i] = xr[idx];
      float f[8];
      unpack8(v[i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += f[e];
    }
  }
  const float mean = block_sum(sum, red) / float(H);
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
      float f[8];
      unpack8(v[i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) sq += (f[e] - mean) * (f[e] - mean);
    }
  }
  const float var = block_sum(sq, red) / float(H);
  const float rstd = rsqrtf(var + eps);
  uint4* orow = out + row * nv;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    if (idx < nv) {
      float f[8], g[8], b[8];
      unpack8(v[i], f);
      unpack8(__ldg(gamma + idx), g);
      unpack8(__ldg(beta + idx), b);
      uint4 o;
      o.x = pack2((f[0] - mean) * rstd * g[0] + b[0], (f[1] - mean) * rstd * g[1] + b[1]);
      o.y = pack2((f[2] - mean) * rstd * g[2] + b[2], (f[3] - mean) * rstd * g[3] + b[3]);
      o.z = pack2((f[4] - mean) * rstd * g[4] + b[4], (f[5] - mean) * rstd * g[5] + b[5]);
      o.w = pack2((f[6] - mean) * rstd * g[6] + b[6], (f[7] - mean) * rstd * g[7] + b[7]);
      orow[idx] = o;
    }
  }
}

}  // namespace

cudaError_t launch_layernorm(int64_t rows, int H, const __nv_bfloat16* x,
                             const __nv_bfloat16* gamma, const __nv_bfloat16* beta, float eps,
                             __nv_bfloat16* out, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (H <= 0 || H % 8 != 0 || H > kLnMaxH || rows > 0x7fffffff) return cudaErrorInvalidValue;
  layernorm_kernel<<<unsigned(rows), THREADS, 0, stream>>>(
      reinterpret_cast<const uint4*>(x), reinterpret_cast<const uint4*>(gamma),
      reinterpret_cast<const uint4*>(beta), reinterpret_cast<uint4*>(out), H, eps);
  return cudaGetLastError();
}

}  // namespace pb
