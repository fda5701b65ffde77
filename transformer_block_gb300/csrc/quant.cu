// quant.cu — FP8 E4M3 quantization for the FP8 GEMM path: per-row current scaling (each
// row's scale is its largest magnitude / 448, the E4M3 maximum), as in the FP8 recipe of
// the performance notes ("BF16 / FP16 / FP8": E4M3 for the forward pass, only the GEMMs in
// FP8, the scale taken from the current tensor). The steps are fixed in fp32 so that any
// implementation reproduces the codes exactly:
//   amax = max_c |x[r,c]|,   inv = 448 / amax (0 when amax = 0),   scale[r] = amax / 448,
//   code[r,c] = E4M3(x[r,c] * inv)   (round to nearest even, saturating).
#include "kernels.h"
#include "ptx.cuh"

namespace pb {
namespace {

constexpr int THREADS = 256;

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

__device__ __forceinline__ void unpack8(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
    f[2 * e] = p.x;
    f[2 * e + 1] = p.y;
  }
}

// One CTA per row of a bf16 [rows, cols] matrix (cols % 8 == 0, row stride ld_in
// elements): the row is read twice (amax, then the codes), the second time from L2.
__global__ void __launch_bounds__(THREADS) quantize_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                                int64_t cols, int64_t ld_in,
                                                                uint8_t* __restrict__ codes,
                                                                int64_t ld_out,
                                                                float* __restrict__ scales) {
  __shared__ float red[THREADS / 32];
  const int64_t row = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * ld_in);
  const int64_t nv = cols / 8;
  float amax = 0.f;
  for (int64_t i = threadIdx.x; i < nv; i += THREADS) {
    float f[8];
    unpack8(xr[i], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
  }
  amax = block_max(amax, red);
  const float inv = amax > 0.f ? 448.f / amax : 0.f;
  if (threadIdx.x == 0) scales[row] = amax / 448.f;
  uint2* cr = reinterpret_cast<uint2*>(codes + row * ld_out);
  for (int64_t i = threadIdx.x; i < nv; i += THREADS) {
    float f[8];
    unpack8(xr[i], f);
    cr[i] = quant8_e4m3(f, inv);
  }
}

// amax[c] = max(amax[c], max_r |w[r, c]|) over a bf16 [rows, cols] matrix (row stride ld):
// one thread per column (coalesced across the warp), rows split over blockIdx.y. amax
// holds non-negative floats, which order like their bit patterns, so atomicMax on the bits
// is a float max.
__global__ void col_amax_kernel(const __nv_bfloat16* __restrict__ w, int64_t rows, int64_t cols,
                                int64_t ld, int64_t rows_per_block, float* __restrict__ amax) {
  const int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  const int64_t r0 = int64_t(blockIdx.y) * rows_per_block;
  const int64_t r1 = r0 + rows_per_block < rows ? r0 + rows_per_block : rows;
  float m = 0.f;
  for (int64_t r = r0; r < r1; ++r) m = fmaxf(m, fabsf(__bfloat162float(w[r * ld + c])));
  atomicMax(reinterpret_cast<unsigned int*>(amax) + c, __float_as_uint(m));
}

}  // namespace

cudaError_t launch_quantize_rows_e4m3(const __nv_bfloat16* x, int64_t rows, int64_t cols,
                                      int64_t ld_in, uint8_t* codes, int64_t ld_out,
                                      float* scales, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (cols <= 0 || cols % 8 != 0 || ld_in % 8 != 0 || ld_out % 8 != 0 || rows > 0x7fffffff)
    return cudaErrorInvalidValue;
  quantize_rows_kernel<<<unsigned(rows), THREADS, 0, stream>>>(x, cols, ld_in, codes, ld_out,
                                                                scales);
  return cudaGetLastError();
}

cudaError_t launch_col_amax(const __nv_bfloat16* w, int64_t rows, int64_t cols, int64_t ld,
                            float* amax, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const int64_t per = 256;
  const int64_t gx = (cols + 255) / 256, gy = (rows + per - 1) / per;
  if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidValue;
  col_amax_kernel<<<dim3(unsigned(gx), unsigned(gy)), 256, 0, stream>>>(w, rows, cols, ld, per,
                                                                         amax);
  return cudaGetLastError();
}

}  // namespace pb
