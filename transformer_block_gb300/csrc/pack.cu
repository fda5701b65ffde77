// pack.cu — one-time packing of the block's weights (run by pb_create, not per forward).
//
// The pages store a linear layer as W [in, out] with Y = X W (Megatron-LM notes, section
// 2.1). The tensor-core GEMM reads its B operand K-major, [out, in], so each weight is
// transposed once into the two concatenated operands:
//   W1cat [3H + F, H] = [Wqkv | W1]^T        W2cat [H, H + F] = [Wo ; W2]^T
// and the optional biases are gathered into fp32 vectors of the GEMMs' output columns.
// For the SwiGLU block W1 = [W_gate | W_up] is [H, 2F] and its 2F rows of W1cat are
// interleaved in groups of 16: row 32t + i is column 16t + i of W_gate (i < 16) or of W_up
// (i >= 16), so every 32-column block the GEMM epilogue handles holds 16 gate values and
// the 16 up values they multiply.
#include <cuda_fp16.h>

#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace pb {
namespace {

constexpr int TILE = 32;

// Input column of output row c: c itself, or with glu_F > 0 the gate / up interleave
// described above (c in [0, 2 glu_F)).
__device__ __forceinline__ int64_t glu_source(int64_t c, int64_t glu_F) {
  if (glu_F == 0) return c;
  const int64_t t = c / 32, i = c % 32;
  return i < 16 ? 16 * t + i : glu_F + 16 * t + (i - 16);
}

// out[c * ld_out + r] = in[r * ld_in + glu_source(c)], through a padded 32 x 32 shared-memory
// tile so both the reads and the writes are coalesced; TOut is bf16 (a copy), fp16 (a
// conversion, exact inside the fp16 range; values beyond it are reported) or uint8_t: the
// FP8 E4M3 code of the value times 448 / amax[glu_source(c)] (per-output-channel current
// scaling, the same fp32 steps as the row quantizer of quant.cu).
template <typename TOut>
__global__ void transpose_kernel(const __nv_bfloat16* __restrict__ in, int64_t rows, int64_t cols,
                                 int64_t ld_in, TOut* __restrict__ out, int64_t ld_out,
                                 int64_t glu_F, const float* __restrict__ amax, int* status) {
  __shared__ float tile[TILE][TILE + 1];
  const int64_t r0 = int64_t(blockIdx.y) * TILE, c0 = int64_t(blockIdx.x) * TILE;
  for (int i = threadIdx.y; i < TILE; i += blockDim.y) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols)
      tile[i][threadIdx.x] = __bfloat162float(in[r * ld_in + glu_source(c, glu_F)]);
  }
  __syncthreads();
  bool bad = false;
  for (int i = threadIdx.y; i < TILE; i += blockDim.y) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) {
      const float v = tile[threadIdx.x][i];
      if (std::is_same<TOut, uint8_t>::value) {
        const float a = amax[glu_source(c, glu_F)];
        const float inv = a > 0.f ? 448.f / a : 0.f;
        out[c * ld_out + r] = TOut(cvt_e4m3x2(v * inv, 0.f) & 0xFF);
      } else if (sizeof(TOut) == 2 && std::is_same<TOut, __half>::value) {
        bad |= !(fabsf(v) <= 65504.f);
        out[c * ld_out + r] = TOut(__float2half_rn(v));
      } else {
        out[c * ld_out + r] = TOut(__float2bfloat16_rn(v));
      }
    }
  }
  if (bad && status != nullptr) atomicCAS(status, 0, kStatusRange);
}

__global__ void bias_prep_kernel(const __nv_bfloat16* b_qkv, const __nv_bfloat16* b1,
                                 const __nv_bfloat16* b_o, const __nv_bfloat16* b2, int H, int F,
                                 bool glu, float* bias1, float* bias2, float* bias_o,
                                 float* bias_2) {
  const int n1 = 3 * H + (glu ? 2 * F : F);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n1; i += gridDim.x * blockDim.x) {
    float v = 0.f;
    if (i < 3 * H) {
      if (b_qkv) v = __bfloat162float(b_qkv[i]);
    } else if (b1) {
      v = __bfloat162float(b1[glu_source(i - 3 * H, glu ? F : 0)]);
    }
    bias1[i] = v;
    if (i < H) {
      const float o = b_o ? __bfloat162float(b_o[i]) : 0.f;
      const float t = b2 ? __bfloat162float(b2[i]) : 0.f;
      bias2[i] = o + t;
      bias_o[i] = o;
      bias_2[i] = t;
    }
  }
}

}  // namespace

cudaError_t launch_transpose(const __nv_bfloat16* in, int64_t rows, int64_t cols, int64_t ld_in,
                             void* out, int64_t ld_out, bool out_f16, int64_t glu_F, int* status,
                             cudaStream_t stream) {
  if (glu_F != 0 && (cols != 2 * glu_F || glu_F % 16 != 0)) return cudaErrorInvalidValue;
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const int64_t gx = (cols + TILE - 1) / TILE, gy = (rows + TILE - 1) / TILE;
  if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidValue;
  const dim3 grid{unsigned(gx), unsigned(gy), 1u}, block{unsigned(TILE), 8u, 1u};
  if (out_f16)
    transpose_kernel<__half><<<grid, block, 0, stream>>>(in, rows, cols, ld_in,
                                                          static_cast<__half*>(out), ld_out,
                                                          glu_F, nullptr, status);
  else
    transpose_kernel<__nv_bfloat16><<<grid, block, 0, stream>>>(
        in, rows, cols, ld_in, static_cast<__nv_bfloat16*>(out), ld_out, glu_F, nullptr,
        status);
  return cudaGetLastError();
}

cudaError_t launch_transpose_e4m3(const __nv_bfloat16* in, int64_t rows, int64_t cols,
                                  int64_t ld_in, uint8_t* out, int64_t ld_out, int64_t glu_F,
                                  const float* amax, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  if (glu_F != 0 && (cols != 2 * glu_F || glu_F % 16 != 0)) return cudaErrorInvalidValue;
  const int64_t gx = (cols + TILE - 1) / TILE, gy = (rows + TILE - 1) / TILE;
  if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidValue;
  const dim3 grid{unsigned(gx), unsigned(gy), 1u}, block{unsigned(TILE), 8u, 1u};
  transpose_kernel<uint8_t><<<grid, block, 0, stream>>>(in, rows, cols, ld_in, out, ld_out, glu_F,
                                                         amax, nullptr);
  return cudaGetLastError();
}

namespace {
// scales[c] = amax[glu_source(c)] / 448 for the n output channels.
__global__ void amax_to_scales_kernel(const float* amax, int64_t n, int64_t glu_F, float* scales) {
  for (int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; c < n;
       c += int64_t(gridDim.x) * blockDim.x)
    scales[c] = amax[glu_source(c, glu_F)] / 448.f;
}
}  // namespace

cudaError_t launch_amax_to_scales(const float* amax, int64_t n, int64_t glu_F, float* scales,
                                  cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  amax_to_scales_kernel<<<256, 256, 0, stream>>>(amax, n, glu_F, scales);
  return cudaGetLastError();
}

cudaError_t launch_bias_prep(const __nv_bfloat16* b_qkv, const __nv_bfloat16* b1,
                             const __nv_bfloat16* b_o, const __nv_bfloat16* b2, int H, int F,
                             bool glu, float* bias1, float* bias2, float* bias_o, float* bias_2,
                             cudaStream_t stream) {
  bias_prep_kernel<<<256, 256, 0, stream>>>(b_qkv, b1, b_o, b2, H, F, glu, bias1, bias2, bias_o,
                                            bias_2);
  return cudaGetLastError();
}

}  // namespace pb
