// kernels.h — launch interface between the C ABI (pb_api.cu) and the sm_103a kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace pb {

// ---------------------------------------------------------------- per-device set-up
// The runtime keeps a kernel's function attributes (the large dynamic shared memory
// opt-in) per device, and occupancy differs between devices, so launch set-up runs once
// per device ordinal, under std::call_once (safe when several host threads launch at
// once), and its result is kept for that device.
constexpr int kMaxDevices = 128;
struct PerDeviceInit {
  std::once_flag once[kMaxDevices];
  cudaError_t err[kMaxDevices] = {};
  int value[kMaxDevices] = {};
};
// Runs init(device, &value) once for the current device; returns its error and (when
// value_out is not null) the value it stored.
template <class F>
cudaError_t per_device_init(PerDeviceInit& s, F&& init, int* value_out = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(s.once[dev], [&] { s.err[dev] = init(dev, &s.value[dev]); });
  if (value_out != nullptr) *value_out = s.value[dev];
  return s.err[dev];
}

// ---------------------------------------------------------------- LayerNorm (ln.cu)
constexpr int kLnMaxH = 16384;
constexpr int kStatusRange = 7;  // == PB_ERR_RANGE
// x: [rows, H] bf16 (x_f32 false) or fp32; out: bf16 (out_f16 false) or fp16. With fp16
// output a value beyond the fp16 range records kStatusRange in *status (may be null).
// beta == nullptr selects RMSNorm: x / sqrt(mean x^2 + eps) * gamma.
cudaError_t launch_layernorm(int64_t rows, int H, const void* x, bool x_f32,
                             const __nv_bfloat16* gamma, const __nv_bfloat16* beta, float eps,
                             void* out, bool out_f16, int* status, cudaStream_t stream);

// ---------------------------------------------------------------- GEMM (gemm.cu)
// D[M, N] = A[M, K] * B[N, K]^T with tcgen05 on CTA pairs; A and B come in through TMA
// tensor maps (128-byte swizzle, boxes of 128 bytes of K x kGemmBoxRows rows for both:
// 64 elements of a 16-bit operand, 128 of an FP8 one).
constexpr int kGemmBM = 128;       // rows of A per CTA
constexpr int kGemmBN = 256;       // columns of D per CTA pair (128 rows of B per CTA)
constexpr int kGemmBK = 64;        // K elements per stage, 16-bit operands
constexpr int kGemmBK8 = 128;      // K elements per stage, FP8 operands
constexpr int kGemmBoxRows = 128;

// Operand types of the GEMM: both operands have the same one.
enum OpType : int { kOpBf16 = 0, kOpF16 = 1, kOpE4m3 = 2 };

enum EpiKind : int {
  kEpiStore = 0,     // C = bf16(D)
  kEpiBlockIn = 1,   // D = xn [Wqkv | W1]: route q|k, v (transposed per head), GeLU(h)
  kEpiResidual = 2,  // y = bf16(D + bias + x)
  kEpiBwdAct = 3,    // D = dy [Wo ; W2]^T: d_attn (bf16), and dh = D * act'(h) into dz
  kEpiGrad = 4,      // fp32 gradient store (or accumulate), split by rows or columns
};

// Operand layouts: bit 0 set = A is MN-major (stored [K, M], M contiguous), bit 1 = B is
// MN-major ([K, N]). K-major operands are [M, K] / [N, K], K contiguous.
enum GemmLayout : int { kKK = 0, kMK = 1, kKM = 2, kMM = 3 };

struct EpiParams {
  // TMA stores of the 16-bit row-major outputs (tma_store): kEpiBlockIn writes q|k through
  // tm_out0 ([T, 2H]) and GeLU(h) through tm_out1 ([T, H + F]), kEpiResidual writes y
  // through tm_out0 ([T, N]); boxes of 32 columns x 32 rows, 64-byte swizzle. Each
  // epilogue warp stages its 32 x 32 chunk in shared memory and one lane issues the copy,
  // so the stores leave the load/store path the main loop's operand traffic uses.
  CUtensorMap tm_out0;  // the type carries the alignment TMA needs
  CUtensorMap tm_out1;
  bool tma_store;
  int M, N;
  int* status;  // device status word (fp16 range errors), may be null
  // kEpiStore
  __nv_bfloat16* c;
  int64_t ldc;
  // kEpiBlockIn. Output column c of this GEMM is routed as column c + col_base of
  // [q | k | v | h]: 0 for the parallel block's one GEMM over [Wqkv | W1], 3H for a GEMM
  // over W1 alone (the serial block's MLP input projection).
  int col_base;
  // SwiGLU: the h columns are [gate | up] interleaved in 16s (see launch_transpose); each
  // 32-column block gives 16 outputs silu(gate) * up at act column H + (c - 3H) / 2.
  bool glu;
  int H, F, S, nh, dh;
  int64_t seq_pad;
  __nv_bfloat16* qk;   // [T, 2H]
  __nv_bfloat16* vt;   // [B*nh*dh, seq_pad]
  void* act;           // [T, H + F]; GeLU(h) goes to columns [H, H + F)
  bool act_f16;        // act holds fp16 (else bf16)
  // kEpiBlockIn / kEpiResidual: fp32 bias of the N output columns, or null
  const float* bias;
  // FP8 operands: D[m, n] is scale_a[m] * scale_b[n] times the accumulated sum (per-row
  // scales of A and per-output-channel scales of B), applied before the bias; null = 1.
  const float* scale_a;
  const float* scale_b;
  // kEpiResidual
  const void* resid;  // [M, N], fp32 if resid_f32 else bf16
  void* y;            // [M, N], fp32 if y_f32 else bf16
  bool resid_f32;
  bool y_f32;
  // kEpiBlockIn: when set, the pre-activation h (after its bias) is also stored here,
  // [T, N - 3H] bf16 in W1cat row order (training forward). kEpiBwdAct reads it back.
  __nv_bfloat16* hpre;
  // kEpiBwdAct (N = H + F): columns [0, H) are d_attn = dy Wo^T -> d_attn [T, H] bf16;
  // column H + f is d act_f = dy W2^T -> dh = d act_f * gelu'(h_f) at dz column 3H + f
  // (SwiGLU: d gate and d up at the W1cat-order columns of feature f), dz row stride ldz.
  __nv_bfloat16* d_attn;
  __nv_bfloat16* dz;
  int64_t ldz;
  // kEpiGrad: D[m, n] -> g0[m * ld0 + n] while m < split_row and n < split_col; rows from
  // split_row on -> g1[(m - split_row) * ld1 + n]; columns from split_col on ->
  // g1[m * ld1 + (n - split_col)], with glu the W1cat interleave undone (column
  // split_col + 32t + i is gate feature 16t + i for i < 16, else up feature F + 16t + i - 16).
  // accumulate: add to what is there (fp32 gradient accumulation).
  float* g0;
  float* g1;
  int64_t ld0, ld1;
  int split_row, split_col;
  bool accumulate;
};

// Stream-K work space: the tiles of the last waves are split along K across all CTA
// pairs; a pair whose K segment does not start at 0 leaves its fp32 partial tile here and
// publishes it with a per-warp flag (the launch's epoch value). The one warp that reads a
// flag clears it after use, so every launch that completes leaves the flags at zero.
constexpr int kSkMaxClusters = 96;
constexpr size_t kSkPartialBytes = size_t(2) * 128 * 256 * 4;  // one pair tile, fp32
constexpr size_t kSkFlagBytes = size_t(2) * 4 * 8;             // 2 CTAs x 4 warps x u64
constexpr size_t kSkScratchBytes = size_t(kSkMaxClusters) * (kSkPartialBytes + kSkFlagBytes);

size_t gemm_smem_bytes();
// op: the type of A and B (K % 64 == 0, K % 128 == 0 for kOpE4m3). sk_scratch
// (kSkScratchBytes, 256-byte aligned) may be null: then every tile is computed whole by one
// CTA pair.
cudaError_t launch_gemm(EpiKind kind, OpType op, const CUtensorMap& tmA, const CUtensorMap& tmB,
                        int M, int N, int K, const EpiParams& ep, int num_sms, int* status,
                        uint64_t limit_ns, void* sk_scratch, cudaStream_t stream);
// bf16 operands in the given layout. An MN-major operand's tensor map is [K rows, M (or N)
// columns] in boxes of 64 x 64; K need not be a multiple of 64 (the last block is zero
// filled). Kinds: kEpiStore (any layout), kEpiBwdAct and kEpiGrad (kKM, kMM).
cudaError_t launch_gemm_layout(EpiKind kind, GemmLayout layout, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, int M, int N, int K, const EpiParams& ep,
                               int num_sms, int* status, uint64_t limit_ns, void* sk_scratch,
                               cudaStream_t stream);

// ---------------------------------------------------------------- attention (swa.cu)
struct SwaParams {
  int B, S, H, nh, dh, window;
  int num_q_tiles;
  float scale_log2;    // log2(e) / sqrt(dh)
  void* out;  // attention output, row (b*S + i), columns [head*dh, (head+1)*dh)
  int64_t out_ld;
  bool out_f16;  // write fp16 (else bf16)
  float* lse;    // training forward: [B * nh, lse_ld] log2-sum-exp of each row's scores
                 // (times log2(e) / sqrt(dh)), or null
  int64_t lse_ld;
};
constexpr int kSwaBQ = 128;  // query rows per tile (two tiles per CTA)
constexpr int kSwaBKV = 128;  // keys per tile
// tmQ: the [B][S][2H] q|k buffer in boxes of 64 columns x kSwaBQ rows; tmK: the same buffer
// in boxes of 64 columns x kSwaBKV rows; tmVT: v^T [B*nh*dh][seq_pad] in boxes of kSwaBKV
// keys x dh rows.
cudaError_t launch_swa(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmVT,
                       const SwaParams& p, int* status, uint64_t limit_ns, cudaStream_t stream);

// ---------------------------------------------------------------- attention backward
// (swa_bwd.cu). q | k and v^T as the forward left them, dO = d_attn [B][S][H] bf16, the
// forward's lse and delta[b, head, i] = dO_i . O_i ([B * nh, lse_ld] fp32, lse_ld a multiple
// of 64 >= S). Adds dq (unscaled)
// into dq_acc [T, H] fp32 (zeroed by the caller) and writes dk (scaled by 1/sqrt(dh)) and
// dv as bf16 into dz columns [H, 2H) and [2H, 3H) (row stride ldz). dh == 128.
struct SwaBwdParams {
  int B, S, H, nh, dh, window;
  float scale_log2;  // log2(e) / sqrt(dh)
  float scale;       // 1 / sqrt(dh)
  const float* lse;
  const float* delta;
  int64_t lse_ld;
  float* dq_acc;
  __nv_bfloat16* dz;
  int64_t ldz;
};
// tmQ: q|k in boxes of 64 columns x 64 rows; tmK: the same in boxes of 64 x 128 rows;
// tmVT: v^T in boxes of 64 keys x dh rows; tmDO: d_attn [B][S][H] in boxes of 64 x 64;
// tmDQ: dq_acc [B][S][H] fp32, unswizzled boxes of 32 columns x 64 rows.
cudaError_t launch_swa_bwd(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmVT, const CUtensorMap& tmDO,
                           const CUtensorMap& tmDQ, const SwaBwdParams& p, int* status,
                           uint64_t limit_ns, cudaStream_t stream);

// ---------------------------------------------------------------- backward helpers
// (bwd_aux.cu)
// delta[(b * nh + head) * lse_ld + s] = sum_d dO[t, head*dh + d] * O[t, head*dh + d],
// t = b*S + s (dO: [T, H] bf16; O: the attention output, row stride o_ld).
cudaError_t launch_attn_delta(const __nv_bfloat16* dO, const __nv_bfloat16* O, int64_t o_ld,
                              int B, int S, int nh, int dh, float* delta, int64_t lse_ld,
                              cudaStream_t stream);
// dz[t * ldz + c] = bf16(dq_acc[t * H + c] * scale), c < H.
cudaError_t launch_dq_to_bf16(const float* dq_acc, int64_t T, int H, float scale,
                              __nv_bfloat16* dz, int64_t ldz, cudaStream_t stream);
// Normalisation backward, per row: dx = dy + rstd (g - mean g - xhat mean(g xhat)), g =
// dxn * gamma, xhat = (x - mu) rstd (RMSNorm when rms: mu = 0, no mean g term); also the
// row statistics (mu, rstd) for the parameter gradients. x, dy, dx bf16 [T, H]; dxn fp32.
cudaError_t launch_norm_bwd(int64_t T, int H, const __nv_bfloat16* x,
                            const __nv_bfloat16* gamma, const float* dxn,
                            const __nv_bfloat16* dy, float eps, bool rms, __nv_bfloat16* dx,
                            float2* stats, cudaStream_t stream);
constexpr int kColBlocks = 32;  // row blocks of the column reductions
// dgamma[c] (+)= sum_r dxn[r,c] xhat[r,c], dbeta[c] (+)= sum_r dxn[r,c] (dbeta may be null),
// through partials [2][kColBlocks][H] fp32, rows summed in a fixed order.
cudaError_t launch_norm_param_grads(int64_t T, int H, const __nv_bfloat16* x, const float* dxn,
                                    const float2* stats, float* partials, float* dgamma,
                                    float* dbeta, bool accumulate, cudaStream_t stream);
// Column sums of a bf16 [rows, N] matrix (row stride ld), through partials
// [kColBlocks][N] fp32, rows summed in a fixed order: column c < split goes to out0[c],
// column c >= split to out1[c - split], or with glu_F > 0 to out1 at the SwiGLU
// de-interleave of c - split (group t = (c - split) / 32, i = (c - split) % 32: gate
// feature 16t + i for i < 16, else up feature glu_F + 16t + i - 16). A null out is skipped;
// accumulate adds to it.
cudaError_t launch_col_sums(const __nv_bfloat16* m, int64_t rows, int64_t N, int64_t ld,
                            float* partials, float* out0, float* out1, int64_t split,
                            int64_t glu_F, bool accumulate, cudaStream_t stream);

// ---------------------------------------------------------------- packing (pack.cu)
// out[c * ld_out + r] = in[r * ld_in + c] for r < rows, c < cols; with out_f16 the bf16
// value is converted to fp16 (kStatusRange in *status if it is beyond the fp16 range).
// glu_F > 0 (cols == 2 glu_F): output row c takes input column 16t + i of the gate half
// or of the up half, t = c / 32, i = c % 32 (< 16: gate, else up, i - 16) -- the SwiGLU
// interleave of the first GEMM's B operand.
cudaError_t launch_transpose(const __nv_bfloat16* in, int64_t rows, int64_t cols, int64_t ld_in,
                             void* out, int64_t ld_out, bool out_f16, int64_t glu_F, int* status,
                             cudaStream_t stream);
// bias1[3H + F] = [b_qkv | b1] (0 where absent; with glu b1 is [2F] and is interleaved like
// W1's rows, bias1 [3H + 2F]); bias2[H] = b_o + b2; bias_o[H] = b_o and bias_2[H] = b2
// apart (the serial block adds them in two different GEMMs).
cudaError_t launch_bias_prep(const __nv_bfloat16* b_qkv, const __nv_bfloat16* b1,
                             const __nv_bfloat16* b_o, const __nv_bfloat16* b2, int H, int F,
                             bool glu, float* bias1, float* bias2, float* bias_o, float* bias_2,
                             cudaStream_t stream);

// ---------------------------------------------------------------- FP8 (quant.cu, pack.cu)
// Per-row current scaling to E4M3 (fixed fp32 steps: amax, inv = 448 / amax, scale =
// amax / 448, code = E4M3(x * inv) rounded to nearest even, saturating). x: bf16 [rows,
// cols] with row stride ld_in; codes: [rows, cols] bytes with row stride ld_out; scales:
// [rows] fp32. cols, ld_in, ld_out multiples of 8.
cudaError_t launch_quantize_rows_e4m3(const __nv_bfloat16* x, int64_t rows, int64_t cols,
                                      int64_t ld_in, uint8_t* codes, int64_t ld_out,
                                      float* scales, cudaStream_t stream);
// amax[c] = max(amax[c], max_r |w[r, c]|) for a bf16 [rows, cols] matrix, row stride ld
// (amax must start at 0 or hold an earlier partial result).
cudaError_t launch_col_amax(const __nv_bfloat16* w, int64_t rows, int64_t cols, int64_t ld,
                            float* amax, cudaStream_t stream);
// As launch_transpose, writing the E4M3 code of each value scaled by 448 / amax of its
// output row's source column (per-output-channel current scaling).
cudaError_t launch_transpose_e4m3(const __nv_bfloat16* in, int64_t rows, int64_t cols,
                                  int64_t ld_in, uint8_t* out, int64_t ld_out, int64_t glu_F,
                                  const float* amax, cudaStream_t stream);
// scales[c] = amax[source column of output row c] / 448.
cudaError_t launch_amax_to_scales(const float* amax, int64_t n, int64_t glu_F, float* scales,
                                  cudaStream_t stream);
// LayerNorm (beta != null) or RMSNorm of bf16 / fp32 rows straight to E4M3 codes with
// per-row current scaling: out [rows, H] bytes, scales [rows] fp32.
cudaError_t launch_layernorm_e4m3(int64_t rows, int H, const void* x, bool x_f32,
                                  const __nv_bfloat16* gamma, const __nv_bfloat16* beta,
                                  float eps, uint8_t* out, float* scales, cudaStream_t stream);

// ---------------------------------------------------------------- self-test (gemm.cu)
cudaError_t launch_wait_probe(uint64_t limit_ns, int* status, cudaStream_t stream);

}  // namespace pb
