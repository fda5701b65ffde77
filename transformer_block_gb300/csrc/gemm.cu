// gemm.cu — persistent warp-specialised tcgen05 GEMM on CTA pairs, D = A * B^T, with the
// epilogues of the parallel block's two linear steps fused in:
//   * [q | k | v | h] = LN(x) [Wqkv | W1], GeLU(h) applied in the epilogue (the fused
//     QKV projection of the MegaScale reading notes, section 1.3, widened to the MLP's
//     first linear because both read the same LN output in eq. (4));
//   * y = x + [attn | GeLU(h)] [Wo ; W2] (+ bias), the residual sum of eq. (4) applied
//     in the epilogue of the one GEMM that computes both branch outputs.
//
// Two CTAs of a cluster (one per SM) compute one 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256): each CTA loads, by TMA, its own 128 rows of A and
// its half (128 rows) of the tile's 256 rows of B, 64 elements of K per stage, into a
// 6-stage ring, and holds its 128 x 256 half of the fp32 accumulator in its tensor
// memory (double-buffered, 2 x 256 columns, so the epilogue of one tile overlaps the
// main loop of the next).
//   warp 0     TMA producer (both CTAs); every copy of the pair completes on the even
//              CTA's stage barrier (the pair form of the TMA load), so the MMA issuer
//              waits on one barrier per stage
//   warp 1     even CTA: the MMA-issuing thread; both: tensor-memory owner
//   warps 2-5  epilogue, one TMEM lane quadrant each (warp w reads lanes 32*(w%4)..+31)
// MMA completion is multicast to both CTAs' barriers. Pair tiles are handed out
// round-robin over the clusters, M fastest, so clusters running at the same time share
// B tiles in L2.
#include <atomic>
#include <chrono>
#include <random>

#include "kernels.h"
#include "ptx.cuh"

namespace pb {
namespace {

constexpr int BM = kGemmBM;       // output rows per CTA
constexpr int PM = 2 * kGemmBM;   // output rows per CTA pair
constexpr int BN = kGemmBN;       // output columns per pair tile
constexpr int BK = kGemmBK;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB: this CTA's rows of A (one M tile)
constexpr int B_BYTES = (BN / 2) * BK * 2;  // 16 KB: this CTA's half of B
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
// Per epilogue warp, a 32 x 32 fp32 chunk (rows padded to 33 words: conflict-free both
// ways) for the coalesced gradient stores.
constexpr int STAGE_PITCH = 33;
static_assert(4 * 32 * STAGE_PITCH * 4 >= 4 * 4096, "four warps' two 2 KB store buffers");

// Shared-memory geometry for MT 256-row M tiles per CTA pair and work unit. MT = 1: a
// 256 x 256 tile, six stages of A and B, the accumulator double-buffered in tensor memory
// (2 x 256 columns). MT = 2: a 512 x 256 unit whose two M tiles share every B stage (a
// quarter less operand traffic per FLOP), four stages of two A tiles and B, one 256-column
// accumulator per M tile (not double-buffered).
template <int MT>
struct Geo {
  static_assert(MT == 1 || MT == 2, "one or two M tiles per unit");
  static constexpr int STAGES = MT == 2 ? 4 : 6;
  static constexpr int STAGE_BYTES = MT * A_BYTES + B_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  // 1024-byte aligned: the forward epilogues' TMA-store buffers (64-byte swizzle) live here
  static constexpr size_t EPI_STAGE_OFF =
      (size_t(STAGES) * STAGE_BYTES + 8 * NUM_BARS + 16 + 1023) / 1024 * 1024;
  static constexpr size_t SMEM_BYTES = 1024 + EPI_STAGE_OFF + 4 * 32 * STAGE_PITCH * 4;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of the GEMM");
};

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The GeLU epilogues take erf from Abramowitz & Stegun, Handbook of Mathematical
// Functions, 7.1.26: for x >= 0, 1 - erf(x) = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5)
// exp(-x^2) with t = 1 / (1 + p x), |error| <= 1.5e-7 (about 5e-7 in fp32; GeLU then stays
// within 2e-4 of its value where |GeLU| > 1e-3, a tenth of a bf16 step). For a packed pair
// z: q = 1 - erf(|z| / sqrt 2) and e = exp(-z^2 / 2).
__device__ __forceinline__ void erfc_terms(float z0, float z1, uint64_t& q, uint64_t& e) {
  constexpr float kP = 0.3275911f, kA1 = 0.254829592f, kA2 = -0.284496736f,
                  kA3 = 1.421413741f, kA4 = -1.453152027f, kA5 = 1.061405429f;
  constexpr float kRsqrt2 = 0.70710678118654752f, kLog2e = 1.4426950408889634f;
  const uint64_t x = f2(fabsf(z0) * kRsqrt2, fabsf(z1) * kRsqrt2);
  float d0, d1;
  f2_split(f2_fma(x, f2(kP, kP), f2(1.f, 1.f)), d0, d1);
  const uint64_t t = f2(rcp_approx(d0), rcp_approx(d1));
  uint64_t poly = f2_fma(t, f2(kA5, kA5), f2(kA4, kA4));
  poly = f2_fma(poly, t, f2(kA3, kA3));
  poly = f2_fma(poly, t, f2(kA2, kA2));
  poly = f2_fma(poly, t, f2(kA1, kA1));
  poly = f2_mul(poly, t);
  float g0, g1;
  f2_split(f2_mul(f2_mul(x, x), f2(-kLog2e, -kLog2e)), g0, g1);
  e = f2(ex2_approx(g0), ex2_approx(g1));
  q = f2_mul(poly, e);
}

// GeLU(z) = z Phi(z) = z (1 + erf(z / sqrt 2)) / 2 on a packed pair: with q as above,
// z - z q / 2 for z >= 0 and z q / 2 below.
__device__ __forceinline__ void gelu_pair(float& z0, float& z1) {
  uint64_t q, e;
  erfc_terms(z0, z1, q, e);
  float h0, h1;
  f2_split(f2_mul(f2_mul(f2(z0, z1), f2(0.5f, 0.5f)), q), h0, h1);
  z0 = z0 >= 0.f ? z0 - h0 : h0;
  z1 = z1 >= 0.f ? z1 - h1 : h1;
}

// d0, d1 times GeLU'(z) = Phi(z) + z phi(z), phi the standard normal density
// exp(-z^2 / 2) / sqrt(2 pi), with Phi from the same erf terms.
__device__ __forceinline__ void gelu_grad_pair(float& d0, float& d1, float z0, float z1) {
  constexpr float kRsqrt2pi = 0.39894228040143268f;
  uint64_t q, e;
  erfc_terms(z0, z1, q, e);
  float q0, q1;
  f2_split(q, q0, q1);
  const float p0 = z0 >= 0.f ? 1.f - 0.5f * q0 : 0.5f * q0;
  const float p1 = z1 >= 0.f ? 1.f - 0.5f * q1 : 0.5f * q1;
  float g0, g1;
  f2_split(f2_fma(f2(z0 * kRsqrt2pi, z1 * kRsqrt2pi), e, f2(p0, p1)), g0, g1);
  d0 *= g0;
  d1 *= g1;
}

template <int N>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16* src, float (&v)[N]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < N / 8; ++q) {
    const uint4 u = s4[q];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      v[8 * q + 2 * e] = f.x;
      v[8 * q + 2 * e + 1] = f.y;
    }
  }
}

// n fp32 values to dst (16-byte aligned), added to what is there when accumulate.
template <int N>
__device__ __forceinline__ void store_f32(float* dst, const float* v, bool accumulate) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < N / 4; ++q) {
    float4 o = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    if (accumulate) {
      const float4 a = d[q];
      o.x += a.x;
      o.y += a.y;
      o.z += a.z;
      o.w += a.w;
    }
    d[q] = o;
  }
}

// 32 bytes from one lane in one instruction; p must be 32-byte aligned. A warp's row-wise
// stores touch 32 rows per instruction, and each instruction costs the L1 data path (shared
// with the TMA writes and the MMAs' operand reads of the main loop) about one pass per row
// it touches, so halving the instructions per row halves that cost.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// N consecutive 16-bit values (N a multiple of 8) from one lane: 32-byte stores where dst
// is 32-byte aligned, else 16-byte stores.
template <int N>
__device__ __forceinline__ void store_words16(void* dst, const uint32_t (&w)[N / 2]) {
  if ((reinterpret_cast<uintptr_t>(dst) & 31) == 0 && N % 16 == 0) {
#pragma unroll
    for (int q = 0; q < N / 16; ++q) st_global_v8(static_cast<char*>(dst) + 32 * q, w + 8 * q);
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < N / 8; ++q) d[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
}

template <bool F16>
__device__ __forceinline__ void store_row32(void* dst, const float (&v)[32]) {
  uint32_t w[16];
#pragma unroll
  for (int e = 0; e < 16; ++e)
    w[e] = F16 ? pack_f16x2(v[2 * e], v[2 * e + 1]) : pack_bf16x2(v[2 * e], v[2 * e + 1]);
  store_words16<32>(dst, w);
}

template <bool F16>
__device__ __forceinline__ void store_row16(void* dst, const float (&v)[16]) {
  uint32_t w[8];
#pragma unroll
  for (int e = 0; e < 8; ++e)
    w[e] = F16 ? pack_f16x2(v[2 * e], v[2 * e + 1]) : pack_bf16x2(v[2 * e], v[2 * e + 1]);
  store_words16<16>(dst, w);
}

__device__ __forceinline__ void store_row32_f32(float* dst, const float (&v)[32]) {
  if ((reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) st_global_v8(dst + 8 * q, reinterpret_cast<const uint32_t*>(v + 8 * q));
  } else {
    float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q) d[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
}

// Transposes 16-byte pieces inside each group of 4 lanes: lane 4g + k, holding pieces
// 0..3 of row 4g + k in w (4 words each), ends up holding piece k of row 4g + i as piece i.
// Two exchange rounds: the off-diagonal 2 x 2 blocks of pieces with lane ^ 2, then the
// off-diagonal pieces inside each block with lane ^ 1.
__device__ __forceinline__ void transpose_pieces4(uint32_t (&w)[16]) {
  const int k = int(threadIdx.x & 3);
  const bool hi = (k & 2) != 0, odd = (k & 1) != 0;
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t y = __shfl_xor_sync(0xffffffffu, hi ? w[4 * s + e] : w[4 * (2 + s) + e], 2);
      if (hi)
        w[4 * s + e] = y;
      else
        w[4 * (2 + s) + e] = y;
    }
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t y =
          __shfl_xor_sync(0xffffffffu, odd ? w[4 * (2 * c) + e] : w[4 * (2 * c + 1) + e], 1);
      if (odd)
        w[4 * (2 * c) + e] = y;
      else
        w[4 * (2 * c + 1) + e] = y;
    }
}

// Warp-wide: the warp's 32 x 32 block of 16-bit values (lane l holds row l's 32 values as
// 16 words) to rows [0, nrows) at base (row stride ld_bytes). After the transpose each
// store instruction writes 8 rows x 64 contiguous bytes instead of 32 rows x 16 bytes:
// a quarter of the L1 data-path passes, which the main loop's TMA writes and operand
// reads share.
__device__ __forceinline__ void store_rows32_16b(char* base, int64_t ld_bytes, int nrows,
                                                 uint32_t (&w)[16]) {
  transpose_pieces4(w);
  const int lane = int(threadIdx.x & 31), k = lane & 3, g = lane >> 2;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * g + i;
    if (r < nrows)
      *reinterpret_cast<uint4*>(base + r * ld_bytes + 16 * k) =
          make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
}

template <bool F16>
__device__ __forceinline__ void pack_words16(const float (&v)[32], uint32_t (&w)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e)
    w[e] = F16 ? pack_f16x2(v[2 * e], v[2 * e + 1]) : pack_bf16x2(v[2 * e], v[2 * e + 1]);
}

// A warp's TMA stores: two 2 KB staging buffers (32 rows of 64 bytes) used in turn.
struct StoreStage {
  uint32_t base;  // shared-memory address of the warp's buffers
  uint32_t n;     // stores issued so far
};

// Warp-wide: the warp's 32 rows (lane l holds row row0 + l as 16 words of 16-bit pairs) of
// the 32 columns at col0 to the tensor of `tm`, by one TMA store. Rows past the tensor's
// end are dropped by the copy.
__device__ __forceinline__ void tma_store_rows32(StoreStage& ss, const CUtensorMap* tm, int row0,
                                                 int col0, int M, const uint32_t (&w)[16]) {
  if (row0 >= M) return;  // the whole warp is past the last row (uniform in the warp)
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t buf = ss.base + (ss.n & 1u) * 2048u;
  if (ss.n >= 2) {  // the buffer's previous store (two ago) must have read it
    if (lane == 0) bulk_wait_read_1();
    __syncwarp();
  }
  // 64-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ ((r >> 1) & 3), which
  // also spreads the warp's writes over all banks
  const uint32_t rb = buf + lane * 64u, sw = (lane >> 1) & 3u;
#pragma unroll
  for (uint32_t j = 0; j < 4; ++j)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rb + ((j ^ sw) << 4)),
                 "r"(w[4 * j]), "r"(w[4 * j + 1]), "r"(w[4 * j + 2]), "r"(w[4 * j + 3])
                 : "memory");
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tm, buf, col0, row0);
    bulk_commit();
  }
  ++ss.n;
}

// Epilogue of 32 consecutive columns [col0, col0 + 32) of one output row. Called by all 32
// lanes of a warp together, lane l holding row `row` = the warp's first row + l: the plain
// store is warp-wide (the fused epilogues store row-wise per lane, where the transpose's
// extra instructions cost more than its fewer store passes save).
template <int KIND>
__device__ __forceinline__ void epilogue32(const EpiParams& ep, int row, int col0, float (&v)[32],
                                           StoreStage& ss) {
  if (KIND == kEpiStore) {
    const int row0 = row - int(threadIdx.x & 31);
    const int nrows = ep.M - row0 < 32 ? ep.M - row0 : 32;
    if (nrows <= 0) return;
    if (ep.scale_a != nullptr) {  // FP8 operands: undo the row and channel scales
      const float sa = row < ep.M ? ep.scale_a[row] : 0.f;
      const float4* s4 = reinterpret_cast<const float4*>(ep.scale_b + col0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 sb = __ldg(s4 + q);
        v[4 * q + 0] *= sa * sb.x;
        v[4 * q + 1] *= sa * sb.y;
        v[4 * q + 2] *= sa * sb.z;
        v[4 * q + 3] *= sa * sb.w;
      }
    }
    uint32_t w[16];
    pack_words16<false>(v, w);
    store_rows32_16b(reinterpret_cast<char*>(ep.c + int64_t(row0) * ep.ldc + col0),
                     int64_t(ep.ldc) * 2, nrows, w);
    return;
  }
  // With TMA stores every lane takes part in the warp's copies, rows past M included (the
  // copy drops them); otherwise a lane past M has nothing to do.
  const bool tma = ep.tma_store && (KIND == kEpiResidual || (KIND == kEpiBlockIn && !ep.glu));
  if (row >= ep.M && !tma) return;
  const bool live = row < ep.M;
  if (ep.scale_a != nullptr) {  // FP8 operands: undo the row and channel scales
    const float sa = live ? ep.scale_a[row] : 0.f;
    const float4* s4 = reinterpret_cast<const float4*>(ep.scale_b + col0);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 sb = __ldg(s4 + q);
      v[4 * q + 0] *= sa * sb.x;
      v[4 * q + 1] *= sa * sb.y;
      v[4 * q + 2] *= sa * sb.z;
      v[4 * q + 3] *= sa * sb.w;
    }
  }
  if (KIND != kEpiStore && ep.bias != nullptr) {
    const float4* b4 = reinterpret_cast<const float4*>(ep.bias + col0);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float4 b = __ldg(b4 + q);
      v[4 * q + 0] += b.x;
      v[4 * q + 1] += b.y;
      v[4 * q + 2] += b.z;
      v[4 * q + 3] += b.w;
    }
  }
  if (KIND == kEpiBlockIn) {
    const int H = ep.H;
    const int cc = col0 + ep.col_base;  // column of [q | k | v | h]
    const int row0 = row - int(threadIdx.x & 31);
    if (cc < 2 * H) {  // q | k
      if (tma) {
        uint32_t w[16];
        pack_words16<false>(v, w);
        tma_store_rows32(ss, &ep.tm_out0, row0, cc, ep.M, w);
      } else {
        store_row32<false>(ep.qk + int64_t(row) * (2 * H) + cc, v);
      }
    } else if (cc < 3 * H) {  // v, stored transposed per (sequence, head)
      if (!live) return;
      const int c = cc - 2 * H;
      const int head = c / ep.dh, d0 = c - head * ep.dh;
      const int b = row / ep.S, s = row - b * ep.S;
      __nv_bfloat16* dst =
          ep.vt + (int64_t(b * ep.nh + head) * ep.dh + d0) * ep.seq_pad + s;
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[int64_t(i) * ep.seq_pad] = __float2bfloat16_rn(v[i]);
    } else {
      if (ep.hpre != nullptr && live)  // training forward: keep h for the backward
        store_row32<false>(ep.hpre + int64_t(row) * (ep.N + ep.col_base - 3 * H) + (cc - 3 * H),
                           v);
      if (ep.glu) {
        // [gate | up] of 16 MLP features -> silu(gate) * up, next to the attention output
        // in the second GEMM's A operand
        float o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = v[i] * rcp_approx(1.0f + __expf(-v[i])) * v[16 + i];
        const int64_t off = int64_t(row) * (H + ep.F) + H + (cc - 3 * H) / 2;
        if (ep.act_f16) {
          bool bad = false;
#pragma unroll
          for (int i = 0; i < 16; ++i) bad |= !(fabsf(o[i]) <= kF16Max);
          if (bad) report_range(ep.status);
          store_row16<true>(static_cast<__half*>(ep.act) + off, o);
        } else {
          store_row16<false>(static_cast<__nv_bfloat16*>(ep.act) + off, o);
        }
      } else {  // h -> GeLU(h), next to the attention output in the second GEMM's A operand
#pragma unroll
        for (int i = 0; i < 32; i += 2) gelu_pair(v[i], v[i + 1]);
        const int64_t off = int64_t(row) * (H + ep.F) + H + (cc - 3 * H);
        if (ep.act_f16) {
          bool bad = false;
#pragma unroll
          for (int i = 0; i < 32; ++i) bad |= live && !(fabsf(v[i]) <= kF16Max);
          if (bad) report_range(ep.status);
        }
        if (tma) {
          uint32_t w[16];
          if (ep.act_f16)
            pack_words16<true>(v, w);
          else
            pack_words16<false>(v, w);
          tma_store_rows32(ss, &ep.tm_out1, row0, H + (cc - 3 * H), ep.M, w);
        } else if (ep.act_f16) {
          store_row32<true>(static_cast<__half*>(ep.act) + off, v);
        } else {
          store_row32<false>(static_cast<__nv_bfloat16*>(ep.act) + off, v);
        }
      }
    }
  } else if (KIND == kEpiBwdAct) {
    const int H = ep.H;
    if (col0 < H) {  // d_attn = dy Wo^T
      store_row32<false>(ep.d_attn + int64_t(row) * H + col0, v);
      return;
    }
    const int f0 = col0 - H;  // MLP feature of the first column
    const __nv_bfloat16* hp = ep.hpre + int64_t(row) * (ep.glu ? 2 * ep.F : ep.F);
    __nv_bfloat16* dz = ep.dz + int64_t(row) * ep.ldz + 3 * H;
    if (!ep.glu) {
      float h[32];
      load_bf16<32>(hp + f0, h);
#pragma unroll
      for (int i = 0; i < 32; i += 2) gelu_grad_pair(v[i], v[i + 1], h[i], h[i + 1]);
      store_row32<false>(dz + f0, v);
    } else {
      // features f0 .. f0 + 31 are the interleave groups f0 / 16 and f0 / 16 + 1: W1cat
      // columns [2 f0, 2 f0 + 64), 16 gate then 16 up values each
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int c = 2 * f0 + 32 * half;
        float g[16], u[16], dg[16], du[16];
        load_bf16<16>(hp + c, g);
        load_bf16<16>(hp + c + 16, u);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float d = v[16 * half + i];
          const float sg = rcp_approx(1.0f + __expf(-g[i]));
          du[i] = d * g[i] * sg;
          dg[i] = d * u[i] * sg * (1.0f + g[i] * (1.0f - sg));
        }
        store_row16<false>(dz + c, dg);
        store_row16<false>(dz + c + 16, du);
      }
    }
  } else if (KIND == kEpiGrad) {
    if (row >= ep.split_row) {
      store_f32<32>(ep.g1 + int64_t(row - ep.split_row) * ep.ld1 + col0, v, ep.accumulate);
    } else if (col0 >= ep.split_col) {
      const int c = col0 - ep.split_col;
      float* base = ep.g1 + int64_t(row) * ep.ld1;
      if (ep.glu) {  // undo the W1cat interleave: 16 gate then 16 up features
        store_f32<16>(base + c / 2, v, ep.accumulate);
        store_f32<16>(base + ep.F + c / 2, v + 16, ep.accumulate);
      } else {
        store_f32<32>(base + c, v, ep.accumulate);
      }
    } else {
      store_f32<32>(ep.g0 + int64_t(row) * ep.ld0 + col0, v, ep.accumulate);
    }
  } else {  // kEpiResidual: y = D + bias + x
    const int64_t off = int64_t(live ? row : 0) * ep.N + col0;
    if (ep.resid_f32) {
      const float4* x4 = reinterpret_cast<const float4*>(static_cast<const float*>(ep.resid) + off);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 f = x4[q];
        v[4 * q + 0] += f.x;
        v[4 * q + 1] += f.y;
        v[4 * q + 2] += f.z;
        v[4 * q + 3] += f.w;
      }
    } else {
      const uint4* x4 =
          reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(ep.resid) + off);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 u = x4[q];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
          float2 f = __bfloat1622float2(p);
          v[8 * q + 2 * e] += f.x;
          v[8 * q + 2 * e + 1] += f.y;
        }
      }
    }
    if (tma) {
      uint32_t w[16];
      pack_words16<false>(v, w);
      tma_store_rows32(ss, &ep.tm_out0, row - int(threadIdx.x & 31), col0, ep.M, w);
    } else if (ep.y_f32) {
      store_row32_f32(static_cast<float*>(ep.y) + off, v);
    } else {
      store_row32<false>(static_cast<__nv_bfloat16*>(ep.y) + off, v);
    }
  }
}

// Destination of columns [col0 + cq, col0 + cq + 4) of gradient row `row` (kEpiGrad).
__device__ __forceinline__ float* grad_dst(const EpiParams& ep, int row, int col0, int cq) {
  if (row >= ep.split_row) return ep.g1 + int64_t(row - ep.split_row) * ep.ld1 + col0 + cq;
  if (col0 >= ep.split_col) {
    const int c = col0 - ep.split_col;
    float* base = ep.g1 + int64_t(row) * ep.ld1;
    if (ep.glu)  // undo the W1cat interleave: 16 gate then 16 up features
      return cq < 16 ? base + c / 2 + cq : base + ep.F + c / 2 + (cq - 16);
    return base + c + cq;
  }
  return ep.g0 + int64_t(row) * ep.ld0 + col0 + cq;
}

// kEpiGrad for a warp's 32 rows [row0, row0 + 32) x 32 columns: the chunk goes through
// shared memory so that each store instruction writes four whole 128-byte rows (eight
// lanes per row) instead of 32 rows' 16-byte pieces.
__device__ __forceinline__ void grad_store_warp(const EpiParams& ep, int row0, int col0,
                                                const float (&v)[32], float* stage) {
  const int lane = int(threadIdx.x & 31);
#pragma unroll
  for (int i = 0; i < 32; ++i) stage[lane * STAGE_PITCH + i] = v[i];
  __syncwarp();
  const int cq = (lane & 7) * 4;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int r = 4 * it + (lane >> 3);
    const int row = row0 + r;
    if (row < ep.M) {
      const float* sr = stage + r * STAGE_PITCH + cq;
      float4 o = make_float4(sr[0], sr[1], sr[2], sr[3]);
      float4* dst = reinterpret_cast<float4*>(grad_dst(ep, row, col0, cq));
      if (ep.accumulate) {
        const float4 a = *dst;
        o.x += a.x;
        o.y += a.y;
        o.z += a.z;
        o.w += a.w;
      }
      *dst = o;
    }
  }
  __syncwarp();
}

// The work of one CTA pair: first whole units t = cluster, cluster + clusters, ... below
// dp_tiles (a unit is mt M tiles of 256 rows by 256 columns), then its contiguous share
// [cluster * W, (cluster + 1) * W) of the linearised (tile, k-block) iterations of the
// sk_tiles stream-K tiles that follow them: the 256-row M tiles of the remaining units.
struct Sched {
  int num_m, num_n, num_kb;  // num_m counts units of mt x 256 rows
  int cluster, clusters;
  int dp_tiles, sk_tiles, W;
  int mt, group;             // M tiles per unit; units per rasterisation group
};

struct SkParams {
  int dp_tiles, sk_tiles, W;
  float* partials;  // [kSkMaxClusters][2][128][256]
  uint64_t* flags;  // [kSkMaxClusters][2][4]
  uint64_t epoch;
};

struct Unit {
  int row0, tn;  // first row (of the pair) and column block
  int mt;        // M tiles in this unit (a stream-K tile has one)
  int ts;        // stream-K tile index, -1 for a whole unit
  int kb0, kb1;
};

// Unit index -> (unit row block, column block). Units are ordered in groups of `group`
// row blocks (kGroupM pair-rows of 256 in all), M fastest inside a group, so the CTA pairs
// running at the same time cover a compact block of about 2048 rows x (pairs / group)
// columns and share both their A rows and their B columns in L2.
constexpr int kGroupM = 8;
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group, int& m,
                                            int& n) {
  const int per_group = group * num_n;
  const int g = tile / per_group;
  const int first_m = g * group;
  const int gm = min(group, num_m - first_m);
  const int r = tile - g * per_group;
  m = first_m + r % gm;
  n = r / gm;
}

struct UnitIter {
  int t;
  int64_t it, it_end;
  __device__ explicit UnitIter(const Sched& s)
      : t(s.cluster),
        it(int64_t(s.cluster) * s.W),
        it_end(min(int64_t(s.cluster + 1) * s.W, int64_t(s.sk_tiles) * s.num_kb)) {}
  __device__ bool next(const Sched& s, Unit& u) {
    int tm, tn;
    if (t < s.dp_tiles) {
      tile_coords(t, s.num_m, s.num_n, s.group, tm, tn);
      u = Unit{tm * s.mt * 2 * kGemmBM, tn, s.mt, -1, 0, s.num_kb};
      t += s.clusters;
      return true;
    }
    if (it >= it_end) return false;
    const int ts = int(it / s.num_kb);
    const int kb0 = int(it - int64_t(ts) * s.num_kb);
    const int kb1 = int(min(int64_t(s.num_kb), int64_t(kb0) + (it_end - it)));
    tile_coords(s.dp_tiles + ts / s.mt, s.num_m, s.num_n, s.group, tm, tn);
    u = Unit{(tm * s.mt + ts % s.mt) * 2 * kGemmBM, tn, 1, ts, kb0, kb1};
    it += kb1 - kb0;
    return true;
  }
};

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

template <int KIND, int OP, int LAYOUT, int MT>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                int K, const __grid_constant__ EpiParams ep, const SkParams sk, int* status,
                uint64_t limit_ns) {
  static_assert(MT == 1 || LAYOUT == kKK, "two M tiles per unit: K-major operands only");
  constexpr int STAGES = Geo<MT>::STAGES, STAGE_BYTES = Geo<MT>::STAGE_BYTES;
  constexpr int NUM_BARS = Geo<MT>::NUM_BARS;
  constexpr size_t EPI_STAGE_OFF = Geo<MT>::EPI_STAGE_OFF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(STAGES) * STAGE_BYTES);
  // full: both CTAs' copies of a stage landed (used in the even CTA only: the odd CTA's
  // copies complete on the even CTA's barrier). empty: the pair's MMAs are done reading.
  const uint32_t full0 = smem_u32(bars);                   // [STAGES]
  const uint32_t empty0 = smem_u32(bars + STAGES);         // [STAGES]
  const uint32_t tfull0 = smem_u32(bars + 2 * STAGES);     // [2] accumulator ready
  const uint32_t tempty0 = smem_u32(bars + 2 * STAGES + 2);  // [2] accumulator drained (x8)
  const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t warp = warp_id(), lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 8);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, status, limit_ns};
  // Teardown waits for the CTA's own copies and MMAs get at least a second, whatever the
  // wait limit, so shared and tensor memory are never released under them.
  const uint64_t drain_ns = limit_ns > kDrainFloorNs ? limit_ns : kDrainFloorNs;

  Sched sc;
  sc.num_m = (ep.M + MT * PM - 1) / (MT * PM);
  sc.num_n = (ep.N + BN - 1) / BN;
  sc.mt = MT;
  sc.group = kGroupM / MT;
  constexpr int BKE = OP == kOpE4m3 ? kGemmBK8 : BK;  // K elements per stage (128 bytes)
  constexpr bool AMN = (LAYOUT & kMK) != 0, BMN = (LAYOUT & kKM) != 0;
  static_assert(!(AMN || BMN) || OP != kOpE4m3, "MN-major operands are 16-bit");
  sc.num_kb = (K + BKE - 1) / BKE;  // a ragged last block is zero filled by TMA
  sc.cluster = int(blockIdx.x) >> 1;
  sc.clusters = int(gridDim.x) >> 1;
  sc.dp_tiles = sk.dp_tiles;
  sc.sk_tiles = sk.sk_tiles;
  sc.W = sk.W;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      uint32_t last_par[STAGES];
      uint32_t used = 0;
      // The stage's full barrier in the even CTA, as a cluster address.
      const uint32_t full_pair0 = mapa_shared(full0, 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      UnitIter ui(sc);
      Unit u;
      while (ok && ui.next(sc, u)) {
        const int m0 = u.row0 + int(rank) * BM;
        const int n0 = u.tn * BN + int(rank) * (BN / 2);
        const uint32_t stage_tx = 2u * uint32_t(u.mt * A_BYTES + B_BYTES);  // both CTAs
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, wc, 1)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + size_t(stage) * STAGE_BYTES);
          // The even CTA announces both CTAs' bytes; copies that land before it does only
          // drive the transaction count below zero, and the phase cannot complete without
          // its arrival. The odd CTA reuses a stage only after the pair's MMAs read it, so
          // its copies always count toward the phase the MMA issuer waits for next.
          if (leader) mbar_arrive_expect_tx(full0 + 8 * stage, stage_tx);
          // K-major: one box of 128 rows x 64 K; MN-major: two boxes of 64 K-rows x 64
          // elements of M (or N), 8 KB apart
          if (AMN) {
            tma_load_2d_pair(sa, &tmA, full_pair0 + 8 * stage, m0, kb * BKE);
            tma_load_2d_pair(sa + A_BYTES / 2, &tmA, full_pair0 + 8 * stage, m0 + 64, kb * BKE);
          } else {
            // MT = 2: the unit's second M tile 256 rows below, in the stage's second A slot
            for (int g = 0; g < u.mt; ++g)
              tma_load_2d_pair(sa + g * A_BYTES, &tmA, full_pair0 + 8 * stage, kb * BKE,
                               m0 + g * PM);
          }
          if (BMN) {
            tma_load_2d_pair(sa + A_BYTES, &tmB, full_pair0 + 8 * stage, n0, kb * BKE);
            tma_load_2d_pair(sa + A_BYTES + B_BYTES / 2, &tmB, full_pair0 + 8 * stage, n0 + 64,
                             kb * BKE);
          } else {
            tma_load_2d_pair(sa + MT * A_BYTES, &tmB, full_pair0 + 8 * stage, kb * BKE, n0);
          }
          last_par[stage] = phase;
          used |= 1u << stage;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Every copy of the pair must land before either CTA exits: the even CTA waits for
      // its full barriers (which count the odd CTA's bytes too); the odd CTA is held at the
      // final cluster barrier until then.
      if (leader)
        for (int s = 0; s < STAGES; ++s)
          if (used & (1u << s)) mbar_wait_drain(full0 + 8 * s, last_par[s], drain_ns);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc = idesc_f32acc(PM, BN, OP != kOpBf16, AMN, BMN);
      // descriptor start-address step of one MMA (K = 16 or 32 elements, 32 bytes):
      // along a swizzled row (K-major) or two 1024-byte atoms on (MN-major), in 16 B units
      constexpr uint64_t kStepA = AMN ? 128 : 2, kStepB = BMN ? 128 : 2;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_par = 0;
      bool ok = true;
      UnitIter ui(sc);
      Unit u;
      while (ok && ui.next(sc, u)) {
        if (!mbar_wait(tempty0 + 8 * acc, acc_par ^ 1, wc, 2)) break;
        tc_fence_after();
        // MT = 1: accumulator acc of two; MT = 2: M tile g in columns [g * BN, (g + 1) * BN)
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, wc, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + size_t(stage) * STAGE_BYTES);
          const uint64_t da =
              AMN ? sdesc_mnmajor_sw128(sa, A_BYTES / 2) : sdesc_kmajor_sw128(sa);
          const uint64_t db = BMN ? sdesc_mnmajor_sw128(sa + A_BYTES, B_BYTES / 2)
                                  : sdesc_kmajor_sw128(sa + MT * A_BYTES);
          // four products of 32 bytes of K each: K = 16 (16-bit) or 32 (FP8) elements; with
          // MT = 2 each M tile's A slot against the shared B
          for (int g = 0; g < u.mt; ++g) {
            const uint32_t dt = MT == 2 ? tmem_base + uint32_t(g * BN) : d_tmem;
            const uint64_t dag = da + uint64_t((g * A_BYTES) >> 4);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if (OP == kOpE4m3)
                mma_f8kind_ss_pair(dt, dag + kStepA * k, db + kStepB * k, idesc,
                                   (kb > u.kb0) || k > 0);
              else
                mma_f16kind_ss_pair(dt, dag + kStepA * k, db + kStepB * k, idesc,
                                    (kb > u.kb0) || k > 0);
            }
          }
          mma_commit_pair(empty0 + 8 * stage, 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair(tfull0 + 8 * acc, 0x3);
        if (MT == 1) {
          acc ^= 1;
          if (acc == 0) acc_par ^= 1;
        } else {
          acc_par ^= 1;  // one accumulator set
        }
      }
      // Every MMA this thread issued (into both CTAs' tensor memory) must finish before
      // either CTA releases it.
      mma_commit_pair(drain_bar, 0x1);
      mbar_wait_drain(drain_bar, 0, drain_ns);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue warps
    const uint32_t quad = warp & 3;
    float* epi_stage = reinterpret_cast<float*>(smem + EPI_STAGE_OFF) +
                       (warp - 2) * 32 * STAGE_PITCH;
    // the same area as two 2 KB TMA-store buffers per warp (forward kinds only)
    StoreStage ss{smem_u32(smem + EPI_STAGE_OFF) + (warp - 2) * 4096u, 0u};
    int acc = 0;
    uint32_t acc_par = 0;
    UnitIter ui(sc);
    Unit u;
    bool ok = true;
    while (ok && ui.next(sc, u)) {
      if (!mbar_wait_warp(tfull0 + 8 * acc, acc_par, wc, 4)) break;
      tc_fence_after();
      for (int g = 0; g < u.mt; ++g) {  // MT = 2: the unit's two M tiles, one after the other
        const int m0 = u.row0 + g * PM + int(rank) * BM, n0 = u.tn * BN;
        const int row = m0 + int(quad * 32 + lane);
        const uint32_t taddr =
            tmem_base + ((quad * 32u) << 16) + uint32_t((MT == 2 ? g : acc) * BN);
        // This thread's row of a pair's partial tile ([2][128][256] fp32 per cluster).
        const size_t part_off = (size_t(rank) * 128 + quad * 32 + lane) * BN;
        if (u.kb0 > 0) {
          // A K segment that does not start at 0: leave the partial sums for the pair that
          // owns k-block 0 of this tile, then publish them (one flag per warp).
          float* dst = sk.partials + size_t(sc.cluster) * (2 * 128 * BN) + part_off;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(taddr + uint32_t(c * 32), r);
            tmem_ld_wait(r);
            float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              __stcg(d4 + q, make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                         __uint_as_float(r[4 * q + 2]),
                                         __uint_as_float(r[4 * q + 3])));
          }
          __threadfence();
          __syncwarp();
          if (lane == 0)
            st_release_u64(sk.flags + (size_t(sc.cluster) * 2 + rank) * 4 + quad, sk.epoch);
        } else {
          // K segment from 0: this pair finishes the tile. For a stream-K tile, the pairs
          // cluster+1 .. last computed its other K segments; wait for their partials.
          int last = sc.cluster;
          if (u.ts >= 0) last = int(((int64_t(u.ts) + 1) * sc.num_kb - 1) / sc.W);
          for (int c2 = sc.cluster + 1; ok && c2 <= last; ++c2) {
            const uint64_t* f = sk.flags + (size_t(c2) * 2 + rank) * 4 + quad;
            if (ld_acquire_u64(f) != sk.epoch) {
              const uint64_t t0 = globaltimer_ns();
              while (ld_acquire_u64(f) != sk.epoch) {
                __nanosleep(100);
                if (*abort_flag) {
                  ok = false;
                  break;
                }
                if (globaltimer_ns() - t0 > limit_ns) {
                  wait_give_up(wc, 7);
                  ok = false;
                  break;
                }
              }
            }
          }
          ok = __all_sync(0xffffffffu, ok);
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            const int col0 = n0 + c * 32;
            if (col0 >= ep.N) break;
            uint32_t r[32];
            tmem_ld32(taddr + uint32_t(c * 32), r);
            tmem_ld_wait(r);
            if (!ok) continue;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
            for (int c2 = sc.cluster + 1; c2 <= last; ++c2) {
              const float4* p4 = reinterpret_cast<const float4*>(
                  sk.partials + size_t(c2) * (2 * 128 * BN) + part_off + c * 32);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 pv = __ldcg(p4 + q);
                v[4 * q] += pv.x;
                v[4 * q + 1] += pv.y;
                v[4 * q + 2] += pv.z;
                v[4 * q + 3] += pv.w;
              }
            }
            if (KIND == kEpiGrad)
              grad_store_warp(ep, row - int(lane), col0, v, epi_stage);
            else
              epilogue32<KIND>(ep, row, col0, v, ss);
          }
          // Each flag has exactly one reader, this warp: clear what it consumed, so the
          // flags are zero again when the launch ends. A later launch that carries the same
          // epoch value (a repeated launch of identical parameters) then cannot take them
          // for its own. (After a wait that gave up the flags are left as they are; the
          // status word reports that launch.)
          if (ok && lane == 0)
            for (int c2 = sc.cluster + 1; c2 <= last; ++c2)
              sk.flags[(size_t(c2) * 2 + rank) * 4 + quad] = 0;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(tempty0 + 8 * acc);
        else
          mbar_arrive_remote(mapa_shared(tempty0 + 8 * acc, 0));
      }
      if (MT == 1) {
        acc ^= 1;
        if (acc == 0) acc_par ^= 1;
      } else {
        acc_par ^= 1;
      }
    }
    // the warp's TMA stores must have read their buffers, and landed, before the CTA ends
    if (ss.n > 0 && lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still arrive on it or MMA into it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// Process-wide launch counter for the stream-K flags, seeded so that a stale flag left in
// a reused buffer by an earlier process is not taken for this launch's.
uint64_t next_epoch() {
  static std::atomic<uint64_t> counter{
      (uint64_t(std::random_device{}()) << 32) ^
      uint64_t(std::chrono::steady_clock::now().time_since_epoch().count()) ^
      0x9E3779B97F4A7C15ull};
  uint64_t e = ++counter;
  return e == 0 ? ++counter : e;
}

// Stream-K tiles of a two-M-tile launch: at most this many pairs share one tile along K.
constexpr int kSkMaxSplit = 16;

template <int KIND, int OP, int LAYOUT = kKK, int MT = 1>
cudaError_t launch_kind(const CUtensorMap& tmA, const CUtensorMap& tmB, int M, int N, int K,
                        const EpiParams& ep, int num_sms, int* status, uint64_t limit_ns,
                        void* sk_scratch, cudaStream_t stream) {
  constexpr size_t SMEM_BYTES = Geo<MT>::SMEM_BYTES;
  static PerDeviceInit setup;  // per device: shared-memory opt-in and co-resident pairs
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int max_clusters = 0;
  const cudaError_t attr_err = per_device_init(
      setup,
      [&](int dev, int* out) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel<KIND, OP, LAYOUT, MT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(SMEM_BYTES));
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t occ = cfg;
        occ.gridDim = dim3(2 * (sms / 2), 1, 1);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, gemm_kernel<KIND, OP, LAYOUT, MT>, &occ);
        *out = (e == cudaSuccess && n > 0) ? n : 0;
        return e;
      },
      &max_clusters);
  if (attr_err != cudaSuccess) return attr_err;
  if (max_clusters <= 0) return cudaErrorLaunchOutOfResources;
  const int units = ((M + MT * PM - 1) / (MT * PM)) * ((N + BN - 1) / BN);
  const int clusters = units < max_clusters ? units : max_clusters;
  const int bke = OP == kOpE4m3 ? kGemmBK8 : BK;
  const int num_kb = (K + bke - 1) / bke;
  // Stream-K for the last waves when they would leave pairs idle. MT = 1: every full wave
  // but one runs whole tiles; the remaining (clusters + rem) tiles are split evenly along
  // K. MT = 2: every full wave runs whole 512-row units (the traffic saving holds there);
  // the rem units left over are split into their 256-row tiles, and those along K, over at
  // most kSkMaxSplit pairs per tile.
  SkParams sk{};
  sk.dp_tiles = units;
  const int rem = units % clusters;
  if (sk_scratch != nullptr && clusters <= kSkMaxClusters && units > clusters && rem != 0 &&
      num_kb >= 8) {
    int sk_pairs = clusters;
    if (MT == 1) {
      sk.sk_tiles = clusters + rem;
      sk.dp_tiles = units - sk.sk_tiles;
    } else {
      sk.sk_tiles = MT * rem;
      sk.dp_tiles = units - rem;
      if (sk.sk_tiles * kSkMaxSplit < sk_pairs) sk_pairs = sk.sk_tiles * kSkMaxSplit;
    }
    const int64_t iters = int64_t(sk.sk_tiles) * num_kb;
    sk.W = int((iters + sk_pairs - 1) / sk_pairs);
    sk.partials = static_cast<float*>(sk_scratch);
    sk.flags = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(sk_scratch) +
                                           size_t(kSkMaxClusters) * kSkPartialBytes);
    sk.epoch = next_epoch();
  }
  EpiParams e = ep;
  e.M = M;
  e.N = N;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<KIND, OP, LAYOUT, MT>, tmA, tmB, K, e, sk, status,
                            limit_ns);
}

// Two M tiles per unit for the K-major GEMMs whose M spans at least two 256-row tiles and
// whose K is long: the shared B stage cuts operand traffic per FLOP by a quarter, and under
// the power limit the lower traffic keeps the SM clock higher; the accumulator is not
// double-buffered, so the epilogue must be small next to a unit's main loop (measured: a
// gain from K = 12288 on, a loss at K <= 10240).
inline bool two_m_tiles(int M, int K) { return M > PM && K >= 12288; }

}  // namespace

size_t gemm_smem_bytes() { return Geo<1>::SMEM_BYTES; }

namespace {
// The bounded wait of the kernels above, on a barrier that never completes.
__global__ void wait_probe_kernel(uint64_t limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  const WaitCtl wc{&abort_flag, status, limit_ns};
  mbar_wait(smem_u32(&bar), 0, wc, 99);
}
}  // namespace

cudaError_t launch_wait_probe(uint64_t limit_ns, int* status, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

cudaError_t launch_gemm(EpiKind kind, OpType op, const CUtensorMap& tmA, const CUtensorMap& tmB,
                        int M, int N, int K, const EpiParams& ep, int num_sms, int* status,
                        uint64_t limit_ns, void* sk_scratch, cudaStream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
  if (K % (op == kOpE4m3 ? kGemmBK8 : kGemmBK) != 0) return cudaErrorInvalidValue;
#define PB_GEMM_OP(KIND_, OP_)                                                                 \
  return two_m_tiles(M, K) ? launch_kind<KIND_, OP_, kKK, 2>(tmA, tmB, M, N, K, ep, num_sms,     \
                                                          status, limit_ns, sk_scratch, stream) \
                        : launch_kind<KIND_, OP_, kKK, 1>(tmA, tmB, M, N, K, ep, num_sms,     \
                                                          status, limit_ns, sk_scratch, stream)
#define PB_GEMM_CASE(KIND_)                                                                    \
  switch (op) {                                                                                \
    case kOpF16:                                                                               \
      PB_GEMM_OP(KIND_, kOpF16);                                                               \
    case kOpE4m3:                                                                              \
      PB_GEMM_OP(KIND_, kOpE4m3);                                                              \
    default:                                                                                   \
      PB_GEMM_OP(KIND_, kOpBf16);                                                              \
  }
  switch (kind) {
    case kEpiStore:
      PB_GEMM_CASE(kEpiStore);
    case kEpiBlockIn:
      PB_GEMM_CASE(kEpiBlockIn);
    case kEpiResidual:
      PB_GEMM_CASE(kEpiResidual);
    default:
      break;
  }
#undef PB_GEMM_CASE
#undef PB_GEMM_OP
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_layout(EpiKind kind, GemmLayout layout, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, int M, int N, int K, const EpiParams& ep,
                               int num_sms, int* status, uint64_t limit_ns, void* sk_scratch,
                               cudaStream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
  // a K-major operand's rows are K elements: TMA wants a 16-byte multiple
  if (layout != kMM && K % 8 != 0) return cudaErrorInvalidValue;
#define PB_GEMM_LAYOUT(KIND_, LAYOUT_)                                                        return launch_kind<KIND_, kOpBf16, LAYOUT_>(tmA, tmB, M, N, K, ep, num_sms, status,                                                     limit_ns, sk_scratch, stream)
  if (kind == kEpiStore) {
    switch (layout) {
      case kKK: PB_GEMM_LAYOUT(kEpiStore, kKK);
      case kMK: PB_GEMM_LAYOUT(kEpiStore, kMK);
      case kKM: PB_GEMM_LAYOUT(kEpiStore, kKM);
      case kMM: PB_GEMM_LAYOUT(kEpiStore, kMM);
    }
  } else if (kind == kEpiBwdAct && layout == kKM) {
    PB_GEMM_LAYOUT(kEpiBwdAct, kKM);
  } else if (kind == kEpiGrad && layout == kKM) {
    PB_GEMM_LAYOUT(kEpiGrad, kKM);
  } else if (kind == kEpiGrad && layout == kMM) {
    PB_GEMM_LAYOUT(kEpiGrad, kMM);
  }
#undef PB_GEMM_LAYOUT
  return cudaErrorInvalidValue;
}

}  // namespace pb
