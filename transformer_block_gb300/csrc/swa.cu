// swa.cu — flash-style sliding-window causal attention on the tensor cores.
//
// For every sequence b, head j and query i:
//   o_i = sum_{k : 0 <= i - k < w} softmax_k(q_i . k_k / sqrt(dh)) v_k
// (MegaScale reading notes, section 1.1, "Sliding Window Attention", eqs. (5)-(6): each
// token attends to the most recent w tokens; the FlashAttention tiling of section 1.3
// keeps the score matrix on chip, so it never reaches HBM).
//
// One CTA per (query tile of 128 rows, head, sequence). Only the key tiles that meet
// the window [i - w + 1, i] of some query of the tile are visited, and only tiles that
// cross the diagonal or the window's far edge are masked element by element.
//   warp 0     TMA producer: the Q tile once, then K and V^T tiles in a 2-stage ring
//   warp 1     TMEM owner and the single MMA-issuing thread:
//                S_j = Q K_j^T  -> tensor memory (two S buffers, so S_{j+1} is computed
//                                  while the softmax works on S_j)
//                O  += P_j V_j  -> tensor memory (P_j read from shared memory)
//   warps 2-5  softmax, one query row per thread (the thread's TMEM lane): online
//              max / sum in fp32 with exp2 (the 1/sqrt(dh) and log2(e) factors folded
//              into one multiplier), P rounded to bf16 into shared memory, the running
//              output rescaled in tensor memory when the row maximum grows, and the
//              final O / l written as bf16.
// V arrives transposed ([dh, keys] per head, written so by the first GEMM's epilogue),
// so both products read K-major operands.
#include "kernels.h"
#include "ptx.cuh"

namespace pb {
namespace {

constexpr int BQ = kSwaBQ, BKV = kSwaBKV;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;  // S0 [0,128) | S1 [128,256) | O [256, 256+dh)
constexpr int BOX = 128 * 64 * 2;    // one 128-row x 64-column bf16 box: 16 KB

template <int DH>
struct Layout {
  static constexpr int Q_BYTES = BQ * DH * 2;
  static constexpr int K_BYTES = BKV * DH * 2;
  static constexpr int VHALF = DH * 64 * 2;  // V^T box: DH rows x 64 keys
  static constexpr int V_BYTES = 2 * VHALF;
  static constexpr int P_BYTES = BQ * BKV * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = Q_OFF + Q_BYTES;
  static constexpr int STAGE = K_BYTES + V_BYTES;
  static constexpr int P_OFF = KV_OFF + 2 * STAGE;
  static constexpr int BAR_OFF = P_OFF + P_BYTES;
  static constexpr int NUM_BARS = 12;
  // Request enough shared memory that only one CTA fits per SM: the CTA takes all 512
  // tensor-memory columns.
  static constexpr size_t SMEM = 200 * 1024;
  static_assert(BAR_OFF + NUM_BARS * 8 + 16 + 1024 <= SMEM, "shared memory layout");
};

template <int DH>
__global__ void __launch_bounds__(THREADS, 1)
    swa_kernel(const __grid_constant__ CUtensorMap tmQK, const __grid_constant__ CUtensorMap tmVT,
               const SwaParams p, int* status, uint64_t limit_ns) {
  using L = Layout<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  const uint32_t q_full = smem_u32(bars + 0);
  const uint32_t kv_full0 = smem_u32(bars + 1);   // [2]
  const uint32_t kv_empty0 = smem_u32(bars + 3);  // [2]
  const uint32_t s_full0 = smem_u32(bars + 5);    // [2]
  const uint32_t s_free0 = smem_u32(bars + 7);    // [2]
  const uint32_t p_full = smem_u32(bars + 9);
  const uint32_t o_ready = smem_u32(bars + 10);
  const uint32_t drain_bar = smem_u32(bars + 11);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // Heaviest query tiles first: with a window >= seq the last tiles see the most keys.
  const int nbh = p.nh * p.B;
  const int q_tile = p.num_q_tiles - 1 - int(blockIdx.x) / nbh;
  const int head = int(blockIdx.x) % p.nh;
  const int b = (int(blockIdx.x) % nbh) / p.nh;
  const int q0 = q_tile * BQ;
  const int q_hi = min(q0 + BQ - 1, p.S - 1);
  const int k_lo = max(0, q0 - p.window + 1);
  const int kt_begin = k_lo / BKV;
  const int nkv = q_hi / BKV - kt_begin + 1;

  if (cta_should_skip(status)) return;
  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(kv_full0 + 8 * s, 1);
      mbar_init(kv_empty0 + 8 * s, 1);
      mbar_init(s_full0 + 8 * s, 1);
      mbar_init(s_free0 + 8 * s, 4);
    }
    mbar_init(p_full, 4);
    mbar_init(o_ready, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQK);
    tma_prefetch_desc(&tmVT);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, status, limit_ns};
  // Teardown waits for the CTA's own copies and MMAs get at least a second, whatever the
  // wait limit, so shared and tensor memory are never released under them.
  const uint64_t drain_ns = limit_ns > kDrainFloorNs ? limit_ns : kDrainFloorNs;
  const uint32_t sQ = smem_u32(smem + L::Q_OFF);
  const uint32_t sKV = smem_u32(smem + L::KV_OFF);
  const uint32_t sP = smem_u32(smem + L::P_OFF);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      uint32_t last_par[2] = {0, 0};
      uint32_t used = 0;
      mbar_arrive_expect_tx(q_full, L::Q_BYTES);
#pragma unroll
      for (int hb = 0; hb < DH / 64; ++hb)
        tma_load_3d(sQ + hb * BOX, &tmQK, q_full, head * DH + hb * 64, q0, b);
      const int vt_row = (b * p.nh + head) * DH;
      for (int j = 0; j < nkv; ++j) {
        const int st = j & 1;
        const uint32_t par = (j >> 1) & 1;
        if (!mbar_wait(kv_empty0 + 8 * st, par ^ 1, wc, 11)) break;
        const uint32_t base = sKV + st * L::STAGE;
        const int k0 = (kt_begin + j) * BKV;
        mbar_arrive_expect_tx(kv_full0 + 8 * st, L::K_BYTES + L::V_BYTES);
#pragma unroll
        for (int hb = 0; hb < DH / 64; ++hb)
          tma_load_3d(base + hb * BOX, &tmQK, kv_full0 + 8 * st, p.H + head * DH + hb * 64, k0,
                      b);
#pragma unroll
        for (int kh = 0; kh < 2; ++kh)
          tma_load_2d(base + L::K_BYTES + kh * L::VHALF, &tmVT, kv_full0 + 8 * st, k0 + kh * 64,
                      vt_row);
        last_par[st] = par;
        used |= 1u << st;
      }
      mbar_wait_drain(q_full, 0, drain_ns);
      for (int s = 0; s < 2; ++s)
        if (used & (1u << s)) mbar_wait_drain(kv_full0 + 8 * s, last_par[s], drain_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      const uint32_t id_s = idesc_bf16_f32(BQ, BKV);
      const uint32_t id_o = idesc_bf16_f32(BQ, DH);
      const uint32_t t_o = tmem_base + 256;
      bool ok = mbar_wait(q_full, 0, wc, 12);
      // O += P_i V_i, once P_i is in shared memory.
      auto issue_pv = [&](int i) -> bool {
        if (!mbar_wait(p_full, i & 1, wc, 13)) return false;
        tc_fence_after();
        const uint32_t vbase = sKV + (i & 1) * L::STAGE + L::K_BYTES;
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
          const uint64_t da = sdesc_kmajor_sw128(sP + (kk >> 2) * BOX) + 2 * (kk & 3);
          const uint64_t db = sdesc_kmajor_sw128(vbase + (kk >> 2) * L::VHALF) + 2 * (kk & 3);
          mma_f16kind_ss(t_o, da, db, id_o, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(kv_empty0 + 8 * (i & 1));
        mma_commit(o_ready);
        return true;
      };
      for (int j = 0; ok && j < nkv; ++j) {
        const int st = j & 1;
        const uint32_t par = (j >> 1) & 1;
        if (!mbar_wait(kv_full0 + 8 * st, par, wc, 14)) {
          ok = false;
          break;
        }
        if (!mbar_wait(s_free0 + 8 * st, par ^ 1, wc, 15)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kbase = sKV + st * L::STAGE;
        const uint32_t t_s = tmem_base + uint32_t(st * BKV);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint64_t da = sdesc_kmajor_sw128(sQ + (kk >> 2) * BOX) + 2 * (kk & 3);
          const uint64_t db = sdesc_kmajor_sw128(kbase + (kk >> 2) * BOX) + 2 * (kk & 3);
          mma_f16kind_ss(t_s, da, db, id_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full0 + 8 * st);
        if (j > 0 && !issue_pv(j - 1)) ok = false;
      }
      if (ok) issue_pv(nkv - 1);
      mma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, drain_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax
    const uint32_t quad = warp & 3;
    const int r = int(quad * 32 + lane);  // query row inside the tile = TMEM lane
    const int i = q0 + r;                 // query position in the sequence
    const uint32_t lane_addr = (quad * 32u) << 16;
    const float c = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int st = j & 1;
      const uint32_t par = (j >> 1) & 1;
      if (!mbar_wait_warp(s_full0 + 8 * st, par, wc, 16)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[BKV];
#pragma unroll
      for (int ch = 0; ch < BKV / 32; ++ch) {
        uint32_t u[32];
        tmem_ld32(tmem_base + lane_addr + uint32_t(st * BKV + ch * 32), u);
        tmem_ld_wait(u);
#pragma unroll
        for (int e = 0; e < 32; ++e) s[ch * 32 + e] = __uint_as_float(u[e]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free0 + 8 * st);

      const int k0 = (kt_begin + j) * BKV;
      const bool whole = (k0 + BKV - 1 <= q0) && (q0 + BQ - 1 - k0 < p.window);
      if (!whole) {
#pragma unroll
        for (int e = 0; e < BKV; ++e) {
          const int d = i - (k0 + e);
          if (d < 0 || d >= p.window) s[e] = -INFINITY;
        }
      }
      float mx = m;
#pragma unroll
      for (int e = 0; e < BKV; ++e) mx = fmaxf(mx, s[e]);
      const float ms = (mx == -INFINITY) ? 0.f : mx * c;
      const float alpha = ex2_approx(m * c - ms);
      float sum = 0.f;
#pragma unroll
      for (int e = 0; e < BKV; ++e) {
        s[e] = ex2_approx(fmaf(s[e], c, -ms));
        sum += s[e];
      }
      l = l * alpha + sum;
      m = mx;

      if (j > 0) {
        // P_{j-1} V_{j-1} has finished: O is stable and the P buffer is free.
        if (!mbar_wait_warp(o_ready, (j - 1) & 1, wc, 17)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int ch = 0; ch < DH / 32; ++ch) {
            uint32_t u[32];
            const uint32_t ta = tmem_base + lane_addr + 256u + uint32_t(ch * 32);
            tmem_ld32(ta, u);
            tmem_ld_wait(u);
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
            tmem_st32(ta, u);
          }
          tmem_st_wait();
        }
      }
      // P row -> shared memory, K-major with the 128-byte swizzle the MMA expects.
      uint8_t* prow = smem + L::P_OFF + r * 128;
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const float* f = s + kb * 64 + ch * 8;
          uint4 v;
          v.x = pack_bf16x2(f[0], f[1]);
          v.y = pack_bf16x2(f[2], f[3]);
          v.z = pack_bf16x2(f[4], f[5]);
          v.w = pack_bf16x2(f[6], f[7]);
          *reinterpret_cast<uint4*>(prow + kb * BOX + ((ch ^ (r & 7)) << 4)) = v;
        }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && mbar_wait_warp(o_ready, (nkv - 1) & 1, wc, 18)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const int64_t off = (int64_t(b) * p.S + i) * p.out_ld + head * DH;
      bool bad = false;
#pragma unroll
      for (int ch = 0; ch < DH / 32; ++ch) {
        uint32_t u[32];
        tmem_ld32(tmem_base + lane_addr + 256u + uint32_t(ch * 32), u);
        tmem_ld_wait(u);
        if (i < p.S) {
          float o[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(u[e]) * inv_l;
          uint4* d4 = p.out_f16
                          ? reinterpret_cast<uint4*>(static_cast<__half*>(p.out) + off + ch * 32)
                          : reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + off +
                                                     ch * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float* f = o + 8 * q;
            uint4 v;
            if (p.out_f16) {
#pragma unroll
              for (int e = 0; e < 8; ++e) bad |= !(fabsf(f[e]) <= kF16Max);
              v.x = pack_f16x2(f[0], f[1]);
              v.y = pack_f16x2(f[2], f[3]);
              v.z = pack_f16x2(f[4], f[5]);
              v.w = pack_f16x2(f[6], f[7]);
            } else {
              v.x = pack_bf16x2(f[0], f[1]);
              v.y = pack_bf16x2(f[2], f[3]);
              v.z = pack_bf16x2(f[4], f[5]);
              v.w = pack_bf16x2(f[6], f[7]);
            }
            d4[q] = v;
          }
        }
      }
      if (bad) report_range(status);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int DH>
cudaError_t launch_dh(const CUtensorMap& tmQK, const CUtensorMap& tmVT, const SwaParams& p,
                      int* status, uint64_t limit_ns, cudaStream_t stream) {
  using L = Layout<DH>;
  static cudaError_t attr = cudaFuncSetAttribute(
      swa_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(L::SMEM));
  if (attr != cudaSuccess) return attr;
  const int64_t grid = int64_t(p.num_q_tiles) * p.nh * p.B;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  swa_kernel<DH><<<unsigned(grid), THREADS, L::SMEM, stream>>>(tmQK, tmVT, p, status, limit_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_swa(const CUtensorMap& tmQK, const CUtensorMap& tmVT, const SwaParams& p,
                       int* status, uint64_t limit_ns, cudaStream_t stream) {
  if (p.dh == 64) return launch_dh<64>(tmQK, tmVT, p, status, limit_ns, stream);
  if (p.dh == 128) return launch_dh<128>(tmQK, tmVT, p, status, limit_ns, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pb
