// swa_bwd.cu — backward of the sliding-window causal attention on the tensor cores, with
// the probabilities recomputed from q, k and the forward's log-sum-exp instead of stored
// (the selective recomputation of the MegaScale reading notes, section 1.3: the score
// matrix is the expensive activation, recomputed in the backward pass).
//
// For one head of one sequence, with W(i) = {j : 0 <= i - j < w}, s_ij = q_i . k_j / sqrt(dh),
// p_ij = 2^(s_ij log2(e) - L_i) (L_i the forward's log2-sum-exp of row i), do = dL/do:
//   dv_j = sum_i p_ij do_i
//   dp_ij = do_i . v_j,   ds_ij = p_ij (dp_ij - D_i),   D_i = do_i . o_i
//   dq_i = sum_j ds_ij k_j / sqrt(dh),   dk_j = sum_i ds_ij q_i / sqrt(dh)
// (D_i equals sum_j p_ij dp_ij because o_i = sum_j p_ij v_j.)
//
// One CTA per (128-key tile, head, sequence), the key tiles with the most queries first.
// It keeps K and V of its keys in shared memory and dV, dK (fp32) in tensor memory, and
// walks the 64-query steps that reach its keys (from its first key to the last query whose
// window does). Step n, in tensor-memory buffer b = n % 2:
//   S^T  = K Q^T        (M = 128 keys, N = 64 queries)              buffer b, columns 0-63
//   dP^T = V dO^T       (A = V, MN-major from v^T)                  buffer b, columns 64-127
//   P and dS warps: P^T and dS^T (bf16) over S^T and dP^T, dS into shared memory (b)
//   dV  += P^T dO,  dK += dS^T Q   (A from tensor memory, B = dO and Q read MN-major)
//   dQ^T = K^T dS       (M = 128 head dims, N = 64 queries; both operands MN-major) over
//                       buffer b; with dh = 64 the upper 64 rows of K^T are a zero box
//   dQ warps: dQ^T out, each warp's 32 head dims x 64 queries staged in shared memory and
//             added into the fp32 dq accumulator in global memory by one TMA reduction
//             (other key tiles add theirs)
// With two buffers the P/dS math of step n + 1 runs while the tensor cores compute the
// dV, dK and dQ products of step n; buffer b is loaded with the scores of step n + 2 once
// dQ^T of step n has been read out. The MMAs of one thread execute in issue order, so dQ^T
// overwrites P^T only after dV has read it; a commit covers every earlier MMA. The same
// shared-memory tiles serve as K-major and as MN-major operands: a TMA box of 64 16-bit
// elements per row is both.
//   warp 0     TMA producer: K and V once, then per step Q, dO and the step's 64 values
//              of the log-sum-exp and of D (2-stage ring)
//   warp 1     tensor-memory owner and the MMA-issuing thread
//   warps 2-5  P and dS, one key per thread (its TMEM lane)
//   warps 6-9  dQ per step, then the dK and dV rows of the tile
// Tensor memory: buffer 0 [0, 128) | buffer 1 [128, 256) | dV [256, 256 + dh) |
// dK [384, 384 + dh). Head sizes 64 and 128.
#include "kernels.h"
#include "ptx.cuh"

namespace pb {
namespace {

constexpr int BKV = 128;  // keys per CTA
constexpr int BQ = 64;    // queries per step
constexpr int THREADS = 320;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_BUF = 128, T_DP = 64, T_DV = 256, T_DK = 384;
constexpr int K_BOX = BKV * 64 * 2;   // 16 KB: 128 keys x 64 dims
constexpr int K_BYTES = 2 * K_BOX;    // two boxes whatever the head size (see below)
constexpr int QD_BOX = BQ * 64 * 2;   // 8 KB: 64 queries x 64 dims
constexpr int ROWVAL_BYTES = BQ * 4;  // 64 fp32 values of L or D
constexpr int STAGES = 2;
constexpr int DS_BYTES = BKV * BQ * 2;  // dS: 128 key rows x 64 queries
constexpr int DQ_WARP_BYTES = 32 * BQ * 4;  // a dQ warp's staging: 64 queries x 32 dims fp32
// kv_full, q_full[2], q_empty[2], s_full[2], p_full[2], mma_done[2], dq_free[2], drain
constexpr int NUM_BARS = 14;

// Shared-memory layout for head size DH (64 or 128). K always takes two 64-dim boxes: with
// DH = 64 the second is zero, so dQ^T = K^T dS stays an M = 128 product whose rows 64-127
// are zero (the dQ warps of those rows skip their reductions).
template <int DH>
struct BwdLayout {
  static_assert(DH == 64 || DH == 128, "head size");
  static constexpr int K_TX = (DH / 64) * K_BOX;  // bytes the K load brings
  static constexpr int V_HALF = DH * 64 * 2;      // dh rows x 64 keys (from v^T)
  static constexpr int V_BYTES = 2 * V_HALF;
  static constexpr int Q_BYTES = (DH / 64) * QD_BOX;
  static constexpr int STAGE_TX = 2 * Q_BYTES + 2 * ROWVAL_BYTES;  // Q, dO, L, D
  static constexpr int STAGE_BYTES = 2 * Q_BYTES + 1024;           // next stage 1024-aligned
  static constexpr int K_OFF = 0, V_OFF = K_BYTES, ST_OFF = V_OFF + V_BYTES;
  static constexpr int DS_OFF = ST_OFF + STAGES * STAGE_BYTES;
  static constexpr int DQ_OFF = DS_OFF + 2 * DS_BYTES;
  static constexpr int BAR_OFF = DQ_OFF + 4 * DQ_WARP_BYTES;
  static constexpr size_t NEED = size_t(BAR_OFF) + NUM_BARS * 8 + 16 + 1024;
  // one CTA per SM: it takes all tensor-memory columns
  static constexpr size_t SMEM = NEED > 120 * 1024 ? NEED : 120 * 1024;
  static_assert(SMEM <= 227 * 1024 && 2 * SMEM > 228 * 1024, "shared memory layout");
};

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t u[64];
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(u));
  tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
  tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(u));
  tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(u + 32));
#pragma unroll
  for (int e = 0; e < 64; ++e) v[e] = __uint_as_float(u[e]);
}

// The step count of key tile j0: from its first key to the last query whose window
// reaches the tile, in 64-query steps.
__device__ __forceinline__ int num_steps(const SwaBwdParams& p, int j0) {
  const int last = min(p.S - 1, j0 + BKV - 1 + p.window - 1);
  return last / BQ - j0 / BQ + 1;
}

template <int DH>
__global__ void __launch_bounds__(THREADS, 1)
    swa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmVT,
                   const __grid_constant__ CUtensorMap tmDO,
                   const __grid_constant__ CUtensorMap tmDQ, const SwaBwdParams p, int* status,
                   uint64_t limit_ns) {
  using Lb = BwdLayout<DH>;
  constexpr int K_TX = Lb::K_TX, V_HALF = Lb::V_HALF, V_BYTES = Lb::V_BYTES;
  constexpr int Q_BYTES = Lb::Q_BYTES, STAGE_TX = Lb::STAGE_TX, STAGE_BYTES = Lb::STAGE_BYTES;
  constexpr int K_OFF = Lb::K_OFF, V_OFF = Lb::V_OFF, ST_OFF = Lb::ST_OFF;
  constexpr int DS_OFF = Lb::DS_OFF, DQ_OFF = Lb::DQ_OFF, BAR_OFF = Lb::BAR_OFF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  const uint32_t kv_full = smem_u32(bars + 0);
  const uint32_t q_full0 = smem_u32(bars + 1);    // [2] per stage
  const uint32_t q_empty0 = smem_u32(bars + 3);   // [2]
  const uint32_t s_full0 = smem_u32(bars + 5);    // [2] per tensor-memory buffer
  const uint32_t p_full0 = smem_u32(bars + 7);    // [2] (4 P/dS warps)
  const uint32_t mma_done0 = smem_u32(bars + 9);  // [2] the step's dV, dK, dQ^T products
  const uint32_t dq_free0 = smem_u32(bars + 11);  // [2] (4 dQ warps read dQ^T out)
  const uint32_t drain_bar = smem_u32(bars + 13);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (cta_should_skip(status)) return;
  // Work item: key tile (slowest: the tiles with the most queries come first), head, sequence.
  const int per_tile = p.nh * p.B;
  const int jt = int(blockIdx.x) / per_tile;
  const int head = int(blockIdx.x) % p.nh;
  const int b = (int(blockIdx.x) / p.nh) % p.B;
  const int j0 = jt * BKV;
  const int N = num_steps(p, j0);
  const int64_t row_off = int64_t(b * p.nh + head) * p.lse_ld;  // of L and D

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(q_full0 + 8 * s, 1);
      mbar_init(q_empty0 + 8 * s, 1);
      mbar_init(s_full0 + 8 * s, 1);
      mbar_init(p_full0 + 8 * s, 4);
      mbar_init(mma_done0 + 8 * s, 1);
      mbar_init(dq_free0 + 8 * s, 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (DH == 64) {
    // the second K box: zero rows of K^T for the M = 128 dQ^T product
    uint4* kz = reinterpret_cast<uint4*>(smem + K_OFF + K_BOX);
    for (int e = int(threadIdx.x); e < K_BOX / 16; e += THREADS) kz[e] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVT);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmDQ);
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
  const uint64_t drain_ns = limit_ns > kDrainFloorNs ? limit_ns : kDrainFloorNs;
  const uint32_t sK = smem_u32(smem + K_OFF), sV = smem_u32(smem + V_OFF);
  const uint32_t sST = smem_u32(smem + ST_OFF), sDS = smem_u32(smem + DS_OFF);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ producer
      mbar_arrive_expect_tx(kv_full, K_TX + V_BYTES);
#pragma unroll
      for (int c = 0; c < DH / 64; ++c)
        tma_load_3d(sK + c * K_BOX, &tmK, kv_full, p.H + head * DH + 64 * c, j0, b);
#pragma unroll
      for (int c = 0; c < 2; ++c)  // two halves of 64 keys
        tma_load_2d(sV + c * V_HALF, &tmVT, kv_full, j0 + 64 * c, (b * p.nh + head) * DH);
      int issued = 0;
      for (int n = 0; n < N; ++n) {
        const int st = n & 1;
        if (!mbar_wait(q_empty0 + 8 * st, uint32_t((n >> 1) & 1) ^ 1u, wc, 30)) break;
        const uint32_t dst = sST + st * STAGE_BYTES, bar = q_full0 + 8 * st;
        const int i0 = j0 + n * BQ;
        mbar_arrive_expect_tx(bar, STAGE_TX);
#pragma unroll
        for (int c = 0; c < DH / 64; ++c) {
          tma_load_3d(dst + c * QD_BOX, &tmQ, bar, head * DH + 64 * c, i0, b);
          tma_load_3d(dst + Q_BYTES + c * QD_BOX, &tmDO, bar, head * DH + 64 * c, i0, b);
        }
        // the rows' L and D (row stride lse_ld, a multiple of 64: never past the row)
        bulk_load(dst + 2 * Q_BYTES, p.lse + row_off + i0, ROWVAL_BYTES, bar);
        bulk_load(dst + 2 * Q_BYTES + ROWVAL_BYTES, p.delta + row_off + i0, ROWVAL_BYTES, bar);
        issued = n + 1;
      }
      // the CTA's own copies land before it may exit
      mbar_wait_drain(kv_full, 0, drain_ns);
      for (int n = issued - 2 < 0 ? 0 : issued - 2; n < issued; ++n)
        mbar_wait_drain(q_full0 + 8 * (n & 1), uint32_t(n >> 1) & 1u, drain_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------------ MMA issuer
      const uint32_t id_s = idesc_f32acc(BKV, BQ);                        // K, Q K-major
      const uint32_t id_dp = idesc_f32acc(BKV, BQ, false, true, false);   // V MN-major
      const uint32_t id_acc = idesc_f32acc(BKV, DH, false, false, true);  // TMEM A, B MN
      // dQ^T: M = the two 64-dim K boxes (the second zero when DH = 64), both MN-major
      const uint32_t id_dq = idesc_f32acc(128, BQ, false, true, true);
      const uint64_t dK = sdesc_kmajor_sw128(sK), dKmn = sdesc_mnmajor_sw128(sK, K_BOX);
      const uint64_t dVmn = sdesc_mnmajor_sw128(sV, V_HALF);
      // S^T and dP^T of step n into buffer n % 2 (its Q / dO stage is n % 2 too)
      auto issue_scores = [&](int n) -> bool {
        const int st = n & 1;
        if (!mbar_wait(q_full0 + 8 * st, uint32_t(n >> 1) & 1u, wc, 32)) return false;
        tc_fence_after();
        const uint32_t sQ = sST + st * STAGE_BYTES, sDO = sQ + Q_BYTES;
        const uint64_t dQk = sdesc_kmajor_sw128(sQ), dDOk = sdesc_kmajor_sw128(sDO);
        const uint32_t t = tmem_base + uint32_t(st) * T_BUF;
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint64_t ok_ = uint64_t(((kk >> 2) * K_BOX) >> 4) + 2 * (kk & 3);
          const uint64_t oq = uint64_t(((kk >> 2) * QD_BOX) >> 4) + 2 * (kk & 3);
          mma_f16kind_ss(t, dK + ok_, dQk + oq, id_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint64_t oq = uint64_t(((kk >> 2) * QD_BOX) >> 4) + 2 * (kk & 3);
          mma_f16kind_ss(t + T_DP, dVmn + 128 * kk, dDOk + oq, id_dp, kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full0 + 8 * st);
        return true;
      };
      bool ok = mbar_wait(kv_full, 0, wc, 31);
      if (ok) ok = issue_scores(0);
      if (ok && N > 1) ok = issue_scores(1);
      for (int n = 0; ok && n < N; ++n) {
        const int bf = n & 1;
        const uint32_t par = uint32_t(n >> 1) & 1u;
        if (!mbar_wait(p_full0 + 8 * bf, par, wc, 33)) break;
        tc_fence_after();
        const uint32_t t = tmem_base + uint32_t(bf) * T_BUF;
        const uint32_t sQ = sST + bf * STAGE_BYTES, sDO = sQ + Q_BYTES;
        // dV += P^T dO, dK += dS^T Q: K = the step's 64 queries
        const uint64_t dDOmn = sdesc_mnmajor_sw128(sDO, QD_BOX);
        const uint64_t dQmn = sdesc_mnmajor_sw128(sQ, QD_BOX);
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_f16kind_ts(tmem_base + T_DV, t + 8 * kk, dDOmn + 128 * kk, id_acc,
                         (n > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_f16kind_ts(tmem_base + T_DK, t + T_DP + 8 * kk, dQmn + 128 * kk, id_acc,
                         (n > 0 || kk > 0) ? 1u : 0u);
        mma_commit(q_empty0 + 8 * bf);  // Q and dO of this stage are read
        // dQ^T = K^T dS over the buffer's first 64 columns (after dV has read P^T there)
        const uint64_t dDS = sdesc_mnmajor_sw128(sDS + bf * DS_BYTES, DS_BYTES);
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          mma_f16kind_ss(t, dKmn + 128 * kk, dDS + 128 * kk, id_dq, kk > 0 ? 1u : 0u);
        mma_commit(mma_done0 + 8 * bf);
        // the buffer takes step n + 2's scores once dQ^T of step n is out
        if (n + 2 < N) {
          if (!mbar_wait(dq_free0 + 8 * bf, par, wc, 34)) break;
          tc_fence_after();
          if (!issue_scores(n + 2)) break;
        }
      }
      mma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, drain_ns);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------------ P and dS
    const uint32_t quad = warp & 3;
    const int r = int(quad * 32 + lane);  // key of the tile = TMEM lane
    const int key = j0 + r;
    const uint32_t lane_addr = (quad * 32u) << 16;
    const uint64_t c2 = f2(p.scale_log2, p.scale_log2);
    const int sw = r & 7;  // 128-byte swizzle of the row's 16-byte chunks
    for (int n = 0; n < N; ++n) {
      const int bf = n & 1;
      const uint32_t par = uint32_t(n >> 1) & 1u;
      // the scores, and the stage's L and D values (already complete: the scores were
      // computed from the same stage)
      if (!mbar_wait_warp(s_full0 + 8 * bf, par, wc, 35) ||
          !mbar_wait_warp(q_full0 + 8 * bf, par, wc, 37))
        break;
      tc_fence_after();
      const uint32_t t = tmem_base + lane_addr + uint32_t(bf) * T_BUF;
      const float* Ls =
          reinterpret_cast<const float*>(smem + ST_OFF + bf * STAGE_BYTES + 2 * Q_BYTES);
      const float* Ds = Ls + BQ;
      uint8_t* ds_row = smem + DS_OFF + bf * DS_BYTES + r * 128;
      const int i0 = j0 + n * BQ;
      // Every (query, key) of the step inside the window: no element masks. Keys past the
      // sequence cannot occur then (they would lie after every query).
      const bool whole = (i0 >= j0 + BKV - 1) && (i0 + BQ - 1 - j0 < p.window) &&
                         (i0 + BQ - 1 < p.S);
      // two halves of 32 queries: S^T and dP^T in, P^T and dS^T out over them (the halves
      // already read), the dS row to shared memory. Pairs of queries in packed fp32 math;
      // L and D four queries per shared-memory load (the same address in every lane).
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t us[32], ud[32];
        tmem_ld32(t + 32 * hf, us);
        tmem_ld32(t + T_DP + 32 * hf, ud);
        tmem_ld_wait(us);
        tmem_ld_wait_regs(ud);
        const float4* L4 = reinterpret_cast<const float4*>(Ls + 32 * hf);
        const float4* D4 = reinterpret_cast<const float4*>(Ds + 32 * hf);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 l = L4[e / 4], dd = D4[e / 4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int e2 = e + 2 * h;
            const uint64_t x2 = f2_fma(f2(__uint_as_float(us[e2]), __uint_as_float(us[e2 + 1])),
                                       c2, h ? f2(-l.z, -l.w) : f2(-l.x, -l.y));
            float x0, x1;
            f2_split(x2, x0, x1);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if (!whole) {  // q's window holds the key: 0 <= q - key < w, q < S
              const int q = i0 + 32 * hf + e2, d = q - key;
              if (!(d >= 0 && d < p.window && q < p.S)) p0 = 0.f;
              if (!(d + 1 >= 0 && d + 1 < p.window && q + 1 < p.S)) p1 = 0.f;
            }
            const uint64_t p2 = f2(p0, p1);
            const uint64_t g2 = f2_sub(f2(__uint_as_float(ud[e2]), __uint_as_float(ud[e2 + 1])),
                                       h ? f2(dd.z, dd.w) : f2(dd.x, dd.y));
            float s0, s1;
            f2_split(f2_mul(p2, g2), s0, s1);
            pk[e2 / 2] = pack_bf16x2(p0, p1);
            dk[e2 / 2] = pack_bf16x2(s0, s1);
          }
        }
        tmem_st16(t + 16 * hf, pk);
        tmem_st16(t + T_DP + 16 * hf, dk);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
          *reinterpret_cast<uint4*>(ds_row + (((4 * hf + ch) ^ sw) << 4)) =
              make_uint4(dk[4 * ch], dk[4 * ch + 1], dk[4 * ch + 2], dk[4 * ch + 3]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full0 + 8 * bf);
    }
  } else {
    // ------------------------------------------------------------------ dQ, dK, dV out
    const uint32_t quad = warp & 3;
    const int r = int(quad * 32 + lane);  // TMEM lane: head dim of dQ^T, key of dV and dK
    const uint32_t lane_addr = (quad * 32u) << 16;
    float* dq_st = reinterpret_cast<float*>(smem + DQ_OFF + (warp - 6) * DQ_WARP_BYTES);
    const uint32_t s_dq = smem_u32(dq_st);
    bool ok = true;
    for (int n = 0; n < N; ++n) {
      const int bf = n & 1;
      if (!mbar_wait_warp(mma_done0 + 8 * bf, uint32_t(n >> 1) & 1u, wc, 36)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[64];
      tmem_ld64(tmem_base + lane_addr + uint32_t(bf) * T_BUF, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free0 + 8 * bf);
      if (int(quad) * 32 >= DH) continue;  // rows of the zero K box (DH = 64)
      const int i0 = j0 + n * BQ;
      // the warp's [64 queries][32 dims] block of dQ into its staging buffer (once the
      // previous step's reduction has read it), then one TMA add into dq (rows past the
      // sequence are outside the map's bounds and skipped)
      if (lane == 0) bulk_wait_read();
      __syncwarp();
#pragma unroll
      for (int e = 0; e < 64; ++e) dq_st[e * 32 + lane] = v[e];
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_3d(&tmDQ, s_dq, head * DH + int(quad) * 32, i0, b);
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_all();  // before the CTA's shared memory is released
    __syncwarp();
    if (ok) {
      // the last step's commit covers every dV and dK product
      const int key = j0 + r;
      __nv_bfloat16* out = p.dz + (int64_t(b) * p.S + key) * p.ldz + head * DH;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {  // dV to column 2H, dK (scaled) to H
        const uint32_t tcol = which ? T_DK : T_DV;
        const float scale = which ? p.scale : 1.f;
        __nv_bfloat16* dst = out + (which ? p.H : 2 * p.H);
#pragma unroll
        for (int ch = 0; ch < DH / 32; ++ch) {
          uint32_t u[32];
          tmem_ld32(tmem_base + lane_addr + tcol + 32 * ch, u);
          tmem_ld_wait(u);
          if (key < p.S) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * ch);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float* f = reinterpret_cast<const float*>(u) + 8 * q;
              d4[q] = make_uint4(pack_bf16x2(f[0] * scale, f[1] * scale),
                                 pack_bf16x2(f[2] * scale, f[3] * scale),
                                 pack_bf16x2(f[4] * scale, f[5] * scale),
                                 pack_bf16x2(f[6] * scale, f[7] * scale));
            }
          }
        }
      }
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
cudaError_t launch_dh(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmVT,
                      const CUtensorMap& tmDO, const CUtensorMap& tmDQ, const SwaBwdParams& p,
                      int* status, uint64_t limit_ns, cudaStream_t stream) {
  constexpr size_t SMEM = BwdLayout<DH>::SMEM;
  static PerDeviceInit setup;  // per device: the shared-memory opt-in
  const cudaError_t attr = per_device_init(setup, [](int, int*) {
    return cudaFuncSetAttribute(swa_bwd_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(SMEM));
  });
  if (attr != cudaSuccess) return attr;
  const int64_t tiles = (int64_t(p.S) + BKV - 1) / BKV;
  const int64_t grid = tiles * p.nh * p.B;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  swa_bwd_kernel<DH><<<unsigned(grid), THREADS, SMEM, stream>>>(tmQ, tmK, tmVT, tmDO, tmDQ, p,
                                                                 status, limit_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_swa_bwd(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmVT, const CUtensorMap& tmDO,
                           const CUtensorMap& tmDQ, const SwaBwdParams& p, int* status,
                           uint64_t limit_ns, cudaStream_t stream) {
  if (p.lse_ld % BQ != 0 || p.lse_ld < p.S) return cudaErrorInvalidValue;
  if (p.dh == 64) return launch_dh<64>(tmQ, tmK, tmVT, tmDO, tmDQ, p, status, limit_ns, stream);
  if (p.dh == 128) return launch_dh<128>(tmQ, tmK, tmVT, tmDO, tmDQ, p, status, limit_ns, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pb
