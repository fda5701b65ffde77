// swa.cu — flash-style sliding-window causal attention on the tensor cores.
//
// For every sequence b, head j and query i:
//   o_i = sum_{k : 0 <= i - k < w} softmax_k(q_i . k_k / sqrt(dh)) v_k
// (MegaScale reading notes, section 1.1, "Sliding Window Attention", eqs. (5)-(6): each
// token attends to the most recent w tokens; the FlashAttention tiling of section 1.3
// keeps the score matrix on chip, so it never reaches HBM).
//
// Work comes in items: a pair of 128-query tiles of one head of one sequence. Both query
// tiles share every K/V tile the item loads. Items are numbered by pair index, heaviest
// first, then sequence and head. The kernel is persistent: one CTA per SM, and CTA c takes
// items c, 2G - 1 - c, 2G + c, ... of the G CTAs. The rounds alternate direction, so the
// heavy items at the front even out. The K/V rings, the S/P barriers and the tensor memory
// carry over from one item to the next, so the next item's Q and K loads and its first S
// products overlap the current item's last tiles and output. Only key tiles that meet the
// window of some query of the pair are visited. A key tile that one query tile does not
// need is skipped for that tile (no MMA, no softmax). Only tiles that cross the diagonal or
// the window's far edge are masked element by element.
//   warp 0     TMA producer: per item both query tiles (once the previous item's last S
//              products are done), then K tiles (3-stage ring, freed as soon as both S
//              products have read them, loaded one tile ahead of V) and V^T tiles
//              (2-stage ring)
//   warp 1     tensor-memory owner and the single MMA-issuing thread, in the order
//                S0 = Q0 K_j^T, S1 = Q1 K_j^T, then per tile h: O_h += P_h V_j followed
//                by S_h = Q_h K_{j+1}^T
//              so the tensor cores work on one query tile while the other's softmax runs;
//              it waits only for P_h: each mbarrier wait in that thread idles the tensor
//              pipe for about its latency
//   warp 2     watcher: waits for the V tile of each step and the next K tile and adds an
//              arrival to query tile 0's P barrier, so the issuer's wait for P_0 also
//              covers them
//   warp 3     idle (warps 0-3 form the warpgroup whose registers go to the softmax)
//   warps 4-7  softmax of query tile 0, one row per thread (the thread's TMEM lane)
//   warps 8-11 softmax of query tile 1
// Tensor memory: S0 | S1 | O0 | O1 (128 columns each). The softmax writes P (bf16) over
// the first 64 columns of its own S, and the PV product reads it from there (A operand in
// tensor memory); the tensor pipe executes one thread's MMAs in issue order, so the next
// S_h overwrites P_h only after O_h += P_h V has read it.
// Online softmax in fp32 with exp2 (1/sqrt(dh) and log2(e) folded into one multiplier);
// the output is rescaled only when a row maximum grows by more than 2^8, and the final
// O / l uses the same reference maximum as every P, so the result is unchanged up to
// rounding. V arrives transposed ([dh, keys] per head, written so by the first GEMM's
// epilogue), so the PV product reads a K-major operand.
#include "kernels.h"
#include "ptx.cuh"

namespace pb {
namespace {

constexpr int BQ = kSwaBQ, BKV = kSwaBKV;
constexpr int THREADS = 384;
// Registers per thread: at launch (the most 384 threads may have), then per warpgroup: the
// producer / MMA warpgroup gives some up, the two softmax warpgroups take them.
constexpr uint32_t kRegsLaunch = 168, kRegsControl = 96, kRegsSoftmax = 200;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= THREADS * kRegsLaunch,
              "register split exceeds the launch allocation");
constexpr uint32_t TMEM_COLS = 512;
constexpr int BOX = 128 * 64 * 2;          // one 128-row x 64-column 16-bit box: 16 KB
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// One softmax row of a tile: p_k = 2^(s_k c - m) rounded to bf16 into tensor memory at t_s
// (column m holds keys 2m and 2m + 1), 32 keys per store; returns the fp32 sum of the
// unrounded p_k. Scale, shift and sum run on packed pairs.
__device__ __forceinline__ float probs_to_tmem(const float (&s)[kSwaBKV], float c, float m,
                                               uint32_t t_s) {
  const uint64_t c2 = f2(c, c), nm2 = f2(-m, -m);
  uint64_t acc[4] = {0, 0, 0, 0};  // four independent partial sums of pairs
#pragma unroll
  for (int ch = 0; ch < kSwaBKV / 32; ++ch) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint64_t x2 = f2_fma(f2(s[ch * 32 + 2 * e], s[ch * 32 + 2 * e + 1]), c2, nm2);
      float x0, x1;
      f2_split(x2, x0, x1);
      const uint64_t a2 = f2(ex2_approx(x0), ex2_approx(x1));
      acc[e & 3] = f2_add(acc[e & 3], a2);
      float a0, a1;
      f2_split(a2, a0, a1);
      pk[e] = pack_bf16x2(a0, a1);
    }
    tmem_st16(t_s + uint32_t(ch * 16), pk);
  }
  const uint64_t t = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
  float lo, hi;
  f2_split(t, lo, hi);
  return lo + hi;
}

template <int DH>
struct Layout {
  static constexpr int Q_TILE = BQ * DH * 2;
  static constexpr int K_BYTES = BKV * DH * 2;
  static constexpr int VHALF = DH * 64 * 2;  // V^T box: DH rows x 64 keys
  static constexpr int V_BYTES = 2 * VHALF;
  static constexpr int K_STAGES = 3, V_STAGES = 2;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = 2 * Q_TILE;
  static constexpr int V_OFF = K_OFF + K_STAGES * K_BYTES;
  static constexpr int BAR_OFF = V_OFF + V_STAGES * V_BYTES;
  static constexpr int NUM_BARS = 19;
  static constexpr size_t NEED = size_t(BAR_OFF) + NUM_BARS * 8 + 16 + 1024;
  // At least enough shared memory that only one CTA fits per SM: the CTA takes all 512
  // tensor-memory columns.
  static constexpr size_t SMEM = NEED > 200 * 1024 ? NEED : 200 * 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory layout");
};

// One unit of work: a pair of 128-query tiles of one head of one sequence.
struct Item {
  int b, head, q0;
  int kb0, ke0, kb1, ke1;  // key-tile range [kb, ke] of query tile 0 / 1 (empty past seq)
  int kt_begin, U;         // first key tile the pair visits, and how many it visits
};

// Item r of the launch. Longest work first: a pair's key-tile count never falls as the
// pair index grows (it grows until the window is full, then stays), so items run in
// descending pair order, every (sequence, head) of one pair index before the next.
__device__ __forceinline__ Item make_item(const SwaParams& p, int r) {
  const int num_pairs = (p.num_q_tiles + 1) / 2;
  Item it;
  const int pair = num_pairs - 1 - r / (p.nh * p.B);
  it.head = r % p.nh;
  it.b = (r / p.nh) % p.B;
  it.q0 = pair * 2 * BQ;
  int kb[2], ke[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int qb = it.q0 + h * BQ;
    kb[h] = qb < p.S ? max(0, qb - p.window + 1) / BKV : 1;
    ke[h] = qb < p.S ? min(qb + BQ - 1, p.S - 1) / BKV : 0;
  }
  it.kb0 = kb[0];
  it.ke0 = ke[0];
  it.kb1 = kb[1];
  it.ke1 = ke[1];
  it.kt_begin = kb[0];
  it.U = max(ke[0], ke[1]) - kb[0] + 1;
  return it;
}

// Does query tile h of the item need key tile j?
__device__ __forceinline__ bool item_needs(const Item& it, int h, int j) {
  return h ? (j >= it.kb1 && j <= it.ke1) : (j >= it.kb0 && j <= it.ke0);
}

// The n-th item of CTA c among G persistent CTAs: rounds of G items, dealt in alternating
// directions (c, then G - 1 - c), so the heavy items at the front even out across CTAs.
__device__ __forceinline__ int item_index(int n, int c, int G) {
  return n * G + ((n & 1) ? G - 1 - c : c);
}

template <int DH>
__global__ void __launch_bounds__(THREADS, 1)
    swa_kernel(const __grid_constant__ CUtensorMap tmQK, const __grid_constant__ CUtensorMap tmVT,
               const SwaParams p, int* status, uint64_t limit_ns) {
  static_assert(BKV == 128 && BQ == 128, "tile shape of this kernel");
  using L = Layout<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  const uint32_t q_full = smem_u32(bars + 0);
  const uint32_t q_empty = smem_u32(bars + 1);    // the item's last S products are done
  const uint32_t k_full0 = smem_u32(bars + 2);    // [3]
  const uint32_t k_empty0 = smem_u32(bars + 5);   // [3]
  const uint32_t v_full0 = smem_u32(bars + 8);    // [2]
  const uint32_t v_empty0 = smem_u32(bars + 10);  // [2]
  const uint32_t s_full0 = smem_u32(bars + 12);   // [2] per query tile
  const uint32_t p_full0 = smem_u32(bars + 14);   // [2] per query tile (4 warps each)
  const uint32_t o_final0 = smem_u32(bars + 16);  // [2] per query tile: item's last PV done
  const uint32_t drain_bar = smem_u32(bars + 18);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int num_items = ((p.num_q_tiles + 1) / 2) * p.nh * p.B;
  const int G = int(gridDim.x), cta = int(blockIdx.x);

  if (cta_should_skip(status)) return;
  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(k_full0 + 8 * s, 1);
      mbar_init(k_empty0 + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(v_full0 + 8 * s, 1);
      mbar_init(v_empty0 + 8 * s, 1);
      mbar_init(s_full0 + 8 * s, 1);
      // query tile 0: its 4 softmax warps and the watcher (the V and next K tiles landed)
      mbar_init(p_full0 + 8 * s, s == 0 ? 5 : 4);
      mbar_init(o_final0 + 8 * s, 1);
    }
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
  const uint32_t sK = smem_u32(smem + L::K_OFF);
  const uint32_t sV = smem_u32(smem + L::V_OFF);
  if (warp < 4) {
  setmaxnreg_dec<kRegsControl>();
  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      // K and V rings run on across items: load g (counted over the CTA's whole run) goes
      // to stage g % stages. Per stage: parity of its last load (bit s), ever loaded.
      uint32_t kc = 0, vc = 0;
      uint32_t k_par = 0, v_par = 0, k_used = 0, v_used = 0;
      int n_done = 0;
      bool ok = true;
      for (int n = 0; ok; ++n) {
        const int r = item_index(n, cta, G);
        if (r >= num_items) break;
        const Item it = make_item(p, r);
        // The Q tiles of the previous item are free once its last S products completed.
        if (!mbar_wait(q_empty, (n & 1) ^ 1, wc, 20)) break;
        mbar_arrive_expect_tx(q_full, 2 * L::Q_TILE);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int hb = 0; hb < DH / 64; ++hb)
            tma_load_3d(sQ + h * L::Q_TILE + hb * BOX, &tmQK, q_full, it.head * DH + hb * 64,
                        it.q0 + h * BQ, it.b);
        n_done = n + 1;
        const int vt_row = (it.b * p.nh + it.head) * DH;
        auto load_k = [&](int idx) -> bool {
          const uint32_t g = kc + uint32_t(idx);
          const uint32_t st = g % 3, par = (g / 3) & 1;
          if (!mbar_wait(k_empty0 + 8 * st, par ^ 1, wc, 11)) return false;
          const uint32_t dst = sK + st * L::K_BYTES;
          mbar_arrive_expect_tx(k_full0 + 8 * st, L::K_BYTES);
#pragma unroll
          for (int hb = 0; hb < DH / 64; ++hb)
            tma_load_3d(dst + hb * BOX, &tmQK, k_full0 + 8 * st, p.H + it.head * DH + hb * 64,
                        (it.kt_begin + idx) * BKV, it.b);
          k_par = (k_par & ~(1u << st)) | (par << st);
          k_used |= 1u << st;
          return true;
        };
        auto load_v = [&](int idx) -> bool {
          const uint32_t g = vc + uint32_t(idx);
          const uint32_t st = g & 1, par = (g >> 1) & 1;
          if (!mbar_wait(v_empty0 + 8 * st, par ^ 1, wc, 10)) return false;
          const uint32_t dst = sV + st * L::V_BYTES;
          mbar_arrive_expect_tx(v_full0 + 8 * st, L::V_BYTES);
#pragma unroll
          for (int kh = 0; kh < 2; ++kh)
            tma_load_2d(dst + kh * L::VHALF, &tmVT, v_full0 + 8 * st,
                        (it.kt_begin + idx) * BKV + kh * 64, vt_row);
          v_par = (v_par & ~(1u << st)) | (par << st);
          v_used |= 1u << st;
          return true;
        };
        // K runs one tile ahead of V: S_h of the next tile is issued before P_h V of this
        // one can be.
        ok = load_k(0);
        for (int idx = 0; ok && idx < it.U; ++idx) {
          if (idx + 1 < it.U) ok = load_k(idx + 1);
          if (ok) ok = load_v(idx);
        }
        kc += uint32_t(it.U);
        vc += uint32_t(it.U);
      }
      if (n_done > 0) mbar_wait_drain(q_full, uint32_t(n_done - 1) & 1, drain_ns);
      for (uint32_t s = 0; s < 3; ++s)
        if (k_used & (1u << s)) mbar_wait_drain(k_full0 + 8 * s, (k_par >> s) & 1u, drain_ns);
      for (uint32_t s = 0; s < 2; ++s)
        if (v_used & (1u << s)) mbar_wait_drain(v_full0 + 8 * s, (v_par >> s) & 1u, drain_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      const uint32_t id_s = idesc_bf16_f32(BQ, BKV);
      const uint32_t id_o = idesc_bf16_f32(BQ, DH);
      // Shared-memory descriptors: the start-address field is the byte address / 16, so a
      // descriptor for base + offset is the base's descriptor + offset / 16 (all addresses
      // stay below 256 KB, inside the 14-bit field). Built once, outside the issue path.
      const uint64_t dQ = sdesc_kmajor_sw128(sQ), dK = sdesc_kmajor_sw128(sK),
                     dV = sdesc_kmajor_sw128(sV);
      uint32_t kc = 0, vc = 0, tb = 0;  // K, V tiles and union tiles consumed so far
      bool ok = true;
      for (int n = 0; ok; ++n) {
        const int r = item_index(n, cta, G);
        if (r >= num_items) break;
        const Item it = make_item(p, r);
        // S_h = Q_h K^T for union key tile idx (nothing if query tile h does not need it).
        // The item's last S products read Q for the last time: then Q may be reloaded.
        auto issue_s = [&](int h, int idx) {
          const uint32_t st = (kc + uint32_t(idx)) % 3;
          if (item_needs(it, h, it.kt_begin + idx)) {
            const uint64_t da = dQ + uint64_t((h * L::Q_TILE) >> 4);
            const uint64_t db = dK + uint64_t((st * L::K_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < DH / 16; ++kk) {
              const uint64_t off = uint64_t(((kk >> 2) * BOX) >> 4) + 2 * (kk & 3);
              mma_f16kind_ss(tmem_base + uint32_t(h * BKV), da + off, db + off, id_s,
                             kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(s_full0 + 8 * h);
          if (h == 1) {
            mma_commit(k_empty0 + 8 * st);  // both S products have K
            if (idx + 1 == it.U) mma_commit(q_empty);
          }
        };
        if (!mbar_wait(q_full, uint32_t(n) & 1, wc, 12) ||
            !mbar_wait(k_full0 + 8 * (kc % 3), (kc / 3) & 1, wc, 14))
          break;
        tc_fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
        uint32_t pv_started = 0;  // bit h: O_h holds this item's partial sum
        for (int idx = 0; ok && idx < it.U; ++idx) {
          const int j = it.kt_begin + idx;
          const uint32_t gv = vc + uint32_t(idx);
          const uint64_t dv = dV + uint64_t(((gv & 1) * L::V_BYTES) >> 4);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // P_0's phase also certifies that V tile gv and K tile gk have landed (the
            // watcher's arrival), so one wait per query tile and key tile suffices.
            if (!mbar_wait(p_full0 + 8 * h, (tb + uint32_t(idx)) & 1, wc, 13)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (item_needs(it, h, j)) {
              // O_h += P_h V: P_h (bf16) sits in the first 64 columns of S_h. The softmax
              // of query tile h arrives on p_full only after it has read the previous
              // item's O_h out, so the first product may overwrite it.
              const uint32_t t_p = tmem_base + uint32_t(h * BKV);
              const uint32_t t_o = tmem_base + 256u + uint32_t(h * 128);
#pragma unroll
              for (int kk = 0; kk < BKV / 16; ++kk) {
                const uint64_t off = uint64_t(((kk >> 2) * L::VHALF) >> 4) + 2 * (kk & 3);
                mma_f16kind_ts(t_o, t_p + uint32_t(kk * 8), dv + off, id_o,
                               ((pv_started >> h) & 1u) | (kk > 0 ? 1u : 0u));
              }
              pv_started |= 1u << h;
            }
            if (h == 1) mma_commit(v_empty0 + 8 * (gv & 1));  // both PV products have V
            if (idx + 1 == it.U) mma_commit(o_final0 + 8 * h);  // once per item
            if (idx + 1 < it.U) issue_s(h, idx + 1);
          }
        }
        kc += uint32_t(it.U);
        vc += uint32_t(it.U);
        tb += uint32_t(it.U);
      }
      mma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, drain_ns);
    }
    __syncwarp();
  } else if (warp == 2) {
    if (lane == 0) {
      // ---------------------------------------------------------------- watcher
      // Every mbarrier wait in the MMA-issuing thread idles the tensor pipe for about its
      // latency, so that thread waits only for P. This thread waits for the V tile of each
      // step and the K tile of the next one, then adds its arrival to query tile 0's
      // p_full phase. It waits for that phase to complete before the next step, so it
      // never arrives in a later phase; a V or K stage cannot be refilled before the
      // phase completes, because the issuer reads it only afterwards.
      uint32_t kc = 0, vc = 0, tb = 0;
      bool ok = true;
      for (int n = 0; ok; ++n) {
        const int r = item_index(n, cta, G);
        if (r >= num_items) break;
        const Item it = make_item(p, r);
        for (int idx = 0; idx < it.U; ++idx) {
          const uint32_t gv = vc + uint32_t(idx), gk = kc + uint32_t(idx + 1);
          if (!mbar_wait(v_full0 + 8 * (gv & 1), (gv >> 1) & 1, wc, 17) ||
              (idx + 1 < it.U && !mbar_wait(k_full0 + 8 * (gk % 3), (gk / 3) & 1, wc, 15))) {
            ok = false;
            break;
          }
          mbar_arrive(p_full0);
          if (!mbar_wait(p_full0, (tb + uint32_t(idx)) & 1, wc, 19)) {
            ok = false;
            break;
          }
        }
        kc += uint32_t(it.U);
        vc += uint32_t(it.U);
        tb += uint32_t(it.U);
      }
    }
    __syncwarp();
  }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------------ softmax
    const int h = (warp >= 8) ? 1 : 0;  // query tile of this warpgroup
    const uint32_t quad = warp & 3;
    const int r = int(quad * 32 + lane);  // query row inside the tile = TMEM lane
    const uint32_t lane_addr = (quad * 32u) << 16;
    const uint32_t t_s = tmem_base + lane_addr + uint32_t(h * BKV);
    const uint32_t t_o = tmem_base + lane_addr + 256u + uint32_t(h * 128);
    const uint32_t s_full = s_full0 + 8 * h, p_full = p_full0 + 8 * h;
    const float c = p.scale_log2;
    uint32_t tb = 0;  // union tiles of earlier items
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int ri = item_index(n, cta, G);
      if (ri >= num_items) break;
      const Item it = make_item(p, ri);
      const int qb = it.q0 + h * BQ;
      const int i = qb + r;  // query position in the sequence
      const int kb_h = h ? it.kb1 : it.kb0, ke_h = h ? it.ke1 : it.ke0;
      float m_used = -INFINITY, l = 0.f;
      bool has_o = false;
      for (int idx = 0; idx < it.U; ++idx) {
        const int j = it.kt_begin + idx;
        if (!mbar_wait_warp(s_full, (tb + uint32_t(idx)) & 1, wc, 16)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (j >= kb_h && j <= ke_h) {
          // The whole S row, four loads in flight, one wait.
          uint32_t u[BKV];
#pragma unroll
          for (int ch = 0; ch < BKV / 32; ++ch)
            tmem_ld32(t_s + uint32_t(ch * 32), *reinterpret_cast<uint32_t(*)[32]>(u + ch * 32));
          tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(u));
          tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(u + 32));
          tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(u + 64));
          tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(u + 96));
          float s[BKV];
#pragma unroll
          for (int e = 0; e < BKV; ++e) s[e] = __uint_as_float(u[e]);
          const int k0 = j * BKV;
          const bool whole = (k0 + BKV - 1 <= qb) && (qb + BQ - 1 - k0 < p.window);
          if (!whole) {
#pragma unroll
            for (int e = 0; e < BKV; ++e) {
              const int d = i - (k0 + e);
              if (d < 0 || d >= p.window) s[e] = -INFINITY;
            }
          }
          // Row maximum: four independent chains of three-input maxima.
          float mx4[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float a = s[32 * q];
#pragma unroll
            for (int e = 1; e < 31; e += 2) a = max3f(a, s[32 * q + e], s[32 * q + e + 1]);
            mx4[q] = fmaxf(a, s[32 * q + 31]);
          }
          const float mx = fmaxf(max3f(mx4[0], mx4[1], mx4[2]), mx4[3]);
          const float mxs = mx * c;
          // Move the reference maximum only when the row maximum grew by more than 2^8
          // (from -inf, any finite maximum does); O is rescaled below, after P is stored.
          const bool grow = mxs > m_used + kRescaleThreshold;
          const float alpha = grow ? ex2_approx(m_used - mxs) : 1.f;
          if (grow) {
            l *= alpha;
            m_used = mxs;
          }
          const float m_eff = (m_used == -INFINITY) ? 0.f : m_used;
          // P_h over the first 64 columns of S_h (masked keys give exactly 0).
          l += probs_to_tmem(s, c, m_eff, t_s);
          tmem_st_wait();
          if (has_o && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
            for (int ch = 0; ch < DH / 32; ++ch) {
              uint32_t u[32];
              tmem_ld32(t_o + uint32_t(ch * 32), u);
              tmem_ld_wait(u);
#pragma unroll
              for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
              tmem_st32(t_o + uint32_t(ch * 32), u);
            }
            tmem_st_wait();
          }
          has_o = true;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (!ok) break;
      tb += uint32_t(it.U);
      if (has_o && !mbar_wait_warp(o_final0 + 8 * h, uint32_t(n) & 1, wc, 18)) break;
      if (has_o) {
        tc_fence_after();
        const float inv_l = 1.f / l;
        // training forward: the row's log2-sum-exp, from which the backward recomputes P
        if (p.lse != nullptr && i < p.S)
          p.lse[(int64_t(it.b) * p.nh + it.head) * p.lse_ld + i] = m_used + log2f(l);
        const int64_t off = (int64_t(it.b) * p.S + i) * p.out_ld + it.head * DH;
        bool bad = false;
#pragma unroll
        for (int ch = 0; ch < DH / 32; ++ch) {
          uint32_t u[32];
          tmem_ld32(t_o + uint32_t(ch * 32), u);
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
    }  // items
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
  static PerDeviceInit setup;  // per device: the shared-memory opt-in
  const cudaError_t attr = per_device_init(setup, [](int, int*) {
    return cudaFuncSetAttribute(swa_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(L::SMEM));
  });
  if (attr != cudaSuccess) return attr;
  const int64_t items = int64_t((p.num_q_tiles + 1) / 2) * p.nh * p.B;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffff) return cudaErrorInvalidValue;
  // Persistent: one CTA per SM (the CTA holds all 512 tensor-memory columns), each walking
  // its share of the items.
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t grid = items < sms ? items : sms;
  swa_kernel<DH><<<unsigned(grid), THREADS, L::SMEM, stream>>>(tmQK, tmVT, p, status, limit_ns);
  return cudaGetLastError();
}

}  // namespace

// Query and key tiles are both 128 rows, so tmK (the same q|k buffer) is not needed here.
cudaError_t launch_swa(const CUtensorMap& tmQ, const CUtensorMap& /*tmK*/, const CUtensorMap& tmVT,
                       const SwaParams& p, int* status, uint64_t limit_ns, cudaStream_t stream) {
  if (p.dh == 64) return launch_dh<64>(tmQ, tmVT, p, status, limit_ns, stream);
  if (p.dh == 128) return launch_dh<128>(tmQ, tmVT, p, status, limit_ns, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pb
