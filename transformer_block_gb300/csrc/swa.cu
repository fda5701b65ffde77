// swa.cu — flash-style sliding-window causal attention on the tensor cores, CTA pairs.
//
// For every sequence b, head j and query i:
//   o_i = sum_{k : 0 <= i - k < w} softmax_k(q_i . k_k / sqrt(dh)) v_k
// (MegaScale reading notes, section 1.1, "Sliding Window Attention", eqs. (5)-(6): each
// token attends to the most recent w tokens; the FlashAttention tiling of section 1.3
// keeps the score matrix on chip, so it never reaches HBM).
//
// Work comes in items: two 128-query tiles of one head of one sequence. A cluster of two
// CTAs (a CTA pair, one per SM) takes an item, CTA r the query tile q0 + 128 r, and both
// tiles go through the tensor cores together as pair products (tcgen05 cta_group::2,
// M = 256, issued by one thread of the even CTA):
//   S = Q K_j^T    each CTA reads its own Q tile and holds half (64 keys) of key tile K_j
//   O += P V_j     P from each CTA's tensor memory, each CTA holds half (dh/2 rows) of V_j^T
// so a key tile costs each SM half a K tile and half a V tile of loads and shared-memory
// reads, and one issuing thread drives two SMs' tensor cores. Each CTA's tensor memory
// holds two score buffers and O (S_a | S_b | O): S(t + 2) is queued behind O += P(t) V_t
// while the softmax of tile t + 1 runs, so one tile's scores are always being computed
// while the previous tile's probabilities are made.
//   warp 0     TMA producer (both CTAs): the item's Q tile (two slots, so the next item's Q
//              loads while this one runs), K halves (4-stage ring, two tiles ahead of V)
//              and V^T halves (3-stage ring); both CTAs' copies complete on the even
//              CTA's barriers (the pair form of the TMA load)
//   warp 1     even CTA: the MMA-issuing thread; both: tensor-memory owner
//   warp 2     even CTA: watcher: for tile t it waits for V_t, K_{t+2} and (when tile t + 2
//              starts an item) that item's Q, then adds an arrival to P(t)'s barrier, so
//              the issuer waits once per key tile
//   warp 3     idle (warps 0-3 form the warpgroup whose registers go to the softmax)
//   warps 4-11 softmax, two threads per query row (the row's TMEM lane): warps 4-7 take
//              keys 0-63 of the tile, warps 8-11 keys 64-127; the two halves of a row
//              exchange their maxima through shared memory, synchronised by an mbarrier
//              per TMEM lane quadrant (a bounded wait, like every other wait here)
// The softmax writes P (bf16) over the first 64 columns of its score buffer; the tensor
// pipe executes the issuing thread's products in order, so S(t + 2) overwrites P(t) only
// after O += P(t) V_t has read it. A key tile that one query tile of the item does not
// need still goes through the pair products; that CTA writes zeros as its P. Only tiles
// that cross the diagonal or the window's far edge are masked element by element.
// Online softmax in fp32 with exp2 (1/sqrt(dh) and log2(e) folded into one multiplier);
// O is rescaled only when a row maximum grows by more than 2^8 (after the previous PV
// product has finished with O), and the final O / l uses the same reference maximum as
// every P, so the result is unchanged up to rounding. V arrives transposed ([dh, keys] per
// head, written so by the first GEMM's epilogue), so the PV product reads a K-major
// operand. Items are numbered by pair index, heaviest first; the kernel is persistent, CTA
// pair c of G taking items c, 2G - 1 - c, 2G + c, ... (alternating directions).
#include "kernels.h"
#include "ptx.cuh"

namespace pb {
namespace {

constexpr int BQ = kSwaBQ, BKV = kSwaBKV;
static_assert(BQ == 128 && BKV == 128, "tile shape of this kernel");
constexpr int THREADS = 384;
// Registers per thread: at launch (the most 384 threads may have), then per warpgroup: the
// control warpgroup gives some up, the two softmax warpgroups take them.
constexpr uint32_t kRegsLaunch = 168, kRegsControl = 96, kRegsSoftmax = 200;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= THREADS * kRegsLaunch,
              "register split exceeds the launch allocation");
constexpr uint32_t TMEM_COLS = 512;
constexpr int K_STAGES = 4, V_STAGES = 3;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// Softmax warps p_full waits for: 8 per CTA, and the watcher.
constexpr uint32_t kPArrivals = 2 * 8 + 1;

template <int DH>
struct Layout {
  static constexpr int QBOX = BQ * 64 * 2;         // 128 query rows x 64 columns: 16 KB
  static constexpr int Q_TILE = BQ * DH * 2;       // DH / 64 boxes
  static constexpr int KBOX = 64 * 64 * 2;         // 64 keys x 64 columns: 8 KB
  static constexpr int KH_BYTES = 64 * DH * 2;     // this CTA's 64 keys (DH / 64 boxes)
  static constexpr int VBOX = (DH / 2) * 64 * 2;   // DH / 2 rows of V^T x 64 keys
  static constexpr int VH_BYTES = 2 * VBOX;        // DH / 2 rows x 128 keys
  static constexpr int Q_OFF = 0;                  // two slots
  static constexpr int K_OFF = Q_OFF + 2 * Q_TILE;
  static constexpr int V_OFF = K_OFF + K_STAGES * KH_BYTES;
  static constexpr int RED_OFF = V_OFF + V_STAGES * VH_BYTES;
  // row maxima [tile parity][half][128] and row sums [half][128] of the two softmax halves
  static constexpr int RED_BYTES = (2 * 2 * 128 + 2 * 128) * 4;
  static constexpr int BAR_OFF = RED_OFF + RED_BYTES;
  static constexpr int NUM_BARS = 29;
  static constexpr size_t NEED = size_t(BAR_OFF) + NUM_BARS * 8 + 16 + 1024;
  // At least enough shared memory that only one CTA fits per SM: the CTA takes all 512
  // tensor-memory columns.
  static constexpr size_t SMEM = NEED > 200 * 1024 ? NEED : 200 * 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory layout");
  static_assert(QBOX % 1024 == 0 && KBOX % 1024 == 0 && VBOX % 1024 == 0 && V_OFF % 1024 == 0,
                "128-byte swizzled boxes start on 1024-byte boundaries");
};

// One unit of work: a pair of 128-query tiles of one head of one sequence.
struct Item {
  int b, head, q0;
  int kb0, ke0, kb1, ke1;  // key-tile range [kb, ke] of query tile 0 / 1 (empty past seq)
  int kt_begin, U;         // first key tile the item visits, and how many it visits
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

// The n-th item of CTA pair c among G pairs: rounds of G items, dealt in alternating
// directions (c, then G - 1 - c), so the heavy items at the front even out across pairs.
__device__ __forceinline__ int item_index(int n, int c, int G) {
  return n * G + ((n & 1) ? G - 1 - c : c);
}

// Walks the key tiles of a pair's items in order: item n, its tile idx, and g, the tile's
// number over the pair's whole run (which fixes ring stages, buffers and barrier phases).
struct Cursor {
  int n, idx;
  uint32_t g;
  bool valid;
  Item it;
  __device__ void load(const SwaParams& p, int c, int G, int num_items) {
    const int r = item_index(n, c, G);
    valid = r < num_items;
    if (valid) it = make_item(p, r);
  }
  __device__ void start(const SwaParams& p, int c, int G, int num_items) {
    n = 0;
    idx = 0;
    g = 0;
    load(p, c, G, num_items);
  }
  __device__ void next(const SwaParams& p, int c, int G, int num_items) {
    ++g;
    if (++idx == it.U) {
      idx = 0;
      ++n;
      load(p, c, G, num_items);
    }
  }
};

// Half a softmax row: p_k = 2^(s_k c - m) rounded to bf16 into tensor memory at t_p
// (column m holds keys 2m and 2m + 1), 32 keys per store; returns the fp32 sum of the
// unrounded p_k. Scale, shift and sum run on packed pairs.
__device__ __forceinline__ float probs64_to_tmem(const float (&s)[64], float c, float m,
                                                 uint32_t t_p) {
  const uint64_t c2 = f2(c, c), nm2 = f2(-m, -m);
  uint64_t acc[4] = {0, 0, 0, 0};  // four independent partial sums of pairs
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
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
    tmem_st16(t_p + uint32_t(ch * 16), pk);
  }
  const uint64_t t = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
  float lo, hi;
  f2_split(t, lo, hi);
  return lo + hi;
}

template <int DH>
__global__ void __launch_bounds__(THREADS, 1)
    swa_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmVT, const SwaParams p, int* status,
               uint64_t limit_ns) {
  using L = Layout<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  // (E) = used in the even CTA only; (B) = in both CTAs (pair commits reach both).
  const uint32_t q_full0 = smem_u32(bars + 0);    // [2] (E) both CTAs' Q of a slot landed
  const uint32_t q_empty0 = smem_u32(bars + 2);   // [2] (B) the item's last S products done
  const uint32_t k_full0 = smem_u32(bars + 4);    // [4] (E)
  const uint32_t k_empty0 = smem_u32(bars + 8);   // [4] (B)
  const uint32_t v_full0 = smem_u32(bars + 12);   // [3] (E)
  const uint32_t v_empty0 = smem_u32(bars + 15);  // [3] (B)
  const uint32_t s_full0 = smem_u32(bars + 18);   // [2] (B) per score buffer
  const uint32_t p_full0 = smem_u32(bars + 20);   // [2] (E) both CTAs' P of a buffer, watcher
  // (B) a PV product finished. Waited for only before a rescale of O in the softmax of
  // tile t: S(t) done implies PV(t - 2) done, and PV(t) waits for that softmax, so the
  // barrier is then at the phase of PV(t - 1) or just past it (a parity wait is exact).
  const uint32_t pv_done = smem_u32(bars + 22);
  const uint32_t drain_bar = smem_u32(bars + 23); // (E)
  const uint32_t xch0 = smem_u32(bars + 24);      // [4] the two softmax halves of a quadrant
  // (B) an item's last PV product finished (one phase per item: the softmax reads O out
  // only after it, and the next item's first PV waits for that softmax).
  const uint32_t o_final = smem_u32(bars + 28);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red_max = reinterpret_cast<float*>(smem + L::RED_OFF);  // [2][2][128]
  float* red_l = red_max + 2 * 2 * 128;                            // [2][128]

  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  const int num_items = ((p.num_q_tiles + 1) / 2) * p.nh * p.B;
  const int G = int(gridDim.x) >> 1, pc_id = int(blockIdx.x) >> 1;
  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(q_full0 + 8 * s, 1);
      mbar_init(q_empty0 + 8 * s, 1);
      mbar_init(s_full0 + 8 * s, 1);
      mbar_init(p_full0 + 8 * s, kPArrivals);
    }
    for (int s = 0; s < K_STAGES; ++s) {
      mbar_init(k_full0 + 8 * s, 1);
      mbar_init(k_empty0 + 8 * s, 1);
    }
    for (int s = 0; s < V_STAGES; ++s) {
      mbar_init(v_full0 + 8 * s, 1);
      mbar_init(v_empty0 + 8 * s, 1);
    }
    for (int q = 0; q < 4; ++q) mbar_init(xch0 + 8 * q, 2);
    mbar_init(pv_done, 1);
    mbar_init(o_final, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVT);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive or pair copy
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, status, limit_ns};
  // Teardown waits for the pair's own copies and MMAs get at least a second, whatever the
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
        // Each CTA loads its own half of every tile into its own shared memory; the
        // copies complete on the even CTA's barriers, where the even CTA announces both
        // CTAs' bytes. A CTA refills a slot or stage only after the pair products read it
        // (the empty barriers), so its copies always count toward the phase the issuer
        // and the watcher wait for next.
        const uint32_t q_full_e = mapa_shared(q_full0, 0);
        const uint32_t k_full_e = mapa_shared(k_full0, 0);
        const uint32_t v_full_e = mapa_shared(v_full0, 0);
        uint32_t q_used = 0, k_used = 0, v_used = 0, q_par = 0, k_par = 0, v_par = 0;
        Cursor kc, vc;
        kc.start(p, pc_id, G, num_items);
        vc.start(p, pc_id, G, num_items);
        bool ok = true;
        while (ok && vc.valid) {
          // K runs two tiles ahead of V: S(t + 2) is issued right after O += P(t) V_t.
          while (ok && kc.valid && kc.g <= vc.g + 2) {
            const Item& it = kc.it;
            if (kc.idx == 0) {  // a new item: its Q tile first
              const uint32_t slot = uint32_t(kc.n) & 1, par = (uint32_t(kc.n) >> 1) & 1;
              if (!mbar_wait(q_empty0 + 8 * slot, par ^ 1, wc, 20)) {
                ok = false;
                break;
              }
              if (leader) mbar_arrive_expect_tx(q_full0 + 8 * slot, 2 * L::Q_TILE);
#pragma unroll
              for (int hb = 0; hb < DH / 64; ++hb)
                tma_load_3d_pair(sQ + slot * L::Q_TILE + hb * L::QBOX, &tmQ, q_full_e + 8 * slot,
                                 it.head * DH + hb * 64, it.q0 + int(rank) * BQ, it.b);
              q_par = (q_par & ~(1u << slot)) | (par << slot);
              q_used |= 1u << slot;
            }
            const uint32_t st = kc.g % K_STAGES, par = (kc.g / K_STAGES) & 1;
            if (!mbar_wait(k_empty0 + 8 * st, par ^ 1, wc, 11)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(k_full0 + 8 * st, 2 * L::KH_BYTES);
#pragma unroll
            for (int hb = 0; hb < DH / 64; ++hb)
              tma_load_3d_pair(sK + st * L::KH_BYTES + hb * L::KBOX, &tmK, k_full_e + 8 * st,
                               p.H + it.head * DH + hb * 64,
                               (it.kt_begin + kc.idx) * BKV + int(rank) * 64, it.b);
            k_par = (k_par & ~(1u << st)) | (par << st);
            k_used |= 1u << st;
            kc.next(p, pc_id, G, num_items);
          }
          if (!ok) break;
          const Item& it = vc.it;
          const uint32_t st = vc.g % V_STAGES, par = (vc.g / V_STAGES) & 1;
          if (!mbar_wait(v_empty0 + 8 * st, par ^ 1, wc, 10)) break;
          if (leader) mbar_arrive_expect_tx(v_full0 + 8 * st, 2 * L::VH_BYTES);
          const int vt_row = (it.b * p.nh + it.head) * DH + int(rank) * (DH / 2);
#pragma unroll
          for (int kh = 0; kh < 2; ++kh)
            tma_load_2d_pair(sV + st * L::VH_BYTES + kh * L::VBOX, &tmVT, v_full_e + 8 * st,
                             (it.kt_begin + vc.idx) * BKV + kh * 64, vt_row);
          v_par = (v_par & ~(1u << st)) | (par << st);
          v_used |= 1u << st;
          vc.next(p, pc_id, G, num_items);
        }
        // Every copy of the pair must land before either CTA exits: the even CTA waits for
        // its full barriers (which count the odd CTA's bytes too); the odd CTA is held at
        // the final cluster barrier until then.
        if (leader) {
          for (uint32_t s = 0; s < 2; ++s)
            if (q_used & (1u << s)) mbar_wait_drain(q_full0 + 8 * s, (q_par >> s) & 1u, drain_ns);
          for (uint32_t s = 0; s < uint32_t(K_STAGES); ++s)
            if (k_used & (1u << s)) mbar_wait_drain(k_full0 + 8 * s, (k_par >> s) & 1u, drain_ns);
          for (uint32_t s = 0; s < uint32_t(V_STAGES); ++s)
            if (v_used & (1u << s)) mbar_wait_drain(v_full0 + 8 * s, (v_par >> s) & 1u, drain_ns);
        }
      }
    } else if (warp == 1) {
      if (lane == 0 && leader) {
        // ---------------------------------------------------------------- MMA issuer
        const uint32_t id_s = idesc_f32acc(2 * BQ, BKV);
        const uint32_t id_o = idesc_f32acc(2 * BQ, DH);
        // Shared-memory descriptors: the start-address field is the byte address / 16, so
        // a descriptor for base + offset is the base's descriptor + offset / 16 (all
        // addresses stay below 256 KB, inside the 14-bit field).
        const uint64_t dQ = sdesc_kmajor_sw128(sQ), dK = sdesc_kmajor_sw128(sK),
                       dV = sdesc_kmajor_sw128(sV);
        Cursor sc, pc;
        sc.start(p, pc_id, G, num_items);
        pc.start(p, pc_id, G, num_items);
        // S(t) = Q K_t^T into score buffer t & 1 of both CTAs.
        auto issue_s = [&]() {
          const uint32_t st = sc.g % K_STAGES, buf = sc.g & 1, slot = uint32_t(sc.n) & 1;
          const uint64_t da = dQ + uint64_t((slot * L::Q_TILE) >> 4);
          const uint64_t db = dK + uint64_t((st * L::KH_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk)
            mma_f16kind_ss_pair(tmem_base + buf * BKV,
                                da + uint64_t(((kk >> 2) * L::QBOX) >> 4) + 2 * (kk & 3),
                                db + uint64_t(((kk >> 2) * L::KBOX) >> 4) + 2 * (kk & 3), id_s,
                                kk > 0 ? 1u : 0u);
          mma_commit_pair(s_full0 + 8 * buf, 0x3);
          mma_commit_pair(k_empty0 + 8 * st, 0x3);
          if (sc.idx + 1 == sc.it.U) mma_commit_pair(q_empty0 + 8 * slot, 0x3);
          sc.next(p, pc_id, G, num_items);
        };
        bool ok = true;
        // The first two score products; after that the watcher certifies what each needs.
        for (int t = 0; ok && t < 2 && sc.valid; ++t) {
          const uint32_t st = sc.g % K_STAGES;
          if ((sc.idx == 0 && !mbar_wait(q_full0 + 8 * (uint32_t(sc.n) & 1),
                                         (uint32_t(sc.n) >> 1) & 1, wc, 12)) ||
              !mbar_wait(k_full0 + 8 * st, (sc.g / K_STAGES) & 1, wc, 14)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s();
        }
        while (ok && pc.valid) {
          const uint32_t buf = pc.g & 1;
          // P(t) from both CTAs, and (the watcher's arrival) V_t, K_{t+2} and, if tile t + 2
          // starts an item, its Q.
          if (!mbar_wait(p_full0 + 8 * buf, (pc.g >> 1) & 1, wc, 13)) break;
          tc_fence_after();
          const uint32_t vst = pc.g % V_STAGES;
          const uint64_t dv = dV + uint64_t((vst * L::VH_BYTES) >> 4);
          const uint32_t t_p = tmem_base + buf * BKV;
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            mma_f16kind_ts_pair(tmem_base + 2u * BKV, t_p + uint32_t(kk * 8),
                                dv + uint64_t(((kk >> 2) * L::VBOX) >> 4) + 2 * (kk & 3), id_o,
                                (pc.idx > 0 || kk > 0) ? 1u : 0u);
          mma_commit_pair(v_empty0 + 8 * vst, 0x3);
          mma_commit_pair(pv_done, 0x3);
          if (pc.idx + 1 == pc.it.U) mma_commit_pair(o_final, 0x3);
          pc.next(p, pc_id, G, num_items);
          if (sc.valid) issue_s();
        }
        // Every product this thread issued (into both CTAs' tensor memory) must finish
        // before either CTA releases it.
        mma_commit_pair(drain_bar, 0x1);
        mbar_wait_drain(drain_bar, 0, drain_ns);
      }
    } else if (warp == 2) {
      if (lane == 0 && leader) {
        // ---------------------------------------------------------------- watcher
        // Adds one arrival per key tile t to P(t)'s barrier once V_t, K_{t+2} and (if tile
        // t + 2 starts an item) that item's Q have landed, then waits for the phase to
        // complete, so it never arrives in a later phase of the same barrier.
        Cursor w, a;
        w.start(p, pc_id, G, num_items);
        a.start(p, pc_id, G, num_items);
        for (int t = 0; t < 2 && a.valid; ++t) a.next(p, pc_id, G, num_items);
        while (w.valid) {
          const uint32_t vs = w.g % V_STAGES;
          if (!mbar_wait(v_full0 + 8 * vs, (w.g / V_STAGES) & 1, wc, 17)) break;
          if (a.valid) {
            if (!mbar_wait(k_full0 + 8 * (a.g % K_STAGES), (a.g / K_STAGES) & 1, wc, 15)) break;
            if (a.idx == 0 && !mbar_wait(q_full0 + 8 * (uint32_t(a.n) & 1),
                                         (uint32_t(a.n) >> 1) & 1, wc, 21))
              break;
          }
          const uint32_t buf = w.g & 1;
          mbar_arrive(p_full0 + 8 * buf);
          if (!mbar_wait(p_full0 + 8 * buf, (w.g >> 1) & 1, wc, 19)) break;
          w.next(p, pc_id, G, num_items);
          if (a.valid) a.next(p, pc_id, G, num_items);
        }
      }
    }
    __syncwarp();
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------------ softmax
    const uint32_t quad = warp & 3, half = (warp - 4) >> 2;
    const int r = int(quad * 32 + lane);  // query row inside the tile = TMEM lane
    const uint32_t lane_addr = (quad * 32u) << 16;
    const uint32_t t_row = tmem_base + lane_addr;
    const uint32_t t_o = t_row + 2u * BKV + half * (DH / 2);
    const uint32_t xch = xch0 + 8 * quad;  // the row halves' exchange barrier
    uint32_t xn = 0;                       // exchanges so far (its phase)
    // Both halves of the quadrant's rows have written their value to shared memory (and
    // finished their tensor-memory reads of the tile): one arrival per warp, then the
    // bounded wait for the phase.
    auto exchange = [&]() -> bool {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(xch);
      const bool done = mbar_wait_warp(xch, xn & 1, wc, 23);
      ++xn;
      tc_fence_after();
      return done;
    };
    // P(t)'s barrier lives in the even CTA.
    const uint32_t p_full_e = leader ? p_full0 : mapa_shared(p_full0, 0);
    const float c = p.scale_log2;
    Cursor cur;
    cur.start(p, pc_id, G, num_items);
    bool ok = true;
    while (ok && cur.valid) {
      const Item it = cur.it;
      const uint32_t n_item = uint32_t(cur.n);
      const int qb = it.q0 + int(rank) * BQ;
      const int i = qb + r;  // query position in the sequence
      const int kb_h = rank ? it.kb1 : it.kb0, ke_h = rank ? it.ke1 : it.ke0;
      float m_used = -INFINITY, l = 0.f;
      bool has_o = false;
      for (int idx = 0; idx < it.U; ++idx) {
        const uint32_t g = cur.g, buf = g & 1;
        if (!mbar_wait_warp(s_full0 + 8 * buf, (g >> 1) & 1, wc, 16)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_s = t_row + buf * BKV;
        const int j = it.kt_begin + idx;
        if (j >= kb_h && j <= ke_h) {
          uint32_t u[64];
          tmem_ld32(t_s + half * 64, *reinterpret_cast<uint32_t(*)[32]>(u));
          tmem_ld32(t_s + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
          tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(u));
          tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(u + 32));
          float s[64];
#pragma unroll
          for (int e = 0; e < 64; ++e) s[e] = __uint_as_float(u[e]);
          const int k0 = j * BKV;
          const bool whole = (k0 + BKV - 1 <= qb) && (qb + BQ - 1 - k0 < p.window);
          if (!whole) {
            const int kh0 = k0 + int(half) * 64;
#pragma unroll
            for (int e = 0; e < 64; ++e) {
              const int d = i - (kh0 + e);
              if (d < 0 || d >= p.window) s[e] = -INFINITY;
            }
          }
          // Half-row maximum: two independent chains of three-input maxima.
          float a0 = s[0], a1 = s[32];
#pragma unroll
          for (int e = 1; e < 31; e += 2) {
            a0 = max3f(a0, s[e], s[e + 1]);
            a1 = max3f(a1, s[32 + e], s[32 + e + 1]);
          }
          float mx = max3f(a0, a1, fmaxf(s[31], s[63]));
          // The row maximum: exchange with the other half of the row.
          float* slot = red_max + (g & 1) * 256;
          slot[half * 128 + r] = mx;
          if (!exchange()) {
            ok = false;
            break;
          }
          mx = fmaxf(mx, slot[(half ^ 1) * 128 + r]);
          const float mxs = mx * c;
          // Move the reference maximum only when the row maximum grew by more than 2^8
          // (from -inf, any finite maximum does); O is rescaled below, after P is stored.
          // Both halves of a row see the same maximum and take the same decision.
          const bool grow = mxs > m_used + kRescaleThreshold;
          const float alpha = grow ? ex2_approx(m_used - mxs) : 1.f;
          if (grow) {
            l *= alpha;
            m_used = mxs;
          }
          const float m_eff = (m_used == -INFINITY) ? 0.f : m_used;
          // P over this half's 32 columns of the first 64 (masked keys give exactly 0).
          l += probs64_to_tmem(s, c, m_eff, t_s + half * 32);
          tmem_st_wait();
          if (has_o && __any_sync(0xffffffffu, grow)) {
            // O may be rescaled only after the previous PV product has finished with it.
            if (!mbar_wait_warp(pv_done, (g - 1) & 1, wc, 22)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int ch = 0; ch < DH / 64; ++ch) {
              uint32_t v[32];
              tmem_ld32(t_o + uint32_t(ch * 32), v);
              tmem_ld_wait(v);
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
              tmem_st32(t_o + uint32_t(ch * 32), v);
            }
            tmem_st_wait();
          }
          has_o = true;
        } else {
          // Key tile outside this query tile's range: P = 0 for the pair product.
          uint32_t z[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) z[e] = 0u;
          tmem_st16(t_s + half * 32, z);
          tmem_st16(t_s + half * 32 + 16, z);
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(p_full_e + 8 * buf);
          else
            mbar_arrive_remote(p_full_e + 8 * buf);
        }
        cur.next(p, pc_id, G, num_items);
      }
      if (!ok) break;
      if (has_o) {
        // The item's last PV product has finished: O is final.
        if (!mbar_wait_warp(o_final, n_item & 1, wc, 18)) break;
        tc_fence_after();
        red_l[half * 128 + r] = l;
        if (!exchange()) break;
        const float l_row = l + red_l[(half ^ 1) * 128 + r];
        const float inv_l = 1.f / l_row;
        // training forward: the row's log2-sum-exp, from which the backward recomputes P
        if (half == 0 && p.lse != nullptr && i < p.S)
          p.lse[(int64_t(it.b) * p.nh + it.head) * p.lse_ld + i] = m_used + log2f(l_row);
        const int64_t off =
            (int64_t(it.b) * p.S + i) * p.out_ld + it.head * DH + int(half) * (DH / 2);
        bool bad = false;
#pragma unroll
        for (int ch = 0; ch < DH / 64; ++ch) {
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
  cluster_sync();  // no CTA leaves while its peer may still arrive on it or MMA into it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int DH>
cudaError_t launch_dh(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmVT,
                      const SwaParams& p, int* status, uint64_t limit_ns, cudaStream_t stream) {
  using L = Layout<DH>;
  const int64_t items = int64_t((p.num_q_tiles + 1) / 2) * p.nh * p.B;
  if (items <= 0) return cudaSuccess;
  if (items > 0x3fffffff) return cudaErrorInvalidValue;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = L::SMEM;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  // Per device: the shared-memory opt-in and how many CTA pairs fit at once.
  static PerDeviceInit setup;
  int max_pairs = 0;
  const cudaError_t e = per_device_init(
      setup,
      [&](int dev, int* out) {
        cudaError_t r = cudaFuncSetAttribute(swa_kernel<DH>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(L::SMEM));
        if (r != cudaSuccess) return r;
        int sms = 0;
        r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (r != cudaSuccess) return r;
        cudaLaunchConfig_t occ = cfg;
        occ.gridDim = dim3(2 * (sms / 2), 1, 1);
        int n = 0;
        r = cudaOccupancyMaxActiveClusters(&n, swa_kernel<DH>, &occ);
        *out = (r == cudaSuccess && n > 0) ? n : 0;
        return r;
      },
      &max_pairs);
  if (e != cudaSuccess) return e;
  if (max_pairs <= 0) return cudaErrorLaunchOutOfResources;
  // Persistent: every CTA pair that fits at once, each walking its share of the items.
  const int64_t pairs = items < max_pairs ? items : max_pairs;
  cfg.gridDim = dim3(unsigned(2 * pairs), 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, swa_kernel<DH>, tmQ, tmK, tmVT, p, status, limit_ns);
}

}  // namespace

// tmQ: the q|k buffer in boxes of 64 columns x 128 rows (query tiles); tmK: the same buffer
// in boxes of 64 columns x 64 rows (half key tiles); tmVT: v^T in boxes of 64 keys x dh/2
// rows (half V^T tiles).
cudaError_t launch_swa(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmVT,
                       const SwaParams& p, int* status, uint64_t limit_ns, cudaStream_t stream) {
  if (p.dh == 64) return launch_dh<64>(tmQ, tmK, tmVT, p, status, limit_ns, stream);
  if (p.dh == 128) return launch_dh<128>(tmQ, tmK, tmVT, p, status, limit_ns, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pb
