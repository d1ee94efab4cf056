// Fused attention forward on CTA pairs (tcgen05 cta_group::2), bf16, d = 128,
// non-causal: the 2-CTA tile of the FA4 forward ("FlashAttention-4's Softmax
// Tricks", section "The emulated exp2": the 2-CTA non-causal d = 128
// configuration; section "Why exp is the bottleneck": the 1-CTA and 2-CTA
// tables).
//
// A cluster of two CTAs on two SMs shares every product. Each CTA keeps two
// 128-row query tiles (its rows of the pair's two 256-row tiles) and the
// TMEM of the 1-CTA kernel (fwd_bf16.cuh): S0, S1, O0, O1. Per key block of
// 128 keys, the pair's S_t = Q_t K^T is one M = 256 product issued by CTA 0,
// with its rows in each CTA's TMEM and its N = 128 key columns split: CTA 0
// holds keys 0-63 of the block, CTA 1 keys 64-127 (K-major, 128-byte
// swizzle). O_t += P_t V likewise: P from each CTA's TMEM, V's d columns
// split, 0-63 in CTA 0 and 64-127 in CTA 1 (MN-major). So each SM stages
// half of every K and V block: a ring of ten 16 KiB slots instead of five
// 32 KiB ones, and half the K/V traffic from L2. Each CTA loads its own
// halves with plain TMA (no multicast).
//
//   warp 8 (both)   TMA: its Q tiles once per item, its K and V halves per block
//   warp 9 (CTA 0)  MMA issuer for the pair (one elected thread)
//   warp 9 (CTA 1)  forwards its loads' completion to CTA 0's barriers
//   warps 0-7       softmax, thread = query row, as in the 1-CTA kernel; the
//                   hand-over of P counts CTA 1's threads on CTA 0's barrier
//
// The softmax, the rescale rule, the inline correction and the epilogue are
// those of the 1-CTA kernel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fwd_bf16.cuh"
#include "kernel_setup.h"
#include "ptx.cuh"
#include "schedule.h"

namespace attn {

struct Fwd2Cfg {
  static constexpr int D = 128;
  static constexpr uint32_t kQBoxBytes = 128u * 128u;       // 128 rows x 64 columns
  static constexpr uint32_t kTileBytes = 2 * kQBoxBytes;    // one 128 x 128 Q tile
  static constexpr uint32_t kKBoxBytes = 64u * 128u;        // 64 keys x 64 columns
  static constexpr uint32_t kHalfBytes = 16384u;            // a K half (2 boxes) or a V half (1 box)
  static constexpr int kSlots = 10;
  static constexpr uint32_t kRingOff = 2 * kTileBytes;
  static constexpr uint32_t kBarOff = kRingOff + kSlots * kHalfBytes;
  // q_full, peer_q, full[kSlots], peer_full[kSlots], empty[kSlots], s_full[2],
  // p_full[2][2], o_final[2], drain, q_empty
  static constexpr int kNumBars = 2 + 3 * kSlots + 10;
  static constexpr uint32_t kHolderOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kAbortOff = kHolderOff + 4;
  static constexpr uint32_t kSmemBytes = kAbortOff + 4 + 1024;
  static constexpr int kThreads = 384;
  static constexpr uint32_t kRegsSoftmax = 208;
  static constexpr uint32_t kRegsOther = 88;
  static constexpr int kLaunchRegs = 168;
  static constexpr uint32_t kTmemCols = 512;
  __host__ __device__ static constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 256u + (t ? 128u : 0u); }
};

// Bounded wait at cluster scope (a barrier other CTAs arrive on); as
// wait_bar. RELAXED: no acquire (the P hand-over, whose data is TMEM ordered
// by the tcgen05 fences).
template <bool RELAXED>
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                 unsigned int* status, uint32_t where) {
  auto try_once = [&] { return RELAXED ? mbar_try_wait_cluster_relaxed(bar, parity) : mbar_try_wait_cluster(bar, parity); };
  if (try_once()) return true;
  const long long t0 = clock64();
  while (true) {
    if (try_once()) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      *abort_flag = 1u;
      record_status(status, kStatusTimeout, where);
      return false;
    }
  }
}

// args.n_pairs here counts 512-row groups of a head (the pair's two 256-row
// tiles); work items are (head, group).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(384, 1)
    attn_fwd_bf16_2cta_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kh,
                              const __grid_constant__ CUtensorMap tm_v, const FwdArgs args,
                              const __grid_constant__ WorkList wl) {
  using C = Fwd2Cfg;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar_q = sbase + C::kBarOff;
  const uint32_t bar_peer_q = bar_q + 8u;
  auto bar_full = [&](int i) { return bar_q + 8u * (2 + i); };
  auto bar_peer_full = [&](int i) { return bar_q + 8u * (2 + C::kSlots + i); };
  auto bar_empty = [&](int i) { return bar_q + 8u * (2 + 2 * C::kSlots + i); };
  auto bar_s = [&](int t) { return bar_q + 8u * (2 + 3 * C::kSlots + t); };
  auto bar_p = [&](int t, int h) { return bar_q + 8u * (4 + 3 * C::kSlots + 2 * t + h); };
  auto bar_o = [&](int t) { return bar_q + 8u * (8 + 3 * C::kSlots + t); };
  const uint32_t bar_drain = bar_q + 8u * (10 + 3 * C::kSlots);
  const uint32_t bar_qe = bar_q + 8u * (11 + 3 * C::kSlots);
  uint32_t* holder = reinterpret_cast<uint32_t*>(smem + C::kHolderOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kAbortOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int cluster = static_cast<int>(cluster_id_x());
  const int n_clusters = static_cast<int>(cluster_count_x());
  const int total_items = args.bh * args.n_pairs;
  auto item_of = [&](int k) {
    if (args.use_list) {
      const int idx = wl.first[cluster] + k;
      return idx < wl.first[cluster + 1] ? static_cast<int>(wl.item[idx]) : total_items;
    }
    const long long g = n_clusters;
    const long long o = k * g + ((k & 1) ? g - 1 - cluster : cluster);
    return o < total_items ? static_cast<int>(o) : total_items;
  };
  auto coords = [&](int it, int& bh, int& grp) { item_coords(it, args.bh, args.n_pairs, args.band, bh, grp); };
  const int nkv = args.n_kv_blocks;
  // first row of this CTA's tile t in a group: the pair's tile t covers rows
  // [512 g + 256 t, +256), CTA 0 the first 128 of them
  auto tile_row = [&](int grp, int t) { return grp * 512 + t * 256 + static_cast<int>(rank) * 128; };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_peer_q, 1);
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_peer_full(i), 1);
      mbar_init(bar_empty(i), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s(t), 1);
      // CTA 0's 128 softmax threads of the tile, and CTA 1's
      mbar_init(bar_p(t, 0), 256);
      mbar_init(bar_p(t, 1), 256);
      mbar_init(bar_o(t), 1);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_qe, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc_pair(smem_addr(holder), C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  // both CTAs' barriers are initialised before either arrives on the other's
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *holder;

  if (warp >= 8) {
    regs_to<C::kRegsOther, C::kLaunchRegs>();
    if (warp == 8) {
      // ---------------------------------------------------------- TMA (both CTAs): own Q tiles and K/V halves
      const uint32_t leader = elect_one();
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      int seq = 0;
      uint32_t slot = 0, ph = 0;
      bool ok = true;
      int qi = 0;
      for (int it = item_of(0); ok && it < total_items; it = item_of(++qi)) {
        int bh, grp;
        coords(it, bh, grp);
        if (qi > 0) {
          ok = __all_sync(0xffffffffu, wait_bar(bar_qe, (qi - 1) & 1, abort_flag, args.status, 13));
          if (!ok) break;
        }
        if (leader) {
          mbar_arrive_expect_tx(bar_q, 2 * C::kTileBytes);
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int b = 0; b < 2; ++b)
              tma_load_3d_hint(sbase + t * C::kTileBytes + b * C::kQBoxBytes, &tm_q, bar_q, b * 64, tile_row(grp, t),
                               bh, pol_q);
        }
        for (int j = 0; ok && j < nkv; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            ok = __all_sync(0xffffffffu, wait_bar(bar_empty(slot), ph ^ 1u, abort_flag, args.status, 1));
            if (!ok) break;
            if (leader) {
              const uint32_t dst = sbase + C::kRingOff + slot * C::kHalfBytes;
              mbar_arrive_expect_tx(bar_full(slot), C::kHalfBytes);
              if (kv == 0) {
                // keys [128 j + 64 rank, +64), all d columns (two 64-column boxes)
#pragma unroll
                for (int b = 0; b < 2; ++b)
                  tma_load_3d_hint(dst + b * C::kKBoxBytes, &tm_kh, bar_full(slot), b * 64,
                                   j * 128 + static_cast<int>(rank) * 64, bh, pol_kv);
              } else {
                // all 128 keys, d columns [64 rank, +64)
                tma_load_3d_hint(dst, &tm_v, bar_full(slot), static_cast<int>(rank) * 64, j * 128, bh, pol_kv);
              }
            }
            ++seq;
            if (++slot == static_cast<uint32_t>(C::kSlots)) {
              slot = 0;
              ph ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        drain_bar(bar_q, (qi & 1) ^ 1);
        for (int s = seq - C::kSlots < 0 ? 0 : seq - C::kSlots; s < seq; ++s)
          drain_bar(bar_full(s % C::kSlots), (s / C::kSlots) & 1);
      }
      __syncwarp();
    } else if (warp == 9 && rank == 1) {
      // ---------------------------------------------------------- CTA 1: forward load completions to CTA 0
      // In the producer's order: each of this CTA's loads (Q, then K_j and V_j)
      // is reported on CTA 0's matching peer barrier once it has landed here.
      // A slot is refilled only after CTA 0's MMAs have used it, which needs
      // this report first, so the phases seen here never run ahead.
      const uint32_t leader = elect_one();
      const uint32_t peer_q0 = cluster_addr(bar_peer_q, 0);
      uint32_t slot = 0, ph = 0;
      bool ok = true;
      int qi = 0;
      for (int it = item_of(0); ok && it < total_items; it = item_of(++qi)) {
        ok = __all_sync(0xffffffffu, wait_bar(bar_q, qi & 1, abort_flag, args.status, 20));
        if (!ok) break;
        if (leader) mbar_arrive_remote(peer_q0);
        for (int j = 0; ok && j < nkv; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            ok = __all_sync(0xffffffffu, wait_bar(bar_full(slot), ph, abort_flag, args.status, 21));
            if (!ok) break;
            if (leader) mbar_arrive_remote(cluster_addr(bar_peer_full(slot), 0));
            if (++slot == static_cast<uint32_t>(C::kSlots)) {
              slot = 0;
              ph ^= 1u;
            }
          }
        }
      }
      __syncwarp();
    } else if (warp == 9) {
      // ---------------------------------------------------------- CTA 0: MMA issuer for the pair
      const uint32_t leader = elect_one();
      auto commit_both = [&](uint32_t bar) {
        if (leader) tc_commit_pair(bar);
      };
      auto wait = [&](uint32_t bar, uint32_t parity, uint32_t where) {
        return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, args.status, where));
      };
      // the load reports of CTA 1 (release / acquire at cluster scope: CTA 1's
      // shared memory, written by its TMA, is read by these products)
      auto wait_cl = [&](uint32_t bar, uint32_t parity, uint32_t where) {
        return __all_sync(0xffffffffu, wait_bar_cluster<false>(bar, parity, abort_flag, args.status, where));
      };
      // P of both CTAs (relaxed: TMEM, ordered by the tcgen05 fences)
      auto wait_p = [&](uint32_t bar, uint32_t parity, uint32_t where) {
        return __all_sync(0xffffffffu, wait_bar_cluster<true>(bar, parity, abort_flag, args.status, where));
      };
      // a ring slot has landed in both CTAs
      auto wait_slot = [&](uint32_t slot, uint32_t parity, uint32_t where) {
        return wait(bar_full(slot), parity, where) && wait_cl(bar_peer_full(slot), parity, where);
      };
      constexpr uint32_t kIdS = idesc_bf16_f32(256, 128, false);
      constexpr uint32_t kIdO = idesc_bf16_f32(256, D, true);
      constexpr uint32_t kSlotStep = C::kHalfBytes >> 4;
      const uint64_t q0 = smem_desc_sw128(sbase, 16, 1024);
      const uint32_t desc_hi = static_cast<uint32_t>(q0 >> 32);
      const uint32_t q_lo[2] = {static_cast<uint32_t>(q0),
                                static_cast<uint32_t>(smem_desc_sw128(sbase + C::kTileBytes, 16, 1024))};
      const uint32_t k_ring = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kRingOff, 16, 1024));
      // V halves: one 64-column MN atom per CTA (the leading offset is not used)
      const uint32_t v_ring = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kRingOff, C::kHalfBytes, 1024));
      // K-major steps of K = 16: 32 bytes inside a 128-byte swizzle row, the
      // fifth starts the next 64-column box (Q: 16 KiB boxes, K halves: 8 KiB)
      auto q_step = [](int kk) -> uint32_t { return ((kk >> 2) * C::kQBoxBytes + (kk & 3) * 32) >> 4; };
      auto k_step = [](int kk) -> uint32_t { return ((kk >> 2) * C::kKBoxBytes + (kk & 3) * 32) >> 4; };
      auto issue_s = [&](int t, uint32_t slot) {
        const uint32_t a = q_lo[t];
        const uint32_t b = k_ring + slot * kSlotStep;
        const uint32_t d = tmem + C::col_s(t);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_lo_pair(d, a + q_step(kk), b + k_step(kk), desc_hi, kIdS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, uint32_t slot, int h, bool first) {
        const uint32_t b = v_ring + slot * kSlotStep;
        const uint32_t d = tmem + C::col_o(t);
        const uint32_t a = tmem + C::col_s(t);
        if (leader) {
#pragma unroll
          for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
            mma_ts_lo_pair(d, a + kk * 8, b + kk * 128, desc_hi, kIdO, (!first || kk > 0) ? 1u : 0u);
        }
      };
      auto advance2 = [](uint32_t& slot, uint32_t& phase) {
        slot += 2;
        if (slot >= static_cast<uint32_t>(C::kSlots)) {
          slot -= C::kSlots;
          phase ^= 1u;
        }
      };
      uint32_t ks = 0, kph = 0;
      uint32_t vs = 1, vph = 0;
      uint32_t gb = 0;  // blocks of either tile before this item
      bool ok = true;
      int qi = 0;
      for (int it = item_of(0); ok && it < total_items; it = item_of(++qi)) {
        const int n = nkv;
        ok = wait(bar_q, qi & 1, 2) && wait_cl(bar_peer_q, qi & 1, 2) && wait_slot(ks, kph, 3);
        if (!ok) break;
        tc_fence_after();
        issue_s(0, ks);
        commit_both(bar_s(0));
        issue_s(1, ks);
        commit_both(bar_s(1));
        commit_both(bar_empty(ks));
        if (n == 1) commit_both(bar_qe);
        for (int j = 0; ok && j < n; ++j) {
          if (!wait_slot(vs, vph, 4)) {
            ok = false;
            break;
          }
          uint32_t ks_next = ks, kph_next = kph;
          advance2(ks_next, kph_next);
          const uint32_t par = (gb + j) & 1;
          ok = wait_p(bar_p(0, 0), par, 5);
          if (!ok) break;
          tc_fence_after();
          issue_pv(0, vs, 0, j == 0);
          ok = wait_p(bar_p(0, 1), par, 11);
          if (!ok) break;
          tc_fence_after();
          issue_pv(0, vs, 1, false);
          if (j + 1 < n) {
            ok = wait_slot(ks_next, kph_next, 6);
            if (!ok) break;
            tc_fence_after();
            issue_s(0, ks_next);
            commit_both(bar_s(0));
          } else {
            commit_both(bar_o(0));
          }
          ok = wait_p(bar_p(1, 0), par, 7);
          if (!ok) break;
          tc_fence_after();
          issue_pv(1, vs, 0, j == 0);
          ok = wait_p(bar_p(1, 1), par, 12);
          if (!ok) break;
          tc_fence_after();
          issue_pv(1, vs, 1, false);
          commit_both(bar_empty(vs));
          if (j + 1 < n) {
            issue_s(1, ks_next);
            commit_both(bar_s(1));
            commit_both(bar_empty(ks_next));
            if (j + 2 == n) commit_both(bar_qe);
          } else {
            commit_both(bar_o(1));
          }
          ks = ks_next;
          kph = kph_next;
          advance2(vs, vph);
        }
        gb += n;
      }
      // nothing of the pair's may still be executing when TMEM is released
      if (leader) tc_commit_pair_local(bar_drain);
      drain_bar(bar_drain, 0);
      __syncwarp();
    }
  } else {
    // ============================================================ softmax warpgroups (both CTAs)
    regs_to<C::kRegsSoftmax, C::kLaunchRegs>();
    const int t = warp >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + C::col_s(t);
    const uint32_t o_tm = tmem + lane_off + C::col_o(t);
    const float sl2 = args.scale_log2;
    const float2 sl2_2 = make_float2(sl2, sl2);
    // P of this tile is ready: CTA 0's threads arrive on their own barrier;
    // in CTA 1 each warp's threads have waited for their TMEM stores and
    // fenced them (tcgen05.fence::before_thread_sync), the warp synchronises,
    // and one lane arrives for all 32 on CTA 0's barrier: four remote
    // arrivals per hand-over instead of 128, relaxed (the data is TMEM, whose
    // order the tcgen05 fences give; a release at cluster scope here cost
    // ~800 ns per hand-over)
    const uint32_t p_bar[2] = {rank == 0 ? bar_p(t, 0) : cluster_addr(bar_p(t, 0), 0),
                               rank == 0 ? bar_p(t, 1) : cluster_addr(bar_p(t, 1), 0)};
    auto arrive_p = [&](int h) {
      if (rank == 0) {
        mbar_arrive(p_bar[h]);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(p_bar[h], 32u);
      }
    };
    bool ok = true;
    uint32_t gb = 0;
    int qi = 0;
    for (int it = item_of(0); ok && it < total_items; it = item_of(++qi)) {
      int bh, grp;
      coords(it, bh, grp);
      const int grow = tile_row(grp, t) + r;
      const int nt = nkv;
      float m = -INFINITY;
      float2 acc[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) acc[a] = make_float2(0.f, 0.f);
      for (int j = 0; j < nt; ++j) {
        const uint32_t par = (gb + j) & 1;
        ok = wait_bar(bar_s(t), par, abort_flag, args.status, 16 + t);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float2 s[64];
        {
          uint32_t u[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(s_tm + 32 * c, u[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            reg_fence32(u[c]);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              s[16 * c + i] = make_float2(__uint_as_float(u[c][2 * i]), __uint_as_float(u[c][2 * i + 1]));
          }
        }
        const int kv0 = j * 128;
        const bool need_mask = kv0 + 128 > args.n;
        if (need_mask) {
          const int lim = args.n - 1 - kv0;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            if (2 * c > lim) s[c].x = -INFINITY;
            if (2 * c + 1 > lim) s[c].y = -INFINITY;
          }
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmax3(s[i].x, s[i].y, s[8 + i].x);
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[8 + i].y, s[16 + i].x);
#pragma unroll
        for (int c = 16; c < 56; c += 8)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[c + i].y, s[c + 8 + i].x);
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[56 + i].y, -INFINITY);
        const float bm = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        float m_new = fmaxf(m, bm);
        const bool fire = !((m_new - m) * sl2 <= args.tau);
        if (!fire) m_new = m;
        const float corr = fire ? (m == -INFINITY ? 0.f : ex2_mufu((m - m_new) * sl2)) : 1.0f;
        m = m_new;
        const float neg_ms = (m == -INFINITY) ? 0.f : -(m * sl2);
        const float2 neg_ms_2 = make_float2(neg_ms, neg_ms);
        if (fire) {
          const float2 corr_2 = make_float2(corr, corr);
#pragma unroll
          for (int a = 0; a < 8; ++a) acc[a] = __fmul2_rn(acc[a], corr_2);
        }
        if (need_mask)
          softmax_p_half<0, true, 0>(s, sl2_2, neg_ms_2, s_tm, acc);
        else
          softmax_p_half<0, false, 0>(s, sl2_2, neg_ms_2, s_tm, acc);
        if (j > 0 && __any_sync(0xffffffffu, fire)) {
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t ob[32];
            tmem_ld32(o_tm + c, ob);
            tmem_ld_wait();
            reg_fence32(ob);
            const float2 corr_2 = make_float2(corr, corr);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 o2 = __fmul2_rn(make_float2(__uint_as_float(ob[i]), __uint_as_float(ob[i + 1])), corr_2);
              ob[i] = __float_as_uint(o2.x);
              ob[i + 1] = __float_as_uint(o2.y);
            }
            tmem_st32(o_tm + c, ob);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        arrive_p(0);
        if (need_mask)
          softmax_p_half<0, true, 1>(s, sl2_2, neg_ms_2, s_tm, acc);
        else
          softmax_p_half<0, false, 1>(s, sl2_2, neg_ms_2, s_tm, acc);
        tmem_st_wait();
        tc_fence_before();
        arrive_p(1);
      }
      if (ok) {
        ok = wait_bar(bar_o(t), qi & 1, abort_flag, args.status, 18 + t);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a] = __fadd2_rn(acc[a], acc[a + 4]);
        acc[0] = __fadd2_rn(acc[0], acc[2]);
        acc[1] = __fadd2_rn(acc[1], acc[3]);
        const float2 l2 = __fadd2_rn(acc[0], acc[1]);
        const float l = l2.x + l2.y;
        const float inv_l = 1.0f / l;
        const bool valid = grow < args.n;
        const bool o_aligned32 = (reinterpret_cast<uintptr_t>(args.o) & 31u) == 0;
        const uint64_t pol_o = policy_evict_first();
        __nv_bfloat16* orow = args.o + (static_cast<size_t>(bh) * args.n + (valid ? grow : 0)) * D;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t ob[32];
          tmem_ld32(o_tm + c, ob);
          tmem_ld_wait();
          reg_fence32(ob);
          uint32_t pk[16];
          const float2 inv_l_2 = make_float2(inv_l, inv_l);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 o2 =
                __fmul2_rn(make_float2(__uint_as_float(ob[2 * i]), __uint_as_float(ob[2 * i + 1])), inv_l_2);
            pk[i] = pack_bf16x2(o2.x, o2.y);
          }
          if (valid) store_row64(orow + c, pk, o_aligned32, pol_o);
        }
        if (valid) args.lse[static_cast<size_t>(bh) * args.n + grow] = (m * sl2 + lg2_mufu(l)) * 0.69314718055994531f;
      }
      tc_fence_before();
      gb += nt;
    }
  }

  __syncthreads();
  // CTA 0's products read this CTA's shared memory and TMEM: neither CTA
  // frees its TMEM or leaves before the pair's last product has completed
  // (CTA 0's MMA warp drained before reaching here)
  cluster_sync_all();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

// A persistent grid of `clusters` CTA pairs (2 x clusters CTAs of 384 threads).
inline cudaError_t launch_fwd_bf16_2cta(const CUtensorMap& tm_q, const CUtensorMap& tm_kh, const CUtensorMap& tm_v,
                                        const FwdArgs& args, const WorkList& wl, int clusters, cudaStream_t stream) {
  using C = Fwd2Cfg;
  constexpr auto kernel = attn_fwd_bf16_2cta_kernel;
  const cudaError_t e = kernel_ready<kernel>(C::kSmemBytes, C::kLaunchRegs);
  if (e != cudaSuccess) return e;
  kernel<<<static_cast<unsigned>(2 * clusters), C::kThreads, C::kSmemBytes, stream>>>(tm_q, tm_kh, tm_v, args, wl);
  return cudaGetLastError();
}

// How many CTA pairs of the kernel can be resident at once on the current
// device (0 on failure).
inline int fwd_bf16_2cta_max_clusters() {
  using C = Fwd2Cfg;
  constexpr auto kernel = attn_fwd_bf16_2cta_kernel;
  if (kernel_ready<kernel>(C::kSmemBytes, C::kLaunchRegs) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return 0;
  return n;
}

}  // namespace attn
