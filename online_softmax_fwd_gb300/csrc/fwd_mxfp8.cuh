// Fused attention forward with MXFP8 block-scaled MMAs (d = 128), for sm_103a.
//
// Inputs are E4M3 Q, K, V with one E8M0 scale per 32 x 32 block (see
// quant_mxfp8.cu); P is converted to MXFP8 online, per 32 keys ("PyTorch
// FlashAttention-4 adds MXFP8 block-scaled forward and backward for Blackwell",
// section "Softmax conversion and unroll-KV": the block amax of P comes from
// one extra exp of the block's score max, the E8M0 scale from its exponent and
// mantissa bits). The online-softmax recurrence, lagging-max rescale and
// epilogue are those of the bf16 kernel (fwd_bf16.cuh).
//
// Structure: the bf16 kernel's two 128-row Q tiles in ping-pong, persistent
// CTAs over (tile pair, head) work items from the same list schedule, warps
// 0-7 softmax (thread = row), warp 8 TMA, warp 9 MMA. The 512 TMEM columns
// hold S0, S1, O0, O1 (128 each) as in the bf16 kernel, so the scale factors
// go where the same page's section "TMEM allocation and scale factor
// placement" puts them:
//   * the two first S GEMMs of a CTA read their Q and K scales from the O
//     regions, which no MMA has written yet; for later items S0(0) takes the
//     S1 columns 40-47 below, and S1(0) the O1 region again as soon as the
//     softmax of tile 1 has read the previous item's O1 into registers (its
//     epilogue loads all of O before converting and storing it);
//   * an O GEMM of tile t reads P's scales (written by the softmax) and V's
//     scales from free columns of S_t: P as E4M3 takes columns 0-31, so
//     32-35 (P) and 36-39 (V) are free once the softmax has read S_t;
//   * S_t(j+1) reads its Q and K scales from columns 40-47 of the OTHER tile's
//     S region, copied there only after that tile's softmax has loaded its
//     scores (one extra MMA <- softmax barrier per tile, "s_loaded").
// All scale regions are 4-column aligned.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "exp2_fma.cuh"
#include "fwd_bf16.cuh"
#include "mxfp8_common.cuh"
#include "kernel_setup.h"
#include "ptx.cuh"
#include "schedule.h"

namespace attn {

struct FwdMxArgs {
  const uint8_t* q_sf;   // [B*H][tiles][512] scale atoms (S GEMM layout)
  const uint8_t* k_sf;   // [B*H][tiles][512] (S GEMM layout)
  const uint8_t* v_sf;   // [B*H][tiles][512] (O GEMM layout)
  __nv_bfloat16* o;
  float* lse;
  unsigned int* status;
  int n;
  int n_tiles;           // ceil(N / 128)
  int n_pairs;           // ceil(N / 256)
  int bh;
  int band;
  int use_list;          // 1: items from the work list; 0: serpentine rounds
  float scale;
  float scale_log2;
  float tau;
  // rescale log (the LOG instantiations only, else null): as FwdArgs's
  uint8_t* rescale_log;
};

struct MxCfg {
  static constexpr uint32_t kTileBytes = 128u * 128u;  // 128 x 128 E4M3
  static constexpr uint32_t kAtomBytes = 512u;
  static constexpr int kSlots = 8;
  static constexpr uint32_t kRingOff = 2 * kTileBytes;                   // after Q0, Q1
  static constexpr uint32_t kQAtomOff = kRingOff + kSlots * kTileBytes;  // Q0, Q1 atoms
  static constexpr uint32_t kAtomOff = kQAtomOff + 2 * kAtomBytes;       // one atom per ring slot
  static constexpr uint32_t kBarOff = kAtomOff + kSlots * kAtomBytes;
  // q_full, full[kSlots], empty[kSlots], s_full[2], p_full[2], o_final[2], s_loaded[2], drain, q_empty,
  // o_read[2]
  static constexpr int kNumBars = 1 + 2 * kSlots + 12;
  static constexpr uint32_t kHolderOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kAbortOff = kHolderOff + 4;
  static constexpr uint32_t kSmemBytes = kAbortOff + 4 + 1024;
  static constexpr int kThreads = 384;
  static constexpr uint32_t kRegsSoftmax = 208;
  static constexpr uint32_t kRegsOther = 88;
  static constexpr int kLaunchRegs = 168;
  static constexpr uint32_t kTmemCols = 512;
  __host__ __device__ static constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return t ? 384u : 256u; }
  // inside S_t: P (E4M3) 0-31, P scales 32-35, V scales 36-39; scales of the
  // other tile's next S GEMM: Q 40-43, K 44-47
  static constexpr uint32_t kPScale = 32, kVScale = 36, kQScale = 40, kKScale = 44;
};

// PS, the scaling of P: 0 = one E8M0 scale per 32 keys from the block amax;
// 1 = the constant 2^-8 (E8M0 byte 119) with P in E4M3 (same page, same
// section: constant scaling of P stays robust because softmax keeps P in
// [0, 1]; with a stale maximum P reaches 2^tau, so 256 * 2^tau <= 448 needs
// tau <= log2(1.75)); 2 = the same constant with P in E5M2, whose 57344
// leaves room for tau <= log2(224) ("FlashAttention-4's Softmax Tricks",
// section "Where 'exact' breaks: P in FP8"). V stays E4M3.
// UKV selects the unroll-KV schedule ("PyTorch FlashAttention-4 adds MXFP8...",
// section "Softmax conversion and unroll-KV"): in an item's last key block the
// next item's first S GEMM is issued ahead of tile 1's last P V GEMM, and the
// softmax takes P's fp32 row sum after handing P over (P kept in registers; a
// needed O correction then loads O in 32-column parts). Measured slower on
// this kernel (its softmax warps run the epilogue, which hides the boundary
// wait anyway); kept as an opt-in schedule.
// LOG writes each row's rescale decision per key block (see FwdArgs).
template <bool CAUSAL, int EMU, int PS, bool UKV = false, bool LOG = false>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_mxfp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const FwdMxArgs args,
                          const __grid_constant__ WorkList wl) {
  using C = MxCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar_q = sbase + C::kBarOff;
  auto bar_full = [&](int i) { return bar_q + 8u * (1 + i); };
  auto bar_empty = [&](int i) { return bar_q + 8u * (1 + C::kSlots + i); };
  auto bar_s = [&](int t) { return bar_q + 8u * (1 + 2 * C::kSlots + t); };
  auto bar_p = [&](int t) { return bar_q + 8u * (3 + 2 * C::kSlots + t); };
  auto bar_o = [&](int t) { return bar_q + 8u * (5 + 2 * C::kSlots + t); };
  auto bar_ld = [&](int t) { return bar_q + 8u * (7 + 2 * C::kSlots + t); };
  const uint32_t bar_drain = bar_q + 8u * (9 + 2 * C::kSlots);
  const uint32_t bar_qe = bar_q + 8u * (10 + 2 * C::kSlots);  // Q buffers and atoms free again
  // the softmax of tile t has read O_t into registers (epilogue)
  auto bar_oread = [&](int t) { return bar_q + 8u * (11 + 2 * C::kSlots + t); };
  uint32_t* holder = reinterpret_cast<uint32_t*>(smem + C::kHolderOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kAbortOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // work items as in the bf16 kernel: the list, else serpentine rounds
  const int total_items = args.bh * args.n_pairs;
  auto item_of = [&](int k) {
    if (args.use_list) {
      const int idx = wl.first[blockIdx.x] + k;
      return idx < wl.first[blockIdx.x + 1] ? static_cast<int>(wl.item[idx]) : total_items;
    }
    const long long g = gridDim.x;
    const long long o = k * g + ((k & 1) ? g - 1 - blockIdx.x : blockIdx.x);
    return o < total_items ? static_cast<int>(o) : total_items;
  };
  auto coords = [&](int it, int& bh, int& pair) { item_coords(it, args.bh, args.n_pairs, args.band, bh, pair); };
  const int nkv = args.n_tiles;
  auto blocks_of = [&](int pair, int t) { return CAUSAL ? min(2 * pair + 1 + t, nkv) : nkv; };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s(t), 1);
      mbar_init(bar_p(t), 128);
      mbar_init(bar_o(t), 1);
      mbar_init(bar_ld(t), 128);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_qe, 1);
    mbar_init(bar_oread(0), 128);
    mbar_init(bar_oread(1), 128);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_addr(holder), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;

  if (warp >= 8) {
    // ============================================================ producer warpgroup
    regs_to<C::kRegsOther, C::kLaunchRegs>();
    if (warp == 8) {
      // ---------------------------------------------------------- TMA: Q0, Q1 (+ atoms), then K_j, V_j
      const uint32_t leader = elect_one();
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      int seq = 0;
      uint32_t slot = 0, ph = 0;
      bool ok = true;
      int qi = 0;
      for (int it = item_of(0); ok && it < total_items; it = item_of(++qi)) {
        int bh, pair;
        coords(it, bh, pair);
        const int row0 = pair * 256;
        const int n1 = blocks_of(pair, 1);
        const size_t head_atoms = static_cast<size_t>(bh) * nkv;
        // the Q buffers and atoms are free once the previous item's S GEMMs are complete
        if (qi > 0) {
          ok = __all_sync(0xffffffffu, wait_bar(bar_qe, (qi - 1) & 1, abort_flag, args.status, 13));
          if (!ok) break;
        }
        if (leader) {
          mbar_arrive_expect_tx(bar_q, 2 * (C::kTileBytes + C::kAtomBytes));
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            tma_load_3d_hint(sbase + t * C::kTileBytes, &tm_q, bar_q, 0, row0 + 128 * t, bh, pol_q);
            // a tile past N reads zeros through the map; its scales may be any valid atom
            const int qt = min(2 * pair + t, nkv - 1);
            bulk_load(sbase + C::kQAtomOff + t * C::kAtomBytes, args.q_sf + (head_atoms + qt) * C::kAtomBytes,
                      C::kAtomBytes, bar_q);
          }
        }
        for (int j = 0; ok && j < n1; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            ok = __all_sync(0xffffffffu, wait_bar(bar_empty(slot), ph ^ 1u, abort_flag, args.status, 1));
            if (!ok) break;
            if (leader) {
              mbar_arrive_expect_tx(bar_full(slot), C::kTileBytes + C::kAtomBytes);
              tma_load_3d_hint(sbase + C::kRingOff + slot * C::kTileBytes, kv ? &tm_v : &tm_k, bar_full(slot), 0,
                               j * 128, bh, pol_kv);
              bulk_load(sbase + C::kAtomOff + slot * C::kAtomBytes,
                        (kv ? args.v_sf : args.k_sf) + (head_atoms + j) * C::kAtomBytes, C::kAtomBytes,
                        bar_full(slot));
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
    } else if (warp == 9) {
      // ---------------------------------------------------------- MMA issuer (elected lane)
      const uint32_t leader = elect_one();
      auto commit = [&](uint32_t bar) {
        if (leader) tc_commit(bar);
      };
      auto wait = [&](uint32_t bar, uint32_t parity, uint32_t where) {
        return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, args.status, where));
      };
      constexpr uint32_t kSlotStep = C::kTileBytes >> 4;
      // descriptors as low words (start address, leading offset) plus one
      // shared high word (8-row groups 1024 bytes apart, 128-byte swizzle)
      const uint64_t q0 = smem_desc_sw128(sbase, 16, 1024);
      const uint32_t desc_hi = static_cast<uint32_t>(q0 >> 32);
      const uint32_t q_desc[2] = {static_cast<uint32_t>(q0),
                                  static_cast<uint32_t>(smem_desc_sw128(sbase + C::kTileBytes, 16, 1024))};
      const uint32_t ring_k = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kRingOff, 16, 1024));
      const uint32_t ring_v = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kRingOff, C::kTileBytes, 1024));
      auto slot_atom = [&](uint32_t slot) { return sbase + C::kAtomOff + slot * C::kAtomBytes; };
      // S_t = Q_t K^T from ring slot kslot; scales copied to TMEM columns sf_cols (Q) and sf_cols + 4 (K)
      auto issue_s = [&](int t, uint32_t kslot, uint32_t sf_cols) {
        if (leader) {
          sf_copy_to_tmem(tmem + sf_cols, sbase + C::kQAtomOff + t * C::kAtomBytes);
          sf_copy_to_tmem(tmem + sf_cols + 4, slot_atom(kslot));
#pragma unroll
          for (uint32_t kk = 0; kk < 4; ++kk)
            mma_mxf8_ss_lo(tmem + C::col_s(t), q_desc[t] + 2 * kk, ring_k + kslot * kSlotStep + 2 * kk, desc_hi,
                           idesc_mxf8(128, 128, false, kk, kk), kk > 0 ? 1u : 0u, tmem + sf_cols, tmem + sf_cols + 4);
        }
      };
      // O_t += P_t V from ring slot vslot; P_t and its scales in S_t, V's scales copied beside them
      auto issue_pv = [&](int t, uint32_t vslot, bool first) {
        if (leader) {
          const uint32_t s_cols = tmem + C::col_s(t);
          sf_copy_to_tmem(s_cols + C::kVScale, slot_atom(vslot));
#pragma unroll
          for (uint32_t kk = 0; kk < 4; ++kk)
            mma_mxf8_ts_lo(tmem + C::col_o(t), s_cols + 8 * kk, ring_v + vslot * kSlotStep + 256 * kk, desc_hi,
                           idesc_mxf8(128, 128, true, kk, kk, PS == 2), (!first || kk > 0) ? 1u : 0u, s_cols + C::kPScale,
                           s_cols + C::kVScale);
        }
      };
      auto advance2 = [](uint32_t& slot, uint32_t& phase) {
        slot += 2;
        if (slot >= static_cast<uint32_t>(C::kSlots)) {
          slot -= C::kSlots;
          phase ^= 1u;
        }
      };
      // ring positions and barrier phases continue across items
      uint32_t ks = 0, kph = 0;  // K_j
      uint32_t vs = 1, vph = 0;  // V_j
      uint32_t gb0 = 0, gb1 = 0;  // blocks of tile 0 / tile 1 before this item
      bool s0_early = false;       // (UKV) this item's S0(0) went out in the previous item's last block
      bool ok = true;
      int qi = 0;
      for (int it = item_of(0); ok && it < total_items; it = item_of(++qi)) {
        int bh, pair;
        coords(it, bh, pair);
        (void)bh;
        const int n0 = blocks_of(pair, 0);
        const int n1 = blocks_of(pair, 1);
        // (with UKV, re-waiting a phase that already completed returns at once:
        // the next phase of either barrier needs this item's S GEMMs first)
        ok = wait(bar_q, qi & 1, 2) && wait(bar_full(ks), kph, 3);
        if (!ok) break;
        tc_fence_after();
        if (qi == 0) {
          // first S GEMMs of the CTA: scales in the O regions, which no MMA has written yet
          issue_s(0, ks, C::col_o(0));
          commit(bar_s(0));
          issue_s(1, ks, C::col_o(1));
          commit(bar_s(1));
        } else {
          if (!s0_early) {
            // S1's columns 40-47 are free (its last scores were loaded before its last P)
            issue_s(0, ks, C::col_s(1) + C::kQScale);
            commit(bar_s(0));
          }
          // S1(0)'s scales go into O1 once the previous item's O1 has been read
          ok = wait(bar_oread(1), (qi - 1) & 1, 14);
          if (!ok) break;
          tc_fence_after();
          issue_s(1, ks, C::col_o(1));
          commit(bar_s(1));
        }
        s0_early = false;
        commit(bar_empty(ks));
        if (n1 == 1) commit(bar_qe);  // this item's S GEMMs are all issued
        for (int j = 0; ok && j < n1; ++j) {
          if (!wait(bar_full(vs), vph, 4)) {
            ok = false;
            break;
          }
          uint32_t ks_next = ks, kph_next = kph;
          advance2(ks_next, kph_next);
          bool k_next_ready = false;
          if (j < n0) {
            ok = wait(bar_p(0), (gb0 + j) & 1, 5);
            if (!ok) break;
            tc_fence_after();
            issue_pv(0, vs, j == 0);
            if (j + 1 < n0) {
              // S0(j+1)'s scales go into S1's columns 40-47: S1(j) must be loaded
              ok = wait(bar_full(ks_next), kph_next, 6) && wait(bar_ld(1), (gb1 + j) & 1, 9);
              if (!ok) break;
              k_next_ready = true;
              tc_fence_after();
              issue_s(0, ks_next, C::col_s(1) + C::kQScale);
              commit(bar_s(0));
            } else {
              commit(bar_o(0));
            }
          }
          if constexpr (UKV) {
            // the next item's S0(0) ahead of tile 1's last P V: its Q and K_0
            // are loaded once this item's S GEMMs are all issued (they are);
            // its scales go into S1's columns 40-47, free once tile 1 has
            // loaded its last scores
            if (j + 1 == n1 && item_of(qi + 1) < total_items) {
              ok = wait(bar_q, (qi + 1) & 1, 2) && wait(bar_full(ks_next), kph_next, 6) &&
                   wait(bar_ld(1), (gb1 + j) & 1, 9);
              if (!ok) break;
              tc_fence_after();
              issue_s(0, ks_next, C::col_s(1) + C::kQScale);
              commit(bar_s(0));
              s0_early = true;
            }
          }
          ok = wait(bar_p(1), (gb1 + j) & 1, 7);
          if (!ok) break;
          tc_fence_after();
          issue_pv(1, vs, j == 0);
          commit(bar_empty(vs));
          if (j + 1 < n1) {
            if (!k_next_ready) {
              ok = wait(bar_full(ks_next), kph_next, 8);
              if (!ok) break;
            }
            // S1(j+1)'s scales go into S0's columns 40-47: if tile 0 has block
            // j+1, its scores there must have been loaded first
            if (j + 1 < n0) {
              ok = wait(bar_ld(0), (gb0 + j + 1) & 1, 10);
              if (!ok) break;
            }
            tc_fence_after();
            issue_s(1, ks_next, C::col_s(0) + C::kQScale);
            commit(bar_s(1));
            commit(bar_empty(ks_next));
            if (j + 2 == n1) commit(bar_qe);  // that was this item's last S GEMM
          } else {
            commit(bar_o(1));
          }
          ks = ks_next;
          kph = kph_next;
          advance2(vs, vph);
        }
        gb0 += n0;
        gb1 += n1;
      }
      commit(bar_drain);
      drain_bar(bar_drain, 0);
      __syncwarp();
    }
  } else {
    // ============================================================ softmax warpgroups
    regs_to<C::kRegsSoftmax, C::kLaunchRegs>();
    const int t = warp >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + C::col_s(t);
    const uint32_t o_tm = tmem + lane_off + C::col_o(t);
    const float sl2 = args.scale_log2;
    const float2 sl2_2 = make_float2(sl2, sl2);
    bool ok = true;
    uint32_t gb = 0;  // this tile's blocks before the current item (barrier phases)
    int qi = 0;
    for (int it = item_of(0); ok && it < total_items; it = item_of(++qi)) {
    int bh, pair;
    coords(it, bh, pair);
    const int tile_row0 = pair * 256 + 128 * t;
    const int grow = tile_row0 + r;
    const int nt = blocks_of(pair, t);
    float m = -INFINITY;
    float l = 0.f;
    for (int j = 0; j < nt; ++j) {
      ok = __all_sync(0xffffffffu, wait_bar(bar_s(t), (gb + j) & 1, abort_flag, args.status, 16 + t));
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
      // the scores are in registers: the other tile's next S GEMM may now put
      // its scale factors into this region
      tc_fence_before();
      mbar_arrive(bar_ld(t));
      const int kv0 = j * 128;
      const bool need_mask = (kv0 + 128 > args.n) || (CAUSAL && kv0 + 127 > tile_row0);
      if (need_mask) {
        int lim = args.n - 1 - kv0;
        if (CAUSAL) lim = min(lim, grow - kv0);
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          if (2 * c > lim) s[c].x = -INFINITY;
          if (2 * c + 1 > lim) s[c].y = -INFINITY;
        }
      }
      // maxima of the four 32-key blocks (two interleaved chains each)
      float bmx[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float a = fmaxf(s[16 * g].x, s[16 * g].y);
        float c = fmaxf(s[16 * g + 1].x, s[16 * g + 1].y);
#pragma unroll
        for (int i = 2; i < 16; i += 2) {
          a = fmax3(a, s[16 * g + i].x, s[16 * g + i].y);
          c = fmax3(c, s[16 * g + i + 1].x, s[16 * g + i + 1].y);
        }
        bmx[g] = fmaxf(a, c);
      }
      const float bm = fmaxf(fmaxf(bmx[0], bmx[1]), fmaxf(bmx[2], bmx[3]));
      float m_new = fmaxf(m, bm);
      const bool fire = !((m_new - m) * sl2 <= args.tau);
      if (!fire) m_new = m;
      const float corr = fire ? (m == -INFINITY ? 0.f : ex2_mufu((m - m_new) * sl2)) : 1.0f;
      m = m_new;
      const float neg_ms = (m == -INFINITY) ? 0.f : -(m * sl2);
      float lsum = 0.f;
      // P per 32-key block: E8M0 scale from one exp of the block max; P / 2^e
      // = 2^(x - e), so the scale rides in the exp's shift; the fp32 row sum
      // takes each block's P / 2^e times 2^e
      uint32_t pk[32];
      uint32_t sfw = 0;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint32_t sfb = PS != 0 ? 119u : e8m0_for_amax(ex2_mufu(__fmaf_rn(bmx[g], sl2, neg_ms)));
        sfw |= sfb << (8 * g);
        const float shift = neg_ms - static_cast<float>(static_cast<int>(sfb) - 127);
        const float2 shift_2 = make_float2(shift, shift);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const int c = 16 * g + i;
          const float2 x0 = __ffma2_rn(s[c], sl2_2, shift_2);
          const float2 x1 = __ffma2_rn(s[c + 1], sl2_2, shift_2);
          float2 p0, p1;
          if (need_mask) {
            p0 = make_float2(ex2_mufu(x0.x), ex2_mufu(x0.y));
            p1 = make_float2(ex2_mufu(x1.x), ex2_mufu(x1.y));
          } else {
            p0 = make_float2(exp2_col<EMU, false>(2 * c, x0.x), exp2_col<EMU, false>(2 * c + 1, x0.y));
            p1 = make_float2(exp2_col<EMU, false>(2 * c + 2, x1.x), exp2_col<EMU, false>(2 * c + 3, x1.y));
          }
          if constexpr (UKV) {
            s[c] = p0;  // kept for the row sum after the hand-over
            s[c + 1] = p1;
          } else {
            acc[(i >> 1) & 1] = __fadd2_rn(acc[(i >> 1) & 1], p0);
            acc[2 + ((i >> 1) & 1)] = __fadd2_rn(acc[2 + ((i >> 1) & 1)], p1);
          }
          pk[8 * g + i / 2] = PS == 2 ? pack_e5m2x4(p0.x, p0.y, p1.x, p1.y) : pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
        }
        if constexpr (!UKV) {
          acc[0] = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
          lsum = __fmaf_rn(acc[0].x + acc[0].y, __uint_as_float(sfb << 23), lsum);
        }
      }
      tmem_st32(s_tm, pk);                      // P, 4 keys per column
      tmem_st1(s_tm + C::kPScale + quad, sfw);  // row r's scales at column r / 32
      // correction of O once the scores are dead; lands before P is handed
      // over
      const bool warp_rescales = j > 0 && __any_sync(0xffffffffu, fire);
      if constexpr (LOG) {
        if (grow < args.n)
          args.rescale_log[(static_cast<size_t>(bh) * args.n + grow) * nkv + j] =
              static_cast<uint8_t>((fire ? 1u : 0u) | (warp_rescales ? 2u : 0u));
      }
      if (warp_rescales) {
        const float2 corr_2 = make_float2(corr, corr);
        if constexpr (UKV) {
          // 32 columns at a time (P stays in registers for the sum)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t ob[32];
            tmem_ld32(o_tm + 32 * c, ob);
            tmem_ld_wait();
            reg_fence32(ob);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 o2 = __fmul2_rn(make_float2(__uint_as_float(ob[i]), __uint_as_float(ob[i + 1])), corr_2);
              ob[i] = __float_as_uint(o2.x);
              ob[i + 1] = __float_as_uint(o2.y);
            }
            tmem_st32(o_tm + 32 * c, ob);
          }
        } else {
          // all of O at once (one load latency, overlapping the store of P)
          uint32_t ob[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(o_tm + 32 * c, ob[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            reg_fence32(ob[c]);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 o2 =
                  __fmul2_rn(make_float2(__uint_as_float(ob[c][i]), __uint_as_float(ob[c][i + 1])), corr_2);
              ob[c][i] = __float_as_uint(o2.x);
              ob[c][i + 1] = __float_as_uint(o2.y);
            }
            tmem_st32(o_tm + 32 * c, ob[c]);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p(t));
      if constexpr (UKV) {
        // the O GEMM and the next S GEMM run meanwhile
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          float2 acc[4] = {s[16 * g], s[16 * g + 1], s[16 * g + 2], s[16 * g + 3]};
#pragma unroll
          for (int i = 4; i < 16; ++i) acc[i & 3] = __fadd2_rn(acc[i & 3], s[16 * g + i]);
          acc[0] = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
          lsum = __fmaf_rn(acc[0].x + acc[0].y, __uint_as_float(((sfw >> (8 * g)) & 0xffu) << 23), lsum);
        }
      }
      l = l * corr + lsum;
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar_o(t), qi & 1, abort_flag, args.status, 18 + t));
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const bool valid = grow < args.n;
      // rows are 128 or 256 bytes: 32-byte alignment of O decides the store width for all of them
      const bool o_aligned32 = (reinterpret_cast<uintptr_t>(args.o) & 31u) == 0;
      const uint64_t pol_o = policy_evict_first();
      __nv_bfloat16* orow = args.o + (static_cast<size_t>(bh) * args.n + (valid ? grow : 0)) * 128;
      const float2 inv_l_2 = make_float2(inv_l, inv_l);
      // all of O_t into registers first: the next item's S1 GEMM may then put
      // its scale factors into O1
      uint32_t ob[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(o_tm + 32 * c, ob[c]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar_oread(t));
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        reg_fence32(ob[c]);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 o2 =
              __fmul2_rn(make_float2(__uint_as_float(ob[c][2 * i]), __uint_as_float(ob[c][2 * i + 1])), inv_l_2);
          w[i] = pack_bf16x2(o2.x, o2.y);
        }
        if (valid) store_row64(orow + 32 * c, w, o_aligned32, pol_o);
      }
      if (valid) args.lse[static_cast<size_t>(bh) * args.n + grow] = (m * sl2 + lg2_mufu(l)) * 0.69314718055994531f;
    }
    // the next item's O GEMMs overwrite O_t only after this warpgroup's next
    // P is ready, i.e. after these reads
    tc_fence_before();
    gb += nt;
    }
  }

  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <bool CAUSAL, int EMU, int PS, bool UKV = false, bool LOG = false>
cudaError_t launch_fwd_mxfp8(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const FwdMxArgs& args, const WorkList& wl, int ctas, cudaStream_t stream) {
  constexpr auto kernel = attn_fwd_mxfp8_kernel<CAUSAL, EMU, PS, UKV, LOG>;
  // shared-memory opt-in and the setmaxnreg register check, once per device
  const cudaError_t e = kernel_ready<kernel>(MxCfg::kSmemBytes, MxCfg::kLaunchRegs);
  if (e != cudaSuccess) return e;
  kernel<<<static_cast<unsigned>(ctas), MxCfg::kThreads, MxCfg::kSmemBytes, stream>>>(tm_q, tm_k, tm_v, args, wl);
  return cudaGetLastError();
}

}  // namespace attn
