// Fused attention forward, bf16 in / bf16 O + fp32 LSE out, for sm_103a.
//
// One CTA owns two 128-row query tiles of one (batch, head) -- the two Q tiles
// in ping-pong of the FA4 forward pipeline ("Software-Emulated Exponential",
// KernelWiki; "PyTorch FlashAttention-4 adds MXFP8", section "TMEM allocation")
// -- and streams the head's keys and values in 128-row blocks:
//
//   warp 8      TMA producer: Q0, Q1 once; then K_j, V_j into a ring of
//               128 x d bf16 shared-memory slots (128-byte swizzle).
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T (tcgen05, both operands
//               in shared memory, fp32 accumulator in TMEM) and O_t += P_t V_j
//               (A operand P_t read from TMEM, V_j from shared memory).
//   warps 0-3   softmax for tile 0, warps 4-7 for tile 1; thread = query row.
//
// Per key block j, a softmax thread (row i) follows the online recurrence of
// "Flash Attention 4 - the algorithm and the two-MMA problem" ("Online softmax
// - three running states", "Deferred normalization", "The exp2 trick"):
//   load its 128 scores from TMEM; mask keys j > i on the causal diagonal block
//   and keys >= N in a ragged last block ("Lecture 2 - Online Softmax and
//   Numerical Correctness", "Causal masking just changes which blocks
//   contribute"); take the block max of the raw scores; move the running max
//   only if it would grow by more than tau in log2 units, else keep the stale
//   max ("FlashAttention-4's Softmax Tricks", "Conditional rescaling": the
//   SoftmaxSm100.update_row_max rule); if any row of the warp moved, rescale
//   that warp's O rows in TMEM by 2^((m_old - m_new) s log2 e) (correction done
//   in place: the MMA thread issues S_t(j) after O_t += P_t V_{j-1}, and tcgen05
//   operations from one thread complete in order, so when S_t(j) is complete O_t
//   is quiescent until this warp hands P_t(j) over); p = 2^(s log2e * S -
//   s log2e * m) with one FFMA and then the MUFU ex2 or, for a compile-time
//   share of the columns, the software exp2 on the FMA pipe; l += sum p in fp32;
//   P rounded to bf16 and stored over the S columns it replaces, handed over in
//   two halves of 64 keys so the O MMA of the first half overlaps the softmax
//   of the second.
// After the last block: O / l rounded to bf16, and LSE = s m + ln l.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "exp2_fma.cuh"
#include "kernel_setup.h"
#include "ptx.cuh"
#include "schedule.h"

namespace attn {

constexpr uint32_t kStatusTimeout = 5;  // == ATTN_ERR_TIMEOUT

struct FwdArgs {
  __nv_bfloat16* o;
  float* lse;
  unsigned int* status;  // device error word
  int n;                 // sequence length N
  int n_kv_blocks;       // ceil(N / 128)
  int n_pairs;           // ceil(N / 256): Q-tile pairs per head
  int bh;                // B * H
  int band;              // heads per scheduling band (their K/V stay in L2 together)
  int use_list;          // 1: items from the work list; 0: serpentine rounds
  float scale;           // s
  float scale_log2;      // s * log2(e)
  float tau;             // rescale threshold, log2 units
  // Rescale log (only read by the logging instantiations, else null): one
  // byte per (head, row, key block), bit 0 = the row's running max moved at
  // this block, bit 1 = the row's warp rescaled O (any of its 32 rows moved,
  // block > 0).
  uint8_t* rescale_log;
};

template <int D>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kBoxes = D / 64;                     // 64-column (128-byte) swizzle boxes per row
  static constexpr uint32_t kBoxBytes = 128u * 128u;        // 128 rows x 128 bytes
  static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;  // one 128 x d bf16 tile
  static constexpr int kSlots = D == 128 ? 5 : 8;           // K/V ring depth
  static constexpr uint32_t kRingOff = 2 * kTileBytes;      // after Q0, Q1
  static constexpr uint32_t kBarOff = kRingOff + kSlots * kTileBytes;
  // q_full, full[kSlots], empty[kSlots], s_full[2], p_full[2][2 halves], o_final[2], drain, q_empty
  static constexpr int kNumBars = 1 + 2 * kSlots + 10;
  static constexpr uint32_t kHolderOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kAbortOff = kHolderOff + 4;
  static constexpr uint32_t kSmemBytes = kAbortOff + 4 + 1024;  // + slack for 1024-byte alignment
  static constexpr int kThreads = 384;  // 8 softmax warps, TMA warp, MMA warp, 2 spare
  // setmaxnreg split: softmax warpgroups grow, the producer warpgroup shrinks.
  // 2*128*208 + 128*88 = 64512 = 384 threads x 168 registers at launch.
  static constexpr uint32_t kRegsSoftmax = 208;
  static constexpr uint32_t kRegsOther = 88;
  static constexpr int kLaunchRegs = 168;
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: S_t (fp32, 128 columns; P_t as bf16 pairs over its first 64)
  // and O_t (fp32, d columns) for the two query tiles.
  __host__ __device__ static constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 256u + (t ? D : 0); }
};

// ~2 s at the 2 GHz class SM clock.
constexpr long long kWaitLimitCycles = 4000000000LL;
constexpr long long kDrainLimitCycles = 200000000LL;

__device__ __forceinline__ void record_status(unsigned int* status, uint32_t code, uint32_t where) {
  atomicCAS(status, 0u, code | (where << 8));
}

// Wait for phase `parity` of an mbarrier, giving up when another role raised
// the CTA's abort flag or after limit_cycles (then raising it and recording
// ATTN_ERR_TIMEOUT with `where` in the status word).
__device__ __forceinline__ bool wait_bar_limit(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                               unsigned int* status, uint32_t where, long long limit_cycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit_cycles) {
      *abort_flag = 1u;
      record_status(status, kStatusTimeout, where);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         unsigned int* status, uint32_t where) {
  return wait_bar_limit(bar, parity, abort_flag, status, where, kWaitLimitCycles);
}

// Bounded wait used only while draining after an abort.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kDrainLimitCycles) return;
  }
}

template <int EMU, bool MUFU_ONLY>
__device__ __forceinline__ float exp2_col(int c, float x) {
  if constexpr (!MUFU_ONLY && EMU > 0) {
    if ((c & 15) < EMU) return exp2_fma(x);
  }
  return ex2_mufu(x);
}

// p = 2^(S*sl2 + neg_ms) for one half (64 keys, pairs [32 H, 32 H + 32)) of a
// row's 128 scores, rounded to bf16 pairs and stored to TMEM at p_tm (32 bf16
// pairs from column 32 H); the unrounded p are added to the row's partial sums
// acc. The scale-and-shift and the sums use the packed fp32 pair instructions
// (one issue for two lanes of work); eight independent partial sums keep the
// long-latency packed add off the critical path.
template <int EMU, bool MUFU_ONLY, int H>
__device__ __forceinline__ void softmax_p_half(const float2 (&s)[64], float2 sl2_2, float2 neg_ms_2, uint32_t p_tm,
                                               float2 (&acc)[8]) {
#pragma unroll
  for (int chunk = 2 * H; chunk < 2 * H + 2; ++chunk) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = chunk * 16 + i;  // pair index
      const float2 x = __ffma2_rn(s[c], sl2_2, neg_ms_2);
      const float2 p = make_float2(exp2_col<EMU, MUFU_ONLY>(2 * c, x.x), exp2_col<EMU, MUFU_ONLY>(2 * c + 1, x.y));
      acc[i & 7] = __fadd2_rn(acc[i & 7], p);
      pk[i] = pack_bf16x2(p.x, p.y);
    }
    tmem_st16(p_tm + chunk * 16, pk);
  }
}

template <int D, bool CAUSAL, int EMU, bool LOG = false>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const FwdArgs args,
                         const __grid_constant__ WorkList wl) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzle atoms need 1024-byte aligned tiles (shared-window address)
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar_q = sbase + C::kBarOff;
  auto bar_full = [&](int i) { return bar_q + 8u * (1 + i); };
  auto bar_empty = [&](int i) { return bar_q + 8u * (1 + C::kSlots + i); };
  auto bar_s = [&](int t) { return bar_q + 8u * (1 + 2 * C::kSlots + t); };
  // P of a tile is handed over in two halves of 64 keys, so the O MMA of the
  // first half overlaps the softmax of the second
  auto bar_p = [&](int t, int h) { return bar_q + 8u * (3 + 2 * C::kSlots + 2 * t + h); };
  auto bar_o = [&](int t) { return bar_q + 8u * (7 + 2 * C::kSlots + t); };
  const uint32_t bar_drain = bar_q + 8u * (9 + 2 * C::kSlots);
  const uint32_t bar_qe = bar_q + 8u * (10 + 2 * C::kSlots);  // Q buffers free again
  uint32_t* holder = reinterpret_cast<uint32_t*>(smem + C::kHolderOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kAbortOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Persistent: CTA c runs the items of its work list in order; without a
  // list, in round k it takes item k G + c (k even) or k G + G - 1 - c (k odd),
  // G = gridDim.x, a serpentine that evens out the causal items' unequal work.
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
  const int nkv = args.n_kv_blocks;
  // key blocks of tile 0 and tile 1 (n1 >= n0) of a pair
  auto blocks_of = [&](int pair, int t) { return CAUSAL ? min(2 * pair + 1 + t, nkv) : nkv; };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s(t), 1);
      mbar_init(bar_p(t, 0), 128);
      mbar_init(bar_p(t, 1), 128);
      mbar_init(bar_o(t), 1);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_qe, 1);
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
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop (warp-uniform values); one elected lane
    // issues the copies.
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
      // the Q buffers are free once the previous item's S MMAs are complete
      if (qi > 0) {
        ok = __all_sync(0xffffffffu, wait_bar(bar_qe, (qi - 1) & 1, abort_flag, args.status, 13));
        if (!ok) break;
      }
      if (leader) {
        mbar_arrive_expect_tx(bar_q, 2 * C::kTileBytes);
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d_hint(sbase + t * C::kTileBytes + b * C::kBoxBytes, &tm_q, bar_q, b * 64, row0 + 128 * t, bh,
                             pol_q);
      }
      for (int j = 0; ok && j < n1; ++j) {
        for (int kv = 0; kv < 2; ++kv) {
          ok = __all_sync(0xffffffffu, wait_bar(bar_empty(slot), ph ^ 1u, abort_flag, args.status, 1));
          if (!ok) break;
          if (leader) {
            mbar_arrive_expect_tx(bar_full(slot), C::kTileBytes);
            const CUtensorMap* map = kv ? &tm_v : &tm_k;
#pragma unroll
            for (int b = 0; b < C::kBoxes; ++b)
              tma_load_3d_hint(sbase + C::kRingOff + slot * C::kTileBytes + b * C::kBoxBytes, map, bar_full(slot),
                               b * 64, j * 128, bh, pol_kv);
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
      // let the copies already in flight land before the CTA's memory is released
      drain_bar(bar_q, (qi & 1) ^ 1);
      for (int s = seq - C::kSlots < 0 ? 0 : seq - C::kSlots; s < seq; ++s)
        drain_bar(bar_full(s % C::kSlots), (s / C::kSlots) & 1);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop so descriptors and ring positions stay
    // warp-uniform; one elected lane issues the MMAs and commits (a commit
    // tracks the MMAs of the thread that issues it, always the same lane).
    {
      const uint32_t leader = elect_one();
      auto commit = [&](uint32_t bar) {
        if (leader) tc_commit(bar);
      };
      auto wait = [&](uint32_t bar, uint32_t parity, uint32_t where) {
        return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, args.status, where));
      };
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false);
      constexpr uint32_t kIdO = idesc_bf16_f32(128, D, true);
      constexpr uint32_t kSlotStep = C::kTileBytes >> 4;  // descriptor units between ring slots
      // Descriptors are built once and advanced with constant adds to their
      // low word (start address >> 4; every operand lies below 256 KiB, so no
      // carry leaves the field). The high word (8-row groups 1024 bytes apart,
      // 128-byte swizzle) is the same for Q, K and V.
      // Q and K are K-major: the next K=16 slice is 32 bytes further inside a
      // 128-byte swizzle row, the 5th starts the next 64-column box.
      const uint64_t q0 = smem_desc_sw128(sbase, 16, 1024);
      const uint32_t desc_hi = static_cast<uint32_t>(q0 >> 32);
      const uint32_t q_lo[2] = {static_cast<uint32_t>(q0),
                                static_cast<uint32_t>(smem_desc_sw128(sbase + C::kTileBytes, 16, 1024))};
      const uint32_t k_ring = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kRingOff, 16, 1024));
      // V is MN-major: 64-column halves kBoxBytes apart (the leading offset),
      // 8-key groups 1024 bytes apart; the next 16 keys are 2048 bytes further.
      const uint32_t v_ring = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kRingOff, C::kBoxBytes, 1024));
      auto kmajor_step = [](int kk) -> uint32_t { return ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4; };
      auto issue_s = [&](int t, uint32_t slot) {
        const uint32_t a = q_lo[t];
        const uint32_t b = k_ring + slot * kSlotStep;
        const uint32_t d = tmem + C::col_s(t);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_lo(d, a + kmajor_step(kk), b + kmajor_step(kk), desc_hi, kIdS, kk > 0 ? 1u : 0u);
        }
      };
      // O_t += P_t V for keys [64 h, 64 h + 64) of the block
      auto issue_pv = [&](int t, uint32_t slot, int h, bool first) {
        const uint32_t b = v_ring + slot * kSlotStep;
        const uint32_t d = tmem + C::col_o(t);
        const uint32_t a = tmem + C::col_s(t);
        if (leader) {
#pragma unroll
          for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
            mma_ts_lo(d, a + kk * 8, b + kk * 128, desc_hi, kIdO, (!first || kk > 0) ? 1u : 0u);
        }
      };
      // ring positions: K_j is the (2j)-th load, V_j the (2j+1)-th
      auto advance2 = [](uint32_t& slot, uint32_t& phase) {
        slot += 2;
        if (slot >= static_cast<uint32_t>(C::kSlots)) {
          slot -= C::kSlots;
          phase ^= 1u;
        }
      };
      // ring positions continue across items: K_j of an item follows the
      // previous item's last V
      uint32_t ks = 0, kph = 0;  // K_j
      uint32_t vs = 1, vph = 0;  // V_j
      uint32_t gb0 = 0, gb1 = 0;  // blocks of tile 0 / tile 1 before this item (barrier phases)
      bool ok = true;
      int qi = 0;
      for (int it = item_of(0); ok && it < total_items; it = item_of(++qi)) {
        int bh, pair;
        coords(it, bh, pair);
        (void)bh;
        const int n0 = blocks_of(pair, 0);
        const int n1 = blocks_of(pair, 1);
        ok = wait(bar_q, qi & 1, 2) && wait(bar_full(ks), kph, 3);
        if (!ok) break;
        tc_fence_after();
        issue_s(0, ks);
        commit(bar_s(0));
        issue_s(1, ks);
        commit(bar_s(1));
        commit(bar_empty(ks));
        if (n1 == 1) commit(bar_qe);  // this item's S MMAs are all issued
        for (int j = 0; ok && j < n1; ++j) {
          if (!wait(bar_full(vs), vph, 4)) {
            ok = false;
            break;
          }
          uint32_t ks_next = ks, kph_next = kph;
          advance2(ks_next, kph_next);
          bool k_next_ready = false;
          if (j < n0) {
            const uint32_t par = (gb0 + j) & 1;
            ok = wait(bar_p(0, 0), par, 5);
            if (!ok) break;
            tc_fence_after();
            issue_pv(0, vs, 0, j == 0);
            ok = wait(bar_p(0, 1), par, 11);
            if (!ok) break;
            tc_fence_after();
            issue_pv(0, vs, 1, false);
            if (j + 1 < n0) {
              ok = wait(bar_full(ks_next), kph_next, 6);
              if (!ok) break;
              k_next_ready = true;
              tc_fence_after();
              issue_s(0, ks_next);
              commit(bar_s(0));
            } else {
              commit(bar_o(0));
            }
          }
          const uint32_t par1 = (gb1 + j) & 1;
          ok = wait(bar_p(1, 0), par1, 7);
          if (!ok) break;
          tc_fence_after();
          issue_pv(1, vs, 0, j == 0);
          ok = wait(bar_p(1, 1), par1, 12);
          if (!ok) break;
          tc_fence_after();
          issue_pv(1, vs, 1, false);
          commit(bar_empty(vs));
          if (j + 1 < n1) {
            if (!k_next_ready) {
              ok = wait(bar_full(ks_next), kph_next, 8);
              if (!ok) break;
              tc_fence_after();
            }
            issue_s(1, ks_next);
            commit(bar_s(1));
            commit(bar_empty(ks_next));
            if (j + 2 == n1) commit(bar_qe);  // that was this item's last S MMA
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
      // nothing may still be executing when TMEM is released
      commit(bar_drain);
      drain_bar(bar_drain, 0);
    }
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
    // the row sum l as 16 partial sums, reduced once after the last block
    float2 acc[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) acc[a] = make_float2(0.f, 0.f);
    for (int j = 0; j < nt; ++j) {
      const uint32_t par = (gb + j) & 1;
      ok = wait_bar(bar_s(t), par, abort_flag, args.status, 16 + t);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float2 s[64];  // the row's 128 scores as (even, odd) column pairs
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
      // keep the stale max unless it would grow by more than tau (log2 units)
      float m_new = fmaxf(m, bm);
      const bool fire = !((m_new - m) * sl2 <= args.tau);
      if (!fire) m_new = m;
      // 0 while nothing has been accumulated (first block), 1 when the max stays
      const float corr = fire ? (m == -INFINITY ? 0.f : ex2_mufu((m - m_new) * sl2)) : 1.0f;
      m = m_new;
      const float neg_ms = (m == -INFINITY) ? 0.f : -(m * sl2);
      const float2 neg_ms_2 = make_float2(neg_ms, neg_ms);
      if (fire) {
        const float2 corr_2 = make_float2(corr, corr);
#pragma unroll
        for (int a = 0; a < 8; ++a) acc[a] = __fmul2_rn(acc[a], corr_2);
      }
      // first 64 keys of P
      if (need_mask)
        softmax_p_half<EMU, true, 0>(s, sl2_2, neg_ms_2, s_tm, acc);
      else
        softmax_p_half<EMU, false, 0>(s, sl2_2, neg_ms_2, s_tm, acc);
      // correction of O (before any O MMA of this block), for the whole warp
      // if any of its rows moved its max
      const bool warp_rescales = j > 0 && __any_sync(0xffffffffu, fire);
      if constexpr (LOG) {
        if (grow < args.n)
          args.rescale_log[(static_cast<size_t>(bh) * args.n + grow) * nkv + j] =
              static_cast<uint8_t>((fire ? 1u : 0u) | (warp_rescales ? 2u : 0u));
      }
      if (warp_rescales) {
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
      mbar_arrive(bar_p(t, 0));
      // last 64 keys, while the MMA works on the first
      if (need_mask)
        softmax_p_half<EMU, true, 1>(s, sl2_2, neg_ms_2, s_tm, acc);
      else
        softmax_p_half<EMU, false, 1>(s, sl2_2, neg_ms_2, s_tm, acc);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p(t, 1));
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
      // rows are 128 or 256 bytes: 32-byte alignment of O decides the store width for all of them
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
          const float2 o2 = __fmul2_rn(make_float2(__uint_as_float(ob[2 * i]), __uint_as_float(ob[2 * i + 1])), inv_l_2);
          pk[i] = pack_bf16x2(o2.x, o2.y);
        }
        if (valid) store_row64(orow + c, pk, o_aligned32, pol_o);
      }
      if (valid) args.lse[static_cast<size_t>(bh) * args.n + grow] = (m * sl2 + lg2_mufu(l)) * 0.69314718055994531f;
    }
    // the next item's O MMAs overwrite O_t only after this warpgroup's next
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

// Launch one instantiation: a persistent grid of `ctas` CTAs of 384 threads,
// one per SM (at most one per item; the work list, when used, is built for
// that many).
template <int D, bool CAUSAL, int EMU, bool LOG = false>
cudaError_t launch_fwd_bf16(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                            const FwdArgs& args, const WorkList& wl, int ctas, cudaStream_t stream) {
  using C = FwdCfg<D>;
  constexpr auto kernel = attn_fwd_bf16_kernel<D, CAUSAL, EMU, LOG>;
  // shared-memory opt-in and the setmaxnreg register check, once per device
  const cudaError_t e = kernel_ready<kernel>(C::kSmemBytes, C::kLaunchRegs);
  if (e != cudaSuccess) return e;
  kernel<<<static_cast<unsigned>(ctas), C::kThreads, C::kSmemBytes, stream>>>(tm_q, tm_k, tm_v, args, wl);
  return cudaGetLastError();
}

}  // namespace attn
