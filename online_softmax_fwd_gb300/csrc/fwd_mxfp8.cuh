// Fused attention forward with MXFP8 block-scaled MMAs (d = 128), for sm_103a.
//
// Inputs are E4M3 Q, K, V with one E8M0 scale per 32 x 32 block (see
// quant_mxfp8.cu); P is converted to MXFP8 online, per 32 keys ("PyTorch
// FlashAttention-4 adds MXFP8 block-scaled forward and backward for Blackwell",
// section "Softmax conversion and unroll-KV": the block amax of P comes from
// one extra exp of the block's score max, the scale from its exponent and
// mantissa bits). The online-softmax recurrence, tau rescale and epilogue are
// those of the bf16 kernel.
//
// One CTA owns one 128-row Q tile of one (batch, head). The lower-precision
// MMAs are twice as fast, so softmax is the bound; S is double-buffered in
// TMEM so S(j+1) is computed while the softmax works on S(j):
//   TMEM cols   0-127  S buffer 0 (P(j) as E4M3 over its first 32 columns)
//             128-255  S buffer 1
//             256-383  O (fp32)
//             384..411 scale factors, 4 columns each: Q (A of S), K[2] (B of S),
//                      P[2] (A of O), V[2] (B of O)
//   warps 0-7  softmax: warp w owns TMEM lane quadrant w % 4 and the key
//              columns [64 (w / 4), 64 (w / 4) + 64) of each block; the two
//              halves of a row swap their 32-key block maxima through shared
//              memory (published with per-thread sequence numbers)
//   warp 8     TMA: Q tile + its scale atom; then K_0, K_1, V_0, K_2, V_1, ...
//   warp 9     MMA (elected lane): S(j) into buffer j % 2; O += P(j) V_j.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "exp2_fma.cuh"
#include "fwd_bf16.cuh"
#include "mxfp8_common.cuh"
#include "ptx.cuh"

namespace attn {

struct FwdMxArgs {
  const uint8_t* q_sf;   // [B*H][tiles][512] scale atoms (S GEMM layout)
  const uint8_t* k_sf;   // [B*H][tiles][512] (S GEMM layout)
  const uint8_t* v_sf;   // [B*H][tiles][512] (O GEMM layout)
  __nv_bfloat16* o;
  float* lse;
  unsigned int* status;
  int n;
  int n_tiles;           // ceil(N / 128): Q tiles and key blocks per head
  int bh;
  int band;
  float scale;
  float scale_log2;
  float tau;
};

struct MxCfg {
  static constexpr uint32_t kTileBytes = 128u * 128u;   // 128 x 128 E4M3
  static constexpr uint32_t kAtomBytes = 512u;
  static constexpr int kSlots = 8;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kRingOff = kTileBytes;                       // 1024-aligned payloads
  static constexpr uint32_t kQAtomOff = kRingOff + kSlots * kTileBytes;
  static constexpr uint32_t kAtomOff = kQAtomOff + kAtomBytes;           // one atom per ring slot
  static constexpr uint32_t kXchOff = kAtomOff + kSlots * kAtomBytes;    // [2 parity][4 quad][2 half][32][2] floats
  static constexpr uint32_t kXchBytes = 2 * 4 * 2 * 32 * 2 * 4;
  static constexpr uint32_t kLOff = kXchOff + kXchBytes;                 // [2 half][128] floats
  static constexpr uint32_t kSeqOff = kLOff + 2 * 128 * 4;              // [2 half][128] ints
  static constexpr uint32_t kBarOff = kSeqOff + 2 * 128 * 4;
  // q_full, full[kSlots], empty[kSlots], s_full[2], p_full[2], o_done, drain
  static constexpr int kNumBars = 1 + 2 * kSlots + 6;
  static constexpr uint32_t kHolderOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kAbortOff = kHolderOff + 4;
  static constexpr uint32_t kSmemBytes = kAbortOff + 4 + 1024;
  static constexpr int kThreads = 384;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
  static constexpr uint32_t kColSfQ = 384;
  __host__ __device__ static constexpr uint32_t col_s(int b) { return b ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t col_sf_k(int b) { return 388u + 4u * b; }
  __host__ __device__ static constexpr uint32_t col_sf_p(int b) { return 396u + 4u * b; }
  __host__ __device__ static constexpr uint32_t col_sf_v(int b) { return 404u + 4u * b; }
};

// Bounded wait until *seq >= want (a partner thread's publication), giving up
// on the CTA's abort flag or after kWaitLimitCycles.
__device__ __forceinline__ bool wait_seq(const volatile int* seq, int want, volatile uint32_t* abort_flag,
                                         unsigned int* status, uint32_t where) {
  if (*seq >= want) return true;
  const long long t0 = clock64();
  while (*seq < want) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      *abort_flag = 1u;
      record_status(status, kStatusTimeout, where);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

template <bool CAUSAL, int EMU>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_mxfp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const FwdMxArgs args) {
  using C = MxCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar_q = sbase + C::kBarOff;
  auto bar_full = [&](int i) { return bar_q + 8u * (1 + i); };
  auto bar_empty = [&](int i) { return bar_q + 8u * (1 + C::kSlots + i); };
  auto bar_s = [&](int b) { return bar_q + 8u * (1 + 2 * C::kSlots + b); };
  auto bar_p = [&](int b) { return bar_q + 8u * (3 + 2 * C::kSlots + b); };
  const uint32_t bar_o = bar_q + 8u * (5 + 2 * C::kSlots);
  const uint32_t bar_drain = bar_q + 8u * (6 + 2 * C::kSlots);
  uint32_t* holder = reinterpret_cast<uint32_t*>(smem + C::kHolderOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kAbortOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int bh, tile;
  {
    const int per_band = args.band * args.n_tiles;
    const int band_id = blockIdx.x / per_band;
    const int r = blockIdx.x - band_id * per_band;
    const int heads = min(args.band, args.bh - band_id * args.band);
    tile = args.n_tiles - 1 - r / heads;  // heaviest causal tiles first
    bh = band_id * args.band + r % heads;
  }
  const int row0 = tile * 128;
  const int nblk = CAUSAL ? min(tile + 1, args.n_tiles) : args.n_tiles;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_s(b), 1);
      mbar_init(bar_p(b), 256);
    }
    mbar_init(bar_o, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp < 8) reinterpret_cast<int*>(smem + C::kSeqOff)[threadIdx.x] = 0;
  if (warp == 9) {
    tmem_alloc(smem_addr(holder), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;

  // load order shared by the producer and the MMA warp: K_0, K_1, then V_j, K_{j+2}
  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    const uint32_t leader = elect_one();
    const uint64_t pol_q = policy_evict_first();
    const uint64_t pol_kv = policy_evict_last();
    const size_t head_atoms = static_cast<size_t>(bh) * args.n_tiles;
    if (leader) {
      mbar_arrive_expect_tx(bar_q, C::kTileBytes + C::kAtomBytes);
      tma_load_3d_hint(sbase + C::kQOff, &tm_q, bar_q, 0, row0, bh, pol_q);
      bulk_load(sbase + C::kQAtomOff, args.q_sf + (head_atoms + tile) * C::kAtomBytes, C::kAtomBytes, bar_q);
    }
    uint32_t slot = 0, ph = 0;
    int seq = 0;
    bool ok = true;
    auto load = [&](bool is_v, int blk) {
      ok = __all_sync(0xffffffffu, wait_bar(bar_empty(slot), ph ^ 1u, abort_flag, args.status, 1));
      if (!ok) return;
      if (leader) {
        mbar_arrive_expect_tx(bar_full(slot), C::kTileBytes + C::kAtomBytes);
        tma_load_3d_hint(sbase + C::kRingOff + slot * C::kTileBytes, is_v ? &tm_v : &tm_k, bar_full(slot), 0,
                         blk * 128, bh, pol_kv);
        bulk_load(sbase + C::kAtomOff + slot * C::kAtomBytes,
                  (is_v ? args.v_sf : args.k_sf) + (head_atoms + blk) * C::kAtomBytes, C::kAtomBytes, bar_full(slot));
      }
      ++seq;
      if (++slot == static_cast<uint32_t>(C::kSlots)) {
        slot = 0;
        ph ^= 1u;
      }
    };
    load(false, 0);
    if (ok && nblk > 1) load(false, 1);
    for (int j = 0; ok && j < nblk; ++j) {
      load(true, j);
      if (ok && j + 2 < nblk) load(false, j + 2);
    }
    if (!ok) {
      drain_bar(bar_q, 0);
      for (int s = seq - C::kSlots < 0 ? 0 : seq - C::kSlots; s < seq; ++s)
        drain_bar(bar_full(s % C::kSlots), (s / C::kSlots) & 1);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t leader = elect_one();
    auto commit = [&](uint32_t bar) {
      if (leader) tc_commit(bar);
    };
    auto wait = [&](uint32_t bar, uint32_t parity, uint32_t where) {
      return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, args.status, where));
    };
    // E4M3 tiles: one 128-byte swizzle row per matrix row; K-major Q and K
    // advance 32 bytes per K=32 step, MN-major V advances 32 rows (4096 bytes)
    const uint64_t q_desc = smem_desc_sw128(sbase + C::kQOff, 16, 1024);
    const uint64_t ring_k = smem_desc_sw128(sbase + C::kRingOff, 16, 1024);
    const uint64_t ring_v = smem_desc_sw128(sbase + C::kRingOff, C::kTileBytes, 1024);
    constexpr uint64_t kSlotStep = C::kTileBytes >> 4;
    uint32_t slot = 0, ph = 0;
    auto next = [&]() {
      if (++slot == static_cast<uint32_t>(C::kSlots)) {
        slot = 0;
        ph ^= 1u;
      }
    };
    auto issue_s = [&](int b, uint32_t kslot) {
      // K's scales into the buffer's B-scale columns, then 4 MMAs of K = 32
      const uint32_t sfk = tmem + C::col_sf_k(b);
      if (leader) {
        sf_copy_to_tmem(sfk, sbase + C::kAtomOff + kslot * C::kAtomBytes);
#pragma unroll
        for (uint32_t kk = 0; kk < 4; ++kk)
          mma_mxf8_ss(tmem + C::col_s(b), q_desc + 2 * kk, ring_k + kslot * kSlotStep + 2 * kk,
                      idesc_mxf8(128, 128, false, kk, kk), kk > 0 ? 1u : 0u, tmem + C::kColSfQ, sfk);
      }
    };
    auto issue_pv = [&](int b, uint32_t vslot, bool first) {
      const uint32_t sfv = tmem + C::col_sf_v(b);
      if (leader) {
        sf_copy_to_tmem(sfv, sbase + C::kAtomOff + vslot * C::kAtomBytes);
#pragma unroll
        for (uint32_t kk = 0; kk < 4; ++kk)
          mma_mxf8_ts(tmem + C::kColO, tmem + C::col_s(b) + 8 * kk, ring_v + vslot * kSlotStep + 256 * kk,
                      idesc_mxf8(128, 128, true, kk, kk), (!first || kk > 0) ? 1u : 0u, tmem + C::col_sf_p(b),
                      sfv);
      }
    };
    bool ok = wait(bar_q, 0, 2);
    if (ok) {
      tc_fence_after();
      if (leader) sf_copy_to_tmem(tmem + C::kColSfQ, sbase + C::kQAtomOff);
    }
    for (int b = 0; ok && b < 2 && b < nblk; ++b) {
      ok = wait(bar_full(slot), ph, 3);
      if (!ok) break;
      tc_fence_after();
      issue_s(b, slot);
      commit(bar_s(b));
      commit(bar_empty(slot));
      next();
    }
    for (int j = 0; ok && j < nblk; ++j) {
      const int b = j & 1;
      if (!wait(bar_full(slot), ph, 4)) break;  // V_j
      if (!wait(bar_p(b), (j >> 1) & 1, 5)) break;
      tc_fence_after();
      issue_pv(b, slot, j == 0);
      commit(bar_empty(slot));
      next();
      if (j + 2 < nblk) {
        if (!wait(bar_full(slot), ph, 6)) break;  // K_{j+2}
        tc_fence_after();
        issue_s(b, slot);
        commit(bar_s(b));
        commit(bar_empty(slot));
        next();
      } else if (j == nblk - 1) {
        commit(bar_o);
      }
    }
    commit(bar_drain);
    drain_bar(bar_drain, 0);
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int half = warp >> 2;
    const int r = quad * 32 + lane;
    const int grow = row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    float* xch = reinterpret_cast<float*>(smem + C::kXchOff);  // [parity][quad][half][lane][2]
    volatile float* lx = reinterpret_cast<volatile float*>(smem + C::kLOff);  // [half][128]
    volatile int* seqs = reinterpret_cast<volatile int*>(smem + C::kSeqOff);  // [half][128]
    volatile int* my_seq = seqs + half * 128 + r;
    const volatile int* their_seq = seqs + (half ^ 1) * 128 + r;
    const float sl2 = args.scale_log2;
    const float2 sl2_2 = make_float2(sl2, sl2);
    float m = -INFINITY;
    float l = 0.f;  // this half's share of the row sum
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      const int b = j & 1;
      ok = __all_sync(0xffffffffu, wait_bar(bar_s(b), (j >> 1) & 1, abort_flag, args.status, 16 + half));
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_tm = tmem + lane_off + C::col_s(b) + 64 * half;
      float2 s[32];
      {
        uint32_t u[2][32];
        tmem_ld32(s_tm, u[0]);
        tmem_ld32(s_tm + 32, u[1]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          reg_fence32(u[c]);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            s[16 * c + i] = make_float2(__uint_as_float(u[c][2 * i]), __uint_as_float(u[c][2 * i + 1]));
        }
      }
      const int kv0 = j * 128 + 64 * half;
      const bool need_mask = (j * 128 + 128 > args.n) || (CAUSAL && j == tile);
      if (need_mask) {
        int lim = args.n - 1 - kv0;
        if (CAUSAL) lim = min(lim, grow - kv0);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (2 * c > lim) s[c].x = -INFINITY;
          if (2 * c + 1 > lim) s[c].y = -INFINITY;
        }
      }
      // maxima of this half's two 32-key blocks (two interleaved chains each)
      float bmx[2];
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        float a = fmaxf(s[16 * g].x, s[16 * g].y);
        float c = fmaxf(s[16 * g + 1].x, s[16 * g + 1].y);
#pragma unroll
        for (int i = 2; i < 16; i += 2) {
          a = fmax3(a, s[16 * g + i].x, s[16 * g + i].y);
          c = fmax3(c, s[16 * g + i + 1].x, s[16 * g + i + 1].y);
        }
        bmx[g] = fmaxf(a, c);
      }
      // swap with the other half of the row (values double-buffered by block
      // parity; a per-thread sequence number publishes them)
      volatile float* mine = xch + ((((b * 4 + quad) * 2 + half) * 32 + lane) * 2);
      const volatile float* theirs = xch + ((((b * 4 + quad) * 2 + (half ^ 1)) * 32 + lane) * 2);
      mine[0] = bmx[0];
      mine[1] = bmx[1];
      __threadfence_block();
      my_seq[0] = j + 1;
      ok = __all_sync(0xffffffffu, wait_seq(their_seq, j + 1, abort_flag, args.status, 20));
      if (!ok) break;
      __threadfence_block();
      // the four 32-key block maxima of the row, in key order
      const float t0 = theirs[0], t1 = theirs[1];
      const float blk0 = half ? t0 : bmx[0], blk1 = half ? t1 : bmx[1];
      const float blk2 = half ? bmx[0] : t0, blk3 = half ? bmx[1] : t1;
      const float bm = fmaxf(fmaxf(blk0, blk1), fmaxf(blk2, blk3));
      float m_new = fmaxf(m, bm);
      const bool fire = !((m_new - m) * sl2 <= args.tau);
      if (!fire) m_new = m;
      const float corr = fire ? (m == -INFINITY ? 0.f : ex2_mufu((m - m_new) * sl2)) : 1.0f;
      m = m_new;
      const float neg_ms = (m == -INFINITY) ? 0.f : -(m * sl2);
      // E8M0 scale of each of this half's 32-key blocks of P: the block amax is
      // one exp of the block's score max
      const uint32_t sf_mine0 = e8m0_for_amax(ex2_mufu(__fmaf_rn(bmx[0], sl2, neg_ms)));
      const uint32_t sf_mine1 = e8m0_for_amax(ex2_mufu(__fmaf_rn(bmx[1], sl2, neg_ms)));
      // P / 2^e of a block is 2^(x - e): the block's scale goes into the exp's
      // shift, so the conversion needs no multiply; the fp32 row sum takes the
      // scaled block sums times 2^e.
      float lsum = 0.f;
      uint32_t pk[16];
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const uint32_t sfb = g ? sf_mine1 : sf_mine0;
        const float shift = neg_ms - static_cast<float>(static_cast<int>(sfb) - 127);
        const float2 shift_2 = make_float2(shift, shift);
        float2 acc = make_float2(0.f, 0.f);
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
          acc = __fadd2_rn(acc, __fadd2_rn(p0, p1));
          pk[8 * g + i / 2] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
        }
        lsum = __fmaf_rn(acc.x + acc.y, __uint_as_float(sfb << 23), lsum);  // * 2^(sfb - 127)
      }
      tmem_st16(tmem + lane_off + C::col_s(b) + 16 * half, pk);
      // the row's four P scales, one byte per key block, written by half 0
      // (half 1's two are recomputed from the swapped maxima)
      if (half == 0) {
        const uint32_t sf2 = e8m0_for_amax(ex2_mufu(__fmaf_rn(blk2, sl2, neg_ms)));
        const uint32_t sf3 = e8m0_for_amax(ex2_mufu(__fmaf_rn(blk3, sl2, neg_ms)));
        tmem_st1(tmem + lane_off + C::col_sf_p(b) + quad, sf_mine0 | (sf_mine1 << 8) | (sf2 << 16) | (sf3 << 24));
      }
      // correction of this half's O columns once the scores are dead
      if (j > 0 && __any_sync(0xffffffffu, fire)) {
        const float2 corr_2 = make_float2(corr, corr);
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          uint32_t ob[32];
          const uint32_t o_tm = tmem + lane_off + C::kColO + 64 * half + c;
          tmem_ld32(o_tm, ob);
          tmem_ld_wait();
          reg_fence32(ob);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 o2 = __fmul2_rn(make_float2(__uint_as_float(ob[i]), __uint_as_float(ob[i + 1])), corr_2);
            ob[i] = __float_as_uint(o2.x);
            ob[i + 1] = __float_as_uint(o2.y);
          }
          tmem_st32(o_tm, ob);
        }
      }
      l = l * corr + lsum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p(b));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar_o, 0, abort_flag, args.status, 18));
    // the row's sum is the two halves' sums
    if (ok) {
      lx[half * 128 + r] = l;
      __threadfence_block();
      my_seq[0] = nblk + 1;
      ok = __all_sync(0xffffffffu, wait_seq(their_seq, nblk + 1, abort_flag, args.status, 21));
      __threadfence_block();
    }
    if (ok) {
      tc_fence_after();
      const float l_row = lx[r] + lx[128 + r];
      const float inv_l = 1.0f / l_row;
      const bool valid = grow < args.n;
      __nv_bfloat16* orow = args.o + (static_cast<size_t>(bh) * args.n + (valid ? grow : 0)) * 128 + 64 * half;
      const float2 inv_l_2 = make_float2(inv_l, inv_l);
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        uint32_t ob[32];
        tmem_ld32(tmem + lane_off + C::kColO + 64 * half + c, ob);
        tmem_ld_wait();
        reg_fence32(ob);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 o2 = __fmul2_rn(make_float2(__uint_as_float(ob[2 * i]), __uint_as_float(ob[2 * i + 1])), inv_l_2);
          w[i] = pack_bf16x2(o2.x, o2.y);
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
      }
      if (valid && half == 0)
        args.lse[static_cast<size_t>(bh) * args.n + grow] = (m * sl2 + lg2_mufu(l_row)) * 0.69314718055994531f;
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <bool CAUSAL, int EMU>
cudaError_t launch_fwd_mxfp8(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const FwdMxArgs& args, cudaStream_t stream) {
  auto kernel = attn_fwd_mxfp8_kernel<CAUSAL, EMU>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MxCfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long ctas = static_cast<long long>(args.bh) * args.n_tiles;
  kernel<<<static_cast<unsigned>(ctas), MxCfg::kThreads, MxCfg::kSmemBytes, stream>>>(tm_q, tm_k, tm_v, args);
  return cudaGetLastError();
}

}  // namespace attn
