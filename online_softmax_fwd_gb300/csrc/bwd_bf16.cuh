// Attention backward, bf16 in / bf16 dQ, dK, dV out, for sm_103a.
//
// The gradient of O = softmax(s Q K^T) V with P rebuilt from the forward's
// LSE ("Lecture 2 - Online Softmax and Numerical Correctness", section "Use
// it in the real stack": the LSE side output makes the backward cheap), as
// the five products of "PyTorch FlashAttention-4 adds MXFP8 block-scaled
// forward and backward for Blackwell", section "TMEM allocation and scale
// factor placement", with dK and dV accumulated in TMEM for the whole life of
// a CTA. One CTA owns a 128-key tile j of one (batch, head) and streams the
// head's 128-row query tiles i (causal: i >= j):
//
//   S^T  = K_j Q_i^T            (keys x queries, fp32 in TMEM)
//   dP^T = V_j dO_i^T
//   P^T  = exp2(S^T s log2 e - LSE_i log2 e)       (masked entries 0)
//   dS^T = P^T * (dP^T - D_i),  D = rowsum(dO * O)
//   dV_j += P^T dO_i,   dK_j += dS^T Q_i           (A operands from TMEM)
//   dQ_i (+)= dS K_j                               (fp32 reduction in global)
//
//   warps 0-7   thread = key row (warps w and w + 4 share rows and split the
//               128 queries): P^T and dS^T, then the dK, dV epilogue
//   warps 8-11  thread = query row: dQ_i out of TMEM, through shared memory
//               (at d = 128 the stage's dO_i buffer, free once the dV product
//               has read it and handed back to the TMA warp afterwards; at
//               d = 64 a buffer of its own) into TMA reduce-adds onto the fp32 dQ
//   warp 12     TMA: K_j, V_j once; Q_i (with LSE_i log2 e and D_i) into a
//               ring of stages
//   warp 13     MMA issuer (one elected lane)
//   warp 14     TMA: dO_i into the same stages (loaded and released apart
//               from Q_i)
//
// TMEM: S^T at 0 (P^T as bf16 pairs over columns 0-31 and 64-95, each half
// over columns its own warp loaded), dP^T at 128 (dS^T likewise), dV at 256,
// dK at 256 + d, and at d = 64 dQ_i at 384. At d = 128 dQ_i reuses the dP^T
// columns, issued right behind the dK product that reads dS^T from them (one
// thread's products run in issue order), and the next dP^T waits until the
// dQ warps have loaded dQ_i. dS also
// goes to shared memory, keys x queries with queries contiguous, as the
// MN-major A operand of the dQ product.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bwd_common.cuh"
#include "fwd_bf16.cuh"
#include "kernel_setup.h"
#include "ptx.cuh"

namespace attn {

struct BwdArgs {
  const float* lse2;     // -LSE * log2(e), [B*H, np] (0 past N)
  const float* dvec;     // -D = -rowsum(dO * O), [B*H, np] (0 past N)
  float* dq_acc;         // fp32 [B*H, N, d], zeroed before the kernel; receives dS K (unscaled) through tm_dq
  __nv_bfloat16* dk;     // [B*H, N, d]
  __nv_bfloat16* dv;     // [B*H, N, d]
  unsigned int* status;  // device error word
  int n;                 // N
  int np;                // N rounded up to 128 (row stride of lse2 and dvec)
  int n_tiles;           // ceil(N / 128)
  int bh;                // B * H
  float scale;           // s
  float scale_log2;      // s * log2(e)
};

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kBoxes = D / 64;
  static constexpr uint32_t kBoxBytes = 128u * 128u;           // 128 rows x 64 bf16 (one swizzle span)
  static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;   // 128 x d bf16
  static constexpr int kStages = D == 128 ? 2 : 3;             // Q_i, dO_i ring
  static constexpr uint32_t kKOff = 0;
  static constexpr uint32_t kVOff = kTileBytes;
  // stage s: Q_i, dO_i, then LSE_i log2 e and D_i (128 floats each)
  static constexpr uint32_t kStageOff = 2 * kTileBytes;
  static constexpr uint32_t kVecOff = 2 * kTileBytes;          // within a stage
  static constexpr uint32_t kStageBytes = 2 * kTileBytes + 1024;
  static constexpr uint32_t kDsOff = kStageOff + kStages * kStageBytes;
  static constexpr uint32_t kDsBytes = 2 * kBoxBytes;          // 128 keys x 128 queries bf16
  // d = 64 has room for a buffer of its own for dQ on its way out (two fp32
  // 32-column boxes); d = 128 sends dQ through dO's buffer instead
  static constexpr bool kOwnDqBuf = D == 64;
  static constexpr uint32_t kDqBufOff = kDsOff + kDsBytes;
  static constexpr uint32_t kBarOff = kDqBufOff + (kOwnDqBuf ? 2 * kBoxBytes : 0);
  // kv, q_full[kStages], q_free[kStages], do_full[kStages], do_free[kStages], s, dp, p, ds, dv_done, k_done,
  // dq, ds_free, dq_read, fin, drain
  static constexpr int kNumBars = 1 + 4 * kStages + 11;
  static constexpr uint32_t kHolderOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kAbortOff = kHolderOff + 4;
  // the 1024-byte alignment of the tiles takes up to 1008 bytes of slack; at
  // d = 128 only what is left below the 227 KiB limit is reserved, and the
  // kernel checks its own base alignment against it
  static constexpr uint32_t kUsed = kAbortOff + 4;
  static constexpr uint32_t kSmemBytes = kUsed + 1024 <= 232448u ? kUsed + 1024 : 232448u;
  static constexpr uint32_t kSlack = kSmemBytes - kUsed;
  static_assert(kUsed + 256 <= 232448u, "shared memory");
  static constexpr int kThreads = 512;
  static constexpr int kDqWarp0 = 8, kTmaWarp = 12, kMmaWarp = 13, kDoWarp = 14;
  // setmaxnreg: 4 warps x 32 x (2 x 136 + 152 + 88) = 512 threads x 128 at launch
  static constexpr uint32_t kRegsDs = 136;
  static constexpr uint32_t kRegsDq = 152;
  static constexpr uint32_t kRegsProducer = 88;
  static constexpr int kLaunchRegs = 128;
  static_assert(2 * kRegsDs + kRegsDq + kRegsProducer <= 4 * kLaunchRegs, "register split");
  static constexpr uint32_t kTmemCols = 512;
  // dQ_i has columns of its own at d = 64; at d = 128 it reuses dP^T's
  static constexpr bool kDqAlias = D == 128;
  static constexpr uint32_t kColS = 0, kColDp = 128, kColDv = 256, kColDk = 256 + D,
                            kColDq = kDqAlias ? 128 : 256 + 2 * D;
};

// tcgen05 instruction descriptor, kind::f16, bf16 A and B, fp32 D, with the
// major-ness of both operands given
__host__ __device__ constexpr uint32_t idesc_bf16_f32_ab(int m, int n, bool a_mn_major, bool b_mn_major) {
  return idesc_bf16_f32(m, n, b_mn_major) | ((a_mn_major ? 1u : 0u) << 15);
}

// barrier among the 64 threads of P/dS warps w and w + 4 (ids 2 .. 5)
__device__ __forceinline__ void pair_sync(int quad) {
  asm volatile("bar.sync %0, 64;" ::"r"(2 + quad) : "memory");
}
__device__ __forceinline__ bool pair_all(int quad, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %2, 0;\n\t"
      "bar.red.and.pred p, %1, 64, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(2 + quad), "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}
// barrier among the 128 threads of the dQ warpgroup
__device__ __forceinline__ void dq_group_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// the same barrier, returning whether `v` holds in all 128 threads (so the
// group leaves its loop together and never waits at a barrier alone)
__device__ __forceinline__ bool dq_group_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 1, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(512, 1)
    attn_bwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dq, const BwdArgs args) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  if (pad > C::kSlack) {  // the layout does not fit this launch's shared-memory base
    if (threadIdx.x == 0) record_status(args.status, 2u /* ATTN_ERR_UNSUPPORTED */, 39);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + C::kBarOff;
  const uint32_t bar_kv = bar0;
  // a stage's Q_i (with LSE_i log2 e and D_i) and dO_i are loaded and freed separately:
  // Q_i is free after the dK product, dO_i after dQ_i has gone out through its buffer
  auto bar_qfull = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_qfree = [&](int s) { return bar0 + 8u * (1 + C::kStages + s); };
  auto bar_dofull = [&](int s) { return bar0 + 8u * (1 + 2 * C::kStages + s); };
  auto bar_dofree = [&](int s) { return bar0 + 8u * (1 + 3 * C::kStages + s); };
  const uint32_t bar_s = bar0 + 8u * (1 + 4 * C::kStages);
  const uint32_t bar_dp = bar_s + 8u;
  const uint32_t bar_p = bar_s + 16u;
  const uint32_t bar_ds = bar_s + 24u;
  const uint32_t bar_dvdone = bar_s + 32u;
  const uint32_t bar_kdone = bar_s + 40u;
  const uint32_t bar_dq = bar_s + 48u;
  const uint32_t bar_dsfree = bar_s + 56u;
  const uint32_t bar_dqread = bar_s + 64u;
  const uint32_t bar_fin = bar_s + 72u;
  const uint32_t bar_drain = bar_s + 80u;
  uint32_t* holder = reinterpret_cast<uint32_t*>(smem + C::kHolderOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kAbortOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA -> (head, key tile): the key tiles of one head run side by side, so
  // its Q and dO are read from L2 by all of them
  const int bh = blockIdx.x / args.n_tiles;
  const int j = blockIdx.x % args.n_tiles;
  const int i0 = CAUSAL ? j : 0;
  const int n_it = args.n_tiles - i0;

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_qfull(s), 1);
      mbar_init(bar_qfree(s), 1);
      mbar_init(bar_dofull(s), 1);
      // d = 128: arrived by the dQ warpgroup once its reduce-adds have read the buffer; d = 64: by the dV product
      mbar_init(bar_dofree(s), 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_p, 256);
    mbar_init(bar_ds, 256);
    mbar_init(bar_dvdone, 1);
    mbar_init(bar_kdone, 1);
    mbar_init(bar_dq, 1);
    mbar_init(bar_dsfree, 1);
    mbar_init(bar_dqread, 128);
    mbar_init(bar_fin, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_addr(holder), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;

  // (each register-count change sits inside its role's branch: ptxas sizes a
  // region by the setmaxnreg that dominates it)
  if (warp >= C::kTmaWarp) {
  regs_to<C::kRegsProducer, C::kLaunchRegs>();
  if (warp == C::kTmaWarp || warp == C::kDoWarp) {
    // ------------------------------------------------------------ TMA
    // Two loaders, so that neither waits behind the other's buffer: warp 12
    // K_j, V_j (once) and Q_i (with LSE_i log2 e and D_i), warp 14 dO_i.
    const uint32_t leader = elect_one();
    const uint64_t pol_stream = policy_evict_first();  // K_j, V_j: read by this CTA alone
    const uint64_t pol_keep = policy_evict_last();     // Q_i, dO_i: read by every key tile of the head
    const bool q_side = warp == C::kTmaWarp;
    if (q_side && leader) {
      mbar_arrive_expect_tx(bar_kv, 2 * C::kTileBytes);
#pragma unroll
      for (int b = 0; b < C::kBoxes; ++b) {
        tma_load_3d_hint(sbase + C::kKOff + b * C::kBoxBytes, &tm_k, bar_kv, b * 64, j * 128, bh, pol_stream);
        tma_load_3d_hint(sbase + C::kVOff + b * C::kBoxBytes, &tm_v, bar_kv, b * 64, j * 128, bh, pol_stream);
      }
    }
    int issued = 0;
    for (int i = 0; i < n_it; ++i) {
      const int st = i % C::kStages;
      const uint32_t ph = static_cast<uint32_t>(i / C::kStages) & 1u;
      const uint32_t dst = sbase + C::kStageOff + st * C::kStageBytes;
      if (q_side) {
        if (!__all_sync(0xffffffffu, wait_bar(bar_qfree(st), ph ^ 1u, abort_flag, args.status, 30))) break;
        if (leader) {
          const int row = (i0 + i) * 128;
          mbar_arrive_expect_tx(bar_qfull(st), C::kTileBytes + 1024);
#pragma unroll
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d_hint(dst + b * C::kBoxBytes, &tm_q, bar_qfull(st), b * 64, row, bh, pol_keep);
          const size_t vrow = static_cast<size_t>(bh) * args.np + row;
          bulk_g2s(dst + C::kVecOff, args.lse2 + vrow, 512, bar_qfull(st));
          bulk_g2s(dst + C::kVecOff + 512, args.dvec + vrow, 512, bar_qfull(st));
        }
      } else {
        if (!__all_sync(0xffffffffu, wait_bar(bar_dofree(st), ph ^ 1u, abort_flag, args.status, 29))) break;
        if (leader) {
          mbar_arrive_expect_tx(bar_dofull(st), C::kTileBytes);
#pragma unroll
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d_hint(dst + C::kTileBytes + b * C::kBoxBytes, &tm_do, bar_dofull(st), b * 64, (i0 + i) * 128,
                             bh, pol_keep);
        }
      }
      ++issued;
    }
    if (issued < n_it) {
      // a wait gave up: the copies in flight land before the CTA leaves
      if (q_side) drain_bar(bar_kv, 0);
      for (int s = issued - C::kStages < 0 ? 0 : issued - C::kStages; s < issued; ++s)
        drain_bar(q_side ? bar_qfull(s % C::kStages) : bar_dofull(s % C::kStages), (s / C::kStages) & 1);
    }
    __syncwarp();
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t leader = elect_one();
    auto commit = [&](uint32_t bar) {
      if (leader) tc_commit(bar);
    };
    auto wait = [&](uint32_t bar, uint32_t parity, uint32_t where) {
      return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, args.status, where));
    };
    constexpr uint32_t kIdSq = idesc_bf16_f32(128, 128, false);          // S^T, dP^T
    constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, true);            // dV, dK (A from TMEM)
    constexpr uint32_t kIdDq = idesc_bf16_f32_ab(128, D, true, true);    // dQ (A = dS MN-major)
    // low descriptor words (start >> 4, leading offset); the high word (8-row
    // groups 1024 bytes apart, 128-byte swizzle) is shared by all of them
    const uint64_t k0 = smem_desc_sw128(sbase + C::kKOff, 16, 1024);
    const uint32_t desc_hi = static_cast<uint32_t>(k0 >> 32);
    const uint32_t k_km = static_cast<uint32_t>(k0);
    const uint32_t v_km = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kVOff, 16, 1024));
    const uint32_t k_mn = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kKOff, C::kBoxBytes, 1024));
    const uint32_t ds_mn = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kDsOff, C::kBoxBytes, 1024));
    const uint32_t st_km = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kStageOff, 16, 1024));
    const uint32_t st_mn = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kStageOff, C::kBoxBytes, 1024));
    constexpr uint32_t kStageStep = C::kStageBytes >> 4;
    constexpr uint32_t kTileStep = C::kTileBytes >> 4;
    // K-major: the next 16 columns are 32 bytes on inside a swizzle row, every
    // 4th step starts the next 64-column box. MN-major: 16 rows further = 2048 bytes.
    auto kmajor_step = [](int kk) -> uint32_t { return ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4; };
    // Each issue starts from bases the compiler must treat as new values, so it
    // computes the per-step addresses on the spot instead of keeping all of
    // them (five products x 8-16 steps) in registers across the loop.
    auto opaque = [](uint32_t x) {
      asm volatile("" : "+r"(x));
      return x;
    };
    // S^T = K Q_i^T and dP^T = V dO_i^T (contraction over d)
    auto issue_sq = [&](uint32_t a_lo, uint32_t b_lo, uint32_t col) {
      a_lo = opaque(a_lo);
      b_lo = opaque(b_lo);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_lo(tmem + col, a_lo + kmajor_step(kk), b_lo + kmajor_step(kk), desc_hi, kIdSq, kk > 0 ? 1u : 0u);
      }
    };
    // dV += P^T dO_i, dK += dS^T Q_i (contraction over the 128 queries; A's
    // queries 0-63 at columns 0-31 of its region, 64-127 at 64-95)
    auto issue_acc = [&](uint32_t a_col, uint32_t b_lo, uint32_t d_col, bool first) {
      a_col = opaque(a_col);
      b_lo = opaque(b_lo);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_lo(tmem + d_col, tmem + a_col + (kk < 4 ? 8 * kk : 64 + 8 * (kk - 4)), b_lo + kk * 128, desc_hi, kIdAcc,
                    (!first || kk > 0) ? 1u : 0u);
      }
    };
    // dQ_i = dS K_j (contraction over the 128 keys)
    auto issue_dq = [&]() {
      const uint32_t a = opaque(ds_mn), b = opaque(k_mn);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss_lo(tmem + C::kColDq, a + kk * 128, b + kk * 128, desc_hi, kIdDq, kk > 0 ? 1u : 0u);
      }
    };
    bool ok = wait(bar_kv, 0, 31) && wait(bar_qfull(0), 0, 32);
    if (ok) {
      tc_fence_after();
      issue_sq(k_km, st_km, C::kColS);
      commit(bar_s);
      ok = wait(bar_dofull(0), 0, 39);
    }
    if (ok) {
      tc_fence_after();
      issue_sq(v_km, st_km + kTileStep, C::kColDp);
      commit(bar_dp);
    }
    for (int it = 0; ok && it < n_it; ++it) {
      const uint32_t par = static_cast<uint32_t>(it) & 1u;
      const int st = it % C::kStages;
      ok = wait(bar_p, par, 33);
      if (!ok) break;
      tc_fence_after();
      issue_acc(C::kColS, st_mn + st * kStageStep + kTileStep, C::kColDv, it == 0);  // B = dO_i
      commit(bar_dvdone);
      if constexpr (C::kOwnDqBuf) commit(bar_dofree(st));  // dO_i is read by this product alone
      const bool more = it + 1 < n_it;
      const int st1 = (it + 1) % C::kStages;
      if (more) {
        // S^T(i+1) overwrites P^T(i) once the dV product has read it; issued
        // before dK(i) so the P/dS warpgroup finds it ready after dS^T(i)
        ok = wait(bar_qfull(st1), static_cast<uint32_t>((it + 1) / C::kStages) & 1u, 35) &&
             wait(bar_dvdone, par, 36);
        if (!ok) break;
        tc_fence_after();
        issue_sq(k_km, st_km + st1 * kStageStep, C::kColS);
        commit(bar_s);
      }
      ok = wait(bar_ds, par, 34);
      if (!ok) break;
      tc_fence_after();
      issue_acc(C::kColDp, st_mn + st * kStageStep, C::kColDk, it == 0);  // B = Q_i
      commit(bar_qfree(st));
      if constexpr (C::kDqAlias) {
        // dQ_i over dS^T(i), right behind the dK product that reads it: one
        // thread's products run in issue order
        issue_dq();
        commit(bar_dq);
        commit(bar_dsfree);
        if (more) {
          // dP^T(i+1) overwrites dQ_i once the dQ warps have loaded it
          ok = wait(bar_dqread, par, 38) &&
               wait(bar_dofull(st1), static_cast<uint32_t>((it + 1) / C::kStages) & 1u, 46);
          if (!ok) break;
          tc_fence_after();
          issue_sq(v_km, st_km + st1 * kStageStep + kTileStep, C::kColDp);
          commit(bar_dp);
        }
      } else {
        // dQ_i in its own columns once the dQ warps have loaded dQ_{i-1}
        if (it > 0) {
          ok = wait(bar_dqread, par ^ 1u, 38);
          if (!ok) break;
          tc_fence_after();
        }
        issue_dq();
        commit(bar_dq);
        commit(bar_dsfree);
        if (more) {
          // dP^T(i+1) over dS^T(i), behind the dK product that reads it (issue
          // order)
          ok = wait(bar_dofull(st1), static_cast<uint32_t>((it + 1) / C::kStages) & 1u, 46);
          if (!ok) break;
          tc_fence_after();
          issue_sq(v_km, st_km + st1 * kStageStep + kTileStep, C::kColDp);
          commit(bar_dp);
        }
      }
    }
    commit(bar_fin);
    // nothing may still be executing when TMEM is released
    commit(bar_drain);
    drain_bar(bar_drain, 0);
    __syncwarp();
  }
  } else if (warp < C::kDqWarp0) {
    // ------------------------------------------------------------ P^T, dS^T (thread = key row)
    // Warps w and w + 4 share key rows 32 (w % 4) .. and take queries
    // 64 h .. 64 h + 63 (h = w / 4). Each stores its half of P^T and dS^T as
    // bf16 pairs over the first 32 of the 64 fp32 columns it loaded itself.
    regs_to<C::kRegsDs, C::kLaunchRegs>();
    const int quad = warp & 3, h = warp >> 2;
    const int r = quad * 32 + lane;
    const int kj = j * 128 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + C::kColS;
    const uint32_t dp_tm = tmem + lane_off + C::kColDp;
    const float2 sl2_2 = make_float2(args.scale_log2, args.scale_log2);
    const uint32_t ds_row = sbase + C::kDsOff + r * 128;
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      const uint32_t par = static_cast<uint32_t>(it) & 1u;
      const int q0 = (i0 + it) * 128;
      // this query tile's LSE log2 e and D, in its stage
      const uint32_t vec = sbase + C::kStageOff + (it % C::kStages) * C::kStageBytes + C::kVecOff;
      // queries past N, and on the causal diagonal tile keys after the query
      const bool need_mask = (q0 + 128 > args.n) || (CAUSAL && it == 0);
      int lim = args.n - 1 - q0;  // last valid query column
      // S^T(i) is complete, and the stage's vectors have landed (the stage is
      // refilled only after this warpgroup's dS^T(i) has been consumed)
      ok = __all_sync(0xffffffffu, wait_bar(bar_s, par, abort_flag, args.status, 40) &&
                                       wait_bar(bar_qfull(it % C::kStages), static_cast<uint32_t>(it / C::kStages) & 1u,
                                                abort_flag, args.status, 45));
      if (!ok) break;
      tc_fence_after();
      uint32_t pk[32];  // this warp's 64 queries of the P^T row, as bf16 pairs
      {
        uint32_t u[2][32];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) tmem_ld32(s_tm + 32 * (2 * h + kk), u[kk]);
        tmem_ld_wait();
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int k = 2 * h + kk;
          reg_fence32(u[kk]);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 l4 = lds_f4(vec + 4u * (32 * k + 4 * c4));  // -LSE log2 e
            const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(u[kk][4 * c4]), __uint_as_float(u[kk][4 * c4 + 1])),
                                          sl2_2, make_float2(l4.x, l4.y));
            const float2 x23 = __ffma2_rn(make_float2(__uint_as_float(u[kk][4 * c4 + 2]), __uint_as_float(u[kk][4 * c4 + 3])),
                                          sl2_2, make_float2(l4.z, l4.w));
            const float xs[4] = {x01.x, x01.y, x23.x, x23.y};
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = 32 * k + 4 * c4 + e;
              p[e] = ex2_mufu(xs[e]);
              if (need_mask && (c > lim || (CAUSAL && kj > q0 + c))) p[e] = 0.f;
            }
            pk[16 * kk + 2 * c4] = pack_bf16x2(p[0], p[1]);
            pk[16 * kk + 2 * c4 + 1] = pack_bf16x2(p[2], p[3]);
          }
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = pk[16 * kk + e];
          tmem_st16(s_tm + 64 * h + 16 * kk, w);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p);
      // dS^T = P^T (dP^T - D); the dS buffer in shared memory is free once the
      // previous dQ product has read it
      {
        bool w_ok = wait_bar(bar_dp, par, abort_flag, args.status, 41);
        if (w_ok && it > 0) w_ok = wait_bar(bar_dsfree, par ^ 1u, abort_flag, args.status, 42);
        ok = __all_sync(0xffffffffu, w_ok);
      }
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t u[2][32];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) tmem_ld32(dp_tm + 32 * (2 * h + kk), u[kk]);
        tmem_ld_wait();
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int k = 2 * h + kk;
          reg_fence32(u[kk]);
          uint32_t w[16];
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 d4 = lds_f4(vec + 512u + 4u * (32 * k + 4 * c4));  // -D
            const uint32_t a = pk[16 * kk + 2 * c4], b = pk[16 * kk + 2 * c4 + 1];
            const float2 ds01 = __fmul2_rn(make_float2(bf16_lo(a), bf16_hi(a)),
                                           __fadd2_rn(make_float2(__uint_as_float(u[kk][4 * c4]),
                                                                  __uint_as_float(u[kk][4 * c4 + 1])),
                                                      make_float2(d4.x, d4.y)));
            const float2 ds23 = __fmul2_rn(make_float2(bf16_lo(b), bf16_hi(b)),
                                           __fadd2_rn(make_float2(__uint_as_float(u[kk][4 * c4 + 2]),
                                                                  __uint_as_float(u[kk][4 * c4 + 3])),
                                                      make_float2(d4.z, d4.w)));
            w[2 * c4] = pack_bf16x2(ds01.x, ds01.y);
            w[2 * c4 + 1] = pack_bf16x2(ds23.x, ds23.y);
          }
          tmem_st16(dp_tm + 64 * h + 16 * kk, w);
          // shared memory: key row r, queries 32k .. 32k+31 = 16-byte chunks
          // 4(k%2) .. 4(k%2)+3 of box k/2, 128-byte swizzled
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const uint32_t chunk = static_cast<uint32_t>(4 * (k & 1) + v4);
            st_shared_v4(ds_row + (k >> 1) * C::kBoxBytes + ((chunk ^ static_cast<uint32_t>(r & 7)) << 4),
                         w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
          }
        }
      }
      tmem_st_wait();
      fence_async_shared();  // the generic-proxy stores of dS, before the tensor core reads them
      tc_fence_before();
      mbar_arrive(bar_ds);
    }
    // ---------------------------------------------------------- dK, dV epilogue
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar_fin, 0, abort_flag, args.status, 43));
    if (ok) {
      tc_fence_after();
      const bool valid = kj < args.n;
      const size_t off = (static_cast<size_t>(bh) * args.n + (valid ? kj : 0)) * D;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const float mul = which ? args.scale : 1.0f;
        __nv_bfloat16* dst = (which ? args.dk : args.dv) + off;
        const uint32_t src = tmem + lane_off + (which ? C::kColDk : C::kColDv);
#pragma unroll
        for (int c = h * (D / 2); c < (h + 1) * (D / 2); c += 32) {
          uint32_t u[32];
          tmem_ld32(src + c, u);
          tmem_ld_wait();
          reg_fence32(u);
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(u[2 * e]) * mul, __uint_as_float(u[2 * e + 1]) * mul);
          if (valid) {
            uint4* o4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) o4[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
          }
        }
      }
    }
    tc_fence_before();
  } else {
    // ------------------------------------------------------------ dQ (thread = query row)
    regs_to<C::kRegsDq, C::kLaunchRegs>();
    // dQ_i leaves TMEM at once (the next dP^T may then take its columns) and
    // goes out through dO_i's buffer (the dV product that read dO_i is
    // complete before dQ_i is computed) as 32-column fp32 boxes (128-byte
    // rows, 128-byte swizzle), each reduce-added onto the fp32 dQ by one TMA
    // operation; the buffer goes back to the TMA warp once they have read it.
    const int q = (warp - C::kDqWarp0) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp - C::kDqWarp0) * 32) << 16;
    const bool issuer = q == 0;
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      ok = dq_group_all(wait_bar(bar_dq, static_cast<uint32_t>(it) & 1u, abort_flag, args.status, 44));
      if (!ok) break;
      tc_fence_after();
      uint32_t u[D / 32][32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem + lane_off + C::kColDq + 32 * c, u[c]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar_dqread);
      const int st = it % C::kStages;
      // dO_i's buffer, or at d = 64 the dQ buffer
      const uint32_t buf = C::kOwnDqBuf ? sbase + C::kDqBufOff
                                        : sbase + C::kStageOff + st * C::kStageBytes + C::kTileBytes;
      // one 32-column box at a time through the buffer's box slots, each box
      // its own bulk group, so writing the next box overlaps the reduce-add
      // of the previous ones
      constexpr int kSlots = C::kOwnDqBuf ? 2 : C::kBoxes;
      if (C::kOwnDqBuf && it > 0) {
        // the previous dQ's reduce-adds have read the buffer
        if (issuer) bulk_wait_read();
        dq_group_sync();
      }
#pragma unroll
      for (int bb = 0; bb < D / 32; ++bb) {
        const uint32_t slot = buf + (bb % kSlots) * C::kBoxBytes;
        if (bb >= kSlots) {
          // the reduce-add that last used this slot has read it
          if (issuer) {
            if constexpr (kSlots == 2)
              asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            else
              bulk_wait_read();
          }
          dq_group_sync();
        }
        reg_fence32(u[bb]);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          st_shared_v4(slot + q * 128 + ((static_cast<uint32_t>(c4) ^ static_cast<uint32_t>(q & 7)) << 4),
                       u[bb][4 * c4], u[bb][4 * c4 + 1], u[bb][4 * c4 + 2], u[bb][4 * c4 + 3]);
        fence_async_shared();
        dq_group_sync();
        if (issuer) {
          tma_reduce_add_3d(&tm_dq, slot, 32 * bb, (i0 + it) * 128, bh);
          bulk_commit();
        }
      }
      if (!C::kOwnDqBuf && issuer) {
        bulk_wait_read();
        mbar_arrive(bar_dofree(st));
      }
      __syncwarp();
    }
    if (issuer) bulk_wait_all();
  }

  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_bwd_bf16(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                            const CUtensorMap& tm_do, const CUtensorMap& tm_dq, const BwdArgs& args,
                            cudaStream_t stream) {
  using C = BwdCfg<D>;
  constexpr auto kernel = attn_bwd_bf16_kernel<D, CAUSAL>;
  // shared-memory opt-in and the setmaxnreg register check, once per device
  const cudaError_t e = kernel_ready<kernel>(C::kSmemBytes, C::kLaunchRegs);
  if (e != cudaSuccess) return e;
  const long long ctas = static_cast<long long>(args.bh) * args.n_tiles;
  kernel<<<static_cast<unsigned>(ctas), C::kThreads, C::kSmemBytes, stream>>>(tm_q, tm_k, tm_v, tm_do, tm_dq, args);
  return cudaGetLastError();
}

}  // namespace attn
