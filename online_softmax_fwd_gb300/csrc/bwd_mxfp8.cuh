// Attention backward with MXFP8 block-scaled MMAs (d = 128), for sm_103a.
//
// The five products of the bf16 backward (bwd_bf16.cuh), each on the
// block-scaled tensor cores, as "PyTorch FlashAttention-4 adds MXFP8
// block-scaled forward and backward for Blackwell" describes them: Q, K and dO
// quantised in square 32 x 32 blocks, so that one E4M3 payload in shared
// memory serves the products along d and those along the sequence (section
// "Quantization along both axes and jagged tensors"), with a scale-factor atom
// per layout; dS quantised online in square 32 x 32 blocks, so that the dK and
// dQ products read one representation; P converted online with the constant
// scale 2^-8 (section "Softmax conversion and unroll-KV": softmax keeps P in
// [0, 1]). V is quantised in the same square blocks and enters dP alone.
//
// One CTA owns a 128-key tile j of one (batch, head) and streams the head's
// query tiles i (causal: i >= j):
//   S^T  = K_j Q_i^T           A = K_j, B = Q_i     (shared memory, K-major)
//   dP^T = V_j dO_i^T          A = V_j, B = dO_i    (shared memory, K-major)
//   P^T  = exp2(S^T s log2 e - LSE_i log2 e), to E4M3 x 2^8 in TMEM
//   dS^T = P^T (dP^T - D_i),    to E4M3 in 32 x 32 blocks, in TMEM and smem
//   dV_j += P^T dO_i           A = P^T (TMEM), B = dO_i (MN-major)
//   dK_j += dS^T Q_i           A = dS^T (TMEM), B = Q_i (MN-major)
//   dQ_i^T = K_j^T dS^T        A = K_j^T (K-major), B = dS (MN-major)
// dQ is taken transposed (A then comes from a K-major copy of K_j^T the dQ
// warps make once), so that every product has its A operand K-major or in
// TMEM; the fp32 dQ accumulator is kept transposed too, [B*H, d, N], and the
// last kernel turns it back while rounding to bf16.
//
//   warps 0-7   thread = key row; warps w and w + 4 share key rows 32 (w % 4)
//               .. and take queries 64 h .. 64 h + 63 (h = w / 4): P^T, dS^T
//               and their scales, then the dK, dV epilogue
//   warps 8-11  thread = d column: K_j^T once; then dQ_i^T out of TMEM into
//               the dQ buffer (warp 8 + b: d rows 32 b .. 32 b + 31, four
//               boxes of 32 queries) and TMA reduce-adds onto the transposed
//               fp32 dQ
//   warp 12     TMA: K_j, V_j and their atoms once; Q_i (+ 8 - LSE_i log2 e,
//               -D_i and Q's two atoms) into a ring of stages
//   warp 13     MMA issuer (one elected lane); tcgen05.cp of every atom
//   warp 14     TMA: dO_i (+ its two atoms) into the same stages
//
// TMEM (512 columns): S^T 0-127, dP^T 128-255, dV 256-383, dK 384-511; dQ_i^T
// takes the dP^T columns, issued right behind the dK product that reads dS^T
// from them (one thread's products run in issue order), and the next dP^T
// waits until the dQ warps have loaded dQ_i^T. P^T and dS^T as E4M3 (four
// queries per column) take columns 0-15 (queries 0-63, warp h = 0) and 64-79
// (queries 64-127, h = 1) of their region, among the columns each warp loaded
// itself. The scale factors sit in columns of the S^T and dP^T regions that
// are dead at the time (the same page, section "TMEM allocation and scale
// factor placement"):
//   S^T region  32-35 P^T's (the constant), 36-39 dO_i's (dV); 40-47 K^T's and
//               dS's (dQ_i) and 48-55 V's and dO_{i+1}'s (dP_{i+1}), once the
//               P warps have loaded S^T_{i+1}
//   dP^T region 32-35 and 96-99 dS^T's (query blocks 0-1 and 2-3), 36-39
//               Q_i's (dK); 40-47 K's and Q_{i+1}'s (S_{i+1}), once the dS
//               warps have loaded dP^T_i
// The first S and dP products read their scales from the dV and dK regions,
// which no product has written yet. Each extra dependency is one barrier:
// "dP^T loaded" before S_{i+1}, "S^T loaded" before dQ_i.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bwd_common.cuh"
#include "fwd_bf16.cuh"
#include "mxfp8_common.cuh"
#include "kernel_setup.h"
#include "ptx.cuh"

namespace attn {

struct BwdMxArgs {
  const uint8_t* q_sf;    // Q atoms, rows = query (S product), [B*H][tiles][512]
  const uint8_t* q_sf_t;  // Q atoms, rows = d column (dK product)
  const uint8_t* k_sf;    // K atoms, rows = key (S product)
  const uint8_t* k_sf_t;  // K atoms, rows = d column (dQ product)
  const uint8_t* v_sf;    // V atoms, rows = key (dP product)
  const uint8_t* do_sf;   // dO atoms, rows = query (dP product)
  const uint8_t* do_sf_t; // dO atoms, rows = d column (dV product)
  const float* lse2;      // 8 - LSE * log2(e), [B*H, np] (0 past N)
  const float* dvec;      // -D = -rowsum(dO * O), [B*H, np] (0 past N)
  __nv_bfloat16* dk;      // [B*H, N, 128]
  __nv_bfloat16* dv;      // [B*H, N, 128]
  unsigned int* status;
  int n;
  int np;                 // N rounded up to 128
  int n_tiles;            // ceil(N / 128)
  int bh;
  float scale;
  float scale_log2;
};

struct BwdMxCfg {
  static constexpr uint32_t kTileBytes = 128u * 128u;  // 128 x 128 E4M3
  static constexpr uint32_t kAtomBytes = 512u;
  static constexpr int kStages = 2;
  static constexpr uint32_t kKOff = 0;
  static constexpr uint32_t kVOff = kTileBytes;
  // K (rows = key), K (rows = d), V (rows = key)
  static constexpr uint32_t kKvAtomOff = 2 * kTileBytes;
  // stage: Q_i, dO_i, LSE_i log2 e - 8 and D_i, Q_i's atoms (rows = query,
  // rows = d), dO_i's atoms (the same two)
  static constexpr uint32_t kStageOff = 34u * 1024u;
  static constexpr uint32_t kVecOff = 2 * kTileBytes;
  static constexpr uint32_t kQAtomOff = kVecOff + 1024;
  static constexpr uint32_t kDoAtomOff = kQAtomOff + 2 * kAtomBytes;
  static constexpr uint32_t kStageBytes = kDoAtomOff + 2 * kAtomBytes;  // 35 KiB
  static constexpr uint32_t kDsOff = kStageOff + kStages * kStageBytes;  // dS, keys x queries, queries contiguous
  static constexpr uint32_t kDsAtomOff = kDsOff + kTileBytes;            // dS's scales, rows = query (dQ product)
  static constexpr uint32_t kKtOff = (kDsAtomOff + kAtomBytes + 1023u) / 1024u * 1024u;  // K^T, d x keys, keys contiguous
  static constexpr uint32_t kDqBufOff = kKtOff + kTileBytes;
  static constexpr uint32_t kDqBufBytes = 4 * kTileBytes;                // per dQ warp 4 boxes of 32 d x 32 fp32
  static constexpr uint32_t kDqBoxBytes = 32u * 128u;
  static constexpr uint32_t kBarOff = kDqBufOff + kDqBufBytes;
  // kv, q_full[2], q_free[2], do_full[2], do_free[2], s, dp, p, ds, dv_done, k_done, dq, ds_free, dq_read, fin,
  // drain, dp_loaded, s_loaded, kt_ready
  static constexpr int kNumBars = 1 + 4 * kStages + 14;
  static constexpr uint32_t kHolderOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kAbortOff = kHolderOff + 4;
  static constexpr uint32_t kUsed = kAbortOff + 4;
  static constexpr uint32_t kSmemBytes = kUsed + 1024;
  static_assert(kSmemBytes <= 232448u, "shared memory");
  static_assert(kStageOff % 1024 == 0 && kStageBytes % 1024 == 0 && kDsOff % 1024 == 0 && kKtOff % 1024 == 0 &&
                    kDqBufOff % 1024 == 0,
                "1024-byte tiles");
  static_assert(kKvAtomOff + 3 * kAtomBytes <= kStageOff, "K, V atoms");
  static constexpr int kThreads = 512;
  static constexpr int kDqWarp0 = 8, kTmaWarp = 12, kMmaWarp = 13, kDoWarp = 14;
  // setmaxnreg: 4 warps x 32 x (2 x 152 + 120 + 88) = 512 threads x 128 at launch
  static constexpr uint32_t kRegsDs = 152;
  static constexpr uint32_t kRegsDq = 120;
  static constexpr uint32_t kRegsProducer = 88;
  static constexpr int kLaunchRegs = 128;
  static_assert(2 * kRegsDs + kRegsDq + kRegsProducer <= 4 * kLaunchRegs, "register split");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDp = 128, kColDv = 256, kColDk = 384, kColDq = 128;
  // scale-factor columns, offsets inside the S^T and dP^T regions: the A
  // operand's at 32 or 40, the B operand's 4 further
  static constexpr uint32_t kSfTs = 32;  // TMEM-A products: P^T / dS^T (queries 0-63), then dO_i / Q_i
  static constexpr uint32_t kSfTsHi = 96;  // dS^T's scales for queries 64-127
  static constexpr uint32_t kSfDp = 48;    // dP_{i+1} (S^T region)
  static constexpr uint32_t kSfSs = 40;  // shared-memory products: dQ_i and dP_{i+1} (S^T region), S_{i+1} (dP^T region)
  // the constant E8M0 byte of P^T: 2^-8 (P = 1 is held as 256)
  static constexpr uint32_t kPScaleByte = 119u;
};

template <bool CAUSAL>
__global__ void __launch_bounds__(512, 1)
    attn_bwd_mxfp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_dq, const BwdMxArgs args) {
  using C = BwdMxCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + C::kBarOff;
  const uint32_t bar_kv = bar0;
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
  const uint32_t bar_dpld = bar_s + 88u;  // the dS warps have loaded dP^T_i
  const uint32_t bar_sld = bar_s + 96u;   // the P warps have loaded S^T_i
  const uint32_t bar_ktr = bar_s + 104u;  // the dQ warps have written K^T
  uint32_t* holder = reinterpret_cast<uint32_t*>(smem + C::kHolderOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kAbortOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA -> (head, key tile), the key tiles of one head side by side
  const int bh = blockIdx.x / args.n_tiles;
  const int j = blockIdx.x % args.n_tiles;
  const int i0 = CAUSAL ? j : 0;
  const int n_it = args.n_tiles - i0;
  const size_t head_atoms = static_cast<size_t>(bh) * args.n_tiles;

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_qfull(s), 1);
      mbar_init(bar_qfree(s), 1);
      mbar_init(bar_dofull(s), 1);
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
    mbar_init(bar_dpld, 256);
    mbar_init(bar_sld, 256);
    mbar_init(bar_ktr, 128);
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

  // (each register-count change sits inside its role's branch)
  if (warp >= C::kTmaWarp) {
  regs_to<C::kRegsProducer, C::kLaunchRegs>();
  if (warp == C::kTmaWarp || warp == C::kDoWarp) {
    // ------------------------------------------------------------ TMA
    // Two loaders, so that neither waits behind the other's buffer: warp 12
    // K_j, V_j (once) and Q_i, warp 14 dO_i. Q_i's stage frees after the dK
    // product, dO_i's after the dV product, one product apart in time.
    const uint32_t leader = elect_one();
    const uint64_t pol_stream = policy_evict_first();  // K_j, V_j: this CTA alone
    const uint64_t pol_keep = policy_evict_last();     // Q_i, dO_i: every key tile of the head
    const bool q_side = warp == C::kTmaWarp;
    if (q_side && leader) {
      mbar_arrive_expect_tx(bar_kv, 2 * C::kTileBytes + 3 * C::kAtomBytes);
      tma_load_3d_hint(sbase + C::kKOff, &tm_k, bar_kv, 0, j * 128, bh, pol_stream);
      tma_load_3d_hint(sbase + C::kVOff, &tm_v, bar_kv, 0, j * 128, bh, pol_stream);
      const size_t a = (head_atoms + j) * C::kAtomBytes;
      bulk_load(sbase + C::kKvAtomOff, args.k_sf + a, C::kAtomBytes, bar_kv);
      bulk_load(sbase + C::kKvAtomOff + C::kAtomBytes, args.k_sf_t + a, C::kAtomBytes, bar_kv);
      bulk_load(sbase + C::kKvAtomOff + 2 * C::kAtomBytes, args.v_sf + a, C::kAtomBytes, bar_kv);
    }
    int issued = 0;
    for (int i = 0; i < n_it; ++i) {
      const int st = i % C::kStages;
      const uint32_t ph = static_cast<uint32_t>(i / C::kStages) & 1u;
      const uint32_t dst = sbase + C::kStageOff + st * C::kStageBytes;
      const size_t a = (head_atoms + i0 + i) * C::kAtomBytes;
      if (q_side) {
        if (!__all_sync(0xffffffffu, wait_bar(bar_qfree(st), ph ^ 1u, abort_flag, args.status, 50))) break;
        if (leader) {
          const int row = (i0 + i) * 128;
          mbar_arrive_expect_tx(bar_qfull(st), C::kTileBytes + 1024 + 2 * C::kAtomBytes);
          tma_load_3d_hint(dst, &tm_q, bar_qfull(st), 0, row, bh, pol_keep);
          const size_t vrow = static_cast<size_t>(bh) * args.np + row;
          bulk_load(dst + C::kVecOff, args.lse2 + vrow, 512, bar_qfull(st));
          bulk_load(dst + C::kVecOff + 512, args.dvec + vrow, 512, bar_qfull(st));
          bulk_load(dst + C::kQAtomOff, args.q_sf + a, C::kAtomBytes, bar_qfull(st));
          bulk_load(dst + C::kQAtomOff + C::kAtomBytes, args.q_sf_t + a, C::kAtomBytes, bar_qfull(st));
        }
      } else {
        if (!__all_sync(0xffffffffu, wait_bar(bar_dofree(st), ph ^ 1u, abort_flag, args.status, 51))) break;
        if (leader) {
          mbar_arrive_expect_tx(bar_dofull(st), C::kTileBytes + 2 * C::kAtomBytes);
          tma_load_3d_hint(dst + C::kTileBytes, &tm_do, bar_dofull(st), 0, (i0 + i) * 128, bh, pol_keep);
          bulk_load(dst + C::kDoAtomOff, args.do_sf + a, C::kAtomBytes, bar_dofull(st));
          bulk_load(dst + C::kDoAtomOff + C::kAtomBytes, args.do_sf_t + a, C::kAtomBytes, bar_dofull(st));
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
    // descriptor low words (start >> 4, leading offset); the high word (8-row
    // groups 1024 bytes apart, 128-byte swizzle) is shared. A 128 x 128 E4M3
    // tile has 128-byte rows: K-major, the next 32 columns are 32 bytes on;
    // MN-major, the next 32 rows are 4096 bytes on.
    const uint64_t k0 = smem_desc_sw128(sbase + C::kKOff, 16, 1024);
    const uint32_t desc_hi = static_cast<uint32_t>(k0 >> 32);
    const uint32_t k_km = static_cast<uint32_t>(k0);
    const uint32_t v_km = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kVOff, 16, 1024));
    const uint32_t kt_km = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kKtOff, 16, 1024));
    const uint32_t ds_mn = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kDsOff, C::kTileBytes, 1024));
    const uint32_t st_km = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kStageOff, 16, 1024));
    const uint32_t st_mn = static_cast<uint32_t>(smem_desc_sw128(sbase + C::kStageOff, C::kTileBytes, 1024));
    constexpr uint32_t kStageStep = C::kStageBytes >> 4;
    constexpr uint32_t kTileStep = C::kTileBytes >> 4;
    auto stage_addr = [&](int st) { return sbase + C::kStageOff + static_cast<uint32_t>(st) * C::kStageBytes; };
    const uint32_t atom_k = sbase + C::kKvAtomOff, atom_kt = atom_k + C::kAtomBytes,
                   atom_v = atom_k + 2 * C::kAtomBytes;
    auto opaque = [](uint32_t x) {
      asm volatile("" : "+r"(x));
      return x;
    };
    // D = A B^T with both operands in shared memory, A K-major, B K-major
    // (S^T, dP^T) or MN-major (dQ^T): the A and B atoms are copied to TMEM
    // columns sf and sf + 4 first
    auto issue_ss = [&](uint32_t a_lo, uint32_t b_lo, uint32_t d_col, uint32_t sf, uint32_t atom_a, uint32_t atom_b,
                        bool b_mn) {
      a_lo = opaque(a_lo);
      b_lo = opaque(b_lo);
      if (leader) {
        sf_copy_to_tmem(tmem + sf, atom_a);
        sf_copy_to_tmem(tmem + sf + 4, atom_b);
#pragma unroll
        for (uint32_t kk = 0; kk < 4; ++kk)
          mma_mxf8_ss_lo(tmem + d_col, a_lo + 2 * kk, b_lo + (b_mn ? 256 : 2) * kk, desc_hi,
                         idesc_mxf8(128, 128, b_mn, kk, kk), kk > 0 ? 1u : 0u, tmem + sf, tmem + sf + 4);
      }
    };
    // the same product with the scales already in TMEM columns sf, sf + 4
    auto issue_ss_nocp = [&](uint32_t a_lo, uint32_t b_lo, uint32_t d_col, uint32_t sf) {
      a_lo = opaque(a_lo);
      b_lo = opaque(b_lo);
      if (leader) {
#pragma unroll
        for (uint32_t kk = 0; kk < 4; ++kk)
          mma_mxf8_ss_lo(tmem + d_col, a_lo + 2 * kk, b_lo + 2 * kk, desc_hi, idesc_mxf8(128, 128, false, kk, kk),
                         kk > 0 ? 1u : 0u, tmem + sf, tmem + sf + 4);
      }
    };
    // D += A B with A (E4M3) in TMEM region a_reg -- k-steps 0, 1 (queries
    // 0-63) at columns 0-15, k-steps 2, 3 at 64-79 -- its scales at a_reg + 32
    // (P^T: one constant column; dS^T: bytes of query blocks 0, 1 there and of
    // 2, 3 at a_reg + 96), B MN-major in shared memory with its atom copied to
    // a_reg + 36 (dV = P^T dO_i, dK = dS^T Q_i)
    auto issue_ts = [&](uint32_t a_reg, uint32_t b_lo, uint32_t d_col, uint32_t atom_b, bool first, bool split_sf) {
      b_lo = opaque(b_lo);
      if (leader) {
        sf_copy_to_tmem(tmem + a_reg + C::kSfTs + 4, atom_b);
#pragma unroll
        for (uint32_t kk = 0; kk < 4; ++kk)
          mma_mxf8_ts_lo(tmem + d_col, tmem + a_reg + (kk < 2 ? 8 * kk : 64 + 8 * (kk - 2)), b_lo + 256 * kk,
                         desc_hi, idesc_mxf8(128, 128, true, split_sf ? (kk & 1u) : kk, kk),
                         (!first || kk > 0) ? 1u : 0u,
                         tmem + a_reg + (split_sf && kk >= 2 ? C::kSfTsHi : C::kSfTs), tmem + a_reg + C::kSfTs + 4);
      }
    };
    // the first S^T and dP^T take their scales from the dV and dK regions
    bool ok = wait(bar_kv, 0, 52) && wait(bar_qfull(0), 0, 53);
    if (ok) {
      tc_fence_after();
      issue_ss(k_km, st_km, C::kColS, C::kColDv, atom_k, stage_addr(0) + C::kQAtomOff, false);
      commit(bar_s);
      ok = wait(bar_dofull(0), 0, 54);
    }
    if (ok) {
      tc_fence_after();
      issue_ss(v_km, st_km + kTileStep, C::kColDp, C::kColDk, atom_v, stage_addr(0) + C::kDoAtomOff, false);
      commit(bar_dp);
    }
    for (int it = 0; ok && it < n_it; ++it) {
      const uint32_t par = static_cast<uint32_t>(it) & 1u;
      const int st = it % C::kStages;
      const bool more = it + 1 < n_it;
      const int st1 = (it + 1) % C::kStages;
      const uint32_t par1 = static_cast<uint32_t>((it + 1) / C::kStages) & 1u;
      ok = wait(bar_p, par, 55);
      if (!ok) break;
      tc_fence_after();
      // dV += P^T dO_i (B = dO_i MN-major, its atom whose rows are d columns)
      issue_ts(C::kColS, st_mn + st * kStageStep + kTileStep, C::kColDv,
               stage_addr(st) + C::kDoAtomOff + C::kAtomBytes, it == 0, false);
      commit(bar_dvdone);
      commit(bar_dofree(st));  // dO_i: read by dP^T_i (earlier) and this product
      if (more) {
        // S^T_{i+1} overwrites P^T_i once the dV product has read it; its
        // scales go where the dS warps have already loaded dP^T_i
        ok = wait(bar_qfull(st1), par1, 56) && wait(bar_dvdone, par, 57) && wait(bar_dpld, par, 58);
        if (!ok) break;
        tc_fence_after();
        issue_ss(k_km, st_km + st1 * kStageStep, C::kColS, C::kColDp + C::kSfSs, atom_k,
                 stage_addr(st1) + C::kQAtomOff, false);
        commit(bar_s);
      }
      ok = wait(bar_ds, par, 59);
      if (!ok) break;
      tc_fence_after();
      // dK += dS^T Q_i (B = Q_i MN-major, its atom whose rows are d columns)
      issue_ts(C::kColDp, st_mn + st * kStageStep, C::kColDk, stage_addr(st) + C::kQAtomOff + C::kAtomBytes,
               it == 0, true);
      commit(bar_qfree(st));  // Q_i: read by S^T_i and this product
      // dQ_i^T = K^T dS^T over the dP^T columns, issued right behind dK: the
      // tensor core runs one thread's products in issue order, so dK has read
      // dS^T before dQ_i writes over it (as the O product reads P before the
      // next S product overwrites it in the forward kernel). Its scales go
      // into the S^T region once the P warps have loaded S^T_{i+1} (which also
      // means S^T_{i+1}, whose scales sit in the dP^T columns, is complete);
      // K^T is written once.
      ok = (!more || wait(bar_sld, static_cast<uint32_t>(it + 1) & 1u, 61)) && (it > 0 || wait(bar_ktr, 0, 70));
      if (!ok) break;
      tc_fence_after();
      // A = K^T (rows d, its atom whose rows are d columns), B = dS (rows
      // queries, MN-major; the atom the dS warps wrote)
      issue_ss(kt_km, ds_mn, C::kColDq, C::kColS + C::kSfSs, atom_kt, sbase + C::kDsAtomOff, true);
      commit(bar_dq);
      commit(bar_dsfree);
      if (more) {
        // dP^T_{i+1}'s scales go into S^T columns 48-55 as soon as dO_{i+1}
        // has landed (the P warps have loaded S^T_{i+1}); the product itself
        // overwrites dQ_i^T once the dQ warps have loaded it
        ok = wait(bar_dofull(st1), par1, 63);
        if (!ok) break;
        if (leader) {
          sf_copy_to_tmem(tmem + C::kColS + C::kSfDp, atom_v);
          sf_copy_to_tmem(tmem + C::kColS + C::kSfDp + 4, stage_addr(st1) + C::kDoAtomOff);
        }
        ok = wait(bar_dqread, par, 62);
        if (!ok) break;
        tc_fence_after();
        issue_ss_nocp(v_km, st_km + st1 * kStageStep + kTileStep, C::kColDp, C::kColS + C::kSfDp);
        commit(bar_dp);
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
    // Warps w and w + 4 share key rows and split the queries; each stores its
    // half of P^T (dS^T) and its scales over the 64 columns it loaded itself.
    regs_to<C::kRegsDs, C::kLaunchRegs>();
    const int quad = warp & 3, h = warp >> 2;
    const int r = quad * 32 + lane;
    const int kj = j * 128 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + C::kColS;
    const uint32_t dp_tm = tmem + lane_off + C::kColDp;
    const float2 sl2_2 = make_float2(args.scale_log2, args.scale_log2);
    // this thread's row of dS (keys x queries, 128-byte swizzled rows)
    const uint32_t ds_row = sbase + C::kDsOff + r * 128;
    // dQ's B atom: row = query m, block = key block (this warp's quad); every
    // lane l writes its replica row l
    const uint32_t ds_atom = sbase + C::kDsAtomOff + lane * 16 + quad;
    // keys past N take no part (their P is 0), so they do not enter the
    // 32 x 32 blocks' maxima
    const bool key_valid = kj < args.n;
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      const uint32_t par = static_cast<uint32_t>(it) & 1u;
      const int st = it % C::kStages;
      const int q0 = (i0 + it) * 128;
      // this query tile's 8 - LSE log2 e and -D, in its stage
      const uint32_t vec = sbase + C::kStageOff + st * C::kStageBytes + C::kVecOff;
      const bool need_mask = (q0 + 128 > args.n) || (CAUSAL && it == 0) || (j * 128 + 128 > args.n);
      const int lim = key_valid ? args.n - 1 - q0 : -1;  // last valid query column of this row
      ok = __all_sync(0xffffffffu, wait_bar(bar_s, par, abort_flag, args.status, 64) &&
                                       wait_bar(bar_qfull(st), static_cast<uint32_t>(it / C::kStages) & 1u,
                                                abort_flag, args.status, 65));
      if (!ok) break;
      tc_fence_after();
      // P^T 2^8 = exp2(S^T s log2 e + (8 - LSE log2 e)) for this warp's 64 queries
      float p8[64];
      {
        uint32_t u[2][32];
        tmem_ld32(s_tm + 64 * h, u[0]);
        tmem_ld32(s_tm + 64 * h + 32, u[1]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bar_sld);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          reg_fence32(u[kk]);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 l4 = lds_f4(vec + 4u * (64 * h + 32 * kk + 4 * c4));
            const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(u[kk][4 * c4]), __uint_as_float(u[kk][4 * c4 + 1])),
                                          sl2_2, make_float2(l4.x, l4.y));
            const float2 x23 = __ffma2_rn(make_float2(__uint_as_float(u[kk][4 * c4 + 2]), __uint_as_float(u[kk][4 * c4 + 3])),
                                          sl2_2, make_float2(l4.z, l4.w));
            const float xs[4] = {x01.x, x01.y, x23.x, x23.y};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = 64 * h + 32 * kk + 4 * c4 + e;
              float p = ex2_mufu(xs[e]);
              if (need_mask && (c > lim || (CAUSAL && kj > q0 + c))) p = 0.f;
              p8[32 * kk + 4 * c4 + e] = p;
            }
          }
        }
      }
      {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = pack_e4m3x4(p8[4 * e], p8[4 * e + 1], p8[4 * e + 2], p8[4 * e + 3]);
        tmem_st16(s_tm + 64 * h, w);
        // P^T's scales: the constant 2^-8 for every row and k-step
        if (h == 0) tmem_st1(s_tm + C::kSfTs + quad, C::kPScaleByte * 0x01010101u);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p);
      // dS^T = P^T (dP^T - D); dS's shared-memory buffer and atom are free once
      // the previous dQ product has read them
      {
        bool w_ok = wait_bar(bar_dp, par, abort_flag, args.status, 66);
        if (w_ok && it > 0) w_ok = wait_bar(bar_dsfree, par ^ 1u, abort_flag, args.status, 67);
        ok = __all_sync(0xffffffffu, w_ok);
      }
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t u[2][32];
        tmem_ld32(dp_tm + 64 * h, u[0]);
        tmem_ld32(dp_tm + 64 * h + 32, u[1]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bar_dpld);
        uint32_t w[16];
        uint32_t sfw = 0;
        // dS 2^8 = P^T 2^8 (dP^T - D) over two 32 x 32 blocks: 32 queries of
        // this row each, the blocks' 32 rows being the warp's lanes; both
        // blocks' maxima are reduced across the warp side by side
        float amax[2] = {0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          reg_fence32(u[kk]);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 d4 = lds_f4(vec + 512u + 4u * (64 * h + 32 * kk + 4 * c4));  // -D
            const int i = 32 * kk + 4 * c4;
            const float2 t01 = __fmul2_rn(make_float2(p8[i], p8[i + 1]),
                                          __fadd2_rn(make_float2(__uint_as_float(u[kk][4 * c4]),
                                                                 __uint_as_float(u[kk][4 * c4 + 1])),
                                                     make_float2(d4.x, d4.y)));
            const float2 t23 = __fmul2_rn(make_float2(p8[i + 2], p8[i + 3]),
                                          __fadd2_rn(make_float2(__uint_as_float(u[kk][4 * c4 + 2]),
                                                                 __uint_as_float(u[kk][4 * c4 + 3])),
                                                     make_float2(d4.z, d4.w)));
            p8[i] = t01.x;
            p8[i + 1] = t01.y;
            p8[i + 2] = t23.x;
            p8[i + 3] = t23.y;
            amax[kk] = fmax3(amax[kk], fabsf(t01.x), fabsf(t01.y));
            amax[kk] = fmax3(amax[kk], fabsf(t23.x), fabsf(t23.y));
          }
        }
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) {
          amax[0] = fmaxf(amax[0], __shfl_xor_sync(0xffffffffu, amax[0], sh));
          amax[1] = fmaxf(amax[1], __shfl_xor_sync(0xffffffffu, amax[1], sh));
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          // the E8M0 byte of dS is that of dS 2^8 minus 8 (clamped at the
          // bottom of the range, where the codes then carry the difference)
          const uint32_t b8 = e8m0_for_amax(amax[kk]);
          const uint32_t b = b8 < 8u ? 0u : b8 - 8u;
          const float inv = e8m0_inverse(b + 8u);
          const float2 inv_2 = make_float2(inv, inv);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int i = 32 * kk + 4 * e;
            const float2 a = __fmul2_rn(make_float2(p8[i], p8[i + 1]), inv_2);
            const float2 c = __fmul2_rn(make_float2(p8[i + 2], p8[i + 3]), inv_2);
            w[8 * kk + e] = pack_e4m3x4(a.x, a.y, c.x, c.y);
          }
          const uint32_t qb = static_cast<uint32_t>(2 * h + kk);
          sfw |= b << (8 * kk);
          asm volatile("st.shared.u8 [%0], %1;" ::"r"(ds_atom + qb * 4), "r"(b) : "memory");
        }
        // dS for the dQ product: key row r, queries 64h .. 64h + 63 = 16-byte
        // chunks 4h .. 4h + 3 of the 128-byte swizzled row
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          const uint32_t chunk = static_cast<uint32_t>(4 * h + v4);
          st_shared_v4(ds_row + ((chunk ^ static_cast<uint32_t>(r & 7)) << 4), w[4 * v4], w[4 * v4 + 1],
                       w[4 * v4 + 2], w[4 * v4 + 3]);
        }
        // dS^T for the dK product over this warp's own columns, with its
        // scales (query blocks 2h, 2h + 1)
        tmem_st16(dp_tm + 64 * h, w);
        tmem_st1(dp_tm + (h ? C::kSfTsHi : C::kSfTs) + quad, sfw);
      }
      tmem_st_wait();
      fence_async_shared();  // dS and its atom, before the tensor core reads them
      tc_fence_before();
      mbar_arrive(bar_ds);
    }
    // ---------------------------------------------------------- dK, dV epilogue
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar_fin, 0, abort_flag, args.status, 68));
    if (ok) {
      tc_fence_after();
      const size_t off = (static_cast<size_t>(bh) * args.n + (key_valid ? kj : 0)) * 128;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const float mul = which ? args.scale : 1.0f;
        __nv_bfloat16* dst = (which ? args.dk : args.dv) + off;
        const uint32_t src = tmem + lane_off + (which ? C::kColDk : C::kColDv);
#pragma unroll
        for (int c = h * 64; c < (h + 1) * 64; c += 32) {
          uint32_t u[32];
          tmem_ld32(src + c, u);
          tmem_ld_wait();
          reg_fence32(u);
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(u[2 * e]) * mul, __uint_as_float(u[2 * e + 1]) * mul);
          if (key_valid) {
            uint4* o4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) o4[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
          }
        }
      }
    }
    tc_fence_before();
  } else {
    // ------------------------------------------------------------ dQ (thread = d column)
    // Warp 8 + b owns d rows 32 b .. 32 b + 31 of dQ^T: it writes their rows of
    // K^T once, then for every query tile loads their rows of dQ_i^T (two
    // halves of 64 queries; the next dP^T may take the columns after the
    // second) into four boxes of 32 queries -- 32 rows of 32 fp32, 128-byte
    // rows, 128-byte swizzle -- which its lane 0 reduce-adds onto the
    // transposed fp32 dQ.
    regs_to<C::kRegsDq, C::kLaunchRegs>();
    const int wq = warp - C::kDqWarp0;
    const int dcol = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    bool ok = __all_sync(0xffffffffu, wait_bar(bar_kv, 0, abort_flag, args.status, 71));
    if (ok) {
      // K^T row dcol, K-major: key k is byte k % 16 of chunk k / 16, the chunks
      // swizzled by dcol % 8; K_j holds (key k, column dcol) at byte dcol % 16
      // of chunk (dcol / 16) ^ (k % 8) of row k
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t wv[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t word = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = 16 * c + 4 * q4 + e;
            const uint32_t src = sbase + C::kKOff + k * 128 +
                                 (((static_cast<uint32_t>(dcol >> 4)) ^ static_cast<uint32_t>(k & 7)) << 4) +
                                 (dcol & 15);
            uint32_t byte;
            asm volatile("ld.shared.u8 %0, [%1];" : "=r"(byte) : "r"(src) : "memory");
            word |= (byte & 0xFFu) << (8 * e);
          }
          wv[q4] = word;
        }
        st_shared_v4(sbase + C::kKtOff + dcol * 128 + ((static_cast<uint32_t>(c) ^ static_cast<uint32_t>(dcol & 7)) << 4),
                     wv[0], wv[1], wv[2], wv[3]);
      }
      fence_async_shared();  // K^T, before the tensor core reads it
      mbar_arrive(bar_ktr);
    }
    // this lane's row in each box: 16-byte chunk c at ((c ^ lane % 8) << 4)
    const uint32_t boxes = sbase + C::kDqBufOff + static_cast<uint32_t>(wq) * 4u * C::kDqBoxBytes;
    const uint32_t row = boxes + static_cast<uint32_t>(lane) * 128u;
    for (int it = 0; ok && it < n_it; ++it) {
      // this warp's previous reduce-adds have read the boxes
      if (lane == 0 && it > 0) bulk_wait_read();
      __syncwarp();
      ok = __all_sync(0xffffffffu, wait_bar(bar_dq, static_cast<uint32_t>(it) & 1u, abort_flag, args.status, 69));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t u[2][32];
        tmem_ld32(tmem + lane_off + C::kColDq + 64 * half, u[0]);
        tmem_ld32(tmem + lane_off + C::kColDq + 64 * half + 32, u[1]);
        tmem_ld_wait();
        if (half == 1) {
          tc_fence_before();
          mbar_arrive(bar_dqread);
        }
#pragma unroll
        for (int b2 = 0; b2 < 2; ++b2) {
          reg_fence32(u[b2]);
          const uint32_t box_row = row + static_cast<uint32_t>(2 * half + b2) * C::kDqBoxBytes;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(box_row + ((static_cast<uint32_t>(c) ^ static_cast<uint32_t>(lane & 7)) << 4),
                         u[b2][4 * c], u[b2][4 * c + 1], u[b2][4 * c + 2], u[b2][4 * c + 3]);
        }
      }
      fence_async_shared();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int bb = 0; bb < 4; ++bb)
          tma_reduce_add_3d(&tm_dq, boxes + bb * C::kDqBoxBytes, (i0 + it) * 128 + 32 * bb, 32 * wq, bh);
        bulk_commit();
      }
      __syncwarp();
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <bool CAUSAL>
cudaError_t launch_bwd_mxfp8(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const CUtensorMap& tm_do, const CUtensorMap& tm_dq, const BwdMxArgs& args,
                             cudaStream_t stream) {
  using C = BwdMxCfg;
  constexpr auto kernel = attn_bwd_mxfp8_kernel<CAUSAL>;
  // shared-memory opt-in and the setmaxnreg register check, once per device
  const cudaError_t e = kernel_ready<kernel>(C::kSmemBytes, C::kLaunchRegs);
  if (e != cudaSuccess) return e;
  const long long ctas = static_cast<long long>(args.bh) * args.n_tiles;
  kernel<<<static_cast<unsigned>(ctas), C::kThreads, C::kSmemBytes, stream>>>(tm_q, tm_k, tm_v, tm_do, tm_dq, args);
  return cudaGetLastError();
}

}  // namespace attn
