// C ABI of the attention forward library: argument checks, TMA tensor maps,
// dispatch to the kernel instantiations, the device error word and the
// software-exp2 check kernel. See include/attn.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "bwd_bf16.cuh"
#include "bwd_dispatch.h"
#include "bwd_mxfp8.cuh"
#include "exp2_fma.cuh"
#include "fwd_bf16.cuh"
#include "fwd_dispatch.h"
#include "fwd_mxfp8.cuh"
#include "schedule.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr long long kMaxN = 1LL << 24;
constexpr int kMaxCombineParts = 1024;
// log2(448 / 256), rounded down: the largest tau for which P * 2^8 <= 448
constexpr float kPConstMaxTau = 0.807f;
// log2(57344 / 256), rounded down: the same bound for P held in E5M2
constexpr float kPConstE5m2MaxTau = 7.807f;

// Device error word, one per device (each device holds its own copy).
__device__ unsigned int g_attn_status;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Address of g_attn_status on the current device (looked up once per device).
unsigned int* status_word() {
  static std::atomic<unsigned int*> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned int* p = cache[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_attn_status) != cudaSuccess) return nullptr;
  p = static_cast<unsigned int*>(addr);
  cache[dev].store(p, std::memory_order_release);
  return p;
}

// cuTensorMapEncodeTiled is a pure function of its arguments, so a small
// per-thread cache of recent encodings spares repeated calls on the same
// buffers (the common case of a training or serving loop) the host work.
struct MapKey {
  CUtensorMapDataType type;
  CUtensorMapSwizzle swizzle;
  const void* base;
  cuuint64_t dims[3];
  cuuint64_t strides[2];
  cuuint32_t box[3];
};

bool encode_3d(CUtensorMap* m, CUtensorMapDataType type, const void* base, const cuuint64_t (&dims)[3],
               const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3], CUtensorMapSwizzle swizzle) {
  constexpr int kEntries = 8;
  struct Entry {
    MapKey key;
    CUtensorMap map;
    bool valid;
  };
  thread_local Entry cache[kEntries];
  thread_local int next = 0;
  MapKey key;
  std::memset(&key, 0, sizeof key);  // padding bytes take part in the comparison
  key.type = type;
  key.swizzle = swizzle;
  key.base = base;
  std::memcpy(key.dims, dims, sizeof key.dims);
  std::memcpy(key.strides, strides, sizeof key.strides);
  std::memcpy(key.box, box, sizeof key.box);
  for (auto& e : cache)
    if (e.valid && std::memcmp(&e.key, &key, sizeof key) == 0) {
      *m = e.map;
      return true;
    }
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, type, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  Entry& e = cache[next];
  next = (next + 1) % kEntries;
  e.key = key;
  e.map = *m;
  e.valid = true;
  return true;
}

// 3-D map over a contiguous [B*H, N, d] bf16 tensor: d innermost, 64-column
// boxes (128 bytes, the 128-byte swizzle span) of 128 rows; rows past N of a
// head read as zero.
bool make_map(CUtensorMap* m, const void* base, int d, int n, long long bh) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2u, static_cast<cuuint64_t>(d) * 2u * static_cast<cuuint64_t>(n)};
  cuuint32_t box[3] = {64, 128, 1};
  return encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// The same over a [B*H, N, d] bf16 tensor with 64-row boxes: half of a
// 128-key block, the share of one CTA of a pair.
bool make_map_half_rows(CUtensorMap* m, const void* base, int d, int n, long long bh) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2u, static_cast<cuuint64_t>(d) * 2u * static_cast<cuuint64_t>(n)};
  cuuint32_t box[3] = {64, 64, 1};
  return encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 3-D map over a contiguous [B*H, N, 128] E4M3 tensor: one 128-byte swizzle
// row per sequence row, boxes of 128 rows.
bool make_map_e4m3(CUtensorMap* m, const void* base, int n, long long bh) {
  cuuint64_t dims[3] = {128u, static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {128u, 128u * static_cast<cuuint64_t>(n)};
  cuuint32_t box[3] = {128, 128, 1};
  return encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 3-D map over a contiguous [B*H, N, d] fp32 tensor for reduce-adds: 32-column
// boxes (128 bytes, the 128-byte swizzle span) of 128 rows; rows past N are
// not written.
bool make_map_f32(CUtensorMap* m, void* base, int d, int n, long long bh) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4u, static_cast<cuuint64_t>(d) * 4u * static_cast<cuuint64_t>(n)};
  cuuint32_t box[3] = {32, 128, 1};
  return encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 3-D map over a transposed fp32 accumulator [B*H, d, np] for reduce-adds:
// x = the sequence (N valid of a row stride of np), 32 x 32 boxes (128-byte
// rows, 128-byte swizzle); columns past N are not written.
bool make_map_f32_t(CUtensorMap* m, void* base, int d, int n, int np, long long bh) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(bh)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(np) * 4u, static_cast<cuuint64_t>(np) * 4u * static_cast<cuuint64_t>(d)};
  cuuint32_t box[3] = {32, 32, 1};
  return encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// SMs of the current device, queried once per device (the persistent grid size)
int sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// CTA pairs of the 2-CTA forward resident at once on the current device,
// queried once per device
int pair_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  n = attn::fwd_bf16_d128_2cta_max_clusters();
  if (n <= 0) return 0;
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Bytes of a rescale log: one per (head, row, 128-key block).
size_t rescale_log_size(int B, int H, int N) {
  if (B <= 0 || H <= 0 || N <= 0) return 0;
  return static_cast<size_t>(B) * H * N * ((static_cast<size_t>(N) + 127) / 128);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

long long band_for(long long kv_head_bytes, long long bh) {
  // heads whose K and V fit together in ~48 MiB of L2
  long long band = (48LL << 20) / (kv_head_bytes > 0 ? kv_head_bytes : 1);
  if (band < 1) band = 1;
  if (band > bh) band = bh;
  return band;
}

attn_status_t check_fwd_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
                             int H, int N, int d, int causal, float scale, float tau, int emu16, bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(tau) || tau < 0.f || tau > 16.f) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return (d > 0) ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG;
  if (emu16 < 0 || emu16 > 16) return ATTN_ERR_INVALID_ARG;
  if (emu16 > 4) return ATTN_ERR_UNSUPPORTED;
  if (N > kMaxN) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * ((N + 255) / 256) > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) {
    *empty = true;
    return ATTN_OK;
  }
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

__global__ void exp2_emulated_kernel(const float* __restrict__ x, float* __restrict__ y, long long n) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    y[i] = attn::exp2_fma(x[i]);
}

// The bf16 forward: argument checks, tensor maps, work list, dispatch. A
// non-null rescale_log selects the logging instantiation (MUFU exp2 only).
attn_status_t fwd_bf16(const void* q, const void* k, const void* v, void* o, float* lse, uint8_t* rescale_log,
                       int B, int H, int N, int d, int causal, float scale, float tau, int exp2_emu16, void* stream) {
  bool empty = false;
  attn_status_t st = check_fwd_args(q, k, v, o, lse, B, H, N, d, causal, scale, tau, exp2_emu16, &empty);
  if (st != ATTN_OK || empty) return st;
  const long long bh = static_cast<long long>(B) * H;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, d, N, bh) || !make_map(&mk, k, d, N, bh) || !make_map(&mv, v, d, N, bh))
    return ATTN_ERR_CUDA;
  unsigned int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  attn::FwdArgs a;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.status = status;
  a.n = N;
  a.n_kv_blocks = (N + 127) / 128;
  a.scale = scale;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.tau = tau;
  a.rescale_log = rescale_log;
  const int n_pairs = (N + 255) / 256;
  a.n_pairs = n_pairs;
  a.bh = static_cast<int>(bh);
  a.band = static_cast<int>(band_for(4LL * N * d, bh));
  const int sms = sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  // persistent grid: one CTA per SM, items from a list schedule when they fit
  // in one, else in serpentine rounds
  const long long items = bh * n_pairs;
  attn::WorkList wl;
  int ctas = static_cast<int>(std::min<long long>(items, std::min(sms, attn::kListMaxCtas)));
  a.use_list = attn::work_list_for(a.bh, n_pairs, a.n_kv_blocks, a.band, causal != 0, ctas, &wl) ? 1 : 0;
  if (!a.use_list) {
    std::memset(&wl, 0, sizeof(wl));
    ctas = static_cast<int>(std::min<long long>(items, sms));
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (rescale_log)
    e = attn::launch_fwd_bf16_log(d, causal, mq, mk, mv, a, wl, ctas, s);
  else if (d == 64)
    e = causal ? attn::launch_fwd_bf16_d64_c1(exp2_emu16, mq, mk, mv, a, wl, ctas, s)
               : attn::launch_fwd_bf16_d64_c0(exp2_emu16, mq, mk, mv, a, wl, ctas, s);
  else
    e = causal ? attn::launch_fwd_bf16_d128_c1(exp2_emu16, mq, mk, mv, a, wl, ctas, s)
               : attn::launch_fwd_bf16_d128_c0(exp2_emu16, mq, mk, mv, a, wl, ctas, s);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// The MXFP8 forward: argument checks, tensor maps, work list, dispatch;
// unroll_kv selects the unroll-KV schedule (MUFU exp2, per-32-key amax P only).
attn_status_t fwd_mxfp8(const void* q8, const void* q_sf, const void* k8, const void* k_sf, const void* v8,
                        const void* v_sf, void* o, float* lse, int B, int H, int N, int d, int causal, float scale,
                        float tau, int exp2_emu16, int p_scaling, bool unroll_kv, uint8_t* rescale_log,
                        void* stream) {
  if (B < 0 || H < 0 || N < 0 || (causal != 0 && causal != 1)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(tau) || tau < 0.f || tau > 16.f) return ATTN_ERR_INVALID_ARG;
  if (d != 128) return d > 0 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG;
  if (exp2_emu16 < 0 || exp2_emu16 > 16) return ATTN_ERR_INVALID_ARG;
  if (exp2_emu16 != 0 && exp2_emu16 != 2 && exp2_emu16 != 4) return ATTN_ERR_UNSUPPORTED;
  if (p_scaling != ATTN_P_SCALE_BLOCK_AMAX && p_scaling != ATTN_P_SCALE_CONSTANT &&
      p_scaling != ATTN_P_SCALE_CONSTANT_E5M2)
    return ATTN_ERR_INVALID_ARG;
  // constant 2^-8: the largest P, 2^tau, must stay within the format's largest
  // value / 256 (E4M3 448, E5M2 57344)
  if (p_scaling == ATTN_P_SCALE_CONSTANT && !(tau <= kPConstMaxTau)) return ATTN_ERR_INVALID_ARG;
  if (p_scaling == ATTN_P_SCALE_CONSTANT_E5M2 && !(tau <= kPConstE5m2MaxTau)) return ATTN_ERR_INVALID_ARG;
  if (N > kMaxN || static_cast<long long>(B) * H * ((N + 255) / 256) > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!q8 || !q_sf || !k8 || !k_sf || !v8 || !v_sf || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(q_sf) || !aligned16(k_sf) ||
      !aligned16(v_sf) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return ATTN_ERR_MISALIGNED;
  const long long bh = static_cast<long long>(B) * H;
  CUtensorMap mq, mk, mv;
  if (!make_map_e4m3(&mq, q8, N, bh) || !make_map_e4m3(&mk, k8, N, bh) || !make_map_e4m3(&mv, v8, N, bh))
    return ATTN_ERR_CUDA;
  unsigned int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  attn::FwdMxArgs a;
  a.q_sf = static_cast<const uint8_t*>(q_sf);
  a.k_sf = static_cast<const uint8_t*>(k_sf);
  a.v_sf = static_cast<const uint8_t*>(v_sf);
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.status = status;
  a.n = N;
  a.n_tiles = (N + 127) / 128;
  a.n_pairs = (N + 255) / 256;
  a.bh = static_cast<int>(bh);
  a.band = static_cast<int>(band_for(2LL * N * 128, bh));
  a.scale = scale;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.tau = tau;
  a.rescale_log = rescale_log;
  const int sms = sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  // persistent grid with the same work-list schedule as the bf16 kernel
  const long long items = bh * a.n_pairs;
  attn::WorkList wl;
  int ctas = static_cast<int>(std::min<long long>(items, std::min(sms, attn::kListMaxCtas)));
  a.use_list = attn::work_list_for(a.bh, a.n_pairs, a.n_tiles, a.band, causal != 0, ctas, &wl) ? 1 : 0;
  if (!a.use_list) {
    std::memset(&wl, 0, sizeof(wl));
    ctas = static_cast<int>(std::min<long long>(items, sms));
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (rescale_log)
    e = attn::launch_fwd_mxfp8_d128_log(causal, mq, mk, mv, a, wl, ctas, st);
  else if (unroll_kv)
    e = attn::launch_fwd_mxfp8_d128_ukv(causal, mq, mk, mv, a, wl, ctas, st);
  else if (p_scaling == ATTN_P_SCALE_CONSTANT)
    e = attn::launch_fwd_mxfp8_d128_pconst(causal, exp2_emu16, mq, mk, mv, a, wl, ctas, st);
  else if (p_scaling == ATTN_P_SCALE_CONSTANT_E5M2)
    e = attn::launch_fwd_mxfp8_d128_pconst_e5m2(causal, exp2_emu16, mq, mk, mv, a, wl, ctas, st);
  else
    e = attn::launch_fwd_mxfp8_d128(causal, exp2_emu16, mq, mk, mv, a, wl, ctas, st);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                          int d, int causal, float scale, float tau, int exp2_emu16, void* stream) {
  return fwd_bf16(q, k, v, o, lse, nullptr, B, H, N, d, causal, scale, tau, exp2_emu16, stream);
}

attn_status_t attn_fwd_2cta(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                            int d, int causal, float scale, void* stream) {
  bool empty = false;
  attn_status_t st = check_fwd_args(q, k, v, o, lse, B, H, N, d, causal, scale, 8.0f, 0, &empty);
  if (st != ATTN_OK || empty) return st;
  if (d != 128 || causal) return ATTN_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  CUtensorMap mq, mkh, mv;
  if (!make_map(&mq, q, d, N, bh) || !make_map_half_rows(&mkh, k, d, N, bh) || !make_map(&mv, v, d, N, bh))
    return ATTN_ERR_CUDA;
  unsigned int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  attn::FwdArgs a;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.status = status;
  a.n = N;
  a.n_kv_blocks = (N + 127) / 128;
  a.scale = scale;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.tau = 8.0f;
  a.rescale_log = nullptr;
  const int n_groups = (N + 511) / 512;  // a work item: 512 query rows of one head
  a.n_pairs = n_groups;
  a.bh = static_cast<int>(bh);
  a.band = static_cast<int>(band_for(4LL * N * d, bh));
  const int pairs = pair_count();
  if (pairs <= 0) return ATTN_ERR_CUDA;
  const long long items = bh * n_groups;
  attn::WorkList wl;
  int clusters = static_cast<int>(std::min<long long>(items, std::min(pairs, attn::kListMaxCtas)));
  a.use_list = attn::work_list_for(a.bh, n_groups, a.n_kv_blocks, a.band, false, clusters, &wl) ? 1 : 0;
  if (!a.use_list) {
    std::memset(&wl, 0, sizeof(wl));
    clusters = static_cast<int>(std::min<long long>(items, pairs));
  }
  const cudaError_t e =
      attn::launch_fwd_bf16_d128_2cta(mq, mkh, mv, a, wl, clusters, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_combine(const void* o_parts, const float* lse_parts, int parts, void* o, float* lse, int B,
                           int H, int N, int d, void* stream) {
  if (B < 0 || H < 0 || N < 0 || parts < 1 || parts > kMaxCombineParts) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return d > 0 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!o_parts || !lse_parts || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(o)) return ATTN_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(lse_parts) & 3u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return ATTN_ERR_MISALIGNED;
  const int sms = sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  const long long rows = static_cast<long long>(B) * H * N;
  const cudaError_t e =
      attn::launch_attn_combine(o_parts, lse_parts, parts, rows, d, o, lse, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_fwd_rescale_log(const void* q, const void* k, const void* v, void* o, float* lse,
                                   unsigned char* rescale_log, size_t rescale_log_bytes, int B, int H, int N, int d,
                                   int causal, float scale, float tau, void* stream) {
  bool empty = false;
  const attn_status_t st = check_fwd_args(q, k, v, o, lse, B, H, N, d, causal, scale, tau, 0, &empty);
  if (st != ATTN_OK || empty) return st;
  if (!rescale_log || rescale_log_bytes < rescale_log_size(B, H, N)) return ATTN_ERR_INVALID_ARG;
  return fwd_bf16(q, k, v, o, lse, rescale_log, B, H, N, d, causal, scale, tau, 0, stream);
}

size_t attn_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128) || N > kMaxN) return 0;
  const size_t bh = static_cast<size_t>(B) * H;
  const size_t np = (static_cast<size_t>(N) + 127) / 128 * 128;
  const size_t acc = (bh * np * d * 4 + 255) / 256 * 256;
  return acc + 2 * ((bh * np * 4 + 255) / 256 * 256);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                       float scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || H < 0 || N < 0 || (causal != 0 && causal != 1)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return (d > 0) ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG;
  if (N > kMaxN || static_cast<long long>(B) * H * ((N + 127) / 128) > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  // the preparation and conversion kernels put the head index on the grid's y axis
  if (static_cast<long long>(B) * H > 65535) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_bwd_workspace_bytes(B, H, N, d);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_MISALIGNED;
  const long long bh = static_cast<long long>(B) * H;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map(&mq, q, d, N, bh) || !make_map(&mk, k, d, N, bh) || !make_map(&mv, v, d, N, bh) ||
      !make_map(&mdo, dout, d, N, bh))
    return ATTN_ERR_CUDA;
  unsigned int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  const int np = (N + 127) / 128 * 128;
  const size_t acc_bytes = (static_cast<size_t>(bh) * np * d * 4 + 255) / 256 * 256;
  const size_t vec_bytes = (static_cast<size_t>(bh) * np * 4 + 255) / 256 * 256;
  float* dq_acc = static_cast<float*>(workspace);
  CUtensorMap mdq;
  if (!make_map_f32(&mdq, dq_acc, d, N, bh)) return ATTN_ERR_CUDA;
  float* lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_bytes);
  float* dvec = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_bytes + vec_bytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (attn::launch_bwd_prep(o, dout, lse, lse2, dvec, dq_acc, bh, N, np, d, st) != cudaSuccess) return ATTN_ERR_CUDA;
  attn::BwdArgs a;
  a.lse2 = lse2;
  a.dvec = dvec;
  a.dq_acc = dq_acc;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.status = status;
  a.n = N;
  a.np = np;
  a.n_tiles = (N + 127) / 128;
  a.bh = static_cast<int>(bh);
  a.scale = scale;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  cudaError_t e = d == 128 ? attn::launch_bwd_bf16_d128(causal, mq, mk, mv, mdo, mdq, a, st)
                           : attn::launch_bwd_bf16_d64(causal, mq, mk, mv, mdo, mdq, a, st);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  e = attn::launch_bwd_post(dq_acc, dq, bh * N * static_cast<long long>(d), scale, st);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_bwd_mxfp8(const void* q8, const void* q_sf, const void* k8, const void* k_sf, const void* v8,
                             const void* v_sf, const void* o, const void* do8, const void* do_sf, const float* lse,
                             void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                             void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || H < 0 || N < 0 || (causal != 0 && causal != 1)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (d != 128) return d > 0 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG;
  if (N > kMaxN || static_cast<long long>(B) * H * ((N + 127) / 128) > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 65535) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!q8 || !q_sf || !k8 || !k_sf || !v8 || !v_sf || !o || !do8 || !do_sf || !lse || !dq || !dk || !dv)
    return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_bwd_workspace_bytes(B, H, N, d);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(q_sf) || !aligned16(k8) || !aligned16(k_sf) || !aligned16(v8) ||
      !aligned16(v_sf) || !aligned16(o) || !aligned16(do8) || !aligned16(do_sf) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_MISALIGNED;
  const long long bh = static_cast<long long>(B) * H;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map_e4m3(&mq, q8, N, bh) || !make_map_e4m3(&mk, k8, N, bh) || !make_map_e4m3(&mv, v8, N, bh) ||
      !make_map_e4m3(&mdo, do8, N, bh))
    return ATTN_ERR_CUDA;
  unsigned int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  const int np = (N + 127) / 128 * 128;
  const size_t acc_bytes = (static_cast<size_t>(bh) * np * d * 4 + 255) / 256 * 256;
  const size_t vec_bytes = (static_cast<size_t>(bh) * np * 4 + 255) / 256 * 256;
  float* dq_acc = static_cast<float*>(workspace);  // transposed: [B*H, d, np]
  CUtensorMap mdq;
  if (!make_map_f32_t(&mdq, dq_acc, d, N, np, bh)) return ATTN_ERR_CUDA;
  float* lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_bytes);
  float* dvec = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_bytes + vec_bytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (attn::launch_bwd_prep_mxfp8(o, do8, do_sf, lse, lse2, dvec, dq_acc, bh, N, np, st) != cudaSuccess)
    return ATTN_ERR_CUDA;
  // role-2 scale arrays: the atoms whose rows are sequence positions, then
  // those whose rows are d columns
  const size_t sf_bytes = attn_mxfp8_scale_bytes(B, H, N, d);
  auto u8 = [](const void* p) { return static_cast<const uint8_t*>(p); };
  attn::BwdMxArgs a;
  a.q_sf = u8(q_sf);
  a.q_sf_t = u8(q_sf) + sf_bytes;
  a.k_sf = u8(k_sf);
  a.k_sf_t = u8(k_sf) + sf_bytes;
  a.v_sf = u8(v_sf);
  a.do_sf = u8(do_sf);
  a.do_sf_t = u8(do_sf) + sf_bytes;
  a.lse2 = lse2;
  a.dvec = dvec;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.status = status;
  a.n = N;
  a.np = np;
  a.n_tiles = (N + 127) / 128;
  a.bh = static_cast<int>(bh);
  a.scale = scale;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  cudaError_t e = attn::launch_bwd_mxfp8_d128(causal, mq, mk, mv, mdo, mdq, a, st);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  e = attn::launch_bwd_post_t(dq_acc, dq, bh, N, np, scale, st);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                       int causal, float scale, void* stream) {
  return attn_fwd_ex(q, k, v, o, lse, B, H, N, d, causal, scale, 8.0f, 0, stream);
}

size_t attn_mxfp8_scale_bytes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || d != 128) return 0;
  return static_cast<size_t>(B) * H * ((N + 127) / 128) * 512u;
}

attn_status_t attn_mxfp8_quantize(const float* x, void* x_e4m3, void* x_scales, int B, int H, int N, int d, int role,
                                  void* stream) {
  if (B < 0 || H < 0 || N < 0 || role < 0 || role > 2) return ATTN_ERR_INVALID_ARG;
  if (d != 128) return d > 0 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG;
  if (N > kMaxN || static_cast<long long>(B) * H > 65535) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!x || !x_e4m3 || !x_scales) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_e4m3) || !aligned16(x_scales)) return ATTN_ERR_MISALIGNED;
  cudaError_t e = attn::launch_mxfp8_quantize(x, static_cast<uint8_t*>(x_e4m3), static_cast<uint8_t*>(x_scales),
                                              static_cast<long long>(B) * H, N, role, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_fwd_mxfp8_ex(const void* q8, const void* q_sf, const void* k8, const void* k_sf, const void* v8,
                                const void* v_sf, void* o, float* lse, int B, int H, int N, int d, int causal,
                                float scale, float tau, int exp2_emu16, int p_scaling, void* stream) {
  return fwd_mxfp8(q8, q_sf, k8, k_sf, v8, v_sf, o, lse, B, H, N, d, causal, scale, tau, exp2_emu16, p_scaling,
                   false, nullptr, stream);
}

attn_status_t attn_fwd_mxfp8_rescale_log(const void* q8, const void* q_sf, const void* k8, const void* k_sf,
                                         const void* v8, const void* v_sf, void* o, float* lse,
                                         unsigned char* rescale_log, size_t rescale_log_bytes, int B, int H, int N,
                                         int d, int causal, float scale, float tau, void* stream) {
  if (B > 0 && H > 0 && N > 0 && (!rescale_log || rescale_log_bytes < rescale_log_size(B, H, N)))
    return ATTN_ERR_INVALID_ARG;
  return fwd_mxfp8(q8, q_sf, k8, k_sf, v8, v_sf, o, lse, B, H, N, d, causal, scale, tau, 0, ATTN_P_SCALE_BLOCK_AMAX,
                   false, rescale_log, stream);
}

attn_status_t attn_fwd_mxfp8_unroll_kv(const void* q8, const void* q_sf, const void* k8, const void* k_sf,
                                       const void* v8, const void* v_sf, void* o, float* lse, int B, int H, int N,
                                       int d, int causal, float scale, void* stream) {
  return fwd_mxfp8(q8, q_sf, k8, k_sf, v8, v_sf, o, lse, B, H, N, d, causal, scale, 0.0f, 0, ATTN_P_SCALE_BLOCK_AMAX,
                   true, nullptr, stream);
}

attn_status_t attn_fwd_mxfp8(const void* q8, const void* q_sf, const void* k8, const void* k_sf, const void* v8,
                             const void* v_sf, void* o, float* lse, int B, int H, int N, int d, int causal, float scale,
                             void* stream) {
  // tau = 0 for FP8 P: with a stale max a row's largest P is 2^delta instead of
  // exactly 1 and E4M3 rounds it by up to 2^-4 (FlashAttention-4's Softmax
  // Tricks, "Where exact breaks: P in FP8": tau 8 for 16-bit P, 0 for FP8)
  return attn_fwd_mxfp8_ex(q8, q_sf, k8, k_sf, v8, v_sf, o, lse, B, H, N, d, causal, scale, 0.0f, 0,
                           ATTN_P_SCALE_BLOCK_AMAX, stream);
}

attn_status_t attn_exp2_emulated(const float* x, float* y, long long n, void* stream) {
  if (n < 0) return ATTN_ERR_INVALID_ARG;
  if (n == 0) return ATTN_OK;
  if (!x || !y) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 3u) || (reinterpret_cast<uintptr_t>(y) & 3u)) return ATTN_ERR_MISALIGNED;
  const long long want = (n + 255) / 256;
  const int blocks = static_cast<int>(want < 152 * 16 ? want : 152 * 16);
  exp2_emulated_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_get_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned int* p = status_word();
  if (!p) return ATTN_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, p, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (word == 0) return ATTN_OK;
  const unsigned int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  const unsigned int code = word & 0xffu;
  return code == ATTN_ERR_TIMEOUT ? ATTN_ERR_TIMEOUT : ATTN_ERR_CUDA;
}

const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
  }
  return "ATTN_ERR_UNKNOWN";
}

attn_status_t attn_selftest_wait_timeout(long long limit_cycles, void* stream) {
  if (limit_cycles < 1000 || limit_cycles > 10000000000LL) return ATTN_ERR_INVALID_ARG;
  unsigned int* status = status_word();
  if (!status) return ATTN_ERR_CUDA;
  return attn::launch_wait_timeout_selftest(status, limit_cycles, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

int attn_version(void) { return 100; }

}  // extern "C"
