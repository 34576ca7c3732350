// C ABI of the attention library (declared in include/fa.h): argument
// validation, TMA tensor-map encoding, kernel launches, test hooks and the
// device status word. No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_decode.h"
#include "fa_fp8.h"
#include "fa_kernels.h"

namespace {

// First device-side error since the last clear (one per device that loads the library).
__device__ unsigned int g_fa_status;

constexpr int kMaxDevices = 64;
std::atomic<unsigned long long> g_timeout_ns{4000000000ull};
std::atomic<int> g_inject_stall{0};

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  int major = 0;
  unsigned int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encoder() {
  std::call_once(g_encode_once, []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  });
  return g_encode;
}

// Per-device set-up, done once per device with that device current.
fa_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FA_ERR_CUDA;
    di.num_sms = prop.multiProcessorCount;
    di.major = prop.major;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return FA_ERR_CUDA;
    di.status = static_cast<unsigned int*>(p);
    di.ready = true;
  }
  if (di.major != 10) return FA_ERR_UNSUPPORTED;
  *out = &di;
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int p8_of(float p) {
  if (!(p >= 0.f) || !(p < 1.f)) return -1;
  const int v = static_cast<int>(std::floor(static_cast<double>(p) * 256.0 + 0.5));
  return v >= 256 ? -1 : v;
}

fa_status check_common(int B, int H, int N, int d, float scale, float dropout_p, int Hkv) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * H * N;
  if (rows >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (p8_of(dropout_p) < 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// [B*H, N, d] bf16 tensor, boxes of 64 columns x 128 rows, 128-byte swizzle,
// out-of-range elements read as zero.
bool encode_map(CUtensorMap* m, const void* base, int BH, int N, int d) {
  EncodeTiledFn enc = encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t elem[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [outer, rows, inner] tensor of bytes (e4m3 codes) with rows of `inner`
// bytes spaced `row_stride` bytes apart: 128-byte x 128-row boxes, 128-byte
// swizzle, out-of-range elements read as zero.
bool encode_map_u8(CUtensorMap* m, const void* base, int outer, int rows, int inner,
                   int row_stride) {
  EncodeTiledFn enc = encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_stride),
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(row_stride)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t elem[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
             elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

fa::MaskParams make_mask(int B, int H, int Hkv, int N, int causal, const uint8_t* bm,
                         const int32_t* sl, int wl = -1, int wr = -1) {
  fa::MaskParams m;
  m.B = B;
  m.H = H;
  m.Hkv = Hkv;
  m.N = N;
  m.nb = (N + fa::kTile - 1) / fa::kTile;
  m.causal = causal ? 1 : 0;
  m.wl = wl;
  m.wr = wr;
  m.block_mask = bm;
  m.seqlens_k = sl;
  return m;
}

fa::DropParams make_drop(float p, uint64_t seed, uint64_t offset) {
  fa::DropParams d;
  d.p8 = p8_of(p);
  d.keep_scale = static_cast<float>(1.0 / (1.0 - d.p8 / 256.0));
  d.seed_lo = static_cast<uint32_t>(seed);
  d.seed_hi = static_cast<uint32_t>(seed >> 32);
  d.off_lo = static_cast<uint32_t>(offset);
  d.off_hi = static_cast<uint32_t>(offset >> 32);
  // Philox4x32 key schedule (Salmon et al., SC'11): the key grows by the two
  // Weyl constants every round.
  for (int r = 0; r < 10; ++r) {
    d.rk_lo[r] = d.seed_lo + static_cast<uint32_t>(r) * 0x9E3779B9u;
    d.rk_hi[r] = d.seed_hi + static_cast<uint32_t>(r) * 0xBB67AE85u;
  }
  return d;
}

// Launch kinds the stall hook (fa_test_inject_stall) can target.
enum StallTarget { kStallNone = 0, kStallForward = 1, kStallDkdv = 2, kStallDq = 3 };

// 1 if the stall hook is armed for `target` (and then disarm it), else 0.
int take_stall(StallTarget target) {
  if (target == kStallNone) return 0;
  int expected = static_cast<int>(target);
  return g_inject_stall.compare_exchange_strong(expected, 0) ? 1 : 0;
}

fa::SyncParams make_sync(const DeviceInfo* di, StallTarget target) {
  fa::SyncParams s;
  s.status = di->status;
  s.timeout_ns = g_timeout_ns.load();
  s.inject_stall = take_stall(target);
  return s;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Backward workspace for fa_bwd_noalloc: room for D = rowsum(dO * O) of up to
// kNoAllocMaxRows query rows (B*H*N), 16 MiB. It is part of the library's
// device image, so every GPU that loads the library holds it until the
// process exits. In host code `g_noalloc_dsum` is only a host-side stand-in
// for the array; its device address comes from cudaGetSymbolAddress below.
constexpr size_t kNoAllocMaxRows = static_cast<size_t>(1) << 22;
__device__ __align__(256) float g_noalloc_dsum[kNoAllocMaxRows];
void* g_noalloc_addr[kMaxDevices] = {};
std::mutex g_noalloc_mutex;

}  // namespace

extern "C" {

static fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                          int H, int Hkv, int N, int d, float scale, int causal, int wl, int wr,
                          float dropout_p, uint64_t seed, uint64_t offset,
                          const uint8_t* block_mask, const int32_t* seqlens_k, void* stream) {
  fa_status st = check_common(B, H, N, d, scale, dropout_p, Hkv);
  if (st != FA_OK) return st;
  if (wl < -1 || wr < -1) return FA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FA_OK) return st;
  CUtensorMap tq, tk, tv;
  if (!encode_map(&tq, q, B * H, N, d) || !encode_map(&tk, k, B * Hkv, N, d) ||
      !encode_map(&tv, v, B * Hkv, N, d))
    return FA_ERR_CUDA;
  fa::FwdArgs a;
  a.mask = make_mask(B, H, Hkv, N, causal, block_mask, seqlens_k, wl, wr);
  a.drop = make_drop(dropout_p, seed, offset);
  a.sync = make_sync(di, kStallForward);
  a.scale_log2 = scale * fa::kLog2e;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  cudaError_t e = fa::launch_fwd(tq, tk, tv, a, d, a.drop.p8 > 0, di->num_sms,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, float dropout_p, uint64_t seed,
                 uint64_t offset, const uint8_t* block_mask, const int32_t* seqlens_k,
                 void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, H, N, d, scale, causal, -1, -1, dropout_p, seed, offset,
                  block_mask, seqlens_k, stream);
}

fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int H_kv, int N, int d, float scale, int causal, float dropout_p,
                     uint64_t seed, uint64_t offset, const uint8_t* block_mask,
                     const int32_t* seqlens_k, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, -1, -1, dropout_p, seed,
                  offset, block_mask, seqlens_k, stream);
}

fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int H_kv, int N, int d, float scale, int causal, int window_left,
                        int window_right, float dropout_p, uint64_t seed, uint64_t offset,
                        const uint8_t* block_mask, const int32_t* seqlens_k, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, window_left, window_right,
                  dropout_p, seed, offset, block_mask, seqlens_k, stream);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  (void)d;
  if (B < 1 || H < 1 || N < 1) return 0;
  return round256(static_cast<size_t>(B) * H * N * sizeof(float));
}

// Shared validation and set-up of the backward stages. `need` selects which
// pointers must be present: 1 = preprocess (o, dout), 2 = dK/dV, 4 = dQ.
static fa_status bwd_prepare(const void* q, const void* k, const void* v, const void* o,
                             const void* dout, const float* lse, void* dq, void* dk, void* dv,
                             int B, int H, int Hkv, int N, int d, float scale, int causal,
                             int wl, int wr, float dropout_p, uint64_t seed, uint64_t offset,
                             const uint8_t* block_mask, const int32_t* seqlens_k, void* workspace,
                             size_t workspace_bytes, int need, fa::BwdArgs* a, CUtensorMap* maps,
                             DeviceInfo** di) {
  fa_status st = check_common(B, H, N, d, scale, dropout_p, Hkv);
  if (st != FA_OK) return st;
  if (wl < -1 || wr < -1) return FA_ERR_INVALID_ARG;
  if (need & 1) {
    if (!o || !dout || !aligned16(o) || !aligned16(dout)) return FA_ERR_INVALID_ARG;
  }
  if (need & 6) {
    if (!q || !k || !v || !dout || !lse) return FA_ERR_INVALID_ARG;
    for (const void* p : {q, k, v, dout})
      if (!aligned16(p)) return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_INVALID_ARG;
  }
  if ((need & 2) && (!dk || !dv || !aligned16(dk) || !aligned16(dv))) return FA_ERR_INVALID_ARG;
  if ((need & 4) && (!dq || !aligned16(dq))) return FA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < fa_bwd_workspace_size(B, H, N, d) ||
      !aligned16(workspace))
    return FA_ERR_WORKSPACE;
  if ((st = device_info(di)) != FA_OK) return st;
  if (need & 6) {
    if (!encode_map(&maps[0], q, B * H, N, d) || !encode_map(&maps[1], k, B * Hkv, N, d) ||
        !encode_map(&maps[2], v, B * Hkv, N, d) || !encode_map(&maps[3], dout, B * H, N, d))
      return FA_ERR_CUDA;
  }
  a->mask = make_mask(B, H, Hkv, N, causal, block_mask, seqlens_k, wl, wr);
  a->drop = make_drop(dropout_p, seed, offset);
  a->sync = make_sync(*di, kStallNone);
  a->scale = scale;
  a->scale_log2 = scale * fa::kLog2e;
  a->o = static_cast<const __nv_bfloat16*>(o);
  a->dout = static_cast<const __nv_bfloat16*>(dout);
  a->lse = lse;
  a->dsum = static_cast<float*>(workspace);
  a->dq = static_cast<__nv_bfloat16*>(dq);
  a->dk = static_cast<__nv_bfloat16*>(dk);
  a->dv = static_cast<__nv_bfloat16*>(dv);
  return FA_OK;
}

static fa_status bwd_impl(const void* q, const void* k, const void* v, const void* o,
                          const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                          int H, int Hkv, int N, int d, float scale, int causal, int wl, int wr,
                          float dropout_p, uint64_t seed, uint64_t offset,
                          const uint8_t* block_mask, const int32_t* seqlens_k, void* workspace,
                          size_t workspace_bytes, void* stream) {
  fa::BwdArgs a;
  CUtensorMap m[4];
  DeviceInfo* di = nullptr;
  fa_status st = bwd_prepare(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, N, d, scale, causal,
                             wl, wr, dropout_p, seed, offset, block_mask, seqlens_k, workspace,
                             workspace_bytes, 7, &a, m, &di);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool drop = a.drop.p8 > 0;
  cudaError_t e = fa::launch_bwd_preprocess(a, d, di->num_sms, s);
  if (e == cudaSuccess) {
    a.sync.inject_stall = take_stall(kStallDkdv);
    e = fa::launch_bwd_dkdv(m[0], m[1], m[2], m[3], a, d, drop, di->num_sms, s);
  }
  if (e == cudaSuccess) {
    a.sync.inject_stall = take_stall(kStallDq);
    e = fa::launch_bwd_dq(m[0], m[1], m[2], m[3], a, d, drop, di->num_sms, s);
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, float dropout_p, uint64_t seed, uint64_t offset,
                 const uint8_t* block_mask, const int32_t* seqlens_k, void* workspace,
                 size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, H, N, d, scale, causal, -1, -1,
                  dropout_p, seed, offset, block_mask, seqlens_k, workspace, workspace_bytes,
                  stream);
}

fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int H_kv, int N,
                     int d, float scale, int causal, float dropout_p, uint64_t seed,
                     uint64_t offset, const uint8_t* block_mask, const int32_t* seqlens_k,
                     void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N, d, scale, causal, -1, -1,
                  dropout_p, seed, offset, block_mask, seqlens_k, workspace, workspace_bytes,
                  stream);
}

fa_status fa_bwd_window(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                        int H, int H_kv, int N, int d, float scale, int causal, int window_left,
                        int window_right, float dropout_p, uint64_t seed, uint64_t offset,
                        const uint8_t* block_mask, const int32_t* seqlens_k, void* workspace,
                        size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N, d, scale, causal, window_left,
                  window_right, dropout_p, seed, offset, block_mask, seqlens_k, workspace,
                  workspace_bytes, stream);
}

fa_status fa_bwd_preprocess(const void* o, const void* dout, int B, int H, int N, int d,
                            void* workspace, size_t workspace_bytes, void* stream) {
  fa::BwdArgs a;
  CUtensorMap m[4];
  DeviceInfo* di = nullptr;
  fa_status st = bwd_prepare(nullptr, nullptr, nullptr, o, dout, nullptr, nullptr, nullptr,
                             nullptr, B, H, H, N, d, 1.f, 0, -1, -1, 0.f, 0, 0, nullptr, nullptr,
                             workspace, workspace_bytes, 1, &a, m, &di);
  if (st != FA_OK) return st;
  return fa::launch_bwd_preprocess(a, d, di->num_sms, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dout,
                      const float* lse, void* dk, void* dv, int B, int H, int N, int d,
                      float scale, int causal, float dropout_p, uint64_t seed, uint64_t offset,
                      const uint8_t* block_mask, const int32_t* seqlens_k, void* workspace,
                      size_t workspace_bytes, void* stream) {
  fa::BwdArgs a;
  CUtensorMap m[4];
  DeviceInfo* di = nullptr;
  fa_status st = bwd_prepare(q, k, v, nullptr, dout, lse, nullptr, dk, dv, B, H, H, N, d, scale,
                             causal, -1, -1, dropout_p, seed, offset, block_mask, seqlens_k,
                             workspace, workspace_bytes, 2, &a, m, &di);
  if (st != FA_OK) return st;
  a.sync.inject_stall = take_stall(kStallDkdv);
  return fa::launch_bwd_dkdv(m[0], m[1], m[2], m[3], a, d, a.drop.p8 > 0, di->num_sms,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status fa_bwd_dq(const void* q, const void* k, const void* v, const void* dout,
                    const float* lse, void* dq, int B, int H, int N, int d, float scale,
                    int causal, float dropout_p, uint64_t seed, uint64_t offset,
                    const uint8_t* block_mask, const int32_t* seqlens_k, void* workspace,
                    size_t workspace_bytes, void* stream) {
  fa::BwdArgs a;
  CUtensorMap m[4];
  DeviceInfo* di = nullptr;
  fa_status st = bwd_prepare(q, k, v, nullptr, dout, lse, dq, nullptr, nullptr, B, H, H, N, d,
                             scale, causal, -1, -1, dropout_p, seed, offset, block_mask,
                             seqlens_k, workspace, workspace_bytes, 4, &a, m, &di);
  if (st != FA_OK) return st;
  a.sync.inject_stall = take_stall(kStallDq);
  return fa::launch_bwd_dq(m[0], m[1], m[2], m[3], a, d, a.drop.p8 > 0, di->num_sms,
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, float scale, int causal, float dropout_p,
                         uint64_t seed, uint64_t offset, const uint8_t* block_mask,
                         const int32_t* seqlens_k, void* stream) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(N) > kNoAllocMaxRows)
    return FA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  void* scratch = nullptr;
  {
    // First call on this device (with it current): look up the array's device address.
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_addr[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_dsum) != cudaSuccess || p == nullptr)
        return FA_ERR_CUDA;
      g_noalloc_addr[dev] = p;
    }
    scratch = g_noalloc_addr[dev];
  }
  // D is written in full by the first backward kernel before it is read, so
  // the array's contents from an earlier call never matter and nothing is cleared.
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, dropout_p, seed,
                offset, block_mask, seqlens_k, scratch, kNoAllocMaxRows * sizeof(float), stream);
}

// Work split of fa_decode: the (K/V head, key tile) pairs, B * H_kv * n_t of
// them, cut into equal runs of per_cta pairs, one run per CTA; seg_max bounds
// the number of runs that cut one K/V head (1: no head is cut, no combine).
struct DecodePlan {
  int n_t, per_cta, grid, seg_max;
};

static fa_status decode_plan(int B, int H, int Hkv, int Nq, int Nk, int d, int num_ctas,
                             DecodePlan* p) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || num_ctas < 0) return FA_ERR_INVALID_ARG;
  if (Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * Nq >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(H / Hkv) * Nq > fa::kTile) return FA_ERR_UNSUPPORTED;
  p->n_t = (Nk + fa::kTile - 1) / fa::kTile;
  const long long total = static_cast<long long>(B) * Hkv * p->n_t;
  if (total >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  long long ctas = num_ctas;
  long long per = 0;
  if (ctas == 0) {
    DeviceInfo* di = nullptr;
    const fa_status st = device_info(&di);
    if (st != FA_OK) return st;
    ctas = di->num_sms;
    // Whole K/V heads per CTA when that still keeps enough SMs streaming to
    // saturate HBM (measured: 4/5 of them at d = 128, where one CTA streams
    // about 54 GB/s; all but 1/20 at d = 64, where a CTA is slower than its
    // share of HBM): no head is cut, so there are no partial results to write
    // and no combine launch. Otherwise equal runs over all SMs, cutting heads.
    const long long heads = static_cast<long long>(B) * Hkv;
    const long long k = (heads + ctas - 1) / ctas;  // heads per CTA
    const long long busy = (heads + k - 1) / k;      // CTAs that get a head
    if (d == 128 ? busy * 5 >= ctas * 4 : busy * 20 >= ctas * 19) per = k * p->n_t;
  }
  if (ctas > total) ctas = total;
  if (per == 0) per = (total + ctas - 1) / ctas;
  p->per_cta = static_cast<int>(per);
  p->grid = static_cast<int>((total + per - 1) / per);
  if (per % p->n_t == 0) {
    p->seg_max = 1;  // every run holds whole heads
  } else {
    const int bound = (p->n_t - 1) / p->per_cta + 2;
    p->seg_max = bound < p->grid ? bound : p->grid;
  }
  return FA_OK;
}

static size_t decode_ws_bytes(int B, int H, int Nq, int d, const DecodePlan& p) {
  if (p.seg_max <= 1) return 0;
  const size_t slots = static_cast<size_t>(B) * H * Nq * p.seg_max;
  return round256(slots * d * sizeof(float)) + round256(slots * sizeof(float));
}

size_t fa_decode_workspace_size(int B, int H, int H_kv, int Nq, int Nk, int d, int num_ctas) {
  DecodePlan p;
  if (decode_plan(B, H, H_kv, Nq, Nk, d, num_ctas, &p) != FA_OK) return 0;
  return decode_ws_bytes(B, H, Nq, d, p);
}

fa_status fa_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                    int B, int H, int H_kv, int Nq, int Nk, int d, float scale, int causal,
                    int window_left, const int32_t* seqlens_k, int num_ctas, void* workspace,
                    size_t workspace_bytes, void* stream) {
  DecodePlan p;
  fa_status st = decode_plan(B, H, H_kv, Nq, Nk, d, num_ctas, &p);
  if (st != FA_OK) return st;
  if (window_left < -1) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
    return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seqlens_k) & 3u) != 0) return FA_ERR_INVALID_ARG;
  const size_t ws = decode_ws_bytes(B, H, Nq, d, p);
  if (ws > 0 && (workspace == nullptr || workspace_bytes < ws || !aligned16(workspace)))
    return FA_ERR_WORKSPACE;
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FA_OK) return st;
  CUtensorMap tq, tk, tv;
  if (!encode_map(&tq, q, 1, B * H * Nq, d) || !encode_map(&tk, k_cache, B * H_kv, Nk, d) ||
      !encode_map(&tv, v_cache, B * H_kv, Nk, d))
    return FA_ERR_CUDA;
  fa::DecodeArgs a;
  a.B = B;
  a.H = H;
  a.Hkv = H_kv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.causal = causal ? 1 : 0;
  a.wl = window_left;
  a.seqlens_k = seqlens_k;
  a.n_t = p.n_t;
  a.per_cta = p.per_cta;
  a.seg_max = p.seg_max;
  a.scale_log2 = scale * fa::kLog2e;
  a.sync = make_sync(di, kStallForward);
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  const size_t slots = static_cast<size_t>(B) * H * Nq * p.seg_max;
  a.o_part = ws > 0 ? static_cast<float*>(workspace) : nullptr;
  a.lse_part = ws > 0 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                 round256(slots * d * sizeof(float)))
                      : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_decode(tq, tk, tv, a, d, p.grid, s);
  if (e == cudaSuccess && p.seg_max > 1) e = fa::launch_decode_combine(a, d, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_fp8_workspace_size(int B, int H, int d) {
  // B*H amaxes of Q, and of K plus 128 columns of V per K/V head: at most 130 B*H
  if (B < 1 || H < 1 || d != 128) return 0;
  return round256(static_cast<size_t>(B) * H * (2 + 128) * sizeof(unsigned int));
}

int fa_fp8_vt_stride(int N) { return N < 1 ? 0 : (N + 15) / 16 * 16; }

fa_status fa_fp8_quantize_gqa(const void* q, const void* k, const void* v, const float* signs,
                              int B, int H, int Hkv, int N, int d, void* q8, void* k8, void* vt8,
                              float* s_q, float* s_k, float* s_v, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (B < 1 || H < 1 || N < 1 || Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * N >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, v, q8, k8, vt8, s_q, s_k, s_v};  // signs may be null
  for (const void* p : ptrs)
    if (p == nullptr) return FA_ERR_INVALID_ARG;
  const void* tensors[] = {q, k, v, q8, k8, vt8};
  for (const void* p : tensors)
    if (!aligned16(p)) return FA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < fa_fp8_workspace_size(B, H, d) ||
      !aligned16(workspace))
    return FA_ERR_WORKSPACE;
  DeviceInfo* di = nullptr;
  fa_status st = device_info(&di);
  if (st != FA_OK) return st;
  fa::Fp8QuantArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.signs = signs;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.N = N;
  a.Np = fa_fp8_vt_stride(N);
  a.amax = static_cast<unsigned int*>(workspace);
  a.q8 = static_cast<uint8_t*>(q8);
  a.k8 = static_cast<uint8_t*>(k8);
  a.vt8 = static_cast<uint8_t*>(vt8);
  a.s_q = s_q;
  a.s_k = s_k;
  a.s_v = s_v;
  return fa::launch_fp8_quantize(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status fa_fwd_fp8_gqa(const void* q8, const void* k8, const void* vt8, const float* s_q,
                         const float* s_k, const float* s_v, void* o, float* lse, int B, int H,
                         int Hkv, int N, int d, float scale, int causal, const int32_t* seqlens_k,
                         void* stream) {
  fa_status st = check_common(B, H, N, d, scale, 0.f, Hkv);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (!q8 || !k8 || !vt8 || !s_q || !s_k || !s_v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o))
    return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FA_OK) return st;
  const int Np = fa_fp8_vt_stride(N);
  CUtensorMap tq, tk, tv;
  if (!encode_map_u8(&tq, q8, B * H, N, 128, 128) ||
      !encode_map_u8(&tk, k8, B * Hkv, N, 128, 128) ||
      !encode_map_u8(&tv, vt8, B * Hkv, 128, Np, Np))
    return FA_ERR_CUDA;
  fa::Fp8FwdArgs a;
  a.mask = make_mask(B, H, Hkv, N, causal, nullptr, seqlens_k);
  a.sync = make_sync(di, kStallForward);
  a.scale_log2 = scale * fa::kLog2e;
  a.s_q = s_q;
  a.s_k = s_k;
  a.s_v = s_v;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  return fa::launch_fwd_fp8(tq, tk, tv, a, di->num_sms, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status fa_fp8_quantize(const void* q, const void* k, const void* v, const float* signs, int B,
                          int H, int N, int d, void* q8, void* k8, void* vt8, float* s_q,
                          float* s_k, float* s_v, void* workspace, size_t workspace_bytes,
                          void* stream) {
  return fa_fp8_quantize_gqa(q, k, v, signs, B, H, H, N, d, q8, k8, vt8, s_q, s_k, s_v, workspace,
                             workspace_bytes, stream);
}

fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* s_q,
                     const float* s_k, const float* s_v, void* o, float* lse, int B, int H, int N,
                     int d, float scale, int causal, const int32_t* seqlens_k, void* stream) {
  return fa_fwd_fp8_gqa(q8, k8, vt8, s_q, s_k, s_v, o, lse, B, H, H, N, d, scale, causal,
                        seqlens_k, stream);
}

int fa_dropout_p8(float dropout_p) { return p8_of(dropout_p); }

fa_status fa_debug_dropout_keep(uint8_t* keep, int B, int H, int N, float dropout_p,
                                uint64_t seed, uint64_t offset, void* stream) {
  if (keep == nullptr || B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * N >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (p8_of(dropout_p) < 0) return FA_ERR_INVALID_ARG;
  DeviceInfo* di = nullptr;
  fa_status st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = fa::launch_debug_dropout(keep, B, H, N, make_drop(dropout_p, seed, offset),
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_debug_philox(const uint32_t* counters, uint32_t* out, int n, uint32_t key0,
                          uint32_t key1, void* stream) {
  if (counters == nullptr || out == nullptr || n < 0) return FA_ERR_INVALID_ARG;
  if (!aligned16(counters) || !aligned16(out)) return FA_ERR_INVALID_ARG;
  if (n == 0) return FA_OK;
  DeviceInfo* di = nullptr;
  fa_status st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e =
      fa::launch_debug_philox(counters, out, n, key0, key1, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_butterfly_mask(uint8_t* mask_host, int nb) {
  if (mask_host == nullptr || nb < 1 || nb > 65536) return FA_ERR_INVALID_ARG;
  // Partner of block r at stride 2^k is r XOR 2^k; the diagonal is stride 0.
  for (int r = 0; r < nb; ++r) {
    for (int c = 0; c < nb; ++c) {
      const unsigned x = static_cast<unsigned>(r ^ c);
      mask_host[static_cast<size_t>(r) * nb + c] =
          static_cast<uint8_t>(x == 0u || (x & (x - 1u)) == 0u);
    }
  }
  return FA_OK;
}

fa_status fa_device_status(void* stream, int clear) {
  DeviceInfo* di = nullptr;
  fa_status st = device_info(&di);
  if (st != FA_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, di->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_CUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpy(di->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  return static_cast<fa_status>(v);
}

void fa_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }

void fa_test_inject_stall(int mode) {
  g_inject_stall.store(mode >= kStallForward && mode <= kStallDq ? mode : kStallNone);
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension or device";
    case FA_ERR_CUDA: return "CUDA call failed";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
