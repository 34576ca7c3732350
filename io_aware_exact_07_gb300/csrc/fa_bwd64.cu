// Backward kernels for head dimension 64 (the same mathematics as fa_bwd.cu;
// FlashAttention deep-read report, sections 2.5 and 3.3).
//
// At d = 64 tensor memory has room for separate bf16 buffers for the operands
// that the compute warps produce (P^T and dS^T in the key-tile kernel, dS in
// the query-tile kernel), so the next S / dP can be computed as soon as the
// compute warps have *read* the current one instead of after it was consumed.
// Two issuing warps feed the tensor core: one for the shared-memory x
// shared-memory products (S, dP), one for the products that read the compute
// warps' output from tensor memory (dV, dK, dQ); each waits only on its own
// dependencies and tracks its own MMAs with its own commits. Sixteen compute
// warps (four warpgroups, 32 of the 128 columns each) hide the latency of the
// element-wise work.
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

namespace {

constexpr int kD = 64;
constexpr int kComputeWarps = 16;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kProdWarp = 16;
constexpr int kIssueAWarp = 17;  // S^T / dP^T (dK,dV kernel) or S / dP (dQ kernel)
constexpr int kIssueBWarp = 18;  // dV, dK (dK,dV kernel) or dQ (dQ kernel)
constexpr int kThreads = 19 * 32;
constexpr int kTileBytes = kTile * kD * 2;  // 16 KB
constexpr uint64_t kTileDesc = static_cast<uint64_t>(kTileBytes >> 4);
constexpr uint32_t kIdSS = idesc_bf16_f32(128, 128, 0, 0);  // both operands K-major
constexpr uint32_t kIdTS = idesc_bf16_f32(128, kD, 0, 1);   // B operand MN-major

__device__ __forceinline__ float lse2_at(const float* lse, long long idx, bool in_range) {
  if (!in_range) return INFINITY;
  const float l = lse[idx];
  return (l == -INFINITY) ? INFINITY : l * kLog2e;
}

// S (M=128, N=128, K=64) from two K-major shared-memory tiles.
__device__ __forceinline__ void mma_ss_tile(uint32_t d_tmem, uint64_t da, uint64_t db) {
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
    mma_ss(d_tmem, da + off, db + off, kIdSS, kk > 0 ? 1u : 0u);
  }
}
// acc (M=128, N=64) += A[tmem, bf16, 128 x 128] * B[smem, 128 x 64, MN-major].
__device__ __forceinline__ void mma_ts_tile(uint32_t d_tmem, uint32_t a_tmem, uint64_t db,
                                            bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts(d_tmem, a_tmem + kk * 8, db + static_cast<uint64_t>((kk * 2048) >> 4), kIdTS,
           (accumulate || kk > 0) ? 1u : 0u);
}

// ======================================================================== dK, dV
// Tensor memory: dV [0,64), dK [64,128), S^T [128,256), dP^T [256,384),
// P^T bf16 [384,448), dS^T bf16 [448,512).
struct DkdvL {
  static constexpr int kStages = 3;
  static constexpr int kKVOff = 0;                                   // 2 x (K, V)
  static constexpr int kQOff = 4 * kTileBytes;
  static constexpr int kDOOff = kQOff + kStages * kTileBytes;
  static constexpr int kLseOff = kDOOff + kStages * kTileBytes;      // kStages x 128 fp32
  static constexpr int kDsumOff = kLseOff + kStages * 512;
  static constexpr int kDropOff = kDsumOff + kStages * 512;          // 16 warps x 1 KB
  static constexpr int kBarOff = kDropOff + kComputeWarps * 1024;
  static constexpr int kNumBars = 4 + 2 * kStages + 12;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;
  static constexpr uint32_t kColDV = 0, kColDK = 64, kColSt = 128, kColDPt = 256, kColP = 384,
                            kColDS = 448;
};

struct DkdvBars {
  uint32_t kv_full[2], kv_empty[2], q_full[3], q_empty[3];
  uint32_t st_full, st_free, dpt_full, dpt_free, p_ready, p_done, ds_ready, ds_done;
  uint32_t acc_full, acc_free, drain_a, drain_b;
};

template <bool DROPOUT>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv64_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do, const BwdArgs args) {
  using L = DkdvL;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const MaskParams& mk = args.mask;
  const int N = mk.N;
  const int n_t = (N + kTile - 1) / kTile;
  const int n_units = mk.B * mk.H * n_t;

  uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff + 8);
  float* lse_s = reinterpret_cast<float*>(smem + L::kLseOff);
  float* dsum_s = reinterpret_cast<float*>(smem + L::kDsumOff);

  DkdvBars bars;
  {
    int i = 0;
    auto nb = [&]() { return smem_u32(&bar_mem[i++]); };
    for (int b = 0; b < 2; ++b) bars.kv_full[b] = nb();
    for (int b = 0; b < 2; ++b) bars.kv_empty[b] = nb();
    for (int s = 0; s < L::kStages; ++s) bars.q_full[s] = nb();
    for (int s = 0; s < L::kStages; ++s) bars.q_empty[s] = nb();
    bars.st_full = nb();
    bars.st_free = nb();
    bars.dpt_full = nb();
    bars.dpt_free = nb();
    bars.p_ready = nb();
    bars.p_done = nb();
    bars.ds_ready = nb();
    bars.ds_done = nb();
    bars.acc_full = nb();
    bars.acc_free = nb();
    bars.drain_a = nb();
    bars.drain_b = nb();
  }
  if (tid == 0) {
    *abort_flag = 0;
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.kv_full[b], 1);
      mbar_init(bars.kv_empty[b], 1);
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bars.q_full[s], 32);
      mbar_init(bars.q_empty[s], 2 + kComputeWarps);  // both issuers + every compute warp
    }
    mbar_init(bars.st_full, 1);
    mbar_init(bars.st_free, kComputeThreads);
    mbar_init(bars.dpt_full, 1);
    mbar_init(bars.dpt_free, kComputeThreads);
    mbar_init(bars.p_ready, kComputeThreads);
    mbar_init(bars.p_done, 1);
    mbar_init(bars.ds_ready, kComputeThreads);
    mbar_init(bars.ds_done, 1);
    mbar_init(bars.acc_full, 1);
    mbar_init(bars.acc_free, kComputeThreads);
    mbar_init(bars.drain_a, 1);
    mbar_init(bars.drain_b, 1);
    fence_mbar_init();
  }
  if (warp == kIssueAWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t tmo = args.sync.timeout_ns;
  auto fail = [&]() {
    *abort_flag = 1;
    record_error(args.sync.status, kStatusTimeout);
  };
  const uint32_t sKV = smem_u32(smem + L::kKVOff);
  const uint32_t sQ = smem_u32(smem + L::kQOff);
  const uint32_t sDO = smem_u32(smem + L::kDOOff);

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0, q_arms = 0, kv_arms[2] = {0, 0};
    bool ok = true;
    int unit_count = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_count) {
      const int bh = u / n_t, kt = u % n_t;
      const int kv_len = kv_len_of(mk, bh / mk.H);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      const int kb = unit_count & 1;
      const int kuse = unit_count >> 1;
      if (kuse > 0 && !mbar_wait_warp(bars.kv_empty[kb], (kuse - 1) & 1, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      if (lane == 0) {
        mbar_expect_tx(bars.kv_full[kb], 2 * kTileBytes);
        tma_load_3d(sKV + (2 * kb) * kTileBytes, &tm_k, 0, kt * kTile, bh, bars.kv_full[kb]);
        tma_load_3d(sKV + (2 * kb + 1) * kTileBytes, &tm_v, 0, kt * kTile, bh, bars.kv_full[kb]);
      }
      ++kv_arms[kb];
      for (int chunk = 0; chunk * 32 < n_t && ok; ++chunk) {
        uint32_t bits = warp_valid_bits_t(mk, kt, chunk, n_t, n_kv);
        while (bits != 0u) {
          const int qt = chunk * 32 + (__ffs(bits) - 1);
          bits &= bits - 1;
          const int s = it % L::kStages;
          const uint32_t ph = (it / L::kStages) & 1u;
          if (!mbar_wait_warp(bars.q_empty[s], ph ^ 1u, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          float4 l4, d4;
          float* lp = &l4.x;
          float* dp = &d4.x;
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int row = qt * kTile + 4 * lane + r;
            const bool in = row < N;
            const long long idx = static_cast<long long>(bh) * N + row;
            lp[r] = lse2_at(args.lse, idx, in);
            dp[r] = in ? args.dsum[idx] : 0.f;
          }
          reinterpret_cast<float4*>(lse_s + s * 128)[lane] = l4;
          reinterpret_cast<float4*>(dsum_s + s * 128)[lane] = d4;
          if (lane == 0) {
            mbar_expect_tx(bars.q_full[s], 2 * kTileBytes);
            tma_load_3d(sQ + s * kTileBytes, &tm_q, 0, qt * kTile, bh, bars.q_full[s]);
            tma_load_3d(sDO + s * kTileBytes, &tm_do, 0, qt * kTile, bh, bars.q_full[s]);
          } else {
            mbar_arrive(bars.q_full[s]);
          }
          ++q_arms;
          ++it;
        }
      }
    }
    for (int b = 0; b < 2; ++b)
      if (kv_arms[b]) mbar_wait_warp(bars.kv_full[b], (kv_arms[b] - 1) & 1, tmo, nullptr);
#pragma unroll
    for (int s = 0; s < L::kStages; ++s)
      if (q_arms > static_cast<uint32_t>(s))
        mbar_wait_warp(bars.q_full[s], ((q_arms - 1 - s) / L::kStages) & 1, tmo, nullptr);
  } else if (warp == kIssueAWarp) {
    // ------------------------------------------------------------ S^T, dP^T issuer
    const bool leader = lane == 0;
    uint32_t it = 0, gt = 0, stf = 0, dpf = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_count) {
      const int bh = u / n_t, kt = u % n_t;
      const int kv_len = kv_len_of(mk, bh / mk.H);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      const int kb = unit_count & 1;
      (void)bh;
      if (leader && !mbar_wait(bars.kv_full[kb], (unit_count >> 1) & 1, tmo, abort_flag)) {
        fail();
        ok = false;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      const uint64_t dK = sdesc_sw128(sKV + (2 * kb) * kTileBytes, 16, 1024);
      const uint64_t dV = sdesc_sw128(sKV + (2 * kb + 1) * kTileBytes, 16, 1024);
      for (int chunk = 0; chunk * 32 < n_t && ok; ++chunk) {
        const uint32_t vbits = warp_valid_bits_t(mk, kt, chunk, n_t, n_kv);
        if (leader) {
          for (uint32_t bits = vbits; bits != 0u && ok; bits &= bits - 1) {
            const int s = it % L::kStages;
            const uint32_t ph = (it / L::kStages) & 1u;
            if (!mbar_wait(bars.q_full[s], ph, tmo, abort_flag) ||
                (gt > 0 && !mbar_wait(bars.st_free, stf++ & 1, tmo, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_ss_tile(tmem + L::kColSt, dK, sdesc_sw128(sQ + s * kTileBytes, 16, 1024));
            mma_commit(bars.st_full);
            if (gt > 0 && !mbar_wait(bars.dpt_free, dpf++ & 1, tmo, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_ss_tile(tmem + L::kColDPt, dV, sdesc_sw128(sDO + s * kTileBytes, 16, 1024));
            mma_commit(bars.dpt_full);
            mma_commit(bars.q_empty[s]);
            ++gt;
            ++it;
          }
          if (!ok) fail();
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (leader && ok) mma_commit(bars.kv_empty[kb]);
    }
    if (leader) {
      mma_commit(bars.drain_a);
      mbar_wait(bars.drain_a, 0, tmo, nullptr);
    }
    __syncwarp();
  } else if (warp == kIssueBWarp) {
    // ------------------------------------------------------------ dV, dK issuer
    const bool leader = lane == 0;
    uint32_t it = 0, prc = 0, dsc = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_count) {
      const int bh = u / n_t, kt = u % n_t;
      const int kv_len = kv_len_of(mk, bh / mk.H);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      (void)bh;
      bool first = true;
      for (int chunk = 0; chunk * 32 < n_t && ok; ++chunk) {
        const uint32_t vbits = warp_valid_bits_t(mk, kt, chunk, n_t, n_kv);
        if (leader) {
          for (uint32_t bits = vbits; bits != 0u && ok; bits &= bits - 1) {
            const int s = it % L::kStages;
            if (!mbar_wait(bars.p_ready, prc++ & 1, tmo, abort_flag) ||
                (first && unit_count > 0 &&
                 !mbar_wait(bars.acc_free, (unit_count - 1) & 1, tmo, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_ts_tile(tmem + L::kColDV, tmem + L::kColP,
                        sdesc_sw128(sDO + s * kTileBytes, 16384, 1024), !first);
            mma_commit(bars.p_done);
            if (!mbar_wait(bars.ds_ready, dsc++ & 1, tmo, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_ts_tile(tmem + L::kColDK, tmem + L::kColDS,
                        sdesc_sw128(sQ + s * kTileBytes, 16384, 1024), !first);
            mma_commit(bars.ds_done);
            mma_commit(bars.q_empty[s]);
            first = false;
            ++it;
          }
          if (!ok) fail();
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (leader && ok) {
        if (first && unit_count > 0 &&
            !mbar_wait(bars.acc_free, (unit_count - 1) & 1, tmo, abort_flag)) {
          ok = false;
          fail();
        } else {
          mma_commit(bars.acc_full);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (leader) {
      mma_commit(bars.drain_b);
      mbar_wait(bars.drain_b, 0, tmo, nullptr);
    }
    __syncwarp();
  } else if (warp < kComputeWarps) {
    // ------------------------------------------------------------ compute
    // Warpgroup wg owns query columns [32 wg, 32 wg + 32) of every tile; the
    // thread owns one key row.
    const int wg = warp >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tSt = tmem + lane_base + L::kColSt + 32 * wg;
    const uint32_t tDPt = tmem + lane_base + L::kColDPt + 32 * wg;
    const uint32_t tP = tmem + lane_base + L::kColP + 16 * wg;
    const uint32_t tDS = tmem + lane_base + L::kColDS + 16 * wg;
    const float c_log2 = args.scale_log2;
    uint32_t* drop_scratch = reinterpret_cast<uint32_t*>(smem + L::kDropOff + warp * 1024);
    uint32_t it = 0, gt = 0, stc = 0, dpc = 0, pdc = 0, dsc = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_count) {
      const int bh = u / n_t, kt = u % n_t;
      const int kv_len = kv_len_of(mk, bh / mk.H);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      const int key = kt * kTile + r;
      int n_done = 0;
      for (int chunk = 0; chunk * 32 < n_t && ok; ++chunk) {
        uint32_t bits = warp_valid_bits_t(mk, kt, chunk, n_t, n_kv);
        while (bits != 0u && ok) {
          const int qt = chunk * 32 + (__ffs(bits) - 1);
          bits &= bits - 1;
          const int s = it % L::kStages;
          const float* lse_t = lse_s + s * 128 + 32 * wg;
          const float* dsum_t = dsum_s + s * 128 + 32 * wg;
          const int q0 = qt * kTile + 32 * wg;  // first query column of this warpgroup
          uint32_t zb = 0xFFFFFFFFu;            // dropout keep bit per query column
          if constexpr (DROPOUT) {
            // The warp's 32 keys are two 16-key Philox groups; for each of the 32
            // queries both groups are generated (two blocks per lane) and each
            // lane then reads its own key's byte.
            const uint32_t kgroup0 = static_cast<uint32_t>(kt * kTile + quad * 32) >> 4;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const int idx = lane + 32 * m;
              const int c = idx >> 1, gs = idx & 1;
              const uint32_t rowg = static_cast<uint32_t>(bh) * static_cast<uint32_t>(N) +
                                    static_cast<uint32_t>(q0 + c);
              reinterpret_cast<uint4*>(drop_scratch)[c * 2 + gs] =
                  dropout_keep16(args.drop, rowg, kgroup0 + gs);
            }
            __syncwarp();
            zb = 0u;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const uint32_t w = drop_scratch[(c * 2 + (lane >> 4)) * 4 + ((lane & 15) >> 2)];
              zb |= ((w >> (8 * (lane & 3))) & 1u) << c;  // bytes are 0x00 or 0xFF
            }
            __syncwarp();
          }
          // ---- P^T = exp2(S^T c - lse2) for 32 query columns
          if (!mbar_wait_warp(bars.st_full, stc++ & 1, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          float p[32];
          {
            uint32_t sr[32];
            tmem_ld32(tSt, sr);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(bars.st_free);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 l4 = reinterpret_cast<const float4*>(lse_t)[c4];
              p[4 * c4 + 0] = ex2_approx(fmaf(__uint_as_float(sr[4 * c4 + 0]), c_log2, -l4.x));
              p[4 * c4 + 1] = ex2_approx(fmaf(__uint_as_float(sr[4 * c4 + 1]), c_log2, -l4.y));
              p[4 * c4 + 2] = ex2_approx(fmaf(__uint_as_float(sr[4 * c4 + 2]), c_log2, -l4.z));
              p[4 * c4 + 3] = ex2_approx(fmaf(__uint_as_float(sr[4 * c4 + 3]), c_log2, -l4.w));
            }
          }
          if (tile_needs_element_mask(mk, qt, kt, kv_len)) {
            const bool key_ok = key < kv_len;
#pragma unroll
            for (int c = 0; c < 32; ++c)
              p[c] = (key_ok && (!mk.causal || key <= q0 + c)) ? p[c] : 0.f;
          }
          {
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float a0 = ((zb >> (2 * c)) & 1u) ? p[2 * c] : 0.f;
              const float a1 = ((zb >> (2 * c + 1)) & 1u) ? p[2 * c + 1] : 0.f;
              pk[c] = pack_bf16x2(a0, a1);
            }
            if (gt > 0) {  // the previous dV has finished reading the P^T buffer
              if (!mbar_wait_warp(bars.p_done, pdc++ & 1, tmo, abort_flag)) {
                fail();
                ok = false;
                break;
              }
              tc_fence_after();
            }
            tmem_st16(tP, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bars.p_ready);
          }
          // ---- dS^T = P^T (Z dP^T / (1 - p) - D)
          if (!mbar_wait_warp(bars.dpt_full, dpc++ & 1, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          {
            uint32_t dr[32];
            tmem_ld32(tDPt, dr);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(bars.dpt_free);
            uint32_t pk[16];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 d4 = reinterpret_cast<const float4*>(dsum_t)[c4];
              const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
              float ds[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int c = 4 * c4 + e;
                const float z = ((zb >> c) & 1u) ? args.drop.keep_scale : 0.f;
                ds[e] = p[c] * fmaf(z, __uint_as_float(dr[c]), -dv4[e]);
              }
              pk[2 * c4] = pack_bf16x2(ds[0], ds[1]);
              pk[2 * c4 + 1] = pack_bf16x2(ds[2], ds[3]);
            }
            if (gt > 0) {  // the previous dK has finished reading the dS^T buffer
              if (!mbar_wait_warp(bars.ds_done, dsc++ & 1, tmo, abort_flag)) {
                fail();
                ok = false;
                break;
              }
              tc_fence_after();
            }
            tmem_st16(tDS, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bars.ds_ready);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.q_empty[s]);  // lse / D of this stage no longer read
          ++n_done;
          ++gt;
          ++it;
        }
      }
      if (!ok) break;
      // ---- epilogue: dV (warpgroups 0, 1) and dK (2, 3), 32 columns each
      if (!mbar_wait_warp(bars.acc_full, unit_count & 1, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      tc_fence_after();
      const bool is_dv = wg < 2;
      const uint32_t tAcc = tmem + lane_base + (is_dv ? L::kColDV : L::kColDK) + 32 * (wg & 1);
      const float mult = is_dv ? args.drop.keep_scale : args.scale;
      __nv_bfloat16* dst = (is_dv ? args.dv : args.dk) +
                           (static_cast<size_t>(bh) * N + static_cast<size_t>(key)) * kD +
                           32 * (wg & 1);
      uint32_t v[32];
      if (n_done > 0) {
        tmem_ld32(tAcc, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = 0u;
      }
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        pk[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * mult, __uint_as_float(v[2 * k + 1]) * mult);
      if (key < N) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          d4[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      }
      tc_fence_before();
      mbar_arrive(bars.acc_free);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kIssueAWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ======================================================================== dQ
// One unit = one (b, h) head and one 128-row query tile; the loop runs over
// the key tiles it attends to. Tensor memory: S [0,128), dP [128,256),
// dQ [256,320), dS bf16 [320,384).
struct DqL {
  static constexpr int kKStages = 4;
  static constexpr int kVStages = 3;
  static constexpr int kQOff = 0;                                  // 2 x (Q, dO)
  static constexpr int kKOff = 4 * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
  static constexpr int kNumBars = 4 + 2 * kKStages + 2 * kVStages + 10;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 320;
};

struct DqBars {
  uint32_t qd_full[2], qd_empty[2], k_full[4], k_empty[4], v_full[3], v_empty[3];
  uint32_t s_full, s_free, dp_full, dp_free, ds_ready, ds_done, dq_full, dq_free;
  uint32_t drain_a, drain_b;
};

template <bool DROPOUT>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq64_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do, const BwdArgs args) {
  using L = DqL;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const MaskParams& mk = args.mask;
  const int N = mk.N;
  const int n_q = (N + kTile - 1) / kTile;
  const int n_units = mk.B * mk.H * n_q;

  uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff + 8);

  DqBars bars;
  {
    int i = 0;
    auto nb = [&]() { return smem_u32(&bar_mem[i++]); };
    for (int b = 0; b < 2; ++b) bars.qd_full[b] = nb();
    for (int b = 0; b < 2; ++b) bars.qd_empty[b] = nb();
    for (int s = 0; s < L::kKStages; ++s) bars.k_full[s] = nb();
    for (int s = 0; s < L::kKStages; ++s) bars.k_empty[s] = nb();
    for (int s = 0; s < L::kVStages; ++s) bars.v_full[s] = nb();
    for (int s = 0; s < L::kVStages; ++s) bars.v_empty[s] = nb();
    bars.s_full = nb();
    bars.s_free = nb();
    bars.dp_full = nb();
    bars.dp_free = nb();
    bars.ds_ready = nb();
    bars.ds_done = nb();
    bars.dq_full = nb();
    bars.dq_free = nb();
    bars.drain_a = nb();
    bars.drain_b = nb();
  }
  if (tid == 0) {
    *abort_flag = 0;
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.qd_full[b], 1);
      mbar_init(bars.qd_empty[b], 1);
    }
    for (int s = 0; s < L::kKStages; ++s) {
      mbar_init(bars.k_full[s], 1);
      mbar_init(bars.k_empty[s], 1);
    }
    for (int s = 0; s < L::kVStages; ++s) {
      mbar_init(bars.v_full[s], 1);
      mbar_init(bars.v_empty[s], 1);
    }
    mbar_init(bars.s_full, 1);
    mbar_init(bars.s_free, kComputeThreads);
    mbar_init(bars.dp_full, 1);
    mbar_init(bars.dp_free, kComputeThreads);
    mbar_init(bars.ds_ready, kComputeThreads);
    mbar_init(bars.ds_done, 1);
    mbar_init(bars.dq_full, 1);
    mbar_init(bars.dq_free, kComputeThreads);
    mbar_init(bars.drain_a, 1);
    mbar_init(bars.drain_b, 1);
    fence_mbar_init();
  }
  if (warp == kIssueAWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t tmo = args.sync.timeout_ns;
  auto fail = [&]() {
    *abort_flag = 1;
    record_error(args.sync.status, kStatusTimeout);
  };
  const uint32_t sQD = smem_u32(smem + L::kQOff);
  const uint32_t sK = smem_u32(smem + L::kKOff);
  const uint32_t sV = smem_u32(smem + L::kVOff);
  // Unit u: head-major; with a causal mask the longest query tiles of a head first.
  auto unit_coords = [&](int u, int& bh, int& qt) {
    bh = u / n_q;
    qt = u % n_q;
    if (mk.causal) qt = n_q - 1 - qt;
  };
  auto kv_limit = [&](int qt, int n_kv) {
    int jmax = n_kv;
    if (mk.causal && qt + 1 < jmax) jmax = qt + 1;
    return jmax;
  };

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0, k_arms = 0, v_arms = 0, qd_arms[2] = {0, 0};
    bool ok = true;
    int unit_count = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_count) {
      int bh, qt;
      unit_coords(u, bh, qt);
      const int kv_len = kv_len_of(mk, bh / mk.H);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      const int jmax = kv_limit(qt, n_kv);
      const int qb = unit_count & 1, use = unit_count >> 1;
      if (use > 0 && !mbar_wait_warp(bars.qd_empty[qb], (use - 1) & 1, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      if (lane == 0) {
        mbar_expect_tx(bars.qd_full[qb], 2 * kTileBytes);
        tma_load_3d(sQD + (2 * qb) * kTileBytes, &tm_q, 0, qt * kTile, bh, bars.qd_full[qb]);
        tma_load_3d(sQD + (2 * qb + 1) * kTileBytes, &tm_do, 0, qt * kTile, bh, bars.qd_full[qb]);
      }
      ++qd_arms[qb];
      for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
        uint32_t bits = warp_valid_bits(mk, qt, chunk, n_q, n_kv);
        while (bits != 0u) {
          const int j = chunk * 32 + (__ffs(bits) - 1);
          bits &= bits - 1;
          const int ks = it % L::kKStages, vs = it % L::kVStages;
          if (!mbar_wait_warp(bars.k_empty[ks], ((it / L::kKStages) & 1u) ^ 1u, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_expect_tx(bars.k_full[ks], kTileBytes);
            tma_load_3d(sK + ks * kTileBytes, &tm_k, 0, j * kTile, bh, bars.k_full[ks]);
          }
          ++k_arms;
          if (!mbar_wait_warp(bars.v_empty[vs], ((it / L::kVStages) & 1u) ^ 1u, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_expect_tx(bars.v_full[vs], kTileBytes);
            tma_load_3d(sV + vs * kTileBytes, &tm_v, 0, j * kTile, bh, bars.v_full[vs]);
          }
          ++v_arms;
          ++it;
        }
      }
    }
#pragma unroll
    for (int s = 0; s < L::kKStages; ++s)
      if (k_arms > static_cast<uint32_t>(s))
        mbar_wait_warp(bars.k_full[s], ((k_arms - 1 - s) / L::kKStages) & 1, tmo, nullptr);
#pragma unroll
    for (int s = 0; s < L::kVStages; ++s)
      if (v_arms > static_cast<uint32_t>(s))
        mbar_wait_warp(bars.v_full[s], ((v_arms - 1 - s) / L::kVStages) & 1, tmo, nullptr);
    for (int b = 0; b < 2; ++b)
      if (qd_arms[b]) mbar_wait_warp(bars.qd_full[b], (qd_arms[b] - 1) & 1, tmo, nullptr);
  } else if (warp == kIssueAWarp) {
    // ------------------------------------------------------------ S, dP issuer
    const bool leader = lane == 0;
    uint32_t it = 0, gt = 0, sfc = 0, dfc = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_count) {
      int bh, qt;
      unit_coords(u, bh, qt);
      const int kv_len = kv_len_of(mk, bh / mk.H);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      const int jmax = kv_limit(qt, n_kv);
      const int qb = unit_count & 1;
      if (leader && !mbar_wait(bars.qd_full[qb], (unit_count >> 1) & 1, tmo, abort_flag)) {
        fail();
        ok = false;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      const uint64_t dQ = sdesc_sw128(sQD + (2 * qb) * kTileBytes, 16, 1024);
      const uint64_t dDO = sdesc_sw128(sQD + (2 * qb + 1) * kTileBytes, 16, 1024);
      for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
        const uint32_t vbits = warp_valid_bits(mk, qt, chunk, n_q, n_kv);
        if (leader) {
          for (uint32_t bits = vbits; bits != 0u && ok; bits &= bits - 1) {
            const int ks = it % L::kKStages, vs = it % L::kVStages;
            if (!mbar_wait(bars.k_full[ks], (it / L::kKStages) & 1u, tmo, abort_flag) ||
                (gt > 0 && !mbar_wait(bars.s_free, sfc++ & 1, tmo, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_ss_tile(tmem + L::kColS, dQ, sdesc_sw128(sK + ks * kTileBytes, 16, 1024));
            mma_commit(bars.s_full);
            if (!mbar_wait(bars.v_full[vs], (it / L::kVStages) & 1u, tmo, abort_flag) ||
                (gt > 0 && !mbar_wait(bars.dp_free, dfc++ & 1, tmo, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_ss_tile(tmem + L::kColDP, dDO, sdesc_sw128(sV + vs * kTileBytes, 16, 1024));
            mma_commit(bars.dp_full);
            mma_commit(bars.v_empty[vs]);
            ++gt;
            ++it;
          }
          if (!ok) fail();
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (leader && ok) mma_commit(bars.qd_empty[qb]);
    }
    if (leader) {
      mma_commit(bars.drain_a);
      mbar_wait(bars.drain_a, 0, tmo, nullptr);
    }
    __syncwarp();
  } else if (warp == kIssueBWarp) {
    // ------------------------------------------------------------ dQ issuer
    const bool leader = lane == 0;
    uint32_t it = 0, dsc = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_count) {
      int bh, qt;
      unit_coords(u, bh, qt);
      const int kv_len = kv_len_of(mk, bh / mk.H);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      const int jmax = kv_limit(qt, n_kv);
      bool first = true;
      for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
        const uint32_t vbits = warp_valid_bits(mk, qt, chunk, n_q, n_kv);
        if (leader) {
          for (uint32_t bits = vbits; bits != 0u && ok; bits &= bits - 1) {
            const int ks = it % L::kKStages;
            if (!mbar_wait(bars.ds_ready, dsc++ & 1, tmo, abort_flag) ||
                !mbar_wait(bars.k_full[ks], (it / L::kKStages) & 1u, tmo, abort_flag) ||
                (first && unit_count > 0 &&
                 !mbar_wait(bars.dq_free, (unit_count - 1) & 1, tmo, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_ts_tile(tmem + L::kColDQ, tmem + L::kColDS,
                        sdesc_sw128(sK + ks * kTileBytes, 16384, 1024), !first);
            mma_commit(bars.ds_done);
            mma_commit(bars.k_empty[ks]);
            first = false;
            ++it;
          }
          if (!ok) fail();
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (leader && ok) {
        if (first && unit_count > 0 &&
            !mbar_wait(bars.dq_free, (unit_count - 1) & 1, tmo, abort_flag)) {
          ok = false;
          fail();
        } else {
          mma_commit(bars.dq_full);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (leader) {
      mma_commit(bars.drain_b);
      mbar_wait(bars.drain_b, 0, tmo, nullptr);
    }
    __syncwarp();
  } else if (warp < kComputeWarps) {
    // ------------------------------------------------------------ compute
    // Warpgroup wg owns key columns [32 wg, 32 wg + 32) of every tile; the
    // thread owns one query row.
    const int wg = warp >> 2;
    const int quad = warp & 3;
    const int t = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::kColS + 32 * wg;
    const uint32_t tDP = tmem + lane_base + L::kColDP + 32 * wg;
    const uint32_t tDS = tmem + lane_base + L::kColDS + 16 * wg;
    const uint32_t tDQ = tmem + lane_base + L::kColDQ + 16 * wg;
    const float c_log2 = args.scale_log2;
    uint32_t gt = 0, sc = 0, dc = 0, ddc = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_count) {
      int bh, qt;
      unit_coords(u, bh, qt);
      const int row = qt * kTile + t;
      const bool row_in = row < N;
      const long long ridx = static_cast<long long>(bh) * N + row;
      const float lse2 = lse2_at(args.lse, ridx, row_in);
      const float dsum = row_in ? args.dsum[ridx] : 0.f;
      const int kv_len = kv_len_of(mk, bh / mk.H);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      const int jmax = kv_limit(qt, n_kv);
      int n_done = 0;
      for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
        uint32_t bits = warp_valid_bits(mk, qt, chunk, n_q, n_kv);
        while (bits != 0u && ok) {
          const int j = chunk * 32 + (__ffs(bits) - 1);
          bits &= bits - 1;
          uint32_t zb = 0xFFFFFFFFu;  // dropout keep bit per key column
          if constexpr (DROPOUT) {
            zb = 0u;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              const uint4 kw = dropout_keep16(args.drop, static_cast<uint32_t>(ridx),
                                              static_cast<uint32_t>(j * 8 + 2 * wg + g));
              const uint32_t w4[4] = {kw.x, kw.y, kw.z, kw.w};
#pragma unroll
              for (int e = 0; e < 16; ++e) zb |= ((w4[e >> 2] >> (8 * (e & 3))) & 1u) << (16 * g + e);
            }
          }
          int lim = 128;  // keys [0, lim) of this tile are allowed for this row
          if (tile_needs_element_mask(mk, qt, j, kv_len)) {
            lim = kv_len - j * kTile;
            if (mk.causal) {
              const int lc = row - j * kTile + 1;
              lim = lc < lim ? lc : lim;
            }
          }
          const int lim_local = lim - 32 * wg;
          // ---- P = exp2(S c - lse2)
          if (!mbar_wait_warp(bars.s_full, sc++ & 1, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          float p[32];
          {
            uint32_t sr[32];
            tmem_ld32(tS, sr);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(bars.s_free);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float e = ex2_approx(fmaf(__uint_as_float(sr[c]), c_log2, -lse2));
              p[c] = (c < lim_local) ? e : 0.f;
            }
          }
          // ---- dS = P (Z dP / (1 - p) - D)
          if (!mbar_wait_warp(bars.dp_full, dc++ & 1, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t pk[16];
          {
            uint32_t dr[32];
            tmem_ld32(tDP, dr);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(bars.dp_free);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float z0 = ((zb >> (2 * c)) & 1u) ? args.drop.keep_scale : 0.f;
              const float z1 = ((zb >> (2 * c + 1)) & 1u) ? args.drop.keep_scale : 0.f;
              const float d0 = p[2 * c] * fmaf(z0, __uint_as_float(dr[2 * c]), -dsum);
              const float d1 = p[2 * c + 1] * fmaf(z1, __uint_as_float(dr[2 * c + 1]), -dsum);
              pk[c] = pack_bf16x2(d0, d1);
            }
          }
          if (gt > 0) {  // the previous dQ MMA has finished reading the dS buffer
            if (!mbar_wait_warp(bars.ds_done, ddc++ & 1, tmo, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            tc_fence_after();
          }
          tmem_st16(tDS, pk);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bars.ds_ready);
          ++n_done;
          ++gt;
        }
      }
      if (!ok) break;
      // ---- epilogue: dQ = scale * acc, 16 columns per warpgroup
      if (!mbar_wait_warp(bars.dq_full, unit_count & 1, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[16];
      if (n_done > 0) {
        tmem_ld16(tDQ, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = 0u;
      }
      uint32_t o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        o[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * args.scale,
                           __uint_as_float(v[2 * k + 1]) * args.scale);
      if (row_in) {
        uint4* d4 = reinterpret_cast<uint4*>(args.dq + static_cast<size_t>(ridx) * kD + 16 * wg);
        d4[0] = make_uint4(o[0], o[1], o[2], o[3]);
        d4[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
      tc_fence_before();
      mbar_arrive(bars.dq_free);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kIssueAWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <typename K>
cudaError_t set_smem64(K kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

cudaError_t launch_bwd_dkdv64(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const BwdArgs& a, bool dropout, int num_sms,
                              cudaStream_t stream) {
  const int n_t = (a.mask.N + kTile - 1) / kTile;
  const long long units = static_cast<long long>(a.mask.B) * a.mask.H * n_t;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  if (grid <= 0) return cudaSuccess;
  auto kern = dropout ? fa_bwd_dkdv64_kernel<true> : fa_bwd_dkdv64_kernel<false>;
  cudaError_t e = set_smem64(kern, DkdvL::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, DkdvL::kSmemBytes, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq64(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdArgs& a, bool dropout, int num_sms,
                            cudaStream_t stream) {
  const int n_q = (a.mask.N + kTile - 1) / kTile;
  const long long units = static_cast<long long>(a.mask.B) * a.mask.H * n_q;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  if (grid <= 0) return cudaSuccess;
  auto kern = dropout ? fa_bwd_dq64_kernel<true> : fa_bwd_dq64_kernel<false>;
  cudaError_t e = set_smem64(kern, DqL::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, DqL::kSmemBytes, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}

}  // namespace fa
