// Backward kernels (the mathematics of fa_bwd.cu; FlashAttention deep-read
// report, sections 2.5 and 3.3), built from three kinds of warps:
//   - two issuing warps feed the tensor core: "A" issues the products whose
//     operands are both in shared memory (S^T, dP^T in the key-tile kernel;
//     S, dP in the query-tile kernel), "B" the products that read the compute
//     warps' bf16 output from tensor memory (dV, dK; dQ). Each waits only on
//     its own dependencies and tracks its own MMAs with its own commits, so the
//     tensor core keeps receiving work while the other waits;
//   - sixteen compute warps (four warpgroups, 32 of the 128 columns each) do
//     the element-wise work, enough warps per scheduler to hide its latency;
//   - one producer warp streams tiles with TMA.
// Where tensor memory has room (the key-tile kernel at d = 64, the query-tile
// kernel at both head sizes) the bf16 operands produced by the compute warps
// get their own buffers, so the next S / dP is computed as soon as the current
// one has been *read*. In the key-tile kernel at d = 128 (dV, dK, S^T, dP^T
// fill all 512 columns) P^T and dS^T are written over S^T and dP^T, and the
// next S^T / dP^T waits until dV / dK have consumed them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

namespace {

constexpr int kComputeWarps = 16;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kProdWarp = 16;
constexpr int kIssueAWarp = 17;
constexpr int kIssueBWarp = 18;
// Warp 19 idles: it completes the fifth warpgroup, since registers move between
// whole warpgroups.
constexpr int kThreads = 20 * 32;
// Registers per thread: 96 at launch (five warps per sub-partition); the producer
// and issuer warpgroup gives most of its share to the compute warps, which keep
// the per-step P^T / dS^T values of 32 columns live.
constexpr int kRegsLaunch = 96;
constexpr int kRegsCompute = 104;
constexpr int kRegsAux = 56;
static_assert(kComputeThreads * kRegsCompute + (kThreads - kComputeThreads) * kRegsAux <=
                  kThreads * kRegsLaunch,
              "register reallocation exceeds the block's launch allocation");

template <int D>
struct TileT {
  static constexpr int kBytes = kTile * D * 2;
  static constexpr int kChunks = D / 64;  // 64-column (128-byte swizzle) chunks of 16 KB
};

// Barrier arrays are sized for the deepest ring of either head size.
constexpr int kMaxQStages = 4;  // dK/dV kernel: Q / dO ring
constexpr int kMaxKStages = 4;  // dQ kernel: K ring
constexpr int kMaxVStages = 3;  // dQ kernel: V ring

__device__ __forceinline__ float lse2_at(const float* lse, long long idx, bool in_range) {
  if (!in_range) return INFINITY;
  const float l = lse[idx];
  return (l == -INFINITY) ? INFINITY : l * kLog2e;
}

template <int D>
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap* map, int row, int bh,
                                         uint32_t bar) {
#pragma unroll
  for (int c = 0; c < TileT<D>::kChunks; ++c)
    tma_load_3d(dst + c * 16384, map, c * 64, row, bh, bar);
}

// D_tmem (M=128, N=128) = A * B^T over K = D, both K-major shared-memory tiles.
template <int D>
__device__ __forceinline__ void mma_ss_tile(uint32_t d_tmem, uint64_t da, uint64_t db) {
  constexpr uint32_t kId = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
    mma_ss(d_tmem, da + off, db + off, kId, kk > 0 ? 1u : 0u);
  }
}

// acc (M=128, N=D) += A[tmem, bf16, 128 x 128] * B[smem, 128 x D, MN-major].
// The 16-column K step kk of A sits at a_base + (kk / 2) * a_pair + (kk % 2) * 8
// (a_pair = 16: contiguous buffer; 32: pairs written over the fp32 columns
// each warpgroup read).
template <int D>
__device__ __forceinline__ void mma_ts_tile(uint32_t d_tmem, uint32_t a_base, uint32_t a_pair,
                                            uint64_t db, bool accumulate) {
  constexpr uint32_t kId = idesc_bf16_f32(128, D, 0, 1);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts(d_tmem, a_base + (kk >> 1) * a_pair + (kk & 1) * 8,
           db + static_cast<uint64_t>((kk * 2048) >> 4), kId, (accumulate || kk > 0) ? 1u : 0u);
}

// ======================================================================== dK, dV
template <int D>
struct DkdvL {
  static constexpr int T = TileT<D>::kBytes;
  static constexpr bool kSepBuf = (D == 64);       // separate P^T / dS^T buffers
  static constexpr int kKVBufs = (D == 64) ? 2 : 1;
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static_assert(kStages <= kMaxQStages, "Q / dO ring deeper than its barrier arrays");
  static constexpr int kKVOff = 0;                                   // kKVBufs x (K, V)
  static constexpr int kQOff = kKVBufs * 2 * T;
  static constexpr int kDOOff = kQOff + kStages * T;
  static constexpr int kLseOff = kDOOff + kStages * T;               // kStages x 128 fp32
  static constexpr int kDsumOff = kLseOff + kStages * 512;
  static constexpr int kDropOff = kDsumOff + kStages * 512;          // 16 warps x 1 KB
  static constexpr int kBarOff = kDropOff + kComputeWarps * 1024;
  static constexpr int kNumBars = 4 + 2 * kMaxQStages + 13;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;
  static constexpr uint32_t kColDV = 0, kColDK = D, kColSt = 2 * D, kColDPt = 2 * D + 128;
  static constexpr uint32_t kColP = kSepBuf ? 384u : kColSt;
  static constexpr uint32_t kColDS = kSepBuf ? 448u : kColDPt;
  static constexpr uint32_t kPair = kSepBuf ? 16u : 32u;  // A-operand pair stride (columns)
};

struct DkdvBars {
  BarRun kv_full, kv_empty, q_full, q_empty;
  uint32_t st_full, st_free, dpt_full, dpt_free, p_ready, p_done, ds_ready, ds_done;
  uint32_t acc_full, acc_free, drain_a, drain_b;
  uint32_t stall;  // test hook: never completed
};

template <int D, bool DROPOUT, bool GQA, bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_split_kernel(const __grid_constant__ CUtensorMap tm_q,
                             const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v,
                             const __grid_constant__ CUtensorMap tm_do, const BwdArgs args) {
  using L = DkdvL<D>;
  constexpr int T = L::T;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const MaskParams& mk = args.mask;
  const int N = mk.N;
  const int n_t = (N + kTile - 1) / kTile;
  const int n_units = mk.B * mk.Hkv * n_t;
  const int G = GQA ? mk.H / mk.Hkv : 1;  // query heads per K/V head
  const bool rot = mk.seqlens_k != nullptr;  // rotated schedule under key padding

  uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff + 8);
  float* lse_s = reinterpret_cast<float*>(smem + L::kLseOff);
  float* dsum_s = reinterpret_cast<float*>(smem + L::kDsumOff);

  DkdvBars bars;
  {
    int i = 0;
    auto nb = [&]() { return smem_u32(&bar_mem[i++]); };
    auto run = [&](int n) {
      const BarRun r{smem_u32(&bar_mem[i])};
      i += n;
      return r;
    };
    bars.kv_full = run(2);
    bars.kv_empty = run(2);
    bars.q_full = run(kMaxQStages);
    bars.q_empty = run(kMaxQStages);
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
    bars.stall = nb();
  }
  if (tid == 0) {
    *abort_flag = 0;
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.kv_full[b], 1);
      mbar_init(bars.kv_empty[b], 1);
    }
    for (int s = 0; s < kMaxQStages; ++s) {
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
    mbar_init(bars.stall, 1);
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

  if (warp >= kComputeWarps) {
    // producer, issuers and the idle warp: one warpgroup, which hands most of its
    // registers to the compute warpgroups
    regs_dec<kRegsAux>();
    if (warp == kProdWarp) {
      // ------------------------------------------------------------ producer
      uint32_t it = 0, q_arms = 0, kv_arms[2] = {0, 0};
      bool ok = true;
      int unit_count = 0;
      for (int u = sched_unit(0, rot); u < n_units && ok; u = sched_unit(++unit_count, rot)) {
        const int bhk = u / n_t, kt = u % n_t;  // K/V head, key tile
        const int kv_len = kv_len_of(mk, bhk / mk.Hkv);
        const int n_kv = (kv_len + kTile - 1) / kTile;
        const int kb = unit_count % L::kKVBufs;
        const int kuse = unit_count / L::kKVBufs;
        if (kuse > 0 && !mbar_wait_warp(bars.kv_empty[kb], (kuse - 1) & 1, tmo, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_expect_tx(bars.kv_full[kb], 2 * T);
          tma_tile<D>(sKV + (2 * kb) * T, &tm_k, kt * kTile, bhk, bars.kv_full[kb]);
          tma_tile<D>(sKV + (2 * kb + 1) * T, &tm_v, kt * kTile, bhk, bars.kv_full[kb]);
        }
        ++kv_arms[kb];
        for (int bh = group_first_head<GQA>(mk, bhk), bh_end = bh + G; bh < bh_end && ok;
               ++bh) {  // the query heads sharing this K/V head
          for (int chunk = 0; chunk * 32 < n_t && ok; ++chunk) {
            uint32_t bits = warp_valid_bits_t<WIN>(mk, kt, chunk, n_t, n_kv);
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
                lp[r] = -lse2_at(args.lse, idx, in);
                dp[r] = in ? -args.dsum[idx] : 0.f;
              }
              // staged negated: the compute warps add them as packed pairs
              reinterpret_cast<float4*>(lse_s + s * 128)[lane] = l4;
              reinterpret_cast<float4*>(dsum_s + s * 128)[lane] = d4;
              if (lane == 0) {
                mbar_expect_tx(bars.q_full[s], 2 * T);
                tma_tile<D>(sQ + s * T, &tm_q, qt * kTile, bh, bars.q_full[s]);
                tma_tile<D>(sDO + s * T, &tm_do, qt * kTile, bh, bars.q_full[s]);
              } else {
                mbar_arrive(bars.q_full[s]);
              }
              ++q_arms;
              ++it;
            }
          }
        }
      }
      for (int b = 0; b < L::kKVBufs; ++b)
        if (kv_arms[b]) mbar_wait_warp(bars.kv_full[b], (kv_arms[b] - 1) & 1, tmo, nullptr);
  #pragma unroll
      for (int s = 0; s < L::kStages; ++s)
        if (q_arms > static_cast<uint32_t>(s))
          mbar_wait_warp(bars.q_full[s], ((q_arms - 1 - s) / L::kStages) & 1, tmo, nullptr);
    } else if (warp == kIssueAWarp) {
      // ------------------------------------------------------------ S^T, dP^T issuer
      // Before overwriting S^T (dP^T) it waits until the compute warps have read it
      // (separate buffers), or until dV (dK) has consumed the P^T (dS^T) written
      // over it (aliased buffers).
      const bool leader = lane == 0;
      const uint32_t bar_s_ok = L::kSepBuf ? bars.st_free : bars.p_done;
      const uint32_t bar_dp_ok = L::kSepBuf ? bars.dpt_free : bars.ds_done;
      uint32_t it = 0, gt = 0, sfc = 0, dfc = 0;
      bool ok = true;
      if (args.sync.inject_stall && leader) {
        // Test hook: this barrier is never completed, so the bounded wait runs out.
        if (!mbar_wait(bars.stall, 0, tmo, abort_flag)) {
          fail();
          ok = false;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      int unit_count = 0;
      for (int u = sched_unit(0, rot); u < n_units && ok; u = sched_unit(++unit_count, rot)) {
        const int bhk = u / n_t, kt = u % n_t;  // K/V head, key tile
        const int kv_len = kv_len_of(mk, bhk / mk.Hkv);
        const int n_kv = (kv_len + kTile - 1) / kTile;
        const int kb = unit_count % L::kKVBufs;
        if (leader &&
            !mbar_wait(bars.kv_full[kb], (unit_count / L::kKVBufs) & 1, tmo, abort_flag)) {
          fail();
          ok = false;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        const uint64_t dK = sdesc_sw128(sKV + (2 * kb) * T, 16, 1024);
        const uint64_t dV = sdesc_sw128(sKV + (2 * kb + 1) * T, 16, 1024);
        for (int bh = group_first_head<GQA>(mk, bhk), bh_end = bh + G; bh < bh_end && ok;
               ++bh) {  // the query heads sharing this K/V head
          for (int chunk = 0; chunk * 32 < n_t && ok; ++chunk) {
            const uint32_t vbits = warp_valid_bits_t<WIN>(mk, kt, chunk, n_t, n_kv);
            if (leader) {
              for (uint32_t bits = vbits; bits != 0u && ok; bits &= bits - 1) {
                const int s = it % L::kStages;
                const uint32_t ph = (it / L::kStages) & 1u;
                if (!mbar_wait(bars.q_full[s], ph, tmo, abort_flag) ||
                    (gt > 0 && !mbar_wait(bar_s_ok, sfc++ & 1, tmo, abort_flag))) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                mma_ss_tile<D>(tmem + L::kColSt, dK, sdesc_sw128(sQ + s * T, 16, 1024));
                mma_commit(bars.st_full);
                if (gt > 0 && !mbar_wait(bar_dp_ok, dfc++ & 1, tmo, abort_flag)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                mma_ss_tile<D>(tmem + L::kColDPt, dV, sdesc_sw128(sDO + s * T, 16, 1024));
                mma_commit(bars.dpt_full);
                mma_commit(bars.q_empty[s]);
                ++gt;
                ++it;
              }
              if (!ok) fail();
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
          }
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
      for (int u = sched_unit(0, rot); u < n_units && ok; u = sched_unit(++unit_count, rot)) {
        const int bhk = u / n_t, kt = u % n_t;  // K/V head, key tile
        const int kv_len = kv_len_of(mk, bhk / mk.Hkv);
        const int n_kv = (kv_len + kTile - 1) / kTile;
        bool first = true;
        for (int bh = group_first_head<GQA>(mk, bhk), bh_end = bh + G; bh < bh_end && ok;
               ++bh) {  // the query heads sharing this K/V head
          for (int chunk = 0; chunk * 32 < n_t && ok; ++chunk) {
            const uint32_t vbits = warp_valid_bits_t<WIN>(mk, kt, chunk, n_t, n_kv);
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
                mma_ts_tile<D>(tmem + L::kColDV, tmem + L::kColP, L::kPair,
                               sdesc_sw128(sDO + s * T, 16384, 1024), !first);
                mma_commit(bars.p_done);
                if (!mbar_wait(bars.ds_ready, dsc++ & 1, tmo, abort_flag)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                mma_ts_tile<D>(tmem + L::kColDK, tmem + L::kColDS, L::kPair,
                               sdesc_sw128(sQ + s * T, 16384, 1024), !first);
                mma_commit(bars.ds_done);
                mma_commit(bars.q_empty[s]);
                first = false;
                ++it;
              }
              if (!ok) fail();
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
          }
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
    }
  } else {
    regs_inc<kRegsCompute>();
    // ------------------------------------------------------------ compute
    // Warpgroup wg owns query columns [32 wg, 32 wg + 32) of every tile; the
    // thread owns one key row.
    const int wg = warp >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tSt = tmem + lane_base + L::kColSt + 32 * wg;
    const uint32_t tDPt = tmem + lane_base + L::kColDPt + 32 * wg;
    const uint32_t tP = tmem + lane_base + L::kColP + L::kPair * wg;
    const uint32_t tDS = tmem + lane_base + L::kColDS + L::kPair * wg;
    const float c_log2 = args.scale_log2;
    const uint64_t ks2 = f2_pack(args.drop.keep_scale, args.drop.keep_scale);
    uint32_t* drop_scratch = reinterpret_cast<uint32_t*>(smem + L::kDropOff + warp * 1024);
    uint32_t it = 0, gt = 0, stc = 0, dpc = 0, pdc = 0, dsc = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = sched_unit(0, rot); u < n_units && ok; u = sched_unit(++unit_count, rot)) {
      const int bhk = u / n_t, kt = u % n_t;  // K/V head, key tile
      const int kv_len = kv_len_of(mk, bhk / mk.Hkv);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      const int key = kt * kTile + r;
      int n_done = 0;
      for (int bh = group_first_head<GQA>(mk, bhk), bh_end = bh + G; bh < bh_end && ok;
             ++bh) {  // the query heads sharing this K/V head
        for (int chunk = 0; chunk * 32 < n_t && ok; ++chunk) {
          uint32_t bits = warp_valid_bits_t<WIN>(mk, kt, chunk, n_t, n_kv);
          while (bits != 0u && ok) {
            const int qt = chunk * 32 + (__ffs(bits) - 1);
            bits &= bits - 1;
            const int s = it % L::kStages;
            const float* lse_t = lse_s + s * 128 + 32 * wg;
            const float* dsum_t = dsum_s + s * 128 + 32 * wg;
            const int q0 = qt * kTile + 32 * wg;  // first query column of this warpgroup
            // Dropout keep bytes (0x00 / 0xFF) of this thread's key for the 32 query
            // columns, four per word: column c is byte c & 3 of bm[c >> 2].
            uint32_t bm[8];
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
              // this lane's key is byte (lane & 3) of word (lane & 15) >> 2 of the
              // block of its 16-key group: gather it for four columns at a time
              const uint32_t kb = static_cast<uint32_t>(lane & 3);
              const uint32_t sel2 = kb | ((4u + kb) << 4);  // byte kb of a, then byte kb of b
              const uint32_t* wcol = drop_scratch + (lane >> 4) * 4 + ((lane & 15) >> 2);
  #pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint32_t t0 = prmt(wcol[(4 * k + 0) * 8], wcol[(4 * k + 1) * 8], sel2);
                const uint32_t t1 = prmt(wcol[(4 * k + 2) * 8], wcol[(4 * k + 3) * 8], sel2);
                bm[k] = prmt(t0, t1, 0x5410u);
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
            float p[32];  // P^T, fp32, kept until dS^T is formed
            {
              uint32_t sr[32];
              tmem_ld32(tSt, sr);
              tmem_ld_wait();
              if constexpr (L::kSepBuf) {
                tc_fence_before();
                mbar_arrive(bars.st_free);
              }
              const uint64_t c2 = f2_pack(c_log2, c_log2);
  #pragma unroll
              for (int c4 = 0; c4 < 8; ++c4) {
                const ulonglong2 nl = reinterpret_cast<const ulonglong2*>(lse_t)[c4];  // -lse2 pairs
  #pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int c = 4 * c4 + 2 * h;
                  float x0, x1;
                  f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2,
                                   h ? nl.y : nl.x),
                            x0, x1);
                  p[c] = ex2_approx(x0);
                  p[c + 1] = ex2_approx(x1);
                }
              }
            }
            if (tile_needs_element_mask<WIN>(mk, qt, kt, kv_len)) {
              const bool key_ok = key < kv_len;
  #pragma unroll
              for (int c = 0; c < 32; ++c)
                p[c] = (key_ok && (!mk.causal || key <= q0 + c) &&
                        (!WIN || in_window(mk, q0 + c, key)))
                           ? p[c]
                           : 0.f;
            }
            {
              uint32_t pk[16];  // dropped copy for dV
  #pragma unroll
              for (int c = 0; c < 16; ++c) {
                uint32_t pp = pack_bf16x2(p[2 * c], p[2 * c + 1]);
                if constexpr (DROPOUT) pp &= prmt(bm[c >> 1], 0u, (c & 1) ? 0x3322u : 0x1100u);
                pk[c] = pp;
              }
              if constexpr (L::kSepBuf) {
                if (gt > 0) {  // the previous dV has finished reading the P^T buffer
                  if (!mbar_wait_warp(bars.p_done, pdc++ & 1, tmo, abort_flag)) {
                    fail();
                    ok = false;
                    break;
                  }
                  tc_fence_after();
                }
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
              if constexpr (L::kSepBuf) {
                tc_fence_before();
                mbar_arrive(bars.dpt_free);
              }
              uint32_t pk[16];
  #pragma unroll
              for (int c4 = 0; c4 < 8; ++c4) {
                const ulonglong2 nd = reinterpret_cast<const ulonglong2*>(dsum_t)[c4];  // -D pairs
  #pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int c = 4 * c4 + 2 * h;
                  uint32_t dp0 = dr[c], dp1 = dr[c + 1];
                  if constexpr (DROPOUT) {  // keep byte -> all-ones / all-zeros lane mask
                    dp0 &= prmt(bm[c >> 2], 0u, (8u | (c & 3)) * 0x1111u);
                    dp1 &= prmt(bm[c >> 2], 0u, (8u | ((c + 1) & 3)) * 0x1111u);
                  }
                  const uint64_t t = f2_fma(ks2, f2_pack(__uint_as_float(dp0), __uint_as_float(dp1)),
                                            h ? nd.y : nd.x);
                  float a0, a1;
                  f2_unpack(f2_mul(f2_pack(p[c], p[c + 1]), t), a0, a1);
                  pk[2 * c4 + h] = pack_bf16x2(a0, a1);
                }
              }
              if constexpr (L::kSepBuf) {
                if (gt > 0) {  // the previous dK has finished reading the dS^T buffer
                  if (!mbar_wait_warp(bars.ds_done, dsc++ & 1, tmo, abort_flag)) {
                    fail();
                    ok = false;
                    break;
                  }
                  tc_fence_after();
                }
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
      }
      if (!ok) break;
      // ---- epilogue: dV (warpgroups 0, 1) and dK (2, 3), D/2 columns each
      if (!mbar_wait_warp(bars.acc_full, unit_count & 1, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      tc_fence_after();
      constexpr int kHalf = D / 2;
      const bool is_dv = wg < 2;
      const uint32_t tAcc =
          tmem + lane_base + (is_dv ? L::kColDV : L::kColDK) + kHalf * (wg & 1);
      const float mult = is_dv ? args.drop.keep_scale : args.scale;
      __nv_bfloat16* dst = (is_dv ? args.dv : args.dk) +
                           (static_cast<size_t>(bhk) * N + static_cast<size_t>(key)) * D +
                           kHalf * (wg & 1);
#pragma unroll
      for (int c = 0; c < kHalf / 32; ++c) {
        uint32_t v[32];
        if (n_done > 0) {
          tmem_ld32(tAcc + 32 * c, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          pk[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * mult,
                              __uint_as_float(v[2 * k + 1]) * mult);
        if (key < N) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            d4[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
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
// dQ [256, 256+d), dS bf16 [256+d, 320+d).
template <int D>
struct DqL {
  static constexpr int T = TileT<D>::kBytes;
  static constexpr int kQDBufs = (D == 64) ? 2 : 1;
  static constexpr int kKStages = (D == 64) ? 4 : 3;
  static constexpr int kVStages = (D == 64) ? 3 : 2;
  static_assert(kKStages <= kMaxKStages && kVStages <= kMaxVStages,
                "K / V ring deeper than its barrier arrays");
  static constexpr int kQOff = 0;                                  // kQDBufs x (Q, dO)
  static constexpr int kKOff = kQDBufs * 2 * T;
  static constexpr int kVOff = kKOff + kKStages * T;
  static constexpr int kBarOff = kVOff + kVStages * T;
  static constexpr int kNumBars = 4 + 2 * kMaxKStages + 2 * kMaxVStages + 11;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // d = 64: the epilogue stages each compute warp's 32 rows of dQ (1 KB) before
  // storing them coalesced; at d = 128 shared memory has no room for it.
  static constexpr bool kStageDq = (D == 64);
  static constexpr int kStageOff = (kMiscOff + 64 + 127) / 128 * 128;
  static constexpr int kSmemBytes = kStageOff + (kStageDq ? kComputeWarps * 1024 : 0) + 1024;
  static_assert(kSmemBytes <= 232448, "dQ layout exceeds 227 KB of shared memory");
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 256 + D;
};

struct DqBars {
  BarRun qd_full, qd_empty, k_full, k_empty;
  BarRun v_full, v_empty;
  uint32_t s_full, s_free, dp_full, dp_free, ds_ready, ds_done, dq_full, dq_free;
  uint32_t drain_a, drain_b;
  uint32_t stall;  // test hook: never completed
};

template <int D, bool DROPOUT>
struct DqRealloc {
  static constexpr bool value = (D == 128) || DROPOUT;
};

template <int D, bool DROPOUT, bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dq_split_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_do, const BwdArgs args) {
  using L = DqL<D>;
  // Register reallocation pays at d = 128 and with dropout (both keep more values
  // live per compute thread); at d = 64 without dropout the compute warps need no
  // more than the launch allocation and the kernel runs faster without it.
  constexpr bool kRealloc = DqRealloc<D, DROPOUT>::value;
  constexpr int T = L::T;
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
    auto run = [&](int n) {
      const BarRun r{smem_u32(&bar_mem[i])};
      i += n;
      return r;
    };
    bars.qd_full = run(2);
    bars.qd_empty = run(2);
    bars.k_full = run(kMaxKStages);
    bars.k_empty = run(kMaxKStages);
    bars.v_full = run(kMaxVStages);
    bars.v_empty = run(kMaxVStages);
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
    bars.stall = nb();
  }
  if (tid == 0) {
    *abort_flag = 0;
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.qd_full[b], 1);
      mbar_init(bars.qd_empty[b], 1);
    }
    for (int s = 0; s < kMaxKStages; ++s) {
      mbar_init(bars.k_full[s], 1);
      mbar_init(bars.k_empty[s], 1);
    }
    for (int s = 0; s < kMaxVStages; ++s) {
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
    mbar_init(bars.stall, 1);
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

  if (warp >= kComputeWarps) {
    // producer, issuers and the idle warp: one warpgroup, which hands most of its
    // registers to the compute warpgroups
    if constexpr (kRealloc) regs_dec<kRegsAux>();
    if (warp == kProdWarp) {
      // ------------------------------------------------------------ producer
      uint32_t it = 0, k_arms = 0, v_arms = 0, qd_arms[2] = {0, 0};
      bool ok = true;
      int unit_count = 0;
      for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
        int bh, qt;
        unit_coords(u, bh, qt);
        const int kvh = kv_head(mk, bh);  // K/V head of this query head
        const int kv_len = kv_len_of(mk, bh / mk.H);
        const int n_kv = (kv_len + kTile - 1) / kTile;
        const int jmax = kv_limit(qt, n_kv);
        const int qb = unit_count % L::kQDBufs, use = unit_count / L::kQDBufs;
        if (use > 0 && !mbar_wait_warp(bars.qd_empty[qb], (use - 1) & 1, tmo, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_expect_tx(bars.qd_full[qb], 2 * T);
          tma_tile<D>(sQD + (2 * qb) * T, &tm_q, qt * kTile, bh, bars.qd_full[qb]);
          tma_tile<D>(sQD + (2 * qb + 1) * T, &tm_do, qt * kTile, bh, bars.qd_full[qb]);
        }
        ++qd_arms[qb];
        for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
          uint32_t bits = warp_valid_bits<WIN>(mk, qt, chunk, n_q, n_kv);
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
              mbar_expect_tx(bars.k_full[ks], T);
              tma_tile<D>(sK + ks * T, &tm_k, j * kTile, kvh, bars.k_full[ks]);
            }
            ++k_arms;
            if (!mbar_wait_warp(bars.v_empty[vs], ((it / L::kVStages) & 1u) ^ 1u, tmo, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            if (lane == 0) {
              mbar_expect_tx(bars.v_full[vs], T);
              tma_tile<D>(sV + vs * T, &tm_v, j * kTile, kvh, bars.v_full[vs]);
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
      for (int b = 0; b < L::kQDBufs; ++b)
        if (qd_arms[b]) mbar_wait_warp(bars.qd_full[b], (qd_arms[b] - 1) & 1, tmo, nullptr);
    } else if (warp == kIssueAWarp) {
      // ------------------------------------------------------------ S, dP issuer
      const bool leader = lane == 0;
      uint32_t it = 0, gt = 0, sfc = 0, dfc = 0;
      bool ok = true;
      if (args.sync.inject_stall && leader) {
        // Test hook: this barrier is never completed, so the bounded wait runs out.
        if (!mbar_wait(bars.stall, 0, tmo, abort_flag)) {
          fail();
          ok = false;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      int unit_count = 0;
      for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
        int bh, qt;
        unit_coords(u, bh, qt);
        const int kv_len = kv_len_of(mk, bh / mk.H);
        const int n_kv = (kv_len + kTile - 1) / kTile;
        const int jmax = kv_limit(qt, n_kv);
        const int qb = unit_count % L::kQDBufs;
        if (leader &&
            !mbar_wait(bars.qd_full[qb], (unit_count / L::kQDBufs) & 1, tmo, abort_flag)) {
          fail();
          ok = false;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        const uint64_t dQ = sdesc_sw128(sQD + (2 * qb) * T, 16, 1024);
        const uint64_t dDO = sdesc_sw128(sQD + (2 * qb + 1) * T, 16, 1024);
        for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
          const uint32_t vbits = warp_valid_bits<WIN>(mk, qt, chunk, n_q, n_kv);
          if (leader) {
            for (uint32_t bits = vbits; bits != 0u && ok; bits &= bits - 1) {
              const int ks = it % L::kKStages, vs = it % L::kVStages;
              if (!mbar_wait(bars.k_full[ks], (it / L::kKStages) & 1u, tmo, abort_flag) ||
                  (gt > 0 && !mbar_wait(bars.s_free, sfc++ & 1, tmo, abort_flag))) {
                ok = false;
                break;
              }
              tc_fence_after();
              mma_ss_tile<D>(tmem + L::kColS, dQ, sdesc_sw128(sK + ks * T, 16, 1024));
              mma_commit(bars.s_full);
              if (!mbar_wait(bars.v_full[vs], (it / L::kVStages) & 1u, tmo, abort_flag) ||
                  (gt > 0 && !mbar_wait(bars.dp_free, dfc++ & 1, tmo, abort_flag))) {
                ok = false;
                break;
              }
              tc_fence_after();
              mma_ss_tile<D>(tmem + L::kColDP, dDO, sdesc_sw128(sV + vs * T, 16, 1024));
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
      for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
        int bh, qt;
        unit_coords(u, bh, qt);
        const int kv_len = kv_len_of(mk, bh / mk.H);
        const int n_kv = (kv_len + kTile - 1) / kTile;
        const int jmax = kv_limit(qt, n_kv);
        bool first = true;
        for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
          const uint32_t vbits = warp_valid_bits<WIN>(mk, qt, chunk, n_q, n_kv);
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
              mma_ts_tile<D>(tmem + L::kColDQ, tmem + L::kColDS, 16,
                             sdesc_sw128(sK + ks * T, 16384, 1024), !first);
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
    }
  } else {
    if constexpr (kRealloc) regs_inc<kRegsCompute>();
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
    constexpr int kQCols = D / 4;  // dQ columns written by each warpgroup
    const uint32_t tDQ = tmem + lane_base + L::kColDQ + kQCols * wg;
    const float c_log2 = args.scale_log2;
    uint32_t gt = 0, sc = 0, dc = 0, ddc = 0;
    // At d = 128 the dS store's completion is waited for under the next step's
    // S load (measured faster); at d = 64 the dQ MMA must not wait for it
    // (measured slower), so the store is completed at once.
    constexpr bool kDeferDs = (D == 128);
    bool ds_pending = false;  // a dS store issued whose ds_ready arrival is still due
    bool ok = true;
    int unit_count = 0;
    for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
      int bh, qt;
      unit_coords(u, bh, qt);
      const int row = qt * kTile + t;
      const bool row_in = row < N;
      const long long ridx = static_cast<long long>(bh) * N + row;
      const float lse2 = lse2_at(args.lse, ridx, row_in);
      const float dsum = row_in ? args.dsum[ridx] : 0.f;
      const uint64_t c2 = f2_pack(c_log2, c_log2);
      const uint64_t nl2 = f2_pack(-lse2, -lse2);
      const uint64_t nd2 = f2_pack(-dsum, -dsum);
      const uint64_t ks2 = f2_pack(args.drop.keep_scale, args.drop.keep_scale);
      const int kv_len = kv_len_of(mk, bh / mk.H);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      const int jmax = kv_limit(qt, n_kv);
      // sliding window: keys [key_lo, key_hi) are visible to this row
      int key_lo = 0, key_hi = kv_len;
      if constexpr (WIN) {
        if (mk.causal && row + 1 < key_hi) key_hi = row + 1;
        if (mk.wr >= 0 && row + mk.wr + 1 < key_hi) key_hi = row + mk.wr + 1;
        if (mk.wl >= 0) key_lo = row - mk.wl;
      }
      int n_done = 0;
      for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
        uint32_t bits = warp_valid_bits<WIN>(mk, qt, chunk, n_q, n_kv);
        while (bits != 0u && ok) {
          const int j = chunk * 32 + (__ffs(bits) - 1);
          bits &= bits - 1;
          // Dropout keep bytes (0x00 / 0xFF) of this row's 32 key columns, four
          // per word: column c is byte c & 3 of word c >> 2.
          uint32_t kb[8];
          if constexpr (DROPOUT) {
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              const uint4 kw = dropout_keep16(args.drop, static_cast<uint32_t>(ridx),
                                              static_cast<uint32_t>(j * 8 + 2 * wg + g));
              kb[4 * g + 0] = kw.x;
              kb[4 * g + 1] = kw.y;
              kb[4 * g + 2] = kw.z;
              kb[4 * g + 3] = kw.w;
            }
          }
          // WIN: whether this row's visible-key edge falls in the warpgroup's 32 columns
          const bool masked = WIN ? (j * kTile + 32 * wg < key_lo || j * kTile + 32 * wg + 32 > key_hi)
                                  : tile_needs_element_mask<WIN>(mk, qt, j, kv_len);
          // ---- P = exp2(S c - lse2), kept as bf16 pairs
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
            if (kDeferDs && ds_pending) {  // the previous step's dS store completes under this load
              tmem_st_wait();
              tc_fence_before();
              mbar_arrive(bars.ds_ready);
              ds_pending = false;
            }
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(bars.s_free);
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2,
                               nl2),
                        x0, x1);
              p[c] = ex2_approx(x0);
              p[c + 1] = ex2_approx(x1);
            }
            if constexpr (WIN) {
              if (masked) {  // keys [key_lo, key_hi) are allowed for this row
                const int base = j * kTile + 32 * wg;  // key of column 0 of this warpgroup
                const int lim_local = key_hi - base, lo_local = key_lo - base;
#pragma unroll
                for (int c = 0; c < 32; ++c) p[c] = (c >= lo_local && c < lim_local) ? p[c] : 0.f;
              }
            } else if (masked) {  // keys [0, lim) of this tile are allowed for this row
              int lim = kv_len - j * kTile;
              if (mk.causal) {
                const int lc = row - j * kTile + 1;
                lim = lc < lim ? lc : lim;
              }
              const int lim_local = lim - 32 * wg;
#pragma unroll
              for (int c = 0; c < 32; ++c) p[c] = (c < lim_local) ? p[c] : 0.f;
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
              uint32_t dp0 = dr[2 * c], dp1 = dr[2 * c + 1];
              if constexpr (DROPOUT) {
                // keep byte -> all-ones / all-zeros lane mask (sign replicated)
                const uint32_t wd = kb[c >> 1];
                const uint32_t b0 = (2 * c) & 3;
                dp0 &= prmt(wd, 0u, (8u | b0) * 0x1111u);
                dp1 &= prmt(wd, 0u, (8u | (b0 + 1u)) * 0x1111u);
              }
              const uint64_t t =
                  f2_fma(ks2, f2_pack(__uint_as_float(dp0), __uint_as_float(dp1)), nd2);
              float d0, d1;
              f2_unpack(f2_mul(f2_pack(p[2 * c], p[2 * c + 1]), t), d0, d1);
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
          if constexpr (kDeferDs) {
            ds_pending = true;  // completed, and ds_ready arrived, under the next S load
          } else {
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bars.ds_ready);
          }
          ++n_done;
          ++gt;
        }
      }
      if (!ok) break;
      if (ds_pending) {  // the last dQ MMA of the unit needs this step's dS
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bars.ds_ready);
        ds_pending = false;
      }
      // ---- epilogue: dQ = scale * acc, D/4 columns per warpgroup
      if (!mbar_wait_warp(bars.dq_full, unit_count & 1, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[kQCols];
      if (n_done > 0) {
        if constexpr (kQCols == 32) tmem_ld32(tDQ, v);
        else tmem_ld16(tDQ, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int k = 0; k < kQCols; ++k) v[k] = 0u;
      }
      uint32_t o[kQCols / 2];
#pragma unroll
      for (int k = 0; k < kQCols / 2; ++k)
        o[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * args.scale,
                           __uint_as_float(v[2 * k + 1]) * args.scale);
      if constexpr (L::kStageDq) {
        // The warp's 32 rows x 32 bytes go through shared memory so that each
        // store instruction writes 16 rows' whole 32-byte segments instead of 32
        // half segments. Row r's two 16-byte units swap places on rows 4-7 of
        // every 8 (no bank conflicts either way).
        const uint32_t stage = smem_u32(smem + L::kStageOff) + static_cast<uint32_t>(warp * 1024);
        const uint32_t sw = static_cast<uint32_t>(lane >> 2) & 1u;
        st_shared_v4(stage + static_cast<uint32_t>(lane * 32) + (sw << 4), o[0], o[1], o[2], o[3]);
        st_shared_v4(stage + static_cast<uint32_t>(lane * 32) + ((sw ^ 1u) << 4), o[4], o[5], o[6],
                     o[7]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = 16 * i + (lane >> 1);  // row within the warp's 32
          const uint32_t u = static_cast<uint32_t>(lane & 1);
          const uint4 val = ld_shared_v4(stage + static_cast<uint32_t>(r * 32) +
                                         ((u ^ (static_cast<uint32_t>(r >> 2) & 1u)) << 4));
          const int row_r = qt * kTile + quad * 32 + r;
          if (row_r < N)
            *reinterpret_cast<uint4*>(args.dq +
                                      (static_cast<size_t>(bh) * N + static_cast<size_t>(row_r)) * D +
                                      kQCols * wg + 8 * u) = val;
        }
      } else if (row_in) {
        uint4* d4 = reinterpret_cast<uint4*>(args.dq + static_cast<size_t>(ridx) * D + kQCols * wg);
#pragma unroll
        for (int k = 0; k < kQCols / 8; ++k)
          d4[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
      }
      tc_fence_before();
      mbar_arrive(bars.dq_free);
    }
    tmem_st_wait();  // no tensor-memory store may still be in flight on any exit path
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kIssueAWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Shared-memory opt-in, and a check that the kernel was built for the
// register count its in-kernel reallocation assumes: launched with fewer
// registers per thread, the compute warpgroups' increase could never be granted
// and would wait forever, so such a kernel is refused instead of launched.
template <typename K>
cudaError_t set_smem_split(K kern, int bytes, bool realloc) {
  if (realloc) {
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    if (attr.numRegs < kRegsLaunch || attr.maxThreadsPerBlock < kThreads)
      return cudaErrorInvalidConfiguration;
  }
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int D>
cudaError_t launch_dkdv_split_d(const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& tdo, const BwdArgs& a,
                                bool dropout, int grid, cudaStream_t stream) {
  const bool gqa = a.mask.Hkv != a.mask.H, win = a.mask.wl >= 0 || a.mask.wr >= 0;
  auto pick = [&](auto drop) {
    constexpr bool DR = decltype(drop)::value;
    return gqa ? (win ? fa_bwd_dkdv_split_kernel<D, DR, true, true>
                      : fa_bwd_dkdv_split_kernel<D, DR, true, false>)
               : (win ? fa_bwd_dkdv_split_kernel<D, DR, false, true>
                      : fa_bwd_dkdv_split_kernel<D, DR, false, false>);
  };
  auto kern = dropout ? pick(std::true_type{}) : pick(std::false_type{});
  cudaError_t e = set_smem_split(kern, DkdvL<D>::kSmemBytes, true);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, DkdvL<D>::kSmemBytes, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dq_split_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const BwdArgs& a, bool dropout, int grid,
                              cudaStream_t stream) {
  const bool win = a.mask.wl >= 0 || a.mask.wr >= 0;
  auto kern = dropout ? (win ? fa_bwd_dq_split_kernel<D, true, true>
                             : fa_bwd_dq_split_kernel<D, true, false>)
                      : (win ? fa_bwd_dq_split_kernel<D, false, true>
                             : fa_bwd_dq_split_kernel<D, false, false>);
  const bool realloc = dropout ? DqRealloc<D, true>::value : DqRealloc<D, false>::value;
  cudaError_t e = set_smem_split(kern, DqL<D>::kSmemBytes, realloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, DqL<D>::kSmemBytes, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv_split(const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const CUtensorMap& tdo, const BwdArgs& a,
                                  int d, bool dropout, int num_sms, cudaStream_t stream) {
  const int n_t = (a.mask.N + kTile - 1) / kTile;
  const long long units = static_cast<long long>(a.mask.B) * a.mask.Hkv * n_t;  // (K/V head, key tile)
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  if (grid <= 0) return cudaSuccess;
  if (d != 64) return cudaErrorInvalidValue;  // head dimension 128 runs the single-issuer kernel
  return launch_dkdv_split_d<64>(tq, tk, tv, tdo, a, dropout, grid, stream);
}

cudaError_t launch_bwd_dq_split(const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& tdo, const BwdArgs& a,
                                int d, bool dropout, int num_sms, cudaStream_t stream) {
  const int n_q = (a.mask.N + kTile - 1) / kTile;
  const long long units = static_cast<long long>(a.mask.B) * a.mask.H * n_q;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  if (grid <= 0) return cudaSuccess;
  return d == 64 ? launch_dq_split_d<64>(tq, tk, tv, tdo, a, dropout, grid, stream)
                 : launch_dq_split_d<128>(tq, tk, tv, tdo, a, dropout, grid, stream);
}

}  // namespace fa
