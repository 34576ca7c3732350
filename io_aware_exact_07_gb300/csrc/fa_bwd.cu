// Backward pass of exact attention on sm_103a. Nothing of size N x N is
// stored: S and P are recomputed on chip from Q, K and the saved logsumexp
// (FlashAttention deep-read report, sections 2.5 "recomputation" and 3.3
// "backward pass and memory layout"; Attention Kernel page, "why tiling also
// works for training"). With L = sum(O * dO):
//   D_i   = sum_c dO_ic O_ic                       (preprocess kernel)
//   P_ij  = exp(scale q_i.k_j - lse_i), masked; Z_ij the dropout keep bit
//   dV_j  = sum_i P_ij Z_ij/(1-p) dO_i
//   dS_ij = P_ij (Z_ij/(1-p) dO_i.v_j - D_i)
//   dK_j  = scale sum_i dS_ij q_i                  (key-tile kernel: dK, dV)
//   dQ_i  = scale sum_j dS_ij k_j                  (query-tile kernel: dQ)
// The five contractions of the backward (the cross-paper synthesis page notes
// the backward's five matmuls against the forward's two) are split over two
// kernels so that every output tile is owned by exactly one CTA: dQ needs no
// atomics and every result is deterministic. The price is that S and dP are
// computed twice (seven tensor-core contractions instead of five).
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

namespace {

constexpr int kBwdThreads = 352;
constexpr int kProducerWarp = 8;    // K, V and the Q ring (with lse)
constexpr int kMmaWarp = 9;
constexpr int kDOProducerWarp = 10; // the dO ring (with D)

// ------------------------------------------------------------------ preprocess
// D = rowsum(dO * O) in fp32; 8 threads per row, 16-byte loads.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                             const __nv_bfloat16* __restrict__ dout,
                                                             float* __restrict__ dsum,
                                                             long long rows) {
  const int sub = threadIdx.x & 7;
  const unsigned gmask = 0xFFu << (threadIdx.x & 24);
  const long long groups_per_grid = (static_cast<long long>(gridDim.x) * blockDim.x) >> 3;
  for (long long row = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 3;
       row < rows; row += groups_per_grid) {
    float acc = 0.f;
#pragma unroll
    for (int c = sub; c < D / 8; c += 8) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D) + c);
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + row * D) + c);
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
      const uint32_t wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[e]));
        const float2 fb2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb[e]));
        acc = fmaf(fa2.x, fb2.x, acc);
        acc = fmaf(fa2.y, fb2.y, acc);
      }
    }
    acc += __shfl_xor_sync(gmask, acc, 4, 8);
    acc += __shfl_xor_sync(gmask, acc, 2, 8);
    acc += __shfl_xor_sync(gmask, acc, 1, 8);
    if (sub == 0) dsum[row] = acc;
  }
}

// lse in log2 units for recomputing P = exp2(s * scale * log2e - lse2); rows
// outside [0, N) and rows without any allowed key map to +inf, so P = 0.
__device__ __forceinline__ float lse2_of(const float* lse, long long idx, bool in_range) {
  if (!in_range) return INFINITY;
  const float l = lse[idx];
  return (l == -INFINITY) ? INFINITY : l * kLog2e;
}

// ================================================================== dK, dV
// One work unit = one (b, h) head and one 128-row key tile (K_j, V_j stay in
// shared memory); the loop runs over the query tiles that may attend to it.
//   warp 8      TMA producer: K_j, V_j per unit; Q_i (and lse_i via plain
//               loads) through the Q ring.
//   warp 10     TMA producer: dO_i (and D_i via plain loads) through the dO ring.
//   warp 9      MMA issuer: S^T = K Q^T, dP^T = V dO^T (shared-memory
//               operands), dV += P^T dO and dK += dS^T Q (A from tensor memory).
//   warps 0-7   two warpgroups, each owning 64 of the 128 query columns of
//               every tile (thread = key row): P^T = exp2(S^T c - lse2),
//               dropout, dS^T = P^T (Z dP^T / (1-p) - D); P^T and dS^T go back
//               to tensor memory as bf16 over the columns they were read from.
// A Q tile is last read by dK of the step after its own, a dO tile by dV of its
// own step, so the Q ring is one stage deeper than the dO ring (the dropout
// instances keep two Q stages to leave room for their Philox scratch).
// Tensor memory: dV [0, d), dK [d, 2d), S^T [2d, 2d+128), dP^T [2d+128, 2d+256).
template <int D, bool DROPOUT>
struct DkdvLayout {
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kQStages = DROPOUT ? 2 : 3;
  static constexpr int kDOStages = 2;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;
  static constexpr int kDOOff = kQOff + kQStages * kTileBytes;
  static constexpr int kLseOff = kDOOff + kDOStages * kTileBytes;  // kQStages x 128 fp32
  static constexpr int kDsumOff = kLseOff + kQStages * 512;        // kDOStages x 128 fp32
  static constexpr int kDropOff = kDsumOff + kDOStages * 512;      // 8 warps x 2 KB Philox scratch
  static constexpr int kBarOff = kDropOff + (DROPOUT ? 8 * 2048 : 0);
  static constexpr int kNumBars = 2 + 2 * kQStages + 2 * kDOStages + 6 + 2;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // No slack for rounding the base up: the kernel checks that the dynamic
  // shared memory starts on a 1024-byte boundary (the SW128 tiles need it).
  static constexpr int kSmemBytes = kMiscOff + 16;
  static_assert(kSmemBytes <= 232448, "d=128 dK/dV layout exceeds 227 KB of shared memory");
  __device__ static constexpr uint32_t col_dv() { return 0u; }
  __device__ static constexpr uint32_t col_dk() { return static_cast<uint32_t>(D); }
  __device__ static constexpr uint32_t col_st() { return static_cast<uint32_t>(2 * D); }
  __device__ static constexpr uint32_t col_dpt() { return static_cast<uint32_t>(2 * D + 128); }
};

template <int D, bool DROPOUT, bool GQA, bool WIN>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do, const BwdArgs args) {
  using L = DkdvLayout<D, DROPOUT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0u) {  // uniform over the block: nothing has started yet
    if (threadIdx.x == 0) record_error(args.sync.status, kStatusCuda);
    return;
  }
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const MaskParams& mk = args.mask;
  const int N = mk.N;
  const int n_t = (N + kTile - 1) / kTile;  // query tiles == key tiles
  const int n_units = mk.B * mk.Hkv * n_t;
  const int G = GQA ? mk.H / mk.Hkv : 1;  // query heads per K/V head

  uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff + 8);
  float* lse_s = reinterpret_cast<float*>(smem + L::kLseOff);
  float* dsum_s = reinterpret_cast<float*>(smem + L::kDsumOff);

  // ring barriers by stage: full, then empty, Q ring first
  const uint32_t bar0 = smem_u32(bar_mem);
  auto q_full = [&](int s) { return bar0 + 8u * static_cast<uint32_t>(2 + s); };
  auto q_empty = [&](int s) { return bar0 + 8u * static_cast<uint32_t>(2 + L::kQStages + s); };
  auto do_full = [&](int s) {
    return bar0 + 8u * static_cast<uint32_t>(2 + 2 * L::kQStages + s);
  };
  auto do_empty = [&](int s) {
    return bar0 + 8u * static_cast<uint32_t>(2 + 2 * L::kQStages + L::kDOStages + s);
  };
  uint32_t b_kv_full, b_kv_empty, b_st_full, b_dpt_full, b_p_ready, b_ds_ready, b_acc_full,
      b_acc_free, b_drain, b_stall;
  {
    int i = 0;
    auto nb = [&]() { return smem_u32(&bar_mem[i++]); };
    b_kv_full = nb();
    b_kv_empty = nb();
    i += 2 * (L::kQStages + L::kDOStages);
    b_st_full = nb();
    b_dpt_full = nb();
    b_p_ready = nb();
    b_ds_ready = nb();
    b_acc_full = nb();
    b_acc_free = nb();
    b_drain = nb();
    b_stall = nb();  // test hook: never completed
  }
  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(b_kv_full, 1);
    mbar_init(b_kv_empty, 1);
    // full: the 32 producer lanes (lse / D staged by plain stores, one lane
    // also arms the TMA bytes); empty: the MMA commit after the tile's last
    // contraction and one lane of each compute warp once lse / D are read
    for (int s = 0; s < L::kQStages; ++s) {
      mbar_init(q_full(s), 32);
      mbar_init(q_empty(s), 1 + 8);
    }
    for (int s = 0; s < L::kDOStages; ++s) {
      mbar_init(do_full(s), 32);
      mbar_init(do_empty(s), 1 + 8);
    }
    mbar_init(b_st_full, 1);
    mbar_init(b_dpt_full, 1);
    mbar_init(b_p_ready, 256);
    mbar_init(b_ds_ready, 256);
    mbar_init(b_acc_full, 1);
    mbar_init(b_acc_free, 256);
    mbar_init(b_drain, 1);
    mbar_init(b_stall, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
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
  const uint32_t sK = smem_u32(smem + L::kKOff);
  const uint32_t sV = smem_u32(smem + L::kVOff);
  const uint32_t sQ = smem_u32(smem + L::kQOff);
  const uint32_t sDO = smem_u32(smem + L::kDOOff);

  if (warp == kProducerWarp || warp == kDOProducerWarp) {
    // ------------------------------------------------------------ producers
    // Warp 8: K, V per unit and the Q ring with -lse2; warp 10: the dO ring
    // with -D. Each stage's row values go in by plain stores from the 32 lanes
    // before they arrive on the stage's full barrier.
    const bool q_side = warp == kProducerWarp;
    const int n_stages = q_side ? L::kQStages : L::kDOStages;
    const CUtensorMap* tm = q_side ? &tm_q : &tm_do;
    const uint32_t ring = q_side ? sQ : sDO;
    float* rowvals = q_side ? lse_s : dsum_s;
    uint32_t it = 0, kv_arms = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
      const int bhk = u / n_t, kt = u % n_t;  // K/V head, key tile
      const int b = bhk / mk.Hkv;
      const int kv_len = kv_len_of(mk, b);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      if (q_side) {
        if (unit_count > 0 &&
            !mbar_wait_warp(b_kv_empty, (unit_count - 1) & 1, tmo, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_expect_tx(b_kv_full, 2 * L::kTileBytes);
          for (int c = 0; c < L::kChunks; ++c) {
            tma_load_3d(sK + c * 16384, &tm_k, c * 64, kt * kTile, bhk, b_kv_full);
            tma_load_3d(sV + c * 16384, &tm_v, c * 64, kt * kTile, bhk, b_kv_full);
          }
        }
        ++kv_arms;
      }
      for (int bh = group_first_head<GQA>(mk, bhk), bh_end = bh + G; bh < bh_end && ok;
           ++bh) {  // the query heads sharing this K/V head
        for (int chunk = 0; chunk * 32 < n_t && ok; ++chunk) {
          uint32_t bits = warp_valid_bits_t<WIN>(mk, kt, chunk, n_t, n_kv);
          while (bits != 0u) {
            const int qt = chunk * 32 + (__ffs(bits) - 1);
            bits &= bits - 1;
            const int s = static_cast<int>(it % static_cast<uint32_t>(n_stages));
            const uint32_t ph = (it / static_cast<uint32_t>(n_stages)) & 1u;
            const uint32_t full = q_side ? q_full(s) : do_full(s);
            if (!mbar_wait_warp(q_side ? q_empty(s) : do_empty(s), ph ^ 1u, tmo, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            // lse (log2 units) or D of the 128 query rows of this tile, staged
            // negated: the compute warps add them as packed pairs
            float4 v4;
            float* vp = &v4.x;
  #pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int row = qt * kTile + 4 * lane + r;
              const bool in = row < N;
              const long long idx = static_cast<long long>(bh) * N + row;
              vp[r] = q_side ? -lse2_of(args.lse, idx, in) : (in ? -args.dsum[idx] : 0.f);
            }
            reinterpret_cast<float4*>(rowvals + s * 128)[lane] = v4;
            if (lane == 0) {
              mbar_expect_tx(full, L::kTileBytes);
              for (int c = 0; c < L::kChunks; ++c)
                tma_load_3d(ring + s * L::kTileBytes + c * 16384, tm, c * 64, qt * kTile, bh, full);
            } else {
              mbar_arrive(full);
            }
            ++it;
          }
        }
      }
    }
    // no copy may still be in flight when the block exits
    if (kv_arms) mbar_wait_warp(b_kv_full, (kv_arms - 1) & 1, tmo, nullptr);
    for (int s = 0; s < n_stages; ++s)
      if (it > static_cast<uint32_t>(s))
        mbar_wait_warp(q_side ? q_full(s) : do_full(s),
                       ((it - 1 - s) / static_cast<uint32_t>(n_stages)) & 1, tmo, nullptr);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, 0, 1);
    const bool elected = lane == 0;
    uint32_t it = 0, p_cnt = 0, ds_cnt = 0;
    bool ok = true;
    if (args.sync.inject_stall && elected) {
      // Test hook: this barrier is never completed, so the bounded wait runs out.
      if (!mbar_wait(b_stall, 0, tmo, abort_flag)) {
        fail();
        ok = false;
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    int unit_count = 0;
    // acc (+)= A[tmem, 64-column halves at a0 and a0 + 64] * B[smem, MN-major]
    auto issue_acc = [&](uint32_t d_col, uint32_t a_col, uint32_t b_base, bool accumulate) {
      const uint64_t db = sdesc_sw128(b_base, 16384, 1024);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a = tmem + a_col + (kk >> 2) * 64 + (kk & 3) * 8;
        mma_ts(tmem + d_col, a, db + static_cast<uint64_t>((kk * 2048) >> 4), kIdAcc,
               (accumulate || kk > 0) ? 1u : 0u);
      }
    };
    auto issue_ss = [&](uint32_t d_col, uint32_t a_base, uint32_t b_base) {
      const uint64_t da = sdesc_sw128(a_base, 16, 1024);
      const uint64_t db = sdesc_sw128(b_base, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_ss(tmem + d_col, da + (off >> 4), db + (off >> 4), kIdS, kk > 0 ? 1u : 0u);
      }
    };
    for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
      const int bhk = u / n_t, kt = u % n_t;  // K/V head, key tile
      const int b = bhk / mk.Hkv;
      const int kv_len = kv_len_of(mk, b);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      if (!mbar_wait_warp(b_kv_full, unit_count & 1, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      int t = 0;
      int prev_s = -1;
      for (int bh = group_first_head<GQA>(mk, bhk), bh_end = bh + G; bh < bh_end && ok;
             ++bh) {  // the query heads sharing this K/V head
        for (int chunk = 0; chunk * 32 < n_t && ok; ++chunk) {
          uint32_t bits = warp_valid_bits_t<WIN>(mk, kt, chunk, n_t, n_kv);
          while (bits != 0u) {
            bits &= bits - 1;
            const int sq = it % L::kQStages, sd = it % L::kDOStages;
            if (!mbar_wait_warp(q_full(sq), (it / L::kQStages) & 1u, tmo, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            tc_fence_after();
            if (elected) {
              issue_ss(L::col_st(), sK, sQ + sq * L::kTileBytes);  // S^T = K Q^T
              mma_commit(b_st_full);
            }
            __syncwarp();
            if (t > 0) {  // dK += dS^T(prev) Q(prev)
              if (!mbar_wait_warp(b_ds_ready, ds_cnt & 1, tmo, abort_flag)) {
                fail();
                ok = false;
                break;
              }
              ++ds_cnt;
              tc_fence_after();
              if (elected) {
                issue_acc(L::col_dk(), L::col_dpt(), sQ + prev_s * L::kTileBytes, t - 1 > 0);
                mma_commit(q_empty(prev_s));
              }
              __syncwarp();
            }
            if (!mbar_wait_warp(do_full(sd), (it / L::kDOStages) & 1u, tmo, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            tc_fence_after();
            if (elected) {
              issue_ss(L::col_dpt(), sV, sDO + sd * L::kTileBytes);  // dP^T = V dO^T
              mma_commit(b_dpt_full);
            }
            __syncwarp();
            if (!mbar_wait_warp(b_p_ready, p_cnt & 1, tmo, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            ++p_cnt;
            if (t == 0 && unit_count > 0 &&
                !mbar_wait_warp(b_acc_free, (unit_count - 1) & 1, tmo, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            tc_fence_after();
            if (elected) {
              issue_acc(L::col_dv(), L::col_st(), sDO + sd * L::kTileBytes, t > 0);
              mma_commit(do_empty(sd));
            }
            __syncwarp();
            prev_s = sq;
            ++t;
            ++it;
          }
        }
      }
      if (!ok) break;
      if (t > 0) {
        if (!mbar_wait_warp(b_ds_ready, ds_cnt & 1, tmo, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        ++ds_cnt;
        tc_fence_after();
        if (elected) {
          issue_acc(L::col_dk(), L::col_dpt(), sQ + prev_s * L::kTileBytes, t - 1 > 0);
          mma_commit(q_empty(prev_s));
        }
        __syncwarp();
      } else if (unit_count > 0) {
        if (!mbar_wait_warp(b_acc_free, (unit_count - 1) & 1, tmo, abort_flag)) {
          fail();
          ok = false;
          break;
        }
      }
      if (elected) {
        mma_commit(b_acc_full);
        mma_commit(b_kv_empty);
      }
      __syncwarp();
    }
    if (elected) mma_commit(b_drain);
    __syncwarp();
    mbar_wait_warp(b_drain, 0, tmo, nullptr);
  } else {
    // ------------------------------------------------------------ compute
    const int wg = warp >> 2;   // query columns [64 wg, 64 wg + 64)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // key row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tSt = tmem + lane_base + L::col_st() + 64 * wg;
    const uint32_t tDPt = tmem + lane_base + L::col_dpt() + 64 * wg;
    const float c_log2 = args.scale_log2;
    uint32_t* drop_scratch = reinterpret_cast<uint32_t*>(smem + L::kDropOff + warp * 2048);
    uint32_t it = 0, st_cnt = 0, dpt_cnt = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
      const int bhk = u / n_t, kt = u % n_t;  // K/V head, key tile
      const int b = bhk / mk.Hkv;
      const int kv_len = kv_len_of(mk, b);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      const int key = kt * kTile + r;
      int n_done = 0;
      for (int bh = group_first_head<GQA>(mk, bhk), bh_end = bh + G; bh < bh_end && ok;
             ++bh) {  // the query heads sharing this K/V head
        for (int chunk = 0; chunk * 32 < n_t && ok; ++chunk) {
          uint32_t bits = warp_valid_bits_t<WIN>(mk, kt, chunk, n_t, n_kv);
          while (bits != 0u) {
            const int qt = chunk * 32 + (__ffs(bits) - 1);
            bits &= bits - 1;
            const int sq = it % L::kQStages, sd = it % L::kDOStages;
            const float* lse_t = lse_s + sq * 128 + 64 * wg;
            const float* dsum_t = dsum_s + sd * 128 + 64 * wg;
            const int q0 = qt * kTile + 64 * wg;  // first query column of this thread's half
            // Dropout keep bits of this (key, 64 queries) strip.
            uint32_t zb0 = 0xFFFFFFFFu, zb1 = 0xFFFFFFFFu;
            if constexpr (DROPOUT) {
              const uint32_t key0 = static_cast<uint32_t>(kt * kTile + quad * 32);
  #pragma unroll
              for (int m = 0; m < 4; ++m) {
                const int idx = lane + 32 * m;
                const int c = idx >> 1, gs = idx & 1;
                const uint32_t rowg = static_cast<uint32_t>(bh) * static_cast<uint32_t>(N) +
                                      static_cast<uint32_t>(q0 + c);
                const uint4 kw = dropout_keep16(args.drop, rowg, (key0 >> 4) + gs);
                reinterpret_cast<uint4*>(drop_scratch)[c * 2 + gs] = kw;
              }
              __syncwarp();
              zb0 = 0u;
              zb1 = 0u;
  #pragma unroll
              for (int c = 0; c < 64; ++c) {
                const uint32_t w = drop_scratch[(c * 2 + (lane >> 4)) * 4 + ((lane & 15) >> 2)];
                const uint32_t kbit = (w >> (8 * (lane & 3))) & 1u;  // bytes are 0x00 or 0xFF
                if (c < 32) zb0 |= kbit << c;
                else zb1 |= kbit << (c - 32);
              }
              __syncwarp();
            }
            // ---- phase 1: P^T
            if (!mbar_wait_warp(b_st_full, st_cnt & 1, tmo, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            ++st_cnt;
            tc_fence_after();
            float p[64];
            {
              uint32_t sr[64];
              tmem_ld32(tSt, &sr[0]);
              tmem_ld32(tSt + 32, &sr[32]);
              tmem_ld_wait();
              const uint64_t c2 = f2_pack(c_log2, c_log2);
  #pragma unroll
              for (int c4 = 0; c4 < 16; ++c4) {
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
              for (int c = 0; c < 64; ++c) {
                const bool allowed = key_ok && (!mk.causal || key <= q0 + c) &&
                                     (!WIN || in_window(mk, q0 + c, key));
                p[c] = allowed ? p[c] : 0.f;
              }
            }
            {
              uint32_t pk[32];
  #pragma unroll
              for (int c = 0; c < 32; ++c) {
                float a0 = p[2 * c], a1 = p[2 * c + 1];
                if constexpr (DROPOUT) {
                  const uint32_t zw = (c < 16) ? zb0 : zb1;
                  const int sh = (2 * c) & 31;
                  a0 = ((zw >> sh) & 1u) ? a0 : 0.f;
                  a1 = ((zw >> (sh + 1)) & 1u) ? a1 : 0.f;
                }
                pk[c] = pack_bf16x2(a0, a1);
              }
              tmem_st32(tSt, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(b_p_ready);
            // ---- phase 2: dS^T
            if (!mbar_wait_warp(b_dpt_full, dpt_cnt & 1, tmo, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            ++dpt_cnt;
            tc_fence_after();
            {
              uint32_t pk[32];
  #pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t dr[32];
                tmem_ld32(tDPt + 32 * h, dr);
                tmem_ld_wait();
  #pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                  const ulonglong2 nd = reinterpret_cast<const ulonglong2*>(dsum_t)[8 * h + c4];  // -D
  #pragma unroll
                  for (int e = 0; e < 4; e += 2) {
                    const int c = 32 * h + 4 * c4 + e;
                    float z0 = args.drop.keep_scale, z1 = args.drop.keep_scale;
                    if constexpr (DROPOUT) {
                      const uint32_t zw = (c < 32) ? zb0 : zb1;
                      z0 = ((zw >> (c & 31)) & 1u) ? z0 : 0.f;
                      z1 = ((zw >> ((c + 1) & 31)) & 1u) ? z1 : 0.f;
                    }
                    const uint64_t t = f2_fma(f2_pack(z0, z1),
                                              f2_pack(__uint_as_float(dr[4 * c4 + e]),
                                                      __uint_as_float(dr[4 * c4 + e + 1])),
                                              e ? nd.y : nd.x);
                    float a0, a1;
                    f2_unpack(f2_mul(f2_pack(p[c], p[c + 1]), t), a0, a1);
                    pk[16 * h + 2 * c4 + (e >> 1)] = pack_bf16x2(a0, a1);
                  }
                }
              }
              tmem_st32(tDPt, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(b_ds_ready);
            __syncwarp();
            if (lane == 0) {  // lse and D of these stages no longer read
              mbar_arrive(q_empty(sq));
              mbar_arrive(do_empty(sd));
            }
            ++n_done;
            ++it;
          }
        }
      }
      if (!ok) break;
      // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK
      if (!mbar_wait_warp(b_acc_full, unit_count & 1, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tAcc = tmem + lane_base + (wg == 0 ? L::col_dv() : L::col_dk());
      const float mult = (wg == 0) ? args.drop.keep_scale : args.scale;
      __nv_bfloat16* dst_base = (wg == 0) ? args.dv : args.dk;
      __nv_bfloat16* dst = dst_base + (static_cast<size_t>(bhk) * N + static_cast<size_t>(key)) * D;
      const bool row_ok = key < N;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
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
          pk[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * mult, __uint_as_float(v[2 * k + 1]) * mult);
        if (row_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            d4[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(b_acc_free);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <typename K>
cudaError_t set_smem(K kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a, int d, int num_sms, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.mask.B) * a.mask.H * a.mask.N;
  const long long want = (rows * 8 + 255) / 256;
  const int grid = static_cast<int>(want < num_sms * 8LL ? want : num_sms * 8LL);
  if (grid <= 0) return cudaSuccess;
  if (d == 64)
    bwd_preprocess_kernel<64><<<grid, 256, 0, stream>>>(a.o, a.dout, a.dsum, rows);
  else
    bwd_preprocess_kernel<128><<<grid, 256, 0, stream>>>(a.o, a.dout, a.dsum, rows);
  return cudaGetLastError();
}

template <int D, bool DROP>
static cudaError_t launch_dkdv_impl(const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const CUtensorMap& tdo,
                                    const BwdArgs& a, int grid, cudaStream_t stream) {
  const bool gqa = a.mask.Hkv != a.mask.H, win = a.mask.wl >= 0 || a.mask.wr >= 0;
  auto kern = gqa ? (win ? fa_bwd_dkdv_kernel<D, DROP, true, true>
                         : fa_bwd_dkdv_kernel<D, DROP, true, false>)
                  : (win ? fa_bwd_dkdv_kernel<D, DROP, false, true>
                         : fa_bwd_dkdv_kernel<D, DROP, false, false>);
  constexpr int kSmem = DkdvLayout<D, DROP>::kSmemBytes;
  cudaError_t e = set_smem(kern, kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kBwdThreads, kSmem, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdArgs& a, int d, bool dropout,
                            int num_sms, cudaStream_t stream) {
  const int n_t = (a.mask.N + kTile - 1) / kTile;
  const long long units = static_cast<long long>(a.mask.B) * a.mask.Hkv * n_t;  // (K/V head, key tile)
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  if (grid <= 0) return cudaSuccess;
  if (d == 64) return launch_bwd_dkdv_split(tq, tk, tv, tdo, a, d, dropout, num_sms, stream);
  return dropout ? launch_dkdv_impl<128, true>(tq, tk, tv, tdo, a, grid, stream)
                 : launch_dkdv_impl<128, false>(tq, tk, tv, tdo, a, grid, stream);
}

cudaError_t launch_bwd_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdArgs& a, int d, bool dropout,
                          int num_sms, cudaStream_t stream) {
  return launch_bwd_dq_split(tq, tk, tv, tdo, a, d, dropout, num_sms, stream);
}

}  // namespace fa
