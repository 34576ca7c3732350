// FP8 forward of exact attention (FA-3's FP8 with incoherent processing, the
// cross-paper synthesis page on FlashAttention, section 2): Q', K' (rotated)
// and V as e4m3 with scales from fa_fp8.cu, S = Q' K'^T and O += P V on the
// tensor core in FP8 (tcgen05.mma kind::f8f6f4, fp32 accumulators in tensor
// memory), online softmax in fp32 as in the bf16 forward, head dimension 128.
//
// Structure as the bf16 forward's decoupled schedule (one unit = one head and
// 256 query rows, split into two 128-row tiles that ping-pong on the tensor
// core): warp 8 is the TMA producer (Q_a, Q_b, then K_j and V_j^T tiles
// through a ring), warp 9 issues S_x = Q_x K_j^T, warp 10 issues
// O_x += P_x V_j, warps 0-7 run the softmax (thread = query row). What
// differs:
//  - every operand tile is 128 rows of 128 bytes (one 128-byte swizzle
//    chunk); V arrives transposed ([d, keys]) so that all four operands are
//    K-major, and one MMA covers 32 keys or channels;
//  - P is quantised to e4m3 and written to shared memory in the swizzled
//    layout the tensor core reads (so the S buffer is free as soon as the
//    softmax has loaded it); to keep small probabilities above e4m3's
//    subnormal floor, P = exp2(s c - m_ref + 5) and the reference maximum
//    follows the row maximum to within 3 (log2 units), so 2^5 <= max P <= 2^8
//    (e4m3 reaches 448) and weights down to 2^-14 of the row maximum survive
//    (a tighter reference, 1 with offset 7, rescales O more often for 3 %);
//  - the scales: S is multiplied by s_q s_k (folded into the exponent's
//    factor) and O's column c by s_v[c] in the epilogue.
//  - grouped K/V heads (Hkv dividing H): query head h of batch b reads K/V
//    tiles and scales of K/V head b Hkv + h / (H / Hkv).
// Tensor memory: S_a, S_b, O_a, O_b (128 columns each).
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_fp8.h"

namespace fa {

namespace {

constexpr int kF8Threads = 352;
constexpr int kF8ProducerWarp = 8;
constexpr int kF8MmaWarp = 9;
constexpr int kF8PvWarp = 10;
constexpr float kF8Rescale = 3.0f;  // log2 units: the reference follows the row maximum to 3
constexpr float kF8POffset = 5.0f;  // P = exp2(x - m_ref + 5): max P in [2^5, 2^8]

struct F8L {
  static constexpr int kTileBytes = kTile * 128;  // 128 rows x 128 one-byte elements
  static constexpr int kStages = 4;
  static constexpr int kQOff = 0;                  // Q_a, Q_b
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kPOff = kVOff + kStages * kTileBytes;  // P_a, P_b
  static constexpr int kBarOff = kPOff + 2 * kTileBytes;
  // q_full[2], q_empty, k_full/k_empty/v_full/v_empty[S], s_full[2], s_free[2],
  // p_full[2], pv_done[2], o_free[2], drain, drain2, stall
  static constexpr int kNumBars = 3 + 4 * kStages + 10 + 3;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;
  static_assert(kSmemBytes <= 232448, "more shared memory than one CTA may hold");
  __device__ static constexpr uint32_t col_s(int x) { return static_cast<uint32_t>(x) * 128u; }
  __device__ static constexpr uint32_t col_o(int x) { return 256u + static_cast<uint32_t>(x) * 128u; }
};

struct F8Bars {
  BarRun q_full;
  uint32_t q_empty;
  BarRun k_full, k_empty, v_full, v_empty;
  BarRun s_full, s_free, p_full, pv_done, o_free;
  uint32_t drain, drain2, stall;
};

struct F8Unit {
  int bh, bhk, b, qt0;  // query head, its K/V head, batch row, first query tile
};

// Units run head by head, so the query heads of one K/V group are neighbours
// in the schedule and their K/V tiles are read from L2 after the first.
__device__ __forceinline__ F8Unit f8_unit(int u, const MaskParams& m, int n_qblk) {
  F8Unit c;
  const int bh = u / n_qblk;
  int qb = u % n_qblk;
  if (m.causal) qb = n_qblk - 1 - qb;  // longest causal units of a head first
  c.bh = bh;
  c.bhk = kv_head(m, bh);
  c.b = bh / m.H;
  c.qt0 = 2 * qb;
  return c;
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE,
                                                        __NV_E4M3));
}

__device__ __forceinline__ void fence_async_smem_writes() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace

__global__ void __launch_bounds__(kF8Threads, 1)
    fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_vt, const Fp8FwdArgs args) {
  using L = F8L;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const MaskParams& mk = args.mask;
  const int N = mk.N;
  const int n_q = (N + kTile - 1) / kTile;
  const int n_qblk = (n_q + 1) / 2;
  const int n_units = mk.B * mk.H * n_qblk;

  uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff + 8);
  F8Bars bars;
  {
    int i = 0;
    auto nb = [&]() { return smem_u32(&bar_mem[i++]); };
    auto run = [&](int n) {
      const BarRun r{smem_u32(&bar_mem[i])};
      i += n;
      return r;
    };
    bars.q_full = run(2);
    bars.q_empty = nb();
    bars.k_full = run(L::kStages);
    bars.k_empty = run(L::kStages);
    bars.v_full = run(L::kStages);
    bars.v_empty = run(L::kStages);
    bars.s_full = run(2);
    bars.s_free = run(2);
    bars.p_full = run(2);
    bars.pv_done = run(2);
    bars.o_free = run(2);
    bars.drain = nb();
    bars.drain2 = nb();
    bars.stall = nb();
  }
  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bars.q_full[0], 1);
    mbar_init(bars.q_full[1], 1);
    mbar_init(bars.q_empty, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bars.k_full[s], 1);
      mbar_init(bars.k_empty[s], 1);
      mbar_init(bars.v_full[s], 1);
      mbar_init(bars.v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bars.s_full[x], 1);
      mbar_init(bars.s_free[x], 128);
      mbar_init(bars.p_full[x], 128);
      mbar_init(bars.pv_done[x], 1);
      // o_free[x]: the 128 softmax threads of tile x at the end of each
      // epilogue, plus the PV issuer once per unit after its own wait on the
      // previous phase, so that no phase can complete while the PV issuer still
      // waits on the one before it.
      mbar_init(bars.o_free[x], 129);
    }
    mbar_init(bars.drain, 1);
    mbar_init(bars.drain2, 1);
    mbar_init(bars.stall, 1);
    fence_mbar_init();
  }
  if (warp == kF8MmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t tmo = args.sync.timeout_ns;
  auto fail = [&](void) {
    *abort_flag = 1;
    record_error(args.sync.status, kStatusTimeout);
  };
  const uint32_t sQ = smem_u32(smem + L::kQOff);
  const uint32_t sK = smem_u32(smem + L::kKOff);
  const uint32_t sV = smem_u32(smem + L::kVOff);
  const uint32_t sP = smem_u32(smem + L::kPOff);
  constexpr uint32_t kId = idesc_e4m3_f32(128, 128);
  constexpr uint64_t kStep = static_cast<uint64_t>(L::kTileBytes >> 4);

  if (warp == kF8ProducerWarp) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0, k_arms = 0, v_arms = 0, q_armed = 0;
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
    }
    int unit_count = 0;
    for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
      const F8Unit uc = f8_unit(u, mk, n_qblk);
      const int kv_len = kv_len_of(mk, uc.b);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      int jmax = n_kv;
      if (mk.causal && uc.qt0 + 2 < jmax) jmax = uc.qt0 + 2;
      if (unit_count > 0 && !mbar_wait_warp(bars.q_empty, (unit_count - 1) & 1, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      if (lane == 0) {
        for (int x = 0; x < 2; ++x) {
          mbar_expect_tx(bars.q_full[x], L::kTileBytes);
          tma_load_3d(sQ + x * L::kTileBytes, &tm_q, 0, (uc.qt0 + x) * kTile, uc.bh,
                      bars.q_full[x]);
        }
      }
      ++q_armed;
      for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
        uint32_t bits = warp_valid_bits(mk, uc.qt0, chunk, n_q, n_kv) |
                        warp_valid_bits(mk, uc.qt0 + 1, chunk, n_q, n_kv);
        while (bits != 0u) {
          const int j = chunk * 32 + (__ffs(bits) - 1);
          bits &= bits - 1;
          const int s = it % L::kStages;
          const uint32_t ph = (it / L::kStages) & 1u;
          if (!mbar_wait_warp(bars.k_empty[s], ph ^ 1u, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_expect_tx(bars.k_full[s], L::kTileBytes);
            tma_load_3d(sK + s * L::kTileBytes, &tm_k, 0, j * kTile, uc.bhk, bars.k_full[s]);
          }
          ++k_arms;
          if (!mbar_wait_warp(bars.v_empty[s], ph ^ 1u, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_expect_tx(bars.v_full[s], L::kTileBytes);
            // V^T: keys j*128 .. j*128+127 (innermost), all 128 channels
            tma_load_3d(sV + s * L::kTileBytes, &tm_vt, j * kTile, 0, uc.bhk, bars.v_full[s]);
          }
          ++v_arms;
          ++it;
        }
      }
    }
#pragma unroll
    for (int s = 0; s < L::kStages; ++s) {
      if (k_arms > static_cast<uint32_t>(s))
        mbar_wait_warp(bars.k_full[s], ((k_arms - 1 - s) / L::kStages) & 1, tmo, nullptr);
      if (v_arms > static_cast<uint32_t>(s))
        mbar_wait_warp(bars.v_full[s], ((v_arms - 1 - s) / L::kStages) & 1, tmo, nullptr);
    }
    if (q_armed) {
      mbar_wait_warp(bars.q_full[0], (q_armed - 1) & 1, tmo, nullptr);
      mbar_wait_warp(bars.q_full[1], (q_armed - 1) & 1, tmo, nullptr);
    }
  } else if (warp == kF8MmaWarp) {
    // ------------------------------------------------------------ S issuer
    const bool leader = (lane == 0);
    const uint64_t dQa = sdesc_sw128(sQ, 16, 1024);
    const uint64_t dQb = sdesc_sw128(sQ + L::kTileBytes, 16, 1024);
    const uint64_t dK0 = sdesc_sw128(sK, 16, 1024);
    uint32_t it = 0, sf_cnt0 = 0, sf_cnt1 = 0;
    bool s_seen0 = false, s_seen1 = false;
    bool ok = true;
    if (args.sync.inject_stall && leader) {
      // Test hook: a barrier that nothing completes, so the bounded wait runs out.
      if (!mbar_wait(bars.stall, 0, tmo, abort_flag)) {
        fail();
        ok = false;
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    auto issue_S = [&](int x, int s) {
      const uint64_t dq = x ? dQb : dQa;
      const uint64_t dk = dK0 + static_cast<uint64_t>(s) * kStep;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {  // 32 channels (32 bytes) per MMA
        const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
        mma_ss_f8(tmem + L::col_s(x), dq + off, dk + off, kId, kk > 0 ? 1u : 0u);
      }
      mma_commit(bars.s_full[x]);
    };
    int unit_count = 0;
    for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
      const F8Unit uc = f8_unit(u, mk, n_qblk);
      const int kv_len = kv_len_of(mk, uc.b);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      int jmax = n_kv;
      if (mk.causal && uc.qt0 + 2 < jmax) jmax = uc.qt0 + 2;
      const uint32_t uph = unit_count & 1;
      if (leader) {
        ok = mbar_wait(bars.q_full[0], uph, tmo, abort_flag) &&
             mbar_wait(bars.q_full[1], uph, tmo, abort_flag);
        if (!ok) fail();
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
        const uint32_t va = warp_valid_bits(mk, uc.qt0, chunk, n_q, n_kv);
        const uint32_t vb = warp_valid_bits(mk, uc.qt0 + 1, chunk, n_q, n_kv);
        if (leader) {
          uint32_t bits = va | vb;
          while (bits != 0u && ok) {
            const int bit = __ffs(bits) - 1;
            bits &= bits - 1;
            const bool v0 = ((va >> bit) & 1u) != 0u, v1 = ((vb >> bit) & 1u) != 0u;
            const int s = it % L::kStages;
            if (!mbar_wait(bars.k_full[s], (it / L::kStages) & 1u, tmo, abort_flag)) {
              ok = false;
              break;
            }
            if (v0) {  // S_a as soon as the softmax has loaded the previous S_a
              if (s_seen0 && !mbar_wait(bars.s_free[0], sf_cnt0++ & 1, tmo, abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_S(0, s);
              s_seen0 = true;
            }
            if (v1) {
              if (s_seen1 && !mbar_wait(bars.s_free[1], sf_cnt1++ & 1, tmo, abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_S(1, s);
              s_seen1 = true;
            }
            mma_commit(bars.k_empty[s]);
            ++it;
          }
          if (!ok) fail();
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (leader && ok) mma_commit(bars.q_empty);
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (leader) {
      mma_commit(bars.drain);
      mbar_wait(bars.drain, 0, tmo, nullptr);
    }
    __syncwarp();
  } else if (warp == kF8PvWarp) {
    // ------------------------------------------------------------ PV issuer
    const bool leader = (lane == 0);
    const uint64_t dV0 = sdesc_sw128(sV, 16, 1024);
    const uint64_t dPa = sdesc_sw128(sP, 16, 1024);
    const uint64_t dPb = sdesc_sw128(sP + L::kTileBytes, 16, 1024);
    uint32_t it = 0, p_cnt0 = 0, p_cnt1 = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
      const F8Unit uc = f8_unit(u, mk, n_qblk);
      const int kv_len = kv_len_of(mk, uc.b);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      int jmax = n_kv;
      if (mk.causal && uc.qt0 + 2 < jmax) jmax = uc.qt0 + 2;
      bool first0 = true, first1 = true;
      // The first PV of query tile x in a unit overwrites O_x, which the previous
      // unit's epilogue reads: it waits for that epilogue (o_free[x]) and adds
      // this issuer's arrival for the current unit.
      auto claim_o = [&](int x) -> bool {
        if (unit_count > 0 && !mbar_wait(bars.o_free[x], (unit_count - 1) & 1, tmo, abort_flag))
          return false;
        mbar_arrive(bars.o_free[x]);
        return true;
      };
      auto pv = [&](int x, int s, bool first) -> bool {
        // (counters selected by value: a reference to either would put both in
        // local memory)
        const uint32_t pc = x ? p_cnt1 : p_cnt0;
        if (!mbar_wait(bars.p_full[x], pc & 1, tmo, abort_flag)) return false;
        if (x) ++p_cnt1; else ++p_cnt0;
        if (first && !claim_o(x)) return false;
        tc_fence_after();
        const uint64_t dp = x ? dPb : dPa;
        const uint64_t dv = dV0 + static_cast<uint64_t>(s) * kStep;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // 32 keys per MMA
          const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
          mma_ss_f8(tmem + L::col_o(x), dp + off, dv + off, kId, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(bars.pv_done[x]);
        return true;
      };
      for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
        const uint32_t va = warp_valid_bits(mk, uc.qt0, chunk, n_q, n_kv);
        const uint32_t vb = warp_valid_bits(mk, uc.qt0 + 1, chunk, n_q, n_kv);
        if (leader) {
          uint32_t bits = va | vb;
          while (bits != 0u && ok) {
            const int bit = __ffs(bits) - 1;
            bits &= bits - 1;
            const bool v0 = ((va >> bit) & 1u) != 0u, v1 = ((vb >> bit) & 1u) != 0u;
            const int s = it % L::kStages;
            if (!mbar_wait(bars.v_full[s], (it / L::kStages) & 1u, tmo, abort_flag) ||
                (v0 && !pv(0, s, first0)) || (v1 && !pv(1, s, first1))) {
              ok = false;
              break;
            }
            if (v0) first0 = false;
            if (v1) first1 = false;
            mma_commit(bars.v_empty[s]);
            ++it;
          }
          if (!ok) fail();
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (leader && ok) {
        // a query tile without keys in this unit still consumes the epilogue
        // handshake and adds its arrival
        ok = (!first0 || claim_o(0)) && (!first1 || claim_o(1));
        if (!ok) fail();
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (leader) {
      mma_commit(bars.drain2);
      mbar_wait(bars.drain2, 0, tmo, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;    // query tile within the unit
    const int quad = warp & 3;  // tensor-memory lane quadrant
    const int t = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::col_s(x);
    const uint32_t tO = tmem + lane_base + L::col_o(x);
    uint8_t* prow = smem + L::kPOff + x * L::kTileBytes + t * 128;  // this row of P
    uint32_t s_cnt = 0, pv_cnt = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
      const F8Unit uc = f8_unit(u, mk, n_qblk);
      const int qt = uc.qt0 + x;
      const int row = qt * kTile + t;
      const int kv_len = kv_len_of(mk, uc.b);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      int jmax = n_kv;
      if (mk.causal && qt + 1 < jmax) jmax = qt + 1;
      // S of the stored codes times s_q s_k is the score; c folds both into the exponent
      const float c_log2 = args.scale_log2 * args.s_q[uc.bh] * args.s_k[uc.bhk];
      const uint64_t c2 = f2_pack(c_log2, c_log2);
      float m_ref = -INFINITY;
      float l_sum = 0.f;
      int n_done = 0;
      for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
        uint32_t bits = warp_valid_bits(mk, qt, chunk, n_q, n_kv);
        while (bits != 0u) {
          const int j = chunk * 32 + (__ffs(bits) - 1);
          bits &= bits - 1;
          if (!mbar_wait_warp(bars.s_full[x], s_cnt & 1, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          ++s_cnt;
          tc_fence_after();
          uint32_t sr[128];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, &sr[c * 32]);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(bars.s_free[x]);  // S is in registers: the next S may overwrite it
          float s[128];
#pragma unroll
          for (int k = 0; k < 128; ++k) s[k] = __uint_as_float(sr[k]);
          if (tile_needs_element_mask(mk, qt, j, kv_len)) {
            int lim = kv_len - j * kTile;
            if (mk.causal) {
              const int lc = row - j * kTile + 1;
              lim = lc < lim ? lc : lim;
            }
#pragma unroll
            for (int k = 0; k < 128; ++k)
              if (k >= lim) s[k] = -INFINITY;
          }
          float mx[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = fmaxf(s[2 * k], s[2 * k + 1]);
#pragma unroll
          for (int k = 16; k < 128; k += 16)
#pragma unroll
            for (int a = 0; a < 8; ++a) mx[a] = fmax3(mx[a], s[k + 2 * a], s[k + 2 * a + 1]);
          const float m_tile = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                     fmaxf(mx[6], mx[7])) *
                               c_log2;
          const float m_new = fmaxf(m_ref, m_tile);
          const bool grow = m_new > m_ref + kF8Rescale;
          float alpha = 1.f;
          if (grow) {
            alpha = ex2_approx(m_ref - m_new);
            l_sum *= alpha;
            m_ref = m_new;
          }
          const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref - kF8POffset;
          const uint64_t nm2 = f2_pack(-m_use, -m_use);
          uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
          uint32_t pk[32];  // 128 e4m3 codes, four per word, key order
          // P row into shared memory, 128-byte swizzle: 16-byte chunk ch at ch ^ (t & 7).
          // Chunks are stored while the exponentials of the later ones run; the
          // buffer is free once the previous PV of this tile is done, which is
          // awaited halfway through the row (that PV has finished by then in
          // steady state).
          auto store_chunk = [&](int ch) {
            *reinterpret_cast<uint4*>(prow + ((ch ^ (t & 7)) << 4)) =
                make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
          };
          bool pv_ok = true;
#pragma unroll
          for (int e = 0; e < 128; e += 4) {
            float p0, p1, p2, p3;
            f2_unpack(f2_fma(f2_pack(s[e], s[e + 1]), c2, nm2), p0, p1);
            f2_unpack(f2_fma(f2_pack(s[e + 2], s[e + 3]), c2, nm2), p2, p3);
            p0 = ex2_approx(p0);
            p1 = ex2_approx(p1);
            p2 = ex2_approx(p2);
            p3 = ex2_approx(p3);
            rs2[(e >> 2) & 3] = f2_add(rs2[(e >> 2) & 3], f2_add(f2_pack(p0, p1), f2_pack(p2, p3)));
            pk[e >> 2] = e4m3x2(p0, p1) | (e4m3x2(p2, p3) << 16);
            if (e == 60) {  // first half formed: wait for the buffer, store chunks 0-3
              if (n_done > 0) {
                if (!mbar_wait_warp(bars.pv_done[x], pv_cnt & 1, tmo, abort_flag)) {
                  pv_ok = false;
                  break;
                }
                ++pv_cnt;
                tc_fence_after();
              }
#pragma unroll
              for (int ch = 0; ch < 4; ++ch) store_chunk(ch);
            } else if (e > 60 && (e & 15) == 12) {
              store_chunk(e >> 4);
            }
          }
          if (!pv_ok) {
            fail();
            ok = false;
            break;
          }
          {
            const uint64_t t2 = f2_add(f2_add(rs2[0], rs2[1]), f2_add(rs2[2], rs2[3]));
            float r0, r1;
            f2_unpack(t2, r0, r1);
            l_sum += r0 + r1;
          }
          if (n_done > 0 && __any_sync(0xffffffffu, grow)) {  // the previous PV is done
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tmem_st32(tO + c * 32, o);
            }
            tmem_st_wait();
          }
          fence_async_smem_writes();
          tc_fence_before();
          mbar_arrive(bars.p_full[x]);
          ++n_done;
        }
      }
      if (!ok) break;
      // ---- epilogue: O = acc * s_v / l, lse = (m + log2 l - 5) ln 2
      if (n_done > 0) {
        if (!mbar_wait_warp(bars.pv_done[x], pv_cnt & 1, tmo, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        ++pv_cnt;
      }
      tc_fence_after();
      const bool row_ok = row < N;
      const float inv = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
      const float* sv = args.s_v + static_cast<size_t>(uc.bhk) * 128;
      // O goes out 64 columns at a time: the warp puts its 32 rows x 128 bytes into
      // the rows of P_x it writes itself (free once its last PV has completed), then
      // stores them so that every instruction covers four whole 128-byte lines,
      // eight lanes per row, instead of 32 rows with 16 bytes each.
      const uint32_t stage = sP + static_cast<uint32_t>(x * L::kTileBytes + quad * 4096);
      const uint32_t srow = stage + static_cast<uint32_t>(lane * 128);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * h + cc;
          uint32_t o[32];
          if (n_done > 0) {
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = 0u;
          }
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            w[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv * sv[c * 32 + 2 * k],
                               __uint_as_float(o[2 * k + 1]) * inv * sv[c * 32 + 2 * k + 1]);
#pragma unroll
          for (int k = 0; k < 4; ++k)  // 16-byte unit 4 cc + k, swizzled by the row
            st_shared_v4(srow + static_cast<uint32_t>(((4 * cc + k) ^ (lane & 7)) << 4), w[4 * k],
                         w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
        }
        __syncwarp();
        const int u = lane & 7;  // 16-byte unit of the row this lane stores
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 4 * i + (lane >> 3);  // row within the warp's 32
          const uint4 val = ld_shared_v4(stage + static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4)));
          const int orow_i = (uc.qt0 + x) * kTile + quad * 32 + r;
          if (orow_i < N)
            *reinterpret_cast<uint4*>(
                args.o + (static_cast<size_t>(uc.bh) * N + static_cast<size_t>(orow_i)) * 128 +
                64 * h + 8 * u) = val;
        }
        __syncwarp();  // the staging rows are written again by the next half
      }
      if (row_ok)
        args.lse[static_cast<size_t>(uc.bh) * N + row] =
            (l_sum > 0.f) ? (m_ref - kF8POffset + __log2f(l_sum)) * kLn2 : -INFINITY;
      tc_fence_before();
      mbar_arrive(bars.o_free[x]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kF8MmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const Fp8FwdArgs& a, int num_sms, cudaStream_t stream) {
  const int n_q = (a.mask.N + kTile - 1) / kTile;
  const long long units = static_cast<long long>(a.mask.B) * a.mask.H * ((n_q + 1) / 2);
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  if (grid <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fa_fwd_fp8_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, F8L::kSmemBytes);
  if (e != cudaSuccess) return e;
  fa_fwd_fp8_kernel<<<grid, kF8Threads, F8L::kSmemBytes, stream>>>(tq, tk, tvt, a);
  return cudaGetLastError();
}

}  // namespace fa
