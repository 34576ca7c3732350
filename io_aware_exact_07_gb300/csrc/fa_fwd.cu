// Forward pass of exact attention on sm_103a: tiled S = Q K^T, online softmax
// with a running maximum m and sum l, O += P V, writing only O and the row
// logsumexp (FlashAttention deep-read report, sections 2.4 and 3.2; Attention
// Kernel page, "FlashAttention's insight: IO-aware").
//
// Design (per CTA, persistent over work units; one unit = one (b, h) head and
// a block of 256 query rows split into two 128-row query tiles "a" and "b"):
//   warp 8      TMA producer: Q_a, Q_b once per unit, then K_j / V_j tiles
//               through an NS-stage shared-memory ring (128-byte swizzle).
//   warp 9      MMA issuer (one elected lane): S_x = Q_x K_j^T with
//               tcgen05.mma (both operands in shared memory, fp32 accumulator
//               in tensor memory) and O_x += P_x V_j with P_x read from
//               tensor memory (bf16) and V_j from shared memory.
//   warps 0-3   softmax + correction for query tile a (thread = query row,
//   warps 4-7   ... and tile b): tcgen05.ld of the S row, masking, row max,
//               exp2-based probabilities, running sum, dropout, P written back
//               to tensor memory over S as bf16, in-place rescale of the O row
//               when the running maximum grows by more than 2^8; the epilogue
//               divides by l and writes O (bf16) and lse (fp32).
// The two query tiles ping-pong: while the softmax warps of one tile work,
// the tensor core runs the other tile's GEMMs. Tensor memory holds
// S_a, S_b (128 columns each) and O_a, O_b (d columns each).
//
// Loop order differs from the pages' Algorithm 1 (K/V outer, Q inner, O and
// (m, l) written back every step): here the query tile is outer and stays on
// chip, as the FlashAttention-2 summary on the cross-paper synthesis page
// describes, so O and (m, l) are written exactly once.
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

namespace {

constexpr int kFwdThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when m grows by > 2^8

template <int D>
struct FwdLayout {
  static constexpr int kChunks = D / 64;                 // 64-column (128-byte) swizzle chunks
  static constexpr int kTileBytes = kTile * D * 2;       // one 128 x D bf16 tile
  static constexpr int kStages = (D == 64) ? 4 : 2;      // K/V ring depth
  static constexpr int kQOff = 0;                        // Q_a, Q_b
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  // barriers: q_full[2], q_empty, k_full[S], k_empty[S], v_full[S], v_empty[S],
  //           s_full[2], p_full[2], o_full[2], o_free[2], drain, stall
  static constexpr int kNumBars = 2 + 1 + 4 * kStages + 8 + 2;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;  // + slack for 1024-byte alignment
  // tensor-memory columns
  __device__ static constexpr uint32_t col_s(int x) { return static_cast<uint32_t>(x) * 128u; }
  __device__ static constexpr uint32_t col_o(int x) { return 256u + static_cast<uint32_t>(x * D); }
};

struct Bars {
  uint32_t q_full[2], q_empty;
  uint32_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint32_t s_full[2], p_full[2], o_full[2], o_free[2];
  uint32_t drain, stall;
};

struct UnitCoord {
  int bh, b, h, qt0;  // qt0 = index of query tile a (tile b is qt0 + 1)
};

__device__ __forceinline__ UnitCoord decode_unit(int u, int BH, int H, int n_qblk, int causal) {
  UnitCoord c;
  // Heads are processed one after another so that concurrently running CTAs
  // share K/V tiles in L2; with a causal mask the longest query blocks of a
  // head come first.
  const int bh = u / n_qblk;
  int qb = u % n_qblk;
  if (causal) qb = n_qblk - 1 - qb;
  c.bh = bh;
  c.b = bh / H;
  c.h = bh % H;
  c.qt0 = 2 * qb;
  (void)BH;
  return c;
}

}  // namespace

template <int D, bool DROPOUT>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdArgs args) {
  using L = FwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const MaskParams& mk = args.mask;
  const int N = mk.N;
  const int BH = mk.B * mk.H;
  const int n_q = (N + kTile - 1) / kTile;
  const int n_qblk = (n_q + 1) / 2;
  const int n_units = BH * n_qblk;

  uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff + 8);

  Bars bars;
  {
    int i = 0;
    auto nb = [&]() { return smem_u32(&bar_mem[i++]); };
    bars.q_full[0] = nb();
    bars.q_full[1] = nb();
    bars.q_empty = nb();
    for (int s = 0; s < L::kStages; ++s) bars.k_full[s] = nb();
    for (int s = 0; s < L::kStages; ++s) bars.k_empty[s] = nb();
    for (int s = 0; s < L::kStages; ++s) bars.v_full[s] = nb();
    for (int s = 0; s < L::kStages; ++s) bars.v_empty[s] = nb();
    for (int x = 0; x < 2; ++x) bars.s_full[x] = nb();
    for (int x = 0; x < 2; ++x) bars.p_full[x] = nb();
    for (int x = 0; x < 2; ++x) bars.o_full[x] = nb();
    for (int x = 0; x < 2; ++x) bars.o_free[x] = nb();
    bars.drain = nb();
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
      mbar_init(bars.p_full[x], 128);
      mbar_init(bars.o_full[x], 1);
      mbar_init(bars.o_free[x], 128);
    }
    mbar_init(bars.drain, 1);
    mbar_init(bars.stall, 1);
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

  auto fail = [&](void) {
    *abort_flag = 1;
    record_error(args.sync.status, kStatusTimeout);
  };

  const uint32_t sQ = smem_u32(smem + L::kQOff);
  const uint32_t sK = smem_u32(smem + L::kKOff);
  const uint32_t sV = smem_u32(smem + L::kVOff);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0;          // K/V ring position (running over all units)
    uint32_t k_arms = 0, v_arms = 0;  // loads issued into the K / V rings
    uint32_t q_armed = 0;
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    int unit_count = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_count) {
      const UnitCoord uc = decode_unit(u, BH, mk.H, n_qblk, mk.causal);
      const int kv_len = kv_len_of(mk, uc.b);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      int jmax = n_kv;
      if (mk.causal && uc.qt0 + 2 < jmax) jmax = uc.qt0 + 2;
      if (unit_count > 0) {
        if (!mbar_wait_warp(bars.q_empty, (unit_count - 1) & 1, tmo, abort_flag)) {
          fail();
          ok = false;
          break;
        }
      }
      if (lane == 0) {
        for (int x = 0; x < 2; ++x) {
          mbar_expect_tx(bars.q_full[x], L::kTileBytes);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(sQ + x * L::kTileBytes + c * 16384, &tm_q, c * 64, (uc.qt0 + x) * kTile,
                        uc.bh, bars.q_full[x]);
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
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_3d(sK + s * L::kTileBytes + c * 16384, &tm_k, c * 64, j * kTile, uc.bh,
                          bars.k_full[s]);
          }
          ++k_arms;
          if (!mbar_wait_warp(bars.v_empty[s], ph ^ 1u, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_expect_tx(bars.v_full[s], L::kTileBytes);
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_3d(sV + s * L::kTileBytes + c * 16384, &tm_v, c * 64, j * kTile, uc.bh,
                          bars.v_full[s]);
          }
          ++v_arms;
          ++it;
        }
      }
    }
    // Drain: every load this warp issued must land before the CTA exits.
    // Stage s was armed for ring positions s, s + S, ...; wait for the last one.
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
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);  // S = Q K^T, both K-major
    constexpr uint32_t kIdPV = idesc_bf16_f32(128, D, 0, 1);   // O += P V, V MN-major
    uint32_t it = 0;
    uint32_t p_cnt[2] = {0, 0};
    bool ok = true;
    bool issued_any = false;
    const bool elected = (lane == 0);
    if (args.sync.inject_stall) {
      // Test hook: this barrier is never completed, so the bounded wait runs out.
      if (!mbar_wait_warp(bars.stall, 0, tmo, abort_flag)) {
        fail();
        ok = false;
      }
    }
    int unit_count = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_count) {
      const UnitCoord uc = decode_unit(u, BH, mk.H, n_qblk, mk.causal);
      const int kv_len = kv_len_of(mk, uc.b);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      int jmax = n_kv;
      if (mk.causal && uc.qt0 + 2 < jmax) jmax = uc.qt0 + 2;
      const uint32_t uph = unit_count & 1;
      if (!mbar_wait_warp(bars.q_full[0], uph, tmo, abort_flag) ||
          !mbar_wait_warp(bars.q_full[1], uph, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      bool pend[2] = {false, false};
      bool first_pv[2] = {true, true};
      int prev_stage = -1;
      uint32_t prev_ph = 0;

      // PV for the tile of query tile x that was S-issued at the previous ring position.
      auto flush_pv = [&](int x) -> bool {
        if (!pend[x]) return true;
        if (!mbar_wait_warp(bars.p_full[x], p_cnt[x] & 1, tmo, abort_flag)) return false;
        ++p_cnt[x];
        if (first_pv[x] && unit_count > 0) {
          if (!mbar_wait_warp(bars.o_free[x], (unit_count - 1) & 1, tmo, abort_flag)) return false;
        }
        tc_fence_after();
        if (elected) {
          const uint32_t vbase = sV + prev_stage * L::kTileBytes;
          const uint64_t dv0 = sdesc_sw128(vbase, 16384, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            mma_ts(tmem + L::col_o(x), tmem + L::col_s(x) + kk * 8,
                   dv0 + static_cast<uint64_t>((kk * 2048) >> 4), kIdPV,
                   (first_pv[x] && kk == 0) ? 0u : 1u);
          }
        }
        __syncwarp();
        first_pv[x] = false;
        pend[x] = false;
        return true;
      };

      for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
        const uint32_t va = warp_valid_bits(mk, uc.qt0, chunk, n_q, n_kv);
        const uint32_t vb = warp_valid_bits(mk, uc.qt0 + 1, chunk, n_q, n_kv);
        uint32_t bits = va | vb;
        while (bits != 0u) {
          const int bit = __ffs(bits) - 1;
          bits &= bits - 1;
          const bool valid[2] = {((va >> bit) & 1u) != 0u, ((vb >> bit) & 1u) != 0u};
          const int s = it % L::kStages;
          const uint32_t ph = (it / L::kStages) & 1u;
          if (!mbar_wait_warp(bars.k_full[s], ph, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          if (prev_stage >= 0) {
            if (!mbar_wait_warp(bars.v_full[prev_stage], prev_ph, tmo, abort_flag)) {
              fail();
              ok = false;
              break;
            }
          }
          tc_fence_after();
          bool had_pv = pend[0] || pend[1];
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!ok) break;
            if (!flush_pv(x)) {
              fail();
              ok = false;
              break;
            }
            if (valid[x]) {
              if (elected) {
                const uint32_t qb = sQ + x * L::kTileBytes;
                const uint32_t kb = sK + s * L::kTileBytes;
                const uint64_t dq0 = sdesc_sw128(qb, 16, 1024);
                const uint64_t dk0 = sdesc_sw128(kb, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                  mma_ss(tmem + L::col_s(x), dq0 + (off >> 4), dk0 + (off >> 4), kIdS,
                         kk > 0 ? 1u : 0u);
                }
                mma_commit(bars.s_full[x]);
              }
              __syncwarp();
              pend[x] = true;
              issued_any = true;
            }
          }
          if (!ok) break;
          if (elected) {
            if (had_pv) mma_commit(bars.v_empty[prev_stage]);
            mma_commit(bars.k_empty[s]);
          }
          __syncwarp();
          prev_stage = s;
          prev_ph = ph;
          ++it;
        }
      }
      if (!ok) break;
      // Flush the PVs of the last ring position, then release it.
      if (prev_stage >= 0) {
        if (!mbar_wait_warp(bars.v_full[prev_stage], prev_ph, tmo, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (ok && !flush_pv(x)) {
            fail();
            ok = false;
          }
        }
        if (!ok) break;
        if (elected) mma_commit(bars.v_empty[prev_stage]);
        __syncwarp();
      }
      // A query tile with no PV in this unit still consumes the epilogue
      // handshake of the previous unit.
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (ok && first_pv[x] && unit_count > 0) {
          if (!mbar_wait_warp(bars.o_free[x], (unit_count - 1) & 1, tmo, abort_flag)) {
            fail();
            ok = false;
          }
        }
      }
      if (!ok) break;
      if (elected) {
        mma_commit(bars.o_full[0]);
        mma_commit(bars.o_full[1]);
        mma_commit(bars.q_empty);
      }
      __syncwarp();
    }
    // Drain: all issued MMAs must finish before tensor memory is released.
    if (elected) mma_commit(bars.drain);
    __syncwarp();
    mbar_wait_warp(bars.drain, 0, tmo, nullptr);
    (void)issued_any;
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;                 // query tile within the unit (0 = a, 1 = b)
    const int quad = warp & 3;               // tensor-memory lane quadrant of this warp
    const int t = quad * 32 + lane;          // row within the query tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::col_s(x);
    const uint32_t tO = tmem + lane_base + L::col_o(x);
    const float c_log2 = args.scale_log2;
    uint32_t s_cnt = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++unit_count) {
      const UnitCoord uc = decode_unit(u, BH, mk.H, n_qblk, mk.causal);
      const int qt = uc.qt0 + x;
      const int row = qt * kTile + t;
      const int kv_len = kv_len_of(mk, uc.b);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      int jmax = n_kv;
      if (mk.causal && qt + 1 < jmax) jmax = qt + 1;
      float m_ref = -INFINITY;  // reference maximum, scaled log2 units
      float l_sum = 0.f;        // running sum of exp2(s*c - m_ref), undropped
      int n_done = 0;
      const uint32_t row_global = static_cast<uint32_t>(uc.bh) * static_cast<uint32_t>(N) +
                                  static_cast<uint32_t>(row);
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
          float s[128];
#pragma unroll
          for (int k = 0; k < 128; ++k) s[k] = __uint_as_float(sr[k]);
          if (tile_needs_element_mask(mk, qt, j, kv_len)) {
            int lim = kv_len - j * kTile;                 // keys [0, lim) of this tile are valid
            if (mk.causal) {
              const int lc = row - j * kTile + 1;       // causal: key <= row
              lim = lc < lim ? lc : lim;
            }
#pragma unroll
            for (int k = 0; k < 128; ++k)
              if (k >= lim) s[k] = -INFINITY;
          }
          float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
          for (int k = 4; k < 128; k += 4) {
            mx0 = fmaxf(mx0, s[k]);
            mx1 = fmaxf(mx1, s[k + 1]);
            mx2 = fmaxf(mx2, s[k + 2]);
            mx3 = fmaxf(mx3, s[k + 3]);
          }
          const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c_log2;
          const float m_new = fmaxf(m_ref, m_tile);
          const bool grow = m_new > m_ref + kRescaleThreshold;
          float alpha = 1.f;
          if (grow) {
            alpha = ex2_approx(m_ref - m_new);  // 0 when m_ref = -inf
            l_sum *= alpha;
            m_ref = m_new;
          }
          const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
          // P = exp2(s*c - m_ref), summed (undropped) into l, dropout applied,
          // packed to bf16 and stored over S, 64 columns at a time.
          float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t pk[32];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const int k0 = half * 64 + g * 16;
              uint32_t w[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
              if constexpr (DROPOUT) {
                const uint4 keep = dropout_keep16(args.drop, row_global,
                                                  static_cast<uint32_t>(j * 8 + half * 4 + g));
                w[0] = keep.x;
                w[1] = keep.y;
                w[2] = keep.z;
                w[3] = keep.w;
              }
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                float p0 = ex2_approx(fmaf(s[k0 + e], c_log2, -m_use));
                float p1 = ex2_approx(fmaf(s[k0 + e + 1], c_log2, -m_use));
                rs0 += p0;
                rs1 += p1;
                if constexpr (DROPOUT) {
                  p0 = ((w[e >> 2] >> (8 * (e & 3))) & 0xFFu) ? p0 : 0.f;
                  p1 = ((w[(e + 1) >> 2] >> (8 * ((e + 1) & 3))) & 0xFFu) ? p1 : 0.f;
                }
                pk[g * 8 + (e >> 1)] = pack_bf16x2(p0, p1);
              }
            }
            tmem_st32(tS + half * 32, pk);
          }
          l_sum += rs0 + rs1;
          // Rescale the O row in tensor memory (warp-collective loads/stores).
          if (n_done > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tmem_st32(tO + c * 32, o);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bars.p_full[x]);
          ++n_done;
        }
      }
      if (!ok) break;
      // ---- epilogue: O = acc * keep_scale / l, lse = (m + log2 l) * ln 2
      if (!mbar_wait_warp(bars.o_full[x], unit_count & 1, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      tc_fence_after();
      const bool row_ok = row < N;
      const float inv = (l_sum > 0.f) ? args.drop.keep_scale / l_sum : 0.f;
      __nv_bfloat16* orow =
          args.o + (static_cast<size_t>(uc.bh) * N + static_cast<size_t>(row)) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (n_done > 0) {
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          pk[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
      }
      if (row_ok) {
        const float lse = (l_sum > 0.f) ? (m_ref + __log2f(l_sum)) * kLn2 : -INFINITY;
        args.lse[static_cast<size_t>(uc.bh) * N + row] = lse;
      }
      tc_fence_before();
      mbar_arrive(bars.o_free[x]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool DROPOUT>
static cudaError_t launch_fwd_impl(const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const FwdArgs& a, int grid,
                                   cudaStream_t stream) {
  using L = FwdLayout<D>;
  auto kern = fa_fwd_kernel<D, DROPOUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       L::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kFwdThreads, L::kSmemBytes, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, int d, bool dropout, int num_sms, cudaStream_t stream) {
  const int n_q = (a.mask.N + kTile - 1) / kTile;
  const long long units = static_cast<long long>(a.mask.B) * a.mask.H * ((n_q + 1) / 2);
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  if (grid <= 0) return cudaSuccess;
  if (d == 64) {
    return dropout ? launch_fwd_impl<64, true>(tq, tk, tv, a, grid, stream)
                   : launch_fwd_impl<64, false>(tq, tk, tv, a, grid, stream);
  }
  return dropout ? launch_fwd_impl<128, true>(tq, tk, tv, a, grid, stream)
                 : launch_fwd_impl<128, false>(tq, tk, tv, a, grid, stream);
}

}  // namespace fa
