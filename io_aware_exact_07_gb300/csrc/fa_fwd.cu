// Forward pass of exact attention at head dimension 64 on sm_103a: tiled
// S = Q K^T, online softmax with a running maximum m and sum l, O += P V,
// writing only O and the row logsumexp (FlashAttention deep-read report,
// sections 2.4 and 3.2; Attention Kernel page, "FlashAttention's insight:
// IO-aware"). Head dimension 128 has its own kernel (fa_fwd128.cu).
//
// Design (per CTA, persistent over work units; one unit = one (b, h) head and
// a block of 256 query rows split into two 128-row query tiles "a" and "b"):
//   warp 8      TMA producer: Q_a, Q_b once per unit, then K_j / V_j tiles
//               through a four-stage shared-memory ring (128-byte swizzle).
//   warp 9      S issuer (one elected lane): S_x = Q_x K_j^T with tcgen05.mma
//               (both operands in shared memory, fp32 accumulator in tensor
//               memory) as soon as the softmax has read the previous S_x.
//   warp 10     PV issuer (one elected lane): O_x += P_x V_j with P_x read
//               from tensor memory (bf16) and V_j from shared memory.
//   warps 0-3   softmax + correction for query tile a (thread = query row,
//   warps 4-7   ... and tile b): tcgen05.ld of the S row, masking, row max,
//               exp2-based probabilities, running sum, dropout, P written to
//               its own tensor-memory buffer as bf16, in-place rescale of the O
//               row when the running maximum grows by more than 2^8; the
//               epilogue divides by l and writes O (bf16) and lse (fp32).
// The two query tiles ping-pong: while the softmax warps of one tile work,
// the tensor core runs the other tile's GEMMs. Tensor memory holds S_a, S_b
// (128 columns each), P_a, P_b and O_a, O_b (64 columns each).
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

constexpr int kSoftmaxWarps = 8;  // two warpgroups, one per query tile
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kPvWarp = 10;  // second MMA issuer
// Warp 11 idles: it completes the third warpgroup, since registers move between
// whole warpgroups.
constexpr int kFwdThreads = 12 * 32;
// Registers per thread: 168 at launch (three warps per sub-partition); the
// producer and issuer warpgroup gives part of its share to the softmax warps,
// which hold a 128-score row and its packed probabilities.
constexpr int kRegsLaunch = 168;
constexpr int kRegsSoftmax = 200;
constexpr int kRegsAux = 96;
static_assert(kSoftmaxWarps * 32 * kRegsSoftmax + (kFwdThreads - kSoftmaxWarps * 32) * kRegsAux <=
                  kFwdThreads * kRegsLaunch,
              "register reallocation exceeds the block's launch allocation");
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when m grows by > 2^8

template <int D>
struct FwdLayout {
  static_assert(D == 64, "head dimension 128 runs the kernel of fa_fwd128.cu");
  static constexpr int kChunks = D / 64;                 // 64-column (128-byte) swizzle chunks
  static constexpr int kTileBytes = kTile * D * 2;       // one 128 x D bf16 tile
  static constexpr int kStages = 4;                      // K/V ring depth
  static constexpr int kQOff = 0;                        // Q_a, Q_b
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  // barriers: q_full[2], q_empty, k_full[S], k_empty[S], v_full[S], v_empty[S],
  //           s_full[2], p_full[2], o_free[2], s_free[2], pv_done[2], drain, drain2, stall
  static constexpr int kNumBars = 2 + 1 + 4 * kStages + 10 + 3;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // epilogue staging: 4 KB per softmax warp (its 32 rows of O, 128 bytes each)
  static constexpr int kStageOff = (kMiscOff + 64 + 127) / 128 * 128;
  static constexpr int kSmemBytes = kStageOff + 8 * 4096 + 1024;  // + slack for 1024-byte alignment
  // Tensor memory has room for a separate P buffer per query tile
  // (2 x (128 S + 64 P + 64 O) = 512 columns), so the next S can be computed
  // while the softmax still works on the current one.
  __device__ static constexpr uint32_t col_s(int x) { return static_cast<uint32_t>(x) * 128u; }
  __device__ static constexpr uint32_t col_p(int x) { return 256u + 64u * static_cast<uint32_t>(x); }
  __device__ static constexpr uint32_t col_o(int x) { return 384u + 64u * static_cast<uint32_t>(x); }
};

struct Bars {
  BarRun q_full;
  uint32_t q_empty;
  BarRun k_full, k_empty, v_full, v_empty;
  BarRun s_full, p_full, o_free;
  BarRun s_free, pv_done;
  uint32_t drain, drain2, stall;
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

template <int D, bool DROPOUT, bool WIN>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdArgs args) {
  using L = FwdLayout<D>;
  // Without dropout each half of P is stored as soon as it is formed; with
  // dropout (more live registers) both halves are stored at the end, which keeps
  // that instance free of spills.
  constexpr bool kEarlyP = !DROPOUT;
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
    bars.p_full = run(2);
    bars.o_free = run(2);
    bars.s_free = run(2);
    bars.pv_done = run(2);
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
      mbar_init(bars.p_full[x], 128);
      // o_free[x]: the 128 softmax threads of tile x at the end of each
      // epilogue, plus the PV issuer once per unit after its own wait on the
      // previous phase, so that no phase can complete while the PV issuer still
      // waits on the one before it (units without key tiles would otherwise let
      // the epilogues run ahead).
      mbar_init(bars.o_free[x], 129);
      mbar_init(bars.s_free[x], 128);
      mbar_init(bars.pv_done[x], 1);
    }
    mbar_init(bars.drain, 1);
    mbar_init(bars.drain2, 1);
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

  if (warp >= kSoftmaxWarps) {
    // producer, issuers and the idle warp: one warpgroup, which hands most of its
    // registers to the softmax warpgroups
    regs_dec<kRegsAux>();
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
      for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
        const UnitCoord uc = decode_unit(u, BH, mk.H, n_qblk, mk.causal);
        const int kvh = kv_head(mk, uc.bh);  // K/V head of this query head
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
          uint32_t bits = warp_valid_bits<WIN>(mk, uc.qt0, chunk, n_q, n_kv) |
                          warp_valid_bits<WIN>(mk, uc.qt0 + 1, chunk, n_q, n_kv);
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
                tma_load_3d(sK + s * L::kTileBytes + c * 16384, &tm_k, c * 64, j * kTile, kvh,
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
                tma_load_3d(sV + s * L::kTileBytes + c * 16384, &tm_v, c * 64, j * kTile, kvh,
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
      // ------------------------------------------------------------ S issuer
      // Lane 0 alone waits and issues: tcgen05.mma issue blocks while the tensor
      // core is busy (its queue is shallow), so every cycle this thread spends on
      // anything else is a tensor-core bubble. The rest of the warp only helps
      // evaluate the tile lists (one ballot per 32 key tiles).
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);  // S = Q K^T, both K-major
      constexpr uint64_t kStageStep = static_cast<uint64_t>(L::kTileBytes >> 4);
      const bool leader = (lane == 0);
      const uint64_t dQa = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dQb = sdesc_sw128(sQ + L::kTileBytes, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sK, 16, 1024);
      uint32_t it = 0;
      uint32_t sf_cnt0 = 0, sf_cnt1 = 0;
      bool s_seen0 = false, s_seen1 = false;
      bool ok = true;
      if (args.sync.inject_stall && leader) {
        // Test hook: this barrier is never completed, so the bounded wait runs out.
        if (!mbar_wait(bars.stall, 0, tmo, abort_flag)) {
          fail();
          ok = false;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      auto issue_S = [&](int x, int s) {
        const uint64_t dq = x ? dQb : dQa;
        const uint64_t dk = dK0 + static_cast<uint64_t>(s) * kStageStep;
  #pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          mma_ss(tmem + L::col_s(x), dq + off, dk + off, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bars.s_full[x]);
      };
      int unit_count = 0;
      for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
        const UnitCoord uc = decode_unit(u, BH, mk.H, n_qblk, mk.causal);
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
          const uint32_t va = warp_valid_bits<WIN>(mk, uc.qt0, chunk, n_q, n_kv);
          const uint32_t vb = warp_valid_bits<WIN>(mk, uc.qt0 + 1, chunk, n_q, n_kv);
          if (leader) {
            uint32_t bits = va | vb;
            while (bits != 0u && ok) {
              const int bit = __ffs(bits) - 1;
              bits &= bits - 1;
              const bool v0 = ((va >> bit) & 1u) != 0u, v1 = ((vb >> bit) & 1u) != 0u;
              const int s = it % L::kStages;
              const uint32_t ph = (it / L::kStages) & 1u;
              if (!mbar_wait(bars.k_full[s], ph, tmo, abort_flag)) {
                ok = false;
                break;
              }
              // S of this position as soon as the softmax has read the previous S
              // (the PVs come from the PV-issuer warp)
              if (v0) {
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
        // Q is free for the next unit once the last S of this one has completed.
        if (leader && ok) mma_commit(bars.q_empty);
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      // Drain: all issued MMAs must finish before tensor memory is released.
      if (leader) {
        mma_commit(bars.drain);
        mbar_wait(bars.drain, 0, tmo, nullptr);
      }
      __syncwarp();
    } else if (warp == kPvWarp) {
      // ------------------------------------------------------------ PV issuer
      // O_x += P_x V_j as soon as P_x of key tile j is ready, from a second
      // issuing thread, so that the tensor core keeps receiving work while the S
      // issuer waits on its own barriers. Its MMAs are tracked by its own commits
      // (pv_done, v_empty).
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, D, 0, 1);  // O += P V, V MN-major
      constexpr uint64_t kStageStep = static_cast<uint64_t>(L::kTileBytes >> 4);
      const bool leader = (lane == 0);
      const uint64_t dV0 = sdesc_sw128(sV, 16384, 1024);
      uint32_t it = 0, p_cnt0 = 0, p_cnt1 = 0;
      bool ok = true;
      int unit_count = 0;
      for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
        const UnitCoord uc = decode_unit(u, BH, mk.H, n_qblk, mk.causal);
        const int kv_len = kv_len_of(mk, uc.b);
        const int n_kv = (kv_len + kTile - 1) / kTile;
        int jmax = n_kv;
        if (mk.causal && uc.qt0 + 2 < jmax) jmax = uc.qt0 + 2;
        bool first0 = true, first1 = true;
        // The first PV of query tile x in a unit overwrites O_x, which the
        // previous unit's epilogue reads: it waits for that epilogue (o_free[x])
        // and adds this issuer's arrival for the current unit.
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
          const uint64_t dv = dV0 + static_cast<uint64_t>(s) * kStageStep;
  #pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + L::col_o(x), tmem + L::col_p(x) + kk * 8,
                   dv + static_cast<uint64_t>((kk * 2048) >> 4), kIdPV,
                   (first && kk == 0) ? 0u : 1u);
          mma_commit(bars.pv_done[x]);
          return true;
        };
        for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
          const uint32_t va = warp_valid_bits<WIN>(mk, uc.qt0, chunk, n_q, n_kv);
          const uint32_t vb = warp_valid_bits<WIN>(mk, uc.qt0 + 1, chunk, n_q, n_kv);
          if (leader) {
            uint32_t bits = va | vb;
            while (bits != 0u && ok) {
              const int bit = __ffs(bits) - 1;
              bits &= bits - 1;
              const bool v0 = ((va >> bit) & 1u) != 0u, v1 = ((vb >> bit) & 1u) != 0u;
              const int s = it % L::kStages;
              const uint32_t ph = (it / L::kStages) & 1u;
              if (!mbar_wait(bars.v_full[s], ph, tmo, abort_flag) || (v0 && !pv(0, s, first0)) ||
                  (v1 && !pv(1, s, first1))) {
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
          // A query tile without PV in this unit still consumes the epilogue
          // handshake of the previous unit and adds its arrival.
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
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;                 // query tile within the unit (0 = a, 1 = b)
    const int quad = warp & 3;               // tensor-memory lane quadrant of this warp
    const int t = quad * 32 + lane;          // row within the query tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::col_s(x);
    const uint32_t tP = tmem + lane_base + L::col_p(x);
    const uint32_t tO = tmem + lane_base + L::col_o(x);
    const float c_log2 = args.scale_log2;
    uint32_t s_cnt = 0;
    uint32_t pv_cnt = 0;  // PV completions consumed
    bool ok = true;
    int unit_count = 0;
    for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
      const UnitCoord uc = decode_unit(u, BH, mk.H, n_qblk, mk.causal);
      const int qt = uc.qt0 + x;
      const int row = qt * kTile + t;
      const int kv_len = kv_len_of(mk, uc.b);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      int jmax = n_kv;
      if (mk.causal && qt + 1 < jmax) jmax = qt + 1;
      // sliding window: keys [key_lo, key_hi) are visible to this row
      int key_lo = 0, key_hi = kv_len;
      if constexpr (WIN) {
        if (mk.causal && row + 1 < key_hi) key_hi = row + 1;
        if (mk.wr >= 0 && row + mk.wr + 1 < key_hi) key_hi = row + mk.wr + 1;
        if (mk.wl >= 0) key_lo = row - mk.wl;
      }
      float m_ref = -INFINITY;  // reference maximum, scaled log2 units
      float l_sum = 0.f;        // running sum of exp2(s*c - m_ref), undropped
      int n_done = 0;
      const uint32_t row_global = static_cast<uint32_t>(uc.bh) * static_cast<uint32_t>(N) +
                                  static_cast<uint32_t>(row);
      for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
        uint32_t bits = warp_valid_bits<WIN>(mk, qt, chunk, n_q, n_kv);
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
          // S is in registers: the next S may be written over it.
          tc_fence_before();
          mbar_arrive(bars.s_free[x]);
          float s[128];
#pragma unroll
          for (int k = 0; k < 128; ++k) s[k] = __uint_as_float(sr[k]);
          if constexpr (WIN) {
            if (j * kTile < key_lo || (j + 1) * kTile > key_hi) {  // this row's edge is in the tile
              const int lim = key_hi - j * kTile, lo = key_lo - j * kTile;  // keys [lo, lim) valid
#pragma unroll
              for (int k = 0; k < 128; ++k)
                if (k >= lim || k < lo) s[k] = -INFINITY;
            }
          } else if (tile_needs_element_mask<WIN>(mk, qt, j, kv_len)) {
            int lim = kv_len - j * kTile;                 // keys [0, lim) of this tile are valid
            if (mk.causal) {
              const int lc = row - j * kTile + 1;       // causal: key <= row
              lim = lc < lim ? lc : lim;
            }
#pragma unroll
            for (int k = 0; k < 128; ++k)
              if (k >= lim) s[k] = -INFINITY;
          }
          // Row maximum: three-input max over eight independent accumulators.
          float mx[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = fmaxf(s[2 * k], s[2 * k + 1]);
#pragma unroll
          for (int k = 16; k < 128; k += 16)
#pragma unroll
            for (int a = 0; a < 8; ++a) mx[a] = fmax3(mx[a], s[k + 2 * a], s[k + 2 * a + 1]);
          const float mx_row = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                     fmaxf(mx[6], mx[7]));
          const float m_tile = mx_row * c_log2;
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
          // packed to bf16 and stored over S, 64 columns at a time. The scale
          // and subtract and the row sum run on packed pairs of lanes.
          const uint64_t c2 = f2_pack(c_log2, c_log2);
          const uint64_t nm2 = f2_pack(-m_use, -m_use);
          uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};  // four packed partial sums
          uint32_t pk[64];
          bool pv_ok = true;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
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
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(s[k0 + e], s[k0 + e + 1]), c2, nm2), x0, x1);
                float p0 = ex2_approx(x0);
                float p1 = ex2_approx(x1);
                rs2[(e >> 1) & 3] = f2_add(rs2[(e >> 1) & 3], f2_pack(p0, p1));
                uint32_t pp = pack_bf16x2(p0, p1);
                // dropout: keep bytes e, e+1 (0x00 / 0xFF) widened to the two bf16 lanes
                if constexpr (DROPOUT) pp &= prmt(w[e >> 2], 0u, (e & 2) ? 0x3322u : 0x1100u);
                pk[half * 32 + g * 8 + (e >> 1)] = pp;
              }
            }
            if constexpr (kEarlyP) {
              // P has its own buffer, which the previous PV reads: once that PV
              // is done (long before, in steady state), store each half as soon
              // as it is formed so the store overlaps the next half's exponentials.
              if (half == 0 && n_done > 0) {
                if (!mbar_wait_warp(bars.pv_done[x], pv_cnt & 1, tmo, abort_flag)) {
                  pv_ok = false;
                  break;
                }
                ++pv_cnt;
                tc_fence_after();
              }
              tmem_st32(tP + half * 32, &pk[half * 32]);
            }
          }
          if constexpr (!kEarlyP) {
            // The previous PV reads the P buffer and accumulates into O: wait for it.
            if (n_done > 0) {
              if (!mbar_wait_warp(bars.pv_done[x], pv_cnt & 1, tmo, abort_flag)) {
                pv_ok = false;
              } else {
                ++pv_cnt;
                tc_fence_after();
              }
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
          if constexpr (!kEarlyP) {
            tmem_st32(tP, &pk[0]);
            tmem_st32(tP + 32, &pk[32]);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bars.p_full[x]);
          ++n_done;
        }
      }
      if (!ok) break;
      // ---- epilogue: O = acc * keep_scale / l, lse = (m + log2 l) * ln 2
      // the last PV of this unit has completed once its pv_done phase has
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
      const float inv = (l_sum > 0.f) ? args.drop.keep_scale / l_sum : 0.f;
      // The warp puts its 32 rows x 128 bytes of O into its own staging area, then
      // stores them so that every instruction covers four whole 128-byte lines,
      // eight lanes per row, instead of 32 rows with 16 bytes each.
      const uint32_t stage = smem_u32(smem + L::kStageOff) + static_cast<uint32_t>(warp * 4096);
      const uint32_t srow = stage + static_cast<uint32_t>(lane * 128);
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
#pragma unroll
        for (int k = 0; k < 4; ++k)  // 16-byte unit 4 c + k, swizzled by the row
          st_shared_v4(srow + static_cast<uint32_t>(((4 * c + k) ^ (lane & 7)) << 4), pk[4 * k],
                       pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      }
      __syncwarp();
      {
        const int u = lane & 7;  // 16-byte unit of the row this lane stores
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 4 * i + (lane >> 3);  // row within the warp's 32
          const uint4 val = ld_shared_v4(stage + static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4)));
          const int orow_i = qt * kTile + quad * 32 + r;
          if (orow_i < N)
            *reinterpret_cast<uint4*>(
                args.o + (static_cast<size_t>(uc.bh) * N + static_cast<size_t>(orow_i)) * D + 8 * u) =
                val;
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
  const bool win = a.mask.wl >= 0 || a.mask.wr >= 0;
  auto kern = win ? fa_fwd_kernel<D, DROPOUT, true> : fa_fwd_kernel<D, DROPOUT, false>;
  // The in-kernel register reallocation assumes kRegsLaunch registers per thread
  // at launch: with fewer, the softmax warpgroups' increase could never be
  // granted and would wait forever, so such a kernel is refused.
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.numRegs < kRegsLaunch || attr.maxThreadsPerBlock < kFwdThreads)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kFwdThreads, L::kSmemBytes, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, int d, bool dropout, int num_sms, cudaStream_t stream) {
  if (d == 128) return launch_fwd128(tq, tk, tv, a, dropout, num_sms, stream);
  const int n_q = (a.mask.N + kTile - 1) / kTile;
  const long long units = static_cast<long long>(a.mask.B) * a.mask.H * ((n_q + 1) / 2);
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  if (grid <= 0) return cudaSuccess;
  return dropout ? launch_fwd_impl<64, true>(tq, tk, tv, a, grid, stream)
                 : launch_fwd_impl<64, false>(tq, tk, tv, a, grid, stream);
}

}  // namespace fa
