// Forward pass of exact attention at head dimension 128 on sm_103a: the same
// tiled S = Q K^T, online softmax and O += P V as the d = 64 kernel, writing only
// O and the row logsumexp (FlashAttention deep-read report, sections 2.4 and 3.2;
// Attention Kernel page, "FlashAttention's insight: IO-aware").
//
// Design (per CTA, persistent over work units; one unit = one (b, h) head and
// one 128-row query tile):
//   warp 8      TMA producer: Q once per unit, then K_j through a two-stage ring.
//   warp 11     TMA producer: V_j through a two-stage ring.
//   warp 9      S issuer (one elected lane): S_g = Q K_j^T into tensor memory.
//   warp 10     PV issuer (one elected lane): O_g += P_g V_j, P_g and V_j both
//               read from shared memory.
//   warps 0-3   softmax warpgroup g = 0: the key tiles at even positions of the
//   warps 4-7   unit's tile list, and g = 1: those at odd positions (thread =
//               query row): tcgen05.ld of the S row, masking, row maximum,
//               exp2-based probabilities, running sum, dropout, P stored as bf16
//               into its own shared-memory buffer P_g (128-byte swizzle), and
//               in-place rescale of O_g when the reference maximum grows by more
//               than 2^8.
// Each warpgroup thus keeps a partial softmax state (m_g, l_g, O_g) over half of
// the keys. The epilogue merges the two: m = max(m_0, m_1),
// alpha_g = 2^(m_g - m), l = sum_g alpha_g l_g, O = sum_g alpha_g O_g / l, which
// is the block decomposition of the softmax normaliser (FlashAttention deep-read
// report, section 3.1) applied to two interleaved key sets.
//
// Why this shape at d = 128: tensor memory holds S_0, S_1, O_0, O_1 (4 x 128
// columns), so P cannot get a tensor-memory buffer of its own. With P in shared
// memory the next S of a warpgroup no longer waits for the PV that reads its P,
// and with both warpgroups on the same query tile their softmaxes overlap
// instead of alternating. Shared memory: Q (32 KB), K and V rings (2 x 2 x 32 KB)
// and P_0, P_1 (2 x 32 KB), 224 KB in all.
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

namespace {

constexpr int kD = 128;
constexpr int kQkProducerWarp = 8;
constexpr int kSIssuerWarp = 9;
constexpr int kPvIssuerWarp = 10;
constexpr int kVProducerWarp = 11;
constexpr int kThreads = 12 * 32;
// Registers per thread: 168 at launch; the producer and issuer warpgroup gives
// part of its share to the two softmax warpgroups.
constexpr int kRegsLaunch = 168;
constexpr int kRegsSoftmax = 200;
constexpr int kRegsAux = 96;
static_assert(8 * 32 * kRegsSoftmax + 4 * 32 * kRegsAux <= kThreads * kRegsLaunch,
              "register reallocation exceeds the block's launch allocation");
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when m grows by > 2^8

struct Layout {
  static constexpr int kTileBytes = kTile * kD * 2;  // one 128 x 128 bf16 tile
  static constexpr int kStages = 2;                  // K and V ring depth
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kPOff = kVOff + kStages * kTileBytes;  // P_0, P_1
  static constexpr int kBarOff = kPOff + 2 * kTileBytes;
  // barriers: q_full, q_empty, k_full[2], k_empty[2], v_full[2], v_empty[2],
  //           s_full[2], s_free[2], p_full[2], pv_done[2], o_free, xbar[4],
  //           drain, drain2, stall
  static constexpr int kNumBars = 26;
  // abort flag, tensor-memory address, units whose PVs are all issued
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kXchOff = kMiscOff + 16;            // (m, l) per warpgroup and row
  // No alignment slack: the kernel checks that the dynamic shared memory starts
  // on a 1024-byte boundary, which the swizzled tiles need.
  static constexpr int kSmemBytes = kXchOff + 2 * kTile * 8;
  static_assert(kSmemBytes <= 232448, "shared memory exceeds the per-block limit");
  // tensor-memory columns
  __device__ static constexpr uint32_t col_s(int g) { return 128u * static_cast<uint32_t>(g); }
  __device__ static constexpr uint32_t col_o(int g) {
    return 256u + 128u * static_cast<uint32_t>(g);
  }
};

struct Bars {
  uint32_t q_full, q_empty;
  BarRun k_full, k_empty, v_full, v_empty;  // ring stages
  BarRun s_full, s_free, p_full, pv_done;   // per softmax warpgroup
  uint32_t o_free;
  BarRun xbar;  // per tensor-memory lane quadrant: the epilogue's (m, l) exchange
  uint32_t drain, drain2, stall;
};

struct Unit {
  int bh, b, qt;
};

__device__ __forceinline__ Unit decode_unit(int u, int H, int n_q, int causal) {
  // Heads one after another, so that concurrently running CTAs share K/V tiles
  // in L2; with a causal mask the longest query tiles of a head come first.
  Unit c;
  c.bh = u / n_q;
  c.qt = u - c.bh * n_q;
  if (causal) c.qt = n_q - 1 - c.qt;
  c.b = c.bh / H;
  return c;
}

// Key tiles [0, jmax) can hold valid tiles of query tile qt.
__device__ __forceinline__ int key_tile_bound(const MaskParams& mk, int qt, int n_kv) {
  int jmax = n_kv;
  if (mk.causal && qt + 1 < jmax) jmax = qt + 1;
  return jmax;
}

}  // namespace

template <bool DROPOUT, bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FwdArgs args) {
  using L = Layout;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0u) {
    if (threadIdx.x == 0) record_error(args.sync.status, kStatusCuda);
    return;
  }
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
  // units (in this CTA's order) whose PVs have all been issued: a count, not a
  // barrier phase, since the PV issuer may run several units without key tiles
  // ahead of the S issuer
  volatile int* pv_units = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  Bars bars;
  {
    int i = 0;
    auto nb = [&]() { return smem_u32(&bar_mem[i++]); };
    auto run = [&](int n) {
      const BarRun r{smem_u32(&bar_mem[i])};
      i += n;
      return r;
    };
    bars.q_full = nb();
    bars.q_empty = nb();
    bars.k_full = run(2);
    bars.k_empty = run(2);
    bars.v_full = run(2);
    bars.v_empty = run(2);
    bars.s_full = run(2);
    bars.s_free = run(2);
    bars.p_full = run(2);
    bars.pv_done = run(2);
    bars.o_free = nb();
    bars.xbar = run(4);
    bars.drain = nb();
    bars.drain2 = nb();
    bars.stall = nb();
  }

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bars.q_full, 1);
    mbar_init(bars.q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bars.k_full[s], 1);
      mbar_init(bars.k_empty[s], 1);
      mbar_init(bars.v_full[s], 1);
      mbar_init(bars.v_empty[s], 1);
      mbar_init(bars.s_full[s], 1);
      mbar_init(bars.s_free[s], 128);
      mbar_init(bars.p_full[s], 128);
      mbar_init(bars.pv_done[s], 1);
    }
    // o_free: the 256 softmax threads at the end of each epilogue, plus the PV
    // issuer once per unit after its own wait on the previous phase, so that no
    // phase can complete while the PV issuer still waits on the one before it
    // (units without key tiles would otherwise let the epilogues run ahead).
    mbar_init(bars.o_free, 257);
    for (int q = 0; q < 4; ++q) mbar_init(bars.xbar[q], 64);
    *pv_units = 0;
    mbar_init(bars.drain, 1);
    mbar_init(bars.drain2, 1);
    mbar_init(bars.stall, 1);
    fence_mbar_init();
  }
  if (warp == kSIssuerWarp) {
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

  if (warp >= 8) {
    // producers and issuers: one warpgroup, which hands most of its registers
    // to the softmax warpgroups
    regs_dec<kRegsAux>();
    if (warp == kQkProducerWarp || warp == kVProducerWarp) {
      // ------------------------------------------------------------ producers
      const bool is_k = (warp == kQkProducerWarp);
      const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
      const BarRun full = is_k ? bars.k_full : bars.v_full;
      const BarRun empty = is_k ? bars.k_empty : bars.v_empty;
      const uint32_t sRing = is_k ? sK : sV;
      uint32_t it = 0, arms = 0, q_armed = 0;
      bool ok = true;
      if (lane == 0) {
        tma_prefetch_desc(tm);
        if (is_k) tma_prefetch_desc(&tm_q);
      }
      int unit_count = 0;
      for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
        const Unit uc = decode_unit(u, mk.H, n_q, mk.causal);
        const int kvh = kv_head(mk, uc.bh);
        const int n_kv = (kv_len_of(mk, uc.b) + kTile - 1) / kTile;
        const int jmax = key_tile_bound(mk, uc.qt, n_kv);
        if (is_k) {
          if (unit_count > 0 &&
              !mbar_wait_warp(bars.q_empty, (unit_count - 1) & 1, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_expect_tx(bars.q_full, L::kTileBytes);
            for (int c = 0; c < 2; ++c)
              tma_load_3d(sQ + c * 16384, &tm_q, c * 64, uc.qt * kTile, uc.bh, bars.q_full);
          }
          ++q_armed;
        }
        for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
          uint32_t bits = warp_valid_bits<WIN>(mk, uc.qt, chunk, n_q, n_kv);
          while (bits != 0u) {
            const int j = chunk * 32 + (__ffs(bits) - 1);
            bits &= bits - 1;
            const int s = it & 1;
            const uint32_t ph = (it >> 1) & 1u;
            if (!mbar_wait_warp(empty[s], ph ^ 1u, tmo, abort_flag)) {
              fail();
              ok = false;
              break;
            }
            if (lane == 0) {
              mbar_expect_tx(full[s], L::kTileBytes);
              for (int c = 0; c < 2; ++c)
                tma_load_3d(sRing + s * L::kTileBytes + c * 16384, tm, c * 64, j * kTile, kvh,
                            full[s]);
            }
            ++arms;
            ++it;
          }
        }
      }
      // Drain: every load this warp issued must land before the CTA exits.
      // Stage s was armed for ring positions s, s + 2, ...; wait for the last one.
      for (int s = 0; s < 2; ++s)
        if (arms > static_cast<uint32_t>(s))
          mbar_wait_warp(full[s], ((arms - 1 - s) >> 1) & 1, tmo, nullptr);
      if (q_armed) mbar_wait_warp(bars.q_full, (q_armed - 1) & 1, tmo, nullptr);
    } else if (warp == kSIssuerWarp) {
      // ------------------------------------------------------------ S issuer
      // Lane 0 alone waits and issues (tcgen05.mma issue blocks while the tensor
      // core's queue is full); the rest of the warp helps evaluate the tile
      // lists (one ballot per 32 key tiles).
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);  // S = Q K^T, both K-major
      constexpr uint64_t kStageStep = static_cast<uint64_t>(L::kTileBytes >> 4);
      const bool leader = (lane == 0);
      const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sK, 16, 1024);
      uint32_t it = 0, sf0 = 0, sf1 = 0;
      bool seen0 = false, seen1 = false;
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
        const Unit uc = decode_unit(u, mk.H, n_q, mk.causal);
        const int n_kv = (kv_len_of(mk, uc.b) + kTile - 1) / kTile;
        const int jmax = key_tile_bound(mk, uc.qt, n_kv);
        // The tensor core runs products in issue order: the next unit's S products
        // wait until the PV issuer has issued this unit's last PV, so that they
        // do not delay it (the softmax warpgroups' epilogue waits for that PV; they
        // need the next S only after the epilogue).
        if (leader) {
          bool ready = *pv_units >= unit_count;
          if (!ready) {
            const uint64_t t0 = globaltimer_ns();
            while (!(ready = *pv_units >= unit_count)) {
              if (*abort_flag || globaltimer_ns() - t0 > tmo) break;
              __nanosleep(64);  // leave issue slots to the softmax warps meanwhile
            }
          }
          if (!ready || !mbar_wait(bars.q_full, unit_count & 1, tmo, abort_flag)) {
            fail();
            ok = false;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        int pos = 0;  // position in the unit's tile list
        for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
          const uint32_t bits = warp_valid_bits<WIN>(mk, uc.qt, chunk, n_q, n_kv);
          if (leader) {
            uint32_t b = bits;
            int p = pos;
            while (b != 0u && ok) {
              b &= b - 1;
              const int g = p & 1;
              const int s = it & 1;
              const uint32_t ph = (it >> 1) & 1u;
              if (!mbar_wait(bars.k_full[s], ph, tmo, abort_flag)) {
                ok = false;
                break;
              }
              // S_g is free once its warpgroup has read the previous S_g.
              if (g == 0) {
                if (seen0 && !mbar_wait(bars.s_free[0], sf0++ & 1, tmo, abort_flag)) {
                  ok = false;
                  break;
                }
                seen0 = true;
              } else {
                if (seen1 && !mbar_wait(bars.s_free[1], sf1++ & 1, tmo, abort_flag)) {
                  ok = false;
                  break;
                }
                seen1 = true;
              }
              tc_fence_after();
              const uint64_t dk = dK0 + static_cast<uint64_t>(s) * kStageStep;
  #pragma unroll
              for (int kk = 0; kk < kD / 16; ++kk) {
                const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                mma_ss(tmem + L::col_s(g), dQ + off, dk + off, kIdS, kk > 0 ? 1u : 0u);
              }
              mma_commit(bars.s_full[g]);
              mma_commit(bars.k_empty[s]);
              ++it;
              ++p;
            }
            if (!ok) fail();
          }
          pos += __popc(bits);
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
    } else if (warp == kPvIssuerWarp) {
      // ------------------------------------------------------------ PV issuer
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, kD, 0, 1);  // P K-major, V MN-major
      constexpr uint64_t kStageStep = static_cast<uint64_t>(L::kTileBytes >> 4);
      const bool leader = (lane == 0);
      const uint64_t dP0 = sdesc_sw128(sP, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sV, 16384, 1024);
      uint32_t it = 0, pc0 = 0, pc1 = 0;
      bool ok = true;
      int unit_count = 0;
      for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
        const Unit uc = decode_unit(u, mk.H, n_q, mk.causal);
        const int n_kv = (kv_len_of(mk, uc.b) + kTile - 1) / kTile;
        const int jmax = key_tile_bound(mk, uc.qt, n_kv);
        // The first PV of a unit overwrites O_0 or O_1, which the previous unit's
        // epilogue reads: it waits for that epilogue (o_free).
        bool first_any = true, first0 = true, first1 = true;
        int pos = 0;
        for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
          const uint32_t bits = warp_valid_bits<WIN>(mk, uc.qt, chunk, n_q, n_kv);
          if (leader) {
            uint32_t b = bits;
            int p = pos;
            while (b != 0u && ok) {
              b &= b - 1;
              const int g = p & 1;
              const int s = it & 1;
              const uint32_t ph = (it >> 1) & 1u;
              // (selected by value: a reference to either counter would put both
              // in local memory)
              const uint32_t pc = g ? pc1 : pc0;
              if (!mbar_wait(bars.v_full[s], ph, tmo, abort_flag) ||
                  !mbar_wait(bars.p_full[g], pc & 1, tmo, abort_flag)) {
                ok = false;
                break;
              }
              if (g) ++pc1; else ++pc0;
              if (first_any) {
                if (unit_count > 0 &&
                    !mbar_wait(bars.o_free, (unit_count - 1) & 1, tmo, abort_flag)) {
                  ok = false;
                  break;
                }
                mbar_arrive(bars.o_free);
                first_any = false;
              }
              tc_fence_after();
              const bool first = g ? first1 : first0;
              const uint64_t dp = dP0 + static_cast<uint64_t>(g) * kStageStep;
              const uint64_t dv = dV0 + static_cast<uint64_t>(s) * kStageStep;
  #pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk) {
                const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                mma_ss(tmem + L::col_o(g), dp + off, dv + static_cast<uint64_t>((kk * 2048) >> 4),
                       kIdPV, (first && kk == 0) ? 0u : 1u);
              }
              if (g) first1 = false; else first0 = false;
              mma_commit(bars.pv_done[g]);
              mma_commit(bars.v_empty[s]);
              ++it;
              ++p;
            }
            if (!ok) fail();
          }
          pos += __popc(bits);
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        // A unit without any PV still consumes the previous epilogue's handshake
        // and adds its own arrival.
        if (leader && ok && first_any) {
          if (unit_count > 0 && !mbar_wait(bars.o_free, (unit_count - 1) & 1, tmo, abort_flag)) {
            fail();
            ok = false;
          } else {
            mbar_arrive(bars.o_free);
          }
        }
        if (leader && ok) *pv_units = unit_count + 1;  // this unit's PVs are all issued
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
    const int g = warp >> 2;                 // warpgroup: key tiles at positions p, p % 2 == g
    const int quad = warp & 3;               // tensor-memory lane quadrant of this warp
    const int t = quad * 32 + lane;          // row within the query tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::col_s(g);
    const uint32_t tO = tmem + lane_base + L::col_o(g);
    // This row of P_g, with the row's swizzle phase (t mod 8) in address bits 4-6:
    // 16-byte unit v of the row then sits at prow ^ (v << 4).
    const uint32_t prow = sP + static_cast<uint32_t>(g * L::kTileBytes + t * 128 + ((t & 7) << 4));
    float2* xch = reinterpret_cast<float2*>(smem + L::kXchOff);
    const float c_log2 = args.scale_log2;
    uint32_t s_cnt = 0, pv_cnt = 0;
    bool ok = true;
    int unit_count = 0;
    for (int u = sched_unit(0); u < n_units && ok; u = sched_unit(++unit_count)) {
      const Unit uc = decode_unit(u, mk.H, n_q, mk.causal);
      const int row = uc.qt * kTile + t;
      const int kv_len = kv_len_of(mk, uc.b);
      const int n_kv = (kv_len + kTile - 1) / kTile;
      const int jmax = key_tile_bound(mk, uc.qt, n_kv);
      // sliding window: keys [key_lo, key_hi) are visible to this row
      int key_lo = 0, key_hi = kv_len;
      if constexpr (WIN) {
        if (mk.causal && row + 1 < key_hi) key_hi = row + 1;
        if (mk.wr >= 0 && row + mk.wr + 1 < key_hi) key_hi = row + mk.wr + 1;
        if (mk.wl >= 0) key_lo = row - mk.wl;
      }
      float m_ref = -INFINITY;  // reference maximum, scaled log2 units
      float l_sum = 0.f;        // running sum of exp2(s*c - m_ref), undropped
      int n_done = 0;           // key tiles of this warpgroup
      int n_all = 0;            // key tiles of the unit (both warpgroups)
      const uint32_t row_global = static_cast<uint32_t>(uc.bh) * static_cast<uint32_t>(N) +
                                  static_cast<uint32_t>(row);
      for (int chunk = 0; chunk * 32 < jmax && ok; ++chunk) {
        uint32_t bits = warp_valid_bits<WIN>(mk, uc.qt, chunk, n_q, n_kv);
        while (bits != 0u) {
          const int j = chunk * 32 + (__ffs(bits) - 1);
          bits &= bits - 1;
          if ((n_all++ & 1) != g) continue;
          if (!mbar_wait_warp(bars.s_full[g], s_cnt & 1, tmo, abort_flag)) {
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
          // S is in registers: the next S of this warpgroup may be written over it.
          tc_fence_before();
          mbar_arrive(bars.s_free[g]);
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
          } else if (tile_needs_element_mask<WIN>(mk, uc.qt, j, kv_len)) {
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
          const float m_new = fmaxf(m_ref, mx_row * c_log2);
          const bool grow = m_new > m_ref + kRescaleThreshold;
          float alpha = 1.f;
          if (grow) {
            alpha = ex2_approx(m_ref - m_new);  // 0 when m_ref = -inf
            l_sum *= alpha;
            m_ref = m_new;
          }
          const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
          // P = exp2(s*c - m_ref), summed (undropped) into l, dropout applied,
          // packed to bf16 and stored into P_g, which the previous PV reads.
          const uint64_t c2 = f2_pack(c_log2, c_log2);
          const uint64_t nm2 = f2_pack(-m_use, -m_use);
          uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};  // four packed partial sums
          uint32_t pk[64];
          bool pv_ok = true;
          bool stored0 = false;  // first half already in P_g
#pragma unroll
          for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int k0 = half * 64 + q4 * 16;
              uint32_t w[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
              if constexpr (DROPOUT) {
                const uint4 keep = dropout_keep16(args.drop, row_global,
                                                  static_cast<uint32_t>(j * 8 + half * 4 + q4));
                w[0] = keep.x;
                w[1] = keep.y;
                w[2] = keep.z;
                w[3] = keep.w;
              }
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(s[k0 + e], s[k0 + e + 1]), c2, nm2), x0, x1);
                const float p0 = ex2_approx(x0);
                const float p1 = ex2_approx(x1);
                rs2[(e >> 1) & 3] = f2_add(rs2[(e >> 1) & 3], f2_pack(p0, p1));
                uint32_t pp = pack_bf16x2(p0, p1);
                // dropout: keep bytes e, e+1 (0x00 / 0xFF) widened to the two bf16 lanes
                if constexpr (DROPOUT) pp &= prmt(w[e >> 2], 0u, (e & 2) ? 0x3322u : 0x1100u);
                pk[half * 32 + q4 * 8 + (e >> 1)] = pp;
              }
            }
            // 128-byte swizzle: 16-byte unit v of the row's 64-key half h at v ^ (t & 7)
            auto store_half = [&](int h) {
#pragma unroll
              for (int v = 0; v < 8; ++v)
                st_shared_v4(
                    (prow ^ static_cast<uint32_t>(v << 4)) + static_cast<uint32_t>(h * 16384),
                    pk[h * 32 + 4 * v], pk[h * 32 + 4 * v + 1], pk[h * 32 + 4 * v + 2],
                    pk[h * 32 + 4 * v + 3]);
            };
            if (half == 0) {
              // The first half goes out now if the previous PV (which reads P_g)
              // has already completed; otherwise the second half's exponentials
              // come first and the wait moves to the end of the row.
              // (The sliding-window and dropout instances always wait here: their
              // extra per-row state makes the deferred path spill.)
              constexpr bool kAlwaysWait = WIN || DROPOUT;
              const bool ready =
                  n_done == 0 || kAlwaysWait ||
                  __all_sync(0xffffffffu, mbar_test_wait(bars.pv_done[g], pv_cnt & 1));
              if (ready) {
                if (n_done > 0) {
                  if (kAlwaysWait &&
                      !mbar_wait_warp(bars.pv_done[g], pv_cnt & 1, tmo, abort_flag)) {
                    pv_ok = false;
                    break;
                  }
                  ++pv_cnt;
                  tc_fence_after();
                }
                store_half(0);
                stored0 = true;
              }
            } else {
              if (!stored0) {
                if (!mbar_wait_warp(bars.pv_done[g], pv_cnt & 1, tmo, abort_flag)) {
                  pv_ok = false;
                  break;
                }
                ++pv_cnt;
                tc_fence_after();
                store_half(0);
              }
              store_half(1);
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
          // Rescale the O_g row in tensor memory (the previous PV has completed).
          if (n_done > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
            for (int c = 0; c < kD / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tmem_st32(tO + c * 32, o);
            }
            tmem_st_wait();
          }
          // P_g's generic-proxy stores become visible to the tensor core's reads.
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(bars.p_full[g]);
          ++n_done;
        }
      }
      if (!ok) break;
      // ---- epilogue: merge the two warpgroups' partial softmaxes.
      // This warpgroup's last PV has completed once its pv_done phase has.
      if (n_done > 0) {
        if (!mbar_wait_warp(bars.pv_done[g], pv_cnt & 1, tmo, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        ++pv_cnt;
      }
      // The exchange slots are reused once both warpgroups have finished the
      // previous unit's epilogue (o_free completes after every read of them).
      if (unit_count > 0 &&
          !mbar_wait_warp(bars.o_free, (unit_count - 1) & 1, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      xch[g * kTile + t] = make_float2(m_ref, l_sum);
      // The partner row (same lane quadrant, other warpgroup) arrives after its
      // own last PV has completed, so both O_0 and O_1 are final past this wait.
      mbar_arrive(bars.xbar[quad]);
      if (!mbar_wait_warp(bars.xbar[quad], unit_count & 1, tmo, abort_flag)) {
        fail();
        ok = false;
        break;
      }
      tc_fence_after();
      const float2 other = xch[(1 - g) * kTile + t];
      const float m0 = g ? other.x : m_ref, l0 = g ? other.y : l_sum;
      const float m1 = g ? m_ref : other.x, l1 = g ? l_sum : other.y;
      const bool has0 = (n_all + 1) / 2 > 0, has1 = n_all / 2 > 0;  // O_g was written
      const float m = fmaxf(m0, m1);
      const float a0 = (l0 > 0.f) ? ex2_approx(m0 - m) : 0.f;
      const float a1 = (l1 > 0.f) ? ex2_approx(m1 - m) : 0.f;
      const float l = a0 * l0 + a1 * l1;
      const float inv = (l > 0.f) ? args.drop.keep_scale / l : 0.f;
      const float w0 = a0 * inv, w1 = a1 * inv;
      const bool row_ok = row < N;
      // This warpgroup writes output columns [64 g, 64 g + 64) from both O_0 and O_1.
      // Each warp first puts its 32 rows x 128 bytes into shared memory (the rows of
      // P_g this warp itself writes, free once its last PV has completed), then
      // stores them so that every instruction covers four whole 128-byte lines,
      // eight lanes per row, instead of 32 rows with 16 bytes each. (The
      // sliding-window instance stores its rows directly: the staging makes it
      // spill.)
      constexpr bool kStaged = !WIN;
      __nv_bfloat16* orow =
          args.o + (static_cast<size_t>(uc.bh) * N + static_cast<size_t>(row)) * kD + 64 * g;
      const uint32_t stage = sP + static_cast<uint32_t>(g * L::kTileBytes + quad * 4096);
      const uint32_t srow = stage + static_cast<uint32_t>(lane * 128);
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 16 columns at a time (fewer live registers)
        const uint32_t col = 64u * static_cast<uint32_t>(g) + 16u * static_cast<uint32_t>(c);
        uint32_t o0[16], o1[16];
        if (has0) tmem_ld16(tmem + lane_base + L::col_o(0) + col, o0);
        if (has1) tmem_ld16(tmem + lane_base + L::col_o(1) + col, o1);
        tmem_ld_wait();
        uint32_t pk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float v0 = 0.f, v1 = 0.f;
          if (has0) {
            v0 = __uint_as_float(o0[2 * k]) * w0;
            v1 = __uint_as_float(o0[2 * k + 1]) * w0;
          }
          if (has1) {
            v0 = fmaf(__uint_as_float(o1[2 * k]), w1, v0);
            v1 = fmaf(__uint_as_float(o1[2 * k + 1]), w1, v1);
          }
          pk[k] = pack_bf16x2(v0, v1);
        }
        if constexpr (kStaged) {
          // 16-byte units 2 c and 2 c + 1 of the row, swizzled by the row (no bank
          // conflicts)
          st_shared_v4(srow + static_cast<uint32_t>(((2 * c) ^ (lane & 7)) << 4), pk[0], pk[1],
                       pk[2], pk[3]);
          st_shared_v4(srow + static_cast<uint32_t>(((2 * c + 1) ^ (lane & 7)) << 4), pk[4], pk[5],
                       pk[6], pk[7]);
        } else if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 16);
          dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      if constexpr (kStaged) {
        __syncwarp();
        const int u = lane & 7;  // 16-byte unit of the row this lane stores
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 4 * i + (lane >> 3);  // row within the warp's 32
          const uint4 val = ld_shared_v4(stage + static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4)));
          const int orow_i = uc.qt * kTile + quad * 32 + r;
          if (orow_i < N)
            *reinterpret_cast<uint4*>(args.o +
                                      (static_cast<size_t>(uc.bh) * N + static_cast<size_t>(orow_i)) *
                                          kD +
                                      64 * g + 8 * u) = val;
        }
      }
      if (row_ok && g == 0) {
        const float lse = (l > 0.f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
        args.lse[static_cast<size_t>(uc.bh) * N + row] = lse;
      }
      tc_fence_before();
      mbar_arrive(bars.o_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kSIssuerWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool DROPOUT>
static cudaError_t launch_fwd128_impl(const CUtensorMap& tq, const CUtensorMap& tk,
                                      const CUtensorMap& tv, const FwdArgs& a, int grid,
                                      cudaStream_t stream) {
  const bool win = a.mask.wl >= 0 || a.mask.wr >= 0;
  auto kern = win ? fa_fwd128_kernel<DROPOUT, true> : fa_fwd128_kernel<DROPOUT, false>;
  // The in-kernel register reallocation assumes kRegsLaunch registers per thread
  // at launch: with fewer, the softmax warpgroups' increase could never be
  // granted and would wait forever, so such a kernel is refused.
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.numRegs < kRegsLaunch || attr.maxThreadsPerBlock < kThreads)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, Layout::kSmemBytes, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

cudaError_t launch_fwd128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdArgs& a, bool dropout, int num_sms, cudaStream_t stream) {
  const int n_q = (a.mask.N + kTile - 1) / kTile;
  const long long units = static_cast<long long>(a.mask.B) * a.mask.H * n_q;
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);
  if (grid <= 0) return cudaSuccess;
  return dropout ? launch_fwd128_impl<true>(tq, tk, tv, a, grid, stream)
                 : launch_fwd128_impl<false>(tq, tk, tv, a, grid, stream);
}

}  // namespace fa
