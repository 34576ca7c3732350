// Short-query attention over a key/value cache ("decode"): Nq new query rows
// per head attend over a cache of Nk keys. The page "FlashAttention — L3
// Cross-Paper Synthesis" (section 3) names this case as the one the
// FlashAttention kernels leave unoptimised: with one or a few query rows
// there is no N x N matrix to keep on chip, and the cost is reading the K/V
// cache from HBM. The kernels are built for that bound:
//  - the query rows of every query head of a K/V group (G = H / Hkv heads x
//    Nq rows, at most 128) form one 128-row query tile, so each K/V tile is
//    read from HBM once for the whole group;
//  - the (K/V head, key tile) pairs are cut into equal runs, one per CTA
//    (one CTA per SM), so every SM streams the same number of tiles and no
//    SM idles in a tail;
//  - a head cut by a run boundary is finished in pieces, each leaving its
//    normalised output and logsumexp; the combine kernel merges them with the
//    online softmax's rule for two blocks (Attention Kernel page, quiz answer
//    2; FlashAttention deep-read report, section 2.4).
//
// Per CTA: warp 4 is the TMA producer (the Q tile once per piece, K and V
// tiles through an NS-stage ring); warp 5 issues S = Q K^T (tcgen05.mma into
// one of three tensor-memory S buffers) and warp 6 issues O += P V (P read from
// tensor memory) as soon as the softmax has written P, so that neither kind of
// MMA waits behind the other's inputs; warps 0-3 run the online softmax with
// one thread per query row (only the warps that hold real rows take part).
// Tensor memory: S_0, S_1, S_2 (128 columns each, P written over S as bf16)
// and O (d columns); three S buffers let the S product of a tile start while
// the two before it are still in softmax or in their PV product.
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_decode.h"

namespace fa {

namespace {

constexpr int kDecThreads = 224;
constexpr int kDecProducerWarp = 4;
constexpr int kDecMmaWarp = 5;  // S issuer; allocates tensor memory
constexpr int kDecPvWarp = 6;   // PV issuer
constexpr int kDecMaxStages = 6;
constexpr float kDecRescale = 8.0f;  // log2 units: rescale O when m grows by > 2^8
constexpr uint32_t kSBufs = 3;       // S / P buffers in tensor memory
constexpr int kCombineWarps = 8;

template <int D>
struct DecL {
  static constexpr int kChunks = D / 64;                // 64-column (128-byte) swizzle chunks
  static constexpr int kTileBytes = kTile * D * 2;      // one 128 x D bf16 tile
  static constexpr int kStages = (D == 64) ? 6 : 3;     // K/V ring depth
  static_assert(kStages <= kDecMaxStages, "K/V ring deeper than its barrier arrays");
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  // q_full, q_empty, k/v full/empty rings, s_full[3], s_free[3], p_full[3],
  // o_full, o_free, drain, drain_pv, stall
  static constexpr int kNumBars = 2 + 4 * kDecMaxStages + 3 * kSBufs + 5;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;  // + slack for 1024-byte alignment
  static_assert(kSmemBytes <= 232448, "more shared memory than one CTA may hold");
  static constexpr uint32_t kColO = kSBufs * 128;  // after the S buffers
  static_assert(kColO + D <= 512, "tensor memory holds the S buffers and O");
};

struct DecBars {
  uint32_t q_full, q_empty;
  BarRun k_full, k_empty;
  BarRun v_full, v_empty;
  BarRun s_full, s_free, p_full;
  uint32_t o_full, o_free, drain, drain_pv, stall;
};

// One piece of a CTA's run: key tiles [j0, j1) of K/V head bkv (j1 already
// clipped to the valid cache length), the piece's index among those of its
// head and their number.
struct Piece {
  int bkv, j0, j1, seg, n_seg;
};

// Valid cache length of batch row b, clamped to [0, Nk].
__device__ __forceinline__ int cache_len(const DecodeArgs& a, int b) {
  if (a.seqlens_k == nullptr) return a.Nk;
  const int L = a.seqlens_k[b];
  return L < 0 ? 0 : (L > a.Nk ? a.Nk : L);
}

// The piece that starts at flattened position pos of CTA cta's run, which
// ends at hi; returns the position after it. Tiles below every row's sliding
// window (row 0 of the group sees the lowest keys) are left out of it.
__device__ __forceinline__ long long make_piece(const DecodeArgs& a, int cta, long long pos,
                                                long long hi, Piece& p) {
  const int bkv = static_cast<int>(pos / a.n_t);
  const long long head0 = static_cast<long long>(bkv) * a.n_t;
  const long long end = hi < head0 + a.n_t ? hi : head0 + a.n_t;
  const int c0 = static_cast<int>(head0 / a.per_cta);
  const int c1 = static_cast<int>((head0 + a.n_t - 1) / a.per_cta);
  const int L = cache_len(a, bkv / a.Hkv);
  const int n_valid = (L + kTile - 1) / kTile;
  p.bkv = bkv;
  p.j0 = static_cast<int>(pos - head0);
  p.j1 = static_cast<int>(end - head0);
  if (p.j1 > n_valid) p.j1 = n_valid;
  if (a.wl >= 0) {
    const int lo = L - a.Nq - a.wl;  // lowest key any row of the group sees
    const int jlo = lo > 0 ? lo / kTile : 0;
    if (p.j0 < jlo) p.j0 = jlo;
  }
  if (p.j1 < p.j0) p.j1 = p.j0;
  p.seg = cta - c0;
  p.n_seg = c1 - c0 + 1;
  return end;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kDecThreads, 1)
    fa_decode_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const DecodeArgs args) {
  using L = DecL<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = args.H / args.Hkv;
  const int M = G * args.Nq;  // real rows of the query tile
  const long long total = static_cast<long long>(args.B) * args.Hkv * args.n_t;
  const long long lo = static_cast<long long>(blockIdx.x) * args.per_cta;
  const long long hi = lo + args.per_cta < total ? lo + args.per_cta : total;

  uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff + 8);
  const int n_sw = (M + 31) / 32;  // softmax warps holding real rows

  DecBars bars;
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
    bars.k_full = run(kDecMaxStages);
    bars.k_empty = run(kDecMaxStages);
    bars.v_full = run(kDecMaxStages);
    bars.v_empty = run(kDecMaxStages);
    bars.s_full = run(kSBufs);
    bars.s_free = run(kSBufs);
    bars.p_full = run(kSBufs);
    bars.o_full = nb();
    bars.o_free = nb();
    bars.drain = nb();
    bars.drain_pv = nb();
    bars.stall = nb();
  }
  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bars.q_full, 1);
    mbar_init(bars.q_empty, 1);
    for (int s = 0; s < kDecMaxStages; ++s) {
      mbar_init(bars.k_full[s], 1);
      mbar_init(bars.k_empty[s], 1);
      mbar_init(bars.v_full[s], 1);
      mbar_init(bars.v_empty[s], 1);
    }
    for (uint32_t x = 0; x < kSBufs; ++x) {
      mbar_init(bars.s_full[x], 1);
      mbar_init(bars.s_free[x], 1);
      mbar_init(bars.p_full[x], 32 * n_sw);
    }
    mbar_init(bars.o_full, 1);
    mbar_init(bars.o_free, 32 * n_sw);
    mbar_init(bars.drain, 1);
    mbar_init(bars.drain_pv, 1);
    mbar_init(bars.stall, 1);
    fence_mbar_init();
  }
  if (warp == kDecMmaWarp) {
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

  if (warp == kDecProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t it = 0, k_arms = 0, v_arms = 0, q_arms = 0;
      bool ok = true;
      int np = 0;
      for (long long pos = lo; pos < hi && ok; ++np) {
        Piece pc;
        pos = make_piece(args, blockIdx.x, pos, hi, pc);
        if (np > 0 && !mbar_wait(bars.q_empty, (np - 1) & 1, tmo, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        mbar_expect_tx(bars.q_full, L::kTileBytes);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sQ + c * 16384, &tm_q, c * 64, pc.bkv * M, 0, bars.q_full);
        ++q_arms;
        for (int j = pc.j0; j < pc.j1; ++j) {
          const int s = it % L::kStages;
          const uint32_t ph = (it / L::kStages) & 1u;
          if (!mbar_wait(bars.k_empty[s], ph ^ 1u, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          mbar_expect_tx(bars.k_full[s], L::kTileBytes);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(sK + s * L::kTileBytes + c * 16384, &tm_k, c * 64, j * kTile, pc.bkv,
                        bars.k_full[s]);
          ++k_arms;
          if (!mbar_wait(bars.v_empty[s], ph ^ 1u, tmo, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          mbar_expect_tx(bars.v_full[s], L::kTileBytes);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(sV + s * L::kTileBytes + c * 16384, &tm_v, c * 64, j * kTile, pc.bkv,
                        bars.v_full[s]);
          ++v_arms;
          ++it;
        }
      }
      // Drain: every load issued here must land before the CTA exits. Stage s
      // was armed for ring positions s, s + NS, ...; wait for the last one.
      for (int s = 0; s < L::kStages; ++s) {
        if (k_arms > static_cast<uint32_t>(s))
          mbar_wait(bars.k_full[s], ((k_arms - 1 - s) / L::kStages) & 1, tmo, nullptr);
        if (v_arms > static_cast<uint32_t>(s))
          mbar_wait(bars.v_full[s], ((v_arms - 1 - s) / L::kStages) & 1, tmo, nullptr);
      }
      if (q_arms) mbar_wait(bars.q_full, (q_arms - 1) & 1, tmo, nullptr);
    }
    __syncwarp();
  } else if (warp == kDecMmaWarp) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);  // S = Q K^T, both K-major
      constexpr uint64_t kStageStep = static_cast<uint64_t>(L::kTileBytes >> 4);
      const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sK, 16, 1024);
      uint32_t it = 0;
      bool ok = true;
      // Test hook: a barrier that nothing completes, so the bounded wait runs out.
      if (args.sync.inject_stall && !mbar_wait(bars.stall, 0, tmo, abort_flag)) ok = false;
      int np = 0;
      for (long long pos = lo; pos < hi && ok; ++np) {
        Piece pc;
        pos = make_piece(args, blockIdx.x, pos, hi, pc);
        if (!mbar_wait(bars.q_full, np & 1, tmo, abort_flag)) {
          ok = false;
          break;
        }
        for (int j = pc.j0; j < pc.j1; ++j) {
          const int s = it % L::kStages;
          const uint32_t x = it % kSBufs;
          if (!mbar_wait(bars.k_full[s], (it / L::kStages) & 1u, tmo, abort_flag)) {
            ok = false;
            break;
          }
          // S buffer x was last read as P by the PV kSBufs positions back.
          if (it >= kSBufs &&
              !mbar_wait(bars.s_free[x], ((it / kSBufs) - 1) & 1u, tmo, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dk = dK0 + static_cast<uint64_t>(s) * kStageStep;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
            mma_ss(tmem + x * 128u, dQ + off, dk + off, kIdS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bars.k_empty[s]);
          mma_commit(bars.s_full[x]);
          ++it;
        }
        if (!ok) break;
        mma_commit(bars.q_empty);  // Q may be replaced once these S products are done
      }
      if (!ok) fail();
      // Drain: every issued MMA must finish before tensor memory is released.
      mma_commit(bars.drain);
      mbar_wait(bars.drain, 0, tmo, nullptr);
    }
    __syncwarp();
  } else if (warp == kDecPvWarp) {
    // ------------------------------------------------------------ PV issuer
    if (lane == 0) {
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, D, 0, 1);  // O += P V, V MN-major
      constexpr uint64_t kStageStep = static_cast<uint64_t>(L::kTileBytes >> 4);
      const uint64_t dV0 = sdesc_sw128(sV, 16384, 1024);
      uint32_t it = 0;
      bool ok = true;
      int n_full = 0;  // pieces with at least one key tile so far (O handshakes)
      for (long long pos = lo; pos < hi && ok;) {
        Piece pc;
        pos = make_piece(args, blockIdx.x, pos, hi, pc);
        for (int j = pc.j0; j < pc.j1; ++j) {
          const int s = it % L::kStages;
          const uint32_t x = it % kSBufs;
          const bool first = j == pc.j0;
          if (!mbar_wait(bars.p_full[x], (it / kSBufs) & 1u, tmo, abort_flag) ||
              !mbar_wait(bars.v_full[s], (it / L::kStages) & 1u, tmo, abort_flag) ||
              // the epilogue of the previous piece with keys has read O
              (first && n_full > 0 &&
               !mbar_wait(bars.o_free, (n_full - 1) & 1, tmo, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dv = dV0 + static_cast<uint64_t>(s) * kStageStep;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + L::kColO, tmem + x * 128u + kk * 8,
                   dv + static_cast<uint64_t>((kk * 2048) >> 4), kIdPV,
                   (first && kk == 0) ? 0u : 1u);
          mma_commit(bars.v_empty[s]);
          mma_commit(bars.s_free[x]);  // also tells the softmax that this PV is done
          ++it;
        }
        if (!ok) break;
        if (pc.j1 > pc.j0) {
          mma_commit(bars.o_full);  // O of this piece is complete with its last PV
          ++n_full;
        }
      }
      if (!ok) fail();
      mma_commit(bars.drain_pv);
      mbar_wait(bars.drain_pv, 0, tmo, nullptr);
    }
    __syncwarp();
  } else if (warp < n_sw) {
    // ------------------------------------------------------------ softmax
    const int r = warp * 32 + lane;  // query-tile row = tensor-memory lane
    const bool real = r < M;
    const int i = r % args.Nq;       // query row within its head
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem + lane_base + L::kColO;
    const float c_log2 = args.scale_log2;
    uint32_t it = 0;
    bool ok = true;
    int np = 0;
    int n_full = 0;  // pieces with at least one key tile so far
    for (long long pos = lo; pos < hi && ok; ++np) {
      Piece pc;
      pos = make_piece(args, blockIdx.x, pos, hi, pc);
      const int Lb = cache_len(args, pc.bkv / args.Hkv);
      int vis = Lb;  // keys [key_lo, vis) are visible to this row
      if (args.causal) {
        const int lc = Lb - args.Nq + i + 1;
        vis = lc < vis ? lc : vis;
      }
      const int key_lo = args.wl >= 0 ? Lb - args.Nq + i - args.wl : 0;
      float m_ref = -INFINITY;  // reference maximum, scaled log2 units
      float l_sum = 0.f;        // running sum of exp2(s*c - m_ref)
      for (int j = pc.j0; j < pc.j1; ++j) {
        const uint32_t x = it % kSBufs;
        const uint32_t tS = tmem + lane_base + x * 128u;
        if (!mbar_wait_warp(bars.s_full[x], (it / kSBufs) & 1u, tmo, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, &sr[c * 32]);
        tmem_ld_wait();
        float s[128];
#pragma unroll
        for (int k = 0; k < 128; ++k) s[k] = __uint_as_float(sr[k]);
        const int lim = vis - j * kTile;     // keys [lo, lim) of this tile are visible
        const int lo = key_lo - j * kTile;
        if (lim < kTile || lo > 0) {
#pragma unroll
          for (int k = 0; k < 128; ++k)
            if (k >= lim || k < lo) s[k] = -INFINITY;
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
        const bool grow = m_new > m_ref + kDecRescale;
        float alpha = 1.f;
        if (grow) {
          alpha = ex2_approx(m_ref - m_new);  // 0 when m_ref = -inf
          l_sum *= alpha;
          m_ref = m_new;
        }
        // Rescale the O row once the PV of the previous tile has finished with
        // it (the s_free phase of its buffer; the PV before that on the same
        // buffer completed before this tile's S was issued).
        if (j > pc.j0 && __any_sync(0xffffffffu, grow)) {
          if (!mbar_wait_warp(bars.s_free[(it - 1) % kSBufs], ((it - 1) / kSBufs) & 1u, tmo,
                              abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
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
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        const uint64_t c2 = f2_pack(c_log2, c_log2);
        const uint64_t nm2 = f2_pack(-m_use, -m_use);
        uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            const int k = half * 64 + e;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[k], s[k + 1]), c2, nm2), x0, x1);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            rs2[(e >> 1) & 3] = f2_add(rs2[(e >> 1) & 3], f2_pack(p0, p1));
            pk[e >> 1] = pack_bf16x2(p0, p1);
          }
          tmem_st32(tS + half * 32, pk);  // P (bf16 pairs) over the S columns already read
        }
        {
          const uint64_t t2 = f2_add(f2_add(rs2[0], rs2[1]), f2_add(rs2[2], rs2[3]));
          float r0, r1;
          f2_unpack(t2, r0, r1);
          l_sum += r0 + r1;
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bars.p_full[x]);
        ++it;
      }
      if (!ok) break;
      // ---- epilogue: O / l and lse, final or one piece of a cut head
      const bool any = pc.j1 > pc.j0;
      if (any) {
        if (!mbar_wait_warp(bars.o_full, n_full & 1, tmo, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const size_t row = static_cast<size_t>(pc.bkv) * M + r;  // flat [B, H, Nq] row
      const float inv = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
      const float lse = (l_sum > 0.f) ? (m_ref + __log2f(l_sum)) * kLn2 : -INFINITY;
      const bool direct = pc.n_seg == 1;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (any) {
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0u;
        }
        if (!real) continue;
        if (direct) {
          uint4* dst = reinterpret_cast<uint4*>(args.o + row * D + c * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(o[8 * k + 2 * e]) * inv,
                                 __uint_as_float(o[8 * k + 2 * e + 1]) * inv);
            dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(
              args.o_part + (row * args.seg_max + pc.seg) * D + c * 32);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                 __uint_as_float(o[4 * k + 2]) * inv,
                                 __uint_as_float(o[4 * k + 3]) * inv);
        }
      }
      if (real) {
        if (direct)
          args.lse[row] = lse;
        else
          args.lse_part[row * args.seg_max + pc.seg] = lse;
      }
      if (any) {  // O may now be overwritten by the next piece's first PV
        tc_fence_before();
        mbar_arrive(bars.o_free);
        ++n_full;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kDecMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge of the pieces of each cut head, one warp per query row: with
// lse_s = m_s + ln l_s and normalised O_s, the whole-cache result is
// O = sum_s e^{lse_s - m} O_s / sum_s e^{lse_s - m}, lse = m + ln sum_s e^{lse_s - m},
// m = max_s lse_s (the two-block merge of the online softmax applied piecewise).
template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
    fa_decode_combine_kernel(const DecodeArgs a) {
  constexpr int kPer = D / 32;  // columns per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(a.B) * a.H * a.Nq;
  const long long row = static_cast<long long>(blockIdx.x) * kCombineWarps + warp;
  if (row >= rows) return;
  const int M = (a.H / a.Hkv) * a.Nq;
  const long long head0 = (row / M) * a.n_t;
  const int n_seg = static_cast<int>((head0 + a.n_t - 1) / a.per_cta - head0 / a.per_cta) + 1;
  if (n_seg == 1) return;  // finished by its only CTA
  const float* lp = a.lse_part + row * a.seg_max;
  float m = -INFINITY;
  for (int s = 0; s < n_seg; ++s) m = fmaxf(m, lp[s]);
  float acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
  float den = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < n_seg; ++s) {
      const float w = ex2_approx((lp[s] - m) * kLog2e);  // 0 for an empty piece
      den += w;
      const float* op = a.o_part + (row * a.seg_max + s) * D + lane * kPer;
      if constexpr (kPer == 4) {
        const float4 v = *reinterpret_cast<const float4*>(op);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
        acc[2] += w * v.z;
        acc[3] += w * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(op);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  __nv_bfloat16* dst = a.o + row * D + lane * kPer;
  if constexpr (kPer == 4) {
    uint2 w;
    w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0) a.lse[row] = den > 0.f ? m + __logf(den) : -INFINITY;
}

cudaError_t launch_decode(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecodeArgs& a, int d, int grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (d == 64) {
    auto kern = fa_decode_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DecL<64>::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kDecThreads, DecL<64>::kSmemBytes, stream>>>(tq, tk, tv, a);
  } else {
    auto kern = fa_decode_kernel<128>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DecL<128>::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kDecThreads, DecL<128>::kSmemBytes, stream>>>(tq, tk, tv, a);
  }
  return cudaGetLastError();
}

cudaError_t launch_decode_combine(const DecodeArgs& a, int d, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.B) * a.H * a.Nq;
  const long long blocks = (rows + kCombineWarps - 1) / kCombineWarps;
  if (blocks <= 0) return cudaSuccess;
  if (d == 64)
    fa_decode_combine_kernel<64><<<static_cast<unsigned>(blocks), kCombineWarps * 32, 0, stream>>>(a);
  else
    fa_decode_combine_kernel<128><<<static_cast<unsigned>(blocks), kCombineWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
