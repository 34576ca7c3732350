// Shared device-side pieces of the attention kernels: launch parameters,
// tile validity (causal / key padding / block-sparse), the Philox dropout
// generator and the device status word.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kTile = 128;               // query / key tile edge (rows), and block-mask granularity
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device status codes (mirror fa_status in include/fa.h).
constexpr unsigned kStatusCuda = 3u;     // a launch found its configuration unusable
constexpr unsigned kStatusTimeout = 5u;

// A run of consecutive mbarriers (8 bytes each) addressed by index. An array of
// barrier addresses indexed by a ring stage would be placed in local memory, so
// every handshake would first load its barrier's address from there.
struct BarRun {
  uint32_t base;
  __device__ __forceinline__ uint32_t operator[](int i) const {
    return base + 8u * static_cast<uint32_t>(i);
  }
};

struct MaskParams {
  int B, H, N;
  int Hkv;                      // K/V heads (H for per-head attention; H / Hkv query heads share one)
  int nb;                       // ceil(N / 128): tiles per side, block-mask row length
  int causal;
  int wl, wr;                   // sliding window: keys i - wl .. i + wr visible (-1: unbounded)
  const uint8_t* block_mask;    // [nb, nb] or null
  const int32_t* seqlens_k;     // [B] or null
};

struct DropParams {
  int p8;                       // drop iff Philox byte < p8
  float keep_scale;             // 1 / (1 - p8 / 256)
  uint32_t seed_lo, seed_hi, off_lo, off_hi;
  // Philox round keys, (seed_lo + r W0, seed_hi + r W1) mod 2^32 for rounds
  // r = 0..9, filled on the host so that a kernel reads them as constant
  // operands instead of bumping the key every round.
  uint32_t rk_lo[10], rk_hi[10];
};

struct SyncParams {
  unsigned int* status;         // device status word (first error wins)
  unsigned long long timeout_ns;
  int inject_stall;             // test hook: wait on a barrier that never completes
};

__device__ __forceinline__ void record_error(unsigned int* status, unsigned code) {
  atomicCAS(status, 0u, code);
}

// K/V head of query head bh = b*H + h: grouped-query attention gives the H / Hkv
// query heads h of a group the K/V head h / (H / Hkv) of the same batch row.
__device__ __forceinline__ int kv_head(const MaskParams& m, int bh) {
  const int b = bh / m.H, h = bh - b * m.H;
  return b * m.Hkv + h / (m.H / m.Hkv);
}

// First query head bh = b*H + h of the group that shares K/V head bhk = b*Hkv + j;
// the group is the G = H / Hkv consecutive heads from there. With one query head
// per K/V head (GQA false) that is bhk itself.
template <bool GQA>
__device__ __forceinline__ int group_first_head(const MaskParams& m, int bhk) {
  if constexpr (!GQA) return bhk;
  return (bhk / m.Hkv) * m.H + (bhk % m.Hkv) * (m.H / m.Hkv);
}

// Number of valid keys of batch b (key padding clamps to [0, N]).
__device__ __forceinline__ int kv_len_of(const MaskParams& m, int b) {
  if (m.seqlens_k == nullptr) return m.N;
  int L = m.seqlens_k[b];
  return L < 0 ? 0 : (L > m.N ? m.N : L);
}

// Static schedule of the persistent kernels: in round k the CTAs take the
// positions [k G, k G + G) of the work list, G = gridDim.x, in forward order
// on even rounds and in reverse order on odd rounds. Every role of a CTA walks
// the same sequence. With a causal mask the work list is ordered longest unit
// first within each head, so a CTA that drew a long unit in one round draws a
// short one in the next and the per-CTA totals stay within a few percent of
// each other; head-major order keeps the CTAs of a round on a few heads, whose
// K/V tiles they then share in L2. Returns a position >= the list length once
// the CTA has no more work (positions grow with k).
// With rotate set, round k instead shifts the positions by k: the dK/dV work
// list under key padding has its empty units (key tiles past a batch row's
// length) at the same places in every head, so the alternation would hand some
// CTAs a key tile and its mirror, both often empty, in every round, and others
// none; rotating lets every CTA meet every key tile.
__device__ __forceinline__ int sched_unit(int k, bool rotate = false) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  if (rotate) return k * G + (c + k) % G;
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Whether the (query tile qt, key tile kt) pair has any allowed element.
// n_kv = ceil(kv_len / 128), n_q = ceil(N / 128). With a sliding window (WIN:
// a separate kernel instance, so that kernels without one keep their code)
// the pair is skipped when the band i - wl <= j <= i + wr misses the tile.
template <bool WIN = false>
__device__ __forceinline__ bool tile_valid(const MaskParams& m, int qt, int kt, int n_q,
                                           int n_kv) {
  if (qt >= n_q || kt >= n_kv) return false;
  if (m.causal && kt > qt) return false;
  if constexpr (WIN) {
    if (m.wl >= 0 && kt * kTile + (kTile - 1) + m.wl < qt * kTile) return false;
    if (m.wr >= 0 && kt * kTile > qt * kTile + (kTile - 1) + m.wr) return false;
  }
  if (m.block_mask != nullptr && m.block_mask[qt * m.nb + kt] == 0) return false;
  return true;
}

// Whether the pair needs a per-element mask (causal diagonal, key tile
// crossing kv_len, or a sliding-window edge inside the tile). Query rows
// beyond N are never written, so the query tail needs none.
template <bool WIN = false>
__device__ __forceinline__ bool tile_needs_element_mask(const MaskParams& m, int qt, int kt,
                                                        int kv_len) {
  if constexpr (WIN) {
    if (m.wl >= 0 && kt * kTile < qt * kTile + (kTile - 1) - m.wl) return true;
    if (m.wr >= 0 && kt * kTile + (kTile - 1) > qt * kTile + m.wr) return true;
  }
  return (m.causal && kt == qt) || ((kt + 1) * kTile > kv_len);
}

// Whether key j is inside query i's sliding window.
__device__ __forceinline__ bool in_window(const MaskParams& m, int i, int j) {
  return (m.wl < 0 || j >= i - m.wl) && (m.wr < 0 || j <= i + m.wr);
}

// Bits j in [32*c, 32*c + 32) that are valid for query tile qt, computed by a
// whole warp (one candidate per lane).
template <bool WIN = false>
__device__ __forceinline__ uint32_t warp_valid_bits(const MaskParams& m, int qt, int chunk,
                                                    int n_q, int n_kv) {
  const int lane = threadIdx.x & 31;
  const bool v = tile_valid<WIN>(m, qt, chunk * 32 + lane, n_q, n_kv);
  return __ballot_sync(0xffffffffu, v);
}

// Same, transposed: query tiles qt in [32*c, 32*c + 32) valid for key tile kt.
template <bool WIN = false>
__device__ __forceinline__ uint32_t warp_valid_bits_t(const MaskParams& m, int kt, int chunk,
                                                      int n_q, int n_kv) {
  const int lane = threadIdx.x & 31;
  const bool v = tile_valid<WIN>(m, chunk * 32 + lane, kt, n_q, n_kv);
  return __ballot_sync(0xffffffffu, v);
}

// ------------------------------------------------------------------ Philox
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC'11): ten rounds of two 32x32 -> 64-bit multiplies by the
// round multipliers, the high halves xored with the other counter words and
// the key, with the key advanced by the Weyl increments between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// The same generator with the round keys taken from DropParams.
__device__ __forceinline__ uint4 philox4x32_10_rk(uint4 c, const DropParams& d) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    // one widening multiply gives both halves of each 64-bit product
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c.x;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c.z;
    const uint32_t lo0 = static_cast<uint32_t>(p0), hi0 = static_cast<uint32_t>(p0 >> 32);
    const uint32_t lo1 = static_cast<uint32_t>(p1), hi1 = static_cast<uint32_t>(p1 >> 32);
    c = make_uint4(hi1 ^ c.y ^ d.rk_lo[r], lo1, hi0 ^ c.w ^ d.rk_hi[r], lo0);
  }
  return c;
}

// Byte permute: result byte i = byte sel.nibble[i] of the 8-byte value {b, a}
// (a = bytes 0-3); a nibble with bit 3 set replicates that byte's sign bit.
// Used to turn dropout keep bytes (0x00 / 0xFF) into lane masks.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Keep masks for the 16 keys [16*g, 16*g + 16) of query row `row_global`
// ((b*H + h)*N + i): each byte is 0xFF where the element is kept, 0 where dropped.
__device__ __forceinline__ uint4 dropout_keep16(const DropParams& d, uint32_t row_global,
                                                uint32_t key_group) {
  const uint4 r = philox4x32_10_rk(make_uint4(key_group, row_global, d.off_lo, d.off_hi), d);
  const uint32_t thr = static_cast<uint32_t>(d.p8) * 0x01010101u;
  // Per-byte unsigned compare x >= p8 in SWAR form: the subtraction of the low
  // seven bits cannot borrow across bytes (bit 7 of each minuend byte is set),
  // so bit 7 of each byte of dif is [low7(x) >= low7(p8)]; x >= p8 when x's
  // top bit is set and p8's is not, or when they agree and dif's is set. The
  // byte permute then spreads each byte's top bit to 0xFF or 0x00.
  auto ge = [thr](uint32_t x) {
    const uint32_t dif = (x | 0x80808080u) - (thr & 0x7F7F7F7Fu);
    const uint32_t top = (x & ~thr) | (~(x ^ thr) & dif);
    return prmt(top, 0u, 0xBA98u);
  };
  return make_uint4(ge(r.x), ge(r.y), ge(r.z), ge(r.w));
}

// bf16x2 helpers for the epilogues.
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) { return pack_bf16x2(lo, hi); }

}  // namespace fa
