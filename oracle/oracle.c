/*
 * Oracle for exact scaled-dot-product attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * CPU definition that the GPU kernels are checked against. Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it;
 * the library's own code path never does. It shares no code, header or table
 * with the CUDA sources.
 *
 * What it computes (fp64 throughout, inputs are bf16 values widened exactly):
 *
 *   Standard attention ("Algorithm 0" in the deep-read report on FlashAttention,
 *   section 3.1): S = Q K^T, P = softmax(S), O = P V, evaluated directly from
 *   that definition with no tiling and no online softmax. The fused options
 *   that the same report lists for the one-kernel forward (section 3.2: masking
 *   and dropout done on chip) are applied as plain element-wise steps:
 *
 *     allowed(i,j) = [!causal || j <= i] && [j < L_b] && [block_mask[i/128][j/128]]
 *                    && [wl < 0 || j >= i - wl] && [wr < 0 || j <= i + wr]
 *
 *   The last two factors are the sliding (local) window: a key is visible to a
 *   query only within wl positions before it and wr after it (a negative value
 *   leaves that side unbounded). The cross-paper synthesis page on
 *   FlashAttention lists sliding-window attention among the variants an
 *   IO-aware kernel should cover (section 5), and the Attention Kernel page
 *   counts sliding windows among the sparse patterns whose blocks are skipped
 *   (its section on xFormers, cuDNN and sparse attention).
 *     s_ij   = scale * q_i . k_j                          (allowed pairs only)
 *     lse_i  = m_i + ln sum_j exp(s_ij - m_i),   m_i = max_j s_ij
 *     P_ij   = exp(s_ij - lse_i)                          (0 where not allowed)
 *     O_i    = sum_j P_ij * Z_ij / (1 - p8/256) * v_j
 *
 *   lse is the natural-log row statistic that replaces the pair (m, l) the
 *   report says the forward keeps (section 2.5); a fully masked row has O = 0
 *   and lse = -inf.
 *
 *   Backward of L = sum(O * dO), the analytic gradient of the definition above
 *   (the report's section 3.3 says the backward rebuilds S and P and forms dP,
 *   dS and the gradients of Q, K and V; the formulas are the calculus of the
 *   softmax):
 *     dV_j  = sum_i P_ij Z_ij/(1-p) dO_i
 *     dP_ij = Z_ij/(1-p) * (dO_i . v_j)
 *     D_i   = sum_j P_ij dP_ij
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale * sum_j dS_ij k_j
 *     dK_j  = scale * sum_i dS_ij q_i
 *   To avoid storing N x N matrices the definition is evaluated in two passes:
 *   one over query rows (lse_i, D_i, dQ_i) and one over key rows (dK_j, dV_j),
 *   each recomputing s_ij from q and k. Every quantity is still the literal
 *   formula above.
 *
 *   Dropout mask Z (the pages only say dropout is fused on chip; the counter
 *   mapping is this library's documented choice): Philox4x32-10 as published
 *   by Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as
 *   1, 2, 3" (SC'11), with
 *     key     = (lo32(seed), hi32(seed))
 *     counter = (j >> 4, r, lo32(offset), hi32(offset)),  r = (b*H + h)*N + i
 *   The 16 output bytes (word w = (j&15)>>2, byte (j&3), little endian) serve
 *   the 16 columns of that group; Z_ij = 0 (dropped) iff byte < p8, where
 *   p8 = round(256 p) and the keep scale is 1/(1 - p8/256).
 *
 *   Butterfly block mask ("fixed butterfly sparsity", report section 2.6 and
 *   3.5): with nb = ceil(N/128) blocks per side, block (r, c) is kept iff
 *   r XOR c is 0 or a power of two below nb.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BLOCK 128

/* ------------------------------------------------------------------ Philox */

/* Philox4x32 round and key schedule, from the SC'11 paper's definition:
 * two 32x32->64 multiplies by the round multipliers, outputs permuted and
 * xored with the key; the key is bumped by the Weyl constants between rounds. */
static const uint32_t PHILOX_M0 = 0xD2511F53u;
static const uint32_t PHILOX_M1 = 0xCD9E8D57u;
static const uint32_t PHILOX_W0 = 0x9E3779B9u;
static const uint32_t PHILOX_W1 = 0xBB67AE85u;

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    uint64_t prod0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
    uint64_t prod1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* Dropout threshold in 1/256 units: round(256 p), computed in double. */
int oracle_p8(double p) { return (int)floor(p * 256.0 + 0.5); }

/* Z_ij for one element: 1 = kept, 0 = dropped. */
static int keep_bit(int b, int h, int i, int j, int H, int N, int p8, uint64_t seed,
                    uint64_t offset) {
  if (p8 <= 0) return 1;
  uint64_t r = ((uint64_t)b * (uint64_t)H + (uint64_t)h) * (uint64_t)N + (uint64_t)i;
  uint32_t ctr[4] = {(uint32_t)(j >> 4), (uint32_t)r, (uint32_t)offset,
                     (uint32_t)(offset >> 32)};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  int byte_index = j & 15;
  uint32_t word = out[byte_index >> 2];
  int byte = (int)((word >> (8 * (byte_index & 3))) & 0xFFu);
  return byte >= p8;
}

/* keep[n][i][j] for the listed heads (head n is batch head_b[n], head head_h[n]). */
void oracle_dropout_keep(uint8_t* keep, int n_heads, const int* head_b, const int* head_h, int H,
                         int N, int p8, uint64_t seed, uint64_t offset) {
  long total = (long)n_heads * N;
#pragma omp parallel for schedule(static)
  for (long t = 0; t < total; ++t) {
    int n = (int)(t / N), i = (int)(t % N);
    for (int j = 0; j < N; ++j)
      keep[t * (long)N + j] = (uint8_t)keep_bit(head_b[n], head_h[n], i, j, H, N, p8, seed, offset);
  }
}

/* --------------------------------------------------------------- butterfly */

void oracle_butterfly(uint8_t* mask, int nb) {
  for (int r = 0; r < nb; ++r)
    for (int c = 0; c < nb; ++c) {
      int x = r ^ c;
      int keep = (x == 0);
      for (int s = 1; s < nb; s <<= 1)
        if (x == s) keep = 1;
      mask[(long)r * nb + c] = (uint8_t)keep;
    }
}

/* --------------------------------------------------------------- attention */

typedef struct {
  int H, N, d, causal, p8;
  int wl, wr;  /* sliding window: keys i - wl .. i + wr (negative: unbounded) */
  double scale, keep_scale;
  uint64_t seed, offset;
  const uint8_t* block_mask;
  const int* seqlens_k;
  int nb;
} params_t;

static params_t make_params(int H, int N, int d, double scale, int causal, int p8, uint64_t seed,
                            uint64_t offset, const uint8_t* block_mask, const int* seqlens_k,
                            int wl, int wr) {
  params_t P;
  P.wl = wl;
  P.wr = wr;
  P.H = H;
  P.N = N;
  P.d = d;
  P.causal = causal;
  P.p8 = p8 > 0 ? p8 : 0;
  P.scale = scale;
  P.keep_scale = 1.0 / (1.0 - (double)P.p8 / 256.0);
  P.seed = seed;
  P.offset = offset;
  P.block_mask = block_mask;
  P.seqlens_k = seqlens_k;
  P.nb = (N + ORACLE_BLOCK - 1) / ORACLE_BLOCK;
  return P;
}

static int allowed(const params_t* P, int b, int i, int j) {
  if (P->causal && j > i) return 0;
  if (P->wl >= 0 && j < i - P->wl) return 0;
  if (P->wr >= 0 && j > i + P->wr) return 0;
  if (P->seqlens_k && j >= P->seqlens_k[b]) return 0;
  if (P->block_mask && !P->block_mask[(long)(i / ORACLE_BLOCK) * P->nb + (j / ORACLE_BLOCK)])
    return 0;
  return 1;
}

static double dot(const double* a, const double* b, int d) {
  double s = 0.0;
  for (int k = 0; k < d; ++k) s += a[k] * b[k];
  return s;
}

/* Row statistics of query row i of one head: fills s[j] for allowed j and
 * returns lse_i (-inf if no key is allowed). */
static double row_lse(const params_t* P, int b, int i, const double* qi, const double* kh,
                      double* s) {
  double m = -INFINITY;
  for (int j = 0; j < P->N; ++j) {
    if (!allowed(P, b, i, j)) continue;
    s[j] = P->scale * dot(qi, kh + (long)j * P->d, P->d);
    if (s[j] > m) m = s[j];
  }
  if (m == -INFINITY) return -INFINITY;
  double l = 0.0;
  for (int j = 0; j < P->N; ++j)
    if (allowed(P, b, i, j)) l += exp(s[j] - m);
  return m + log(l);
}

/* Forward: o [n_heads, N, d], lse [n_heads, N]. Tensors are [n_heads, N, d]. */
int oracle_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
               int n_heads, const int* head_b, const int* head_h, int H, int N, int d,
               double scale, int causal, int p8, uint64_t seed, uint64_t offset,
               const uint8_t* block_mask, const int* seqlens_k, int window_left,
               int window_right) {
  if (n_heads < 0 || N < 0 || d <= 0) return 1;
  params_t P = make_params(H, N, d, scale, causal, p8, seed, offset, block_mask, seqlens_k,
                           window_left, window_right);
  long total = (long)n_heads * N;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 8)
    for (long t = 0; t < total; ++t) {
      int n = (int)(t / N), i = (int)(t % N);
      int b = head_b[n], h = head_h[n];
      const double* qi = q + t * d;
      const double* kh = k + (long)n * N * d;
      const double* vh = v + (long)n * N * d;
      double* oi = o + t * d;
      for (int c = 0; c < d; ++c) oi[c] = 0.0;
      double L = row_lse(&P, b, i, qi, kh, s);
      lse[t] = L;
      if (L == -INFINITY) continue;
      for (int j = 0; j < N; ++j) {
        if (!allowed(&P, b, i, j)) continue;
        double p = exp(s[j] - L);
        if (!keep_bit(b, h, i, j, H, N, P.p8, seed, offset)) continue;
        double w = p * P.keep_scale;
        const double* vj = vh + (long)j * d;
        for (int c = 0; c < d; ++c) oi[c] += w * vj[c];
      }
    }
    free(s);
  }
  return 0;
}

/* Backward of L = sum(O * dO). Outputs dq, dk, dv [n_heads, N, d] and
 * D [n_heads, N] (D_i = sum_j P_ij dP_ij). */
int oracle_bwd(const double* q, const double* k, const double* v, const double* dout, double* dq,
               double* dk, double* dv, double* D, int n_heads, const int* head_b,
               const int* head_h, int H, int N, int d, double scale, int causal, int p8,
               uint64_t seed, uint64_t offset, const uint8_t* block_mask, const int* seqlens_k,
               int window_left, int window_right) {
  if (n_heads < 0 || N < 0 || d <= 0) return 1;
  params_t P = make_params(H, N, d, scale, causal, p8, seed, offset, block_mask, seqlens_k,
                           window_left, window_right);
  long total = (long)n_heads * N;
  double* lse = (double*)malloc(sizeof(double) * (total > 0 ? total : 1));
  if (!lse) return 2;
  /* Pass 1, over query rows i: lse_i, D_i and dQ_i. */
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (N > 0 ? N : 1));
    double* dp = (double*)malloc(sizeof(double) * (N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 8)
    for (long t = 0; t < total; ++t) {
      int n = (int)(t / N), i = (int)(t % N);
      int b = head_b[n], h = head_h[n];
      const double* qi = q + t * d;
      const double* doi = dout + t * d;
      const double* kh = k + (long)n * N * d;
      const double* vh = v + (long)n * N * d;
      double* dqi = dq + t * d;
      for (int c = 0; c < d; ++c) dqi[c] = 0.0;
      double L = row_lse(&P, b, i, qi, kh, s);
      lse[t] = L;
      D[t] = 0.0;
      if (L == -INFINITY) continue;
      double Di = 0.0;
      for (int j = 0; j < N; ++j) {
        if (!allowed(&P, b, i, j)) continue;
        double z = keep_bit(b, h, i, j, H, N, P.p8, seed, offset) ? P.keep_scale : 0.0;
        dp[j] = z * dot(doi, vh + (long)j * d, d);
        Di += exp(s[j] - L) * dp[j];
      }
      D[t] = Di;
      for (int j = 0; j < N; ++j) {
        if (!allowed(&P, b, i, j)) continue;
        double ds = exp(s[j] - L) * (dp[j] - Di);
        const double* kj = kh + (long)j * d;
        for (int c = 0; c < d; ++c) dqi[c] += scale * ds * kj[c];
      }
    }
    free(s);
    free(dp);
  }
  /* Pass 2, over key rows j: dK_j and dV_j. */
#pragma omp parallel for schedule(dynamic, 8)
  for (long t = 0; t < total; ++t) {
    int n = (int)(t / N), j = (int)(t % N);
    int b = head_b[n], h = head_h[n];
    const double* kj = k + t * d;
    const double* vj = v + t * d;
    const double* qh = q + (long)n * N * d;
    const double* doh = dout + (long)n * N * d;
    double* dkj = dk + t * d;
    double* dvj = dv + t * d;
    for (int c = 0; c < d; ++c) {
      dkj[c] = 0.0;
      dvj[c] = 0.0;
    }
    for (int i = 0; i < N; ++i) {
      if (!allowed(&P, b, i, j)) continue;
      long row = (long)n * N + i;
      if (lse[row] == -INFINITY) continue;
      const double* qi = qh + (long)i * d;
      const double* doi = doh + (long)i * d;
      double sij = scale * dot(qi, kj, d);
      double pij = exp(sij - lse[row]);
      double z = keep_bit(b, h, i, j, H, N, P.p8, seed, offset) ? P.keep_scale : 0.0;
      double dpij = z * dot(doi, vj, d);
      double dsij = pij * (dpij - D[row]);
      for (int c = 0; c < d; ++c) {
        dvj[c] += pij * z * doi[c];
        dkj[c] += scale * dsij * qi[c];
      }
    }
  }
  free(lse);
  return 0;
}
