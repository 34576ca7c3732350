/*
 * fa.h — C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * The library computes exact scaled-dot-product attention the IO-aware way:
 * the forward pass streams K/V tiles through on-chip memory, keeps a running
 * row maximum and sum (online softmax) and writes only O and the per-row
 * logsumexp; the backward pass recomputes S and P on chip from that
 * logsumexp and produces dQ, dK and dV without writing any N x N matrix to
 * device memory.  (FlashAttention deep-read report, sections 2.4 "tiling and
 * incremental softmax", 2.5 "recomputation", 3.2 "Algorithm 1" and 3.3
 * "backward pass and memory layout"; Attention Kernel page, "FlashAttention's
 * insight: IO-aware" and "why tiling also works for training".)
 *
 * Conventions shared by every entry point
 *   - q, k, v, o, dout, dq, dk, dv: bf16, contiguous, layout [B, H, N, d]
 *     (row-major; element (b,h,i,c) at ((b*H + h)*N + i)*d + c). Device
 *     pointers, 16-byte aligned. A [B, N, H, d] tensor must be transposed
 *     by the caller first.
 *   - lse: fp32 [B, H, N], natural-log logsumexp of the scaled scores of each
 *     query row (this replaces the pair (m, l) that the pages store); a row
 *     with no allowed key gets -inf and O = 0 for that row.
 *   - d (head dimension) must be 64 or 128; N >= 1; B, H >= 1;
 *     B*H*N < 2^31.
 *   - scale > 0 multiplies Q K^T (the usual value is 1/sqrt(d)).
 *   - causal != 0 masks key j for query i when j > i (square, top-left aligned).
 *   - seqlens_k (nullable): device int32 [B]; keys j >= seqlens_k[b] are
 *     masked for every query row of batch b (key padding; query rows are still
 *     computed). Values are clamped to [0, N].
 *   - block_mask (nullable): device uint8 [nb, nb], nb = ceil(N / 128), row
 *     major, shared by all (b, h): a zero byte at (r, c) removes every pair
 *     with query block r and key block c (FlashAttention deep-read report,
 *     sections 2.6 and 3.5, block-sparse attention; blocks are 128 x 128).
 *     The C entry points receive only the two pointers and cannot check the
 *     sizes of these arrays: a shorter seqlens_k or block_mask makes the
 *     kernels read past its end. (The Python binding checks both shapes.)
 *   - dropout_p in [0, 1): dropout on the normalised probabilities, applied
 *     on chip (deep-read report section 3.2). It is quantised to
 *     p8 = round(256 p) and the effective rate is p8/256 (see fa_dropout_p8).
 *     Element (b,h,i,j) is dropped iff byte (j & 15) of
 *       Philox4x32-10(counter = (j >> 4, (b*H + h)*N + i, lo32(offset), hi32(offset)),
 *                     key = (lo32(seed), hi32(seed)))
 *     is below p8 (byte index j&15 = word (j&15)>>2, little-endian byte j&3),
 *     Philox as published by Salmon, Moraes, Dror and Shaw (SC'11). Kept
 *     elements are scaled by 1/(1 - p8/256). fa_fwd and fa_bwd must be given
 *     the same seed and offset. The logsumexp is that of the undropped softmax.
 *   - stream: a cudaStream_t (NULL = legacy default stream). Every call is
 *     asynchronous on that stream; the return value reports argument errors
 *     and launch failures only.
 *   - The library never allocates device memory. The caller owns every buffer.
 *   - Device-side failures (a bounded wait that ran out) are recorded in a
 *     per-device status word; fa_device_status() reads and optionally clears it.
 */
#ifndef FA_GB300_H_
#define FA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null/unaligned pointer, bad size, bad value */
  FA_ERR_UNSUPPORTED = 2, /* head dimension other than 64/128, not an sm_100-family GPU */
  FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, attribute) */
  FA_ERR_WORKSPACE = 4,   /* workspace missing or smaller than fa_bwd_workspace_size() */
  FA_ERR_TIMEOUT = 5      /* a device-side wait ran out (reported by fa_device_status) */
} fa_status;

/* Forward pass: O = softmax(scale * Q K^T, masked) V, plus lse.
 * Writes o [B,H,N,d] bf16 and lse [B,H,N] fp32 (both device). */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, float dropout_p, uint64_t seed,
                 uint64_t offset, const uint8_t* block_mask, const int32_t* seqlens_k,
                 void* stream);

/* Bytes of device workspace fa_bwd needs (the per-row D = rowsum(dO * O), fp32 [B,H,N],
 * rounded up to 256 bytes). */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/* Backward pass of L = sum(O * dO) for the forward above. o and lse are the
 * forward's outputs for the same inputs and options. Writes dq, dk, dv
 * (bf16 [B,H,N,d], device). workspace: device, >= fa_bwd_workspace_size(),
 * 16-byte aligned; its contents on entry do not matter. Three kernels run in
 * order on `stream`: D = rowsum(dO * O); dK and dV (one pass over key tiles,
 * recomputing S^T and P^T); dQ (one pass over query tiles, recomputing S and P).
 * dQ is accumulated without atomics, so every output is deterministic. */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, float dropout_p, uint64_t seed, uint64_t offset,
                 const uint8_t* block_mask, const int32_t* seqlens_k, void* workspace,
                 size_t workspace_bytes, void* stream);

/* Grouped-query attention (query heads sharing K/V heads, which the page
 * "Attention Kernel: FlashAttention 与它的后继者", section on FlashAttention's
 * IO-aware insight, names as a further cut of K/V reads): H query heads and
 * H_kv K/V heads, H a multiple of H_kv, query head h of batch row b attending
 * with K/V head h / (H / H_kv).
 * q, o, dout, dq: bf16 [B,H,N,d]; k, v, dk, dv: bf16 [B,H_kv,N,d]; lse:
 * fp32 [B,H,N]. dk and dv of a K/V head are the sums over the query heads
 * that share it, formed on chip (the key-tile kernel walks every query head
 * of the group), so they stay atomic-free and deterministic. Dropout keys on
 * the query head, as for H independent heads. H_kv = H is fa_fwd / fa_bwd;
 * H_kv = 1 is multi-query attention. Errors as for fa_fwd / fa_bwd, plus
 * FA_ERR_INVALID_ARG when H_kv < 1 or H % H_kv != 0. The workspace is
 * fa_bwd_workspace_size(B, H, N, d). */
fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int H_kv, int N, int d, float scale, int causal, float dropout_p,
                     uint64_t seed, uint64_t offset, const uint8_t* block_mask,
                     const int32_t* seqlens_k, void* stream);
fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int H_kv, int N,
                     int d, float scale, int causal, float dropout_p, uint64_t seed,
                     uint64_t offset, const uint8_t* block_mask, const int32_t* seqlens_k,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Sliding-window (local) attention, with every other option of fa_fwd_gqa /
 * fa_bwd_gqa: key j is visible to query i only if
 * i - window_left <= j <= i + window_right (-1 leaves that side unbounded);
 * it composes with causal (which caps j <= i), key padding and the block mask.
 * The cross-paper synthesis page on FlashAttention lists sliding-window
 * attention among the variants an IO-aware kernel should cover (section 5),
 * and the Attention Kernel page counts sliding windows among the sparse
 * patterns whose blocks are skipped (section on xFormers, cuDNN and sparse
 * attention). The kernels skip every 128 x 128 tile the band misses and mask
 * elements only on tiles an edge crosses, so the work is O(N * window).
 * Arguments, layouts, outputs and errors are those of fa_fwd_gqa /
 * fa_bwd_gqa, plus FA_ERR_INVALID_ARG when a window bound is below -1. */
fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int H_kv, int N, int d, float scale, int causal, int window_left,
                        int window_right, float dropout_p, uint64_t seed, uint64_t offset,
                        const uint8_t* block_mask, const int32_t* seqlens_k, void* stream);
fa_status fa_bwd_window(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                        int H, int H_kv, int N, int d, float scale, int causal, int window_left,
                        int window_right, float dropout_p, uint64_t seed, uint64_t offset,
                        const uint8_t* block_mask, const int32_t* seqlens_k, void* workspace,
                        size_t workspace_bytes, void* stream);

/* The three stages fa_bwd runs, for callers that schedule or time them
 * separately. They must run in this order on one stream with the same
 * workspace (it carries D from the first stage to the other two); dK/dV and
 * dQ are independent of each other once D exists.
 *   fa_bwd_preprocess: D = rowsum(dO * O) into the workspace.
 *   fa_bwd_dkdv:       dK, dV (one CTA owns each 128-row key tile).
 *   fa_bwd_dq:         dQ (one CTA owns each 128-row query tile). */
fa_status fa_bwd_preprocess(const void* o, const void* dout, int B, int H, int N, int d,
                            void* workspace, size_t workspace_bytes, void* stream);
fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dout,
                      const float* lse, void* dk, void* dv, int B, int H, int N, int d,
                      float scale, int causal, float dropout_p, uint64_t seed, uint64_t offset,
                      const uint8_t* block_mask, const int32_t* seqlens_k, void* workspace,
                      size_t workspace_bytes, void* stream);
fa_status fa_bwd_dq(const void* q, const void* k, const void* v, const void* dout,
                    const float* lse, void* dq, int B, int H, int N, int d, float scale,
                    int causal, float dropout_p, uint64_t seed, uint64_t offset,
                    const uint8_t* block_mask, const int32_t* seqlens_k, void* workspace,
                    size_t workspace_bytes, void* stream);

/* fa_bwd without a caller-provided workspace: for callers that cannot allocate
 * device memory themselves, such as plugins inside a host framework that owns
 * all device memory and offers them no workspace, or code that must not call
 * cudaMalloc / cudaFree because those can synchronise the device or fail under
 * a fixed memory budget. This entry point allocates nothing: D = rowsum(dO * O)
 * goes to a static device array of 2^22 floats (16 MiB) that every GPU loading
 * the library holds until the process exits. The pages have no counterpart of
 * this call; it exists only for such callers.
 *   - Arguments and outputs are exactly those of fa_bwd minus the workspace.
 *   - B*H*N above 2^22 (4,194,304 query rows) is rejected with FA_ERR_WORKSPACE
 *     before any device work.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address; make that first call before any stream capture.
 *   - All calls on a device share the one array. Its contents left by an earlier
 *     call do not matter (D is fully rewritten before it is read), but two calls
 *     whose kernels overlap on the GPU (different streams, or one device used
 *     from several threads without ordering) race on it: order them. */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, float scale, int causal, float dropout_p,
                         uint64_t seed, uint64_t offset, const uint8_t* block_mask,
                         const int32_t* seqlens_k, void* stream);

/* Short-query attention over a key/value cache (decode): Nq new query rows
 * per head attend over a cache of Nk keys, forward only. The page
 * "FlashAttention — L3 Cross-Paper Synthesis" (section 3) names this case,
 * bound by reading the K/V cache from HBM, as one the FlashAttention kernels
 * leave unoptimised. Query rows are the last Nq positions of each sequence:
 * row i of batch b sits at position L_b - Nq + i, where L_b = seqlens_k[b]
 * (clamped to [0, Nk]; Nk when seqlens_k is null). Without causal it sees
 * cache keys j < L_b; with causal, j <= L_b - Nq + i as well. A row that
 * sees no key gets O = 0 and lse = -inf. window_left >= 0 adds a sliding window:
 * row i sees only keys j >= L_b - Nq + i - window_left (cache tiles below every
 * row's window are not read); -1 for none.
 *   q, o:          bf16 [B, H, Nq, d], contiguous, 16-byte aligned (device)
 *   k_cache, v_cache: bf16 [B, H_kv, Nk, d], contiguous, 16-byte aligned
 *   lse:           fp32 [B, H, Nq], natural log (device)
 *   seqlens_k:     int32 [B] (device) or NULL
 *   H a multiple of H_kv (query head h reads K/V head h / (H / H_kv)), with
 *   (H / H_kv) * Nq <= 128: the query rows of a K/V group form one tile, so
 *   every K/V tile is read from HBM once per group. d = 64 or 128.
 *   num_ctas: number of CTAs the (K/V head, key tile) pairs are divided
 *   among in equal runs; 0 = automatic: whole K/V heads per CTA when that
 *   keeps at least 4/5 of the SMs busy, else one CTA per SM with heads cut
 *   between them. A K/V head cut between two CTAs is finished by a
 *   second, small kernel that merges the pieces' normalised outputs with the
 *   online softmax's merge rule; it needs the caller's workspace of
 *   fa_decode_workspace_size(...) bytes (16-byte aligned, device; 0 when no
 *   head is cut, and then workspace may be NULL). The result does not depend
 *   on num_ctas beyond fp32 rounding of the merge.
 * Errors: FA_ERR_INVALID_ARG (null or unaligned pointers, sizes < 1, H not a
 * multiple of H_kv, scale not positive and finite, num_ctas < 0,
 * window_left < -1),
 * FA_ERR_UNSUPPORTED (d not 64/128, (H / H_kv) * Nq > 128, not an sm_100-family
 * GPU), FA_ERR_WORKSPACE, FA_ERR_CUDA. Asynchronous on `stream`; nothing is
 * allocated. */
size_t fa_decode_workspace_size(int B, int H, int H_kv, int Nq, int Nk, int d, int num_ctas);
fa_status fa_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                    int B, int H, int H_kv, int Nq, int Nk, int d, float scale, int causal,
                    int window_left, const int32_t* seqlens_k, int num_ctas, void* workspace,
                    size_t workspace_bytes, void* stream);

/* FP8 forward with incoherent processing (FA-3's FP8 path, which the
 * cross-paper synthesis page on FlashAttention names in its section 2), head
 * dimension 128, forward only.
 * fa_fp8_quantize: Q' = Q M and K' = K M with M = diag(signs) H / sqrt(128),
 *   H the Sylvester Hadamard matrix (signs: fp32 [128] of +-1, device; NULL
 *   means no rotation), each stored as e4m3 codes with one scale per head,
 *   s = amax / 448 (1 for an all-zero head); V as e4m3 with one scale per
 *   (head, column), written transposed.
 *     q, k, v:  bf16 [B, H, N, 128] (device, 16-byte aligned)
 *     q8, k8:   uint8 [B, H, N, 128] (e4m3 codes, rounded to nearest even,
 *               saturating at 448)
 *     vt8:      uint8 [B, H, 128, Np], Np = fa_fp8_vt_stride(N) (N rounded up
 *               to 16; keys N .. Np-1 are written as zero)
 *     s_q, s_k: fp32 [B, H]; s_v: fp32 [B, H, 128]
 *     workspace: fa_fp8_workspace_size(B, H, 128) bytes (device, 16-byte aligned)
 * fa_fwd_fp8: attention of Q^ = dec(q8) s_q, K^ = dec(k8) s_k, V^ = dec(vt8)^T s_v
 *   (rotated Q and K give the same scores), both products on the tensor core
 *   in FP8 with fp32 accumulation; P is rounded to e4m3 for the PV product
 *   (kept between 2^5 and 2^8 at each row's maximum, so weights down to 2^-14
 *   of it are represented). Causal and key padding as fa_fwd. o: bf16
 *   [B, H, N, 128]; lse: fp32 [B, H, N] (natural log).
 * Accuracy contract (the exactness of fa_fwd does not carry over): against
 * exact attention of the dequantised inputs, |O - O^| <= 2^-4 sum_j P_ij |v^_j|
 * + 2^-15 sum_j |v^_j| (the e4m3 rounding of P, with underflow below 2^-9)
 * + 1.5 bf16 half-ulps of O; lse within 1e-3. Against the bf16 inputs the
 * error adds the quantisation of Q, K, V, which the rotation reduces when
 * channels carry outliers.
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED (d != 128), FA_ERR_WORKSPACE,
 * FA_ERR_CUDA. Asynchronous on `stream`; nothing is allocated. */
size_t fa_fp8_workspace_size(int B, int H, int d);
int fa_fp8_vt_stride(int N);
fa_status fa_fp8_quantize(const void* q, const void* k, const void* v, const float* signs, int B,
                          int H, int N, int d, void* q8, void* k8, void* vt8, float* s_q,
                          float* s_k, float* s_v, void* workspace, size_t workspace_bytes,
                          void* stream);
fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* s_q,
                     const float* s_k, const float* s_v, void* o, float* lse, int B, int H, int N,
                     int d, float scale, int causal, const int32_t* seqlens_k, void* stream);

/* Grouped K/V heads (H_kv dividing H; query head h of batch b uses K/V head
 * b H_kv + h / (H / H_kv), as fa_fwd_gqa): the same two calls with k, v, k8
 * shaped [B, H_kv, N, 128], vt8 [B, H_kv, 128, Np], s_k [B, H_kv] and s_v
 * [B, H_kv, 128]; q, q8, s_q, o and lse keep H. The workspace of
 * fa_fp8_workspace_size(B, H, 128) bytes also covers this case. fa_fp8_quantize
 * and fa_fwd_fp8 are these with H_kv = H. FA_ERR_INVALID_ARG also when H_kv < 1
 * or H is not a multiple of H_kv. */
fa_status fa_fp8_quantize_gqa(const void* q, const void* k, const void* v, const float* signs,
                              int B, int H, int H_kv, int N, int d, void* q8, void* k8, void* vt8,
                              float* s_q, float* s_k, float* s_v, void* workspace,
                              size_t workspace_bytes, void* stream);
fa_status fa_fwd_fp8_gqa(const void* q8, const void* k8, const void* vt8, const float* s_q,
                         const float* s_k, const float* s_v, void* o, float* lse, int B, int H,
                         int H_kv, int N, int d, float scale, int causal,
                         const int32_t* seqlens_k, void* stream);

/* Quantised dropout threshold round(256 p) used by fa_fwd / fa_bwd (-1 if p is
 * outside [0, 1)). The effective dropout rate is fa_dropout_p8(p) / 256. */
int fa_dropout_p8(float dropout_p);

/* Test hook: writes keep[b][h][i][j] (uint8 0/1, device, [B,H,N,N]) for the
 * dropout mask that fa_fwd / fa_bwd use with these arguments, computed by the
 * same device Philox code. */
fa_status fa_debug_dropout_keep(uint8_t* keep, int B, int H, int N, float dropout_p,
                                uint64_t seed, uint64_t offset, void* stream);

/* Test hook: raw Philox4x32-10 blocks from the device generator the kernels
 * use: out[4*t .. 4*t+3] = Philox(counter[4*t .. 4*t+3], key) for t < n.
 * counters and out are device uint32 arrays. */
fa_status fa_debug_philox(const uint32_t* counters, uint32_t* out, int n, uint32_t key0,
                          uint32_t key1, void* stream);

/* Host helper: the butterfly block mask (FlashAttention deep-read report,
 * sections 2.6 and 3.5, "fixed butterfly sparsity pattern"): with nb blocks per
 * side, mask[r*nb + c] = 1 iff r XOR c is 0 or a power of two below nb.
 * Writes nb*nb bytes to host memory. */
fa_status fa_butterfly_mask(uint8_t* mask_host, int nb);

/* Reads the status word of the current device after synchronising `stream`;
 * returns FA_OK or the first device-side error recorded since the last clear:
 * FA_ERR_TIMEOUT (a bounded wait ran out), or FA_ERR_CUDA when a kernel found
 * its launch unusable and returned without work (the d = 128 forward and the
 * d = 128 key-tile backward kernel use nearly all 227 KB of shared memory with
 * no alignment slack and check that their dynamic shared memory starts on a
 * 1024-byte boundary).
 * clear != 0 resets it to FA_OK.
 * The word is one per device, shared by every call on that device: the
 * forward entry points take no workspace to hold a per-call word. An error
 * recorded by a kernel on one stream is therefore seen by whichever caller
 * reads the word next, also from another stream or thread; callers that need
 * to attribute errors to one call must order their calls and read the word
 * between them. */
fa_status fa_device_status(void* stream, int clear);

/* Upper bound on every device-side wait, in nanoseconds (default 4e9). A wait
 * that runs out records FA_ERR_TIMEOUT and the kernel exits early. */
void fa_set_wait_timeout_ns(uint64_t ns);

/* Test hook for failure detection (host-side injection; nothing faults or
 * traps on the GPU). The armed launch waits on a barrier that nothing
 * completes, so its bounded wait runs out and the kernel returns with
 * FA_ERR_TIMEOUT recorded; the hook is consumed by that launch and later
 * launches run normally. mode selects the launch:
 *   1: the next forward-type kernel (fa_fwd and its _gqa / _window forms,
 *      fa_decode, fa_fwd_fp8, fa_fwd_fp8_gqa);
 *   2: the next dK/dV kernel (fa_bwd and its _gqa / _window / _noalloc forms,
 *      fa_bwd_dkdv);
 *   3: the next dQ kernel (the same backward calls, fa_bwd_dq).
 * mode 0 (or any other value) clears it. */
void fa_test_inject_stall(int mode);

/* Static description of an error code. */
const char* fa_status_string(fa_status s);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H_ */
