/*
 * smla.h -- C ABI of libsmla: the FP8 lightning indexer, per-token top-k and
 * sparse MLA prefill attention for GB300 (sm_103a).
 *
 * Every entry point takes plain device pointers and sizes, validates them on
 * the host, enqueues its kernels asynchronously on `stream` and returns an
 * smla_status_t.  The caller owns every buffer; the library allocates no
 * device memory.  No C++ exception crosses this boundary.  A call that
 * returns anything but SMLA_OK has enqueued nothing (except SMLA_ERR_CUDA,
 * where a launch was attempted and failed); smla_last_error() then holds a
 * message for the calling thread.
 *
 * Errors found on the device (an index or page id outside the pool, a
 * pipeline wait that gave up) are recorded in a per-device error word
 * instead of faulting; the kernel that found them skips the offending
 * access and finishes.  smla_check_device_errors() reads and clears that
 * word.  Outputs of a call that recorded a device error are unspecified.
 *
 * Layouts are row-major and dense unless a stride is given.  "e4m3" is the
 * float8_e4m3fn byte format; "bf16" is bfloat16 bits.  Each call states the
 * alignment its pointers need; a misaligned pointer returns
 * SMLA_ERR_INVALID_ARG.
 */
#ifndef SMLA_H_
#define SMLA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SMLA_OK = 0,
  SMLA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer */
  SMLA_ERR_UNSUPPORTED = 2,  /* valid but outside the shapes this build implements */
  SMLA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  SMLA_ERR_TIMEOUT = 4,      /* a device pipeline wait gave up (device error word) */
  SMLA_ERR_DEVICE_CHECK = 5  /* an index / page id was out of range (device error word) */
} smla_status_t;

enum { SMLA_BF16 = 0, SMLA_E4M3 = 1 };

/* Ragged batch of B sequences over a paged cache (all pointers on the device).
 * Sequence b owns query tokens cu_q[b] .. cu_q[b+1]-1 and kv_len[b] cached
 * tokens; its q_len = cu_q[b+1]-cu_q[b] new tokens are the LAST q_len cached
 * positions, so its token i sits at pos = kv_len[b] - q_len + i and may
 * attend to logical keys 0..pos.  Logical key j of sequence b is physical
 * row page_table[b*max_pages + j/page_size]*page_size + j%page_size.
 * T = cu_q[B] (passed on the host so that no call reads device memory to
 * size its grid).  Requires q_len <= kv_len for every sequence.  The three
 * pointers must be 4-byte aligned. */
typedef struct {
  const int32_t* cu_q;        /* [B+1] */
  const int32_t* kv_len;      /* [B] */
  const int32_t* page_table;  /* [B, max_pages] physical page ids */
  int32_t B;
  int32_t max_pages;
  int32_t page_size;          /* power of two, 8..4096 */
  int32_t T;
} smla_seqs_t;

/* Stage 1 -- FP8 lightning-indexer scores.
 * "sparse_index_fp8_sm100" (Modular Mojo kernel page), module summary and
 * section "Layout (crux)":
 *   scores[t, key] = k_scale[phys(key)] * sum_h relu(q[t,h,:] . k_pool[phys(key),:]) * q_scale[t,h]
 * for every logical key 0..pos(t) of t's sequence; every other entry of row
 * t (key > pos(t), up to score_stride) is written as -inf (the causal tail
 * fill, fused).
 *   q        e4m3 [T, H_idx, 128]
 *   q_scale  f32  [T, H_idx]
 *   k_pool   e4m3 [phys_rows, 128]  paged indexer keys
 *   k_scale  f32  [phys_rows]       per physical row
 *   scores   f32  [T, score_stride] (output; score_stride >= max kv_len, multiple of 4)
 * H_idx must be 4, 8, 16, 32 or 64 (SMLA_ERR_UNSUPPORTED otherwise).
 * Alignment: q, k_pool and scores 16 bytes; q_scale and k_scale 4 bytes.
 * The dot products run on tcgen05 FP8 tensor cores with f32 accumulation. */
smla_status_t smla_indexer_scores(const uint8_t* q, const float* q_scale, const uint8_t* k_pool,
                                  const float* k_scale, int64_t phys_rows, smla_seqs_t seqs,
                                  int32_t H_idx, float* scores, int64_t score_stride,
                                  cudaStream_t stream);

/* Stage 2 -- per-token top-k over the causally valid keys.
 * "sparse_index_fp8_sm100" (the indexer's score buffer is this stage's
 * input; the page verifies the result as a top-k set match) and
 * "mla_sm100_prefill_sparse_fp8" (indices in physical-row space + per-query
 * topk_lengths):
 *   topk_lengths[t] = min(k, pos(t)+1)
 *   indices[t, 0..len) = physical rows of the len largest scores[t, 0..pos(t)],
 *                        ties broken toward the lower logical key, emitted in
 *                        ascending logical-key order
 *   indices[t, len..k) = 0xFFFFFFFF
 *   scores   f32 [T, score_stride] (entries past pos(t) do not affect the
 *            result; a row's last 16-byte load may read up to three of them)
 *   indices  u32 [T, k] (output), topk_lengths u32 [T] (output)
 * workspace: caller-owned device scratch of at least
 * smla_topk_workspace_size(T, score_stride, k) bytes (16-byte aligned; may
 * be NULL when that size is 0, which it is for every shape this build
 * selects in one pass per row); its contents on entry do not matter and are
 * unspecified on return.  A smaller workspace_bytes returns
 * SMLA_ERR_INVALID_ARG.
 * 1 <= k <= 65536. NaN scores are unsupported (their order is unspecified).
 * Alignment: scores 16 bytes; indices and topk_lengths 4 bytes. */
size_t smla_topk_workspace_size(int32_t T, int64_t score_stride, int32_t k);
smla_status_t smla_topk(const float* scores, int64_t score_stride, smla_seqs_t seqs, int32_t k,
                        uint32_t* indices, uint32_t* topk_lengths, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);

/* Stages 1 + 2 fused -- indexer scores and per-token top-k in one pass, the
 * score rows kept in the SM's shared memory instead of an HBM buffer.
 * "sparse_index_fp8_sm100" (module summary: the scorer is a drop-in for the
 * buffer the top-k stage reads, and the fusions that follow it are left to
 * later work).  Outputs exactly what smla_indexer_scores followed by
 * smla_topk produce: the same scores (same MMAs and epilogue arithmetic in
 * the same order), the same selection rule (ties to the lower logical key),
 * indices u32 [T, k] in ascending logical-key order with the 0xFFFFFFFF
 * tail, topk_lengths u32 [T].
 *   q, q_scale, k_pool, k_scale, phys_rows, seqs, H_idx: as smla_indexer_scores
 *   score_stride: a bound on every kv_len (>= max kv_len, multiple of 4), as
 *                 the unfused pair's score row stride
 *   k, indices, topk_lengths: as smla_topk
 * Rows of up to 128 * H_idx keys (8192 at H_idx 64) stay on chip and need no
 * workspace; for a larger score_stride the call runs the unfused pair with
 * the score buffer [T, score_stride] in `workspace`.  workspace: caller-owned
 * device scratch of at least smla_indexer_topk_workspace_size(T,
 * score_stride, H_idx, k) bytes (16-byte aligned; NULL when that is 0);
 * contents on entry do not matter, unspecified on return.  Errors and
 * alignment as for the two stages. */
size_t smla_indexer_topk_workspace_size(int32_t T, int64_t score_stride, int32_t H_idx, int32_t k);
smla_status_t smla_indexer_topk(const uint8_t* q, const float* q_scale, const uint8_t* k_pool,
                                const float* k_scale, int64_t phys_rows, smla_seqs_t seqs, int32_t H_idx,
                                int64_t score_stride, int32_t k, uint32_t* indices, uint32_t* topk_lengths,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Stage 3 -- sparse MLA prefill attention.
 * "mla_sm100_prefill_sparse_fp8" (Modular Mojo function page: arguments,
 * scale_block_size modes) and "mla_prefill_sparse_qkv_fp8" (K and V share
 * the latent rows; V = the first v_depth columns).  For each token t and
 * head h, with n = topk_lengths[t] and K_j = dequant(latent_pool[indices[t,j]]):
 *   s_j = softmax_scale * q[t,h,:] . K_j,
 *   p_j = exp(s_j) / (exp(sink_h) + sum_i exp(s_i))   (sink_h = attn_sink[h], or no term when NULL),
 *   out[t,h,:] = bf16_rne( sum_j p_j * K_j[0:v_depth] )     (zeros if n == 0)
 *   q            [T, H, 576], bf16 (q_dtype SMLA_BF16) or e4m3 (SMLA_E4M3)
 *   latent_pool  e4m3 [phys_rows, 576] (512 nope + 64 rope)
 *   scales       f32 [phys_rows, ceil(576/scale_block_size)]; NULL when
 *                scale_block_size == 0 (unit scale); scale_block_size >= 576
 *                means one scale per row; 32 means 18 block scales per row
 *   indices      u32 [T, indices_stride] physical rows; topk_lengths u32 [T]
 *                (each <= indices_stride)
 *   attn_sink    f32 [H] or NULL: one logit per head, in the units of the
 *                scaled logits s_j, that joins every softmax denominator and
 *                carries no value (the page names the argument without
 *                defining it; this is the reading taken)
 *   out          bf16 [T, H, v_depth] (output)
 * Supported: H in {16, 32, 48, 64} or any multiple of 64; v_depth == 512;
 * scale_block_size in {0, 32} or >= 576, where 32 (block scales) requires e4m3
 * q.  Alignment: q, latent_pool and out 16 bytes; indices, topk_lengths,
 * scales and attn_sink 4 bytes.  Other shapes return SMLA_ERR_UNSUPPORTED,
 * misaligned pointers SMLA_ERR_INVALID_ARG; nothing is launched then.
 * Runs on tcgen05 FP8 tensor cores with f32 TMEM accumulation: e4m3 q is
 * used natively; bf16 q and the softmax weights P (bf16-accuracy path) are
 * carried as two e4m3 terms (hi + lo) so that the products stay on the FP8
 * pipe; blockwise-scaled rows are dequantised to the same two-term form. */
smla_status_t smla_sparse_prefill(const void* q, int32_t q_dtype, const uint8_t* latent_pool,
                                  int64_t phys_rows, const float* scales, int32_t scale_block_size,
                                  const uint32_t* indices, int32_t indices_stride,
                                  const uint32_t* topk_lengths, int32_t T, int32_t H,
                                  int32_t v_depth, float softmax_scale, const float* attn_sink,
                                  uint16_t* out, cudaStream_t stream);

/* Sparse MLA prefill over a BF16 latent cache: "mla_sm100_prefill_sparse_fp8"
 * names itself the FP8 KV-cache variant of "mla_sm100_prefill_sparse"; this
 * is that BF16-cache form.  The same computation as smla_sparse_prefill with
 * K_j = latent_pool[indices[t,j]] read as bf16 (no scales):
 *   q            bf16 [T, H, 576]
 *   latent_pool  bf16 [phys_rows, 576] (512 nope + 64 rope)
 *   indices, topk_lengths, attn_sink, out, H, v_depth: as smla_sparse_prefill
 * Alignment: q, latent_pool and out 16 bytes; indices, topk_lengths and
 * attn_sink 4 bytes.  The products run as tcgen05 kind::f16 (bf16 x bf16)
 * MMAs with f32 TMEM accumulation; P is rounded to bf16. */
smla_status_t smla_sparse_prefill_bf16_cache(const uint16_t* q, const uint16_t* latent_pool, int64_t phys_rows,
                                             const uint32_t* indices, int32_t indices_stride,
                                             const uint32_t* topk_lengths, int32_t T, int32_t H,
                                             int32_t v_depth, float softmax_scale, const float* attn_sink,
                                             uint16_t* out, cudaStream_t stream);

/* Dense causal MLA prefill over the paged latent cache, for prompts short
 * enough that a top-k selection would keep every key.  "SM100MLA" (the
 * dense MLA prefill struct page) and "mla_sm100_prefill_blockscale" (dense
 * MLA prefill with a block-scaled FP8 cache): token t of sequence b attends
 * to every logical key 0..pos(t) of b (pos as in smla_seqs_t), reached
 * through the page table, so no indices are read:
 *   out[t,h,:] = sum_{j <= pos(t)} p_j * K_j[0:v_depth],
 *   K_j = dequant(latent_pool[phys(b, j)]), p and the sink as for
 *   smla_sparse_prefill.
 * This equals smla_sparse_prefill with indices[t] = phys(b, 0..pos(t)) and
 * topk_lengths[t] = pos(t)+1.  T = seqs.T; q [T, H, 576] and out
 * [T, H, 512] as there; the other arguments, supported shapes, alignment
 * and errors as for smla_sparse_prefill. */
smla_status_t smla_dense_prefill(const void* q, int32_t q_dtype, const uint8_t* latent_pool,
                                 int64_t phys_rows, const float* scales, int32_t scale_block_size,
                                 smla_seqs_t seqs, int32_t H, int32_t v_depth, float softmax_scale,
                                 const float* attn_sink, uint16_t* out, cudaStream_t stream);

/* Sparse MLA decode: the sparse attention of smla_sparse_prefill for few
 * query tokens (one or two per sequence), the other serving phase of the
 * same cache and indices ("mla_prefill_sparse_qkv_fp8", which names the
 * FP8 decode QK / PV machinery the prefill reuses).  Same arguments, result
 * and rules as smla_sparse_prefill.  When the (token, 64-head group) pairs
 * are too few to fill the GPU, each token's key blocks are divided among
 * several CTAs, whose partial outputs and log-sum-exps go to `workspace`
 * and are merged by a second kernel.  workspace: caller-owned device
 * scratch of at least smla_sparse_decode_workspace_size(T, H,
 * indices_stride) bytes on the current device (16-byte aligned; NULL when
 * that size is 0); contents on entry do not matter, unspecified on return;
 * too small returns SMLA_ERR_INVALID_ARG. */
size_t smla_sparse_decode_workspace_size(int32_t T, int32_t H, int32_t indices_stride);
smla_status_t smla_sparse_decode(const void* q, int32_t q_dtype, const uint8_t* latent_pool,
                                 int64_t phys_rows, const float* scales, int32_t scale_block_size,
                                 const uint32_t* indices, int32_t indices_stride,
                                 const uint32_t* topk_lengths, int32_t T, int32_t H,
                                 int32_t v_depth, float softmax_scale, const float* attn_sink,
                                 uint16_t* out, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/* smla_sparse_decode without a workspace, for callers that cannot allocate
 * device memory at the point where they decode: code running inside another
 * runtime's enqueue step that forbids allocation (an inference-engine
 * plugin, say), or a serving loop whose device memory is all reserved by a
 * pool it may not go around, or where a cudaMalloc would stall the loop.
 * The papers have no counterpart of this call; it is an integration
 * convenience.
 * Same arguments, result and rules as smla_sparse_decode, minus workspace
 * and workspace_bytes: the split partials live in a fixed 32 MiB scratch
 * array that the library declares in device memory.  Every GPU that loads
 * the library holds those 32 MiB until the process exits.  The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 * The first call on a device looks the array's device address up (once,
 * with that device current) and should come before any stream capture.
 * The split count is the one smla_sparse_decode uses; on a 152-SM GB300 it
 * never needs more than about 20 MB.  Sizes that would need more than 32 MiB
 * return SMLA_ERR_UNSUPPORTED with a message naming the need, and nothing
 * is launched.  All calls share the one array, which keeps the last call's
 * contents; every entry a call reads back is written first by that call, so
 * nothing has to start at zero.  Calls whose kernels overlap on the GPU
 * (different streams, or other host threads) race on the array: order them
 * on one stream. */
smla_status_t smla_sparse_decode_noalloc(const void* q, int32_t q_dtype, const uint8_t* latent_pool,
                                         int64_t phys_rows, const float* scales, int32_t scale_block_size,
                                         const uint32_t* indices, int32_t indices_stride,
                                         const uint32_t* topk_lengths, int32_t T, int32_t H,
                                         int32_t v_depth, float softmax_scale, const float* attn_sink,
                                         uint16_t* out, cudaStream_t stream);

/* Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns SMLA_OK, SMLA_ERR_DEVICE_CHECK (out-of-range index or page
 * id), SMLA_ERR_TIMEOUT (a pipeline wait gave up) or SMLA_ERR_CUDA. */
smla_status_t smla_check_device_errors(cudaStream_t stream);

/* Self-test of the device timeout path: enqueues one kernel whose only
 * thread waits, with a limit of limit_us microseconds (1 .. 1000000), on a
 * pipeline barrier that nothing completes, exactly as the stage kernels
 * wait on theirs.  When the limit passes, the kernel records the timeout
 * in the device error word and returns, so the next
 * smla_check_device_errors() reports SMLA_ERR_TIMEOUT.  No library function
 * calls it; it exists so that the timeout path can be tested without a
 * hung kernel. */
smla_status_t smla_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream);

/* Copies the calling thread's last error message (NUL-terminated, truncated
 * to n bytes) and returns its full length. */
size_t smla_last_error(char* buf, size_t n);

/* Library version, "major.minor.patch". */
const char* smla_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SMLA_H_ */
