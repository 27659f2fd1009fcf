// Host-side internals shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/smla.h"

namespace smla {

// Records a message for smla_last_error() and returns `st`.
smla_status_t fail(smla_status_t st, const char* fmt, ...);
smla_status_t fail_cuda(cudaError_t e, const char* what);

// uint8 tensor map of the given rank: dims[0] innermost (elements = bytes),
// strides[i] = byte stride of dimension i + 1, box per dimension, 64- or
// 128-byte swizzle, zero fill out of bounds.  False when cuTensorMapEncodeTiled rejects it.
bool encode_tma_u8(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                   const uint32_t* box, int swizzle_bytes);
// 2-D uint8 tensor map [rows][inner] (row pitch = inner bytes), box
// [box_rows][box_inner], 128- (default) or 64-byte swizzle, zero fill out of
// bounds.
bool encode_tma_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                      uint32_t box_rows, int swizzle_bytes = 128);

// Number of SMs of the current device (cached per device).
int device_sm_count();

smla_status_t launch_indexer(const uint8_t* q, const float* q_scale, const uint8_t* k_pool, const float* k_scale,
                             int64_t phys_rows, const smla_seqs_t& seqs, int h_idx, float* scores,
                             int64_t score_stride, unsigned* err, cudaStream_t stream);

// Fused indexer + top-k (score rows in shared memory): the longest row it
// holds for this H_idx, and its launcher (kv_len <= that cap).
int indexer_topk_row_cap(int h_idx);
smla_status_t launch_indexer_topk(const uint8_t* q, const float* q_scale, const uint8_t* k_pool, const float* k_scale,
                                  int64_t phys_rows, const smla_seqs_t& seqs, int h_idx, int k, uint32_t* indices,
                                  uint32_t* topk_lengths, unsigned* err, cudaStream_t stream);

smla_status_t launch_topk(const float* scores, int64_t score_stride, const smla_seqs_t& seqs, int k,
                          uint32_t* indices, uint32_t* topk_lengths, unsigned* err, cudaStream_t stream);

// One launch of the attention kernel: sparse (indices + lengths) or dense
// causal (seqs non-null: every key 0..pos through the page table), with an
// optional per-head sink and, for nsplit > 1, split-K partials instead of
// the bf16 output.
struct AttnArgs {
  const void* q;
  int q_dtype;
  const uint8_t* latent;
  int64_t phys_rows;
  const float* scales;
  int sbs;
  const uint32_t* indices;
  int indices_stride;
  const uint32_t* topk_lengths;
  const smla_seqs_t* seqs;
  int T, H;
  float softmax_scale;
  const float* sink;
  uint16_t* out;
  int nsplit;
  float* part_o;    // [T, nsplit, H, 512]
  float* part_lse;  // [T, nsplit, H]
  int cache_bf16;   // latent_pool holds bf16 [phys_rows, 576] (q bf16, no scales)
};
smla_status_t launch_attention(const AttnArgs& a, unsigned* err, cudaStream_t stream);

// Split-K decode: the split count for these sizes, the workspace it needs,
// and the kernel that combines the partials into the bf16 output.
int decode_splits(int T, int H, int indices_stride);
size_t decode_workspace_bytes(int T, int H, int nsplit);
// Fixed scratch of smla_sparse_decode_noalloc (a static device array): its
// size, and its device address on the current device when `need` bytes fit
// (SMLA_ERR_UNSUPPORTED otherwise; nullptr when need is 0).
size_t noalloc_scratch_bytes();
smla_status_t noalloc_scratch_for(size_t need, void** out);
smla_status_t launch_decode_combine(const float* part_o, const float* part_lse, const float* sink, int T, int H,
                                    int nsplit, uint16_t* out, cudaStream_t stream);

}  // namespace smla
