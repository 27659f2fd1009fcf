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

smla_status_t launch_topk(const float* scores, int64_t score_stride, const smla_seqs_t& seqs, int k,
                          uint32_t* indices, uint32_t* topk_lengths, unsigned* err, cudaStream_t stream);

smla_status_t launch_sparse_prefill(const void* q, int q_dtype, const uint8_t* latent, int64_t phys_rows,
                                    const float* scales, int sbs, const uint32_t* indices, int indices_stride,
                                    const uint32_t* topk_lengths, int T, int H, float softmax_scale,
                                    uint16_t* out, unsigned* err, cudaStream_t stream);

}  // namespace smla
