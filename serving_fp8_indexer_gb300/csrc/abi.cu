// The C ABI (include/smla.h): host-side argument validation, the per-device
// error word, tensor-map encoding and dispatch to the stage launchers.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {

namespace {
thread_local std::string g_last_error;
std::mutex g_mu;
constexpr int kMaxDevices = 64;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
}  // namespace

// One word per device; kernels atomicOr error bits into it.
__device__ unsigned int g_smla_device_errors;

smla_status_t fail(smla_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

smla_status_t fail_cuda(cudaError_t e, const char* what) {
  return fail(SMLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool encode_tma_u8(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                   const uint32_t* box, int swizzle_bytes) {
  if (rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], estr[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    estr[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  // The CUDA driver entry point is looked up through the runtime, so the library
  // does not link libcuda directly (it loads on machines without a CUDA driver).
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn encode = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return false;
      encode = reinterpret_cast<EncodeFn>(fn);
    }
  }
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
                            d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tma_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                      uint32_t box_rows, int swizzle_bytes) {
  const uint64_t dims[2] = {inner, rows};
  const uint64_t strides[1] = {inner};
  const uint32_t box[2] = {box_inner, box_rows};
  return encode_tma_u8(map, base, 2, dims, strides, box, swizzle_bytes);
}

static smla_status_t device_err_ptr(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SMLA_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_smla_device_errors);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(device error word)");
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_err_ptr[dev];
  return SMLA_OK;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sm_count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

// One warp: lane 0 initialises an mbarrier expecting one arrival that never
// comes and waits on its first phase with the given limit (the stage
// kernels' bounded wait); the wait gives up, records kErrTimeout and the
// kernel returns.
__global__ void selftest_wait_kernel(unsigned* err, unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    mbar_wait(smem_u32(&bar), 0, err, limit_ns);
  }
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

static smla_status_t check_seqs(const smla_seqs_t& s) {
  if (s.T < 0 || s.B < 0) return fail(SMLA_ERR_INVALID_ARG, "seqs: T=%d B=%d must be >= 0", s.T, s.B);
  if (s.T == 0) return SMLA_OK;
  if (s.B < 1) return fail(SMLA_ERR_INVALID_ARG, "seqs: B must be >= 1 when T > 0");
  if (!s.cu_q || !s.kv_len || !s.page_table) return fail(SMLA_ERR_INVALID_ARG, "seqs: null pointer");
  if (!aligned4(s.cu_q) || !aligned4(s.kv_len) || !aligned4(s.page_table))
    return fail(SMLA_ERR_INVALID_ARG, "seqs: pointers must be 4-byte aligned");
  if (s.max_pages < 1) return fail(SMLA_ERR_INVALID_ARG, "seqs: max_pages must be >= 1");
  if (s.page_size < 8 || s.page_size > 4096 || (s.page_size & (s.page_size - 1)))
    return fail(SMLA_ERR_UNSUPPORTED, "seqs: page_size %d must be a power of two in [8, 4096]", s.page_size);
  return SMLA_OK;
}

}  // namespace smla

using namespace smla;

extern "C" {

const char* smla_version(void) { return "0.1.0"; }

size_t smla_last_error(char* buf, size_t n) {
  const std::string& m = g_last_error;
  if (buf && n) {
    const size_t c = m.size() < n - 1 ? m.size() : n - 1;
    std::memcpy(buf, m.data(), c);
    buf[c] = '\0';
  }
  return m.size();
}

smla_status_t smla_indexer_scores(const uint8_t* q, const float* q_scale, const uint8_t* k_pool,
                                  const float* k_scale, int64_t phys_rows, smla_seqs_t seqs, int32_t H_idx,
                                  float* scores, int64_t score_stride, cudaStream_t stream) {
  g_last_error.clear();
  smla_status_t st = check_seqs(seqs);
  if (st != SMLA_OK) return st;
  if (H_idx != 4 && H_idx != 8 && H_idx != 16 && H_idx != 32 && H_idx != 64)
    return fail(SMLA_ERR_UNSUPPORTED, "H_idx=%d: supported 4, 8, 16, 32, 64", H_idx);
  if (score_stride < 4 || (score_stride & 3))
    return fail(SMLA_ERR_INVALID_ARG, "score_stride=%lld must be a positive multiple of 4",
                static_cast<long long>(score_stride));
  if (seqs.T == 0) return SMLA_OK;
  if (!q || !q_scale || !k_pool || !k_scale || !scores) return fail(SMLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(scores) || !aligned4(q_scale) || !aligned4(k_scale))
    return fail(SMLA_ERR_INVALID_ARG, "q, k_pool, scores must be 16-byte aligned; scales 4-byte aligned");
  if (phys_rows < 1 || phys_rows >= (int64_t(1) << 31))
    return fail(SMLA_ERR_INVALID_ARG, "phys_rows=%lld out of range", static_cast<long long>(phys_rows));
  if (static_cast<int64_t>(seqs.T) * H_idx >= (int64_t(1) << 31))
    return fail(SMLA_ERR_UNSUPPORTED, "T*H_idx too large");
  unsigned* err = nullptr;
  st = device_err_ptr(&err);
  if (st != SMLA_OK) return st;
  return launch_indexer(q, q_scale, k_pool, k_scale, phys_rows, seqs, H_idx, scores, score_stride, err, stream);
}

size_t smla_topk_workspace_size(int32_t T, int64_t score_stride, int32_t k) {
  (void)T;
  (void)score_stride;
  (void)k;
  // Every supported row is selected by one CTA in one pass over its scores:
  // no scratch beyond shared memory.
  return 0;
}

smla_status_t smla_topk(const float* scores, int64_t score_stride, smla_seqs_t seqs, int32_t k, uint32_t* indices,
                        uint32_t* topk_lengths, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  g_last_error.clear();
  smla_status_t st = check_seqs(seqs);
  if (st != SMLA_OK) return st;
  if (k < 1 || k > 65536) return fail(SMLA_ERR_UNSUPPORTED, "k=%d must be in [1, 65536]", k);
  if (score_stride < 4 || (score_stride & 3))
    return fail(SMLA_ERR_INVALID_ARG, "score_stride=%lld must be a positive multiple of 4",
                static_cast<long long>(score_stride));
  const size_t need = smla_topk_workspace_size(seqs.T, score_stride, k);
  if (workspace_bytes < need || (need && !workspace))
    return fail(SMLA_ERR_INVALID_ARG, "workspace: %zu bytes given, %zu needed", workspace_bytes, need);
  if (workspace && !aligned16(workspace)) return fail(SMLA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (seqs.T == 0) return SMLA_OK;
  if (!scores || !indices || !topk_lengths) return fail(SMLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(scores) || !aligned4(indices) || !aligned4(topk_lengths))
    return fail(SMLA_ERR_INVALID_ARG, "scores must be 16-byte aligned; outputs 4-byte aligned");
  unsigned* err = nullptr;
  st = device_err_ptr(&err);
  if (st != SMLA_OK) return st;
  return launch_topk(scores, score_stride, seqs, k, indices, topk_lengths, err, stream);
}

}  // extern "C"

namespace smla {
// Host-side checks shared by the attention entry points; T is the number of
// query tokens, `keyed` says whether indices / topk_lengths are used.
static smla_status_t check_attn(const void* q, int32_t q_dtype, const void* latent_pool, int64_t phys_rows,
                                const float* scales, int32_t scale_block_size, bool keyed, const uint32_t* indices,
                                int32_t indices_stride, const uint32_t* topk_lengths, int32_t T, int32_t H,
                                int32_t v_depth, float softmax_scale, const float* attn_sink, const void* out) {
  if (T < 0) return fail(SMLA_ERR_INVALID_ARG, "T=%d must be >= 0", T);
  if (q_dtype != SMLA_BF16 && q_dtype != SMLA_E4M3) return fail(SMLA_ERR_INVALID_ARG, "q_dtype=%d", q_dtype);
  if (!(H >= 1 && ((H <= 64 && H % 16 == 0) || H % 64 == 0)))
    return fail(SMLA_ERR_UNSUPPORTED, "H=%d: supported 16, 32, 48, 64 or a multiple of 64", H);
  if (v_depth != 512) return fail(SMLA_ERR_UNSUPPORTED, "v_depth=%d: only 512 is supported", v_depth);
  if (!(scale_block_size == 0 || scale_block_size == 32 || scale_block_size >= 576))
    return fail(SMLA_ERR_UNSUPPORTED, "scale_block_size=%d: supported 0, 32 or >= 576", scale_block_size);
  if (scale_block_size == 32 && q_dtype == SMLA_BF16)
    return fail(SMLA_ERR_UNSUPPORTED, "scale_block_size=32 (block scales) requires e4m3 q");
  if (scale_block_size != 0 && !scales) return fail(SMLA_ERR_INVALID_ARG, "scales is NULL with scale_block_size != 0");
  if (!(softmax_scale == softmax_scale) || softmax_scale > 3.0e38f || softmax_scale < -3.0e38f)
    return fail(SMLA_ERR_INVALID_ARG, "softmax_scale must be finite");
  if (keyed && indices_stride < 1) return fail(SMLA_ERR_INVALID_ARG, "indices_stride must be >= 1");
  if (T == 0) return SMLA_OK;
  if (!q || !latent_pool || !out || (keyed && (!indices || !topk_lengths)))
    return fail(SMLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(latent_pool) || !aligned16(out) ||
      (keyed && (!aligned4(indices) || !aligned4(topk_lengths))) || (scales && !aligned4(scales)) ||
      (attn_sink && !aligned4(attn_sink)))
    return fail(SMLA_ERR_INVALID_ARG,
                "q, latent_pool, out must be 16-byte aligned; indices, scales and attn_sink 4-byte aligned");
  if (phys_rows < 1 || phys_rows >= (int64_t(1) << 31))
    return fail(SMLA_ERR_INVALID_ARG, "phys_rows=%lld out of range", static_cast<long long>(phys_rows));
  if (static_cast<int64_t>(T) * H >= (int64_t(1) << 31)) return fail(SMLA_ERR_UNSUPPORTED, "T*H too large");
  return SMLA_OK;
}
}  // namespace smla

extern "C" {

smla_status_t smla_sparse_prefill(const void* q, int32_t q_dtype, const uint8_t* latent_pool, int64_t phys_rows,
                                  const float* scales, int32_t scale_block_size, const uint32_t* indices,
                                  int32_t indices_stride, const uint32_t* topk_lengths, int32_t T, int32_t H,
                                  int32_t v_depth, float softmax_scale, const float* attn_sink, uint16_t* out,
                                  cudaStream_t stream) {
  g_last_error.clear();
  smla_status_t st = check_attn(q, q_dtype, latent_pool, phys_rows, scales, scale_block_size, true, indices,
                                indices_stride, topk_lengths, T, H, v_depth, softmax_scale, attn_sink, out);
  if (st != SMLA_OK || T == 0) return st;
  unsigned* err = nullptr;
  st = device_err_ptr(&err);
  if (st != SMLA_OK) return st;
  AttnArgs a{q, q_dtype, latent_pool, phys_rows, scales, scale_block_size, indices, indices_stride, topk_lengths,
             nullptr, T, H, softmax_scale, attn_sink, out, 1, nullptr, nullptr};
  return launch_attention(a, err, stream);
}

size_t smla_indexer_topk_workspace_size(int32_t T, int64_t score_stride, int32_t H_idx, int32_t k) {
  (void)k;
  if (T <= 0 || score_stride <= 0) return 0;
  if (score_stride <= indexer_topk_row_cap(H_idx)) return 0;  // rows stay on chip
  // longer rows: the score buffer [T, score_stride] f32 goes to the workspace
  return (static_cast<size_t>(T) * static_cast<size_t>(score_stride) * sizeof(float) + 255) & ~size_t(255);
}

smla_status_t smla_indexer_topk(const uint8_t* q, const float* q_scale, const uint8_t* k_pool, const float* k_scale,
                                int64_t phys_rows, smla_seqs_t seqs, int32_t H_idx, int64_t score_stride, int32_t k,
                                uint32_t* indices, uint32_t* topk_lengths, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
  g_last_error.clear();
  smla_status_t st = check_seqs(seqs);
  if (st != SMLA_OK) return st;
  if (H_idx != 4 && H_idx != 8 && H_idx != 16 && H_idx != 32 && H_idx != 64)
    return fail(SMLA_ERR_UNSUPPORTED, "H_idx=%d: supported 4, 8, 16, 32, 64", H_idx);
  if (k < 1 || k > 65536) return fail(SMLA_ERR_UNSUPPORTED, "k=%d must be in [1, 65536]", k);
  if (score_stride < 4 || (score_stride & 3))
    return fail(SMLA_ERR_INVALID_ARG, "score_stride=%lld must be a positive multiple of 4",
                static_cast<long long>(score_stride));
  const size_t need = smla_indexer_topk_workspace_size(seqs.T, score_stride, H_idx, k);
  if (workspace_bytes < need || (need && !workspace))
    return fail(SMLA_ERR_INVALID_ARG, "workspace: %zu bytes given, %zu needed", workspace_bytes, need);
  if (workspace && !aligned16(workspace)) return fail(SMLA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (seqs.T == 0) return SMLA_OK;
  if (!q || !q_scale || !k_pool || !k_scale || !indices || !topk_lengths)
    return fail(SMLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(k_pool) || !aligned4(q_scale) || !aligned4(k_scale) || !aligned4(indices) ||
      !aligned4(topk_lengths))
    return fail(SMLA_ERR_INVALID_ARG, "q and k_pool must be 16-byte aligned; scales and outputs 4-byte aligned");
  if (phys_rows < 1 || phys_rows >= (int64_t(1) << 31))
    return fail(SMLA_ERR_INVALID_ARG, "phys_rows=%lld out of range", static_cast<long long>(phys_rows));
  if (static_cast<int64_t>(seqs.T) * H_idx >= (int64_t(1) << 31)) return fail(SMLA_ERR_UNSUPPORTED, "T*H_idx too large");
  unsigned* err = nullptr;
  st = device_err_ptr(&err);
  if (st != SMLA_OK) return st;
  if (need == 0)
    return launch_indexer_topk(q, q_scale, k_pool, k_scale, phys_rows, seqs, H_idx, k, indices, topk_lengths, err,
                               stream);
  float* scores = static_cast<float*>(workspace);
  st = launch_indexer(q, q_scale, k_pool, k_scale, phys_rows, seqs, H_idx, scores, score_stride, err, stream);
  if (st != SMLA_OK) return st;
  return launch_topk(scores, score_stride, seqs, k, indices, topk_lengths, err, stream);
}

smla_status_t smla_sparse_prefill_bf16_cache(const uint16_t* q, const uint16_t* latent_pool, int64_t phys_rows,
                                             const uint32_t* indices, int32_t indices_stride,
                                             const uint32_t* topk_lengths, int32_t T, int32_t H, int32_t v_depth,
                                             float softmax_scale, const float* attn_sink, uint16_t* out,
                                             cudaStream_t stream) {
  g_last_error.clear();
  smla_status_t st = check_attn(q, SMLA_BF16, latent_pool, phys_rows, nullptr, 0, true, indices, indices_stride,
                                topk_lengths, T, H, v_depth, softmax_scale, attn_sink, out);
  if (st != SMLA_OK || T == 0) return st;
  unsigned* err = nullptr;
  st = device_err_ptr(&err);
  if (st != SMLA_OK) return st;
  AttnArgs a{q, SMLA_BF16, reinterpret_cast<const uint8_t*>(latent_pool), phys_rows, nullptr, 0, indices,
             indices_stride, topk_lengths, nullptr, T, H, softmax_scale, attn_sink, out, 1, nullptr, nullptr, 1};
  return launch_attention(a, err, stream);
}

smla_status_t smla_dense_prefill(const void* q, int32_t q_dtype, const uint8_t* latent_pool, int64_t phys_rows,
                                 const float* scales, int32_t scale_block_size, smla_seqs_t seqs, int32_t H,
                                 int32_t v_depth, float softmax_scale, const float* attn_sink, uint16_t* out,
                                 cudaStream_t stream) {
  g_last_error.clear();
  smla_status_t st = check_seqs(seqs);
  if (st != SMLA_OK) return st;
  st = check_attn(q, q_dtype, latent_pool, phys_rows, scales, scale_block_size, false, nullptr, 0, nullptr, seqs.T,
                  H, v_depth, softmax_scale, attn_sink, out);
  if (st != SMLA_OK || seqs.T == 0) return st;
  unsigned* err = nullptr;
  st = device_err_ptr(&err);
  if (st != SMLA_OK) return st;
  AttnArgs a{q, q_dtype, latent_pool, phys_rows, scales, scale_block_size, nullptr, 0, nullptr,
             &seqs, seqs.T, H, softmax_scale, attn_sink, out, 1, nullptr, nullptr};
  return launch_attention(a, err, stream);
}

size_t smla_sparse_decode_workspace_size(int32_t T, int32_t H, int32_t indices_stride) {
  if (T <= 0 || H <= 0 || indices_stride <= 0) return 0;
  return decode_workspace_bytes(T, H, decode_splits(T, H, indices_stride));
}

}  // extern "C"

namespace smla {
// smla_sparse_decode, and with use_static the allocation-free variant whose
// split partials go to the library's fixed device scratch instead of a
// caller workspace.
static smla_status_t sparse_decode_impl(const void* q, int32_t q_dtype, const uint8_t* latent_pool,
                                        int64_t phys_rows, const float* scales, int32_t scale_block_size,
                                        const uint32_t* indices, int32_t indices_stride,
                                        const uint32_t* topk_lengths, int32_t T, int32_t H, int32_t v_depth,
                                        float softmax_scale, const float* attn_sink, uint16_t* out, void* workspace,
                                        size_t workspace_bytes, bool use_static, cudaStream_t stream) {
  g_last_error.clear();
  smla_status_t st = check_attn(q, q_dtype, latent_pool, phys_rows, scales, scale_block_size, true, indices,
                                indices_stride, topk_lengths, T, H, v_depth, softmax_scale, attn_sink, out);
  if (st != SMLA_OK) return st;
  const int nsplit = T > 0 ? decode_splits(T, H, indices_stride) : 1;
  const size_t need = decode_workspace_bytes(T, H, nsplit);
  if (use_static && T > 0) {
    st = noalloc_scratch_for(need, &workspace);
    if (st != SMLA_OK) return st;
    workspace_bytes = need;
  }
  if (workspace_bytes < need || (need && !workspace))
    return fail(SMLA_ERR_INVALID_ARG, "workspace: %zu bytes given, %zu needed", workspace_bytes, need);
  if (workspace && !aligned16(workspace)) return fail(SMLA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (T == 0) return SMLA_OK;
  unsigned* err = nullptr;
  st = device_err_ptr(&err);
  if (st != SMLA_OK) return st;
  // workspace: partial outputs [T, nsplit, H, 512] f32, then (at the next
  // 256-byte boundary) log2-sum-exps [T, nsplit, H] f32
  float* part_o = static_cast<float*>(workspace);
  const size_t o_bytes = (static_cast<size_t>(T) * nsplit * H * 512 * sizeof(float) + 255) & ~size_t(255);
  float* part_lse = nsplit > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + o_bytes) : nullptr;
  AttnArgs a{q, q_dtype, latent_pool, phys_rows, scales, scale_block_size, indices, indices_stride, topk_lengths,
             nullptr, T, H, softmax_scale, attn_sink, out, nsplit, nsplit > 1 ? part_o : nullptr, part_lse};
  st = launch_attention(a, err, stream);
  if (st != SMLA_OK || nsplit == 1) return st;
  return launch_decode_combine(part_o, part_lse, attn_sink, T, H, nsplit, out, stream);
}

}  // namespace smla

extern "C" {

smla_status_t smla_sparse_decode(const void* q, int32_t q_dtype, const uint8_t* latent_pool, int64_t phys_rows,
                                 const float* scales, int32_t scale_block_size, const uint32_t* indices,
                                 int32_t indices_stride, const uint32_t* topk_lengths, int32_t T, int32_t H,
                                 int32_t v_depth, float softmax_scale, const float* attn_sink, uint16_t* out,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return sparse_decode_impl(q, q_dtype, latent_pool, phys_rows, scales, scale_block_size, indices, indices_stride,
                            topk_lengths, T, H, v_depth, softmax_scale, attn_sink, out, workspace, workspace_bytes,
                            false, stream);
}

smla_status_t smla_sparse_decode_noalloc(const void* q, int32_t q_dtype, const uint8_t* latent_pool,
                                         int64_t phys_rows, const float* scales, int32_t scale_block_size,
                                         const uint32_t* indices, int32_t indices_stride,
                                         const uint32_t* topk_lengths, int32_t T, int32_t H, int32_t v_depth,
                                         float softmax_scale, const float* attn_sink, uint16_t* out,
                                         cudaStream_t stream) {
  return sparse_decode_impl(q, q_dtype, latent_pool, phys_rows, scales, scale_block_size, indices, indices_stride,
                            topk_lengths, T, H, v_depth, softmax_scale, attn_sink, out, nullptr, 0, true, stream);
}

smla_status_t smla_check_device_errors(cudaStream_t stream) {
  g_last_error.clear();
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_smla_device_errors, sizeof(v));
  if (e != cudaSuccess) return fail_cuda(e, "read device error word");
  if (v == 0) return SMLA_OK;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_smla_device_errors, &zero, sizeof(zero));
  if (e != cudaSuccess) return fail_cuda(e, "clear device error word");
  if (v & kErrTimeout) return fail(SMLA_ERR_TIMEOUT, "device error word 0x%x: a pipeline wait gave up", v);
  return fail(SMLA_ERR_DEVICE_CHECK, "device error word 0x%x: index/page/shape out of range", v);
}

smla_status_t smla_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream) {
  g_last_error.clear();
  if (limit_us < 1 || limit_us > 1000000)
    return fail(SMLA_ERR_INVALID_ARG, "limit_us=%u must be in [1, 1000000]", limit_us);
  unsigned* err = nullptr;
  const smla_status_t st = device_err_ptr(&err);
  if (st != SMLA_OK) return st;
  selftest_wait_kernel<<<1, 32, 0, stream>>>(err, static_cast<unsigned long long>(limit_us) * 1000ull);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "selftest launch");
  return SMLA_OK;
}

}  // extern "C"
