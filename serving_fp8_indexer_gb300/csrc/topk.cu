// Stage 2: per-token top-k over the causally valid keys.
//
// The score buffer "the top-k stage consumes" ("sparse_index_fp8_sm100"
// page) feeds per-query physical-row indices and topk_lengths
// ("mla_sm100_prefill_sparse_fp8" page).  The pages do not describe the
// selection algorithm; this one is a radix select:
//   * one CTA per token; the token's valid scores (keys 0..pos) are read
//     once from HBM (float4, coalesced) into shared memory as
//     order-preserving 32-bit keys;
//   * three histogram passes (11 + 11 + 10 bits, shared-memory atomics)
//     pin the exact k-th largest key value;
//   * one stable compaction pass in logical-key order emits every key above
//     that value plus the lowest-keyed ties, mapped to physical rows through
//     the page table.
// Tokens with pos + 1 <= k take every valid key without selecting.
#include <algorithm>

#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {
namespace tk {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;

struct Params {
  const float* scores;
  int64_t stride;
  const int32_t* cu_q;
  const int32_t* kv_len;
  const int32_t* page_table;
  int B, max_pages, page_size, T;
  int k;
  uint32_t* indices;
  uint32_t* lens;
  int cache_cap;  // floats of the row cached in shared memory
  unsigned* err;
};

// Larger float -> larger unsigned key (-0 sorts just below +0).
__device__ __forceinline__ uint32_t ordered(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive block-wide prefix sum over kThreads values; returns the prefix
// and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += x;
    }
    if (lane < kWarps) warp_tot[lane] = wi - w;  // exclusive warp offsets
    if (lane == kWarps - 1) warp_tot[kWarps] = wi;
  }
  __syncthreads();
  const int r = warp_tot[warp] + incl - v;
  *total = warp_tot[kWarps];
  __syncthreads();
  return r;
}

__device__ __forceinline__ uint32_t phys_row(const Params& p, int b, int key) {
  const int page = key / p.page_size;
  const int pid = page < p.max_pages ? p.page_table[static_cast<int64_t>(b) * p.max_pages + page] : -1;
  if (pid < 0) {
    atomicOr(p.err, kErrPage);
    return 0xFFFFFFFFu;
  }
  return static_cast<uint32_t>(pid) * static_cast<uint32_t>(p.page_size) + static_cast<uint32_t>(key % p.page_size);
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const Params p) {
  extern __shared__ uint32_t cache[];
  __shared__ uint32_t hist[kBins];
  __shared__ int warp_tot[kWarps + 1];
  __shared__ int sh_b, sh_bin, sh_above;

  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid == 0) {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (p.cu_q[mid + 1] <= t) lo = mid + 1; else hi = mid;
    }
    sh_b = lo;
  }
  __syncthreads();
  const int b = sh_b;
  const int q_len = p.cu_q[b + 1] - p.cu_q[b];
  const int kvl = p.kv_len[b];
  int n = kvl - q_len + (t - p.cu_q[b]) + 1;  // valid keys 0..pos
  if (n < 1 || n > p.stride || kvl < q_len) {
    if (tid == 0) atomicOr(p.err, kErrShape);
    n = max(0, min(n, static_cast<int>(p.stride)));
  }
  const int k = p.k;
  uint32_t* out = p.indices + static_cast<int64_t>(t) * k;

  if (n <= k) {
    for (int key = tid; key < n; key += kThreads) out[key] = phys_row(p, b, key);
    for (int i = n + tid; i < k; i += kThreads) out[i] = 0xFFFFFFFFu;
    if (tid == 0) p.lens[t] = static_cast<uint32_t>(n);
    return;
  }

  const float* row = p.scores + static_cast<int64_t>(t) * p.stride;
  const bool cached = n <= p.cache_cap;
  if (cached) {
    const int n4 = n >> 2;
    const float4* row4 = reinterpret_cast<const float4*>(row);
    for (int i = tid; i < n4; i += kThreads) {
      const float4 v = __ldcs(row4 + i);  // read once: stream past L2
      uint4 u;
      u.x = ordered(v.x); u.y = ordered(v.y); u.z = ordered(v.z); u.w = ordered(v.w);
      reinterpret_cast<uint4*>(cache)[i] = u;
    }
    for (int i = (n4 << 2) + tid; i < n; i += kThreads) cache[i] = ordered(row[i]);
  }
  auto key_at = [&](int i) -> uint32_t { return cached ? cache[i] : ordered(row[i]); };

  // ---- radix select of the k-th largest ordered key
  uint32_t prefix = 0;
  int krem = k;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
#pragma unroll
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass], wd = widths[pass];
    const uint32_t mask = (1u << wd) - 1u;
    for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t u = key_at(i);
      if (pass == 0 || (u >> (sh + wd)) == prefix) atomicAdd(&hist[(u >> sh) & mask], 1u);
    }
    __syncthreads();
    // Count of elements in bins above each thread's bins: scan in reverse.
    const int rt = kThreads - 1 - tid;  // thread rt owns bins [rt*4, rt*4+4)
    int local = 0;
#pragma unroll
    for (int j = 0; j < kBinsPerThread; ++j) local += hist[rt * kBinsPerThread + j];
    int total;
    int above = block_exclusive_scan(local, warp_tot, &total);
    int c = above;
#pragma unroll
    for (int j = kBinsPerThread - 1; j >= 0; --j) {
      const int bin = rt * kBinsPerThread + j;
      const int h = hist[bin];
      if (c < krem && c + h >= krem) {
        sh_bin = bin;
        sh_above = c;
      }
      c += h;
    }
    __syncthreads();
    prefix = (prefix << wd) | static_cast<uint32_t>(sh_bin);
    krem -= sh_above;
    __syncthreads();
  }
  const uint32_t thr = prefix;  // exact k-th largest key; krem ties of it are taken

  // ---- stable compaction in logical-key order
  int base = 0, tie_base = 0;
  for (int start = 0; start < n; start += kThreads * 4) {
    uint32_t u[4];
    int neq = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = start + tid * 4 + j;
      u[j] = i < n ? key_at(i) : 0u;
      neq += (i < n && u[j] == thr) ? 1 : 0;
    }
    int eq_total;
    int tie_rank = tie_base + block_exclusive_scan(neq, warp_tot, &eq_total);
    bool sel[4];
    int nsel = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = start + tid * 4 + j;
      bool s = false;
      if (i < n) {
        if (u[j] > thr) s = true;
        else if (u[j] == thr) { s = tie_rank < krem; ++tie_rank; }
      }
      sel[j] = s;
      nsel += s ? 1 : 0;
    }
    int sel_total;
    int pos = base + block_exclusive_scan(nsel, warp_tot, &sel_total);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (sel[j]) {
        if (pos < k) out[pos] = phys_row(p, b, start + tid * 4 + j);
        else atomicOr(p.err, kErrShape);
        ++pos;
      }
    base += sel_total;
    tie_base += eq_total;
  }
  if (tid == 0) p.lens[t] = static_cast<uint32_t>(k);
}

}  // namespace tk

smla_status_t launch_topk(const float* scores, int64_t score_stride, const smla_seqs_t& seqs, int k,
                          uint32_t* indices, uint32_t* topk_lengths, unsigned* err, cudaStream_t stream) {
  using namespace tk;
  if (seqs.T == 0) return SMLA_OK;
  // Cache the whole row when it fits in 160 KB of shared memory; otherwise
  // every pass re-reads it (from L2).
  const int64_t cap = std::min<int64_t>(score_stride, 40 * 1024);
  const size_t smem = static_cast<size_t>((cap + 3) & ~int64_t(3)) * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return fail_cuda(e, "topk smem attribute");
  Params p{scores, score_stride, seqs.cu_q, seqs.kv_len, seqs.page_table, seqs.B, seqs.max_pages,
           seqs.page_size, seqs.T, k, indices, topk_lengths, static_cast<int>(cap), err};
  topk_kernel<<<seqs.T, kThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "topk launch");
  return SMLA_OK;
}

}  // namespace smla
