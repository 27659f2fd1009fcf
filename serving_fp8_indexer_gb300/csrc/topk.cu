// Stage 2: per-token top-k over the causally valid keys.
//
// Input: the indexer's score buffer ("sparse_index_fp8_sm100" page, module
// summary); output: the per-query physical-row indices and topk_lengths the
// sparse attention reads ("mla_sm100_prefill_sparse_fp8" page, arguments).
// The pages do not describe the selection algorithm; this one is a radix
// select:
//   * one CTA per token; the token's valid scores (keys 0..pos) are read
//     once from HBM (float4, coalesced) into shared memory as
//     order-preserving 32-bit keys;
//   * the row's min/max (taken while loading) give the highest bit in which
//     the keys differ; one 11-bit histogram pass over the row from there
//     finds the bin holding the k-th largest;
//   * one pass over warp-contiguous key ranges counts each range's keys
//     above that bin and lists the bin's keys (the candidates);
//   * a short candidate list is ranked directly (score descending, key
//     ascending: the lowest-keyed ties win), marking the taken ones in a
//     bitmap; a long one falls back to more 11-bit digit passes;
//   * one stable compaction pass in logical-key order (warp ballots over the
//     same ranges) emits every key above the bin plus the taken candidates,
//     mapped to physical rows through the page table.
// Tokens with pos + 1 <= k take every valid key without selecting.
// Rows of at most 16384 keys take the register-resident kernel instead (the
// row held in registers, a thread's loads all issued before any is used,
// digit passes over the registers); when the last digit's bin is taken
// whole -- no tie at the threshold, the usual case for continuous scores --
// a key is taken iff it is >= that bin's lowest key, and the compaction
// carries one flag a key instead of two (measured on the end-to-end chunk:
// 0.466 -> 0.367 ms, identical indices).
#include <algorithm>

#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {
namespace tk {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;
constexpr int kRankCap = 128;  // candidates ranked pairwise; longer lists take more digit passes

struct Params {
  const float* scores;
  int64_t stride;
  const int32_t* cu_q;
  const int32_t* kv_len;
  const int32_t* page_table;
  int B, max_pages, page_size, T;
  int page_shift;  // log2(page_size)
  int k;
  uint32_t* indices;
  uint32_t* lens;
  int cache_cap;  // floats of the row cached in shared memory
  int cand_cap;   // keys of the boundary bin kept in the candidate list
  int pt_cap;     // page ids staged in shared memory
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
  const int page = key >> p.page_shift;
  const int pid = page < p.max_pages ? p.page_table[static_cast<int64_t>(b) * p.max_pages + page] : -1;
  if (pid < 0) {
    atomicOr(p.err, kErrPage);
    return 0xFFFFFFFFu;
  }
  return (static_cast<uint32_t>(pid) << p.page_shift) | static_cast<uint32_t>(key & (p.page_size - 1));
}

// Writes the physical row of logical key i to out[o] (page ids from the
// shared-memory copy `ptab` of the sequence's first nptab pages when it holds
// key i's page).
__device__ __forceinline__ void emit(const Params& p, int b, const int* ptab, int nptab, uint32_t* out, int o,
                                     int i) {
  if (o >= p.k) {
    atomicOr(p.err, kErrShape);
    return;
  }
  if (ptab && (i >> p.page_shift) < nptab) {
    const int pid = ptab[i >> p.page_shift];
    out[o] = pid >= 0 ? (static_cast<uint32_t>(pid) << p.page_shift) | static_cast<uint32_t>(i & (p.page_size - 1))
                      : phys_row(p, b, i);
  } else {
    out[o] = phys_row(p, b, i);
  }
}

// Finds the digit bin holding the krem-th largest candidate (bins counted
// from the top), returns it and subtracts the count above it from krem.
// *bin_count (if given) receives the bin's own count.
__device__ __forceinline__ int select_bin(const uint32_t* hist, int& krem, int* warp_tot, int* sh_bin,
                                          int* sh_above, int* bin_count = nullptr) {
  const int tid = threadIdx.x;
  const int rt = kThreads - 1 - tid;  // thread rt owns bins [rt*4, rt*4+4)
  int local = 0;
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) local += hist[rt * kBinsPerThread + j];
  int total;
  int c = block_exclusive_scan(local, warp_tot, &total);
#pragma unroll
  for (int j = kBinsPerThread - 1; j >= 0; --j) {
    const int bin = rt * kBinsPerThread + j;
    const int h = hist[bin];
    if (c < krem && c + h >= krem) {
      *sh_bin = bin;
      *sh_above = c;
      if (bin_count) *bin_count = h;
    }
    c += h;
  }
  __syncthreads();
  const int bin = *sh_bin;
  krem -= *sh_above;
  __syncthreads();
  return bin;
}

// Sequence b of token t (the number of sequence ends cu_q[b+1] <= t) and its
// number of valid keys n = pos + 1; flags and clamps inconsistent shapes.
__device__ __forceinline__ void token_row(const Params& p, int t, int* sh_b, int& b, int& n) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    int cnt = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int bb = b0 + tid;
      cnt += __popc(__ballot_sync(0xffffffffu, bb < p.B && p.cu_q[bb + 1] <= t));
    }
    if (tid == 0) *sh_b = min(cnt, p.B - 1);
  }
  __syncthreads();
  b = *sh_b;
  const int q_len = p.cu_q[b + 1] - p.cu_q[b];
  const int kvl = p.kv_len[b];
  n = kvl - q_len + (t - p.cu_q[b]) + 1;  // valid keys 0..pos
  if (n < 1 || n > p.stride || kvl < q_len) {
    if (tid == 0) atomicOr(p.err, kErrShape);
    n = max(0, min(n, static_cast<int>(p.stride)));
  }
}

// Register-resident selection for rows of at most 2048 * E4 keys: thread tid
// holds the keys 4 * (e * 512 + tid) + u (e < E4, u < 4), read once as
// float4.  11-bit digit histograms over the keys still matching the prefix
// find the k-th largest ordered key (stopping early once the bin holding it
// is taken whole); one compaction in key order (e, tid, u) then emits the
// keys above it and the lowest-keyed krem of its ties, from per-warp prefix
// sums of the two counts.
template <int E4>
__global__ void __launch_bounds__(kThreads, E4 <= 4 ? 3 : 1) topk_reg_kernel(const Params p) {
  constexpr int E = 4 * E4;
  __shared__ uint32_t hist[kBins];
  __shared__ int warp_tot[kWarps + 1];
  __shared__ uint32_t s_wmin[kWarps], s_wmax[kWarps];
  __shared__ uint32_t cnt_w[E4][kWarps];  // per (e, warp): gt count | tie count << 16
  __shared__ uint32_t cnt_p[(E4 + 3) / 4][kWarps];  // per warp: taken counts, four e per word
  __shared__ int ptab[256 * E4];          // page ids of the token's sequence (n / 8 pages at most)
  __shared__ int sh_b, sh_bin, sh_above, sh_cnt;

  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int b, n;
  token_row(p, t, &sh_b, b, n);
  const int k = p.k;
  uint32_t* out = p.indices + static_cast<int64_t>(t) * k;
  if (n <= k) {
    for (int key = tid; key < n; key += kThreads) out[key] = phys_row(p, b, key);
    for (int i = n + tid; i < k; i += kThreads) out[i] = 0xFFFFFFFFu;
    if (tid == 0) p.lens[t] = static_cast<uint32_t>(n);
    return;
  }
  if (n > 2048 * E4) {  // the host picks E4 from the row stride; never taken
    if (tid == 0) atomicOr(p.err, kErrShape);
    return;
  }
  const float* row = p.scores + static_cast<int64_t>(t) * p.stride;
  uint32_t u[E];
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  // All of the thread's loads are issued before any is used.  The row is
  // 16-byte aligned with a stride that is a multiple of 4, so the float4
  // holding key n-1 lies in the row; its entries past n are never used.
  float4 v4[E4];
#pragma unroll
  for (int e = 0; e < E4; ++e) {
    const int key0 = 4 * (e * kThreads + tid);
    v4[e] = key0 < n ? __ldcs(reinterpret_cast<const float4*>(row + key0)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int e = 0; e < E4; ++e) {
    const int key0 = 4 * (e * kThreads + tid);
    const float4 v = v4[e];
    const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      u[4 * e + q] = ordered(f[q]);
      if (key0 + q < n) {
        kmin = min(kmin, u[4 * e + q]);
        kmax = max(kmax, u[4 * e + q]);
      }
    }
  }
  auto valid = [&](int i) { return 4 * ((i >> 2) * kThreads + tid) + (i & 3) < n; };
  // n <= 2048 * E4 and page_size >= 8, so the valid keys span at most 256 * E4 pages
  const int npages = min(p.max_pages, (n + p.page_size - 1) >> p.page_shift);
  for (int i = tid; i < npages; i += kThreads) ptab[i] = p.page_table[static_cast<int64_t>(b) * p.max_pages + i];
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    s_wmin[warp] = kmin;
    s_wmax[warp] = kmax;
  }
  __syncthreads();
  kmin = s_wmin[0];
  kmax = s_wmax[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    kmin = min(kmin, s_wmin[w]);
    kmax = max(kmax, s_wmax[w]);
  }
  // ---- digits.  Keys matching (hi_mask, hi_val) are the candidates; krem of
  // them are still to be taken.
  int krem = k;
  uint32_t hi_mask = 0xffffffffu, hi_val = kmax;  // all keys equal: every key ties kmax
  bool whole = false;                             // the candidates are all taken
  const uint32_t diff = kmin ^ kmax;
  if (diff != 0) {
    int top = 31 - __clz(diff);
    hi_mask = top == 31 ? 0u : ~((2u << top) - 1u);
    hi_val = kmax & hi_mask;
    bool first = true;
    while (top >= 0) {
      const int sh = max(0, top - 10);
      const uint32_t dmask = (1u << (top - sh + 1)) - 1u;
      for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
      __syncthreads();
      if (first) {  // every valid key lies between kmin and kmax, so it has their common prefix
#pragma unroll
        for (int i = 0; i < E; ++i)
          if (valid(i)) atomicAdd(&hist[(u[i] >> sh) & dmask], 1u);
        first = false;
      } else {
#pragma unroll
        for (int i = 0; i < E; ++i)
          if (valid(i) && (u[i] & hi_mask) == hi_val) atomicAdd(&hist[(u[i] >> sh) & dmask], 1u);
      }
      __syncthreads();
      const int bin = select_bin(hist, krem, warp_tot, &sh_bin, &sh_above, &sh_cnt);
      hi_val |= static_cast<uint32_t>(bin) << sh;
      hi_mask |= dmask << sh;
      top = sh - 1;
      if (sh_cnt == krem) {  // uniform: read after the barrier inside select_bin
        whole = true;
        break;
      }
    }
  }
  if (whole) {
    // ---- compaction when the last digit's bin was taken whole: the taken
    // keys are exactly the valid keys >= hi_val (no tie to break), one flag
    // a key.  Key 4e+j of this thread has its flag at bit 4e+j of mk; the
    // per-e counts (<= 4 a thread, <= 128 a warp) are packed four e to a
    // word for one lane scan.
    constexpr int NP = (E4 + 3) / 4;
    static_assert(E4 <= 8, "the taken flags of a thread fit one 32-bit word");
    uint32_t mk = 0u, cw[NP];
#pragma unroll
    for (int w = 0; w < NP; ++w) cw[w] = 0u;
#pragma unroll
    for (int e = 0; e < E4; ++e) {
      uint32_t m = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) m |= (valid(4 * e + j) && u[4 * e + j] >= hi_val ? 1u : 0u) << j;
      mk |= m << (4 * e);
      cw[e >> 2] |= static_cast<uint32_t>(__popc(m)) << (8 * (e & 3));
    }
    uint32_t lx[NP];
#pragma unroll
    for (int w = 0; w < NP; ++w) {
      uint32_t x = cw[w];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      lx[w] = x - cw[w];
      if (lane == 31) cnt_p[w][warp] = x;
    }
    __syncthreads();
    if (warp == 0) {
      // exclusive base of each (e, warp) in key order (e major)
      uint32_t run = 0u;
#pragma unroll
      for (int e = 0; e < E4; ++e) {
        const uint32_t v = lane < kWarps ? (cnt_p[e >> 2][lane] >> (8 * (e & 3))) & 0xffu : 0u;
        uint32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        if (lane < kWarps) cnt_w[e][lane] = run + x - v;
        run += __shfl_sync(0xffffffffu, x, 31);
      }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E4; ++e) {
      const uint32_t m = (mk >> (4 * e)) & 0xfu;
      if (m == 0u) continue;
      int o = static_cast<int>(cnt_w[e][warp] + ((lx[e >> 2] >> (8 * (e & 3))) & 0xffu));
      if (o + __popc(m) > k) {
        atomicOr(p.err, kErrShape);
        continue;
      }
      const int key0 = 4 * (e * kThreads + tid);
      const int pg = key0 >> p.page_shift;  // page_size >= 8: the four keys share a page
      const int pid = pg < npages ? ptab[pg] : -1;
      if (pid < 0) atomicOr(p.err, kErrPage);
      const uint32_t row0 = pid < 0 ? 0xFFFFFFFFu
                                    : (static_cast<uint32_t>(pid) << p.page_shift) |
                                          static_cast<uint32_t>(key0 & (p.page_size - 1));
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if ((m >> j) & 1u) out[o++] = pid < 0 ? row0 : row0 + j;
    }
    if (tid == 0) p.lens[t] = static_cast<uint32_t>(k);
    return;
  }
  // ---- compaction in key order.  Per key two flags, taken once: gt (above
  // the candidates' prefix, or a candidate of a bin taken whole) and tie (a
  // candidate, taken while fewer than krem ties precede it).  Key 4e+j of
  // this thread has its gt flag at bit j and its tie flag at bit 4+j of byte
  // e&3 of fl[e>>2].
  const uint32_t bin_max = hi_val | ~hi_mask;
  uint32_t fl[(E4 + 3) / 4];
#pragma unroll
  for (int w = 0; w < (E4 + 3) / 4; ++w) fl[w] = 0u;
#pragma unroll
  for (int e = 0; e < E4; ++e) {
    uint32_t byte = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = 4 * e + j;
      const bool ok = valid(i);
      const bool cand = ok && (u[i] & hi_mask) == hi_val;
      const bool gt = (ok && u[i] > bin_max) || (whole && cand);
      const bool tie = !whole && cand;
      byte |= (gt ? 1u : 0u) << j;
      byte |= (tie ? 1u : 0u) << (4 + j);
    }
    fl[e >> 2] |= byte << (8 * (e & 3));
  }
  auto flags = [&](int e) { return (fl[e >> 2] >> (8 * (e & 3))) & 0xffu; };
  // Lane prefix sums of the two counts, two e per 32-bit word: e's gt count
  // in bits 16(e&1)..+7 and its tie count in the next 8 bits.  A warp holds
  // at most 128 of either per e, so the 8-bit fields never carry.
  constexpr int NW = (E4 + 1) / 2;
  uint32_t lex[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    uint32_t c = 0u;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (2 * w + h >= E4) continue;
      const uint32_t f = flags(2 * w + h);
      c |= (static_cast<uint32_t>(__popc(f & 0xfu)) | (static_cast<uint32_t>(__popc(f >> 4)) << 8)) << (16 * h);
    }
    uint32_t x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    lex[w] = x - c;
    if (lane == 31) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (2 * w + h >= E4) continue;
        const uint32_t tot = (x >> (16 * h)) & 0xffffu;
        cnt_w[2 * w + h][warp] = (tot & 0xffu) | ((tot >> 8) << 16);  // gt | tie << 16
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive prefix over (e, warp) in key order, both counts in one word
    // (a row holds at most 2048 * E4 <= 16384 keys); lane l takes entries
    // l, l + 32, ...
    uint32_t run = 0u;
    for (int base = 0; base < E4 * kWarps; base += 32) {
      const int idx = base + lane;
      const uint32_t v = idx < E4 * kWarps ? cnt_w[idx / kWarps][idx % kWarps] : 0u;
      uint32_t x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      __syncwarp();
      if (idx < E4 * kWarps) cnt_w[idx / kWarps][idx % kWarps] = run + x - v;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  __syncthreads();
  // The emitted position of a taken key is the number of taken keys before
  // it: the gt keys before it plus min(ties before it, krem).
#pragma unroll
  for (int e = 0; e < E4; ++e) {
    const uint32_t f = flags(e);
    if (f == 0u) continue;
    const uint32_t cw = cnt_w[e][warp];
    const uint32_t lx = (lex[e >> 1] >> (16 * (e & 1))) & 0xffffu;
    int gb = static_cast<int>((cw & 0xffffu) + (lx & 0xffu));
    int qb = static_cast<int>((cw >> 16) + (lx >> 8));
    const int key0 = 4 * (e * kThreads + tid);
    const int pg = key0 >> p.page_shift;  // page_size >= 8: the four keys share a page
    const int pid = pg < npages ? ptab[pg] : -1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool gt = (f >> j) & 1u, tie = (f >> (4 + j)) & 1u;
      if (gt || (tie && qb < krem)) {
        const int o = gb + min(qb, krem);
        if (o >= k) {
          atomicOr(p.err, kErrShape);
        } else if (pid < 0) {
          atomicOr(p.err, kErrPage);
          out[o] = 0xFFFFFFFFu;
        } else {
          out[o] = (static_cast<uint32_t>(pid) << p.page_shift) |
                   static_cast<uint32_t>((key0 + j) & (p.page_size - 1));
        }
      }
      gb += gt ? 1 : 0;
      qb += tie ? 1 : 0;
    }
  }
  if (tid == 0) p.lens[t] = static_cast<uint32_t>(k);
}

__global__ void __launch_bounds__(kThreads, 3) topk_kernel(const Params p) {
  extern __shared__ uint32_t smem_dyn[];
  uint32_t* cache = smem_dyn;                 // the row, as ordered keys
  uint32_t* cand = smem_dyn + p.cache_cap;    // candidate list
  int* ptab = reinterpret_cast<int*>(cand + p.cand_cap);  // page ids of the token's sequence
  __shared__ uint32_t hist[kBins];
  __shared__ int warp_tot[kWarps + 1];
  __shared__ uint32_t s_wmin[kWarps], s_wmax[kWarps];
  __shared__ int sh_b, sh_bin, sh_above, s_ncand;

  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid < 32) {
    // sequence of token t: the number of sequence ends cu_q[b+1] <= t
    int cnt = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int bb = b0 + tid;
      cnt += __popc(__ballot_sync(0xffffffffu, bb < p.B && p.cu_q[bb + 1] <= t));
    }
    if (tid == 0) sh_b = min(cnt, p.B - 1);
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

  // the sequence's page ids, for the logical -> physical row mapping
  const int npages = min(p.max_pages, (n + p.page_size - 1) / p.page_size);
  const bool pt_cached = npages <= p.pt_cap;
  for (int i = tid; i < (pt_cached ? npages : 0); i += kThreads)
    ptab[i] = p.page_table[static_cast<int64_t>(b) * p.max_pages + i];
  const float* row = p.scores + static_cast<int64_t>(t) * p.stride;
  const bool cached = n <= p.cache_cap;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  if (cached) {
    const int n4 = n >> 2;
    const float4* row4 = reinterpret_cast<const float4*>(row);
    for (int i = tid; i < n4; i += kThreads) {
      const float4 v = __ldcs(row4 + i);  // read once: stream past L2
      uint4 u;
      u.x = ordered(v.x); u.y = ordered(v.y); u.z = ordered(v.z); u.w = ordered(v.w);
      reinterpret_cast<uint4*>(cache)[i] = u;
      kmin = min(kmin, min(min(u.x, u.y), min(u.z, u.w)));
      kmax = max(kmax, max(max(u.x, u.y), max(u.z, u.w)));
    }
    for (int i = (n4 << 2) + tid; i < n; i += kThreads) {
      const uint32_t u = ordered(row[i]);
      cache[i] = u;
      kmin = min(kmin, u);
      kmax = max(kmax, u);
    }
  } else {
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t u = ordered(row[i]);
      kmin = min(kmin, u);
      kmax = max(kmax, u);
    }
  }
  auto key_at = [&](int i) -> uint32_t { return cached ? cache[i] : ordered(row[i]); };

  // ---- the bin of the k-th largest ordered key.  Bits above the highest
  // bit in which the row's keys differ are common to every key, so the first
  // 11-bit digit starts there.
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if ((tid & 31) == 0) {
    s_wmin[tid >> 5] = kmin;
    s_wmax[tid >> 5] = kmax;
  }
  for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
  if (tid == 0) s_ncand = 0;
  __syncthreads();
  kmin = s_wmin[0];
  kmax = s_wmax[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) {
    kmin = min(kmin, s_wmin[w]);
    kmax = max(kmax, s_wmax[w]);
  }
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t lt = (1u << lane) - 1u;
  // warp w owns the keys [w*span, (w+1)*span); lane l reads key base + 32m + l
  const int span = ((n + kWarps - 1) / kWarps + 31) & ~31;
  const int w0 = min(n, warp * span), w1 = min(n, w0 + span);
  const uint32_t diff = kmin ^ kmax;
  int krem = k;
  uint32_t thr = kmax;  // all keys equal: every key is a tie of kmax
  if (diff != 0) {
    int top = 31 - __clz(diff);
    uint32_t hi_mask = top == 31 ? 0u : ~((2u << top) - 1u);
    uint32_t hi_val = kmax & hi_mask;
    // pass over the whole row
    int sh = max(0, top - 10);
    uint32_t dmask = (1u << (top - sh + 1)) - 1u;
    for (int i = tid; i < n; i += kThreads) atomicAdd(&hist[(key_at(i) >> sh) & dmask], 1u);
    __syncthreads();
    int bin = select_bin(hist, krem, warp_tot, &sh_bin, &sh_above);
    hi_val |= static_cast<uint32_t>(bin) << sh;
    hi_mask |= dmask << sh;
    top = sh - 1;
    // krem keys are still to be taken from the bin (hi_val, hi_mask); every key
    // above the bin's largest value is taken
    const uint32_t bin_max = hi_val | ~hi_mask;
    // ---- candidates: count each range's keys above the bin, list the bin's keys
    int nabove = 0;
    const int ncand_cap = p.cand_cap;
    for (int base = w0; base < w1; base += 32) {
      const int i = base + lane;
      const uint32_t u = i < w1 ? key_at(i) : 0u;
      nabove += __popc(__ballot_sync(0xffffffffu, i < w1 && u > bin_max));
      const bool inb = i < w1 && (u & hi_mask) == hi_val;
      const uint32_t bm = __ballot_sync(0xffffffffu, inb);
      if (bm) {
        int c0 = 0;
        if (lane == 0) c0 = atomicAdd(&s_ncand, __popc(bm));
        c0 = __shfl_sync(0xffffffffu, c0, 0);
        const int slot = c0 + __popc(bm & lt);
        if (inb && slot < ncand_cap) cand[slot] = static_cast<uint32_t>(i);
      }
    }
    __syncthreads();  // s_wmin / s_wmax / hist are reused below
    const int nc = s_ncand;
    if (nc <= kRankCap && n <= kBins * 32) {
      // ---- short list: rank each candidate by (score desc, key asc); the
      // first krem are taken, marked in a bitmap (hist reused) and counted
      // per warp range.
      uint32_t* taken = hist;
      int* above_w = reinterpret_cast<int*>(s_wmin);
      int* cand_w = reinterpret_cast<int*>(s_wmax);
      for (int i = tid; i < (n + 31) / 32; i += kThreads) taken[i] = 0u;
      if (lane == 0) above_w[warp] = nabove;
      if (tid < kWarps) cand_w[tid] = 0;
      __syncthreads();
      for (int c = tid; c < nc; c += kThreads) {
        const int ic = static_cast<int>(cand[c]);
        const uint32_t uc = key_at(ic);
        int rank = 0;
        for (int d = 0; d < nc; ++d) {
          const int id = static_cast<int>(cand[d]);
          const uint32_t ud = key_at(id);
          rank += (ud > uc || (ud == uc && id < ic)) ? 1 : 0;
        }
        if (rank < krem) {
          atomicOr(&taken[ic >> 5], 1u << (ic & 31));
          atomicAdd(&cand_w[ic / span], 1);
        }
      }
      __syncthreads();
      // ---- one stable compaction pass in logical-key order
      int pos = 0;
      for (int w = 0; w < warp; ++w) pos += above_w[w] + cand_w[w];
      for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t u = i < w1 ? key_at(i) : 0u;
        const bool sel = i < w1 && (u > bin_max || ((u & hi_mask) == hi_val && ((taken[i >> 5] >> (i & 31)) & 1u)));
        const uint32_t bsel = __ballot_sync(0xffffffffu, sel);
        if (sel) emit(p, b, pt_cached ? ptab : nullptr, npages, out, pos + __popc(bsel & lt), i);
        pos += __popc(bsel);
      }
      if (tid == 0) p.lens[t] = static_cast<uint32_t>(k);
      return;
    }
    // ---- long list: resolve the remaining digits on the candidates (or on
    // the whole row when the list overflowed), then the two-pass compaction
    const bool in_list = nc <= ncand_cap;
    while (top >= 0) {
      sh = max(0, top - 10);
      dmask = (1u << (top - sh + 1)) - 1u;
      for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
      __syncthreads();
      if (in_list) {
        for (int i = tid; i < nc; i += kThreads) {
          const uint32_t u = key_at(static_cast<int>(cand[i]));
          if ((u & hi_mask) == hi_val) atomicAdd(&hist[(u >> sh) & dmask], 1u);
        }
      } else {
        for (int i = tid; i < n; i += kThreads) {
          const uint32_t u = key_at(i);
          if ((u & hi_mask) == hi_val) atomicAdd(&hist[(u >> sh) & dmask], 1u);
        }
      }
      __syncthreads();
      bin = select_bin(hist, krem, warp_tot, &sh_bin, &sh_above);
      hi_val |= static_cast<uint32_t>(bin) << sh;
      hi_mask |= dmask << sh;
      top = sh - 1;
    }
    thr = hi_val;
  }
  // thr = exact k-th largest key; krem of its ties are taken (lowest keys first)

  // ---- stable compaction in logical-key order, two passes: per-range counts
  // of keys above thr and of ties, then the ballot-ordered writes.
  __syncthreads();  // s_wmin / s_wmax are reused below
  int ngt = 0, neq = 0;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t u = i < w1 ? key_at(i) : 0u;
    ngt += __popc(__ballot_sync(0xffffffffu, i < w1 && u > thr));
    neq += __popc(__ballot_sync(0xffffffffu, i < w1 && u == thr));
  }
  if (lane == 0) {
    s_wmin[warp] = static_cast<uint32_t>(ngt);
    s_wmax[warp] = static_cast<uint32_t>(neq);
  }
  __syncthreads();
  int sel_base = 0, tie_base = 0;
  for (int w = 0; w < warp; ++w) {
    const int g = static_cast<int>(s_wmin[w]), e = static_cast<int>(s_wmax[w]);
    sel_base += g + max(0, min(e, krem - tie_base));
    tie_base += e;
  }
  int pos = sel_base, tie = tie_base;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t u = i < w1 ? key_at(i) : 0u;
    const bool gt = i < w1 && u > thr, eq = i < w1 && u == thr;
    const uint32_t beq = __ballot_sync(0xffffffffu, eq);
    const int my_tie = tie + __popc(beq & lt);
    const bool sel = gt || (eq && my_tie < krem);
    const uint32_t bsel = __ballot_sync(0xffffffffu, sel);
    if (sel) emit(p, b, pt_cached ? ptab : nullptr, npages, out, pos + __popc(bsel & lt), i);
    pos += __popc(bsel);
    tie += __popc(beq);
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
  const int64_t cap = (std::min<int64_t>(score_stride, 40 * 1024) + 3) & ~int64_t(3);
  const int64_t cand_cap = 2048;
  const int64_t pt_cap = std::min<int64_t>(seqs.max_pages, 4096);
  const size_t smem = static_cast<size_t>(cap + cand_cap + pt_cap) * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return fail_cuda(e, "topk smem attribute");
  Params p{scores, score_stride, seqs.cu_q, seqs.kv_len, seqs.page_table, seqs.B, seqs.max_pages,
           seqs.page_size, seqs.T, __builtin_ctz(static_cast<unsigned>(seqs.page_size)), k, indices, topk_lengths,
           static_cast<int>(cap), static_cast<int>(cand_cap), static_cast<int>(pt_cap), err};
  if (score_stride <= 2048 * 4)
    topk_reg_kernel<4><<<seqs.T, kThreads, 0, stream>>>(p);
  else if (score_stride <= 2048 * 8)
    topk_reg_kernel<8><<<seqs.T, kThreads, 0, stream>>>(p);
  else
    topk_kernel<<<seqs.T, kThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "topk launch");
  return SMLA_OK;
}

}  // namespace smla
