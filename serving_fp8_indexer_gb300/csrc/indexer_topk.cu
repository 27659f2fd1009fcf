// Fused FP8 lightning indexer + per-token top-k: the score rows never leave
// the SM.
//
// "sparse_index_fp8_sm100" (module summary) computes
//   score[t, key] = k_scale[key] * sum_h relu(q[t,h] . k[key]) * q_scale[t,h]
// into a score buffer that the top-k stage then reads; the page leaves the
// causal -inf fill and its fusion with the following stages to later work.
// Here the two stages run in one persistent kernel: a CTA owns a tile of TOK
// query tokens (MMA N = TOK * H_idx = 128 (token, head) columns) and computes
// every key tile up to the tile's last position on the tensor cores, exactly
// as the standalone indexer does (same MMA, same relu / q_scale / head-sum /
// k_scale arithmetic in the same order, so the scores are the same floats).
// The epilogue writes each token's scores for keys 0..pos into a shared-
// memory row (two buffers of TOK x L floats, L = 16384 / TOK), and four
// selector warps take the token tile's top-k from those rows while the
// epilogue already fills the other buffer with the next tile.  The selection
// is a radix select over order-preserving 32-bit keys (11-bit digits from the
// highest bit in which the row differs) with a stable compaction in logical
// key order; it emits physical rows (page table) and topk_lengths, and ties
// at the k-th value go to the lower logical key, as smla_topk does.
//
// Warp roles (20 warps): 0 TMA producer (q per
// tile, K tiles through the page table), 1 MMA issuer and TMEM owner, 2-3
// idle, 4-11 epilogue (TMEM lane quarter x 64-column half), 12-15
// selectors.
#include <algorithm>

#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {
namespace fit {

constexpr int kDepth = 128;
constexpr int kBM = 128;                  // keys per tile (MMA M)
constexpr int kBN = 128;                  // (token, head) columns per tile (MMA N)
constexpr int kStages = 3;                // K tile ring
constexpr int kEpiWarps = 8;
constexpr int kSelGroups = 2;             // selector groups: one token of a tile each at a time
constexpr int kGrpWarps = 4;
constexpr int kGrpThreads = 32 * kGrpWarps;
constexpr int kSelWarps = kSelGroups * kGrpWarps;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kSelThreads = 32 * kSelWarps;
constexpr int kEpiWarp0 = 4;
constexpr int kSelWarp0 = kEpiWarp0 + kEpiWarps;
constexpr int kThreads = 32 * (kSelWarp0 + kSelWarps);
static_assert(kThreads == 640 && kEpiWarp0 % 4 == 0, "epilogue warp w reads TMEM lane quarter w % 4");
constexpr int kSliceCols = kBN / 2;       // columns per epilogue warp
constexpr int kRowCap = 16384;            // floats per score buffer (TOK rows of L)
constexpr int kMaxPages = 1024;           // page ids staged per tile
constexpr int kBins = 2048;               // 11-bit digits
constexpr int kBinsPerThread = kBins / kGrpThreads;
constexpr int kMaxE4 = 16;                // float4 groups per selector thread (rows of <= 8192 keys)
// TMEM accumulators (measured on the end-to-end chunk: four, letting the
// MMA run three tiles ahead, 2.464 ms; two 2.467 ms)
constexpr int kAcc = 2;
constexpr uint32_t kTmemCols = kAcc * kBN;
constexpr int kBarEpi = 1, kBarSel0 = 2;  // named barriers: epilogue, selector group g at kBarSel0 + g
constexpr int kMaxTok = kBN / 4;          // tokens per tile at the smallest H_idx
static_assert(kGrpThreads * 4 * kMaxE4 == 8192, "a selector group's per-group counts cover a row of 8192 keys");

struct Params {
  const float* q_scale;
  const float* k_scale;
  int64_t phys_rows;
  const int32_t* cu_q;
  const int32_t* kv_len;
  const int32_t* page_table;
  int B, max_pages, page_size, page_shift;
  int L;         // score row capacity (keys) = kRowCap / TOK
  int k;
  uint32_t* indices;
  uint32_t* lens;
  int box_rows;  // rows per K TMA box = min(page_size, 128)
  unsigned* err;
};

struct __align__(1024) Smem {
  uint8_t q[kBN * kDepth];           // SW128 K-major: 128 rows x 128 B
  uint8_t k[kStages][kBM * kDepth];  // SW128 K-major
  float scores[2][kRowCap];          // [buffer][token * L + key]
  int pages[2][kMaxPages];           // the tile's sequence page ids, per score buffer
  int ppages[kMaxPages];             // the producer's copy for the tile it is loading
  struct Sel {  // one selector group's scratch
    uint32_t hist[kBins];
    uint32_t cnt_w[kMaxE4][kGrpWarps];  // per (float4 group, warp): gt count | tie count << 16
    int wtot[kGrpWarps + 1];
    int sh_bin, sh_above, sh_cnt;
  } sel[kSelGroups];
  float qs[kBN];
  // each token's smallest and largest score of the tile (order-preserving
  // keys), taken by the epilogue while it writes the rows
  uint32_t tmin[2][kMaxTok], tmax[2][kMaxTok];
  unsigned long long bar_q, bar_qfree, bar_kfull[kStages], bar_kempty[kStages], bar_afull[kAcc], bar_aempty[kAcc];
  unsigned long long bar_sfull[2], bar_sfree[2], bar_drain;
  uint32_t tmem_base;
  int k_issued, k_landed, q_issued, q_landed;
};

// Tile w -> (sequence b, token tile tt); b = -1 past the last tile.  The whole
// warp calls.  Sequences whose shape is invalid (kv_len < q_len, or rows
// longer than L) contribute no tiles and are flagged.
__device__ __forceinline__ void tile_of(const Params& p, int w, int TOK, int& b, int& tt) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  b = -1;
  tt = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int bb = b0 + lane;
    int n = 0;
    if (bb < p.B) {
      const int ql = p.cu_q[bb + 1] - p.cu_q[bb];
      const int kl = p.kv_len[bb];
      const bool ok = kl >= ql && kl <= p.L;
      n = (ql > 0 && ok) ? (ql + TOK - 1) / TOK : 0;
      if (ql > 0 && !ok) atomicOr(p.err, kErrShape);
    }
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = base + incl - n;
    const unsigned ball = __ballot_sync(0xffffffffu, n > 0 && w >= excl && w < excl + n);
    if (ball) {
      const int src = __ffs(ball) - 1;
      b = __shfl_sync(0xffffffffu, bb, src);
      tt = __shfl_sync(0xffffffffu, w - excl, src);
      return;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
}

struct Tile {
  int b, t0, ntok, pos0, nt;  // first token, tokens, position of the first, key tiles
};
__device__ __forceinline__ Tile tile_make(const Params& p, int b, int tt, int TOK) {
  Tile x;
  x.b = b;
  const int cu0 = p.cu_q[b];
  const int q_len = p.cu_q[b + 1] - cu0;
  const int kvl = p.kv_len[b];
  x.t0 = cu0 + tt * TOK;
  x.ntok = min(TOK, q_len - tt * TOK);
  x.pos0 = kvl - q_len + tt * TOK;
  x.nt = (x.pos0 + x.ntok - 1) / kBM + 1;  // key tiles up to the last token's position
  return x;
}

// Larger float -> larger unsigned key (-0 sorts just below +0).
__device__ __forceinline__ uint32_t ordered(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t phys_of(const int* pages, int shift, int key) {
  const int pid = pages[key >> shift];
  return pid < 0 ? 0xFFFFFFFFu : (static_cast<uint32_t>(pid) << shift) | static_cast<uint32_t>(key & ((1 << shift) - 1));
}

// Exclusive prefix of v over a selector group's threads (thread order);
// returns it and leaves the total in g.wtot[kGrpWarps].  tid: the thread's
// index in the group; bar: the group's named barrier.
__device__ __forceinline__ int sel_scan(Smem::Sel& g, int v, int tid, int bar) {
  const int lane = tid & 31, wp = tid >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) g.wtot[wp] = incl;
  named_bar_sync(bar, kGrpThreads);
  if (tid == 0) {
    int run = 0;
    for (int i = 0; i < kGrpWarps; ++i) {
      const int x = g.wtot[i];
      g.wtot[i] = run;
      run += x;
    }
    g.wtot[kGrpWarps] = run;
  }
  named_bar_sync(bar, kGrpThreads);
  return g.wtot[wp] + incl - v;
}

// Top-k of one score row in shared memory (n > k valid keys) by one selector
// group: writes the physical rows of the k selected keys, in ascending
// logical-key order, to out[0..k).  kmin / kmax: the row's smallest and
// largest order-preserving keys (taken by the epilogue).  Thread tid (of the
// group's 128) handles the keys 4 * (e * 128 + tid) + u (u < 4) of every
// float4 group e; each pass reads them again from the row (conflict-free
// float4 loads) rather than holding them in registers.
__device__ __forceinline__ void select_row(Smem::Sel& g, int tid, int bar, const float* row, int n, int k,
                                           uint32_t kmin, uint32_t kmax, const int* pages, int shift, uint32_t* out,
                                           unsigned* err) {
  const int lane = tid & 31, wp = tid >> 5;
  const int E4 = (n + 4 * kGrpThreads - 1) / (4 * kGrpThreads);
  const float4* row4 = reinterpret_cast<const float4*>(row);
  // this thread's four keys of group e, as ordered keys, and how many of the
  // four are valid
  auto group = [&](int e, uint32_t (&u)[4]) -> int {
    const int key0 = 4 * (e * kGrpThreads + tid);
    const float4 v = row4[e * kGrpThreads + tid];  // inside the row: key0 + 3 < L
    u[0] = ordered(v.x);
    u[1] = ordered(v.y);
    u[2] = ordered(v.z);
    u[3] = ordered(v.w);
    return min(4, max(0, n - key0));
  };
  // ---- digits: keys matching (hi_mask, hi_val) are the candidates, krem of
  // them still to be taken
  int krem = k;
  uint32_t hi_mask = 0xffffffffu, hi_val = kmax;  // all keys equal: every key ties kmax
  bool whole = false;                             // the candidates are all taken
  const uint32_t diff = kmin ^ kmax;
  if (diff != 0) {
    int top = 31 - __clz(diff);
    hi_mask = top == 31 ? 0u : ~((2u << top) - 1u);
    hi_val = kmax & hi_mask;
    while (top >= 0) {
      const int sh = max(0, top - 10);
      const uint32_t dmask = (1u << (top - sh + 1)) - 1u;
      named_bar_sync(bar, kGrpThreads);  // readers of the previous histogram are done
      for (int i = tid; i < kBins; i += kGrpThreads) g.hist[i] = 0;
      named_bar_sync(bar, kGrpThreads);
#pragma unroll 4
      for (int e = 0; e < E4; ++e) {
        uint32_t u[4];
        const int nv = group(e, u);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q < nv && (u[q] & hi_mask) == hi_val) atomicAdd(&g.hist[(u[q] >> sh) & dmask], 1u);
      }
      named_bar_sync(bar, kGrpThreads);
      // bin of the krem-th largest candidate: thread rt owns bins [rt*16, rt*16+16)
      const int rt = kGrpThreads - 1 - tid;
      int local = 0;
#pragma unroll
      for (int j = 0; j < kBinsPerThread; ++j) local += g.hist[rt * kBinsPerThread + j];
      int c = sel_scan(g, local, tid, bar);
#pragma unroll
      for (int j = kBinsPerThread - 1; j >= 0; --j) {
        const int bin = rt * kBinsPerThread + j;
        const int h = g.hist[bin];
        if (c < krem && c + h >= krem) {
          g.sh_bin = bin;
          g.sh_above = c;
          g.sh_cnt = h;
        }
        c += h;
      }
      named_bar_sync(bar, kGrpThreads);
      const int bin = g.sh_bin;
      krem -= g.sh_above;
      const int cnt = g.sh_cnt;
      hi_val |= static_cast<uint32_t>(bin) << sh;
      hi_mask |= dmask << sh;
      top = sh - 1;
      if (cnt == krem) {
        whole = true;
        break;
      }
    }
  }
  // ---- compaction in key order (e, tid, u): gt = above the candidates (or
  // a candidate of a bin taken whole), tie = a candidate, taken while fewer
  // than krem ties precede it.  Pass 1 counts both per (e, warp); pass 2
  // recomputes the flags and lane prefixes and emits.
  const uint32_t bin_max = hi_val | ~hi_mask;
  // flags of group e: gt at bits 0..3, tie at bits 4..7
  auto flags = [&](int e) -> uint32_t {
    uint32_t u[4];
    const int nv = group(e, u);
    uint32_t f = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool ok = j < nv;
      const bool cand = ok && (u[j] & hi_mask) == hi_val;
      const bool gt = (ok && u[j] > bin_max) || (whole && cand);
      const bool tie = !whole && cand;
      f |= (gt ? 1u : 0u) << j;
      f |= (tie ? 1u : 0u) << (4 + j);
    }
    return f;
  };
  // lane prefix of both counts (8-bit fields: a warp holds at most 128 of
  // either per group); returns the exclusive prefix, *tot the warp's totals
  auto lane_prefix = [&](uint32_t f, uint32_t* tot) -> uint32_t {
    const uint32_t c = static_cast<uint32_t>(__popc(f & 0xfu)) | (static_cast<uint32_t>(__popc(f >> 4)) << 8);
    uint32_t x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    *tot = __shfl_sync(0xffffffffu, x, 31);
    return x - c;
  };
#pragma unroll 4
  for (int e = 0; e < kMaxE4; ++e) {
    uint32_t tot = 0u;
    if (e < E4) lane_prefix(flags(e), &tot);
    if (lane == 0) g.cnt_w[e][wp] = (tot & 0xffu) | ((tot >> 8) << 16);
  }
  named_bar_sync(bar, kGrpThreads);
  if (tid < 32) {
    // exclusive prefix over (e, warp) in key order; both counts in one word
    uint32_t run = 0u;
    for (int base = 0; base < kMaxE4 * kGrpWarps; base += 32) {
      const int idx = base + lane;
      const uint32_t v = g.cnt_w[idx / kGrpWarps][idx % kGrpWarps];
      uint32_t x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      __syncwarp();
      g.cnt_w[idx / kGrpWarps][idx % kGrpWarps] = run + x - v;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  named_bar_sync(bar, kGrpThreads);
#pragma unroll 2
  for (int e = 0; e < E4; ++e) {
    const uint32_t f = flags(e);
    uint32_t tot;
    const uint32_t lx = lane_prefix(f, &tot);
    if (f == 0u) continue;
    const uint32_t cw = g.cnt_w[e][wp];
    int gb = static_cast<int>((cw & 0xffffu) + (lx & 0xffu));
    int qb = static_cast<int>((cw >> 16) + ((lx >> 8) & 0xffu));
    const int key0 = 4 * (e * kGrpThreads + tid);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool gt = (f >> j) & 1u, tie = (f >> (4 + j)) & 1u;
      if (gt || (tie && qb < krem)) {
        const int o = gb + min(qb, krem);
        if (o < k) {
          const uint32_t r = phys_of(pages, shift, key0 + j);
          if (r == 0xFFFFFFFFu) atomicOr(err, kErrPage);
          out[o] = r;
        } else {
          atomicOr(err, kErrShape);
        }
      }
      gb += gt ? 1 : 0;
      qb += tie ? 1 : 0;
    }
  }
  named_bar_sync(bar, kGrpThreads);  // g.cnt_w / hist are reused by the next row
}

template <int HIDX>
__global__ void __launch_bounds__(kThreads, 1)
    fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, const Params p) {
  constexpr int TOK = kBN / HIDX;             // tokens per tile
  constexpr int SLICE_TOK = kSliceCols / HIDX;  // tokens per epilogue column half
  constexpr uint32_t IDESC = idesc_e4m3_f32(kBM, kBN, 0, 0);
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = p.L;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&s.bar_q), 1);
    mbar_init(smem_u32(&s.bar_qfree), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&s.bar_kfull[i]), 1);
      mbar_init(smem_u32(&s.bar_kempty[i]), 1);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(smem_u32(&s.bar_afull[i]), 1);
      mbar_init(smem_u32(&s.bar_aempty[i]), kEpiThreads);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.bar_sfull[i]), kEpiThreads);
      mbar_init(smem_u32(&s.bar_sfree[i]), kSelThreads);
    }
    mbar_init(smem_u32(&s.bar_drain), 1);
    fence_mbar_init();
    s.k_issued = s.k_landed = s.q_issued = s.q_landed = 0;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    int g = 0, it = 0;
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
    }
    for (int w = blockIdx.x; ok; w += gridDim.x, ++it) {
      int b, tt;
      tile_of(p, w, TOK, b, tt);
      if (b < 0) break;
      const Tile x = tile_make(p, b, tt, TOK);
      const int npg = min(kMaxPages, (x.nt * kBM + p.page_size - 1) >> p.page_shift);
      __syncwarp();  // the previous tile's page reads are done
      for (int i = lane; i < npg; i += 32)
        s.ppages[i] = i < p.max_pages ? p.page_table[static_cast<int64_t>(b) * p.max_pages + i] : -1;
      __syncwarp();
      if (lane == 0) {
        // q of this tile, once the previous tile's MMAs have read s.q
        if (it > 0) ok = mbar_wait(smem_u32(&s.bar_qfree), (it - 1) & 1, p.err);
        if (ok) {
          mbar_arrive_expect_tx(smem_u32(&s.bar_q), kBN * kDepth);
          tma_load_2d(smem_u32(s.q), &tm_q, 0, x.t0 * HIDX, smem_u32(&s.bar_q));
          s.q_issued = it + 1;
        }
        const int nbox = kBM / p.box_rows;
        for (int i = 0; ok && i < x.nt; ++i, ++g) {
          const int st = g % kStages;
          if (!mbar_wait(smem_u32(&s.bar_kempty[st]), ((g / kStages) & 1) ^ 1, p.err)) {
            ok = false;
            break;
          }
          int nload = 0;
          int rows[kBM / 8];
          for (int bx = 0; bx < nbox; ++bx) {
            const int key0 = i * kBM + bx * p.box_rows;
            rows[bx] = -1;
            if (key0 > x.pos0 + x.ntok - 1) continue;  // past the tile's last position
            const int pi = key0 >> p.page_shift;
            const int pid = pi < npg ? s.ppages[pi] : -1;
            const int64_t row = static_cast<int64_t>(pid) * p.page_size + (key0 & (p.page_size - 1));
            if (pid < 0 || row + p.box_rows > p.phys_rows) {
              atomicOr(p.err, kErrPage);
              continue;
            }
            rows[bx] = static_cast<int>(row);
            ++nload;
          }
          mbar_arrive_expect_tx(smem_u32(&s.bar_kfull[st]), nload * p.box_rows * kDepth);
          for (int bx = 0; bx < nbox; ++bx)
            if (rows[bx] >= 0)
              tma_load_2d(smem_u32(s.k[st]) + bx * p.box_rows * kDepth, &tm_k, 0, rows[bx],
                          smem_u32(&s.bar_kfull[st]));
          s.k_issued = g + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    int g = 0, it = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok; w += gridDim.x, ++it) {
      int b, tt;
      tile_of(p, w, TOK, b, tt);
      if (b < 0) break;
      const Tile x = tile_make(p, b, tt, TOK);
      if (lane == 0) {
        ok = mbar_wait(smem_u32(&s.bar_q), it & 1, p.err);
        if (ok) s.q_landed = it + 1;
        const uint32_t q_base = smem_u32(s.q);
        for (int i = 0; ok && i < x.nt; ++i, ++g) {
          const int st = g % kStages, a = g % kAcc;
          if (!mbar_wait(smem_u32(&s.bar_kfull[st]), (g / kStages) & 1, p.err)) {
            ok = false;
            break;
          }
          s.k_landed = g + 1;
          if (!mbar_wait(smem_u32(&s.bar_aempty[a]), ((g / kAcc) & 1) ^ 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k_base = smem_u32(s.k[st]);
#pragma unroll
          for (int kk = 0; kk < kDepth / 32; ++kk) {
            const uint64_t ad = make_sdesc(k_base + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = make_sdesc(q_base + kk * 32, 16, 1024, kSwizzle128B);
            mma_f8f6f4_ss(tmem + a * kBN, ad, bd, IDESC, kk > 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&s.bar_kempty[st]));
          mma_commit(smem_u32(&s.bar_afull[a]));
        }
        if (ok) mma_commit(smem_u32(&s.bar_qfree));  // s.q is free once these MMAs complete
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0) {
      // no MMA may still write TMEM when the CTA tears down
      mma_commit(smem_u32(&s.bar_drain));
      mbar_wait(smem_u32(&s.bar_drain), 0, p.err);
    }
    __syncwarp();
  } else if (warp < kEpiWarp0) {
    // warps 2-3: no role
  } else if (warp < kSelWarp0) {
    // ---------------------------------------------------------------- epilogue
    const int et = threadIdx.x - kEpiWarp0 * 32;
    const int quarter = warp & 3;               // TMEM lanes this warp may access
    const int half = (warp - kEpiWarp0) >> 2;   // columns [half*64, half*64 + 64)
    const int row = quarter * 32 + lane;        // key within the tile
    int g = 0, it = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok; w += gridDim.x, ++it) {
      int b, tt;
      tile_of(p, w, TOK, b, tt);
      if (b < 0) break;
      const Tile x = tile_make(p, b, tt, TOK);
      const int buf = it & 1;
      // the selectors are done with this buffer (tile it - 2)
      if (it >= 2 && !named_bar_and(kBarEpi, kEpiThreads, mbar_wait(smem_u32(&s.bar_sfree[buf]), ((it >> 1) - 1) & 1, p.err))) {
        ok = false;
        break;
      }
      const int npg = min(kMaxPages, (x.nt * kBM + p.page_size - 1) >> p.page_shift);
      for (int i = et; i < npg; i += kEpiThreads)
        s.pages[buf][i] = i < p.max_pages ? p.page_table[static_cast<int64_t>(b) * p.max_pages + i] : -1;
      if (et < kBN) {
        const int tok = et / HIDX, h = et % HIDX;
        s.qs[et] = tok < x.ntok ? p.q_scale[static_cast<int64_t>(x.t0 + tok) * HIDX + h] : 0.f;
      }
      if (et < TOK) {
        s.tmin[buf][et] = 0xffffffffu;
        s.tmax[buf][et] = 0u;
      }
      named_bar_sync(kBarEpi, kEpiThreads);
      const int* pg = s.pages[buf];
      const float* qs = s.qs + half * kSliceCols;
      float* srow = s.scores[buf];
      // k_scale of this lane's key in tile i, from the staged page ids, two tiles ahead
      auto load_ks = [&](int i) -> float {
        const int key = i * kBM + row;
        if (i >= x.nt || key > x.pos0 + x.ntok - 1) return 0.f;
        const int pi = key >> p.page_shift;
        const int pid = pi < npg ? pg[pi] : -1;
        const int64_t pr = (static_cast<int64_t>(pid) << p.page_shift) + (key & (p.page_size - 1));
        return (pid >= 0 && pr < p.phys_rows) ? __ldg(p.k_scale + pr) : 0.f;
      };
      float ks_next = load_ks(0), ks_next2 = load_ks(1);
      for (int i = 0; i < x.nt; ++i, ++g) {
        const int a = g % kAcc;
        const float ks = ks_next;
        ks_next = ks_next2;
        ks_next2 = load_ks(i + 2);
        // warp-uniform (the tcgen05.ld below is warp-collective); a warp that
        // gives up leaves the loop, and the vote after it stops all of them
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&s.bar_afull[a]), (g / kAcc) & 1, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float acc[SLICE_TOK];
#pragma unroll
        for (int j = 0; j < SLICE_TOK; ++j) acc[j] = 0.f;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + a * kBN + half * kSliceCols;
        // relu, x q_scale, summed over each token's heads in head order (the
        // standalone indexer's order, so both produce the same floats); 32
        // columns a load
#pragma unroll
        for (int cb = 0; cb < kSliceCols; cb += 32) {
          uint32_t v[32];
          tmem_ld32(taddr + cb, v);
          tmem_wait_ld_regs(v);
          if (cb + 32 == kSliceCols) {
            tc_fence_before();
            mbar_arrive(smem_u32(&s.bar_aempty[a]));  // the accumulator is in registers
          }
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 q4 = *reinterpret_cast<const float4*>(qs + cb + j);
            const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int uu = 0; uu < 4; ++uu) {
              const int tj = (cb + j + uu) / HIDX;
              acc[tj] = fmaf(fmaxf(__uint_as_float(v[j + uu]), 0.f), qq[uu], acc[tj]);
            }
          }
        }
        const int key = i * kBM + row;
#pragma unroll
        for (int j = 0; j < SLICE_TOK; ++j) {
          const int tok = half * SLICE_TOK + j;
          const bool valid = tok < x.ntok && key <= x.pos0 + tok;
          const float sc = ks * acc[j];
          if (valid) srow[tok * L + key] = sc;
          // the token's smallest and largest score so far (order-preserving keys)
          const uint32_t u = ordered(sc);
          const uint32_t wmn = __reduce_min_sync(0xffffffffu, valid ? u : 0xffffffffu);
          const uint32_t wmx = __reduce_max_sync(0xffffffffu, valid ? u : 0u);
          if (lane == 0 && tok < x.ntok && wmn <= wmx) {
            atomicMin(&s.tmin[buf][tok], wmn);
            atomicMax(&s.tmax[buf][tok], wmx);
          }
        }
      }
      // every epilogue thread arrives here once per tile: a give-up by any
      // warp stops all of them together (no named barrier is left waiting),
      // and no warp restages q_scale while another still reads it
      if (!named_bar_and(kBarEpi, kEpiThreads, ok)) break;
      mbar_arrive(smem_u32(&s.bar_sfull[buf]));  // the tile's score rows are complete
    }
  } else {
    // ---------------------------------------------------------------- selectors
    // group gi takes tokens gi, gi + 2, ... of each tile
    const int gi = (warp - kSelWarp0) / kGrpWarps;
    const int st_id = threadIdx.x - (kSelWarp0 + gi * kGrpWarps) * 32;
    const int bar = kBarSel0 + gi;
    Smem::Sel& sg = s.sel[gi];
    int it = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok; w += gridDim.x, ++it) {
      int b, tt;
      tile_of(p, w, TOK, b, tt);
      if (b < 0) break;
      const Tile x = tile_make(p, b, tt, TOK);
      const int buf = it & 1;
      if (!named_bar_and(bar, kGrpThreads, mbar_wait(smem_u32(&s.bar_sfull[buf]), (it >> 1) & 1, p.err))) {
        ok = false;
        break;
      }
      const int* pg = s.pages[buf];
      for (int tok = gi; tok < x.ntok; tok += kSelGroups) {
        const int t = x.t0 + tok;
        const int n = x.pos0 + tok + 1;  // valid keys 0..pos
        uint32_t* out = p.indices + static_cast<int64_t>(t) * p.k;
        if (n <= p.k) {
          for (int key = st_id; key < n; key += kGrpThreads) {
            const uint32_t r = phys_of(pg, p.page_shift, key);
            if (r == 0xFFFFFFFFu) atomicOr(p.err, kErrPage);
            out[key] = r;
          }
          for (int i = n + st_id; i < p.k; i += kGrpThreads) out[i] = 0xFFFFFFFFu;
          if (st_id == 0) p.lens[t] = static_cast<uint32_t>(n);
        } else {
          select_row(sg, st_id, bar, s.scores[buf] + tok * L, n, p.k, s.tmin[buf][tok], s.tmax[buf][tok], pg,
                     p.page_shift, out, p.err);
          if (st_id == 0) p.lens[t] = static_cast<uint32_t>(p.k);
        }
      }
      named_bar_sync(bar, kGrpThreads);
      mbar_arrive(smem_u32(&s.bar_sfree[buf]));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // after a wait gave up: TMA loads still in flight land before the CTA exits
  // (bounded waits; in the normal case every issued load has landed)
  if (threadIdx.x == 0) {
    for (int i = s.q_landed; i < s.q_issued; ++i) mbar_wait(smem_u32(&s.bar_q), i & 1, p.err);
    for (int i = s.k_landed; i < s.k_issued; ++i)
      mbar_wait(smem_u32(&s.bar_kfull[i % kStages]), (i / kStages) & 1, p.err);
  }
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int HIDX>
static cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const Params& p, int grid,
                            cudaStream_t stream) {
  const size_t smem = sizeof(Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(fused_kernel<HIDX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  fused_kernel<HIDX><<<grid, kThreads, smem, stream>>>(tq, tk, p);
  return cudaGetLastError();
}

}  // namespace fit

int indexer_topk_row_cap(int h_idx) { return h_idx > 0 ? fit::kRowCap / (fit::kBN / h_idx) : 0; }

smla_status_t launch_indexer_topk(const uint8_t* q, const float* q_scale, const uint8_t* k_pool, const float* k_scale,
                                  int64_t phys_rows, const smla_seqs_t& seqs, int h_idx, int k, uint32_t* indices,
                                  uint32_t* topk_lengths, unsigned* err, cudaStream_t stream) {
  using namespace fit;
  static_assert(sizeof(Smem) + 1024 <= 232448, "fused indexer + top-k shared memory exceeds a CTA's 227 KB");
  if (seqs.T == 0 || seqs.B == 0) return SMLA_OK;
  const int tok = kBN / h_idx;
  const int L = indexer_topk_row_cap(h_idx);
  const int box_rows = std::min(seqs.page_size, kBM);
  if ((static_cast<int64_t>(L) + seqs.page_size - 1) / seqs.page_size > kMaxPages)
    return fail(SMLA_ERR_UNSUPPORTED, "fused indexer + top-k: page_size %d too small for %d-key rows", seqs.page_size, L);
  CUtensorMap tq, tk;
  if (!encode_tma_2d_u8(&tq, q, kDepth, static_cast<uint64_t>(seqs.T) * h_idx, kDepth, kBN))
    return fail(SMLA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the fused indexer q tensor map");
  if (!encode_tma_2d_u8(&tk, k_pool, kDepth, static_cast<uint64_t>(phys_rows), kDepth, box_rows))
    return fail(SMLA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the fused indexer K tensor map");
  // persistent: at most one CTA per SM (shared memory), no more than there are tiles
  const int64_t tiles_max = (static_cast<int64_t>(seqs.T) + tok - 1) / tok + seqs.B;
  const int grid = static_cast<int>(std::min<int64_t>(tiles_max, device_sm_count()));
  Params p{q_scale, k_scale, phys_rows, seqs.cu_q, seqs.kv_len, seqs.page_table, seqs.B, seqs.max_pages,
           seqs.page_size, __builtin_ctz(static_cast<unsigned>(seqs.page_size)), L, k, indices, topk_lengths,
           box_rows, err};
  cudaError_t e;
  switch (h_idx) {
    case 4: e = launch_t<4>(tq, tk, p, grid, stream); break;
    case 8: e = launch_t<8>(tq, tk, p, grid, stream); break;
    case 16: e = launch_t<16>(tq, tk, p, grid, stream); break;
    case 32: e = launch_t<32>(tq, tk, p, grid, stream); break;
    case 64: e = launch_t<64>(tq, tk, p, grid, stream); break;
    default: return fail(SMLA_ERR_UNSUPPORTED, "H_idx must be 4, 8, 16, 32 or 64");
  }
  if (e != cudaSuccess) return fail_cuda(e, "fused indexer + top-k launch");
  return SMLA_OK;
}

}  // namespace smla
