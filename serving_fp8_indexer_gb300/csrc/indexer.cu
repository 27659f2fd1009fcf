// Stage 1: FP8 lightning-indexer scores on tcgen05 tensor cores.
//
// "sparse_index_fp8_sm100" (Modular Mojo kernel page), module summary and
// "Layout (crux)":
//   score[t, key] = k_scale[key] * sum_h relu(q[t,h] . k[key]) * q_scale[t,h]
// computed as S^T = K . Q^T with the key tile as the MMA M dimension, so the
// head reduction of a key's row stays inside one thread after tcgen05.ld.
//
// GB300 design (not the page's SM100 one):
//   * MMA 128 keys (M) x 256 (token, head) columns (N) x 128 depth (K),
//     kind::f8f6f4 e4m3 x e4m3 -> f32 in TMEM; 4 instructions of K = 32.
//     With H_idx = 64 one tile covers 4 tokens (256 / H_idx in general).
//   * A work item is (sequence, token tile of up to 4 groups, key chunk).
//     Q and q_scale are loaded once per item; K tiles stream through a
//     4-stage TMA ring, one box per page (page_size >= 128: one box per
//     tile), so the paged cache is read in place.  Each K tile serves every
//     token group of the item (4 MMA tiles of N = 256): a K tile feeding
//     only one group left the kernel bound by the L2 -> shared-memory
//     stream of K (measured on the end-to-end chunk: 1 group 1.63 ms,
//     2 groups 1.44, 4 groups 1.35).  Key tiles wholly past the last
//     token's position are not computed, only filled with -inf.
//   * Two TMEM accumulators (2 x 256 columns) let the MMA of one group run
//     while the epilogue warps drain the previous one (each warp: one TMEM
//     lane quarter x one 64-column slice, read 32 columns at a time): relu,
//     x q_scale, sum over the token's heads in head order, x k_scale,
//     causal -inf, coalesced f32 stores.  Sixteen epilogue warps at 32
//     columns a load hide the TMEM load and FMA latencies that eight warps
//     at 64 columns (168 registers a thread) did not (1.35 -> 1.18 ms);
//     splitting a token's sum into independent chains, or pairing heads in
//     f32x2 FMAs, measured no better at sixteen warps.  The
//     item's page ids are staged in shared memory and each lane's k_scale
//     is loaded two tiles ahead, so no L2 round trip sits in a tile's
//     epilogue (measured: with the lookup inline, the epilogue waited on it
//     and a tile took ~4x its MMA time).
//   * Warp roles: warp 0 TMA producer, warp 1 MMA issuer (and TMEM owner),
//     warps 2.. epilogue.
#include <algorithm>

#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {
namespace idx {

constexpr int kDepth = 128;
constexpr int kBM = 128;      // keys per tile (MMA M)
constexpr int kBN = 256;      // (token, head) columns per tile (MMA N)
constexpr int kStages = 4;
constexpr int kGroups = 4;    // token groups (MMA tiles of N = 256) sharing each K tile
// Epilogue warps (a multiple of 4: one per TMEM lane quarter and column
// slice).
constexpr int kEpiThreads = 32 * 16;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kSlices = kEpiThreads / 128;   // column slices; 4 TMEM lane quarters each
constexpr int kSliceCols = kBN / kSlices;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxItemPages = 1024;  // the host sizes key chunks to stay within this

struct Params {
  const float* q_scale;
  const float* k_scale;
  int64_t phys_rows;
  const int32_t* cu_q;
  const int32_t* kv_len;
  const int32_t* page_table;
  int B, max_pages, page_size, T;
  int page_shift;  // log2(page_size)
  float* scores;
  int64_t score_stride;
  int chunk_tiles;  // key tiles per work item
  int box_rows;     // rows per K TMA box = min(page_size, 128)
  unsigned* err;
};

struct __align__(1024) Smem {
  uint8_t q[kGroups][kBN * kDepth];   // SW128 K-major: 256 rows x 128 B per token group
  uint8_t k[kStages][kBM * kDepth];   // SW128 K-major: 128 rows x 128 B each
  float qs[kGroups * kBN];
  int pages[kMaxItemPages];           // page ids of the item's key chunk
  unsigned long long bar_q, bar_kfull[kStages], bar_kempty[kStages], bar_afull[2], bar_aempty[2], bar_drain;
  uint32_t tmem_base;
  int item_b, item_tt, item_kc;
  // TMA loads issued by the producer and landings seen by the MMA issuer, so
  // that a CTA whose wait gave up still waits (bounded) for the copies it has
  // in flight before it exits
  int k_issued, k_landed, q_landed;
};

template <int HIDX>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const Params p) {
  constexpr int TOK = kBN / HIDX;      // tokens per group (one MMA tile)
  constexpr int TOKI = kGroups * TOK;  // tokens per item
  constexpr int SLICE_TOK = kSliceCols / HIDX;  // tokens per epilogue column slice
  constexpr uint32_t IDESC = idesc_e4m3_f32(kBM, kBN, 0, 0);

  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int CW = p.chunk_tiles * kBM;

  // ---- resolve this CTA's work item (warp 0 scans the sequences)
  if (warp == 0) {
    int base = 0, found_b = -1, found_tt = 0, found_kc = 0;
    const int target = blockIdx.x;
    for (int b0 = 0; b0 < p.B && found_b < 0; b0 += 32) {
      const int b = b0 + lane;
      int n = 0, ntt = 0, nkc = 0;
      if (b < p.B) {
        const int ql = p.cu_q[b + 1] - p.cu_q[b];
        const int kl = p.kv_len[b];
        ntt = (ql + TOKI - 1) / TOKI;
        nkc = (kl + CW - 1) / CW;
        n = (ql > 0 && kl >= ql && kl <= p.score_stride) ? ntt * nkc : 0;
        if (ql > 0 && (kl < ql || kl > p.score_stride)) atomicOr(p.err, kErrShape);
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int excl = base + incl - n;
      const bool mine = n > 0 && target >= excl && target < excl + n;
      const unsigned ball = __ballot_sync(0xffffffffu, mine);
      if (ball) {
        const int src = __ffs(ball) - 1;
        if (lane == src) {
          const int r = target - excl;
          found_b = b;
          found_tt = r / nkc;
          found_kc = r % nkc;
        }
        found_b = __shfl_sync(0xffffffffu, found_b, src);
        found_tt = __shfl_sync(0xffffffffu, found_tt, src);
        found_kc = __shfl_sync(0xffffffffu, found_kc, src);
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      s.item_b = found_b;
      s.item_tt = found_tt;
      s.item_kc = found_kc;
    }
  }
  __syncthreads();
  if (s.item_b < 0) return;

  const int b = s.item_b, tt = s.item_tt, kc = s.item_kc;
  const int cu0 = p.cu_q[b];
  const int q_len = p.cu_q[b + 1] - cu0;
  const int kvl = p.kv_len[b];
  const int t0 = cu0 + tt * TOKI;
  const int ntok = min(TOKI, q_len - tt * TOKI);
  const int pos0 = kvl - q_len + tt * TOKI;
  const int ngroups = (ntok + TOK - 1) / TOK;  // groups holding tokens (MMA tiles per K tile)
  const int key_lo = kc * CW;
  const int key_hi = min(key_lo + CW, kvl);
  const int64_t cover_hi = (key_hi == kvl) ? p.score_stride : key_hi;  // last chunk also fills past kv_len
  const int max_pos = pos0 + ntok - 1;
  const int kt_begin = key_lo / kBM;
  const int kt_end = min((key_hi + kBM - 1) / kBM, max_pos / kBM + 1);
  const int n_tiles = max(0, kt_end - kt_begin);

  // ---- setup: barriers, TMEM, q_scale tile
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&s.bar_q), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&s.bar_kfull[i]), 1);
      mbar_init(smem_u32(&s.bar_kempty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.bar_afull[i]), 1);
      mbar_init(smem_u32(&s.bar_aempty[i]), kEpiThreads);
    }
    mbar_init(smem_u32(&s.bar_drain), 1);
    fence_mbar_init();
    s.k_issued = 0;
    s.k_landed = 0;
    s.q_landed = 0;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  // pages of the keys [key_lo, key_lo + CW) (-1 past the sequence's table)
  const int page_lo = key_lo >> p.page_shift;
  const int npg = min(kMaxItemPages, ((key_lo + CW - 1) >> p.page_shift) - page_lo + 1);
  if (warp >= 2) {
    const int c = threadIdx.x - 64;  // column (token-in-item, head)
    for (int cc = c; cc < kGroups * kBN; cc += kEpiThreads) {
      const int tok = cc / HIDX, h = cc % HIDX;
      s.qs[cc] = (tok < ntok) ? p.q_scale[static_cast<int64_t>(t0 + tok) * HIDX + h] : 0.f;
    }
    for (int i = c; i < npg; i += kEpiThreads) {
      const int pg = page_lo + i;
      s.pages[i] = pg < p.max_pages ? p.page_table[static_cast<int64_t>(b) * p.max_pages + pg] : -1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      mbar_arrive_expect_tx(smem_u32(&s.bar_q), ngroups * kBN * kDepth);
      for (int g = 0; g < ngroups; ++g)
        tma_load_2d(smem_u32(s.q[g]), &tm_q, 0, (t0 + g * TOK) * HIDX, smem_u32(&s.bar_q));
      const int nbox = kBM / p.box_rows;
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % kStages;
        if (!mbar_wait(smem_u32(&s.bar_kempty[st]), ((i / kStages) & 1) ^ 1, p.err)) break;
        ++issued;
        const int kt = kt_begin + i;
        int nload = 0;
        int rows[kBM / 8];
        for (int bx = 0; bx < nbox; ++bx) {
          const int key0 = kt * kBM + bx * p.box_rows;
          rows[bx] = -1;
          if (key0 >= kvl) continue;
          // the item's page ids are staged in shared memory (no L2 round trip per box)
          const int pi = (key0 >> p.page_shift) - page_lo;
          const int pid = pi < npg ? s.pages[pi] : -1;
          const int64_t row = static_cast<int64_t>(pid) * p.page_size + key0 % p.page_size;
          if (pid < 0 || row + p.box_rows > p.phys_rows) {
            atomicOr(p.err, kErrPage);
            continue;
          }
          rows[bx] = static_cast<int>(row);
          ++nload;
        }
        // A tile whose boxes were all rejected still arrives (with no bytes).
        mbar_arrive_expect_tx(smem_u32(&s.bar_kfull[st]), nload * p.box_rows * kDepth);
        for (int bx = 0; bx < nbox; ++bx)
          if (rows[bx] >= 0)
            tma_load_2d(smem_u32(s.k[st]) + bx * p.box_rows * kDepth, &tm_k, 0, rows[bx],
                        smem_u32(&s.bar_kfull[st]));
      }
      s.k_issued = issued;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_tiles > 0) {
      bool ok = mbar_wait(smem_u32(&s.bar_q), 0, p.err);
      s.q_landed = ok ? 1 : 0;
      int landed = 0;
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int st = i % kStages;
        if (!mbar_wait(smem_u32(&s.bar_kfull[st]), (i / kStages) & 1, p.err)) break;
        landed = i + 1;
        const uint32_t k_base = smem_u32(s.k[st]);
        // MMA tile m = (K tile i, group g) into accumulator m & 1
        for (int g = 0; ok && g < ngroups; ++g) {
          const int m = i * ngroups + g, a = m & 1;
          if (!mbar_wait(smem_u32(&s.bar_aempty[a]), ((m >> 1) & 1) ^ 1, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t q_base = smem_u32(s.q[g]);
#pragma unroll
          for (int kk = 0; kk < kDepth / 32; ++kk) {
            const uint64_t ad = make_sdesc(k_base + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = make_sdesc(q_base + kk * 32, 16, 1024, kSwizzle128B);
            mma_f8f6f4_ss(tmem + a * kBN, ad, bd, IDESC, kk > 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&s.bar_afull[a]));
        }
        if (!ok) break;
        mma_commit(smem_u32(&s.bar_kempty[st]));
      }
      s.k_landed = landed;
      // Make sure no MMA is still writing TMEM when the CTA tears down.
      mma_commit(smem_u32(&s.bar_drain));
      mbar_wait(smem_u32(&s.bar_drain), 0, p.err);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;      // TMEM lanes this warp may access
    const int slice = ew >> 2;         // columns [slice*kSliceCols, +kSliceCols)
    const int row = quarter * 32 + lane;
    const float* qs_slice = s.qs + slice * kSliceCols;
    // k_scale of this lane's key (physical row) in tile i, from the staged page ids
    auto load_ks = [&](int i) -> float {
      const int key = (kt_begin + i) * kBM + row;
      if (i >= n_tiles || key >= kvl) return 0.f;
      const int pi = (key >> p.page_shift) - page_lo;
      const int pid = pi < npg ? s.pages[pi] : -1;
      const int64_t prow = (static_cast<int64_t>(pid) << p.page_shift) + (key & (p.page_size - 1));
      return (pid >= 0 && prow < p.phys_rows) ? __ldg(p.k_scale + prow) : 0.f;
    };
    float ks_next = load_ks(0), ks_next2 = load_ks(1);
    bool eok = true;
    for (int i = 0; eok && i < n_tiles; ++i) {
      const int kt = kt_begin + i;
      const int key = kt * kBM + row;
      const float ks = ks_next;
      ks_next = ks_next2;
      ks_next2 = load_ks(i + 2);
      for (int g = 0; g < ngroups; ++g) {
        const int m = i * ngroups + g, a = m & 1;
        const float* qs = qs_slice + g * kBN;
        // warp-uniform: the tcgen05.ld below is warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&s.bar_afull[a]), (m >> 1) & 1, p.err))) {
          eok = false;
          break;
        }
        tc_fence_after();
        float acc[SLICE_TOK];
#pragma unroll
        for (int j = 0; j < SLICE_TOK; ++j) acc[j] = 0.f;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + a * kBN + slice * kSliceCols;
#pragma unroll
        for (int cb = 0; cb < kSliceCols; cb += 32) {
          uint32_t v[32];
          tmem_ld32(taddr + cb, v);
          tmem_wait_ld_regs(v);
          if (cb + 32 == kSliceCols) {  // the accumulator is in registers: the MMA may reuse it
            tc_fence_before();
            mbar_arrive(smem_u32(&s.bar_aempty[a]));
          }
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 q4 = *reinterpret_cast<const float4*>(qs + cb + j);
            const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int tj = (cb + j + u) / HIDX;
              acc[tj] = fmaf(fmaxf(__uint_as_float(v[j + u]), 0.f), qq[u], acc[tj]);
            }
          }
        }
        if (key >= key_lo && key < cover_hi) {
#pragma unroll
          for (int j = 0; j < SLICE_TOK; ++j) {
            const int tok = g * TOK + slice * SLICE_TOK + j;
            if (tok < ntok) {
              const float v = (key <= pos0 + tok) ? ks * acc[j] : -INFINITY;
              p.scores[static_cast<int64_t>(t0 + tok) * p.score_stride + key] = v;
            }
          }
        }
      }
    }
    // -inf for the covered keys no computed tile reached.
    const int64_t fill_lo = max(static_cast<int64_t>(key_lo), static_cast<int64_t>(kt_end) * kBM);
    const int et = threadIdx.x - 64;
    for (int tok = 0; tok < ntok; ++tok) {
      float* dst = p.scores + static_cast<int64_t>(t0 + tok) * p.score_stride;
      for (int64_t key = fill_lo + et; key < cover_hi; key += kEpiThreads) dst[key] = -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // After a wait gave up: TMA loads still in flight land before the CTA
  // exits (bounded waits; in the normal case every issued load has landed).
  if (threadIdx.x == 0 && n_tiles > 0) {
    if (!s.q_landed) mbar_wait(smem_u32(&s.bar_q), 0, p.err);
    for (int i = s.k_landed; i < s.k_issued; ++i)
      mbar_wait(smem_u32(&s.bar_kfull[i % kStages]), (i / kStages) & 1, p.err);
  }
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

static_assert(sizeof(Smem) + 1024 <= 232448, "indexer shared memory exceeds a CTA's 227 KB");

template <int HIDX>
static cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const Params& p, int grid,
                            cudaStream_t stream) {
  const size_t smem = sizeof(Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(indexer_kernel<HIDX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  indexer_kernel<HIDX><<<grid, kThreads, smem, stream>>>(tq, tk, p);
  return cudaGetLastError();
}

}  // namespace idx

// Host launcher: builds the two tensor maps, sizes the work items and launches.
smla_status_t launch_indexer(const uint8_t* q, const float* q_scale, const uint8_t* k_pool, const float* k_scale,
                             int64_t phys_rows, const smla_seqs_t& seqs, int h_idx, float* scores,
                             int64_t score_stride, unsigned* err, cudaStream_t stream) {
  using namespace idx;
  if (seqs.T == 0 || seqs.B == 0) return SMLA_OK;
  const int tok = kGroups * kBN / h_idx;
  const int box_rows = std::min(seqs.page_size, kBM);
  CUtensorMap tq, tk;
  if (!encode_tma_2d_u8(&tq, q, kDepth, static_cast<uint64_t>(seqs.T) * h_idx, kDepth, kBN))
    return fail(SMLA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the indexer Q tensor map");
  if (!encode_tma_2d_u8(&tk, k_pool, kDepth, static_cast<uint64_t>(phys_rows), kDepth, box_rows))
    return fail(SMLA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the indexer K tensor map");
  // Key chunk per work item: enough items to give every SM about two.
  const int64_t key_tiles = (score_stride + kBM - 1) / kBM;
  const int64_t est_tt = (seqs.T + tok - 1) / tok;
  const int64_t want = 2 * static_cast<int64_t>(device_sm_count());
  int64_t chunk = (est_tt * key_tiles + want - 1) / want;
  chunk = std::max<int64_t>(1, std::min<int64_t>(chunk, key_tiles));
  // the item's page ids are staged in shared memory (kMaxItemPages)
  chunk = std::min<int64_t>(chunk, static_cast<int64_t>(kMaxItemPages - 2) * seqs.page_size / kBM);
  chunk = std::max<int64_t>(1, chunk);
  const int64_t nchunk = (key_tiles + chunk - 1) / chunk;
  const int64_t grid = (est_tt + seqs.B) * nchunk;  // upper bound; CTAs past the last item exit at once
  if (grid > 0x7fffffff) return fail(SMLA_ERR_UNSUPPORTED, "indexer grid too large");
  Params p{q_scale, k_scale, phys_rows, seqs.cu_q, seqs.kv_len, seqs.page_table, seqs.B, seqs.max_pages,
           seqs.page_size, seqs.T, __builtin_ctz(static_cast<unsigned>(seqs.page_size)), scores, score_stride,
           static_cast<int>(chunk), box_rows, err};
  cudaError_t e;
  switch (h_idx) {
    case 4: e = launch_t<4>(tq, tk, p, static_cast<int>(grid), stream); break;
    case 8: e = launch_t<8>(tq, tk, p, static_cast<int>(grid), stream); break;
    case 16: e = launch_t<16>(tq, tk, p, static_cast<int>(grid), stream); break;
    case 32: e = launch_t<32>(tq, tk, p, static_cast<int>(grid), stream); break;
    case 64: e = launch_t<64>(tq, tk, p, static_cast<int>(grid), stream); break;
    default: return fail(SMLA_ERR_UNSUPPORTED, "H_idx must be 4, 8, 16, 32 or 64");
  }
  if (e != cudaSuccess) return fail_cuda(e, "indexer launch");
  return SMLA_OK;
}

}  // namespace smla
