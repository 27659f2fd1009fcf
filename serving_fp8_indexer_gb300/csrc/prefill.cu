// Stage 3: sparse MLA prefill attention on tcgen05 FP8 tensor cores.
//
// What it computes ("mla_sm100_prefill_sparse_fp8" function page; K and V
// share the latent rows per "mla_prefill_sparse_qkv_fp8"): for token t,
// head h and the n = topk_lengths[t] gathered latent rows K_j,
//   out[t,h,:] = sum_j softmax_j(softmax_scale * q[t,h] . K_j) * K_j[0:512].
//
// GB300 design.  A work item is (token, group of 64 heads); persistent CTAs
// (one per SM) take the items in turn, and an item's keys are processed in
// blocks of 128 gathered rows.  The block's keys are the
// MMA M dimension and the heads the N dimension:
//   S^T[128 keys x 64 heads] = K_blk . Q^T           (TMEM, 64 columns)
//   O^T[512 vcols x 64 heads] += V_blk^T . P^T       (TMEM, 4 x 64 columns)
// so the 128-head, 512-wide output of a token never has to sit in TMEM at
// once (a [heads x 512] f32 accumulator alone would fill all 512 columns)
// and every MMA is M = 128 at full rate.  V^T is the same gathered buffer
// read MN-major (V = the first 512 columns of K).
//
// All products run on the FP8 pipe (kind::f8f6f4, f32 accumulation):
//   * e4m3 q is used as is; bf16 q is split once per item into two e4m3
//     terms q*2^e = hi + lo (per-head power-of-two 2^e keeps lo in range),
//     both multiplied into the same S accumulator (error ~2^-8 relative);
//   * P is quantised to one e4m3 term (native FP8-P path) or, for the bf16
//     path, to hi + lo like q;
//   * blockwise-scaled rows (32-wide scales) are gathered raw with their
//     block scales and split in shared memory into e4m3 hi + lo of
//     x * s_blk / s_row, after which every row carries one scale s_row.
// A per-row scale s_j (tensorwise, or s_row) enters exactly: the logit is
// z = acc * s_j * c_h, the PV operand is exp2(z + log2 s_j - m) and the
// normaliser sums exp2(z - m), so out = sum_j p_j s_j Vraw_j / sum_j p_j.
//
// Softmax: keys are TMEM lanes, so a head's maximum is a cross-lane
// reduction (warp redux on order-preserving ints, then shared-memory atomic
// max across the 4 lane quarters).  The reference m sits 2^4 below the
// largest logit seen when it was set (so that the weights near the maximum
// keep e4m3's precision) and is only raised when a block exceeds it by more
// than 2^8 (lazy rescale), keeping P <= 256 inside the e4m3 range; raising
// it rescales O^T and the row sums.
//
// Pipeline: NST gather slots (2 when they fit in shared memory).  The
// producers fetch the next block's row indices and scales while the current
// block's rows are in flight, so a slot refill starts with its copies.  PV
// runs key-quarter by key-quarter (32 rows of the slot per step, the four
// O^T tiles interleaved) and commits each quarter back to the gather, so the
// rows of block j+NST start arriving while PV of block j is still running.
// QK and PV have an issuing warp each: QK of block j+1 runs under the
// softmax of block j (S is loaded into registers first and then released),
// and PV of block j never queues behind the issue of QK j+1.  Each QK and PV
// is issued as one straight run of MMAs (measured: splitting a block's QK
// into five separately issued groups doubled its tensor-pipe time), and
// consecutive MMAs always target different accumulators (QK alternates two
// S^T accumulators, PV rotates over the four O^T tiles): an MMA waits for
// the previous one on the same accumulator.
//
// Warp roles (24 warps): warps 0-7 softmax / epilogue (lane quarter w%4,
// head half w/4; thread = one key x 32 heads), warp 8 QK issuer and TMEM
// owner, warp 9 PV issuer, warps 10-23 gather producers (cp.async 16 B into
// the SW64 layout; for blockwise rows also the block scales).
#include <algorithm>
#include <cstddef>

#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {
namespace pf {

constexpr int kD = 576;           // qk depth
constexpr int kDV = 512;          // v depth
constexpr int kNH = 64;           // heads per CTA (MMA N)
constexpr int kBK = 128;          // keys per block (MMA M of QK)
constexpr int kChunks = kD / 64;  // 64-byte K chunks per row (SW64)
constexpr int kQBytes = kChunks * kNH * 64;   // 36864
constexpr int kKVBytes = kChunks * kBK * 64;  // 73728
constexpr int kChunkBytes = kBK * 64;         // 8192: one 64-column chunk of a block
constexpr int kRope = 8;                      // chunk index of columns 512..575
constexpr int kRowQ = 4;                      // key quarters a slot is released in
constexpr int kBlkScales = kD / 32;           // 32-column block scales per row (blockwise rows)
constexpr int kSoftWarps = 8;
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kMmaWarp = 8;   // QK issuer, TMEM owner
constexpr int kPvWarp = 9;    // PV issuer
constexpr int kProdWarp0 = 10;
// Producer warps: the gather is bound by the requests kept in flight, so
// more warps gather faster (measured on this access pattern: 7 warps ~4.9,
// 16 warps ~7.4 TB/s from L2).  24 warps in all launch with 80 registers a
// thread; the softmax warpgroups then raise theirs to kSoftRegs and the
// others drop to kLowRegs (setmaxnreg), within the launch allocation.
__host__ __device__ constexpr int prod_warps(int) { return 14; }
__host__ __device__ constexpr int threads_for(int kvp) { return kSoftThreads + 64 + 32 * prod_warps(kvp); }
constexpr int kLaunchRegs = 80;
constexpr int kSoftRegs = 160;
constexpr int kLowRegs = 40;
static_assert(kSoftThreads * kSoftRegs + (threads_for(1) - kSoftThreads) * kLowRegs <= threads_for(1) * kLaunchRegs,
              "register split exceeds the launch allocation");
static_assert(kSoftWarps % 4 == 0 && kMmaWarp % 4 == 0, "roles must split on warpgroup boundaries");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 256;  // S^T accumulators from 256; O^T tiles at [0, 256)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTau = 8.0f;      // lazy-rescale threshold (log2 units): P stays <= 2^8
// The reference a head's weights are taken against sits this far (log2
// units) below the largest logit seen when it was set, so that the block
// maximum's weight is 2^4 rather than 1.  The two-term (hi + lo) e4m3 P then
// keeps about 2^-8 relative precision for weights down to 2^-6 of the
// maximum (with the maximum at 1, lo fell below e4m3's normal range, 2^-6,
// for weights under 2^-2 of it, and those weights carried an absolute error
// of about 2^-10).  A later block rescales once it exceeds the reference by
// 2^8, i.e. the previous maximum by 2^4.
constexpr float kPOffset = 4.0f;
constexpr int kOrdMin = static_cast<int>(0x80000000u);

enum Scale { kUnit = 0, kRow = 1, kBlock = 2 };

// Where a token's keys come from.
enum Keys {
  kIndexed = 0,  // sparse: indices[t, 0 .. topk_lengths[t]) (physical rows)
  kCausal = 1,   // dense: every logical key 0..pos(t) of t's sequence, through the page table
};

struct Params {
  const void* q;
  const uint8_t* latent;
  int64_t phys_rows;
  const float* scales;
  int nscale;  // scales per row
  const uint32_t* indices;
  int indices_stride;
  const uint32_t* lens;
  int T, H;
  float softmax_scale;
  uint16_t* out;
  unsigned* err;
  int q_box3d;  // q tensor map is 3-D: one load brings all column boxes of an item
  int keys;     // Keys
  // kCausal: the ragged batch (smla_seqs_t)
  const int32_t* cu_q;
  const int32_t* kv_len;
  const int32_t* page_table;
  int B, max_pages, page_shift;
  // attention sink: one logit per head (natural-log units, like the scaled
  // logits) that joins every softmax denominator and carries no value; null
  // for none
  const float* sink;
  // split-K: a token's key blocks are divided among nsplit work items, each
  // writing its normalised partial output (f32) and log2-sum-exp per head
  // to part_o [T, nsplit, H, 512] / part_lse [T, nsplit, H]; nsplit == 1
  // writes the bf16 output directly
  int nsplit;
  float* part_o;
  float* part_lse;
};

// EB: bytes per latent element in the cache: 1 (e4m3) or 2 (bf16 cache;
// then q is bf16, one term, and QK / PV run as kind::f16 bf16 MMAs).
template <int QP, int KVP, int PP, int NST, int EB = 1>
struct Smem {
  // Q as the QK B operand, [chunk][QP x 64 rows][64 B]: for bf16 q the hi
  // rows 0..63 and lo rows 64..127 of a chunk are one 128-row operand; with
  // a bf16 cache, 18 chunks of 64 rows
  uint8_t q[QP * EB * kQBytes];
  uint8_t kv[NST][KVP][EB * kKVBytes];
  uint8_t plo[PP == 2 ? kChunkBytes : 16];  // P lo term (bf16 path)
  uint32_t idx[kBK];
  float srow[NST][kBK];  // per-row scale (1 for unit)
  // blockwise rows: each row's 18 block scales, then 1 / s_row per row
  float bsc[KVP == 2 ? kBK * kBlkScales + kBK : 4];
  alignas(16) float cs[kNH];    // softmax_scale * log2(e) / 2^e_h (read as float4)
  alignas(16) float negm[kNH];  // minus the reference maximum per head, log2 units (read as float4)
  float delta[kNH];      // reference raise of the current block
  float fac[kNH];        // rescale factor of the current block; 1 / row sum at the end
  int mx[kNH];           // block maximum per head (order-preserving ints)
  unsigned long long bar_qraw, bar_q, bar_kv_full[NST], bar_kv_empty[NST][kRowQ];
  unsigned long long bar_s_full, bar_s_free, bar_p_full[kRowQ], bar_pv_done;  // P published per key quarter
  unsigned long long bar_kv_split;         // blockwise rows: the block's hi / lo terms are written
  unsigned long long bar_kv_q[kRowQ];      // blockwise rows: key quarter q has landed (raw) with s_row
  uint32_t tmem_base;
  int q_issued;  // TMA q loads requested by the QK warp (read at exit)
};

__device__ __forceinline__ int ord_int(float f) {
  const int b = __float_as_int(f);
  return b >= 0 ? b : b ^ 0x7fffffff;
}
__device__ __forceinline__ float ord_float(int o) { return __int_as_float(o >= 0 ? o : o ^ 0x7fffffff); }

__device__ __forceinline__ uint32_t sw64(int row, int c4) { return static_cast<uint32_t>((c4 ^ ((row >> 1) & 3)) << 4); }

// e4m3 hi + lo split of 16 floats (|x| <= 448) into two 16-byte chunks.
// The residual is formed in f16x2: x -> f16 (2^-11), hi = e4m3(x_f16),
// lo = e4m3(x_f16 - hi) (exact subtraction); |x - hi - lo| <~ 2^-9 |x|.
__device__ __forceinline__ void split16(const float (&x)[16], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t a = f32x2_to_f16x2(x[4 * i + 0], x[4 * i + 1]);
    const uint32_t b = f32x2_to_f16x2(x[4 * i + 2], x[4 * i + 3]);
    const uint16_t ha = f16x2_to_e4m3x2(a), hb = f16x2_to_e4m3x2(b);
    const uint16_t la = f16x2_to_e4m3x2(hsub2(a, e4m3x2_to_f16x2(ha)));
    const uint16_t lb = f16x2_to_e4m3x2(hsub2(b, e4m3x2_to_f16x2(hb)));
    h[i] = static_cast<uint32_t>(ha) | (static_cast<uint32_t>(hb) << 16);
    l[i] = static_cast<uint32_t>(la) | (static_cast<uint32_t>(lb) << 16);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}
// The same split for 8 floats into two 8-byte halves of a chunk.
__device__ __forceinline__ void split8(const float (&x)[8], uint2& hi, uint2& lo) {
  uint32_t h[2], l[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t a = f32x2_to_f16x2(x[4 * i + 0], x[4 * i + 1]);
    const uint32_t b = f32x2_to_f16x2(x[4 * i + 2], x[4 * i + 3]);
    const uint16_t ha = f16x2_to_e4m3x2(a), hb = f16x2_to_e4m3x2(b);
    const uint16_t la = f16x2_to_e4m3x2(hsub2(a, e4m3x2_to_f16x2(ha)));
    const uint16_t lb = f16x2_to_e4m3x2(hsub2(b, e4m3x2_to_f16x2(hb)));
    h[i] = static_cast<uint32_t>(ha) | (static_cast<uint32_t>(hb) << 16);
    l[i] = static_cast<uint32_t>(la) | (static_cast<uint32_t>(lb) << 16);
  }
  hi = make_uint2(h[0], h[1]);
  lo = make_uint2(l[0], l[1]);
}
// Splits f16x2 a into e4m3 hi + lo: hi = a rounded to e4m3 by the conversion
// (nearest even, e4m3's subnormals included) and read back, lo = a - hi
// (exact in f16).  Three conversions a pair and no integer operations: the
// blockwise split is bound by the ALU pipe (measured: rounding hi with
// integer operations on the f16 bits, two conversions a pair, 4.93 ms
// against 4.51 ms for this form on the blockwise workload).
__device__ __forceinline__ void split_f16x2_cvt(uint32_t a, uint16_t& hi, uint16_t& lo) {
  hi = f16x2_to_e4m3x2(a);
  lo = f16x2_to_e4m3x2(hsub2(a, e4m3x2_to_f16x2(hi)));
}
__device__ __forceinline__ uint4 quant16(const float (&x)[16]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = static_cast<uint32_t>(f32x2_to_e4m3x2(x[4 * i], x[4 * i + 1])) |
           (static_cast<uint32_t>(f32x2_to_e4m3x2(x[4 * i + 2], x[4 * i + 3])) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Blockwise rows: the softmax warps split a landed key quarter (rows 32q ..
// 32q + 31) in place.  A piece is 16 bytes (16 e4m3 values) of one row; a
// warp covers 8 rows x 4 pieces of one 64-byte chunk (512 contiguous bytes:
// no bank conflicts).  x = e4m3 * (s_blk / s_row) in f16 (the product needs 8
// significant bits, f16 keeps 11), hi = x rounded to e4m3's 3 mantissa bits
// (nearest even), lo = x - hi (exact); hi overwrites the raw piece, lo goes
// to the second buffer (split_f16x2_cvt).  bsc holds 18 block scales per
// row, then 1 / s_row per row.  Piece i of the quarter is in row
// 32q + ((i >> 2) & 31), 16-byte column c4 = i & 3 of chunk i >> 7; the
// thread stride 256 keeps a thread's row and c4 and steps its chunk by 2.
__device__ __forceinline__ void split_quarter(uint8_t* hi_buf, uint8_t* lo_buf, const float* bsc, int q) {
  // All of a thread's pieces are read first, then converted and written, so
  // that their conversion chains interleave (a piece is only ever read and
  // rewritten by its own thread).
  constexpr int kIt = (32 * 36 + kSoftThreads - 1) / kSoftThreads;
  static_assert(kSoftThreads == 256, "a thread keeps its row and column; its chunk steps by 2");
  const int row = 32 * q + ((threadIdx.x >> 2) & 31), c4 = threadIdx.x & 3, kc0 = threadIdx.x >> 7;
  const uint32_t off0 = kc0 * kChunkBytes + row * 64 + sw64(row, c4);
  const float* bs = bsc + row * kBlkScales + 2 * kc0 + (c4 >> 1);  // chunk kc0 + 2 it: block scale bs[4 it]
  const float isr = bsc[kBK * kBlkScales + row];
  uint4 raw[kIt];
  float ratio[kIt];
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    if (threadIdx.x + it * kSoftThreads < 32 * 36) {
      raw[it] = *reinterpret_cast<const uint4*>(hi_buf + off0 + it * (2 * kChunkBytes));
      ratio[it] = bs[4 * it] * isr;
    }
  }
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    if (threadIdx.x + it * kSoftThreads < 32 * 36) {
      const uint32_t off = off0 + it * (2 * kChunkBytes);
      const uint32_t r2 = f32x2_to_f16x2(ratio[it], ratio[it]);
      const uint32_t wv[4] = {raw[it].x, raw[it].y, raw[it].z, raw[it].w};
      uint32_t h[4], l[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint16_t ha, hb, la, lb;
        split_f16x2_cvt(hmul2(e4m3x2_to_f16x2(static_cast<uint16_t>(wv[k] & 0xffffu)), r2), ha, la);
        split_f16x2_cvt(hmul2(e4m3x2_to_f16x2(static_cast<uint16_t>(wv[k] >> 16)), r2), hb, lb);
        h[k] = static_cast<uint32_t>(ha) | (static_cast<uint32_t>(hb) << 16);
        l[k] = static_cast<uint32_t>(la) | (static_cast<uint32_t>(lb) << 16);
      }
      *reinterpret_cast<uint4*>(hi_buf + off) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(lo_buf + off) = make_uint4(l[0], l[1], l[2], l[3]);
    }
  }
}

// Issues QK of one block: S^T[128 keys x QP*64] over the 576 columns (for
// bf16 q the hi and lo products side by side, one N = 128 MMA per K step, so
// each key tile is read once for both), the MMAs rotating over NACC
// accumulators (MMA i of the block goes to accumulator i % NACC; the first
// NACC overwrite).  Every operand offset is a compile-time constant.
template <int QP, int KVP, int NACC, int EB>
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint64_t a0, uint64_t b0, uint32_t idesc) {
  constexpr int kQN = QP * kNH;
#pragma unroll
  for (int kc = 0; kc < kChunks * EB; ++kc)
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)  // two 32-byte K steps per 64-byte chunk
#pragma unroll
      for (int kp = 0; kp < KVP; ++kp) {
        const int i = (kc * 2 + kk) * KVP + kp;
        // descriptor address fields are in 16-byte units: add offsets >> 4
        const uint64_t ad = a0 + static_cast<uint64_t>((kp * EB * kKVBytes + kc * kChunkBytes + kk * 32) >> 4);
        const uint64_t bd = b0 + static_cast<uint64_t>((kc * kQN * 64 + kk * 32) >> 4);
        if (EB == 2)
          mma_f16_ss(s_tmem + (i % NACC) * kQN, ad, bd, idesc, i < NACC ? 0u : 1u);
        else
          mma_f8f6f4_ss(s_tmem + (i % NACC) * kQN, ad, bd, idesc, i < NACC ? 0u : 1u);
      }
}

// Split-K: the item's normalised partial output O^T / l as f32, thread = one
// value column of 32 heads (a warp store covers 32 consecutive columns of one
// head); heads from nh on are outside the item.  Out of line: the split path
// is rare, and inlined it cost the block loop registers (measured 2 % on the
// end-to-end chunk).
__device__ __noinline__ void store_partial(float* po, uint32_t taddr, const float* linv, int nh) {
#pragma unroll 1
  for (int tile = 0; tile < 4; ++tile) {
    uint32_t v[32];
    tmem_ld32(taddr + tile * kNH, v);
    tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < 32; ++h)
      if (h < nh) __stcs(po + static_cast<int64_t>(h) * kDV + tile * 128, __uint_as_float(v[h]) * linv[h]);
  }
}

// The row sum l = sum_j exp2(z_j - m) of one head (negm = -m, log2 units)
// in the two rarer modes: split-K writes the partial's log2-sum-exp m +
// log2 l to part_lse[prow] (the combine adds the sink); otherwise the sink
// term exp2(sink * log2e - m) joins l.  Out of line, like store_partial.
__device__ __noinline__ float split_or_sink(const Params& p, int64_t prow, int head, float l, float negm) {
  if (p.nsplit > 1) {
    p.part_lse[prow] = l > 0.f ? log2f(l) - negm : -INFINITY;
    return l;
  }
  return l + ex2_approx(fmaf(p.sink[head], kLog2e, negm));
}

// One work item: a token, one group of 64 heads and (split-K) one range of
// the token's key blocks.
struct Item {
  int t, h0, hv;
  int n;     // the token's keys (all splits)
  int j0;    // first key block of this item
  int nblk;  // key blocks of this item (0: nothing to attend to)
  int s;     // split index
  int b;     // sequence of the token (kCausal)
};
__device__ __forceinline__ int item_token(const Params& p, int w, int groups) { return w / (groups * p.nsplit); }

// Sequence of token t (kCausal): the last b with cu_q[b] <= t.
__device__ __forceinline__ int seq_of(const Params& p, int t) {
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu_q[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The token's key count: its selection length (kIndexed) or pos + 1
// (kCausal); `b` receives the sequence for kCausal.
template <int KEYS>
__device__ __forceinline__ int token_keys(const Params& p, int t, int& b) {
  if (KEYS == kCausal) {
    b = seq_of(p, t);
    const int q_len = p.cu_q[b + 1] - p.cu_q[b];
    const int n = p.kv_len[b] - q_len + (t - p.cu_q[b]) + 1;
    if (n < 0 || n > (p.max_pages << p.page_shift)) {
      if (threadIdx.x == 0) atomicOr(p.err, kErrShape);
      return 0;
    }
    return n;
  }
  b = 0;
  int n = static_cast<int>(p.lens[t]);
  if (n > p.indices_stride) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrShape);
    n = p.indices_stride;
  }
  return n;
}

// item w given its token's key count n (and sequence b)
__device__ __forceinline__ Item item_make(const Params& p, int w, int groups, int n, int b) {
  Item it;
  const int tg = w / p.nsplit;
  it.s = w - tg * p.nsplit;
  it.t = tg / groups;
  it.h0 = (tg % groups) * kNH;
  it.hv = min(kNH, p.H - it.h0);
  it.n = n;
  it.b = b;
  const int nb = (n + kBK - 1) / kBK;
  const int per = (nb + p.nsplit - 1) / p.nsplit;
  it.j0 = min(nb, it.s * per);
  it.nblk = min(nb, it.j0 + per) - it.j0;
  return it;
}
template <int KEYS>
__device__ __forceinline__ Item item_at(const Params& p, int w, int groups) {
  int b;
  const int n = token_keys<KEYS>(p, item_token(p, w, groups), b);
  return item_make(p, w, groups, n, b);
}

// Persistent CTAs: CTA c takes the work items c, c + gridDim.x, ... in turn,
// and every pipeline barrier keeps counting across items (a block's slot and
// phases come from its index g over all of this CTA's blocks), so the next
// item's first rows are gathered, and its q split, while the current item's
// last blocks and epilogue run.
template <int QP, int KVP, int PP, int NST, int SC, int KEYS, int EB>
__global__ void __launch_bounds__(threads_for(KVP), 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tq, const Params p) {
  using S = Smem<QP, KVP, PP, NST, EB>;
  static_assert(EB == 1 || (QP == 1 && KVP == 1 && PP == 1 && SC == kUnit),
                "a bf16 cache takes bf16 q as one term, single-term P and no scales");
  constexpr int kCh = kChunks * EB;       // 64-byte chunks per cache row
  constexpr int kSlotBytes = EB * kKVBytes;
  constexpr int kRopeCh = kRope * EB;     // chunk of column 512 (P goes there)
  static_assert(!(PP == 2 && KVP == 2), "P lo has a buffer only when rows are single-term");
  static_assert(KVP == 1 || NST == 1, "the blockwise quarter barriers complete once per block (one slot)");
  static_assert(offsetof(S, kv) % 1024 == 0 && offsetof(S, plo) % 1024 == 0,
                "swizzled operand tiles need 1024-byte alignment");
  static_assert(offsetof(S, cs) % 16 == 0 && offsetof(S, negm) % 16 == 0, "cs / negm are read as float4");
  // S^T accumulators: the block's QK MMAs alternate between two of them
  // (summed by the softmax), because an MMA waits for the previous one on
  // its accumulator but not for other MMAs (measured: two alternating
  // accumulators already run a block's QK as fast as three).
  constexpr int kSAcc = 2;
  constexpr int kQN = QP * kNH;  // QK MMA N
  static_assert(kSAcc == 2, "the softmax sums exactly two S accumulators");
  static_assert(kTmemS + kQN * kSAcc <= kTmemCols, "TMEM budget");
  constexpr int kThreads = threads_for(KVP);
  constexpr int kProdThreads = 32 * prod_warps(KVP);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The swizzled operand tiles need 1024-byte alignment; the launch asks
  // for exactly sizeof(S) bytes, so the dynamic window must start aligned.
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrShape);
    return;
  }
  S& s = *reinterpret_cast<S*>(smem_raw);
  const int groups = (p.H + kNH - 1) / kNH;
  const int items = p.T * groups * p.nsplit;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&s.bar_qraw), 1);
    mbar_init(smem_u32(&s.bar_q), kSoftThreads);
    for (int i = 0; i < NST; ++i) {
      // each producer thread arrives twice per block: once when it has issued
      // its copies (releasing its s.srow / s.idx writes) and once, through
      // cp.async.mbarrier.arrive.noinc, when those copies have landed
      mbar_init(smem_u32(&s.bar_kv_full[i]), 2 * kProdThreads);
      for (int q = 0; q < kRowQ; ++q) mbar_init(smem_u32(&s.bar_kv_empty[i][q]), 1);
    }
    mbar_init(smem_u32(&s.bar_s_full), 1);
    mbar_init(smem_u32(&s.bar_s_free), kSoftThreads);
    for (int q = 0; q < kRowQ; ++q) mbar_init(smem_u32(&s.bar_p_full[q]), kSoftThreads / kRowQ);
    mbar_init(smem_u32(&s.bar_pv_done), 1);
    mbar_init(smem_u32(&s.bar_kv_split), kSoftThreads);
    for (int q = 0; q < kRowQ; ++q) mbar_init(smem_u32(&s.bar_kv_q[q]), kProdThreads);
    fence_mbar_init();
    tma_prefetch_desc(&tq);
  }
  if (threadIdx.x < kNH) s.mx[threadIdx.x] = kOrdMin;
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&s.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  int q_waited = 0;  // TMA q loads waited by the softmax warps (bar_qraw phases)

  if (warp < kSoftWarps) {
    // =================================================================== softmax / epilogue
    setmaxnreg_inc<kSoftRegs>();
    const int r = threadIdx.x & 127;        // key lane = TMEM lane
    const int half = warp >> 2;             // heads [32*half, 32*half + 32)
    const int hb = half * 32;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // ---- q of an item into s.q (its QK B operand).  The QK warp requests
    // the item's 64 q rows with TMA (see there) in the SW64 layout, head =
    // row, 64-byte column box c at c * 4096.  e4m3 q lands in its final
    // layout.  For bf16 q, box pair (2kc, 2kc+1) covers exactly the bytes of
    // chunk kc's hi and lo rows, so the split into e4m3 hi + lo (per-head
    // power of two putting the largest |q| * 2^e in [128, 256)) runs in
    // place, each head's bytes read and rewritten by the same eight lanes.
    auto wait_q = [&]() -> bool {
      const bool r = named_bar_and(1, kSoftThreads, mbar_wait(smem_u32(&s.bar_qraw), q_waited & 1, p.err));
      ++q_waited;
      return r;
    };
    // waits for item I's q rows, splits bf16 q, sets s.cs and releases s.q to QK
    auto convert_q = [&](const Item& I) -> bool {
      if (!wait_q()) return false;
      if (QP == 2) {
        // 8 lanes per head (two rounds of 32 heads): lane r8 of a head holds
        // elements 8 * (r8 + 8k) .. +7 of the row (box 2k + r8 / 4, piece r8 % 4)
        const int r8 = threadIdx.x & 7;
        uint4 v[2][9];
#pragma unroll
        for (int rd = 0; rd < 2; ++rd) {
          const int hh = 32 * rd + (threadIdx.x >> 3);
#pragma unroll
          for (int k = 0; k < 9; ++k)
            v[rd][k] = hh < I.hv ? *reinterpret_cast<const uint4*>(&s.q[(2 * k + (r8 >> 2)) * (kNH * 64) + hh * 64 +
                                                                         sw64(hh, r8 & 3)])
                                 : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int rd = 0; rd < 2; ++rd) {
          const int hh = 32 * rd + (threadIdx.x >> 3);
          float amax = 0.f;
#pragma unroll
          for (int k = 0; k < 9; ++k) {
            const uint32_t wv[4] = {v[rd][k].x, v[rd][k].y, v[rd][k].z, v[rd][k].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              amax = fmaxf(amax, fabsf(__uint_as_float(wv[u] << 16)));
              amax = fmaxf(amax, fabsf(__uint_as_float(wv[u] & 0xffff0000u)));
            }
          }
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          __syncwarp();  // the head's eight lanes have read all of its bytes
          int e = 0;
          if (amax > 0.f) {
            int ex;
            frexpf(amax, &ex);  // amax = m * 2^ex, m in [0.5, 1)
            e = 8 - ex;
          }
          const float sigma = ldexpf(1.f, e);
#pragma unroll
          for (int k = 0; k < 9; ++k) {
            const uint32_t wv[4] = {v[rd][k].x, v[rd][k].y, v[rd][k].z, v[rd][k].w};
            float x[8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              x[2 * u] = __uint_as_float(wv[u] << 16) * sigma;
              x[2 * u + 1] = __uint_as_float(wv[u] & 0xffff0000u) * sigma;
            }
            uint2 hi, lo;
            split8(x, hi, lo);
            const int e0 = 8 * (r8 + 8 * k);  // first element of the piece
            const int kc = e0 >> 6, c4 = (e0 & 63) >> 4;
            const uint32_t off = kc * (kQN * 64) + hh * 64 + sw64(hh, c4) + (e0 & 8);
            *reinterpret_cast<uint2*>(&s.q[off]) = hi;
            *reinterpret_cast<uint2*>(&s.q[off + kNH * 64]) = lo;
          }
          if (r8 == 0) s.cs[hh] = p.softmax_scale * kLog2e / sigma;
        }
      } else {
        // e4m3 q is in place; rows past the item's heads (another token's) are zeroed
        if (I.hv < kNH)
          for (int i = threadIdx.x; i < kCh * kNH * 4; i += kSoftThreads) {
            const int row = (i >> 2) % kNH;
            if (row >= I.hv) *reinterpret_cast<uint4*>(&s.q[(i >> 2) * 64 + (i & 3) * 16]) = make_uint4(0, 0, 0, 0);
          }
        if (threadIdx.x < kNH) s.cs[threadIdx.x] = p.softmax_scale * kLog2e;
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&s.bar_q));
      return true;
    };
    int gb = 0;  // index of the item's first block among this CTA's blocks
    bool ok = true;
    bool q_in = false;  // s.q holds the current item's converted q
    Item I = item_at<KEYS>(p, blockIdx.x, groups);
    for (int w = blockIdx.x; ok && w < items; w += gridDim.x) {
      const int wn = w + static_cast<int>(gridDim.x);  // this CTA's next item
      const int n = I.n, nblk = I.nblk;
      const int n_item = n - I.j0 * kBK;  // the token's keys from this item's first block on
      uint16_t* out_t = p.out + (static_cast<int64_t>(I.t) * p.H + I.h0) * kDV;
      // split-K partials of this item: rows (t * nsplit + s) * H + h of
      // [T, nsplit, H, 512] and [T, nsplit, H]
      auto part_row = [&]() { return (static_cast<int64_t>(I.t) * p.nsplit + I.s) * p.H + I.h0; };
      if (nblk == 0) {
        // nothing to attend to: zeros (no softmax mass), or for a split an
        // empty partial (log-sum-exp -inf, which the combine skips); the QK
        // warp skips the item
        if (p.nsplit > 1) {
          if (threadIdx.x < I.hv) p.part_lse[part_row() + threadIdx.x] = -INFINITY;
        } else {
          for (int i = threadIdx.x; i < I.hv * kDV / 8; i += kSoftThreads)
            __stcs(reinterpret_cast<uint4*>(out_t) + i, make_uint4(0, 0, 0, 0));
        }
        if (wn < items) I = item_at<KEYS>(p, wn, groups);
        continue;
      }
      if (!q_in && !convert_q(I)) { ok = false; break; }  // first item, or after an empty one
      q_in = false;
      // key count of item wn's token: loaded now, used by the epilogue
      int b_next = 0;
      const int n_next = wn < items ? token_keys<KEYS>(p, item_token(p, wn, groups), b_next) : 0;
      if (threadIdx.x < kNH) s.negm[threadIdx.x] = 0.f;  // block 0 sets the reference
      named_bar_sync(1, kSoftThreads);
      // lv[h]: this key lane's share of head hb+h's softmax denominator,
      // summed over the blocks (P / s_row, in the current reference's units)
      float lv[32];
#pragma unroll
      for (int h = 0; h < 32; ++h) lv[h] = 0.f;

      for (int j = 0; j < nblk; ++j) {
        const int g = gb + j;
        const int slot = g % NST;
        // S^T of block j is ready; kv_full is also waited so that the
        // producers' per-row scales are visible to this thread.
        bool wt = true;
        if (KVP == 2) {
          // Blockwise rows land raw, key quarter by key quarter, each with its
          // rows' s_row: split each quarter in place as it lands, then
          // release the block to QK.
#pragma unroll 1
          for (int q = 0; q < kRowQ; ++q) {
            wt = wt && mbar_wait(smem_u32(&s.bar_kv_q[q]), g & 1, p.err);
            if (wt) split_quarter(s.kv[slot][0], s.kv[slot][KVP - 1], s.bsc, q);
          }
          fence_proxy_async_smem();
          mbar_arrive(smem_u32(&s.bar_kv_split));
        } else {
          wt = mbar_wait(smem_u32(&s.bar_kv_full[slot]), (g / NST) & 1, p.err);
        }
        wt = wt && mbar_wait(smem_u32(&s.bar_s_full), g & 1, p.err);
        if (!named_bar_and(1, kSoftThreads, wt)) { ok = false; break; }
        tc_fence_after();
        float y[32];
        {
          // S = sum of the two accumulators' QP term columns, two loads per wait
          uint32_t v0[32], v1[32];
          tmem_ld32(tmem + lane_base + kTmemS + hb, v0);
          tmem_ld32(tmem + lane_base + kTmemS + (QP == 2 ? kNH : kQN) + hb, v1);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) y[h] = __uint_as_float(v0[h]) + __uint_as_float(v1[h]);
          if (QP == 2) {
            tmem_ld32(tmem + lane_base + kTmemS + kQN + hb, v0);
            tmem_ld32(tmem + lane_base + kTmemS + kQN + kNH + hb, v1);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 32; ++h) y[h] += __uint_as_float(v0[h]) + __uint_as_float(v1[h]);
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&s.bar_s_free));  // S may now be overwritten by the next QK
        const float sr = SC == kUnit ? 1.f : s.srow[slot][r];
        const float lg = SC == kUnit ? 0.f : __log2f(sr);
        // y = logit (log2 units) minus the head's reference maximum m_h,
        //   y = S * s_row * c_h - m_h,
        // and the PV operand is exp2(y + log2 s_row).  Block 0 has m = 0: it
        // computes the logits themselves and sets the references to its maxima.
        float ymax = -INFINITY;
        {
          const float4* c4p = reinterpret_cast<const float4*>(s.cs + hb);
          const float4* m4p = reinterpret_cast<const float4*>(s.negm + hb);
          float ym[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four independent max chains
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 c = c4p[q], m = m4p[q];
            const float cc[4] = {c.x, c.y, c.z, c.w}, mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int h = 4 * q + k;
              y[h] = fmaf(y[h], SC == kUnit ? cc[k] : sr * cc[k], mm[k]);
              ym[k] = fmaxf(ym[k], y[h]);
            }
          }
          ymax = fmaxf(fmaxf(ym[0], ym[1]), fmaxf(ym[2], ym[3]));
        }
        if ((j + 1) * kBK > n_item && j * kBK + r >= n_item) {  // lanes past the token's keys (its last block only)
#pragma unroll
          for (int h = 0; h < 32; ++h) y[h] = -INFINITY;
          ymax = -INFINITY;
        }
        // Fast path: no element exceeds its head's reference by more than tau.
        if (named_bar_or(1, kSoftThreads, j == 0 || ymax + lg > kTau)) {
          // Slow path (always taken by block 0): t_h = block maximum of y + lg
          // per head across the 128 key lanes.  Block 0 sets m_h = t_h -
          // kPOffset; a later block raises m_h by d_h = t_h - kPOffset where
          // t_h > tau and scales O^T and the row sums of that head by
          // exp2(-d_h).
          int mine = kOrdMin;
#pragma unroll
          for (int h = 0; h < 32; ++h) {
            const int m = __reduce_max_sync(0xffffffffu, ord_int(y[h] + lg));
            if (lane == h) mine = m;
          }
          atomicMax(&s.mx[hb + lane], mine);
          named_bar_sync(1, kSoftThreads);
          if ((warp & 3) == 0) {
            const int hh = hb + lane;
            const float t = ord_float(s.mx[hh]);
            s.mx[hh] = kOrdMin;
            float d = 0.f, f = 1.f;
            if (j == 0 || t > kTau) {
              d = t - kPOffset;
              if (j > 0) f = exp2f(-d);
              s.negm[hh] -= d;
            }
            s.delta[hh] = d;
            s.fac[hh] = f;
          }
          named_bar_sync(1, kSoftThreads);
#pragma unroll
          for (int h = 0; h < 32; ++h) y[h] -= s.delta[hb + h];
          if (j > 0) {
#pragma unroll
            for (int h = 0; h < 32; ++h) lv[h] *= s.fac[hb + h];
            // O^T holds blocks < j: wait for the last PV, then scale each head's column.
            wt = mbar_wait(smem_u32(&s.bar_pv_done), (g - 1) & 1, p.err);
            if (!named_bar_and(1, kSoftThreads, wt)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int part = 0; part < 8; ++part) {  // 4 tiles x 2 halves of this warp's 32 heads
              uint32_t v[16];
              const int c0 = (part & 1) * 16;
              const uint32_t a = tmem + lane_base + (part >> 1) * kNH + hb + c0;
              tmem_ld16(a, v);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < 16; ++h) v[h] = __float_as_uint(__uint_as_float(v[h]) * s.fac[hb + c0 + h]);
              tmem_st16(a, v);
            }
            tmem_wait_st();
            // every lane quarter is rescaled before any quarter's P is
            // published: each PV MMA of this block writes all 128 lanes
            tc_fence_before();
            named_bar_sync(1, kSoftThreads);
          }
        }
        // ---- P row r (this thread's 32 heads) and the row sums
        const float isr = 1.f / sr;
        uint8_t* p_hi = &s.kv[slot][0][kRopeCh * kChunkBytes];
        uint4 lo_keep[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float x[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int h = c * 16 + k;
            x[k] = ex2_approx(SC == kUnit ? y[h] : y[h] + lg);  // 0 past the selection
            lv[h] = SC == kUnit ? lv[h] + x[k] : fmaf(x[k], isr, lv[h]);
          }
          const int c4 = half * 2 + c;
          if (EB == 2) {
            // bf16 P: heads hb .. hb+31 fill chunk kRopeCh + half, 16 heads
            // (two 16-byte pieces) per c
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
              w[k] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            uint8_t* prow = p_hi + half * kChunkBytes + r * 64;
            *reinterpret_cast<uint4*>(prow + sw64(r, 2 * c)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(prow + sw64(r, 2 * c + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
          } else if (PP == 2) {
            uint4 hi;
            split16(x, hi, lo_keep[c]);
            *reinterpret_cast<uint4*>(p_hi + r * 64 + sw64(r, c4)) = hi;
          } else {
            *reinterpret_cast<uint4*>(p_hi + r * 64 + sw64(r, c4)) = quant16(x);
          }
        }
        // This warp's key quarter of the previous block's PV (possibly the
        // previous item's last) must have completed: it reads this quarter's
        // P-lo rows, and P is published per key quarter only once the quarter
        // before it was consumed (so p_full[q] never runs a phase ahead).  No
        // barrier here: one quarter's warps publish before another's, and PV
        // starts on the first quarters.  A timeout is recorded, not taken.
        if (g > 0) mbar_wait(smem_u32(&s.bar_kv_empty[(g - 1) % NST][warp & 3]), ((g - 1) / NST) & 1, p.err);
        if (PP == 2) {
#pragma unroll
          for (int c = 0; c < 2; ++c) *reinterpret_cast<uint4*>(s.plo + r * 64 + sw64(r, half * 2 + c)) = lo_keep[c];
        }
        fence_proxy_async_smem();
        tc_fence_before();  // this thread's TMEM reads (S) precede the PV it releases
        mbar_arrive(smem_u32(&s.bar_p_full[warp & 3]));
      }
      if (!ok) break;
      gb += nblk;

      // ---- epilogue: row sums across the 128 key lanes (no PV needed yet)
      float* linv = s.fac;  // reused: row sums, then 1 / row sum per head
      if (threadIdx.x < kNH) linv[threadIdx.x] = 0.f;
      named_bar_sync(1, kSoftThreads);
      {
        // Transpose-reduce: after log2(32) halving exchanges (31 shuffles),
        // lane l holds the sum over the warp's 32 key lanes for head hb + l.
#pragma unroll
        for (int step = 16; step >= 1; step >>= 1) {
          const bool upper = (lane & step) != 0;
#pragma unroll
          for (int i = 0; i < step; ++i) {
            const float send = upper ? lv[i] : lv[i + step];
            const float keep = upper ? lv[i + step] : lv[i];
            lv[i] = keep + __shfl_xor_sync(0xffffffffu, send, step);
          }
        }
        atomicAdd(&linv[hb + lane], lv[0]);
      }
      // the next item's q while this item's last PV runs, so the next QK
      // overlaps this epilogue
      Item In{};
      if (wn < items) {
        In = item_make(p, wn, groups, n_next, b_next);
        if (In.nblk > 0) {
          if (!convert_q(In)) { ok = false; break; }
          q_in = true;
        }
      }
      // ---- O^T / l -> bf16 once the last PV has completed
      const bool done = named_bar_and(1, kSoftThreads, mbar_wait(smem_u32(&s.bar_pv_done), (gb - 1) & 1, p.err));
      if (threadIdx.x < kNH) {
        // l = sum_j exp2(z_j - m); the reference m is -negm (log2 units)
        float l = linv[threadIdx.x];
        if ((p.nsplit > 1 || p.sink != nullptr) && threadIdx.x < I.hv)
          l = split_or_sink(p, part_row() + threadIdx.x, I.h0 + threadIdx.x, l, s.negm[threadIdx.x]);
        linv[threadIdx.x] = l > 0.f ? 1.f / l : 0.f;
      }
      named_bar_sync(1, kSoftThreads);
      if (done && p.nsplit > 1) {
        tc_fence_after();
        store_partial(p.part_o + (part_row() + hb) * kDV + r, tmem + lane_base + hb, linv + hb, I.hv - hb);
      } else if (done) {
        tc_fence_after();
        // thread = one value column.  Lane pairs swap one value per two heads,
        // so the even lane holds columns (c, c+1) of head h and the odd lane
        // those of head h+1: one 4-byte bf16x2 store each.
        const bool odd = (lane & 1) != 0;
#pragma unroll 1
        for (int tile = 0; tile < 4; ++tile) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + tile * kNH + hb, v);
          tmem_wait_ld();
          uint32_t* o2 = reinterpret_cast<uint32_t*>(out_t + tile * 128 + (r & ~1));
#pragma unroll
          for (int h = 0; h < 32; h += 2) {
            const float a = __uint_as_float(v[h]) * linv[hb + h];
            const float b = __uint_as_float(v[h + 1]) * linv[hb + h + 1];
            const float got = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
            const __nv_bfloat162 pr = odd ? __floats2bfloat162_rn(got, b) : __floats2bfloat162_rn(a, got);
            const int head = hb + h + (odd ? 1 : 0);
            if (head < I.hv) __stcs(o2 + static_cast<int64_t>(head) * (kDV / 2), *reinterpret_cast<const uint32_t*>(&pr));
          }
        }
      }
      // The O^T reads precede the next item's first PV: every softmax thread
      // passes that item's start barrier before any of them publishes P.
      tc_fence_before();
      // linv (s.fac) is rewritten by the next item's slow path only after the
      // named barrier at that item's start; every thread has read it by then
      I = In;
    }
  } else if (warp == kMmaWarp) {
    // =================================================================== QK issuer
    // QK of block g once its rows have landed, its item's q is in place and
    // the softmax of block g-1 has released S.  The whole warp runs the loop;
    // one elected lane issues.
    setmaxnreg_dec<kLowRegs>();
    const bool leader = elect_one();
    constexpr uint32_t IDESC_QK = EB == 2 ? idesc_bf16_f32(kBK, kQN, 0, 0) : idesc_e4m3_f32(kBK, kQN, 0, 0);
    const uint64_t qk_b0 = make_sdesc(smem_u32(s.q), 16, 512, kSwizzle64B);
    const uint64_t kv_a0 = make_sdesc(smem_u32(s.kv[0][0]), 16, 512, kSwizzle64B);
    // q of the CTA's next item with keys, requested once the last QK of the
    // item before it has completed (s.q is then free).  With a 3-D tensor
    // map one load brings all column boxes, else one load per box.
    constexpr int kQBoxes = QP == 2 ? 2 * kChunks : kCh;
    const uint64_t q_policy = make_policy_evict_first();  // q is read once
    int q_issued = 0;
    auto issue_q = [&](int w) {
      ++q_issued;
      if (leader) {
        const int tg = w / p.nsplit;  // (token, head group) of item w
        const int row = tg / groups * p.H + (tg % groups) * kNH;
        mbar_arrive_expect_tx(smem_u32(&s.bar_qraw), kQBoxes * kNH * 64);
        if (p.q_box3d) {
          tma_load_3d_hint(smem_u32(s.q), &tq, 0, row, 0, smem_u32(&s.bar_qraw), q_policy);
        } else {
#pragma unroll 1
          for (int c = 0; c < kQBoxes; ++c)
            tma_load_2d_hint(smem_u32(s.q) + c * (kNH * 64), &tq, 64 * c, row, smem_u32(&s.bar_qraw), q_policy);
        }
      }
      __syncwarp();
    };
    auto next_nonempty = [&](int w) {
      for (w += gridDim.x; w < items; w += gridDim.x)
        if (item_at<KEYS>(p, w, groups).nblk > 0) return w;
      return items;
    };
    int qn = 0, gb = 0;
    bool ok = true;
    {
      const int w0 = item_at<KEYS>(p, blockIdx.x, groups).nblk > 0 ? static_cast<int>(blockIdx.x) : next_nonempty(blockIdx.x);
      if (w0 < items) issue_q(w0);
    }
    for (int w = blockIdx.x; ok && w < items; w += gridDim.x) {
      const Item I = item_at<KEYS>(p, w, groups);
      if (I.nblk == 0) continue;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s.bar_q), qn & 1, p.err));
      ++qn;
      for (int j = 0; ok && j < I.nblk; ++j) {
        const int g = gb + j;
        const bool wt = (g == 0 || mbar_wait(smem_u32(&s.bar_s_free), (g - 1) & 1, p.err)) &&
                        (KVP == 2 ? mbar_wait(smem_u32(&s.bar_kv_split), g & 1, p.err)
                                  : mbar_wait(smem_u32(&s.bar_kv_full[g % NST]), (g / NST) & 1, p.err));
        if (!__all_sync(0xffffffffu, wt)) { ok = false; break; }
        fence_proxy_async_smem();  // the producers' cp.async rows, seen through the barrier, before the MMAs read them
        tc_fence_after();  // after the softmax's tcgen05.ld of S
        const uint64_t slot_off = static_cast<uint64_t>(((g % NST) * KVP * kSlotBytes) >> 4);
        if (leader) {
          issue_qk<QP, KVP, kSAcc, EB>(tmem + kTmemS, kv_a0 + slot_off, qk_b0, IDESC_QK);
          mma_commit(smem_u32(&s.bar_s_full));
        }
        __syncwarp();
      }
      gb += I.nblk;
      if (!ok) break;
      const int wn = next_nonempty(w);
      if (wn < items) {
        // s.q is overwritten only after this item's last QK has completed
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s.bar_s_full), (gb - 1) & 1, p.err));
        if (ok) issue_q(wn);
      }
    }
    if (leader) s.q_issued = q_issued;
  } else if (warp == kPvWarp) {
    // =================================================================== PV issuer
    // PV of block g, key quarter by key quarter as the softmax warps publish
    // P per quarter.  A warp of its own, so that PV is never queued behind
    // the issue of the next QK.  Every PV MMA writes all 128 O^T lanes: an
    // item's first PV overwrites O^T, and the softmax publishes no P before
    // all its warps have read the previous item's O^T (the item-start
    // barrier) and, after a rescale, rescaled all lanes (a barrier).
    setmaxnreg_dec<kLowRegs>();
    const bool leader = elect_one();
    constexpr uint32_t IDESC_PV = EB == 2 ? idesc_bf16_f32(128, kNH, 1, 1) : idesc_e4m3_f32(128, kNH, 1, 1);
    const uint64_t pv_a0 = make_sdesc(smem_u32(s.kv[0][0]), kChunkBytes, 512, kSwizzle64B);
    const uint64_t plo0 = make_sdesc(smem_u32(s.plo), kChunkBytes, 512, kSwizzle64B);
    int gb = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok && w < items; w += gridDim.x) {
      const Item I = item_at<KEYS>(p, w, groups);
      for (int j = 0; j < I.nblk; ++j) {
        const int g = gb + j;
        // O^T[512 vcols x 64 heads] += V^T P^T over the block's 128 keys, one
        // 32-key quarter at a time (issued once that quarter's P is written)
        // with the four 128-column tiles interleaved; each quarter's rows go
        // back to the gather when its MMAs complete.  P hi sits in the slot's
        // rope chunk, P lo in its own buffer.
        const int slot = g % NST;
        const uint64_t slot_off = static_cast<uint64_t>((slot * KVP * kSlotBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < kRowQ; ++ks) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&s.bar_p_full[ks]), g & 1, p.err))) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();  // V rows landed by cp.async (ordered through the softmax's wait)
          tc_fence_after();  // after the softmax's TMEM reads and rescale of O^T
          if (leader) {
#pragma unroll
            for (int pp = 0; pp < PP; ++pp)
#pragma unroll
              for (int kp = 0; kp < KVP; ++kp)
#pragma unroll
                for (int tile = 0; tile < 4; ++tile)
#pragma unroll
                  for (int kst = 0; kst < EB; ++kst) {  // K steps of 32 (e4m3) or 16 (bf16) keys
                    const uint32_t pacc = (j > 0 || pp > 0 || kp > 0 || ks > 0 || kst > 0) ? 1u : 0u;
                    // value tile: 128 columns = 2 * EB chunks; key rows 32 ks + 16 kst (bf16)
                    const int krow = ks * 32 + kst * 16;
                    const uint64_t ad = pv_a0 + slot_off +
                                        static_cast<uint64_t>((kp * kSlotBytes + (2 * EB * tile) * kChunkBytes + krow * 64) >> 4);
                    const uint64_t bd = pp == 0 ? pv_a0 + slot_off + static_cast<uint64_t>((kRopeCh * kChunkBytes + krow * 64) >> 4)
                                                : plo0 + static_cast<uint64_t>((ks * 32 * 64) >> 4);
                    if (EB == 2)
                      mma_f16_ss(tmem + tile * kNH, ad, bd, IDESC_PV, pacc);
                    else
                      mma_f8f6f4_ss(tmem + tile * kNH, ad, bd, IDESC_PV, pacc);
                  }
            mma_commit(smem_u32(&s.bar_kv_empty[slot][ks]));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (leader) mma_commit(smem_u32(&s.bar_pv_done));
        __syncwarp();
      }
      gb += I.nblk;
    }
  } else {
    // =================================================================== gather producers
    setmaxnreg_dec<kLowRegs>();
    const int pt = threadIdx.x - kProdWarp0 * 32;
    const uint64_t keep = make_policy_evict_last();  // the latent pool stays in L2 over the q / out streams
    // The gather threads: kGRows rows x kPieces 16-byte pieces at a time;
    // thread pt copies piece pc of its rows (consecutive threads on
    // consecutive pieces of a row).
    constexpr int kPieces = 36 * EB;  // 16-byte pieces of a cache row
    constexpr int kGRows = kProdThreads / kPieces;
    constexpr int kGThreads = kGRows * kPieces;
    const int pc = pt % kPieces, pr = pt / kPieces;
    const uint8_t* src_c = p.latent + pc * 16;
    bool ok = true;
    int gb = 0;
    for (int w = blockIdx.x; ok && w < items; w += gridDim.x) {
      const Item I = item_at<KEYS>(p, w, groups);
      const int n = I.n;
      if (I.nblk == 0) continue;
      const uint32_t* tok_idx = p.indices + static_cast<int64_t>(I.t) * p.indices_stride;
      const int32_t* pages = p.page_table + static_cast<int64_t>(I.b) * p.max_pages;
      // physical row of the token's key i: its index (kIndexed) or its
      // logical key through the page table (kCausal); out-of-range rows are
      // reported and replaced by row 0
      auto key_row = [&](int i) -> uint32_t {
        int64_t row;
        if (KEYS == kCausal) {
          const int pid = pages[i >> p.page_shift];
          row = (static_cast<int64_t>(pid) << p.page_shift) | (i & ((1 << p.page_shift) - 1));
          if (pid < 0 || row >= p.phys_rows) {
            atomicOr(p.err, kErrPage);
            row = 0;
          }
        } else {
          row = tok_idx[i];
          if (row >= p.phys_rows) {
            atomicOr(p.err, kErrIndex);
            row = 0;
          }
        }
        return static_cast<uint32_t>(row);
      };
      // lanes past the token's keys gather its key 0 again (finite values
      // that the softmax weights by zero)
      const uint32_t first = pt < kBK ? key_row(0) : 0u;
      // Thread pt < 128 owns row pt of every block: its physical row (and
      // tensorwise scale) are loaded one block ahead.
      uint32_t nxt_row = 0;
      float nxt_sr = 1.f;
      auto load_row = [&](int jb) {
        const int key = (I.j0 + jb) * kBK + pt;
        nxt_row = key < n ? key_row(key) : first;
      };
      auto load_scale = [&]() {  // block scales are gathered with the rows
        if (SC == kRow) nxt_sr = p.scales[static_cast<int64_t>(nxt_row) * p.nscale];
      };
      if (pt < kBK) {
        load_row(0);
        load_scale();
      }
      for (int j = 0; j < I.nblk; ++j) {
        const int g = gb + j;
        const int slot = g % NST;
        const uint32_t par = ((g / NST) & 1) ^ 1;
        const bool wt = mbar_wait(smem_u32(&s.bar_kv_empty[slot][0]), par, p.err);
        if (!named_bar_and(2, kProdThreads, ok && wt)) { ok = false; break; }
        if (pt < kBK) {
          s.idx[pt] = nxt_row;
          if (SC != kBlock) s.srow[slot][pt] = nxt_sr;
        }
        named_bar_sync(2, kProdThreads);
        // Key quarter q (rows 32q..32q+31) is refilled once PV of block g-NST
        // has finished with it: 32 rows x 36 16-byte pieces, consecutive
        // threads on consecutive pieces of a row, into the SW64 operand
        // layout.  Blockwise rows land raw (e4m3) in the hi buffer, and the
        // row's 18 block scales (one thread per row) in s.bsc; each quarter is
        // published (kv_q) once landed, with s_row and 1 / s_row of its rows,
        // and the softmax warps split it while later quarters land (measured:
        // publishing only after all four quarters were issued was slower).
        auto publish_quarter = [&](int qq) {
          if (pt < 32) {
            const int row = 32 * qq + pt;
            float sr = 0.f;
#pragma unroll
            for (int b = 0; b < kBlkScales; ++b) sr = fmaxf(sr, s.bsc[row * kBlkScales + b]);
            sr = sr > 0.f ? sr : 1.f;
            s.srow[slot][row] = sr;
            s.bsc[kBK * kBlkScales + row] = 1.f / sr;
          }
          mbar_arrive(smem_u32(&s.bar_kv_q[qq]));
        };
        for (int q = 0; q < kRowQ; ++q) {
          if (q > 0 && ok) ok = mbar_wait(smem_u32(&s.bar_kv_empty[slot][q]), par, p.err);
          if (ok) {
            // Thread pt < kGThreads copies piece pc of rows pr, pr + kGRows, ...
            // of the quarter (pc and pr fixed per thread).
            if (pt < kGThreads) {
              const uint32_t cbase = smem_u32(s.kv[slot][0]) + (pc >> 2) * kChunkBytes;
#pragma unroll
              for (int k = 0; k < (32 + kGRows - 1) / kGRows; ++k) {
                const int rq = pr + k * kGRows;
                if (rq < 32) {
                  const int row = 32 * q + rq;
                  cp_async16_hint(cbase + row * 64 + sw64(row, pc & 3),
                                  src_c + static_cast<int64_t>(s.idx[row]) * (kD * EB), keep);
                }
              }
            }
            if (KVP == 2 && pt < 32) {
              const int row = 32 * q + pt;
              const float* src = p.scales + static_cast<int64_t>(s.idx[row]) * p.nscale;
#pragma unroll
              for (int b = 0; b < kBlkScales; ++b) cp_async4(smem_u32(&s.bsc[row * kBlkScales + b]), src + b);
            }
          }
          if (KVP == 2) {  // quarter q - 1 is published once it has landed, while q is in flight
            cp_async_commit();
            if (q > 0) {
              cp_async_wait_group<1>();
              publish_quarter(q - 1);
            }
          }
        }
        if (KVP != 2) {
          // The slot is full once every producer's copies have landed; the
          // producers do not wait for that themselves but go on to the next
          // block, so the gathers of both slots can be in flight at once.
          // The QK issuer fences (async proxy) after its wait.
          mbar_arrive(smem_u32(&s.bar_kv_full[slot]));
          cp_async_mbar_arrive_noinc(smem_u32(&s.bar_kv_full[slot]));
        }
        // the next block's row and scale load while this block's rows land
        if (pt < kBK && j + 1 < I.nblk) {
          load_row(j + 1);
          load_scale();
        }
        if (KVP == 2) {
          cp_async_wait_all();
          publish_quarter(kRowQ - 1);
        }
      }
      gb += I.nblk;
    }
    cp_async_wait_all();  // no copy is still landing when the CTA tears down
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // a q load still in flight after an error is waited for (bounded) before exit
  if (threadIdx.x == 0 && s.q_issued > q_waited) mbar_wait(smem_u32(&s.bar_qraw), q_waited & 1, p.err);
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

template <int QP, int KVP, int PP, int NST, int SC, int KEYS, int EB = 1>
static smla_status_t launch_k(const CUtensorMap& tq, const Params& p, cudaStream_t stream) {
  const size_t smem = sizeof(Smem<QP, KVP, PP, NST, EB>);
  static_assert(sizeof(Smem<QP, KVP, PP, NST, EB>) <= 232448, "the variant's shared memory exceeds a CTA's 227 KB");
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<QP, KVP, PP, NST, SC, KEYS, EB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return fail_cuda(e, "prefill smem attribute");
  // The register split (setmaxnreg) draws on the launch allocation: refuse a
  // build whose register count would leave the softmax's increase waiting.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, prefill_kernel<QP, KVP, PP, NST, SC, KEYS, EB>);
  if (e != cudaSuccess) return fail_cuda(e, "prefill attributes");
  if (fa.numRegs != kLaunchRegs)
    return fail(SMLA_ERR_UNSUPPORTED, "prefill kernel built with %d registers a thread, the register split needs %d",
                fa.numRegs, kLaunchRegs);
  // persistent: one CTA per SM (shared memory allows no more), at most one per item
  const int64_t items = static_cast<int64_t>(p.T) * ((p.H + kNH - 1) / kNH) * p.nsplit;
  const dim3 grid(static_cast<unsigned>(std::min<int64_t>(items, device_sm_count())));
  prefill_kernel<QP, KVP, PP, NST, SC, KEYS, EB><<<grid, threads_for(KVP), smem, stream>>>(tq, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "prefill launch");
  return SMLA_OK;
}

template <int QP, int KVP, int PP, int NST, int SC>
static smla_status_t launch_t(const CUtensorMap& tq, const Params& p, cudaStream_t stream) {
  return p.keys == kCausal ? launch_k<QP, KVP, PP, NST, SC, kCausal>(tq, p, stream)
                           : launch_k<QP, KVP, PP, NST, SC, kIndexed>(tq, p, stream);
}

}  // namespace pf

smla_status_t launch_attention(const AttnArgs& a, unsigned* err, cudaStream_t stream) {
  using namespace pf;
  const int sbs = a.sbs;
  const int nscale = sbs == 0 ? 0 : (kD + sbs - 1) / sbs;
  Params p{};
  p.q = a.q;
  p.latent = a.latent;
  p.phys_rows = a.phys_rows;
  p.scales = a.scales;
  p.nscale = nscale;
  p.indices = a.indices;
  p.indices_stride = a.indices_stride;
  p.lens = a.topk_lengths;
  p.T = a.T;
  p.H = a.H;
  p.softmax_scale = a.softmax_scale;
  p.out = a.out;
  p.err = err;
  p.sink = a.sink;
  p.nsplit = a.nsplit < 1 ? 1 : a.nsplit;
  p.part_o = a.part_o;
  p.part_lse = a.part_lse;
  if (a.seqs) {
    p.keys = kCausal;
    p.cu_q = a.seqs->cu_q;
    p.kv_len = a.seqs->kv_len;
    p.page_table = a.seqs->page_table;
    p.B = a.seqs->B;
    p.max_pages = a.seqs->max_pages;
    p.page_shift = __builtin_ctz(static_cast<unsigned>(a.seqs->page_size));
  } else {
    p.keys = kIndexed;
  }
  const bool bf16 = a.q_dtype == SMLA_BF16;
  if (bf16 && sbs != 0 && sbs < kD) return fail(SMLA_ERR_UNSUPPORTED, "bf16 q with block scales is not built (shared memory)");
  // q rows [T * H] x (576 elements) as bytes, loaded as 64-byte column boxes
  // of 64 rows: preferably one 3-D box (x = byte in the box, y = row, z =
  // box index with a 64-byte stride), else a 2-D map with one load per box.
  CUtensorMap tq;
  const int T = a.T, H = a.H;
  const uint64_t pitch = static_cast<uint64_t>(kD) * (bf16 ? 2 : 1);
  const uint32_t nbox = static_cast<uint32_t>(pitch / 64);
  {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(T) * H, nbox};
    const uint64_t strides[2] = {pitch, 64};
    const uint32_t box[3] = {64, static_cast<uint32_t>(kNH), nbox};
    p.q_box3d = encode_tma_u8(&tq, a.q, 3, dims, strides, box, 64) ? 1 : 0;
  }
  if (!p.q_box3d && !encode_tma_2d_u8(&tq, a.q, pitch, static_cast<uint64_t>(T) * H, 64, kNH, 64))
    return fail(SMLA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the prefill q tensor map");
  if (a.cache_bf16) {
    // bf16 cache: bf16 x bf16 MMAs, one gather slot (a 128-row block of
    // 1152-byte rows and the 64-head bf16 q fill shared memory)
    if (!bf16 || sbs != 0 || p.keys != kIndexed)
      return fail(SMLA_ERR_UNSUPPORTED, "a bf16 cache takes bf16 q, no scales and indexed keys");
    return launch_k<1, 1, 1, 1, kUnit, kIndexed, 2>(tq, p, stream);
  }
  if (sbs == 0) return bf16 ? launch_t<2, 1, 2, 2, kUnit>(tq, p, stream) : launch_t<1, 1, 1, 2, kUnit>(tq, p, stream);
  if (sbs >= kD) return bf16 ? launch_t<2, 1, 2, 2, kRow>(tq, p, stream) : launch_t<1, 1, 1, 2, kRow>(tq, p, stream);
  return launch_t<1, 2, 1, 1, kBlock>(tq, p, stream);
}

}  // namespace smla
