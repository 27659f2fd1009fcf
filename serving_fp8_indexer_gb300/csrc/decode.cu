// Split-K sparse MLA decode: host-side split choice and the kernel that
// combines the splits' partial outputs.
//
// With one or two query tokens per sequence, (token, 64-head group) work
// items cannot fill the GPU (8 sequences x 2 tokens x 2 head groups = 32 of
// 152 SMs).  The attention kernel therefore divides each token's key blocks
// among nsplit work items; each writes its partial output normalised by its
// own softmax denominator, O_s = sum_{j in s} p_j V_j / l_s (f32), and its
// log2-sum-exp L_s = m_s + log2 l_s.  This kernel merges them:
//   out = sum_s 2^(L_s - M) O_s / (sum_s 2^(L_s - M) + 2^(sink*log2e - M)),
// M the largest of the L_s (and of the sink term), which equals the softmax
// over all of the token's keys (and the sink) in one pass.
#include <algorithm>
#include <mutex>

#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {
namespace dec {

constexpr int kDV = 512;
constexpr int kThreads = kDV / 4;  // four value columns a thread (one float4)
constexpr float kLog2e = 1.4426950408889634f;

// One CTA per (token, head) output row.
__global__ void __launch_bounds__(kThreads) combine_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_lse,
                                                           const float* __restrict__ sink, int H, int nsplit,
                                                           uint16_t* __restrict__ out) {
  const int row = blockIdx.x;  // t * H + h
  const int t = row / H, h = row - t * H;
  const int64_t base = static_cast<int64_t>(t) * nsplit * H + h;  // split s at base + s * H
  float m = sink ? sink[h] * kLog2e : -INFINITY;
  for (int sp = 0; sp < nsplit; ++sp) m = fmaxf(m, part_lse[base + static_cast<int64_t>(sp) * H]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (m != -INFINITY) {
    if (sink) den = exp2f(sink[h] * kLog2e - m);
    for (int sp = 0; sp < nsplit; ++sp) {
      const float lse = part_lse[base + static_cast<int64_t>(sp) * H];
      if (lse == -INFINITY) continue;  // an empty split: its partial was never written
      const float wgt = exp2f(lse - m);
      den += wgt;
      const float4 o = __ldcs(reinterpret_cast<const float4*>(part_o + (base + static_cast<int64_t>(sp) * H) * kDV) +
                              threadIdx.x);
      acc.x = fmaf(wgt, o.x, acc.x);
      acc.y = fmaf(wgt, o.y, acc.y);
      acc.z = fmaf(wgt, o.z, acc.z);
      acc.w = fmaf(wgt, o.w, acc.w);
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 v;
  v.x = *reinterpret_cast<const uint32_t*>(&lo);
  v.y = *reinterpret_cast<const uint32_t*>(&hi);
  reinterpret_cast<uint2*>(out + static_cast<int64_t>(row) * kDV)[threadIdx.x] = v;
}

// Scratch for smla_sparse_decode_noalloc: the split partials of one call
// live here instead of in a caller-provided workspace.  Every GPU that loads
// the library holds these bytes until the process exits.  Host code must not
// use the array's name as a device address: it is a host-side stand-in; the
// device address comes from cudaGetSymbolAddress (noalloc_scratch below).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

}  // namespace dec

int decode_splits(int T, int H, int indices_stride) {
  constexpr int kNH = 64, kBK = 128;
  const int64_t base = static_cast<int64_t>(T) * ((H + kNH - 1) / kNH);  // (token, head group) items
  const int sms = device_sm_count();
  const int nb = (std::max(indices_stride, 1) + kBK - 1) / kBK;  // key blocks of the longest selection
  if (base <= 0 || base >= sms || nb <= 1) return 1;
  // as many splits as one wave of persistent CTAs holds, then evened out so
  // that every split of a full-length selection gets the same block count
  const int s0 = static_cast<int>(std::min<int64_t>(sms / base, nb));
  const int per = (nb + s0 - 1) / s0;
  return (nb + per - 1) / per;
}

size_t decode_workspace_bytes(int T, int H, int nsplit) {
  if (nsplit <= 1 || T <= 0) return 0;
  const size_t rows = static_cast<size_t>(T) * nsplit * H;
  const size_t o_bytes = (rows * dec::kDV * sizeof(float) + 255) & ~size_t(255);
  return o_bytes + ((rows * sizeof(float) + 255) & ~size_t(255));
}

smla_status_t launch_decode_combine(const float* part_o, const float* part_lse, const float* sink, int T, int H,
                                    int nsplit, uint16_t* out, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(T) * H;
  if (rows <= 0) return SMLA_OK;
  if (rows > 0x7fffffff) return fail(SMLA_ERR_UNSUPPORTED, "decode combine grid too large");
  dec::combine_kernel<<<static_cast<unsigned>(rows), dec::kThreads, 0, stream>>>(part_o, part_lse, sink, H, nsplit,
                                                                                  out);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(e, "decode combine launch");
  return SMLA_OK;
}

// Device address of the static scratch on the current device, looked up
// once per device (with that device current) and cached.
static smla_status_t noalloc_scratch(void** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SMLA_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, dec::g_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(decode scratch)");
    addr[dev] = p;
  }
  *out = addr[dev];
  return SMLA_OK;
}

size_t noalloc_scratch_bytes() { return dec::kNoAllocScratchBytes; }

smla_status_t noalloc_scratch_for(size_t need, void** out) {
  if (need > dec::kNoAllocScratchBytes)
    return fail(SMLA_ERR_UNSUPPORTED,
                "smla_sparse_decode_noalloc: these sizes need %zu bytes of split scratch, more than its fixed %zu; "
                "use smla_sparse_decode with a workspace",
                need, dec::kNoAllocScratchBytes);
  *out = nullptr;
  if (need == 0) return SMLA_OK;
  return noalloc_scratch(out);
}

}  // namespace smla
