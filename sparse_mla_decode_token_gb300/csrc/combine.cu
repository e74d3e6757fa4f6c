// Split-K combine: merges S normalised partials of every (token, head).
//
// The partial layout [T, H, S, 512] plus [T, H, S] base-2 LSEs follows the
// split partials of the FlashInfer cake_sparse_mla_sm120_dsv4_nvfp4_decode page
// (Parameters: mid_out, mid_lse).  With LSE_s the base-2 log-sum-exp of split s:
//   LSE = log2 sum_s 2^{LSE_s},   O = sum_s 2^{LSE_s - LSE} O_s,
// then the sink joins the normaliser, O *= 1 / (1 + 2^{sink*log2(e) - LSE})
// (cake page, Parameters: attn_sink), then O *= bmm2_scale and is rounded to
// BF16.  A head whose splits are all empty gets O = 0 and LSE = -inf.
#include "common.cuh"
#include "kernels.h"

namespace smla {
namespace {

constexpr int kHeadsPerCta = 2;
constexpr int kThreadsPerHead = kHeadDim / 4;   // 4 dims per thread

__global__ void __launch_bounds__(kHeadsPerCta * kThreadsPerHead)
combine_kernel(const DecodeParams p) {
  const int S = p.num_splits;
  const int hl = threadIdx.x / kThreadsPerHead;
  const int d = (threadIdx.x % kThreadsPerHead) * 4;
  const int64_t th = (int64_t)blockIdx.x * kHeadsPerCta + hl;   // flattened (t, h)
  if (th >= (int64_t)p.sum_q * p.H) return;
  const int h = (int)(th % p.H);
  const float* lse_s = p.part_lse + th * S;

  float mx = -INFINITY;
  for (int s = 0; s < S; ++s) mx = fmaxf(mx, __ldg(lse_s + s));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      float ls = __ldg(lse_s + s);
      if (ls == -INFINITY) continue;
      float w = fast_exp2(ls - mx);
      float4 o = __ldg(reinterpret_cast<const float4*>(p.part_o + (th * S + s) * kHeadDim + d));
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
      wsum += w;
    }
  }
  float lse = -INFINITY, f = 0.f;
  if (wsum > 0.f) {
    lse = mx + fast_log2(wsum);
    f = load_scale(p.bmm2, p.bmm2_dev) / wsum;
    if (p.sinks != nullptr) f *= 1.f / (1.f + fast_exp2(__ldg(p.sinks + h) * kLog2e - lse));
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * f, acc.y * f);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * f, acc.w * f);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p.out + th * kHeadDim + d) = packed;
  if (d == 0 && p.out_lse != nullptr) p.out_lse[th] = lse;
}

}  // namespace

cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream) {
  const int64_t heads = (int64_t)p.sum_q * p.H;
  const int64_t grid = (heads + kHeadsPerCta - 1) / kHeadsPerCta;
  combine_kernel<<<(unsigned)grid, kHeadsPerCta * kThreadsPerHead, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
