// Split-K combine: merges S normalised partials of every (token, head).
//
// The partial layout [T, H, S, 512] (BF16) plus [T, H, S] (fp32) base-2 LSEs follows the
// split partials of the FlashInfer cake_sparse_mla_sm120_dsv4_nvfp4_decode page
// (Parameters: mid_out, mid_lse).  With LSE_s the base-2 log-sum-exp of split s:
//   LSE = log2 sum_s 2^{LSE_s},   O = sum_s 2^{LSE_s - LSE} O_s,
// then the sink joins the normaliser, O *= 1 / (1 + 2^{sink*log2(e) - LSE})
// (cake page, Parameters: attn_sink), then O *= bmm2_scale and is rounded to
// BF16.  A head whose splits are all empty gets O = 0 and LSE = -inf.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace smla {
namespace {

constexpr int kHeadsPerCta = 2;
constexpr int kThreadsPerHead = kHeadDim / 4;   // 4 dims per thread

// Merges n normalised partials of one (token, head) into its output row: the
// thread's kVec dims d..d+kVec-1 (kVec = 4 or 8).  lse_at(k) is partial k's
// base-2 LSE, row_at(k) points at its kVec BF16 dims.
template <int kVec, class LseAt, class RowAt>
__device__ __forceinline__ void merge_partials(const DecodeParams& p, int h, int n, int d, LseAt lse_at, RowAt row_at,
                                               __nv_bfloat16* out_row, float* out_lse) {
  using V = typename std::conditional<kVec == 8, uint4, uint2>::type;
  // loads in batches of kBatch independent requests, so that their latencies overlap
  constexpr int kBatch = 8;
  float mx = -INFINITY;
  for (int s0 = 0; s0 < n; s0 += kBatch) {
    float l[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) l[k] = s0 + k < n ? lse_at(s0 + k) : -INFINITY;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) mx = fmaxf(mx, l[k]);
  }
  float acc[kVec];
#pragma unroll
  for (int i = 0; i < kVec; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int s0 = 0; s0 < n; s0 += kBatch) {
      float w[kBatch];
      V o[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const bool in = s0 + k < n;
        const float ls = in ? lse_at(s0 + k) : -INFINITY;
        w[k] = ls == -INFINITY ? 0.f : fast_exp2(ls - mx);   // an empty partial is all zero
        if (in) o[k] = __ldg(row_at(s0 + k));
        else memset(&o[k], 0, sizeof(V));
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&o[k]);
#pragma unroll
        for (int i = 0; i < kVec / 2; ++i) {
          const float2 a = __bfloat1622float2(b2[i]);
          acc[2 * i] = fmaf(w[k], a.x, acc[2 * i]);
          acc[2 * i + 1] = fmaf(w[k], a.y, acc[2 * i + 1]);
        }
        wsum += w[k];
      }
    }
  }
  float lse = -INFINITY, f = 0.f;
  if (wsum > 0.f) {
    lse = mx + fast_log2(wsum);
    f = load_scale(p.bmm2, p.bmm2_dev) / wsum;
    if (p.sinks != nullptr) f *= 1.f / (1.f + fast_exp2(__ldg(p.sinks + h) * kLog2e - lse));
  }
  V packed;
  uint32_t* pw = reinterpret_cast<uint32_t*>(&packed);
#pragma unroll
  for (int i = 0; i < kVec / 2; ++i) {
    __nv_bfloat162 v = __floats2bfloat162_rn(acc[2 * i] * f, acc[2 * i + 1] * f);
    pw[i] = *reinterpret_cast<uint32_t*>(&v);
  }
  *reinterpret_cast<V*>(out_row + d) = packed;
  if (d == 0 && out_lse != nullptr) *out_lse = lse;
}

__global__ void __launch_bounds__(kHeadsPerCta * kThreadsPerHead)
combine_kernel(const DecodeParams p) {
  const int S = p.num_splits;
  const int hl = threadIdx.x / kThreadsPerHead;
  const int d = (threadIdx.x % kThreadsPerHead) * 4;
  const int64_t th = (int64_t)blockIdx.x * kHeadsPerCta + hl;   // flattened (t, h)
  if (th >= (int64_t)p.sum_q * p.H) return;
  const int h = (int)(th % p.H);
  const float* lse_s = p.part_lse + th * S;
  const uint2* o_s = reinterpret_cast<const uint2*>(p.part_o + th * S * kHeadDim + d);   // 4 BF16 dims
  // the split kernel's partials become visible here (programmatic dependent launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  merge_partials<4>(
      p, h, S, d, [&](int k) { return __ldg(lse_s + k); }, [&](int k) { return o_s + (int64_t)k * (kHeadDim / 4); },
      p.out + th * kHeadDim, p.out_lse ? p.out_lse + th : nullptr);
}

}  // namespace

cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream) {
  const int64_t heads = (int64_t)p.sum_q * p.H;
  const int64_t grid = (heads + kHeadsPerCta - 1) / kHeadsPerCta;
  // Programmatic dependent launch: the combine grid may be scheduled while the
  // split kernel drains; griddepcontrol.wait in the kernel orders its reads
  // after the split kernel's writes.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kHeadsPerCta * kThreadsPerHead);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace smla
