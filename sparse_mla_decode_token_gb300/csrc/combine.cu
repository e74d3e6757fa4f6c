// Split-K combine: merges S normalised partials of every (token, head); and
// the merge of the pieces of tokens that the balanced mode cuts.
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

// Balanced mode: cluster c of P took the columns [g(c), g(c + 1)) of the
// token-major column space, g(c) = floor(T W c / P).  A token cut by one or
// more of these boundaries has a head piece (slot 2c + 1 of the cluster where
// it starts) and one piece per later cluster that covers part of it (slot 2c'
// of each).  Block (b, four heads) merges the token cut at g(b + 1) if that is
// the token's first cut; a thread takes 8 dims of one head.
constexpr int kPieceHeadsPerCta = 4;
constexpr int kPieceThreadsPerHead = kHeadDim / 8;

template <class I>
__device__ __forceinline__ bool piece_merge_of(const DecodeParams& p, I clusters, I b, int* t_out, int* n_out) {
  const I W = (I)p.W, total = (I)p.sum_q * W;
  const I cut = total * (b + 1) / clusters;
  if (cut % W == 0) return false;                 // a token edge: nothing cut here
  const I t = cut / W;
  if (total * b / clusters > t * W) return false; // an earlier boundary cuts this token
  I last = b + 1;                                 // the last cluster that covers part of token t
  while (last + 1 < clusters && total * (last + 1) / clusters < (t + 1) * W) ++last;
  *t_out = (int)t;
  *n_out = (int)(last - b + 1);
  return true;
}

__global__ void __launch_bounds__(kPieceHeadsPerCta * kPieceThreadsPerHead)
combine_pieces_kernel(const DecodeParams p, int clusters, const __nv_bfloat16* piece_o, const float* piece_lse) {
  const int hblocks = (p.H + kPieceHeadsPerCta - 1) / kPieceHeadsPerCta;
  const int b = blockIdx.x / hblocks;
  const int h = (blockIdx.x % hblocks) * kPieceHeadsPerCta + threadIdx.x / kPieceThreadsPerHead;
  const int d = (threadIdx.x % kPieceThreadsPerHead) * 8;
  if (h >= p.H) return;
  int t = 0, n = 0;
  // 32-bit arithmetic where T W P fits (divisions are the cost here)
  const bool small = (uint64_t)p.sum_q * (uint64_t)p.W * (uint64_t)clusters < (1ull << 32);
  const bool merge = small ? piece_merge_of<uint32_t>(p, (uint32_t)clusters, (uint32_t)b, &t, &n)
                           : piece_merge_of<uint64_t>(p, (uint64_t)clusters, (uint64_t)b, &t, &n);
  if (!merge) return;
  const int64_t H = p.H;
  auto slot = [&](int k) -> int64_t { return k == 0 ? 2 * (int64_t)b + 1 : 2 * ((int64_t)b + k); };
  asm volatile("griddepcontrol.wait;" ::: "memory");
  merge_partials<8>(
      p, h, n, d, [&](int k) { return __ldg(piece_lse + slot(k) * H + h); },
      [&](int k) { return reinterpret_cast<const uint4*>(piece_o + (slot(k) * H + h) * kHeadDim + d); },
      p.out + ((int64_t)t * H + h) * kHeadDim, p.out_lse ? p.out_lse + (int64_t)t * H + h : nullptr);
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

cudaError_t launch_combine_pieces(const DecodeParams& p, int clusters, const __nv_bfloat16* piece_o,
                                  const float* piece_lse, cudaStream_t stream) {
  const int64_t grid = (int64_t)(clusters - 1) * ((p.H + kPieceHeadsPerCta - 1) / kPieceHeadsPerCta);
  if (grid <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kPieceHeadsPerCta * kPieceThreadsPerHead);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_pieces_kernel, p, clusters, piece_o, piece_lse);
}

}  // namespace smla
