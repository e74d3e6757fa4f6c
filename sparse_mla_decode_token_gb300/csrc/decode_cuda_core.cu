// CUDA-core sparse MLA decode kernel (fp32 FMA; no tensor cores).
//
// One CTA computes one (token, split, group of 16 heads).  It walks the split's
// columns 32 at a time: warp 0 compacts the valid slots of the 32 columns
// (ballot), all threads gather those rows into shared memory as fp32, each
// warp forms the 32 logits of two heads and runs the online softmax with
// warp shuffles, then every thread updates its 2 output dims of all 16 heads.
// This kernel is the plain reference point of the library; the tcgen05
// kernel carries the throughput.
#include "common.cuh"
#include "kernels.h"

namespace smla {
namespace {

constexpr int kHeadsPerCta = 16;
constexpr int kTile = 32;            // columns per step == slots per tile
constexpr int kThreads = 256;
constexpr int kKvPitch = kHeadDim + 1;   // fp32 row pitch: conflict-free column reads

struct CudaCoreSmem {
  float q[kHeadsPerCta][kHeadDim];       // q * bmm1 * log2(e)
  float kv[kTile][kKvPitch];             // gathered rows, fp32
  float p[kHeadsPerCta][kTile];          // softmax numerators of the tile
  float alpha[kHeadsPerCta];             // rescale of the running output
  float m[kHeadsPerCta];                 // running max (base-2 logits)
  float l[kHeadsPerCta];                 // running sum
  int64_t row_off[kTile];                // element offsets of the valid slots
  int from_swa[kTile];
  int n_valid;
};

__device__ __forceinline__ void decode8(const uint4 raw, float* dst, bool bf16) {
  if (bf16) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 f = __bfloat1622float2(h[k]);
      dst[2 * k] = f.x;
      dst[2 * k + 1] = f.y;
    }
  }
}

__device__ __forceinline__ void decode16_e4m3(const uint4 raw, float* dst) {
  const __nv_fp8x2_storage_t* h = reinterpret_cast<const __nv_fp8x2_storage_t*>(&raw);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h[k], __NV_E4M3);
    float2 f = __half22float2(*reinterpret_cast<__half2*>(&hr));
    dst[2 * k] = f.x;
    dst[2 * k + 1] = f.y;
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads)
decode_cuda_core_kernel(const DecodeParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  CudaCoreSmem& sm = *reinterpret_cast<CudaCoreSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int HG = p.H / kHeadsPerCta;
  const int hg = blockIdx.x % HG;
  const int rest = blockIdx.x / HG;
  const int s = rest % p.num_splits;
  const int t = rest / p.num_splits;
  const int h0 = hg * kHeadsPerCta;

  const TokenInfo ti = token_info(p, t);
  int c0, c1;
  split_range(ti.n_lim, p.num_splits, s, &c0, &c1);
  const float qscale = load_scale(p.bmm1, p.bmm1_dev) * kLog2e;
  const float bmm2 = load_scale(p.bmm2, p.bmm2_dev);

  // Q of 16 heads, pre-scaled so that logits come out in base-2 units.
  {
    const int elems = kHeadsPerCta * kHeadDim;
    constexpr int kPer = kBf16 ? 8 : 16;
    for (int c = tid; c < elems / kPer; c += kThreads) {
      int e = c * kPer, h = e / kHeadDim, d = e % kHeadDim;
      const unsigned char* src = reinterpret_cast<const unsigned char*>(p.q) +
          ((int64_t)t * p.q_stride_token + (int64_t)(h0 + h) * kHeadDim + d) * (kBf16 ? 2 : 1);
      uint4 raw = __ldg(reinterpret_cast<const uint4*>(src));
      float v[16];
      if (kBf16) decode8(raw, v, true); else decode16_e4m3(raw, v);
#pragma unroll
      for (int k = 0; k < kPer; ++k) sm.q[h][d + k] = v[k] * qscale;
    }
  }
  // Each warp owns heads (warp, warp + 8) for the softmax; every lane keeps the
  // running max / sum of both.
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float acc[kHeadsPerCta][2];
#pragma unroll
  for (int h = 0; h < kHeadsPerCta; ++h) acc[h][0] = acc[h][1] = 0.f;
  __syncthreads();

  for (int cb = c0; cb < c1; cb += kTile) {
    // a2: compact the valid slots of columns [cb, cb + 32)
    if (warp == 0) {
      int j = cb + lane;
      bool swa = false;
      int64_t off = (j < c1) ? slot_row_offset(p, ti, t, j, &swa) : -1;
      unsigned ball = __ballot_sync(0xffffffffu, off >= 0);
      if (off >= 0) {
        int slot = __popc(ball & ((1u << lane) - 1u));
        sm.row_off[slot] = off;
        sm.from_swa[slot] = swa;
      }
      if (lane == 0) sm.n_valid = __popc(ball);
    }
    __syncthreads();
    const int nv = sm.n_valid;
    if (nv == 0) { __syncthreads(); continue; }

    // a3: gather rows (16-byte vector loads) into fp32 shared memory
    {
      constexpr int kPer = kBf16 ? 8 : 16;
      constexpr int kChunks = kHeadDim / kPer;
      for (int c = tid; c < nv * kChunks; c += kThreads) {
        int r = c / kChunks, d = (c % kChunks) * kPer;
        const unsigned char* base = reinterpret_cast<const unsigned char*>(sm.from_swa[r] ? p.swa : p.comp);
        uint4 raw = __ldg(reinterpret_cast<const uint4*>(base + (sm.row_off[r] + d) * (kBf16 ? 2 : 1)));
        float v[16];
        if (kBf16) decode8(raw, v, true); else decode16_e4m3(raw, v);
#pragma unroll
        for (int k = 0; k < kPer; ++k) sm.kv[r][d + k] = v[k];
      }
    }
    __syncthreads();

    // a4: logits of heads (warp, warp + 8) against slot `lane`
    float sc[2] = {0.f, 0.f};
    if (lane < nv) {
      const float* kr = sm.kv[lane];
      const float* q0 = sm.q[warp];
      const float* q1 = sm.q[warp + 8];
#pragma unroll 8
      for (int d = 0; d < kHeadDim; ++d) {
        float kv = kr[d];
        sc[0] = fmaf(q0[d], kv, sc[0]);
        sc[1] = fmaf(q1[d], kv, sc[1]);
      }
    } else {
      sc[0] = sc[1] = -INFINITY;
    }
    // a5: online softmax (base 2)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float mx = sc[k];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float m_new = fmaxf(m_run[k], mx);
      float alpha = (m_run[k] == -INFINITY) ? 0.f : fast_exp2(m_run[k] - m_new);
      float pj = (lane < nv) ? fast_exp2(sc[k] - m_new) : 0.f;
      float sum = pj;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      l_run[k] = l_run[k] * alpha + sum;
      m_run[k] = m_new;
      int h = warp + 8 * k;
      sm.p[h][lane] = pj;
      if (lane == 0) sm.alpha[h] = alpha;
    }
    __syncthreads();

    // a6: acc[h][:] = alpha * acc + sum_j p[h][j] * kv[j][:]
#pragma unroll
    for (int h = 0; h < kHeadsPerCta; ++h) {
      float a = sm.alpha[h];
      acc[h][0] *= a;
      acc[h][1] *= a;
    }
    for (int j = 0; j < nv; ++j) {
      float v0 = sm.kv[j][tid], v1 = sm.kv[j][tid + 256];
#pragma unroll
      for (int h = 0; h < kHeadsPerCta; ++h) {
        float pj = sm.p[h][j];
        acc[h][0] = fmaf(pj, v0, acc[h][0]);
        acc[h][1] = fmaf(pj, v1, acc[h][1]);
      }
    }
    __syncthreads();
  }

  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      sm.m[warp + 8 * k] = m_run[k];
      sm.l[warp + 8 * k] = l_run[k];
    }
  }
  __syncthreads();

  // a7 / a9 epilogue
#pragma unroll
  for (int h = 0; h < kHeadsPerCta; ++h) {
    const float l = sm.l[h];
    const float lse = (l > 0.f) ? sm.m[h] + fast_log2(l) : -INFINITY;
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    const int hh = h0 + h;
    if (p.num_splits == 1) {
      float f = inv * bmm2;
      if (p.sinks != nullptr && l > 0.f)
        f *= 1.f / (1.f + fast_exp2(__ldg(p.sinks + hh) * kLog2e - lse));
      __nv_bfloat16* o = p.out + ((int64_t)t * p.H + hh) * kHeadDim;
      o[tid] = __float2bfloat16_rn(acc[h][0] * f);
      o[tid + 256] = __float2bfloat16_rn(acc[h][1] * f);
      if (tid == 0 && p.out_lse) p.out_lse[(int64_t)t * p.H + hh] = lse;
    } else {
      const int64_t row = ((int64_t)t * p.H + hh) * p.num_splits + s;
      __nv_bfloat16* o = p.part_o + row * kHeadDim;
      o[tid] = __float2bfloat16_rn(acc[h][0] * inv);
      o[tid + 256] = __float2bfloat16_rn(acc[h][1] * inv);
      if (tid == 0) p.part_lse[row] = lse;
    }
  }
}

}  // namespace

int cuda_core_smem_bytes() { return (int)sizeof(CudaCoreSmem); }
int cuda_core_threads() { return kThreads; }
int cuda_core_ctas_per_split(int H) { return H / kHeadsPerCta; }

cudaError_t launch_decode_cuda_core(const DecodeParams& p, int grid, cudaStream_t stream) {
  const int smem = cuda_core_smem_bytes();
  cudaError_t e;
  if (p.dtype == SMLA_BF16) {
    e = cudaFuncSetAttribute(decode_cuda_core_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    decode_cuda_core_kernel<true><<<grid, kThreads, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(decode_cuda_core_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    decode_cuda_core_kernel<false><<<grid, kThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace smla
