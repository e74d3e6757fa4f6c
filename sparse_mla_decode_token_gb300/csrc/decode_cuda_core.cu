// CUDA-core sparse MLA decode kernel (fp32 FMA; no tensor cores).
//
// One CTA computes one (token, split, group of 16 heads).  It walks the split's
// columns 32 at a time: warp 0 compacts the valid slots of the 32 columns
// (ballot), all threads gather those rows into shared memory as fp32, each
// warp forms the 32 logits of two heads and runs the online softmax with
// warp shuffles, then every thread updates its 2 output dims of all 16 heads.
// This kernel is the plain reference point of the library; the tcgen05
// kernels carry the throughput.  It is also the kernel of the packed KV row
// forms (584-byte packed FP8, 384-byte NVFP4; layouts in include/smla.h),
// whose rows it dequantises while gathering them into shared memory.
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

// Packed FP8 row (584 bytes, 8-byte aligned): work item c < 56 decodes NoPE
// dims [8c, 8c + 8) (E4M3 times 2^(e - 127) of their 64-dim block), item
// 56 + i RoPE dims [448 + 4i, 448 + 4i + 4) (BF16).
__device__ __forceinline__ void packed_fp8_item(const unsigned char* row, int c, float* dst) {
  if (c < 56) {
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(row + 8 * c));
    const float scale = ldexpf(1.0f, (int)__ldg(row + 448 + c / 8) - 127);
    float v[16];
    decode16_e4m3(make_uint4(raw.x, raw.y, 0u, 0u), v);
#pragma unroll
    for (int k = 0; k < 8; ++k) dst[8 * c + k] = v[k] * scale;
  } else {
    const int i = c - 56;
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(row + 456 + 8 * i));
    float v[8];
    decode8(make_uint4(raw.x, raw.y, 0u, 0u), v, true);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[448 + 4 * i + k] = v[k];
  }
}
constexpr int kPackedFp8Items = 56 + 16;

// NVFP4 row (384 bytes, 16-byte aligned): work item c < 14 decodes NoPE dims
// [32c, 32c + 32) (E2M1, low nibble first, times the E4M3 scale of their
// 16-dim block and the row's fp32 scale), item 14 + i RoPE dims 448 + 2i,
// 449 + 2i (BF16).
__device__ __forceinline__ void nvfp4_item(const unsigned char* row, int c, float* dst) {
  if (c < 14) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(row + 16 * c));
    const float g = __ldg(reinterpret_cast<const float*>(row + 380));
    const float s0 = e4m3_value(__ldg(row + 224 + 2 * c)) * g, s1 = e4m3_value(__ldg(row + 225 + 2 * c)) * g;
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const uint32_t code = (w[k >> 3] >> (4 * (k & 7))) & 0xFu;
      dst[32 * c + k] = e2m1_value(code) * (k < 16 ? s0 : s1);
    }
  } else {
    const int i = c - 14;
    const uint32_t raw = __ldg(reinterpret_cast<const uint32_t*>(row + 252 + 4 * i));
    float v[8];
    decode8(make_uint4(raw, 0u, 0u, 0u), v, true);
    dst[448 + 2 * i] = v[0];
    dst[449 + 2 * i] = v[1];
  }
}
constexpr int kNvfp4Items = 14 + 32;

// kKind: SMLA_BF16 / SMLA_E4M3 rows and query, or a packed KV form with a BF16 query.
template <int kKind>
__global__ void __launch_bounds__(kThreads)
decode_cuda_core_kernel(const DecodeParams p) {
  constexpr bool kBf16 = kKind != SMLA_E4M3;                          // query elements
  constexpr bool kPacked = kKind == SMLA_PACKED_FP8 || kKind == SMLA_NVFP4;
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

    // a3: gather rows (16-byte vector loads) into fp32 shared memory;
    // packed rows are dequantised on the way
    if constexpr (kPacked) {
      constexpr int kItems = kKind == SMLA_PACKED_FP8 ? kPackedFp8Items : kNvfp4Items;
      for (int c = tid; c < nv * kItems; c += kThreads) {
        const int r = c / kItems, item = c % kItems;
        const unsigned char* row =
            reinterpret_cast<const unsigned char*>(sm.from_swa[r] ? p.swa : p.comp) + sm.row_off[r];
        if constexpr (kKind == SMLA_PACKED_FP8) packed_fp8_item(row, item, sm.kv[r]);
        else nvfp4_item(row, item, sm.kv[r]);
      }
    } else {
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
  auto launch = [&](auto kernel) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
  };
  switch (p.dtype) {
    case SMLA_BF16: return launch(decode_cuda_core_kernel<SMLA_BF16>);
    case SMLA_E4M3: return launch(decode_cuda_core_kernel<SMLA_E4M3>);
    case SMLA_PACKED_FP8: return launch(decode_cuda_core_kernel<SMLA_PACKED_FP8>);
    case SMLA_NVFP4: return launch(decode_cuda_core_kernel<SMLA_NVFP4>);
  }
  return cudaErrorInvalidValue;
}

}  // namespace smla
