// Shared device-side definitions of the sparse MLA decode kernels.
//
// Token metadata and slot selection follow the FlashInfer
// trtllm_batch_decode_sparse_mla_dsv4 page (description, SM100/SM103
// paragraph; Parameters: sparse_indices, sparse_topk_lens, seq_lens,
// cum_seq_lens_q) and the msa_sparse_decode_attention page (description:
// right-aligned decode positions).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/smla.h"

namespace smla {

constexpr int kHeadDim = SMLA_HEAD_DIM;   // 448 NoPE + 64 RoPE
constexpr int kSwaCols = SMLA_SWA_COLS;   // fixed SWA columns of the index table
constexpr float kLog2e = 1.4426950408889634f;

// Resolved, kernel-side copy of smla_args (strides already defaulted).
struct DecodeParams {
  int32_t sum_q, batch, H, W, dtype, num_splits;
  const void* q;
  int64_t q_stride_token;
  const void* swa;
  int64_t swa_rows, swa_stride;
  const void* comp;
  int64_t comp_rows, comp_stride;
  const int32_t* ind;
  int64_t ind_stride;
  const int32_t* topk;
  const int32_t* seq_lens;
  const int32_t* cum;
  const float* sinks;
  float bmm1, bmm2;
  const float* bmm1_dev;
  const float* bmm2_dev;
  __nv_bfloat16* out;
  float* out_lse;
  __nv_bfloat16* part_o;   // [T, H, S, 512] BF16 normalised split partials (S > 1)
  float* part_lse;   // [T, H, S] fp32 base-2 LSE of each partial (S > 1)
  int32_t* err;
  // page-table form of the compressed segment (bt == nullptr: index form)
  const int32_t* bt;       // [T, max_pages] page IDs
  int64_t bt_stride;
  int32_t page_size;
  const int32_t* hca;      // [B] window + compressed slots backing each request
  const int32_t* swa_lens; // [T] visible window per token, or nullptr (seq_lens rule)
};

struct TokenInfo {
  int b, i, q_len, pos, w_swa, n_lim;
};

// Step a1: request b(t) (binary search of cum_seq_lens_q, or t / q_len when
// the query is dense), right-aligned position pos = seq_len - q_len + i, SWA
// window w_swa = min(128, max(0, pos + 1)) (or clamp(swa_topk_lens[t], 0, 128)
// when per-row window lengths are given) and active columns
// n_lim = clamp(sparse_topk_lens[t], 0, W), in the page-table form further
// capped at max(128, hca_seq_lens[b]) (the request's backed slots).
__device__ __forceinline__ TokenInfo token_info(const DecodeParams& p, int t) {
  TokenInfo ti;
  if (p.cum != nullptr) {
    int lo = 0, hi = p.batch - 1;   // largest b with cum[b] <= t
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.cum + mid) <= t) lo = mid; else hi = mid - 1;
    }
    ti.b = lo;
    ti.i = t - __ldg(p.cum + lo);
    ti.q_len = __ldg(p.cum + lo + 1) - __ldg(p.cum + lo);
  } else {
    ti.q_len = p.sum_q / p.batch;
    ti.b = t / ti.q_len;
    ti.i = t - ti.b * ti.q_len;
  }
  ti.pos = __ldg(p.seq_lens + ti.b) - ti.q_len + ti.i;
  const int visible = p.swa_lens ? __ldg(p.swa_lens + t) : ti.pos + 1;
  ti.w_swa = min(kSwaCols, max(0, visible));
  int n = p.topk ? __ldg(p.topk + t) : p.W;
  ti.n_lim = min(max(n, 0), p.W);
  if (p.bt) ti.n_lim = min(ti.n_lim, max(kSwaCols, __ldg(p.hca + ti.b)));
  return ti;
}

// Page-table form: row of compressed slot c of token t (c < W - 128, so the
// table column is in range), or -2 when that row lies outside the pool.
__device__ __forceinline__ int paged_row(const DecodeParams& p, int t, int c) {
  const int64_t page = __ldg(p.bt + (int64_t)t * p.bt_stride + c / p.page_size);
  const int64_t row = page * p.page_size + c % p.page_size;
  return (row >= 0 && row < p.comp_rows) ? (int)row : -2;
}

// Step a2 for one column: returns the element offset of the selected row in
// its pool and sets *from_swa, or returns -1 when the slot is masked.  An
// index < -1 or past the pool is treated as masked and flagged in *err.
__device__ __forceinline__ int64_t slot_row_offset(const DecodeParams& p, const TokenInfo& ti,
                                                   int t, int j, bool* from_swa) {
  if (j >= ti.n_lim) return -1;
  bool swa = j < kSwaCols;
  int idx = (!swa && p.bt) ? paged_row(p, t, j - kSwaCols) : __ldg(p.ind + (int64_t)t * p.ind_stride + j);
  if (idx == -1) return -1;
  *from_swa = swa;
  if (swa && j >= ti.w_swa) return -1;
  int64_t rows = swa ? p.swa_rows : p.comp_rows;
  if (idx < 0 || (int64_t)idx >= rows) {
    if (p.err) atomicOr(p.err, SMLA_DEVERR_INDEX_OUT_OF_RANGE);
    return -1;
  }
  return (int64_t)idx * (swa ? p.swa_stride : p.comp_stride);
}

// Column range [c0, c1) of split s: the active columns split evenly.
__device__ __forceinline__ void split_range(int n_lim, int S, int s, int* c0, int* c1) {
  int per = (n_lim + S - 1) / S;
  *c0 = min(n_lim, s * per);
  *c1 = min(n_lim, *c0 + per);
}

__device__ __forceinline__ float load_scale(float v, const float* dev) {
  return dev ? __ldg(dev) : v;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Element decoders of the packed KV forms.
// E2M1 element values by code (OCP MX specification, FP4 E2M1: sign, two
// exponent bits with bias 1, one mantissa bit).
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  const uint32_t mag = code & 7u;
  const float v = mag < 2u ? 0.5f * (float)mag : (float)(2u + (mag & 1u)) * (float)(1u << ((mag >> 1) - 1u)) * 0.5f;
  return (code & 8u) ? -v : v;
}

__device__ __forceinline__ float e4m3_value(uint32_t byte) {
  __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(byte & 0xFFu), __NV_E4M3);
  return __half2float(*reinterpret_cast<__half*>(&hr.x));
}

}  // namespace smla
