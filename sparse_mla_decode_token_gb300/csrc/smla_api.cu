// Host side of the C ABI: validation, planner and launches.
//
// Argument semantics follow the FlashInfer trtllm_batch_decode_sparse_mla_dsv4
// page (signature and Parameters).  The planner mirrors the adaptive split
// described on the msa_sparse_decode_attention page (Parameters: force_fused:
// many chunks per token at low batch, a single fused chunk at high batch) and
// the split cap of the cake_sparse_mla_sm120_dsv4_nvfp4_decode page
// (Parameters: num_splits, max_splits).  Everything here reads shapes only:
// no device memory is read, nothing is allocated and nothing synchronises.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <string>

#include "common.cuh"
#include "kernels.h"

namespace smla {
namespace {

thread_local std::string g_last_error;

smla_status fail(smla_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
smla_status fail(smla_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Bytes of a query element, and of a KV row element (the packed forms count
// their rows in bytes: row = 584 / 384 elements of one byte).
int elem_bytes(int dtype) { return dtype == SMLA_E4M3 ? 1 : 2; }
int kv_elem_bytes(int dtype) { return dtype == SMLA_BF16 ? 2 : 1; }
bool packed_dtype(int dtype) { return dtype == SMLA_PACKED_FP8 || dtype == SMLA_NVFP4; }
int64_t kv_row_elems(int dtype) { return dtype == SMLA_PACKED_FP8 ? 584 : dtype == SMLA_NVFP4 ? 384 : kHeadDim; }
int kv_stride_align(int dtype) { return dtype == SMLA_PACKED_FP8 ? 8 : 16; }

// Shape checks shared by planning and decoding.
smla_status check_shapes(const smla_args* a) {
  if (a == nullptr) return fail(SMLA_ERR_INVALID_ARG, "args is NULL");
  if (a->dtype != SMLA_BF16 && a->dtype != SMLA_E4M3 && !packed_dtype(a->dtype))
    return fail(SMLA_ERR_INVALID_ARG, "dtype %d is not an smla_dtype", a->dtype);
  if (a->num_heads != 64 && a->num_heads != 128)
    return fail(SMLA_ERR_UNSUPPORTED, "num_heads %d: only 64 or 128 heads are supported", a->num_heads);
  if (a->sum_q < 0) return fail(SMLA_ERR_INVALID_ARG, "sum_q %d < 0", a->sum_q);
  if (a->batch < 1) return fail(SMLA_ERR_INVALID_ARG, "batch %d < 1", a->batch);
  if (a->width < kSwaCols)
    return fail(SMLA_ERR_INVALID_ARG, "width %d < %d fixed SWA columns", a->width, kSwaCols);
  if (a->cum_seq_lens_q == nullptr && a->sum_q % a->batch != 0)
    return fail(SMLA_ERR_INVALID_ARG, "sum_q %d is not a multiple of batch %d (pass cum_seq_lens_q for varlen)",
                a->sum_q, a->batch);
  if (a->num_splits < 0 || a->num_splits > SMLA_MAX_SPLITS)
    return fail(SMLA_ERR_INVALID_ARG, "num_splits %d outside [0, %d]", a->num_splits, SMLA_MAX_SPLITS);
  if (a->max_splits < 0 || a->max_splits > SMLA_MAX_SPLITS)
    return fail(SMLA_ERR_INVALID_ARG, "max_splits %d outside [0, %d]", a->max_splits, SMLA_MAX_SPLITS);
  if (a->schedule < SMLA_SCHEDULE_AUTO || a->schedule > SMLA_SCHEDULE_BALANCED)
    return fail(SMLA_ERR_INVALID_ARG, "schedule %d is not an smla_schedule", a->schedule);
  if (a->kernel != SMLA_KERNEL_AUTO && a->kernel != SMLA_KERNEL_CUDA_CORE && a->kernel != SMLA_KERNEL_TCGEN05 &&
      a->kernel != SMLA_KERNEL_TCGEN05_HEAD_OWNED && a->kernel != SMLA_KERNEL_TCGEN05_SLOT_SPLIT &&
      a->kernel != SMLA_KERNEL_TCGEN05_TOKEN_PAIRS)
    return fail(SMLA_ERR_INVALID_ARG, "kernel %d is not a smla_kernel", a->kernel);
  if (a->swa_rows < 0 || a->comp_rows < 0)
    return fail(SMLA_ERR_INVALID_ARG, "negative pool row count");
  const int eb = elem_bytes(a->dtype);
  const int64_t min_qs = (int64_t)a->num_heads * kHeadDim;
  const int64_t qs = a->q_stride_token ? a->q_stride_token : min_qs;
  if (qs < min_qs || (qs * eb) % 16 != 0)
    return fail(SMLA_ERR_INVALID_ARG, "q_stride_token %lld must be >= H*512 and a multiple of 16 bytes",
                (long long)qs);
  const int64_t row = kv_row_elems(a->dtype);
  const int keb = kv_elem_bytes(a->dtype), kal = kv_stride_align(a->dtype);
  const int64_t ss = a->swa_row_stride ? a->swa_row_stride : row;
  const int64_t cs = a->comp_row_stride ? a->comp_row_stride : row;
  if (ss < row || (ss * keb) % kal != 0 || cs < row || (cs * keb) % kal != 0)
    return fail(SMLA_ERR_INVALID_ARG, "pool row strides (%lld, %lld) must be >= %lld and multiples of %d bytes",
                (long long)ss, (long long)cs, (long long)row, kal);
  const int index_cols = a->comp_block_tables ? kSwaCols : a->width;   // columns the index table holds
  const int64_t is = a->indices_row_stride ? a->indices_row_stride : index_cols;
  if (is < index_cols)
    return fail(SMLA_ERR_INVALID_ARG, "indices_row_stride %lld < %d index columns", (long long)is, index_cols);
  if (a->comp_block_tables) {
    if (a->comp_page_size < 1 || a->comp_max_pages < 1)
      return fail(SMLA_ERR_INVALID_ARG, "comp_page_size %d and comp_max_pages %d must be >= 1",
                  a->comp_page_size, a->comp_max_pages);
    const int64_t bts = a->block_table_stride ? a->block_table_stride : a->comp_max_pages;
    if (bts < a->comp_max_pages)
      return fail(SMLA_ERR_INVALID_ARG, "block_table_stride %lld < comp_max_pages %d", (long long)bts,
                  a->comp_max_pages);
    if ((int64_t)(a->width - kSwaCols) > (int64_t)a->comp_max_pages * a->comp_page_size)
      return fail(SMLA_ERR_INVALID_ARG, "width %d: %d compressed columns exceed comp_max_pages * comp_page_size = %lld",
                  a->width, a->width - kSwaCols, (long long)a->comp_max_pages * a->comp_page_size);
    if (a->comp_rows > 0x7fffffffLL)
      return fail(SMLA_ERR_UNSUPPORTED, "comp_rows %lld: page-table rows must fit in int32", (long long)a->comp_rows);
  }
  return SMLA_OK;
}

// Pointer checks of a call with sum_q > 0.  Every array the kernels read or
// write must be present where required and aligned to its access width: the
// 16-byte rows (q, pools, out) for TMA and vector accesses, every int32 or
// float32 array to 4 bytes.  A misaligned pointer would otherwise reach the
// device as a misaligned access.
smla_status check_pointers(const smla_args* a) {
  if (!a->q || !a->swa_kv || !a->compressed_kv || !a->sparse_indices || !a->seq_lens || !a->out)
    return fail(SMLA_ERR_INVALID_ARG, "q, swa_kv, compressed_kv, sparse_indices, seq_lens and out are required");
  if (a->comp_block_tables && !a->hca_seq_lens)
    return fail(SMLA_ERR_INVALID_ARG, "hca_seq_lens is required with comp_block_tables");
  if (!aligned(a->q, 16) || !aligned(a->swa_kv, 16) || !aligned(a->compressed_kv, 16) || !aligned(a->out, 16))
    return fail(SMLA_ERR_INVALID_ARG, "q, swa_kv, compressed_kv and out must be 16-byte aligned");
  const struct {
    const void* ptr;
    const char* name;
  } words[] = {
      {a->sparse_indices, "sparse_indices"}, {a->sparse_topk_lens, "sparse_topk_lens"},
      {a->seq_lens, "seq_lens"},             {a->cum_seq_lens_q, "cum_seq_lens_q"},
      {a->sinks, "sinks"},                   {a->bmm1_scale_dev, "bmm1_scale_dev"},
      {a->bmm2_scale_dev, "bmm2_scale_dev"}, {a->out_lse, "out_lse"},
      {a->error_word, "error_word"},         {a->comp_block_tables, "comp_block_tables"},
      {a->hca_seq_lens, "hca_seq_lens"},     {a->swa_topk_lens, "swa_topk_lens"},
  };
  for (const auto& w : words)
    if (w.ptr && !aligned(w.ptr, 4)) return fail(SMLA_ERR_INVALID_ARG, "%s must be 4-byte aligned", w.name);
  return SMLA_OK;
}

// Opt-in host validation of a call's index data (host copies).  It reports
// what the operation's contract calls an error -- a read index or page-table
// row outside its pool, which the kernels mask and flag -- and what it leaves
// undefined: a cum_seq_lens_q that does not start at 0, decreases or does not
// end at sum_q.  Lengths the contract clamps (sparse_topk_lens,
// swa_topk_lens, hca_seq_lens, a seq_len shorter than its query) are clamped
// here as in the kernels: token t of request b sits at position
// seq_lens[b] - q_len + i; SWA column j < 128 is read when j < n_lim and
// j < the window; compressed column j >= 128 when j < n_lim; in the
// page-table form slot c when c < n_lim - 128, n_lim being capped at
// max(128, hca_seq_lens[b]).  The first bad entry is reported by location.
smla_status validate_host(const smla_args* a) {
  smla_status st = check_shapes(a);
  if (st != SMLA_OK) return st;
  if (a->sum_q == 0) return SMLA_OK;
  if (!a->sparse_indices || !a->seq_lens)
    return fail(SMLA_ERR_INVALID_ARG, "sparse_indices and seq_lens are required");
  const bool paged = a->comp_block_tables != nullptr;
  if (paged && !a->hca_seq_lens) return fail(SMLA_ERR_INVALID_ARG, "hca_seq_lens is required with comp_block_tables");
  const int T = a->sum_q, B = a->batch, W = a->width;
  const int32_t* cum = a->cum_seq_lens_q;
  if (cum) {
    if (cum[0] != 0) return fail(SMLA_ERR_INVALID_ARG, "cum_seq_lens_q[0] = %d, not 0", cum[0]);
    for (int b = 0; b < B; ++b)
      if (cum[b + 1] < cum[b])
        return fail(SMLA_ERR_INVALID_ARG, "cum_seq_lens_q gives request %d a negative length (%d -> %d)", b,
                    cum[b], cum[b + 1]);
    if (cum[B] != T) return fail(SMLA_ERR_INVALID_ARG, "cum_seq_lens_q[%d] = %d, not sum_q = %d", B, cum[B], T);
  }
  const int64_t is = a->indices_row_stride ? a->indices_row_stride : (paged ? kSwaCols : W);
  const int64_t bts = paged ? (a->block_table_stride ? a->block_table_stride : a->comp_max_pages) : 0;
  int b = 0;
  for (int t = 0; t < T; ++t) {
    int i, q_len;
    if (cum) {
      while (cum[b + 1] <= t) ++b;         // cum[B] == T > t: ends at a request that holds t
      i = t - cum[b];
      q_len = cum[b + 1] - cum[b];
    } else {
      q_len = T / B;
      b = t / q_len;
      i = t - b * q_len;
    }
    const int64_t visible = a->swa_topk_lens ? (int64_t)a->swa_topk_lens[t] : (int64_t)a->seq_lens[b] - q_len + i + 1;
    const int w = (int)std::min<int64_t>(kSwaCols, std::max<int64_t>(0, visible));
    int n_lim = std::min(std::max(a->sparse_topk_lens ? a->sparse_topk_lens[t] : W, 0), W);
    if (paged) n_lim = std::min(n_lim, std::max(kSwaCols, a->hca_seq_lens[b]));
    const int32_t* row = a->sparse_indices + (int64_t)t * is;
    for (int j = 0; j < std::min(n_lim, w); ++j)
      if (row[j] != -1 && (row[j] < -1 || row[j] >= a->swa_rows))
        return fail(SMLA_ERR_INVALID_ARG, "token %d (request %d) column %d: index %d outside the SWA pool of %lld rows",
                    t, b, j, row[j], (long long)a->swa_rows);
    if (!paged) {
      for (int j = kSwaCols; j < n_lim; ++j)
        if (row[j] != -1 && (row[j] < -1 || row[j] >= a->comp_rows))
          return fail(SMLA_ERR_INVALID_ARG,
                      "token %d (request %d) column %d: index %d outside the compressed pool of %lld rows", t, b, j,
                      row[j], (long long)a->comp_rows);
    } else {
      const int32_t* bt = a->comp_block_tables + (int64_t)t * bts;
      for (int c = 0; c < n_lim - kSwaCols; ++c) {
        const int64_t page = bt[c / a->comp_page_size];
        const int64_t r = page * a->comp_page_size + c % a->comp_page_size;
        if (page < 0 || r >= a->comp_rows)
          return fail(SMLA_ERR_INVALID_ARG,
                      "token %d (request %d) compressed slot %d: page %lld (table column %d) gives row %lld, outside "
                      "the compressed pool of %lld rows",
                      t, b, c, (long long)page, c / a->comp_page_size, (long long)r, (long long)a->comp_rows);
      }
    }
  }
  return SMLA_OK;
}

// Kernel and schedule that SMLA_KERNEL_AUTO / SMLA_SCHEDULE_AUTO select: the
// slot-split kernel for E4M3 rows (unless the balanced schedule is asked
// for, which only the dims-split kernel runs), the dims-split kernel for BF16.
// E4M3 rows with 64 heads, at most SMLA_TC_MAX_SPLIT_COLS / 2 columns and
// more tokens than SM pairs take the slot-split kernel's token-pair form:
// half the units, so one wave fewer (measured 8-10 % faster at 128 and 300
// tokens of 640 columns, even at 152 tokens of 1152; slower when one wave
// holds every token anyway).
constexpr int kAutoSchedule = SMLA_SCHEDULE_GRID;
int auto_kernel(const smla_args* a, int sms) {
  const int schedule = a->schedule == SMLA_SCHEDULE_AUTO ? kAutoSchedule : a->schedule;
  if (a->dtype != SMLA_E4M3 || schedule == SMLA_SCHEDULE_BALANCED) return SMLA_KERNEL_TCGEN05;
  if (a->num_heads == 64 && a->width <= SMLA_TC_MAX_SPLIT_COLS / 2 && a->sum_q > sms / 2)
    return SMLA_KERNEL_TCGEN05_TOKEN_PAIRS;
  return SMLA_KERNEL_TCGEN05_SLOT_SPLIT;
}

std::atomic<int> g_sm_count[64];   // per device; 0 = not queried yet (callers may be on several threads)

smla_status sm_count(int device, int* out) {
  if (device < 0 || device >= 64) return fail(SMLA_ERR_INVALID_ARG, "device %d out of range", device);
  int n = g_sm_count[device].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return fail(SMLA_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    g_sm_count[device].store(n, std::memory_order_relaxed);
  }
  *out = n;
  return SMLA_OK;
}

// The plan as a pure function of the shapes, the split controls and the SM
// count (no device is queried).  The caller has checked the shapes.
smla_status plan_checked(const smla_args* a, int sms, smla_plan* plan) {
  if (sms < 1) return fail(SMLA_ERR_INVALID_ARG, "sm_count %d < 1", sms);
  memset(plan, 0, sizeof(*plan));
  const int max_splits = a->max_splits ? a->max_splits : SMLA_DEFAULT_MAX_SPLITS;
  // The packed KV forms run the dims-split tensor-core kernel (its BF16
  // pipeline behind dequantising producers, exact tiles), or the CUDA-core
  // kernel when that is asked for; the E4M3-only and token-pair forms do not
  // take them.
  const int kernel = packed_dtype(a->dtype)
                         ? (a->kernel == SMLA_KERNEL_CUDA_CORE ? SMLA_KERNEL_CUDA_CORE : SMLA_KERNEL_TCGEN05)
                     : a->kernel == SMLA_KERNEL_AUTO ? auto_kernel(a, sms)
                                                     : a->kernel;
  int S = a->num_splits;
  // token units of the grid: tokens, or token pairs for the token-pair kernel
  int64_t units = a->sum_q;
  if (kernel == SMLA_KERNEL_TCGEN05 || kernel == SMLA_KERNEL_TCGEN05_HEAD_OWNED ||
      kernel == SMLA_KERNEL_TCGEN05_SLOT_SPLIT || kernel == SMLA_KERNEL_TCGEN05_TOKEN_PAIRS) {
    // 2-CTA clusters: balanced mode, else one cluster per (token, split) or
    // (token pair, split).  The head-owned and slot-split forms are E4M3 only
    // (BF16 takes the dims-split kernel), the token-pair form H = 64 only
    // (H = 128 takes the dims-split kernel); all three run the grid schedule.
    const bool head_owned = kernel == SMLA_KERNEL_TCGEN05_HEAD_OWNED && a->dtype == SMLA_E4M3;
    const bool slot_split = kernel == SMLA_KERNEL_TCGEN05_SLOT_SPLIT && a->dtype == SMLA_E4M3;
    const bool pairs_of_tokens = kernel == SMLA_KERNEL_TCGEN05_TOKEN_PAIRS && a->num_heads == 64;
    // E4M3 token pairs run the slot-split kernel's pair form, whose union list
    // holds at most SMLA_TC_MAX_SPLIT_COLS entries: half of that per token
    const bool slot_pairs = pairs_of_tokens && a->dtype == SMLA_E4M3;
    const int col_cap = slot_pairs ? SMLA_TC_MAX_SPLIT_COLS / 2 : SMLA_TC_MAX_SPLIT_COLS;
    plan->kernel = head_owned        ? SMLA_KERNEL_TCGEN05_HEAD_OWNED
                   : slot_split      ? SMLA_KERNEL_TCGEN05_SLOT_SPLIT
                   : pairs_of_tokens ? SMLA_KERNEL_TCGEN05_TOKEN_PAIRS
                                     : SMLA_KERNEL_TCGEN05;
    if (pairs_of_tokens) units = (a->sum_q + 1) / 2;
    plan->ctas_per_split = 2;
    plan->threads = head_owned ? tc_head_owned_threads()
                    : (slot_split || slot_pairs) ? tc_slot_threads() : tc_grid_threads();
    plan->smem_bytes = head_owned                   ? tc_head_owned_smem_bytes()
                       : (slot_split || slot_pairs) ? tc_slot_smem_bytes()
                                                    : tc_grid_smem_bytes(a->dtype, pairs_of_tokens);
    const int s_min = (a->width + col_cap - 1) / col_cap;
    if (s_min > SMLA_MAX_SPLITS)
      return fail(SMLA_ERR_UNSUPPORTED, "width %d needs more than %d splits", a->width, SMLA_MAX_SPLITS);
    if (S != 0 && S < s_min)
      return fail(SMLA_ERR_INVALID_ARG, "num_splits %d < %d: the tcgen05 kernel takes at most %d columns per split",
                  S, s_min, col_cap);
    const int64_t pairs = sms / 2 > 0 ? sms / 2 : 1;
    const int schedule = a->schedule == SMLA_SCHEDULE_AUTO ? kAutoSchedule : a->schedule;
    if (schedule == SMLA_SCHEDULE_BALANCED && S == 0 && a->max_splits == 0 && !head_owned && !slot_split &&
        !pairs_of_tokens && !packed_dtype(a->dtype) &&
        a->width <= SMLA_TC_MAX_SPLIT_COLS && a->sum_q <= (int64_t)(SMLA_TC_MAX_UNITS - 2) * pairs) {
      // Balanced mode: P clusters, one per SM pair, take equal shares of the
      // T x W columns, each share at least 64 columns.  A share of at most
      // (SMLA_TC_MAX_UNITS - 2) W columns touches at most SMLA_TC_MAX_UNITS - 1
      // tokens, and no unit is wider than W.  Wider tables and larger batches
      // take grid mode (the latter in many waves, where a partial last wave
      // costs little).
      const int64_t total = (int64_t)a->sum_q * a->width;
      int64_t P = total / 64;
      if (P > pairs) P = pairs;
      if (P < 1) P = 1;
      plan->num_splits = 1;
      plan->clusters = (int32_t)P;
      plan->grid = (int32_t)(2 * P);
      plan->threads = tc_threads();
      plan->smem_bytes = tc_smem_bytes(a->dtype);
      if (P > 1) {
        const size_t rows = (size_t)2 * P * a->num_heads;
        // BF16 normalised pieces, their fp32 base-2 LSEs (a copy per CTA of a
        // pair), then one counter per cut token and CTA
        plan->workspace_bytes = align_up(rows * kHeadDim * sizeof(__nv_bfloat16), 256) +
                                align_up(2 * rows * sizeof(float), 256) + align_up((size_t)2 * P * sizeof(uint32_t), 256);
      }
      return SMLA_OK;
    }
    if (S == 0) {
      // as many splits as keep every cluster in one wave (a second, partial
      // wave costs a whole unit of time for a few clusters)
      int64_t want = units > 0 ? pairs / units : 1;
      // keep >= 64 columns per split (a token pair's split reads up to twice the columns)
      const int64_t by_width = ((pairs_of_tokens ? 2 : 1) * (int64_t)a->width + 63) / 64;
      if (want > by_width) want = by_width;
      if (want > max_splits) want = max_splits;
      if (want < s_min) want = s_min;
      S = (int)(want < 1 ? 1 : want);
    }
  } else {
    plan->kernel = SMLA_KERNEL_CUDA_CORE;
    plan->ctas_per_split = cuda_core_ctas_per_split(a->num_heads);
    plan->threads = cuda_core_threads();
    plan->smem_bytes = cuda_core_smem_bytes();
    const int resident = 2;                         // CTAs per SM at this smem size
    if (S == 0) {
      const int64_t units = (int64_t)a->sum_q * plan->ctas_per_split;
      const int64_t target = (int64_t)sms * resident;
      int64_t want = units > 0 ? (target + units - 1) / units : 1;
      const int64_t by_width = (a->width + 255) / 256;  // keep >= 256 columns per split
      if (want > by_width) want = by_width;
      if (want > max_splits) want = max_splits;
      S = (int)(want < 1 ? 1 : want);
    }
  }
  plan->num_splits = S;
  const int64_t grid = units * S * plan->ctas_per_split;
  if (grid > 0x7fffffff) return fail(SMLA_ERR_UNSUPPORTED, "grid of %lld CTAs is too large", (long long)grid);
  plan->grid = (int32_t)grid;
  if (S > 1) {
    const size_t rows = (size_t)a->sum_q * a->num_heads * S;
    // BF16 normalised partials, then fp32 base-2 LSEs
    plan->workspace_bytes = align_up(rows * kHeadDim * sizeof(__nv_bfloat16), 256) + align_up(rows * sizeof(float), 256);
  }
  return SMLA_OK;
}

// Plan for a device ordinal: shapes are checked before the device is queried.
smla_status make_plan(const smla_args* a, int device, smla_plan* plan) {
  smla_status st = check_shapes(a);
  if (st != SMLA_OK) return st;
  int sms = 0;
  st = sm_count(device, &sms);
  if (st != SMLA_OK) return st;
  return plan_checked(a, sms, plan);
}

}  // namespace

smla_status record_error(smla_status st, const char* msg) {
  g_last_error = msg;
  return st;
}

}  // namespace smla

using namespace smla;

extern "C" {

smla_status smla_plan_decode(const smla_args* args, int device, smla_plan* plan) {
  if (plan == nullptr) return fail(SMLA_ERR_INVALID_ARG, "plan is NULL");
  return make_plan(args, device, plan);
}

smla_status smla_plan_decode_for_sm_count(const smla_args* args, int sm_count, smla_plan* plan) {
  if (plan == nullptr) return fail(SMLA_ERR_INVALID_ARG, "plan is NULL");
  smla_status st = check_shapes(args);
  if (st != SMLA_OK) return st;
  return plan_checked(args, sm_count, plan);
}

smla_status smla_validate_host(const smla_args* args) { return validate_host(args); }

smla_status smla_workspace_size(const smla_args* args, int device, size_t* bytes) {
  if (bytes == nullptr) return fail(SMLA_ERR_INVALID_ARG, "bytes is NULL");
  smla_plan plan;
  smla_status st = make_plan(args, device, &plan);
  if (st != SMLA_OK) return st;
  *bytes = plan.workspace_bytes;
  return SMLA_OK;
}

smla_status smla_decode(const smla_args* a, void* stream_ptr) {
  // host-only checks (shapes, then pointers) come before any CUDA call
  smla_status st = check_shapes(a);
  if (st != SMLA_OK) return st;
  if (a->sum_q == 0) return SMLA_OK;   // empty batch: nothing to launch
  st = check_pointers(a);
  if (st != SMLA_OK) return st;
  int device = 0;
  cudaError_t ce = cudaGetDevice(&device);
  if (ce != cudaSuccess) return fail(SMLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
  int sms = 0;
  st = sm_count(device, &sms);
  if (st != SMLA_OK) return st;
  smla_plan plan;
  st = plan_checked(a, sms, &plan);
  if (st != SMLA_OK) return st;
  if (plan.workspace_bytes > 0) {
    if (a->workspace == nullptr || a->workspace_bytes < plan.workspace_bytes)
      return fail(SMLA_ERR_WORKSPACE_TOO_SMALL, "workspace of %zu bytes given, %zu needed",
                  a->workspace ? a->workspace_bytes : (size_t)0, plan.workspace_bytes);
    if (!aligned(a->workspace, 256)) return fail(SMLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  }

  DecodeParams p;
  memset(&p, 0, sizeof(p));
  p.sum_q = a->sum_q;
  p.batch = a->batch;
  p.H = a->num_heads;
  p.W = a->width;
  p.dtype = a->dtype;
  p.num_splits = plan.num_splits;
  p.q = a->q;
  p.q_stride_token = a->q_stride_token ? a->q_stride_token : (int64_t)a->num_heads * kHeadDim;
  p.swa = a->swa_kv;
  p.swa_rows = a->swa_rows;
  p.swa_stride = a->swa_row_stride ? a->swa_row_stride : kv_row_elems(a->dtype);
  p.comp = a->compressed_kv;
  p.comp_rows = a->comp_rows;
  p.comp_stride = a->comp_row_stride ? a->comp_row_stride : kv_row_elems(a->dtype);
  p.ind = a->sparse_indices;
  p.ind_stride = a->indices_row_stride ? a->indices_row_stride : (a->comp_block_tables ? kSwaCols : a->width);
  if (a->comp_block_tables) {
    p.bt = a->comp_block_tables;
    p.bt_stride = a->block_table_stride ? a->block_table_stride : a->comp_max_pages;
    p.page_size = a->comp_page_size;
    p.hca = a->hca_seq_lens;
  }
  p.swa_lens = a->swa_topk_lens;
  p.topk = a->sparse_topk_lens;
  p.seq_lens = a->seq_lens;
  p.cum = a->cum_seq_lens_q;
  p.sinks = a->sinks;
  p.bmm1 = a->bmm1_scale;
  p.bmm2 = a->bmm2_scale;
  p.bmm1_dev = a->bmm1_scale_dev;
  p.bmm2_dev = a->bmm2_scale_dev;
  p.out = reinterpret_cast<__nv_bfloat16*>(a->out);
  p.out_lse = a->out_lse;
  p.err = a->error_word;
  if (plan.num_splits > 1) {
    const size_t rows = (size_t)a->sum_q * a->num_heads * plan.num_splits;
    p.part_o = reinterpret_cast<__nv_bfloat16*>(a->workspace);
    p.part_lse = reinterpret_cast<float*>(reinterpret_cast<char*>(a->workspace) +
                                          align_up(rows * kHeadDim * sizeof(__nv_bfloat16), 256));
  }
  __nv_bfloat16* piece_o = nullptr;
  float* piece_lse = nullptr;
  uint32_t* piece_cnt = nullptr;
  if (plan.clusters > 1) {
    const size_t rows = (size_t)2 * plan.clusters * a->num_heads;
    char* w = reinterpret_cast<char*>(a->workspace);
    piece_o = reinterpret_cast<__nv_bfloat16*>(w);
    w += align_up(rows * kHeadDim * sizeof(__nv_bfloat16), 256);
    piece_lse = reinterpret_cast<float*>(w);
    w += align_up(2 * rows * sizeof(float), 256);
    piece_cnt = reinterpret_cast<uint32_t*>(w);
  }

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
  if (a->profile_event_begin) {
    ce = cudaEventRecord(reinterpret_cast<cudaEvent_t>(a->profile_event_begin), stream);
    if (ce != cudaSuccess) return fail(SMLA_ERR_CUDA, "cudaEventRecord: %s", cudaGetErrorString(ce));
  }
  if (piece_cnt != nullptr) {
    // the pieces of each cut token count themselves here: zero before the launch
    ce = cudaMemsetAsync(piece_cnt, 0, (size_t)2 * plan.clusters * sizeof(uint32_t), stream);
    if (ce != cudaSuccess) return fail(SMLA_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(ce));
  }
  if (plan.kernel == SMLA_KERNEL_TCGEN05_HEAD_OWNED)
    ce = launch_decode_tc_head_owned(p, plan.grid, stream);
  else if (plan.kernel == SMLA_KERNEL_TCGEN05_SLOT_SPLIT)
    ce = launch_decode_tc_slot(p, plan.grid, false, stream);
  else if (plan.kernel == SMLA_KERNEL_TCGEN05_TOKEN_PAIRS && a->dtype == SMLA_E4M3)
    ce = launch_decode_tc_slot(p, plan.grid, true, stream);
  else if (plan.kernel == SMLA_KERNEL_TCGEN05 && plan.clusters > 0)
    ce = launch_decode_tc(p, plan.grid, plan.clusters, piece_o, piece_lse, piece_cnt, stream);
  else if (plan.kernel == SMLA_KERNEL_TCGEN05 || plan.kernel == SMLA_KERNEL_TCGEN05_TOKEN_PAIRS)
    ce = launch_decode_tc_grid(p, plan.grid, plan.kernel == SMLA_KERNEL_TCGEN05_TOKEN_PAIRS, stream);
  else
    ce = launch_decode_cuda_core(p, plan.grid, stream);
  if (ce != cudaSuccess) return fail(SMLA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(ce));
  if (plan.num_splits > 1) {
    ce = launch_combine(p, stream);
    if (ce != cudaSuccess) return fail(SMLA_ERR_CUDA, "combine launch: %s", cudaGetErrorString(ce));
  }
  if (a->profile_event_end) {
    ce = cudaEventRecord(reinterpret_cast<cudaEvent_t>(a->profile_event_end), stream);
    if (ce != cudaSuccess) return fail(SMLA_ERR_CUDA, "cudaEventRecord: %s", cudaGetErrorString(ce));
  }
  return SMLA_OK;
}

const char* smla_status_string(smla_status s) {
  switch (s) {
    case SMLA_OK: return "SMLA_OK";
    case SMLA_ERR_INVALID_ARG: return "SMLA_ERR_INVALID_ARG";
    case SMLA_ERR_UNSUPPORTED: return "SMLA_ERR_UNSUPPORTED";
    case SMLA_ERR_WORKSPACE_TOO_SMALL: return "SMLA_ERR_WORKSPACE_TOO_SMALL";
    case SMLA_ERR_CUDA: return "SMLA_ERR_CUDA";
  }
  return "SMLA_ERR_UNKNOWN";
}

const char* smla_last_error(void) { return g_last_error.c_str(); }

int smla_abi_version(void) { return SMLA_ABI_VERSION; }

}  // extern "C"
