/*
 * smla.h -- C ABI of the GB300 (sm_103a) DeepSeek-V4 sparse MLA decode library.
 *
 * The operation (FlashInfer trtllm_batch_decode_sparse_mla_dsv4, description,
 * SM100/SM103 paragraph, and its Parameters list): every flattened query token
 * t has H heads (64 or 128) of dimension 512 (448 NoPE + 64 RoPE dims; FlashInfer
 * cake_sparse_mla_sm120_dsv4_nvfp4_decode, Parameters: q).  All heads share one
 * latent KV row per selected slot.  Row t of the index table selects the slots:
 * columns 0..127 are rows of the sliding-window (SWA) pool, the remaining
 * columns are rows of the compressed pool, and -1 masks a slot (cake page,
 * Parameters: indices).  Per head h:
 *
 *   l_j  = bmm1_scale * <q[t,h,:], kv_j>
 *   O    = bmm2_scale * sum_j e^{l_j} kv_j / (sum_j e^{l_j} + e^{sinks[h]})
 *   LSE2 = log2 sum_j e^{l_j}            (base 2; cake page, Parameters: out_lse)
 *
 * O is written as BF16; LSE2 as float32.  The slots of token t are the columns
 * j < clamp(sparse_topk_lens[t], 0, W) whose index is not -1 and, for SWA
 * columns, j < min(128, pos + 1) where pos = seq_lens[b] - q_len_b + i is the
 * right-aligned position of token i of request b (msa_sparse_decode_attention
 * page, description), or j < clamp(swa_topk_lens[t], 0, 128) when per-row
 * window lengths are given.  A token with no slot gets O = 0 and LSE2 = -inf.
 *
 * The compressed columns come either from the index table (index form) or
 * from per-token page tables (page-table form, see comp_block_tables below).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers on the current CUDA device unless
 *    stated otherwise.  The caller owns every buffer, including the workspace;
 *    the library never allocates, never synchronises the device and never
 *    copies an input.  A wrong output layout is rejected, never copied into
 *    (msa_sparse_decode_attention page, Parameters: out).
 *  - Host-detectable problems return a status synchronously and launch
 *    nothing.  smla_last_error() gives a one-line reason (thread-local).
 *  - Launches are stream-ordered on the stream given; no host synchronisation.
 */
#ifndef SMLA_H
#define SMLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SMLA_ABI_VERSION 9
#define SMLA_HEAD_DIM 512      /* 448 NoPE + 64 RoPE */
#define SMLA_SWA_COLS 128      /* fixed SWA columns at the front of the index table */
#define SMLA_MAX_SPLITS 64     /* upper bound on split-K partials per token */
#define SMLA_DEFAULT_MAX_SPLITS 32

typedef enum smla_status {
  SMLA_OK = 0,
  SMLA_ERR_INVALID_ARG = 1,        /* null/misaligned pointer, bad size or stride */
  SMLA_ERR_UNSUPPORTED = 2,        /* e.g. num_heads not in {64, 128} */
  SMLA_ERR_WORKSPACE_TOO_SMALL = 3,
  SMLA_ERR_CUDA = 4                /* a CUDA runtime call or launch failed */
} smla_status;

/* Element types.  The packed forms take a BF16 query and KV pools of uint8
 * rows whose row strides (swa_row_stride, comp_row_stride) count bytes; the
 * pages (FlashInfer trtllm_batch_decode_sparse_mla_dsv4, description,
 * SM120/SM121 paragraph; cake_sparse_mla_sm120_dsv4_nvfp4_decode, Parameters:
 * kv_cache) give only their sizes, the layouts are this library's reading:
 *   SMLA_PACKED_FP8 (584 bytes, stride a multiple of 8): bytes [0, 448) the
 *     448 NoPE values in E4M3, [448, 455) seven UE8M0 exponents e (NoPE dim d
 *     scaled by 2^(e[d / 64] - 127)), byte 455 unused, [456, 584) the 64 RoPE
 *     values in BF16;
 *   SMLA_NVFP4 (384 bytes, stride a multiple of 16): bytes [0, 224) the 448
 *     NoPE values in E2M1 (dim 2i in the low nibble of byte i), [224, 252)
 *     28 E4M3 block scales (dim d scaled by scale[d / 16]), [252, 380) the 64
 *     RoPE values in BF16, [380, 384) an fp32 scale of every NoPE value.
 * The packed forms run the TCGEN05 kernel's BF16 pipeline, whose producers
 * load each selected row and write it dequantised into the BF16 tile, exactly
 * (packed FP8: E4M3 times a power of two; NVFP4: E2M1 times its E4M3 block
 * scale, the fp32 row scale applied in fp32 to the logits and to P of the
 * NoPE output dims); any other tensor-core request plans to TCGEN05, and
 * SMLA_KERNEL_CUDA_CORE runs the CUDA-core kernel, which dequantises into
 * fp32 shared memory. */
typedef enum smla_dtype {
  SMLA_BF16 = 0,                   /* bfloat16 query and KV rows */
  SMLA_E4M3 = 1,                   /* per-tensor-scaled FP8 E4M3 ("fn") query and KV rows */
  SMLA_PACKED_FP8 = 2,             /* BF16 query, 584-byte packed FP8 KV rows */
  SMLA_NVFP4 = 3                   /* BF16 query, 384-byte NVFP4 KV rows */
} smla_dtype;

/* Kernel selection (smla_args.kernel).  The tensor-core kernels run on pairs
 * of CTAs, CTA r keeping output dims [256 r, 256 r + 256) of every head; they
 * differ in how the logits are split between the CTAs.  TCGEN05: each CTA
 * gathers its dims half of every row, computes partial logits, and both CTAs
 * add the peer's partial and run the softmax of every head.
 * TCGEN05_SLOT_SPLIT (E4M3 rows; BF16 rows take TCGEN05): CTA r gathers the
 * full rows of half of every 128-slot tile, computes their complete logits,
 * and the pair exchanges per-head maxima, E4M3 P halves and the rows' other
 * output half instead of partial logits.  TCGEN05_HEAD_OWNED (E4M3 rows;
 * BF16 rows take TCGEN05): each CTA runs the softmax of half the heads and
 * sends the peer their E4M3 P; slower (a round trip per tile), kept as an
 * alternative.  TCGEN05_TOKEN_PAIRS (H = 64; H = 128 takes TCGEN05): the
 * TCGEN05 kernel with two consecutive tokens of the flattened batch (2u,
 * 2u + 1) per CTA pair, token 2u's heads in MMA rows 0-63 and token 2u + 1's
 * in rows 64-127, over the union of the two tokens' selected rows: a row both
 * tokens select (the shared SWA window of a request's consecutive tokens,
 * shared compressed rows) is gathered once, and each head's softmax takes
 * only its own token's slots.  When either token selects some row more than
 * once the unit shares nothing (each slot still counts once per selection).
 * The grid has ceil(T / 2) x S pairs.  E4M3 rows run the slot-split kernel's
 * pair form (the second token's heads fill the 128 rows its P exchange
 * already carries), which takes at most 1152 columns of each token per split
 * (the split count rises to meet that); BF16 rows the dims-split kernel's.
 * AUTO picks TCGEN05_SLOT_SPLIT for E4M3 rows (TCGEN05 when the BALANCED
 * schedule is asked for; TCGEN05_TOKEN_PAIRS for 64 heads, at most 1152
 * columns and more tokens than SM pairs: half the units, one wave fewer) and
 * TCGEN05 for BF16 rows. */
/* Work hand-out of the TCGEN05 kernel (smla_args.schedule).  GRID: one CTA
 * pair per (token, split), the split count from num_splits / max_splits.
 * BALANCED (with num_splits == 0 and max_splits == 0, W <= 2304 and T <= 14
 * pairs; else GRID): one pair per two SMs (smla_plan.clusters pairs), pair c
 * taking the c-th of equal shares of the T x W selected columns: whole
 * tokens plus the pieces of the tokens cut at its share's ends.  A piece goes
 * to the workspace with its LSE and counts itself on its token's counter
 * (the call zeroes the counters with cudaMemsetAsync before the launch); the
 * token's last piece to finish merges them into the output.  BALANCED runs a
 * separate kernel (several units per CTA pair, a warpgroup for the exchange
 * of partial logits); on a GB300 it measured slower than GRID for batches of
 * 38 to 300 tokens except just past a wave (77 tokens), so AUTO is GRID. */
typedef enum smla_schedule {
  SMLA_SCHEDULE_AUTO = 0,
  SMLA_SCHEDULE_GRID = 1,
  SMLA_SCHEDULE_BALANCED = 2
} smla_schedule;

typedef enum smla_kernel {
  SMLA_KERNEL_AUTO = 0,
  SMLA_KERNEL_CUDA_CORE = 1,          /* plain CUDA-core kernel (fp32 FMA) */
  SMLA_KERNEL_TCGEN05 = 2,            /* tcgen05 / TMEM tensor-core kernel */
  SMLA_KERNEL_TCGEN05_HEAD_OWNED = 3, /* tcgen05 kernel, softmax split between the CTAs by head */
  SMLA_KERNEL_TCGEN05_SLOT_SPLIT = 4, /* tcgen05 kernel, each CTA of a pair takes half of every tile's slots */
  SMLA_KERNEL_TCGEN05_TOKEN_PAIRS = 5 /* tcgen05 kernel, two tokens of 64 heads per CTA pair over their rows' union */
} smla_kernel;

/* Bits the kernels OR into *error_word (device-side detection, no trap). */
#define SMLA_DEVERR_INDEX_OUT_OF_RANGE 0x1  /* index < -1 or >= pool rows: slot treated as masked */
#define SMLA_DEVERR_TIMEOUT 0x2             /* a bounded on-device wait expired; outputs are invalid */
#define SMLA_DEVERR_INTERNAL 0x4            /* an internal limit was hit; outputs are invalid */

/*
 * Arguments of one decode call.  Zero-initialise and fill what you use.
 * Strides are in ELEMENTS; 0 selects the dense default given in brackets.
 */
typedef struct smla_args {
  int32_t sum_q;        /* flattened query tokens T (0 = nothing to do) */
  int32_t batch;        /* requests B >= 1 */
  int32_t num_heads;    /* H: 64 or 128 (vLLM get_padded_num_q_heads) */
  int32_t width;        /* index-table columns W >= 128 (W == 128: SWA-only layer) */
  int32_t dtype;        /* smla_dtype of q, swa_kv and compressed_kv (one type for all three; the
                           packed forms: BF16 q, packed KV rows) */

  /* query [T, H, 512]; heads and dims contiguous; token stride [H*512] */
  const void* q;
  int64_t q_stride_token;

  /* SWA pool rows [swa_rows, 512]; row stride [512], a multiple of 16 bytes (packed forms:
     rows of 584 / 384 bytes, stride in bytes [the row size], a multiple of 8 / 16) */
  const void* swa_kv;
  int64_t swa_rows;
  int64_t swa_row_stride;

  /* compressed pool rows [comp_rows, 512]; may alias swa_kv (SWA-only layers) */
  const void* compressed_kv;
  int64_t comp_rows;
  int64_t comp_row_stride;

  /* int32 index table [T, W], row stride [W]; physical row = page*page_size+offset */
  const int32_t* sparse_indices;
  int64_t indices_row_stride;

  const int32_t* sparse_topk_lens;  /* [T] int32, or NULL = W for every token */
  const int32_t* seq_lens;          /* [B] int32 original KV lengths, required */
  const int32_t* cum_seq_lens_q;    /* [B+1] int32 varlen offsets, or NULL = uniform T/B */
  const float* sinks;               /* [H] float32 sink logits (natural-log units), or NULL */

  float bmm1_scale;                 /* QK and softmax scale (FP8: scale*q_scale*kv_scale) */
  float bmm2_scale;                 /* VO scale (FP8: kv_scale) */
  const float* bmm1_scale_dev;      /* optional device float32 overriding bmm1_scale */
  const float* bmm2_scale_dev;      /* optional device float32 overriding bmm2_scale */

  void* out;                        /* [T, H, 512] BF16, contiguous, 16-byte aligned */
  float* out_lse;                   /* [T, H] float32 base-2 LSE, contiguous, or NULL */

  void* workspace;                  /* caller-owned scratch, >= smla_workspace_size() bytes, 256-byte aligned */
  size_t workspace_bytes;

  int32_t num_splits;               /* 0 = planner; else forced split count in [1, SMLA_MAX_SPLITS] */
  int32_t max_splits;               /* 0 = SMLA_DEFAULT_MAX_SPLITS; planner upper bound */
  int32_t kernel;                   /* smla_kernel */
  int32_t schedule;                 /* smla_schedule: how TCGEN05 hands out column ranges */

  int32_t* error_word;              /* optional device int32; kernels OR SMLA_DEVERR_* bits into it */

  /* Optional cudaEvent_t handles recorded on the stream immediately before
   * the decode kernel and after the last kernel of the call (the decode
   * kernel when the plan has no combine, else the combine, which is launched
   * as a programmatic dependent of the decode kernel).  For profiling. */
  void* profile_event_begin;
  void* profile_event_end;

  /* Page-table form of the compressed segment (trtllm_batch_decode_sparse_mla_dsv4
   * page, Parameters: hca_compressed_block_tables, hca_seq_lens,
   * hca_sparse_indices_format).  With comp_block_tables != NULL the index
   * table holds only the 128 SWA columns (indices_row_stride >= 128, default
   * 128) and compressed slot c of token t -- logical column 128 + c, c < W - 128
   * -- is row  comp_block_tables[t * block_table_stride + c / comp_page_size]
   * * comp_page_size + c % comp_page_size  of compressed_kv.  Request b backs
   * hca_seq_lens[b] - 128 compressed slots (the count includes the 128 window
   * slots); slots past it are never read and their table entries may hold
   * anything; sparse_topk_lens (logical columns) may cut further.  Requires
   * W - 128 <= comp_max_pages * comp_page_size.  A row at or past comp_rows
   * is treated as masked and flagged with SMLA_DEVERR_INDEX_OUT_OF_RANGE.
   * Runs of consecutive rows (pages of a multiple of 64 rows) are loaded
   * with whole-tile copies instead of row gathers. */
  const int32_t* comp_block_tables; /* [T, comp_max_pages] int32 page IDs, or NULL = index form */
  int64_t block_table_stride;       /* row stride in elements [comp_max_pages] */
  int32_t comp_max_pages;           /* page-table columns >= 1 */
  int32_t comp_page_size;           /* rows per compressed page >= 1 */
  const int32_t* hca_seq_lens;      /* [B] int32, required with comp_block_tables */

  /* Per-row visible sliding-window lengths (same page, Parameters:
   * swa_topk_lens), either form: SWA column j of token t is visible iff
   * j < clamp(swa_topk_lens[t], 0, 128); replaces the seq_lens rule.
   * NULL = the seq_lens rule. */
  const int32_t* swa_topk_lens;
} smla_args;

/* The resolved launch plan (shape-based: it never reads device memory). */
typedef struct smla_plan {
  int32_t kernel;            /* smla_kernel actually used (TCGEN05_HEAD_OWNED on BF16 rows reports TCGEN05) */
  int32_t num_splits;        /* S: column ranges per token; S > 1 adds a combine launch (1 in balanced mode) */
  int32_t ctas_per_split;    /* CTAs cooperating on one unit of work */
  int32_t grid;              /* CTAs of the main decode launch */
  int32_t threads;           /* threads per CTA of the main decode launch */
  int32_t smem_bytes;        /* dynamic shared memory per CTA */
  int32_t clusters;          /* balanced mode: P CTA pairs with equal column shares (grid = 2 P; P > 1 adds a
                                memset of the piece counters); 0: one pair per (token, split) */
  size_t workspace_bytes;    /* workspace the call needs (0 without a combine) */
} smla_plan;

/*
 * Plan a call for the device ordinal `device` (SM count and limits are read
 * from it).  Validates args like smla_decode except pointers and workspace.
 * The plan depends only on shapes, the device and num_splits/max_splits/kernel.
 */
smla_status smla_plan_decode(const smla_args* args, int device, smla_plan* plan);

/*
 * The same plan for a device with `sm_count` streaming multiprocessors,
 * without querying any device: a pure function of the shapes, the split
 * controls and sm_count (smla_plan_decode is this with the device's SM count).
 * For planning ahead of time, or for another device than the current one.
 * SMLA_ERR_INVALID_ARG if sm_count < 1 or plan is NULL; shape errors as
 * smla_plan_decode.
 */
smla_status smla_plan_decode_for_sm_count(const smla_args* args, int sm_count, smla_plan* plan);

/*
 * Opt-in validation of a call's index data on HOST copies: sparse_indices,
 * sparse_topk_lens, seq_lens, cum_seq_lens_q, comp_block_tables,
 * hca_seq_lens and swa_topk_lens must point to host memory here; q, the
 * pools, out and the other device pointers are ignored.  After the shape
 * checks of smla_decode it reports what the contract calls an error or leaves
 * undefined, by location:
 *   - a cum_seq_lens_q that does not start at 0, decreases or does not end
 *     at sum_q;
 *   - an index the kernels would read that is neither -1 nor a row of its
 *     pool;
 *   - a page-table slot the kernels would read whose row lies outside the
 *     compressed pool.
 * Lengths are clamped as the kernels clamp them (sparse_topk_lens to
 * [0, width], the window to [0, 128], the footprint by hca_seq_lens), and
 * entries the kernels never read are not checked.  Returns
 * SMLA_ERR_INVALID_ARG with the first bad entry's location in
 * smla_last_error().  smla_decode does not call it: the kernels mask and flag
 * bad indices instead (SMLA_DEVERR_INDEX_OUT_OF_RANGE).
 */
smla_status smla_validate_host(const smla_args* args);

/* Workspace bytes smla_decode will need for these args on `device`. */
smla_status smla_workspace_size(const smla_args* args, int device, size_t* bytes);

/*
 * Run the decode on `stream` (a cudaStream_t, NULL = legacy default stream) on
 * the current device.  Asynchronous; allocation- and synchronisation-free.
 * Writes out (and out_lse if given).  Returns SMLA_ERR_* without launching on
 * a host-detectable problem, SMLA_ERR_CUDA if a launch fails.  Shapes and
 * pointers are checked before any CUDA call: a missing required pointer (q,
 * swa_kv, compressed_kv, sparse_indices, seq_lens, out; hca_seq_lens with
 * comp_block_tables), a row pointer (q, swa_kv, compressed_kv, out) not
 * 16-byte aligned, or an int32 / float32 array not 4-byte aligned is
 * SMLA_ERR_INVALID_ARG.  Pointed-to values are never read on the host.
 */
smla_status smla_decode(const smla_args* args, void* stream);

/*
 * Allocation-free variant of smla_decode (the documentation pages have no
 * counterpart; it exists for callers that cannot allocate device memory, e.g.
 * an inference runtime's plugin enqueue callback that must not allocate, a
 * process whose device memory is fully reserved by another allocator, or a
 * plain C caller with no device allocator of its own).
 *
 * Same arguments and results as smla_decode, except that args->workspace and
 * args->workspace_bytes are ignored: the split-K scratch is a library-owned
 * __device__ array of SMLA_STATIC_WORKSPACE_BYTES that every GPU loading the
 * library holds until the process exits.  Calls that need more scratch than
 * that (see smla_workspace_size) return SMLA_ERR_WORKSPACE_TOO_SMALL and launch
 * nothing; lower num_splits / max_splits or use smla_decode.  The function
 * calls no allocator.
 *
 * The first call in each CUDA context (normally the device's primary context)
 * looks up the array's device address in that context and caches it; make
 * that first call before any stream capture.  Every call on a device shares
 * the one array, and each launch
 * overwrites the scratch it reads, so nothing needs clearing between calls;
 * but calls whose kernels overlap on the GPU (different streams, no ordering)
 * race on the array and give wrong results.  Order them on one stream.
 */
#define SMLA_STATIC_WORKSPACE_BYTES (64u << 20)
smla_status smla_decode_static_workspace(const smla_args* args, void* stream);

/* Static text for a status code. */
const char* smla_status_string(smla_status status);

/* One-line reason for the last non-OK status returned on this thread. */
const char* smla_last_error(void);

/* SMLA_ABI_VERSION of the loaded library. */
int smla_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SMLA_H */
