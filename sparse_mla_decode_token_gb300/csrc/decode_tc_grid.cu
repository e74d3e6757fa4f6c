// tcgen05 / TMEM sparse MLA decode kernel for sm_103a, grid schedule.
//
// Work unit: one (token, split) runs on a cluster of two CTAs (the balanced
// schedule's kernel, decode_tcgen05.cu, works through several units per
// cluster instead).  CTA r of the pair owns output dims [256 r, 256 r + 256):
// an fp32 accumulator for 128 heads x 512 dims is 256 KB, the whole tensor
// memory of one SM, so the output is split across the pair.  Per tile of up to N selected slots (N = 64 for E4M3,
// 32 for BF16):
//
//   set-up (all warps)  stage the split's index columns and compact the valid
//                       slots (per-warp ballots and scans) into a list: SWA
//                       slots, then compressed slots; tiles are runs of N list
//                       entries of one pool (masked slots are never loaded)
//   producer warps 0-3  the pair's half of every selected row (256 dims) with
//                       TMA tile::gather4 (four rows of 128 bytes per request)
//                       into a 128-byte-swizzled, UMMA-canonical shared-memory
//                       tile of a 7-stage (E4M3) or 6-stage (BF16) ring; a
//                       warp's TMA requests are served one after another, so a
//                       tile's 32 requests are spread over the two warps of
//                       one of two groups taking alternate tiles; a tile of N
//                       consecutive rows is one box copy per 128-byte block
//   QK warps 4-6        S_r = Q_r K_r^T   (M = 128 heads, N slots, K = 256 dims)
//                       into one of three TMEM S buffers, warp 4 + b issuing
//                       the tiles of buffer b; warp 4 also allocates and
//                       frees TMEM
//   PV warp 7           O_r += P V_r      (M = 128 heads, N = 256 dims, K = N slots,
//                       P read from TMEM); a separate issuer so that no QK
//                       waits behind a PV that waits for the softmax
//   softmax warps 8-15  two warpgroups taking whole tiles in turn (warpgroup
//                       g takes tiles j with j % 2 == g), one thread per head:
//                       read S_r from TMEM, push it to the peer CTA with
//                       st.async (completing bytes on the peer's mbarrier) as
//                       24-bit floats (four values in three words), add
//                       the peer's partial (S = S_0 + S_1; each CTA adds its
//                       own exact half), settle the running reference maximum m(j) from
//                       m(j-1) (handed over by the other warpgroup through
//                       shared memory), exponentials in base 2 with lazy
//                       rescaling of O, write P (BF16 or E4M3) into TMEM;
//                       finally normalise O and store it (the BF16 output or
//                       split partial rows, staged through shared memory for
//                       256-byte row-segment stores) plus the LSE.  Each
//                       warpgroup pushes its next tile's partial S before its
//                       exponentials; one warpgroup's exponentials overlap the
//                       other's loads and exchange.
//
// Two variants of the same pipeline: kPair (H = 64) runs two tokens per unit
// over the union of their selected rows, their heads in MMA rows 0-63 and
// 64-127 (see Cfg); kPack (packed FP8 and NVFP4 rows) replaces the TMA
// gathers by producers that load the packed rows and write them dequantised
// into the BF16 tiles (see packed_fp8_dims64 / nvfp4_dims64).
//
// The operation follows the FlashInfer trtllm_batch_decode_sparse_mla_dsv4 page
// (description, SM100/SM103 paragraph; Parameters); the base-2 LSE, the sink in
// the normaliser and the split partials follow the cake_sparse_mla_sm120 page
// (Parameters: out_lse, attn_sink, mid_out / mid_lse).
//
// Every mbarrier wait is bounded (2 s); on expiry the CTA raises an abort flag,
// ORs SMLA_DEVERR_TIMEOUT into the error word, lets every role leave its loop,
// waits for its own copies and MMAs, frees its TMEM and returns.  No role
// waits on an unbounded hardware barrier inside its loop.
#include <cuda.h>
#include <cuda_fp4.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kMaxN = 64;            // largest tile (slots per tile)
constexpr int kHalfDims = 256;       // output dims per CTA
constexpr int kProducerWarps = 4;    // TMA gathers
constexpr int kProducerGroups = 2;   // tiles alternate between two groups of two warps that share each tile
constexpr int kMmaWarp = kProducerWarps;        // first QK issuer; allocates and frees TMEM
constexpr int kQkWarps = 3;                     // QK issuers: warp kMmaWarp + i issues the tiles k with k % 3 == i
constexpr int kPvWarp = kMmaWarp + kQkWarps;    // PV issue
constexpr int kSoftmaxWarp0 = kPvWarp + 1;
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = (kSoftmaxWarp0 + kSoftmaxWarps) * 32;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCols = SMLA_TC_MAX_SPLIT_COLS;
constexpr int kMaxChunks = kMaxCols / 32;                 // 32-column chunks of a staged index row
constexpr int kChunksPerWarp = (kMaxChunks + kWarps - 1) / kWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;        // O: 256 fp32 columns
constexpr uint32_t kSCol = 256;      // S: three buffers of N fp32 columns, then P: two buffers of 16 columns
constexpr int kSBufs = 3;
static_assert(kQkWarps == kSBufs, "one QK issuer per S buffer");
constexpr float kRescaleThreshold = 8.f;   // log2 units: P stays <= 2^8
constexpr int kExactRefTiles = 8;          // E4M3 P: chains of at most this many tiles follow the exact maximum
constexpr int kMaxStages = 8;

struct TcSmall {
  uint64_t kv_full[kMaxStages];
  uint64_t kv_empty[kMaxStages];
  uint64_t s_full[kSBufs], s_empty[kSBufs], p_full[2], p_empty[2];
  uint64_t xin_full[2], xout_free[2];
  uint64_t m_ready[2];                   // m_buf[g] written by warpgroup g's four warps
  uint64_t lsum_full;
  uint64_t o_full;                       // every PV done (committed by the PV warp)
  uint64_t qk0_done;                     // the CTA's first QK done (single use)
  uint64_t qk_done;                      // every QK done (one commit per QK warp)
  float m_end[2][128];                   // final reference maximum per [warpgroup][head]
  float m_buf[2][128];                   // reference maximum after the last tile of warpgroup g
  float lsum[2][128];                    // [warpgroup][head]
  int32_t chunk_off[kMaxChunks];        // compacted-slot count of each 32-column chunk, then its offset
  int32_t nswa;                          // valid slots in the SWA columns of the split (token pair: of the union)
  int32_t nvalid;                        // valid slots of the split (token pair: of the union)
  // token pairs only: token B's chunk counts, the chunk counts of B's rows
  // that token A does not select, and the per-token list sizes
  int32_t chunk_off_b[kMaxChunks];
  int32_t only_b_chunk[kMaxChunks];
  int32_t nswa_a, nswa_b, n_a, n_b, only_b_swa, dup;
  float rscale[kMaxStages][kMaxN];       // NVFP4 rows: each stage row's fp32 NoPE scale
  uint32_t tmem_base;
  int32_t abort_flag;
};

// kPair: a unit holds two tokens of 64 heads each (rows 0-63 of the 128-row
// MMA tile token A, rows 64-127 token B) over the union of their selected
// rows: the compacted list can hold both tokens' columns, and a per-tile
// membership mask tells each row which list entries are its own.
template <bool kFp8, bool kPair = false>
struct Cfg {
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kN = kFp8 ? 64 : 32;                    // slots per tile
  static constexpr int kRegions = kHalfDims * kElem / 128;     // 128-byte column blocks per half row
  static constexpr int kChunks = kHalfDims * kElem / 16;       // 16-byte chunks per half row
  static constexpr int kStages = kFp8 ? 7 : 6;                 // KV ring (FP8: the smaller exchange buffers make room for a 7th)
  static constexpr int kKStep = 32 / kElem;                    // MMA K per instruction
  static constexpr int kK1 = kHalfDims / kKStep;               // QK K steps
  static constexpr int kK2 = kN / kKStep;                      // PV K steps
  static constexpr int kPCols = kN * kElem / 4;                // TMEM columns of one P buffer
  static constexpr uint32_t kPCol = kSCol + kSBufs * kN;
  static constexpr int kRegionQ = 128 * 128;                   // 128 rows x 128 B
  static constexpr int kRegionKV = kN * 128;                   // N rows x 128 B
  static constexpr int kQBytes = kRegions * kRegionQ;
  static constexpr int kStageBytes = kRegions * kRegionKV;
  static constexpr int kXBytes = 128 * kN * 3;                 // one exchange buffer: 128 rows of N 24-bit logits
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQBytes;
  static constexpr int kOffX = kOffKV + kStages * kStageBytes;
  static constexpr int kIdxCap = (kPair ? 2 : 1) * kMaxCols;  // list entries (a token pair: the union)
  static constexpr int kMaxTiles = kIdxCap / kN + 2;           // the SWA and compressed runs may each end in a partial tile
  static constexpr int kOffIdx = kOffX + 2 * kXBytes;
  static constexpr int kOffMask = kOffIdx + kIdxCap * 4;       // token pairs: uint64 masks [2][kMaxTiles]
  static constexpr int kOffSmall = kOffMask + (kPair ? 2 * kMaxTiles * 8 : 0);
  static constexpr int kSmemBytes = kOffSmall + (int)sizeof(TcSmall) + 1024;   // + alignment slack
  // token-pair set-up scratch, in the KV stages before the first gather: an
  // open-addressing hash of token A's rows (keys, then A's list indices),
  // each token's compacted list, one membership byte per union entry, and
  // one "B selects it too" byte per entry of A's list
  static constexpr int kHashSlots = 4096;                      // > kMaxCols (A's keys): probing always ends
  static constexpr int kScrVals = kHashSlots * 4;
  static constexpr int kScrListA = 2 * kHashSlots * 4;
  static constexpr int kScrListB = kScrListA + kMaxCols * 4;
  static constexpr int kScrMemb = kScrListB + kMaxCols * 4;
  static constexpr int kScrShared = kScrMemb + kIdxCap;
  static constexpr int kScrEnd = kScrShared + kMaxCols;
  static_assert(!kPair || kScrEnd <= kStages * kStageBytes, "token-pair scratch fits in the KV stages");
  static_assert(kScrVals % 16 == 0 && kScrListA % 16 == 0 && kScrShared % 16 == 0,
                "scratch arrays start on 16-byte boundaries");
  static_assert(kHashSlots > kMaxCols && (kHashSlots & (kHashSlots - 1)) == 0, "hash table size");
  static_assert(kStages <= kMaxStages, "barrier arrays");
  static_assert(kStages >= 3, "PV lags QK by two tiles: a third stage keeps the producer going");
  static_assert(kN <= kMaxN, "row lists");
  static_assert(kPCols == 16, "P buffer width");
  static_assert(kN % 32 == 0, "tiles are whole 32-column groups");
  static_assert(kPCol + 2 * kPCols <= kTmemCols, "tensor memory budget");
  static_assert(kStages * kStageBytes >= 2 * 128 * 256, "BF16 partial staging fits in the KV stages");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Kernel parameters: the shared decode parameters plus two TMA descriptors per
// KV pool ([rows, 512] with the pool's row stride; 128-byte swizzle): box =
// 128 bytes x 1 row for tile::gather4, and 128 bytes x N rows for whole-tile
// copies of N consecutive rows.
struct TcParams {
  CUtensorMap tm_swa;
  CUtensorMap tm_comp;
  CUtensorMap tm_swa_run;
  CUtensorMap tm_comp_run;
  DecodeParams p;
};

// Packed FP8 rows (kPack = SMLA_PACKED_FP8) run the BF16 pipeline: the
// producers load each selected row's bytes with plain loads (a 584-byte row
// pitch is no TMA stride) and write its 256 dims of this CTA's output half as
// BF16 into the stage, in the layout a TMA gather leaves.  Dims [d, d + 64)
// of a row (d a multiple of 64) as 32 BF16 pairs: the NoPE E4M3 values times
// 2^(e - 127) of their 64-dim block (exact in BF16), or the 64 RoPE values
// (BF16 bits copied).
__device__ __forceinline__ void packed_fp8_dims64(const unsigned char* row, int d, uint32_t (&out)[32]) {
  if (d >= 448) {                                    // RoPE: BF16 as stored, 8-byte aligned
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint2 x = __ldg(reinterpret_cast<const uint2*>(row + 456) + i);
      out[2 * i] = x.x;
      out[2 * i + 1] = x.y;
    }
    return;
  }
  const float scale = ldexpf(1.0f, (int)__ldg(row + 448 + d / 64) - 127);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint2 x = __ldg(reinterpret_cast<const uint2*>(row + d) + i);
    const uint32_t w[2] = {x.x, x.y};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)((w[h] >> (16 * k)) & 0xFFFFu), __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<__half2*>(&hr));
        out[4 * i + 2 * h + k] = pack_bf16x2(f.x * scale, f.y * scale);
      }
    }
  }
}

// NVFP4 rows (kPack = SMLA_NVFP4) take the same path with exact tiles: dims
// [d, d + 64) as 32 BF16 pairs, the NoPE E2M1 values times the E4M3 scale of
// their 16-dim block (a product of two 8-bit codes, exact in BF16), or the 64
// RoPE values.  The row's fp32 scale g multiplies the NoPE dims only, so it
// stays out of the tile: each CTA applies it to its partial logits in fp32
// (CTA 1 keeps its NoPE and RoPE dims in separate accumulators) and to the P
// of its NoPE output dims.
__device__ __forceinline__ void nvfp4_dims64(const unsigned char* row, int d, uint32_t (&out)[32]) {
  if (d >= 448) {                                    // RoPE: BF16 as stored, 4-byte aligned
#pragma unroll
    for (int i = 0; i < 32; ++i) out[i] = __ldg(reinterpret_cast<const uint32_t*>(row + 252) + i);
    return;
  }
  const uint32_t sc = __ldg(reinterpret_cast<const uint32_t*>(row + 224 + d / 16));   // four block scales
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(row + d / 2) + i);   // 32 dims, low nibble first
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int b = 0; b < 2; ++b) {                    // the two 16-dim blocks of these 32 dims
      // E2M1 pairs converted by the hardware, times the block scale in fp16:
      // at most six significant bits and within [2^-10, 2688], so exact
      const __half2 bs = __float2half2_rn(e4m3_value((sc >> (8 * (2 * i + b))) & 0xFFu));
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t byte = (w[2 * b + (k >> 2)] >> (8 * (k & 3))) & 0xFFu;
        __half2_raw hr = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)byte, __NV_E2M1);
        const float2 f = __half22float2(__hmul2(*reinterpret_cast<__half2*>(&hr), bs));
        out[16 * i + 8 * b + k] = pack_bf16x2(f.x, f.y);
      }
    }
  }
}

// kPartial: the launch has num_splits > 1 and writes BF16 split partials; its
// epilogue stages the partial rows in shared memory for contiguous stores (a
// separate instantiation, so that the single-split code is compiled alone).
// kPair: H = 64 and a unit is (token pair, split), see Cfg.
// kPack: 0, or SMLA_PACKED_FP8 / SMLA_NVFP4 (BF16 pipeline: kFp8 false, kPair false).
template <bool kFp8, bool kPartial, bool kPair, int kPack>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ TcParams P) {
  static_assert(kPack == 0 || (!kFp8 && !kPair), "packed rows run the BF16 single-token pipeline");
  constexpr bool kNv = kPack == SMLA_NVFP4;
  using C = Cfg<kFp8, kPair>;
  // NVFP4: CTA 1's RoPE logits (three buffers) and the P of the NoPE output
  // dims (P times each slot's row scale; two buffers) after the P buffers
  constexpr uint32_t kSRCol = C::kPCol + 2 * C::kPCols;
  constexpr uint32_t kPGCol = kSRCol + kSBufs * C::kN;
  static_assert(!kNv || kPGCol + 2 * C::kPCols <= kTmemCols, "tensor memory budget (NVFP4)");
  const DecodeParams& p = P.p;
  constexpr int kN = C::kN;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_addr - raw_addr);
  TcSmall& sm = *reinterpret_cast<TcSmall*>(base + C::kOffSmall);
  int32_t* idx_s = reinterpret_cast<int32_t*>(base + C::kOffIdx);
  uint64_t* mask_a = reinterpret_cast<uint64_t*>(base + C::kOffMask);   // token pairs: [tile] rows of token A
  uint64_t* mask_b = mask_a + C::kMaxTiles;                             // token pairs: [tile] rows of token B
  const uint32_t q_addr = base_addr + C::kOffQ;
  const uint32_t kv_addr = base_addr + C::kOffKV;
  const uint32_t x_addr = base_addr + C::kOffX;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const int S = p.num_splits;
  const int unit = blockIdx.x >> 1;
  const int s = unit % S;
  const int t = kPair ? 2 * (unit / S) : unit / S;   // the token (a pair: token A; token B is t + 1)
  const bool has_b = kPair && t + 1 < p.sum_q;       // an odd token count leaves the last pair one token
  const int H = p.H;
  const int rows_used = kPair ? (has_b ? 128 : 64) : H;   // MMA rows that carry a head
  // Column range of this split, from the table width only (so that the index
  // loads need not wait for any device value): [c0, c0 + ceil(W / S)); in the
  // page-table form rounded up to whole 64-slot runs, so that every full tile
  // of compressed slots lies on one page when pages hold a multiple of 64 rows.
  int per_split = (p.W + S - 1) / S;
  if (p.bt) per_split = (per_split + kMaxN - 1) / kMaxN * kMaxN;
  const int c0 = min(p.W, s * per_split);
  int c1 = min(p.W, c0 + per_split);
  if (c1 - c0 > kMaxCols) {           // the planner prevents this; never read past the staging buffer
    if (p.err && tid == 0) atomicOr(p.err, SMLA_DEVERR_INTERNAL);
    c1 = c0 + kMaxCols;
  }

  auto bar = [&](const uint64_t& b) { return smem_addr(&b); };

  // ---------------------------------------------------------------- set-up
  // Q first: its copies need nothing but (t, rank)
  if constexpr (!kPair) {
    const unsigned char* qb = reinterpret_cast<const unsigned char*>(p.q) +
                              ((int64_t)t * p.q_stride_token + (int64_t)rank * kHalfDims) * C::kElem;
    for (int c = tid; c < H * C::kChunks; c += kThreads) {
      const int h = c / C::kChunks, cc = c % C::kChunks;
      cp_async_16(q_addr + (cc >> 3) * C::kRegionQ + sw128_offset(h, cc & 7),
                  qb + (int64_t)h * kHeadDim * C::kElem + cc * 16);
    }
  } else {
    // MMA row h: head h & 63 of token t + (h >> 6)
    for (int c = tid; c < rows_used * C::kChunks; c += kThreads) {
      const int h = c / C::kChunks, cc = c % C::kChunks;
      const unsigned char* qb = reinterpret_cast<const unsigned char*>(p.q) +
                                ((int64_t)(t + (h >> 6)) * p.q_stride_token + (int64_t)(h & 63) * kHeadDim +
                                 (int64_t)rank * kHalfDims) * C::kElem;
      cp_async_16(q_addr + (cc >> 3) * C::kRegionQ + sw128_offset(h, cc & 7), qb + cc * 16);
    }
  }
  // the split's index columns, in flight together with the token metadata loads
  const int nchunks = (c1 - c0 + 31) / 32;
  auto load_cols = [&](int tok, int32_t (&r)[kChunksPerWarp]) {
    const int32_t* irow = p.ind + (int64_t)tok * p.ind_stride;
    if (p.bt == nullptr) {             // index form (a loop of its own: the FP8 code keeps its registers)
#pragma unroll
      for (int q = 0; q < kChunksPerWarp; ++q) {
        const int col = c0 + (warp + q * kWarps) * 32 + lane;
        r[q] = (col < c1) ? __ldg(irow + col) : -1;
      }
    } else {                           // page-table form: compressed rows from the page table
#pragma unroll
      for (int q = 0; q < kChunksPerWarp; ++q) {
        const int col = c0 + (warp + q * kWarps) * 32 + lane;
        r[q] = -1;
        if (col < c1) r[q] = col >= kSwaCols ? paged_row(p, tok, col - kSwaCols) : __ldg(irow + col);
      }
    }
  };
  int32_t rv[kChunksPerWarp];
  int32_t rvb[kChunksPerWarp];         // token pairs: token B's columns (unused otherwise)
  load_cols(t, rv);
  if (has_b) load_cols(t + 1, rvb);
  const TokenInfo ti = token_info(p, t);
  const int c1a = min(c1, max(c0, ti.n_lim));    // active columns of the split
  int c1b = c0, w_swa_b = 0;
  if (has_b) {
    const TokenInfo tib = token_info(p, t + 1);
    c1b = min(c1, max(c0, tib.n_lim));
    w_swa_b = tib.w_swa;
  }
  // a2 for one loaded column: the row, or -1 when the slot is masked (an
  // index < -1 or past the pool is masked and flagged)
  auto check_slot = [&](int idx, int col, int c1t, int w_swa) -> int {
    if (col >= c1t) return -1;
    const bool swa = col < kSwaCols;
    if (idx == -1 || (swa && col >= w_swa)) return -1;
    const int64_t nrows = swa ? p.swa_rows : p.comp_rows;
    if (idx < 0 || (int64_t)idx >= nrows) {
      if (p.err && rank == 0) atomicOr(p.err, SMLA_DEVERR_INDEX_OUT_OF_RANGE);
      return -1;
    }
    return idx;
  };
  // per-chunk valid counts of this warp's chunks (k = warp + q * kWarps) and
  // the valid SWA slots, for one token's loaded columns (valid rows stay in r)
  auto count_chunks = [&](int32_t (&r)[kChunksPerWarp], int c1t, int w_swa, int32_t* cnt, int32_t* nswa_out) {
#pragma unroll
    for (int q = 0; q < kChunksPerWarp; ++q) {
      const int k = warp + q * kWarps;
      if (k < nchunks) {
        const int col = c0 + k * 32 + lane;
        r[q] = check_slot(r[q], col, c1t, w_swa);
        const unsigned ball = __ballot_sync(0xffffffffu, r[q] >= 0);
        const unsigned ball_swa = __ballot_sync(0xffffffffu, r[q] >= 0 && col < kSwaCols);
        if (lane == 0) {
          cnt[k] = __popc(ball);
          if (ball_swa) atomicAdd(nswa_out, __popc(ball_swa));
        }
      }
    }
  };
  // every warp scans the chunk counts itself (at most kMaxChunks = 72, three
  // shuffle scans), which saves a serialised scan and a block barrier:
  // chunk_base[q] = entries before chunk warp + q * kWarps; returns the total
  auto scan_chunks = [&](const int32_t* cnt, int nch, int (&chunk_base)[kChunksPerWarp]) -> int {
    int carry = 0;
#pragma unroll
    for (int q = 0; q < kChunksPerWarp; ++q) chunk_base[q] = 0;
    for (int base0 = 0; base0 < nch; base0 += 32) {
      const int k = base0 + lane;
      const int v = k < nch ? cnt[k] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      // exclusive prefix of this warp's chunks k = warp + q * kWarps in this group of 32
#pragma unroll
      for (int q = 0; q < kChunksPerWarp; ++q) {
        const int kq = warp + q * kWarps;
        const int excl = __shfl_sync(0xffffffffu, incl - v, kq & 31);
        if ((kq >> 5) == (base0 >> 5)) chunk_base[q] = carry + excl;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    return carry;
  };
  auto init_barriers = [&]() {
    for (int i = 0; i < C::kStages; ++i) {
      // TMA: one arrival with the byte count; packed rows: one per warp of the producer group
      mbar_init(bar(sm.kv_full[i]), kPack ? kProducerWarps / kProducerGroups : 1);
      mbar_init(bar(sm.kv_empty[i]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(sm.p_full[b]), kSoftmaxWarps / 2);
      mbar_init(bar(sm.p_empty[b]), 1);
      mbar_init(bar(sm.xin_full[b]), 1);
      mbar_init(bar(sm.xout_free[b]), kSoftmaxWarps / 2);
      mbar_init(bar(sm.m_ready[b]), kSoftmaxWarps / 2);
    }
    mbar_init(bar(sm.lsum_full), kSoftmaxWarps);
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(bar(sm.s_full[b]), 1);
      mbar_init(bar(sm.s_empty[b]), kSoftmaxWarps / 2);
    }
    mbar_init(bar(sm.o_full), 1);
    mbar_init(bar(sm.qk0_done), 1);
    mbar_init(bar(sm.qk_done), kQkWarps);
    sm.abort_flag = 0;
    sm.nswa = 0;
  };
  auto zero_kv_stages = [&]() {
    // rows past a tile's slot count then hold finite data
    const uint4 z = make_uint4(0, 0, 0, 0);
    uint4* zp = reinterpret_cast<uint4*>(base + C::kOffKV);
    const int zn = C::kStages * C::kStageBytes / 16;
    for (int i = tid; i < zn; i += kThreads) zp[i] = z;
  };
  auto zero_q_rows = [&](int from) {   // Q rows [from, 128) carry no head
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int kb = 0; kb < C::kRegions; ++kb) {
      uint4* qz = reinterpret_cast<uint4*>(base + C::kOffQ + kb * C::kRegionQ + from * 128);
      for (int i = tid; i < (128 - from) * 8; i += kThreads) qz[i] = z;
    }
  };
  if constexpr (!kPair) {
    if (H < 128) zero_q_rows(H);
    if constexpr (kNv) {                 // rows past a tile's count meet P = 0: their scale must be finite
      float* rs = &sm.rscale[0][0];
      for (int i = tid; i < kMaxStages * kMaxN; i += kThreads) rs[i] = 0.f;
    }
    if (tid == 0) {
      init_barriers();
      fence_mbar_init_cluster();
    }
    __syncthreads();
    // a2: compaction of the split's columns [c0, c1) into idx_s: valid SWA
    // slots first, then valid compressed slots, each in column order
    count_chunks(rv, c1a, ti.w_swa, sm.chunk_off, &sm.nswa);
    __syncthreads();
    int chunk_base[kChunksPerWarp];
    const int total = scan_chunks(sm.chunk_off, nchunks, chunk_base);
    if (warp == 0 && lane == 0) sm.nvalid = total;
#pragma unroll
    for (int q = 0; q < kChunksPerWarp; ++q) {
      const int k = warp + q * kWarps;
      if (k < nchunks) {
        const unsigned ball = __ballot_sync(0xffffffffu, rv[q] >= 0);
        if (rv[q] >= 0) idx_s[chunk_base[q] + __popc(ball & ((1u << lane) - 1u))] = rv[q];
      }
    }
    // First use of a stage by a partial tile: the rows past those the
    // gathers write must be finite (they meet P = 0 in the PV); later uses
    // find rows an earlier tile wrote there, so the stages are not zeroed whole
    {
      const int nsw = sm.nswa, nv = total;
      const int tsw = (nsw + kN - 1) / kN;
      const int nt = tsw + (nv - nsw + kN - 1) / kN;
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int jz = 0; jz < min(nt, C::kStages); ++jz) {
        const int start = jz < tsw ? jz * kN : nsw + (jz - tsw) * kN;
        const int n = min(kN, (jz < tsw ? nsw : nv) - start);
        const int nw = kPack ? n : (n + 3) & ~3;   // rows the gathers write (gather4: in fours)
        if (nw >= kN) continue;
        const int per_region = (kN - nw) * 8;      // 16-byte chunks per 128-byte column block
        for (int i = tid; i < C::kRegions * per_region; i += kThreads)
          reinterpret_cast<uint4*>(base + C::kOffKV + jz * C::kStageBytes + (i / per_region) * C::kRegionKV +
                                   nw * 128)[i % per_region] = z;
      }
    }
  } else {
    // f1, the rows shared by a pair's tokens gathered once.  Each token's
    // valid slots are compacted as above; token A's rows go into a hash of
    // (pool, row) keys, which B's rows look up; the union list is token A's
    // list with B's rows that A does not select inserted after A's SWA and
    // compressed runs, in B's order:
    //   [A SWA] [B-only SWA] [A compressed] [B-only compressed]
    // A row that either token selects more than once counts once per slot in
    // that token's softmax, which a shared entry cannot express: then the
    // union is the plain concatenation of the two lists (nothing shared).
    // The construction is deterministic, so both CTAs of the pair build the
    // same list (the hash slots may differ; the flags read back do not).
    uint32_t* hkeys = reinterpret_cast<uint32_t*>(base + C::kOffKV);
    int32_t* hvals = reinterpret_cast<int32_t*>(base + C::kOffKV + C::kScrVals);
    int32_t* list_a = reinterpret_cast<int32_t*>(base + C::kOffKV + C::kScrListA);
    int32_t* list_b = reinterpret_cast<int32_t*>(base + C::kOffKV + C::kScrListB);
    uint8_t* memb = base + C::kOffKV + C::kScrMemb;
    uint8_t* shared_a = base + C::kOffKV + C::kScrShared;
    auto hkey = [](int row, bool comp) { return pair_key(row, comp); };
    {
      const uint4 e4 = make_uint4(kPairEmpty, kPairEmpty, kPairEmpty, kPairEmpty), z = make_uint4(0, 0, 0, 0);
      for (int i = tid; i < C::kHashSlots / 4; i += kThreads) reinterpret_cast<uint4*>(hkeys)[i] = e4;
      for (int i = tid; i < kMaxCols / 16; i += kThreads) reinterpret_cast<uint4*>(shared_a)[i] = z;
      for (int i = tid; i < 2 * C::kMaxTiles; i += kThreads) mask_a[i] = 0ull;
    }
    if (!has_b) zero_q_rows(64);
    if (tid == 0) {
      init_barriers();
      sm.nswa_a = sm.nswa_b = sm.only_b_swa = sm.dup = 0;
      fence_mbar_init_cluster();
    }
    __syncthreads();
    count_chunks(rv, c1a, ti.w_swa, sm.chunk_off, &sm.nswa_a);
    if (has_b) count_chunks(rvb, c1b, w_swa_b, sm.chunk_off_b, &sm.nswa_b);
    __syncthreads();
    const int nswa_a = sm.nswa_a, nswa_b = sm.nswa_b;
    {
      int chunk_base[kChunksPerWarp];
      const int n_a = scan_chunks(sm.chunk_off, nchunks, chunk_base);
      if (warp == 0 && lane == 0) sm.n_a = n_a;
#pragma unroll
      for (int q = 0; q < kChunksPerWarp; ++q) {
        const int k = warp + q * kWarps;
        if (k < nchunks) {
          const unsigned ball = __ballot_sync(0xffffffffu, rv[q] >= 0);
          if (rv[q] >= 0) {
            const int e = chunk_base[q] + __popc(ball & ((1u << lane) - 1u));
            list_a[e] = rv[q];
            pair_insert_a<C::kHashSlots>(hkeys, hvals, &sm.dup, hkey(rv[q], e >= nswa_a), e);
          }
        }
      }
      int n_b = 0;
      if (has_b) {
        n_b = scan_chunks(sm.chunk_off_b, nchunks, chunk_base);
#pragma unroll
        for (int q = 0; q < kChunksPerWarp; ++q) {
          const int k = warp + q * kWarps;
          if (k < nchunks) {
            const unsigned ball = __ballot_sync(0xffffffffu, rvb[q] >= 0);
            if (rvb[q] >= 0) {
              const int e = chunk_base[q] + __popc(ball & ((1u << lane) - 1u));
              list_b[e] = rvb[q];
            }
          }
        }
      }
      if (warp == 0 && lane == 0) sm.n_b = n_b;
    }
    __syncthreads();
    const int n_a = sm.n_a, n_b = sm.n_b;
    // B's entries that A does not select (all of them once a repeat is
    // known), counted per 32-entry chunk of B's list; a B entry that A
    // selects claims A's entry and marks it shared
    const int nch_b = (n_b + 31) / 32;
    unsigned only_b[kChunksPerWarp];
    auto count_only_b = [&](bool all) {
#pragma unroll
      for (int q = 0; q < kChunksPerWarp; ++q) {
        const int k = warp + q * kWarps;
        only_b[q] = 0u;
        if (k < nch_b) {
          const int i = k * 32 + lane;
          bool ob = i < n_b;
          if (ob && !all) {
            const int ia = pair_claim_a<C::kHashSlots>(hkeys, hvals, &sm.dup, hkey(list_b[i], i >= nswa_b));
            if (ia >= 0) shared_a[ia] = 1;
            ob = ia < 0;
          }
          only_b[q] = __ballot_sync(0xffffffffu, ob);
          const unsigned ob_swa = __ballot_sync(0xffffffffu, ob && i < nswa_b);
          if (lane == 0) {
            sm.only_b_chunk[k] = __popc(only_b[q]);
            if (ob_swa) atomicAdd(&sm.only_b_swa, __popc(ob_swa));
          }
        }
      }
    };
    const bool dup_a = sm.dup != 0;
    count_only_b(dup_a);
    __syncthreads();
    const bool dup = sm.dup != 0;
    if (dup && !dup_a) {                   // B repeats a shared row: share nothing after all
      if (tid == 0) sm.only_b_swa = 0;
      __syncthreads();
      count_only_b(true);
      __syncthreads();
    }
    const int bs = sm.only_b_swa;          // B-only SWA entries (they come first in B's order)
    const int nswa_u = nswa_a + bs;
    {
      int chunk_base[kChunksPerWarp];
      const int n_only = scan_chunks(sm.only_b_chunk, nch_b, chunk_base);
      if (warp == 0 && lane == 0) {
        sm.nswa = nswa_u;
        sm.nvalid = n_a + n_only;
      }
#pragma unroll
      for (int q = 0; q < kChunksPerWarp; ++q) {
        const int k = warp + q * kWarps;
        if (k < nch_b && ((only_b[q] >> lane) & 1u)) {
          const int r = chunk_base[q] + __popc(only_b[q] & ((1u << lane) - 1u));
          const int e = r < bs ? nswa_a + r : nswa_u + (n_a - nswa_a) + (r - bs);
          idx_s[e] = list_b[k * 32 + lane];
          memb[e] = 2;
        }
      }
      for (int i = tid; i < n_a; i += kThreads) {
        const int row = list_a[i];
        const bool comp = i >= nswa_a;
        const int e = comp ? nswa_u + (i - nswa_a) : i;
        idx_s[e] = row;
        memb[e] = (uint8_t)(1u | ((!dup && shared_a[i]) ? 2u : 0u));
      }
    }
    __syncthreads();
    {
      // per-tile membership masks (bit i: entry i of the tile)
      const int nswa_t = sm.nswa, nvalid_t = sm.nvalid;
      const int tswa_t = (nswa_t + kN - 1) / kN;
      const int ntiles_t = tswa_t + (nvalid_t - nswa_t + kN - 1) / kN;
      for (int j = warp; j < ntiles_t; j += kWarps) {
        const int start = j < tswa_t ? j * kN : nswa_t + (j - tswa_t) * kN;
        const int n = min(kN, (j < tswa_t ? nswa_t : nvalid_t) - start);
        uint64_t ma = 0ull, mb = 0ull;
#pragma unroll
        for (int hb = 0; hb < kN / 32; ++hb) {
          const int i = hb * 32 + lane;
          const uint32_t m = i < n ? memb[start + i] : 0u;
          ma |= (uint64_t)__ballot_sync(0xffffffffu, (m & 1u) != 0u) << (32 * hb);
          mb |= (uint64_t)__ballot_sync(0xffffffffu, (m & 2u) != 0u) << (32 * hb);
        }
        if (lane == 0) {
          mask_a[j] = ma;
          mask_b[j] = mb;
        }
      }
    }
    __syncthreads();                     // the scratch in the KV stages is dead
    zero_kv_stages();
  }
  {
    if (warp == kMmaWarp) tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
    // Q is read by the tensor core (async proxy): every thread waits for its
    // own Q copies and fences them into the async proxy before the barrier,
    // so no QK can start on a Q row that is not yet visible to it
    asm volatile("cp.async.wait_all;" ::: "memory");
    fence_proxy_async_smem();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
  }
  const uint32_t tmem = sm.tmem_base;
  const Ctx cx{&sm.abort_flag, p.err};
  // tiles: runs of up to N compacted slots of one pool
  const int nswa = sm.nswa, nvalid = sm.nvalid;
  const int tswa = (nswa + kN - 1) / kN;
  const int ntiles = tswa + (nvalid - nswa + kN - 1) / kN;
  auto tile_start = [&](int j) { return j < tswa ? j * kN : nswa + (j - tswa) * kN; };
  auto tile_n = [&](int j) { return min(kN, (j < tswa ? nswa : nvalid) - tile_start(j)); };

  if (warp < kProducerWarps) {
    // ============================================================ producer
    // A warp's TMA requests are served one after another (about 50 ns per
    // gather4), so a tile's requests are spread over the three warps of its
    // group; two groups take alternate tiles (measured: one group of six
    // sharing every tile reaches ~15 GB/s per SM from HBM, warps owning whole
    // tiles ~24 GB/s but with a long issue time per tile; two groups of three
    // were fastest in the full kernel).  A full tile of N consecutive rows (a
    // page run of the page-table form, or a run in the index table) is one
    // box copy per 128-byte column block instead.
    if (tid == 0) {
      prefetch_tensormap(&P.tm_swa);
      prefetch_tensormap(&P.tm_comp);
      prefetch_tensormap(&P.tm_swa_run);
      prefetch_tensormap(&P.tm_comp_run);
    }
    // Producer group pg (kWarpsPerGroup warps) gathers tiles pg, pg + kProducerGroups, ...
    constexpr int kWarpsPerGroup = kProducerWarps / kProducerGroups;
    const int pg = warp / kWarpsPerGroup, pw = warp % kWarpsPerGroup;
    int j = pg;                              // after the loop: past the last tile this group issued
    for (; j < ntiles; j += kProducerGroups) {
      const int st = j % C::kStages;
      if (!warp_wait(cx, bar(sm.kv_empty[st]), ((j / C::kStages) & 1) ^ 1)) break;
      const int start = tile_start(j), n = tile_n(j);
      const uint32_t stage = kv_addr + st * C::kStageBytes;
      const int32_t* rows = idx_s + start;
      if constexpr (kPack != 0) {
        // thread i of the group: row i / 2, column blocks 2 (i % 2) and 2 (i % 2) + 1 of this CTA's half
        const int gi = pw * 32 + lane, r = gi >> 1;
        if (r < n) {
          const bool swa = j < tswa;
          const unsigned char* row = reinterpret_cast<const unsigned char*>(swa ? p.swa : p.comp) +
                                     (int64_t)rows[r] * (swa ? p.swa_stride : p.comp_stride);
          if (kNv && (gi & 1) == 0) sm.rscale[st][r] = __ldg(reinterpret_cast<const float*>(row + 380));
#pragma unroll 1
          for (int kk = 0; kk < 2; ++kk) {
            const int kb = 2 * (gi & 1) + kk;
            uint32_t v[32];
            if constexpr (kNv)
              nvfp4_dims64(row, (int)rank * kHalfDims + 64 * kb, v);
            else
              packed_fp8_dims64(row, (int)rank * kHalfDims + 64 * kb, v);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              st_shared_v4(stage + kb * C::kRegionKV + sw128_offset(r, c),
                           make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]));
          }
        }
        fence_proxy_async_smem();            // the tile is read by the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(sm.kv_full[st]));
        continue;
      }
      const int n4 = (n + 3) & ~3;           // gather4 moves four rows: the last row repeats
      if (pw == 0 && lane == 0) mbar_arrive_expect_tx(bar(sm.kv_full[st]), (uint32_t)(C::kRegions * n4 * 128));
      bool run = false;                      // rows[r] == rows[0] + r for every r < N
      if (n == kN) {
        const uint32_t r0 = (uint32_t)rows[0];
        bool ok = true;
#pragma unroll
        for (int r = lane; r < kN; r += 32) ok = ok && (uint32_t)rows[r] == r0 + (uint32_t)r;
        run = __all_sync(0xffffffffu, ok);
      }
      if (run) {
        // every row of the box was checked against the pool's row count in the set-up
        const void* tmap = j < tswa ? static_cast<const void*>(&P.tm_swa_run) : static_cast<const void*>(&P.tm_comp_run);
        if (pw == 0 && lane < C::kRegions)
          tma_load_2d(stage + lane * C::kRegionKV, tmap, (int)rank * kHalfDims + lane * (128 / C::kElem), rows[0],
                      bar(sm.kv_full[st]));
      } else {
        const void* tmap = j < tswa ? static_cast<const void*>(&P.tm_swa) : static_cast<const void*>(&P.tm_comp);
        const int groups = (n4 / 4) * C::kRegions;
        for (int gi = pw + kWarpsPerGroup * lane; gi < groups; gi += kWarpsPerGroup * 32) {
          const int kb = gi % C::kRegions, r0 = (gi / C::kRegions) * 4;
          tma_gather4(stage + kb * C::kRegionKV + r0 * 128, tmap, (int)rank * kHalfDims + kb * (128 / C::kElem),
                      rows[r0], rows[min(r0 + 1, n - 1)], rows[min(r0 + 2, n - 1)], rows[min(r0 + 3, n - 1)],
                      bar(sm.kv_full[st]));
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // Leave no TMA write of this group in flight, also after an abort: wait
    // (bounded, not cut short by the abort flag) for the last tiles it issued,
    // at most one per stage.  Normally the consumers have waited for them.
    // (Packed rows are written with plain stores: nothing is in flight.)
    if constexpr (kPack == 0)
      for (int jj = max(pg, min(j, ntiles) - C::kStages); jj < min(j, ntiles); ++jj)
        if ((jj - pg) % kProducerGroups == 0) drain_wait(bar(sm.kv_full[jj % C::kStages]), (jj / C::kStages) & 1);
  } else if (warp < kMmaWarp + kQkWarps) {
    // ============================================================ QK issue
    // QK and PV are issued by different warps so that a QK never waits behind
    // a PV (which waits for the softmax): the QK of tile k depends only on its
    // data and a free S buffer.  A thread's chain of dependent MMAs into one
    // accumulator is issued about one instruction per 150 ns (measured), so
    // the tiles' QK chains are spread over three warps, one per S buffer,
    // whose MMAs the tensor core interleaves.
    constexpr uint32_t idesc_qk = idesc(kFp8, 128, kN, false);
    const int qi = warp - kMmaWarp;
    // The other issuers start only once the CTA's first QK has completed:
    // on a GB300, a QK issued by a second warp before the first one finished
    // gave wrong logits for some heads in repeated runs (observed, cause
    // not identified); after that the issuers' chains overlap freely.
    bool ok = qi == 0 || ntiles <= qi || warp_wait(cx, bar(sm.qk0_done), 0);
    for (int k = qi; ok && k < ntiles; k += kQkWarps) {
      const int st = k % C::kStages;
      if (!warp_wait(cx, bar(sm.kv_full[st]), (k / C::kStages) & 1)) break;
      const int b = k % kSBufs;
      if (!warp_wait(cx, bar(sm.s_empty[b]), ((k / kSBufs) & 1) ^ 1)) break;
      fence_proxy_async_smem();
      tc_fence_after();
      if (lane == 0) {
        const uint32_t stage = kv_addr + st * C::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < C::kK1; ++kk) {
          const uint64_t a = desc_sw128(q_addr + (kk >> 2) * C::kRegionQ + (kk & 3) * 32, 16, 1024);
          const uint64_t kd = desc_sw128(stage + (kk >> 2) * C::kRegionKV + (kk & 3) * 32, 16, 1024);
          if (kNv && rank == 1 && kk >= C::kK1 - 4)     // CTA 1's dims 448-511: the RoPE logits apart
            mma<kFp8>(tmem + kSRCol + b * kN, a, kd, idesc_qk, kk > C::kK1 - 4 ? 1u : 0u);
          else
            mma<kFp8>(tmem + kSCol + b * kN, a, kd, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(sm.s_full[b]));
        if (k == 0) mma_commit(bar(sm.qk0_done));
      }
      __syncwarp();
    }
    if (lane == 0) mma_commit(bar(sm.qk_done));   // completes once every QK issued above is done
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ============================================================ PV issue
    constexpr uint32_t idesc_pv = idesc(kFp8, 128, kHalfDims, true);
    for (int jj = 0; jj < ntiles; ++jj) {
      const int b = jj & 1, st = jj % C::kStages;
      if (!warp_wait(cx, bar(sm.p_full[b]), (jj >> 1) & 1)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t stage = kv_addr + st * C::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < C::kK2; ++kk) {
          const uint64_t v = desc_sw128(stage + kk * (C::kKStep / 8) * 1024, C::kRegionKV, 1024);
          const uint32_t pk = b * C::kPCols + kk * (C::kKStep * C::kElem / 4);
          const uint32_t acc = (jj > 0 || kk > 0) ? 1u : 0u;
          if constexpr (kNv) {
            // NoPE output dims take P times the row scale, CTA 1's RoPE dims (its last 64) P
            if (rank == 0) {
              mma_tmem_a<kFp8>(tmem + kOCol, tmem + kPGCol + pk, v, idesc_pv, acc);
            } else {
              constexpr uint32_t idesc_nope = idesc(kFp8, 128, kHalfDims - 64, true);
              constexpr uint32_t idesc_rope = idesc(kFp8, 128, 64, true);
              const uint64_t vr = desc_sw128(stage + 3 * C::kRegionKV + kk * (C::kKStep / 8) * 1024, C::kRegionKV, 1024);
              mma_tmem_a<kFp8>(tmem + kOCol, tmem + kPGCol + pk, v, idesc_nope, acc);
              mma_tmem_a<kFp8>(tmem + kOCol + kHalfDims - 64, tmem + C::kPCol + pk, vr, idesc_rope, acc);
            }
          } else {
            mma_tmem_a<kFp8>(tmem + kOCol, tmem + C::kPCol + pk, v, idesc_pv, acc);
          }
        }
        mma_commit(bar(sm.p_empty[b]));
        mma_commit(bar(sm.kv_empty[st]));
      }
      __syncwarp();
    }
    if (lane == 0) mma_commit(bar(sm.o_full));    // completes once every PV issued above is done
    __syncwarp();
  } else {
    // ============================================================ softmax / epilogue
    // Two warpgroups take turns: warpgroup g handles tiles j with j % 2 == g
    // (all N slots; S, P and exchange buffer g).  The only hand-off between
    // consecutive tiles is the running reference maximum m(j), published by
    // the warpgroup of tile j as soon as it is known, so one warpgroup's
    // exponentials overlap the other's loads and exchange.
    const int g = (warp - kSoftmaxWarp0) >> 2;        // warpgroup
    const int q4 = warp & 3;                           // TMEM lane quadrant of this warp
    const int h = q4 * 32 + lane;                      // MMA row (a token pair: head h & 63 of token t + (h >> 6))
    const bool active = q4 * 32 < rows_used;           // warp-uniform
    const bool leader = (warp - kSoftmaxWarp0) % 4 == 0 && lane == 0;   // one thread per warpgroup
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    const float c = load_scale(p.bmm1, p.bmm1_dev) * kLog2e;
    const uint32_t xbytes = (uint32_t)(rows_used * kN * 3);   // bytes the peer pushes per tile (24-bit logits)
    const uint64_t* my_mask = (h < 64) ? mask_a : mask_b;     // token pairs: this row's entries of each tile
    constexpr uint32_t kBarStride = (uint32_t)sizeof(uint64_t);
    const uint32_t x_mine = x_addr + g * C::kXBytes;
    const uint32_t x_peer = map_to_rank(x_mine, peer);
    const uint32_t xin_full_peer = map_to_rank(bar(sm.xin_full[0]), peer) + g * kBarStride;
    const uint32_t xout_free_peer = map_to_rank(bar(sm.xout_free[0]), peer) + g * kBarStride;
    const uint32_t p_cols = C::kPCol + g * C::kPCols;  // P buffer g
    if (leader) mbar_arrive_expect_tx(bar(sm.xin_full[g]), xbytes);
    if (!active) {
      // rows of absent heads: P = 0, so O stays 0 there
      uint32_t zr[C::kPCols];
#pragma unroll
      for (int i = 0; i < C::kPCols; ++i) zr[i] = 0u;
      tmem_st16(tl + p_cols, zr);
      if constexpr (kNv) tmem_st16(tl + kPGCol + g * C::kPCols, zr);
      tmem_wait_st();
    }
    // send this CTA's partial S of tile jj (a tile of my warpgroup) to the peer
    auto push = [&](int jj) -> bool {
      const int sb = jj % kSBufs;
      if (!warp_wait(cx, bar(sm.s_full[sb]), (jj / kSBufs) & 1)) return false;
      // NVFP4: the row scales came with the tile (plain stores before the producers' arrival)
      if (kNv && !warp_wait(cx, bar(sm.kv_full[jj % C::kStages]), (jj / C::kStages) & 1)) return false;
      tc_fence_after();
      if (jj >= 2 && !warp_wait(cx, bar(sm.xout_free[g]), ((jj >> 1) & 1) ^ 1, true)) return false;
      if (active) {
        const uint32_t xb = x_peer + (uint32_t)(h * 16);
#pragma unroll
        for (int hb = 0; hb < kN / 16; ++hb) {
          uint32_t v[16];
          tmem_ld16(tl + kSCol + sb * kN + hb * 16, v);
          tmem_wait_ld();
          if constexpr (kNv) {
            // this CTA's share of the logit: g S over its NoPE dims, plus CTA 1's RoPE part
            const float* rs = sm.rscale[jj % C::kStages] + hb * 16;
            uint32_t vr[16];
            if (rank == 1) {
              tmem_ld16(tl + kSRCol + sb * kN + hb * 16, vr);
              tmem_wait_ld();
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
              v[i] = __float_as_uint(rs[i] * __uint_as_float(v[i]) + (rank == 1 ? __uint_as_float(vr[i]) : 0.f));
          }
          // 24-bit logits: the low mantissa byte is dropped after rounding;
          // values a, b, c, d travel as [a1 a2 a3 d1] [b1 b2 b3 d2] [c1 c2 c3 d3]
          uint32_t w[12];
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {
            const uint32_t d = v[4 * gq + 3] + 0x80u;
            w[3 * gq] = __byte_perm(v[4 * gq] + 0x80u, d, 0x5321);
            w[3 * gq + 1] = __byte_perm(v[4 * gq + 1] + 0x80u, d, 0x6321);
            w[3 * gq + 2] = __byte_perm(v[4 * gq + 2] + 0x80u, d, 0x7321);
          }
#pragma unroll
          for (int q = 0; q < 3; ++q)
            st_async_v4(xb + (uint32_t)((hb * 3 + q) * 128 * 16), __uint_as_float(w[4 * q]),
                        __uint_as_float(w[4 * q + 1]), __uint_as_float(w[4 * q + 2]), __uint_as_float(w[4 * q + 3]),
                        xin_full_peer);
        }
      }
      return true;
    };

    float m_last = -INFINITY, l_run = 0.f;            // reference and row sum of my warpgroup's tiles
    // E4M3 P keeps 3 mantissa bits: under a lagging reference a row's largest P
    // (up to 2^8) is rounded by up to 1/16, which shows when few slots carry the
    // mass, so short tile chains move the reference on every new maximum (the
    // same choice in both CTAs: ntiles is the pair's).
    const float thr = (kFp8 && ntiles <= kExactRefTiles) ? 0.f : kRescaleThreshold;
    bool ok = true;
    if (g < ntiles) ok = push(g);
    int j = g;
    const uint64_t c2 = f2_pack(c, c);
    for (; ok && j < ntiles; j += 2) {
      const int n_cur = tile_n(j);
      const int sb = j % kSBufs;
      // S(j) is final (this warpgroup pushed it): its TMEM load overlaps the wait for the peer's half
      float sv[kN];
      if (active) {
#pragma unroll
        for (int hb = 0; hb < kN / 32; ++hb) {
          uint32_t r[32];
          tmem_ld32(tl + kSCol + sb * kN + hb * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[hb * 32 + i] = __uint_as_float(r[i]);
        }
        if constexpr (kNv) {                      // as pushed: g S (+ CTA 1's RoPE part)
          tmem_wait_ld();
          const float* rs = sm.rscale[j % C::kStages];
          if (rank == 1) {
#pragma unroll
            for (int hb = 0; hb < kN / 32; ++hb) {
              uint32_t r[32];
              tmem_ld32(tl + kSRCol + sb * kN + hb * 32, r);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) sv[hb * 32 + i] = rs[hb * 32 + i] * sv[hb * 32 + i] + __uint_as_float(r[i]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < kN; ++i) sv[i] *= rs[i];
          }
        }
      }
      if (!(ok = warp_wait(cx, bar(sm.xin_full[g]), (j >> 1) & 1, true))) break;
      tc_fence_after();
      float mt = -INFINITY;
      if (active) {
        tmem_wait_ld();
        const uint4* xp = reinterpret_cast<const uint4*>(base + C::kOffX + g * C::kXBytes) + h;
#pragma unroll
        for (int hb = 0; hb < kN / 16; ++hb) {
          uint32_t w[12];
#pragma unroll
          for (int q = 0; q < 3; ++q) {
            const uint4 x = xp[(hb * 3 + q) * 128];
            w[4 * q] = x.x;
            w[4 * q + 1] = x.y;
            w[4 * q + 2] = x.z;
            w[4 * q + 3] = x.w;
          }
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {
            const uint32_t w0 = w[3 * gq], w1 = w[3 * gq + 1], w2 = w[3 * gq + 2];
            const float pa = __uint_as_float(w0 << 8), pb = __uint_as_float(w1 << 8), pc = __uint_as_float(w2 << 8);
            const float pd = __uint_as_float(__byte_perm(__byte_perm(w0, w1, 0x7373), w2, 0x7103));
            const int i = hb * 16 + 4 * gq;
            f2_unpack(f2_mul(f2_add(f2_pack(sv[i], sv[i + 1]), f2_pack(pa, pb)), c2), sv[i], sv[i + 1]);
            f2_unpack(f2_mul(f2_add(f2_pack(sv[i + 2], sv[i + 3]), f2_pack(pc, pd)), c2), sv[i + 2], sv[i + 3]);
          }
        }
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if constexpr (kPair) {
          // only the entries of this row's token (the tile's other entries are the other token's)
          const uint64_t mrow = my_mask[j];
#pragma unroll
          for (int i = 0; i < kN; ++i)
            if ((mrow >> i) & 1ull) m4[i & 3] = fmaxf(m4[i & 3], sv[i]);
        } else if (n_cur >= kN) {
#pragma unroll
          for (int i = 0; i < kN; ++i) m4[i & 3] = fmaxf(m4[i & 3], sv[i]);
        } else {
#pragma unroll
          for (int i = 0; i < kN; ++i)
            if (i < n_cur) m4[i & 3] = fmaxf(m4[i & 3], sv[i]);
        }
        mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      }
      if (leader) mbar_arrive_expect_tx(bar(sm.xin_full[g]), xbytes);   // for tile j + 2
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(sm.s_empty[sb]));                         // S buffer sb may be overwritten
        mbar_arrive_cluster_relaxed(xout_free_peer);               // exchange buffer g read out
      }
      // ---- reference maximum: m(j) = mt if it exceeds m(j-1) by the threshold, else m(j-1)
      float m_prev = -INFINITY;
      if (j > 0) {
        if (!(ok = warp_wait(cx, bar(sm.m_ready[g ^ 1]), ((j - 1) >> 1) & 1))) break;
        m_prev = sm.m_buf[g ^ 1][h];
      }
      const float m_cur = (mt > m_prev + thr) ? mt : m_prev;
      sm.m_buf[g][h] = m_cur;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(sm.m_ready[g]));
      // ---- look ahead: my next tile's partial S to the peer (before this tile's
      // exponentials, so that the peer has it by the time it gets there)
      if (j + 2 < ntiles && !(ok = push(j + 2))) break;
      // ---- P = 2^(x - m(j)); this warpgroup's row sum, rescaled to m(j)
      if (!(ok = warp_wait(cx, bar(sm.p_empty[g]), ((j >> 1) & 1) ^ 1))) break;   // PV(j - 2) done
      tc_fence_after();
      if (active) {
        l_run *= (m_last == -INFINITY) ? 0.f : fast_exp2(m_last - m_cur);
        m_last = m_cur;
        const uint64_t nm2 = f2_pack(-m_cur, -m_cur);
#pragma unroll
        for (int i = 0; i < kN; i += 2) {
          float x0, x1;
          f2_unpack(f2_add(f2_pack(sv[i], sv[i + 1]), nm2), x0, x1);
          sv[i] = fast_exp2(x0);
          sv[i + 1] = fast_exp2(x1);
        }
        if constexpr (kPair) {
          const uint64_t mrow = my_mask[j];
#pragma unroll
          for (int i = 0; i < kN; ++i)
            if (!((mrow >> i) & 1ull)) sv[i] = 0.f;
        } else if (n_cur < kN) {
#pragma unroll
          for (int i = 0; i < kN; ++i)
            if (i >= n_cur) sv[i] = 0.f;
        }
        uint64_t s4[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < kN; i += 2) s4[(i >> 1) & 1] = f2_add(s4[(i >> 1) & 1], f2_pack(sv[i], sv[i + 1]));
        float s0, s1, s2, s3;
        f2_unpack(s4[0], s0, s1);
        f2_unpack(s4[1], s2, s3);
        l_run += (s0 + s1) + (s2 + s3);
        uint32_t pr[C::kPCols];
        if constexpr (kFp8) {
#pragma unroll
          for (int i = 0; i < C::kPCols; ++i)
            pr[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(sv[4 * i], sv[4 * i + 1]), __NV_SATFINITE, __NV_E4M3) |
                    ((uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(sv[4 * i + 2], sv[4 * i + 3]), __NV_SATFINITE, __NV_E4M3) << 16);
        } else {
#pragma unroll
          for (int i = 0; i < C::kPCols; ++i) pr[i] = pack_bf16x2(sv[2 * i], sv[2 * i + 1]);
        }
        tmem_st16(tl + p_cols, pr);
        if constexpr (kNv) {                      // P of the NoPE output dims: times each slot's row scale
          const float* rs = sm.rscale[j % C::kStages];
#pragma unroll
          for (int i = 0; i < C::kPCols; ++i) pr[i] = pack_bf16x2(sv[2 * i] * rs[2 * i], sv[2 * i + 1] * rs[2 * i + 1]);
          tmem_st16(tl + kPGCol + g * C::kPCols, pr);
        }
      }
      // ---- O rescale when the reference moved (O holds tiles < j at m(j-1))
      const bool rescale = active && j > 0 && m_cur != m_prev;
      if (__any_sync(0xffffffffu, rescale)) {
        if (!(ok = warp_wait(cx, bar(sm.p_empty[g ^ 1]), ((j - 1) >> 1) & 1))) break;
        tc_fence_after();
        const float alpha = rescale ? fast_exp2(m_prev - m_cur) : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < kHalfDims / 16; ++cc) {
          uint32_t r[16];
          tmem_ld16(tl + kOCol + cc * 16, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st16(tl + kOCol + cc * 16, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(sm.p_full[g]));
    }
    // total row sum: both warpgroups' sums brought to the final reference
    if (active) {
      sm.lsum[g][h] = l_run;
      sm.m_end[g][h] = m_last;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(sm.lsum_full));
    if (ok) ok = warp_wait(cx, bar(sm.lsum_full), 0);
    if (ok && ntiles > 0) {
      ok = warp_wait(cx, bar(sm.o_full), 0);
      tc_fence_after();
    }
    if (active) {
      float l_tot = 0.f, m_fin = -INFINITY;
      if (ok) {
        const float ma = sm.m_end[0][h], mb = sm.m_end[1][h];
        m_fin = fmaxf(ma, mb);
        if (m_fin != -INFINITY) {
          if (ma != -INFINITY) l_tot += sm.lsum[0][h] * fast_exp2(ma - m_fin);
          if (mb != -INFINITY) l_tot += sm.lsum[1][h] * fast_exp2(mb - m_fin);
        }
      }
      const bool have = ok && ntiles > 0 && l_tot > 0.f;
      const float lse = have ? m_fin + fast_log2(l_tot) : -INFINITY;
      float f = have ? 1.f / l_tot : 0.f;
      if (S == 1) {
        f *= load_scale(p.bmm2, p.bmm2_dev);
        if (p.sinks != nullptr && have) f *= 1.f / (1.f + fast_exp2(__ldg(p.sinks + (kPair ? (h & 63) : h)) * kLog2e - lse));
      }
      const int64_t row_th = kPair ? (int64_t)(t + (h >> 6)) * H + (h & 63) : (int64_t)t * H + h;
      // The BF16 rows (the output, or a split partial) go through shared
      // memory (the KV stages are free once every PV is done), so that the
      // global stores below are whole 256-byte row segments rather than one
      // 16-byte piece per row per warp instruction.  Warpgroup g stages its
      // 128 columns; 16-byte chunks are XOR-swizzled by the row to spread banks.
      unsigned char* row = base + C::kOffKV + g * (128 * 256) + h * 256;
#pragma unroll 1
      for (int cc = 0; cc < kHalfDims / 64; ++cc) {
        const int col = g * (kHalfDims / 2) + cc * 32;
        float v[32];
        if (have) {
          uint32_t r[32];
          tmem_ld32(tl + kOCol + col, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * f;
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(row + (((cc * 4 + q) ^ (h & 7)) << 4)) =
              make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                         pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
      }
      if (rank == 0 && g == 0) {
        if (kPartial)
          p.part_lse[row_th * S + s] = lse;
        else if (p.out_lse)
          p.out_lse[row_th] = lse;
      }
    }
    // copy-out of this warpgroup's staged columns, 256 contiguous bytes per
    // row (half a warp per row): the output row, or the split partial row
    {
      asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(128) : "memory");
      const unsigned char* stg = base + C::kOffKV + g * (128 * 256);
      const int w4 = (warp - kSoftmaxWarp0) & 3;
      const int col0 = (int)rank * kHalfDims + g * (kHalfDims / 2);
      const int c = lane & 15;
      for (int r = w4 + 4 * (lane >> 4); r < rows_used; r += 8) {
        const uint4 x = *reinterpret_cast<const uint4*>(stg + r * 256 + ((c ^ (r & 7)) << 4));
        const int64_t row = kPair ? (int64_t)(t + (r >> 6)) * H + (r & 63) : (int64_t)t * H + r;
        *reinterpret_cast<uint4*>((kPartial ? p.part_o + (row * S + s) * kHeadDim : p.out + row * kHeadDim) +
                                  col0 + c * 8) = x;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == kMmaWarp) {
    // no MMA may still use TMEM (bounded, and not cut short by the abort flag)
    drain_wait(bar(sm.qk_done), 0);
    drain_wait(bar(sm.o_full), 0);
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  tc_fence_before();
  cluster_sync();                          // the peer is done with this CTA's shared memory
}

}  // namespace

int tc_grid_smem_bytes(int dtype, bool pair) {
  // E4M3 rows run the FP8 geometry; BF16 and the packed forms the BF16 one
  if (pair) return dtype == SMLA_E4M3 ? Cfg<true, true>::kSmemBytes : Cfg<false, true>::kSmemBytes;
  return dtype == SMLA_E4M3 ? Cfg<true>::kSmemBytes : Cfg<false>::kSmemBytes;
}
int tc_grid_threads() { return kThreads; }

cudaError_t launch_decode_tc_grid(const DecodeParams& p, int grid, bool pair, cudaStream_t stream) {
  if (pair && p.H != 64) return cudaErrorInvalidValue;   // two tokens of 64 heads fill the 128 MMA rows
  const bool packed = p.dtype == SMLA_PACKED_FP8 || p.dtype == SMLA_NVFP4;
  if (pair && packed) return cudaErrorInvalidValue;
  TcParams P;
  memset(&P, 0, sizeof(P));
  P.p = p;
  const int smem = tc_grid_smem_bytes(p.dtype, pair);
  auto launch = [&](auto kernel) -> cudaError_t {
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    kernel<<<grid, kThreads, smem, stream>>>(P);
    return cudaSuccess;
  };
  const bool partial = p.num_splits > 1;
  if (packed) {                         // no tensor maps: the producers load the rows themselves
    cudaError_t e;
    if (p.dtype == SMLA_PACKED_FP8)
      e = partial ? launch(decode_tc_kernel<false, true, false, SMLA_PACKED_FP8>)
                  : launch(decode_tc_kernel<false, false, false, SMLA_PACKED_FP8>);
    else
      e = partial ? launch(decode_tc_kernel<false, true, false, SMLA_NVFP4>)
                  : launch(decode_tc_kernel<false, false, false, SMLA_NVFP4>);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  // a pool of fewer than N rows holds no run of N rows: its run map is never used
  const int64_t run_rows = p.dtype == SMLA_BF16 ? Cfg<false>::kN : Cfg<true>::kN;
  const int swa_run = (int)std::max<int64_t>(1, std::min(run_rows, p.swa_rows));
  const int comp_run = (int)std::max<int64_t>(1, std::min(run_rows, p.comp_rows));
  cudaError_t e = encode_pool_map(&P.tm_swa, p.swa, p.swa_rows, p.swa_stride, p.dtype, 1);
  if (e == cudaSuccess) e = encode_pool_map(&P.tm_comp, p.comp, p.comp_rows, p.comp_stride, p.dtype, 1);
  if (e == cudaSuccess) e = encode_pool_map(&P.tm_swa_run, p.swa, p.swa_rows, p.swa_stride, p.dtype, swa_run);
  if (e == cudaSuccess) e = encode_pool_map(&P.tm_comp_run, p.comp, p.comp_rows, p.comp_stride, p.dtype, comp_run);
  if (e != cudaSuccess) return e;
  if (pair) {
    if (p.dtype == SMLA_BF16)
      e = partial ? launch(decode_tc_kernel<false, true, true, 0>) : launch(decode_tc_kernel<false, false, true, 0>);
    else
      e = partial ? launch(decode_tc_kernel<true, true, true, 0>) : launch(decode_tc_kernel<true, false, true, 0>);
  } else if (p.dtype == SMLA_BF16) {
    e = partial ? launch(decode_tc_kernel<false, true, false, 0>) : launch(decode_tc_kernel<false, false, false, 0>);
  } else {
    e = partial ? launch(decode_tc_kernel<true, true, false, 0>) : launch(decode_tc_kernel<true, false, false, 0>);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace smla
