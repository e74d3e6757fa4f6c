// tcgen05 / TMEM sparse MLA decode kernel for sm_103a.
//
// A cluster of two CTAs works through a list of units; a unit is the columns
// [c0, c1) of one token's index row.  Units are handed out in one of two ways:
//
//   grid mode        one unit per cluster: (token, split s of S)
//   balanced mode    cluster c of P takes the c-th of P equal, contiguous
//                    shares of the token-major column space (T tokens x W
//                    columns): whole tokens, plus the piece of a token cut at
//                    either end of the share.  Whole tokens write the output;
//                    a piece writes its normalised partial and LSE, counts
//                    itself on its token's counter, and the token's last
//                    piece to finish merges the others with its own fp32 O
//                    into the output.  Every cluster gets the same number of columns,
//                    so no SM pair idles through a last, partial wave, and a
//                    unit's index compaction and first gathers overlap the
//                    previous unit's last tiles.
//
// CTA r of the pair owns output dims [256 r, 256 r + 256): an fp32 accumulator
// for 128 heads x 512 dims is 256 KB, the whole tensor memory of one SM, so
// the output is split across the pair.  Per tile of up to N selected slots
// (N = 64 for E4M3, 32 for BF16):
//
//   producer warps 0-3  per unit, the index compaction: the unit's columns are
//                       loaded, masked and compacted (ballots and scans) into
//                       a list: SWA slots, then compressed slots; tiles are runs
//                       of N list entries of one pool (masked slots are never
//                       loaded); then the pair's half of every selected row
//                       (256 dims) with TMA tile::gather4 (four rows of 128
//                       bytes per request) into a 128-byte-swizzled,
//                       UMMA-canonical shared-memory tile of a 7-stage (E4M3)
//                       or 6-stage (BF16) ring; two groups of two warps take
//                       alternate tiles; a tile of N consecutive rows is one box
//                       copy per 128-byte block
//   QK warps 4-6        per unit, the token's query half (TMA box loads, issued
//                       by warp 4 once every QK of the previous unit is done),
//                       then S_r = Q_r K_r^T (M = 128 heads, N slots, K = 256
//                       dims) into one of three TMEM S buffers; warp 4 + b
//                       issues the tiles of buffer b (one thread's chain of
//                       dependent MMAs runs at about one instruction per
//                       150 ns, so the chains overlap); warp 4 also allocates
//                       and frees TMEM
//   PV warp 7           O_r += P V_r (M = 128 heads, N = 256 dims, K = N slots,
//                       P read from TMEM); a unit's first PV waits until the
//                       previous unit's O has been read out
//   softmax warps 8-15  two warpgroups taking whole tiles in turn (warpgroup g
//                       takes tiles j with j % 2 == g), one thread per head:
//                       read S_r from TMEM, push it to the peer CTA with
//                       st.async (completing bytes on the peer's mbarrier) as
//                       24-bit floats (four values in three words), add the
//                       peer's partial (S = S_0 + S_1; each CTA adds its own
//                       exact half), settle the running reference maximum m(j)
//                       from m(j-1) (handed over by the other warpgroup through
//                       shared memory), exponentials in base 2 with lazy
//                       rescaling of O, write P (BF16 or E4M3) into TMEM; at a
//                       unit's end both warpgroups normalise O and store it
//                       (the BF16 output, or BF16 normalised partials) plus the
//                       LSE.  Each warpgroup pushes its next tile's partial S
//                       before its exponentials; one warpgroup's exponentials
//                       overlap the other's loads and exchange.
//
// Tiles are numbered across the units of a cluster, so the rings of KV
// stages, S / P buffers and exchange buffers run on without a break between
// units.
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

#include <algorithm>
#include <atomic>

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
constexpr int kProducerWarps = 4;    // index compaction and TMA gathers
constexpr int kProducerGroups = 2;   // tiles alternate between two groups of two warps that share each tile
constexpr int kMmaWarp = kProducerWarps;        // first QK issuer; loads Q; allocates and frees TMEM
constexpr int kQkWarps = 3;                     // QK issuers: warp kMmaWarp + i issues the tiles j with j % 3 == i
constexpr int kPvWarp = kMmaWarp + kQkWarps;    // PV issue
constexpr int kSoftmaxWarp0 = 8;
constexpr int kSoftmaxWarps = 8;
constexpr int kPushWarp0 = kSoftmaxWarp0 + kSoftmaxWarps;   // partial-S exchange, one warp per TMEM lane quadrant
constexpr int kPushWarps = 4;
constexpr int kThreads = (kPushWarp0 + kPushWarps) * 32;
// Registers per thread of each warpgroup after the role split (setmaxnreg):
// the launch gives every thread kLaunchRegs; the MMA and push warpgroups hand
// registers back, the two softmax warpgroups take them, the producers keep
// theirs (their index compaction holds two 18-entry arrays per lane).
constexpr int kLaunchRegs = 65536 / kThreads / 8 * 8;
constexpr int kRegsProducer = kLaunchRegs;
constexpr int kRegsMma = 40;
constexpr int kRegsSoftmax = 136;
constexpr int kRegsPush = 64;
static_assert(128 * (kRegsProducer + kRegsMma + kRegsPush) + 256 * kRegsSoftmax <= kThreads * kLaunchRegs,
              "the warpgroups' registers after the split fit in what the launch holds");
constexpr int kMaxCols = SMLA_TC_MAX_SPLIT_COLS;
constexpr int kMaxChunks = kMaxCols / 32;                 // 32-column chunks of a unit
constexpr int kMaxUnits = SMLA_TC_MAX_UNITS;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;        // O: 256 fp32 columns
constexpr uint32_t kSCol = 256;      // S: three buffers of N fp32 columns, then P: two buffers of 16 columns
constexpr int kSBufs = 3;
// One QK issuer per S buffer: an issuer then waits on its buffer's phases in
// order.  An issuer taking tiles of several buffers could wait two phases
// ahead of a buffer's release, which a parity wait cannot tell from one phase
// behind.
static_assert(kQkWarps == kSBufs, "one QK issuer per S buffer");
constexpr float kRescaleThreshold = 8.f;   // log2 units: P stays <= 2^8
constexpr int kExactRefTiles = 8;          // E4M3 P: chains of at most this many tiles follow the exact maximum
constexpr int kMaxStages = 8;
static_assert(kPvWarp >= kMmaWarp + kQkWarps && kPvWarp < kSoftmaxWarp0, "warp roles");
static_assert(kMmaWarp % 4 == 0 && kPvWarp == kMmaWarp + 3, "the QK and PV warps form one warpgroup");
static_assert(kSoftmaxWarp0 % 4 == 0 && kPushWarp0 % 4 == 0, "warpgroups start at multiples of four warps");

// A unit of work: columns [c0, c1) of token t, and where its result goes.
struct Unit {
  int32_t t, c0, c1;
  int32_t partial;           // 0: the output (bmm2, sink, BF16 out, out_lse); 1: a normalised partial
  int64_t part_row;          // partial: element offset of head 0's row
  int64_t lse_row;           // partial: offset of head 0's LSE
  int32_t part_hstride;      // partial: elements between consecutive heads' rows
  int32_t lse_hstride;       // partial: entries between consecutive heads' LSEs
  // balanced mode, a piece of a cut token: the token's pieces are the head
  // piece of cluster merge_first (slot 2 merge_first + 1) and the continuing
  // pieces of the next merge_n - 1 clusters (slot 2 c'); the last of them to
  // finish merges all into the output
  int32_t merge_first, merge_n;
  // written by the producers once the unit is compacted
  int32_t nswa, nvalid, ntiles, tile0;
  int32_t swa_tail, last_tail;   // slots of the last SWA tile and of the last tile
};

struct TcSmall {
  uint64_t kv_full[kMaxStages];
  uint64_t kv_empty[kMaxStages];
  uint64_t s_full[kSBufs], s_empty[kSBufs], p_full[2], p_empty[2];
  uint64_t xin_full[2], xout_free[2];
  uint64_t m_ready[2];                   // m_buf[g] written by warpgroup g's four warps
  uint64_t unit_ready[kMaxUnits];        // unit u compacted (single use)
  uint64_t prod_counts;                  // the producer warps' chunk counts of a unit written (one phase per unit)
  uint64_t prod_list;                    // the producer warps' slot lists of a unit written (one phase per unit)
  uint64_t q_full;                       // a unit's Q landed (one phase per unit using Q: the first, and those with tiles)
  uint64_t qk_first;                     // a unit's first QK done (one phase per unit with tiles)
  uint64_t qk_unit_done;                 // every QK of a unit done (one phase per unit using Q)
  uint64_t lsum_full;                    // both warpgroups' row sums of a unit written (one phase per unit)
  uint64_t unit_pv_done;                 // every PV of a unit done (one phase per unit)
  uint64_t o_free;                       // a unit's O read out (one phase per unit)
  uint64_t epi_staged[2];                // warpgroup g's rows of the last unit staged in shared memory (single use)
  uint64_t piece_sync;                   // balanced mode: the softmax warps wrote a piece (one phase per piece)
  uint64_t piece_dec;                    // balanced mode: whether this piece is its token's last one is known
  int32_t piece_last;                    // balanced mode: this CTA merges the token's pieces
  uint64_t o_full;                       // every PV done (committed by the PV warp at the end)
  uint64_t qk_done;                      // every QK done (one commit per QK warp at the end)
  float m_end[2][2][128];                // [unit & 1][warpgroup][head]: final reference maximum
  float lsum[2][2][128];                 // [unit & 1][warpgroup][head]: row sum at m_end
  float m_buf[2][128];                   // reference maximum after the last tile of warpgroup g
  float2 epi[2][128];                    // [warpgroup][head]: bmm2 scale, sink x log2(e) (each thread its own)
  int32_t chunk_cnt[kMaxChunks];         // compacted-slot count of each 32-column chunk
  int32_t chunk_swa[kMaxChunks];         // of which SWA slots
  Unit unit[kMaxUnits];
  int32_t nunits;
  uint32_t tmem_base;
  int32_t abort_flag;
};

template <bool kFp8>
struct Cfg {
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kN = kFp8 ? 64 : 32;                    // slots per tile
  static constexpr int kRegions = kHalfDims * kElem / 128;     // 128-byte column blocks per half row
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
  static constexpr int kOffIdx = kOffX + 2 * kXBytes;
  static constexpr int kOffSmall = kOffIdx + 2 * kMaxCols * 4;             // two slot lists
  static constexpr int kSmemBytes = kOffSmall + (int)sizeof(TcSmall) + 1024;   // + alignment slack
  static_assert(kStages <= kMaxStages, "barrier arrays");
  static_assert(kStages >= 3, "PV lags QK by two tiles: a third stage keeps the producer going");
  static_assert(kN <= kMaxN, "row lists");
  static_assert(kPCols == 16, "P buffer width");
  static_assert(kN % 32 == 0, "tiles are whole 32-column groups");
  static_assert(kPCol + 2 * kPCols <= kTmemCols, "tensor memory budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Kernel parameters: the shared decode parameters; two TMA descriptors per KV
// pool ([rows, 512] with the pool's row stride; 128-byte swizzle): box = 128
// bytes x 1 row for tile::gather4, and 128 bytes x N rows for whole-tile
// copies of N consecutive rows; the query as [T, H, 512] (box 128 bytes x H
// heads x 1 token); and the unit hand-out.
struct TcParams {
  CUtensorMap tm_swa;
  CUtensorMap tm_comp;
  CUtensorMap tm_swa_run;
  CUtensorMap tm_comp_run;
  CUtensorMap tm_q;
  DecodeParams p;
  int32_t clusters;            // balanced mode: P shares; 0: grid mode
  __nv_bfloat16* piece_o;      // balanced mode: [P][2][H][512] BF16 normalised pieces of cut tokens
  float* piece_lse;            // balanced mode: [P][2][2 ranks][H] their base-2 LSEs (each CTA writes its own)
  uint32_t* piece_cnt;         // balanced mode: [P][2 ranks] pieces finished per cut token (zero at launch)
};

// The units of cluster c; returns their count (at most kMaxUnits, which the
// planner guarantees).  In balanced mode a piece goes to slot 2c if it
// continues a token begun by an earlier cluster (c0 > 0), else to slot 2c + 1
// (the head of a token that later clusters continue); cluster c covers the
// columns [g(c), g(c + 1)) of the token-major column space, g(c) = floor(T W c / P).
__device__ int make_units(const TcParams& P, int c, Unit* units) {
  const DecodeParams& p = P.p;
  const int H = p.H;
  if (P.clusters == 0) {
    // Column range of split s, from the table width only (so that the index
    // loads need not wait for any device value): [c0, c0 + ceil(W / S)); in
    // the page-table form rounded up to whole 64-slot runs, so that every full
    // tile of compressed slots lies on one page when pages hold a multiple of
    // 64 rows.
    const int S = p.num_splits;
    const int s = c % S, t = c / S;
    int per_split = (p.W + S - 1) / S;
    if (p.bt) per_split = (per_split + kMaxN - 1) / kMaxN * kMaxN;
    Unit u = {};
    u.t = t;
    u.c0 = min(p.W, s * per_split);
    u.c1 = min(p.W, u.c0 + per_split);
    u.partial = S > 1;
    u.part_row = ((int64_t)t * H * S + s) * kHeadDim;
    u.part_hstride = S * kHeadDim;
    u.lse_row = (int64_t)t * H * S + s;
    u.lse_hstride = S;
    units[0] = u;
    return 1;
  }
  const int64_t W = p.W;
  const int64_t total = (int64_t)p.sum_q * W;
  const int64_t g0 = total * c / P.clusters, g1 = total * (c + 1) / P.clusters;
  int n = 0;
  for (int64_t t = g0 / W; t * W < g1 && n < kMaxUnits; ++t) {
    Unit u = {};
    u.t = (int32_t)t;
    const int64_t lo = g0 - t * W, hi = g1 - t * W;
    u.c0 = (int32_t)(lo > 0 ? lo : 0);
    u.c1 = (int32_t)(hi < W ? hi : W);
    if (u.c0 > 0 || u.c1 < W) {
      const int64_t slot = 2 * (int64_t)c + (u.c0 > 0 ? 0 : 1);
      u.partial = 1;
      u.part_row = slot * H * kHeadDim;
      u.part_hstride = kHeadDim;
      u.lse_row = slot * 2 * H;             // + rank * H
      u.lse_hstride = 1;
      auto g = [&](int64_t cc) { return total * cc / P.clusters; };
      int64_t first = c, last = c;          // the clusters holding the token's first and last column
      while (first > 0 && g(first) > t * W) --first;
      while (last + 1 < P.clusters && g(last + 1) < (t + 1) * W) ++last;
      u.merge_first = (int32_t)first;
      u.merge_n = (int32_t)(last - first + 1);
    }
    units[n++] = u;
  }
  return n;
}

// Step a2 for unit u, by kNW warps (warp index wi): index columns, token
// metadata, masks; compaction of [c0, c1) into list u & 1: valid SWA slots
// first, then valid compressed slots, each in column order; then publishes
// the unit (its first tile tile0) on unit_ready[u].  sync(i) joins the kNW
// warps (i = 0: chunk counts written, 1: list written) and returns false
// after an abort.  List u & 1 was last read by the gathers of unit u - 2,
// all issued before any warp reaches this compaction.
template <int kN, int kNW, class Sync>
__device__ __forceinline__ bool compact_unit(const DecodeParams& p, TcSmall& sm, int32_t* idx_s, int u, int tile0,
                                         int wi, int lane, uint32_t rank, Sync sync, int& o_nswa, int& o_nvalid) {
  constexpr int kChunksPerWarp = (kMaxChunks + kNW - 1) / kNW;
  Unit& U = sm.unit[u];
  const int t = U.t, c0 = U.c0;
  int c1 = U.c1;
  if (c1 - c0 > kMaxCols) {              // the planner prevents this; never write past the list
    if (p.err && wi == 0 && lane == 0) atomicOr(p.err, SMLA_DEVERR_INTERNAL);
    c1 = c0 + kMaxCols;
  }
  int32_t* list = idx_s + (u & 1) * kMaxCols;
  const int nchunks = (c1 - c0 + 31) / 32;
  int32_t rv[kChunksPerWarp];
  if (p.bt == nullptr) {                 // index form: independent loads, all in flight together
    const int32_t* irow = p.ind + (int64_t)t * p.ind_stride;
#pragma unroll
    for (int q = 0; q < kChunksPerWarp; ++q) {
      const int col = c0 + (wi + q * kNW) * 32 + lane;
      rv[q] = col < c1 ? __ldg(irow + col) : -1;
    }
  } else {                               // page-table form: compressed rows from the page table
    const int32_t* irow = p.ind + (int64_t)t * p.ind_stride;
#pragma unroll
    for (int q = 0; q < kChunksPerWarp; ++q) {
      const int col = c0 + (wi + q * kNW) * 32 + lane;
      rv[q] = -1;
      if (col < c1) rv[q] = col >= kSwaCols ? paged_row(p, t, col - kSwaCols) : __ldg(irow + col);
    }
  }
  const TokenInfo ti = token_info(p, t);
  c1 = min(c1, max(c0, ti.n_lim));     // active columns of the unit
#pragma unroll
  for (int q = 0; q < kChunksPerWarp; ++q) {
    const int k = wi + q * kNW;
    if (k < nchunks) {
      const int col = c0 + k * 32 + lane;
      const int idx = rv[q];
      rv[q] = -1;
      if (col < c1) {
        const bool swa = col < kSwaCols;
        bool valid = idx != -1 && (!swa || col < ti.w_swa);
        if (valid) {
          const int64_t nrows = swa ? p.swa_rows : p.comp_rows;
          if (idx < 0 || (int64_t)idx >= nrows) {
            valid = false;
            if (p.err && rank == 0) atomicOr(p.err, SMLA_DEVERR_INDEX_OUT_OF_RANGE);
          }
        }
        if (valid) rv[q] = idx;
      }
      const unsigned ball = __ballot_sync(0xffffffffu, rv[q] >= 0);
      const unsigned ball_swa = __ballot_sync(0xffffffffu, rv[q] >= 0 && col < kSwaCols);
      if (lane == 0) {
        sm.chunk_cnt[k] = __popc(ball);
        sm.chunk_swa[k] = __popc(ball_swa);
      }
    }
  }
  if (!sync(0)) return false;
  // every producer warp scans the chunk counts itself (at most 72)
  int chunk_base[kChunksPerWarp];
  int nvalid = 0, nswa = 0;
#pragma unroll
  for (int q = 0; q < kChunksPerWarp; ++q) chunk_base[q] = 0;
  for (int base0 = 0; base0 < nchunks; base0 += 32) {
    const int k = base0 + lane;
    const int v = k < nchunks ? sm.chunk_cnt[k] : 0;
    int sw = k < nchunks ? sm.chunk_swa[k] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int w = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, o);
#pragma unroll
    for (int q = 0; q < kChunksPerWarp; ++q) {
      const int kq = wi + q * kNW;
      const int excl = __shfl_sync(0xffffffffu, incl - v, kq & 31);
      if ((kq >> 5) == (base0 >> 5)) chunk_base[q] = nvalid + excl;
    }
    nvalid += __shfl_sync(0xffffffffu, incl, 31);
    nswa += sw;
  }
#pragma unroll
  for (int q = 0; q < kChunksPerWarp; ++q) {
    const int k = wi + q * kNW;
    if (k < nchunks) {
      const unsigned ball = __ballot_sync(0xffffffffu, rv[q] >= 0);
      if (rv[q] >= 0) list[chunk_base[q] + __popc(ball & ((1u << lane) - 1u))] = rv[q];
    }
  }
  if (!sync(1)) return false;   // the list is complete; the chunk counts are free
  if (wi == 0 && lane == 0) {
    U.nswa = nswa;
    U.nvalid = nvalid;
    const int tswa = (nswa + kN - 1) / kN, tcomp = (nvalid - nswa + kN - 1) / kN;
    U.ntiles = tswa + tcomp;
    U.tile0 = tile0;
    U.swa_tail = nswa - (tswa - 1) * kN;
    U.last_tail = tcomp > 0 ? nvalid - nswa - (tcomp - 1) * kN : U.swa_tail;
    mbar_arrive(smem_addr(&sm.unit_ready[u]));
  }
  o_nswa = nswa;
  o_nvalid = nvalid;
  return true;
}


template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ TcParams P) {
  using C = Cfg<kFp8>;
  const DecodeParams& p = P.p;
  constexpr int kN = C::kN;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_addr - raw_addr);
  TcSmall& sm = *reinterpret_cast<TcSmall*>(base + C::kOffSmall);
  int32_t* idx_s = reinterpret_cast<int32_t*>(base + C::kOffIdx);
  const uint32_t q_addr = base_addr + C::kOffQ;
  const uint32_t kv_addr = base_addr + C::kOffKV;
  const uint32_t x_addr = base_addr + C::kOffX;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const int H = p.H;

  auto bar = [&](const uint64_t& b) { return smem_addr(&b); };

  // ---------------------------------------------------------------- set-up
  int nswa0 = 0, nvalid0 = 0;               // unit 0's counts (every thread of the set-up's compaction has them)
  {
    if (tid == 0) {
      prefetch_tensormap(&P.tm_q);
      prefetch_tensormap(&P.tm_swa);
      prefetch_tensormap(&P.tm_comp);
      prefetch_tensormap(&P.tm_swa_run);
      prefetch_tensormap(&P.tm_comp_run);
    }
    // zero the KV stages (rows past a tile's slot count then hold finite
    // data) and the Q rows of absent heads (the Q box loads only H rows);
    // each thread orders its stores before later TMA writes to the same bytes
    const uint4 z = make_uint4(0, 0, 0, 0);
    uint4* zp = reinterpret_cast<uint4*>(base + C::kOffKV);
    const int zn = C::kStages * C::kStageBytes / 16;
    for (int i = tid; i < zn; i += kThreads) zp[i] = z;
    if (H < 128) {
      for (int kb = 0; kb < C::kRegions; ++kb) {
        uint4* qz = reinterpret_cast<uint4*>(base + C::kOffQ + kb * C::kRegionQ + H * 128);
        for (int i = tid; i < (128 - H) * 8; i += kThreads) qz[i] = z;
      }
    }
    fence_proxy_async_smem();
    if (tid == 0) {
      // the first unit's Q first: its load needs only the unit's token
      mbar_init(bar(sm.q_full), 1);
      fence_mbar_init_cluster();
      fence_proxy_async_smem();
      sm.nunits = make_units(P, blockIdx.x >> 1, sm.unit);
      if (sm.nunits > 0) {
        mbar_arrive_expect_tx(bar(sm.q_full), (uint32_t)(C::kRegions * H * 128));
        for (int kb = 0; kb < C::kRegions; ++kb)
          tma_load_3d(q_addr + kb * C::kRegionQ, &P.tm_q, (int)rank * kHalfDims + kb * (128 / C::kElem), 0,
                      sm.unit[0].t, bar(sm.q_full));
      }
      for (int i = 0; i < C::kStages; ++i) {
        mbar_init(bar(sm.kv_full[i]), 1);
        mbar_init(bar(sm.kv_empty[i]), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(bar(sm.p_full[b]), kSoftmaxWarps / 2);
        mbar_init(bar(sm.p_empty[b]), 1);
        mbar_init(bar(sm.xin_full[b]), 1);
        mbar_init(bar(sm.xout_free[b]), kSoftmaxWarps / 2);
        mbar_init(bar(sm.m_ready[b]), kSoftmaxWarps / 2);
      }
      for (int b = 0; b < kSBufs; ++b) {
        mbar_init(bar(sm.s_full[b]), 1);
        mbar_init(bar(sm.s_empty[b]), kSoftmaxWarps / 2 + kPushWarps);   // read by one softmax warpgroup and the push warps
      }
      for (int u = 0; u < kMaxUnits; ++u) mbar_init(bar(sm.unit_ready[u]), 1);
      mbar_init(bar(sm.prod_counts), kProducerWarps);
      mbar_init(bar(sm.prod_list), kProducerWarps);
      mbar_init(bar(sm.qk_first), 1);
      mbar_init(bar(sm.qk_unit_done), kQkWarps);
      mbar_init(bar(sm.lsum_full), kSoftmaxWarps);
      mbar_init(bar(sm.unit_pv_done), 1);
      mbar_init(bar(sm.o_free), kSoftmaxWarps);
      mbar_init(bar(sm.piece_sync), kSoftmaxWarps);
      mbar_init(bar(sm.epi_staged[0]), kSoftmaxWarps / 2);
      mbar_init(bar(sm.epi_staged[1]), kSoftmaxWarps / 2);
      mbar_init(bar(sm.piece_dec), 1);
      mbar_init(bar(sm.o_full), 1);
      mbar_init(bar(sm.qk_done), kQkWarps);
      sm.abort_flag = 0;
      fence_mbar_init_cluster();
    }
    if (warp == kMmaWarp) tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
    __syncthreads();
    // unit 0's index compaction by every warp, before the roles split
    if (sm.nunits > 0)
      compact_unit<kN, kThreads / 32>(p, sm, idx_s, 0, 0, warp, lane, rank, [](int) { __syncthreads(); return true; },
                                      nswa0, nvalid0);
    fence_proxy_async_smem();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
  }
  const uint32_t tmem = sm.tmem_base;
  const Ctx cx{&sm.abort_flag, p.err};
  const int nunits = sm.nunits;

  if (warp < kProducerWarps) {
    // ============================================================ producer
    // The four warps compact each unit's index columns together into a list
    // (two lists alternate), publish the unit, and gather its tiles.  Unit
    // u + 1 is compacted while unit u's tiles are in flight: for unit 0 after
    // its first ring of tiles is issued, for later units before their first
    // tile, when the ring is normally full of the previous unit's tiles.  A
    // warp's TMA requests are served one after another (about 40 ns per
    // gather4), so a tile's requests are spread over the two warps of its
    // group; two groups take alternate tiles.  A full tile of N consecutive
    // rows (a page run of the page-table form, or a run in the index table) is
    // one box copy per 128-byte column block instead.
    constexpr int kWarpsPerGroup = kProducerWarps / kProducerGroups;
    const int pg = warp / kWarpsPerGroup, pw = warp % kWarpsPerGroup;
    // units 1, 2, ... are compacted here (unit 0 in the set-up, by every warp)
    auto compact = [&](int u, int tile0, int& o_nswa, int& o_nvalid) -> bool {
      auto sync = [&](int i) {
        const uint32_t b = i == 0 ? bar(sm.prod_counts) : bar(sm.prod_list);
        __syncwarp();
        if (lane == 0) mbar_arrive(b);
        return warp_wait(cx, b, (u - 1) & 1);
      };
      return compact_unit<kN, kProducerWarps>(p, sm, idx_s, u, tile0, warp, lane, rank, sync, o_nswa, o_nvalid);
    };
    int next_j = pg;                         // the next tile this group issues (after the loop: past its last one)
    int nswa = nswa0, nvalid = nvalid0;      // the current unit's counts
    bool ok = true;
    int tile0 = 0;                           // the current unit's first tile
    for (int u = 0; ok && u < nunits; ++u) {
      const int tswa = (nswa + kN - 1) / kN;
      const int ntiles = tswa + (nvalid - nswa + kN - 1) / kN;
      const int32_t* list = idx_s + (u & 1) * kMaxCols;
      // tiles issued before the next unit's compaction: unit 0's first ring
      const int k_early = u == 0 ? C::kStages : 0;
      int nswa_next = 0, nvalid_next = 0;
      bool compacted = u + 1 >= nunits;
      // ---- gathers of the unit's tiles (global tile j = tile0 + k)
      for (;;) {
        if (!compacted && next_j - tile0 >= min(k_early, ntiles)) {
          if (!(ok = compact(u + 1, tile0 + ntiles, nswa_next, nvalid_next))) break;
          compacted = true;
        }
        if (next_j >= tile0 + ntiles) break;
        const int j = next_j, k = j - tile0;
        const int st = j % C::kStages;
        if (!(ok = warp_wait(cx, bar(sm.kv_empty[st]), ((j / C::kStages) & 1) ^ 1))) break;
        const int start = k < tswa ? k * kN : nswa + (k - tswa) * kN;
        const int n = min(kN, (k < tswa ? nswa : nvalid) - start);
        const int n4 = (n + 3) & ~3;           // gather4 moves four rows: the last row repeats
        if (pw == 0 && lane == 0) mbar_arrive_expect_tx(bar(sm.kv_full[st]), (uint32_t)(C::kRegions * n4 * 128));
        const uint32_t stage = kv_addr + st * C::kStageBytes;
        const int32_t* rows = list + start;
        bool run = false;                      // rows[r] == rows[0] + r for every r < N
        if (n == kN) {
          const uint32_t r0 = (uint32_t)rows[0];
          bool same = true;
#pragma unroll
          for (int r = lane; r < kN; r += 32) same = same && (uint32_t)rows[r] == r0 + (uint32_t)r;
          run = __all_sync(0xffffffffu, same);
        }
        if (run) {
          // every row of the box was checked against the pool's row count in the compaction
          const void* tmap = k < tswa ? static_cast<const void*>(&P.tm_swa_run) : static_cast<const void*>(&P.tm_comp_run);
          if (pw == 0 && lane < C::kRegions)
            tma_load_2d(stage + lane * C::kRegionKV, tmap, (int)rank * kHalfDims + lane * (128 / C::kElem), rows[0],
                        bar(sm.kv_full[st]));
        } else {
          const void* tmap = k < tswa ? static_cast<const void*>(&P.tm_swa) : static_cast<const void*>(&P.tm_comp);
          const int groups = (n4 / 4) * C::kRegions;
          for (int gi = pw + kWarpsPerGroup * lane; gi < groups; gi += kWarpsPerGroup * 32) {
            const int kb = gi % C::kRegions, r0 = (gi / C::kRegions) * 4;
            tma_gather4(stage + kb * C::kRegionKV + r0 * 128, tmap, (int)rank * kHalfDims + kb * (128 / C::kElem),
                        rows[r0], rows[min(r0 + 1, n - 1)], rows[min(r0 + 2, n - 1)], rows[min(r0 + 3, n - 1)],
                        bar(sm.kv_full[st]));
          }
        }
        next_j += kProducerGroups;
      }
      tile0 += ntiles;
      nswa = nswa_next;
      nvalid = nvalid_next;
    }
    // Leave no TMA write of this group in flight, also after an abort: wait
    // (bounded, not cut short by the abort flag) for the last tiles it issued,
    // at most one per stage.  Normally the consumers have waited for them.
    for (int jj = max(pg, next_j - C::kStages); jj < next_j; ++jj)
      if ((jj - pg) % kProducerGroups == 0) drain_wait(bar(sm.kv_full[jj % C::kStages]), (jj / C::kStages) & 1);
  } else if (warp < kSoftmaxWarp0) {
    regs_decrease<kRegsMma>();
    if (warp < kMmaWarp + kQkWarps) {
      // ============================================================ Q load and QK issue
      // QK and PV are issued by different warps so that a QK never waits behind
      // a PV (which waits for the softmax): the QK of tile j depends only on its
      // data, the unit's Q and a free S buffer.  The issuer of the unit's first
      // tile goes first and the others start once that QK has
      // completed (on a GB300 a QK issued by a second warp before the first one
      // finished gave wrong logits for some heads in repeated runs; observed,
      // cause not identified).
      constexpr uint32_t idesc_qk = idesc(kFp8, 128, kN, false);
      const int qi = warp - kMmaWarp;
      const uint32_t qbytes = (uint32_t)(C::kRegions * H * 128);
      // Q of token tq: the first unit's is loaded at the start of the set-up, a
      // later unit's by warp kMmaWarp once every QK of the previous unit that
      // used Q is done.  The first unit counts as using Q even when it has no
      // tile, so that every load is followed by one wait of every QK warp and
      // one commit of each (no parity wait can fall two phases behind or ahead).
      auto load_q = [&](int tq) {
        if (qi == 0 && lane == 0) {
          mbar_arrive_expect_tx(bar(sm.q_full), qbytes);
          for (int kb = 0; kb < C::kRegions; ++kb)
            tma_load_3d(q_addr + kb * C::kRegionQ, &P.tm_q, (int)rank * kHalfDims + kb * (128 / C::kElem), 0, tq,
                        bar(sm.q_full));
        }
        __syncwarp();
      };
      bool ok = true;
      int ne = 0;                              // units that used Q so far
      int nf = 0;                              // units with tiles so far
      for (int u = 0; ok && u < nunits; ++u) {
        if (!(ok = warp_wait(cx, bar(sm.unit_ready[u]), 0))) break;
        const int ntiles = sm.unit[u].ntiles, tile0 = sm.unit[u].tile0, t = sm.unit[u].t;
        if (ntiles == 0 && u > 0) continue;
        if (u > 0) {
          if (qi == 0 && !(ok = warp_wait(cx, bar(sm.qk_unit_done), (ne - 1) & 1))) break;
          load_q(t);
        }
        if (!(ok = warp_wait(cx, bar(sm.q_full), ne & 1))) break;
        const int first = (qi - tile0 % kSBufs + kSBufs) % kSBufs;   // this warp's first tile of the unit (local index)
        if (first > 0 && first < ntiles && !(ok = warp_wait(cx, bar(sm.qk_first), nf & 1))) break;
        for (int k = first; k < ntiles; k += kQkWarps) {
          const int j = tile0 + k;
          const int st = j % C::kStages;
          if (!(ok = warp_wait(cx, bar(sm.kv_full[st]), (j / C::kStages) & 1))) break;
          const int b = j % kSBufs;
          if (!(ok = warp_wait(cx, bar(sm.s_empty[b]), ((j / kSBufs) & 1) ^ 1))) break;
          fence_proxy_async_smem();
          tc_fence_after();
          if (lane == 0) {
            const uint32_t stage = kv_addr + st * C::kStageBytes;
  #pragma unroll
            for (int kk = 0; kk < C::kK1; ++kk) {
              const uint64_t a = desc_sw128(q_addr + (kk >> 2) * C::kRegionQ + (kk & 3) * 32, 16, 1024);
              const uint64_t kd = desc_sw128(stage + (kk >> 2) * C::kRegionKV + (kk & 3) * 32, 16, 1024);
              mma<kFp8>(tmem + kSCol + b * kN, a, kd, idesc_qk, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar(sm.s_full[b]));
            if (k == 0) mma_commit(bar(sm.qk_first));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) mma_commit(bar(sm.qk_unit_done));     // completes once every QK above is done
        __syncwarp();
        ++ne;
        if (ntiles > 0) ++nf;
      }
      if (lane == 0) mma_commit(bar(sm.qk_done));
      __syncwarp();
    } else {
      // ============================================================ PV issue
      constexpr uint32_t idesc_pv = idesc(kFp8, 128, kHalfDims, true);
      bool ok = true;
      for (int u = 0; ok && u < nunits; ++u) {
        if (!(ok = warp_wait(cx, bar(sm.unit_ready[u]), 0))) break;
        // the unit's first PV overwrites O: the previous unit's O must have been
        // read out (waited for every unit, so that this warp runs at most one
        // unit ahead of the epilogue)
        if (u > 0 && !(ok = warp_wait(cx, bar(sm.o_free), (u - 1) & 1))) break;
        const int ntiles = sm.unit[u].ntiles, tile0 = sm.unit[u].tile0;
        for (int k = 0; k < ntiles; ++k) {
          const int j = tile0 + k;
          const int b = j & 1, st = j % C::kStages;
          if (!(ok = warp_wait(cx, bar(sm.p_full[b]), (j >> 1) & 1))) break;
          tc_fence_after();
          if (lane == 0) {
            const uint32_t stage = kv_addr + st * C::kStageBytes;
  #pragma unroll
            for (int kk = 0; kk < C::kK2; ++kk) {
              const uint64_t v = desc_sw128(stage + kk * (C::kKStep / 8) * 1024, C::kRegionKV, 1024);
              mma_tmem_a<kFp8>(tmem + kOCol, tmem + C::kPCol + b * C::kPCols + kk * (C::kKStep * C::kElem / 4), v,
                               idesc_pv, (k > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(bar(sm.p_empty[b]));
            mma_commit(bar(sm.kv_empty[st]));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) mma_commit(bar(sm.unit_pv_done));     // completes once every PV of the unit is done
        __syncwarp();
      }
      if (lane == 0) mma_commit(bar(sm.o_full));    // completes once every PV issued above is done
      __syncwarp();
    }
  } else if (warp < kPushWarp0) {
    regs_increase<kRegsSoftmax>();
    // ============================================================ softmax / epilogue
    // Two warpgroups take turns: warpgroup g handles tiles j with j % 2 == g
    // (all N slots; S, P and exchange buffer g).  The only hand-off between
    // consecutive tiles of a unit is the running reference maximum m(j),
    // published by the warpgroup of tile j as soon as it is known, so one
    // warpgroup's exponentials overlap the other's loads.  The push warps
    // send this CTA's partial S to the peer.
    const int g = (warp - kSoftmaxWarp0) >> 2;        // warpgroup
    const int q4 = warp & 3;                           // TMEM lane quadrant of this warp
    const int h = q4 * 32 + lane;
    const bool active = q4 * 32 < H;                   // warp-uniform
    const bool leader = (warp - kSoftmaxWarp0) % 4 == 0 && lane == 0;   // one thread per warpgroup
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    const float c = load_scale(p.bmm1, p.bmm1_dev) * kLog2e;
    const uint32_t xbytes = (uint32_t)(H * kN * 3);    // bytes the peer pushes per tile (24-bit logits)
    const uint32_t xout_free_peer = map_to_rank(bar(sm.xout_free[g]), peer);
    const uint32_t p_cols = C::kPCol + g * C::kPCols;  // P buffer g
    // the output scales, loaded now so that their latency hides behind the first tile
    if (active)
      sm.epi[g][h] = make_float2(load_scale(p.bmm2, p.bmm2_dev), p.sinks ? __ldg(p.sinks + h) * kLog2e : 0.f);
    if (!active) {
      // rows of absent heads: P = 0, so O stays 0 there
      uint32_t zr[C::kPCols];
#pragma unroll
      for (int i = 0; i < C::kPCols; ++i) zr[i] = 0u;
      tmem_st16(tl + p_cols, zr);
      tmem_wait_st();
    }
    const uint64_t c2 = f2_pack(c, c);
    bool ok = true;
    int npiece = 0;                                    // balanced-mode pieces ended so far
    for (int u = 0; u < nunits; ++u) {
      if (ok) ok = warp_wait(cx, bar(sm.unit_ready[u]), 0);
      const Unit& U = sm.unit[u];
      const int ntiles = ok ? U.ntiles : 0, tile0 = U.tile0;
      const int jend = tile0 + ntiles, jswa = tile0 + (U.nswa + kN - 1) / kN;   // past the unit's last tile / SWA tile
      float m_last = -INFINITY, l_run = 0.f;            // reference and row sum of my warpgroup's tiles of the unit
      // E4M3 P keeps 3 mantissa bits: under a lagging reference a row's largest
      // P (up to 2^8) is rounded by up to 1/16, which shows when few slots carry
      // the mass, so short tile chains move the reference on every new maximum
      // (the same choice in both CTAs: ntiles is the pair's).
      const float thr = (kFp8 && ntiles <= kExactRefTiles) ? 0.f : kRescaleThreshold;
      const int first = (tile0 & 1) == g ? 0 : 1;        // my first tile of the unit (local index)
      for (int j = tile0 + first; ok && j < jend; j += 2) {   // j: tile number within the cluster's work
        // slots of tile j: N but for the unit's last SWA tile and its last tile
        // (read from shared memory where needed, which keeps them out of the
        // registers of the loop)
        const int n_cur = j == jswa - 1 ? *reinterpret_cast<volatile const int32_t*>(&U.swa_tail)
                        : j == jend - 1 ? *reinterpret_cast<volatile const int32_t*>(&U.last_tail) : kN;
        const int sb = j % kSBufs;
        // the peer's half of S(j) lands here: arm for its bytes (they may come first)
        if (leader) mbar_arrive_expect_tx(bar(sm.xin_full[g]), xbytes);
        // this CTA's half: S(j) from TMEM, then the S buffer is free for QK(j + 3)
        if (!(ok = warp_wait(cx, bar(sm.s_full[sb]), (j / kSBufs) & 1))) break;
        tc_fence_after();
        float sv[kN];
        if (active) {
#pragma unroll
          for (int hb = 0; hb < kN / 32; ++hb) {
            uint32_t r[32];
            tmem_ld32(tl + kSCol + sb * kN + hb * 32, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) sv[hb * 32 + i] = __uint_as_float(r[i]);
          }
          tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(sm.s_empty[sb]));
        if (!(ok = warp_wait(cx, bar(sm.xin_full[g]), (j >> 1) & 1, true))) break;
        float mt = -INFINITY;
        if (active) {
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
          if (n_cur >= kN) {
#pragma unroll
            for (int i = 0; i < kN; ++i) m4[i & 3] = fmaxf(m4[i & 3], sv[i]);
          } else {
#pragma unroll
            for (int i = 0; i < kN; ++i)
              if (i < n_cur) m4[i & 3] = fmaxf(m4[i & 3], sv[i]);
          }
          mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(xout_free_peer);   // exchange buffer g read out
        // ---- reference maximum: m(j) = mt if it exceeds m(j-1) by the threshold, else m(j-1)
        float m_prev = -INFINITY;
        if (j > tile0) {
          if (!(ok = warp_wait(cx, bar(sm.m_ready[g ^ 1]), ((j - 1) >> 1) & 1))) break;
          m_prev = sm.m_buf[g ^ 1][h];
        }
        const float m_cur = (mt > m_prev + thr) ? mt : m_prev;
        sm.m_buf[g][h] = m_cur;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(sm.m_ready[g]));
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
          if (n_cur < kN) {
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
        }
        // ---- O rescale when the reference moved (O holds the unit's tiles < j at m(j-1))
        const bool rescale = active && j > tile0 && m_cur != m_prev;
        if (__any_sync(0xffffffffu, rescale)) {
          if (!(ok = warp_wait(cx, bar(sm.p_empty[g ^ 1]), ((j - 1) >> 1) & 1))) break;   // PV(j - 1) done
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

      // ---- the unit's end: both warpgroups' row sums brought to the final reference
      const int ub = u & 1;
      if (active) {
        sm.lsum[ub][g][h] = l_run;
        sm.m_end[ub][g][h] = m_last;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(sm.lsum_full));
      if (ok) ok = warp_wait(cx, bar(sm.lsum_full), u & 1);
      if (ok) {
        ok = warp_wait(cx, bar(sm.unit_pv_done), u & 1);
        tc_fence_after();
      }
      float l_keep = 0.f, lse_keep = -INFINITY;          // this unit's row sum and LSE (for a piece merge)
      // The last unit's rows go out through shared memory (the KV stages are
      // free once its last PV is done): whole 256-byte row segments per half
      // warp instead of one 16-byte piece of 32 rows per warp instruction.
      const bool staged = u == nunits - 1;
      unsigned char* stg = base + C::kOffKV + g * (128 * 256);
      if (active) {
        float l_tot = 0.f, m_fin = -INFINITY;
        if (ok) {
          const float ma = sm.m_end[ub][0][h], mb = sm.m_end[ub][1][h];
          m_fin = fmaxf(ma, mb);
          if (m_fin != -INFINITY) {
            if (ma != -INFINITY) l_tot += sm.lsum[ub][0][h] * fast_exp2(ma - m_fin);
            if (mb != -INFINITY) l_tot += sm.lsum[ub][1][h] * fast_exp2(mb - m_fin);
          }
        }
        const bool have = ok && ntiles > 0 && l_tot > 0.f;
        const float lse = have ? m_fin + fast_log2(l_tot) : -INFINITY;
        float f = have ? 1.f / l_tot : 0.f;
        __nv_bfloat16* dst;
        if (!U.partial) {
          const float2 e = sm.epi[g][h];
          f *= e.x;
          if (p.sinks != nullptr && have) f *= 1.f / (1.f + fast_exp2(e.y - lse));
          dst = p.out + ((int64_t)U.t * H + h) * kHeadDim;
        } else {
          dst = (P.clusters ? P.piece_o : p.part_o) + U.part_row + (int64_t)h * U.part_hstride;
        }
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
          for (int q = 0; q < 4; ++q) {
            const uint4 x = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                       pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
            if (staged)   // 16-byte chunks XOR-swizzled by the row against bank conflicts
              *reinterpret_cast<uint4*>(stg + h * 256 + (((cc * 4 + q) ^ (h & 15)) << 4)) = x;
            else
              reinterpret_cast<uint4*>(dst + (int)rank * kHalfDims + col)[q] = x;
          }
        }
        if (!U.partial) {
          if (rank == 0 && g == 0 && p.out_lse) p.out_lse[(int64_t)U.t * H + h] = lse;
        } else if (P.clusters) {
          if (g == 0) P.piece_lse[U.lse_row + (int64_t)rank * H + h] = lse;   // each CTA its own copy
        } else {
          if (rank == 0 && g == 0) p.part_lse[U.lse_row + (int64_t)h * U.lse_hstride] = lse;
        }
        l_keep = l_tot;
        lse_keep = lse;
      }
      if (staged) {
        // copy-out of this warpgroup's 128 columns: half a warp per row
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(sm.epi_staged[g]));
        if (ok) ok = warp_wait(cx, bar(sm.epi_staged[g]), 0);
        if (ok) {
          __nv_bfloat16* row0 = U.partial ? (P.clusters ? P.piece_o : p.part_o) + U.part_row
                                          : p.out + (int64_t)U.t * H * kHeadDim;
          const int64_t rstride = U.partial ? U.part_hstride : kHeadDim;
          const int ch = lane & 15;
          for (int r = (warp & 3) * 2 + (lane >> 4); r < H; r += 8) {
            const uint4 x = *reinterpret_cast<const uint4*>(stg + r * 256 + ((ch ^ (r & 15)) << 4));
            *reinterpret_cast<uint4*>(row0 + r * rstride + (int)rank * kHalfDims + g * (kHalfDims / 2) + ch * 8) = x;
          }
        }
      }
      if (P.clusters && U.partial) {
        // A piece of a cut token: publish it (device-wide), count it, and if it
        // is the token's last piece to finish, merge all of them (this CTA's
        // half of the dims) into the output.
        __threadfence();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(sm.piece_sync));
        if (warp == kSoftmaxWarp0) {
          const bool all = ok && warp_wait(cx, bar(sm.piece_sync), npiece & 1);
          if (lane == 0) {
            sm.piece_last = all && atomicAdd(P.piece_cnt + 2 * U.merge_first + rank, 1u) == (uint32_t)(U.merge_n - 1);
            __threadfence();
            mbar_arrive(bar(sm.piece_dec));
          }
          __syncwarp();
        }
        if (ok) ok = warp_wait(cx, bar(sm.piece_dec), npiece & 1);
        ++npiece;
        if (ok && *reinterpret_cast<volatile int32_t*>(&sm.piece_last) && active) {
          __threadfence();
          const int own = (int)(U.part_row / ((int64_t)H * kHeadDim));   // this piece's slot
          const int nmerge = U.merge_n, first_c = U.merge_first;
          auto slot = [&](int k) { return k == 0 ? 2 * first_c + 1 : 2 * (first_c + k); };
          auto piece_row = [&](int k) {
            return P.piece_o + ((int64_t)slot(k) * H + h) * kHeadDim + (int)rank * kHalfDims + g * (kHalfDims / 2);
          };
          // the other pieces' 256-byte row segments into L1 while their LSEs load
          for (int k = 0; k < nmerge; ++k)
            if (slot(k) != own) {
              prefetch_l1(piece_row(k));
              prefetch_l1(piece_row(k) + 64);
            }
          // weights 2^(LSE_k - max) of every piece, this one from its fp32 O
          float mx = lse_keep;
          for (int k = 0; k < nmerge; ++k)
            if (slot(k) != own) mx = fmaxf(mx, __ldcg(P.piece_lse + ((int64_t)slot(k) * 2 + rank) * H + h));
          const float w_own = lse_keep == -INFINITY ? 0.f : fast_exp2(lse_keep - mx);
          float wsum = w_own;
          for (int k = 0; k < nmerge; ++k) {
            if (slot(k) == own) continue;
            const float lk = __ldcg(P.piece_lse + ((int64_t)slot(k) * 2 + rank) * H + h);
            wsum += lk == -INFINITY ? 0.f : fast_exp2(lk - mx);
          }
          const bool have_any = mx != -INFINITY && wsum > 0.f;
          const float lse_tot = have_any ? mx + fast_log2(wsum) : -INFINITY;
          const float2 e = sm.epi[g][h];
          float f = have_any ? e.x / wsum : 0.f;
          if (p.sinks != nullptr && have_any) f *= 1.f / (1.f + fast_exp2(e.y - lse_tot));
          const float f_own = l_keep > 0.f ? w_own / l_keep : 0.f;     // O (unnormalised) x this piece's weight
          __nv_bfloat16* out_row = p.out + ((int64_t)U.t * H + h) * kHeadDim + (int)rank * kHalfDims;
#pragma unroll 1
          for (int cc = 0; cc < kHalfDims / 64; ++cc) {
            const int col = g * (kHalfDims / 2) + cc * 32;
            float acc[32];
            {
              uint32_t r[32];
              tmem_ld32(tl + kOCol + col, r);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[i] = f_own != 0.f ? __uint_as_float(r[i]) * f_own : 0.f;
            }
            for (int k = 0; k < nmerge; ++k) {
              if (slot(k) == own) continue;
              const float lk = __ldcg(P.piece_lse + ((int64_t)slot(k) * 2 + rank) * H + h);
              if (lk == -INFINITY) continue;                          // an empty piece is all zero
              const float wk = fast_exp2(lk - mx);
              const uint4* src = reinterpret_cast<const uint4*>(piece_row(k) + cc * 32);
              uint4 x[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) x[q] = src[q];                // L1 hits after the prefetch
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint32_t xs[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float2 fv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[i]));
                  acc[8 * q + 2 * i] = fmaf(wk, fv.x, acc[8 * q + 2 * i]);
                  acc[8 * q + 2 * i + 1] = fmaf(wk, fv.y, acc[8 * q + 2 * i + 1]);
                }
              }
            }
            uint4* o = reinterpret_cast<uint4*>(out_row + col);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              o[q] = make_uint4(pack_bf16x2(acc[8 * q] * f, acc[8 * q + 1] * f), pack_bf16x2(acc[8 * q + 2] * f, acc[8 * q + 3] * f),
                                pack_bf16x2(acc[8 * q + 4] * f, acc[8 * q + 5] * f), pack_bf16x2(acc[8 * q + 6] * f, acc[8 * q + 7] * f));
          }
          if (rank == 0 && g == 0 && p.out_lse) p.out_lse[(int64_t)U.t * H + h] = lse_tot;
        }
      }
      // O read out: the next unit's first PV may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(sm.o_free));
    }
  } else {
    regs_decrease<kRegsPush>();
    // ============================================================ partial-S exchange
    // Warp kPushWarp0 + q sends lanes [32 q, 32 q + 32) of every tile's S (this
    // CTA's half of the logits, heads in TMEM lanes) to the peer's exchange
    // buffer j % 2 with st.async as 24-bit floats (four values in three words),
    // completing bytes on the peer's mbarrier, once the peer has read the
    // buffer's previous tile.  Tiles go in order, as soon as their QK is done.
    const int q4 = warp & 3;
    const int h = q4 * 32 + lane;
    const bool active = q4 * 32 < H;                   // warp-uniform
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t x_peer = map_to_rank(x_addr, peer) + (uint32_t)(h * 16);
    const uint32_t xin_full_peer = map_to_rank(bar(sm.xin_full[0]), peer);
    bool ok = true;
    for (int u = 0; ok && u < nunits; ++u) {
      if (!(ok = warp_wait(cx, bar(sm.unit_ready[u]), 0))) break;
      const int tile0 = sm.unit[u].tile0, jend = tile0 + sm.unit[u].ntiles;
      for (int j = tile0; j < jend; ++j) {
        const int g = j & 1, sb = j % kSBufs;
        if (!(ok = warp_wait(cx, bar(sm.s_full[sb]), (j / kSBufs) & 1))) break;
        tc_fence_after();
        if (j >= 2 && !(ok = warp_wait(cx, bar(sm.xout_free[g]), ((j >> 1) & 1) ^ 1, true))) break;
        if (active) {
          const uint32_t xb = x_peer + (uint32_t)(g * C::kXBytes);
          const uint32_t xbar = xin_full_peer + (uint32_t)(g * sizeof(uint64_t));
#pragma unroll
          for (int hh = 0; hh < kN / 32; ++hh) {
            uint32_t v[32];
            tmem_ld32(tl + kSCol + sb * kN + hh * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int hb = hh * 2 + half;             // 16-slot block
              // the low mantissa byte is dropped after rounding; values a, b,
              // c, d travel as [a1 a2 a3 d1] [b1 b2 b3 d2] [c1 c2 c3 d3]
              uint32_t w[12];
#pragma unroll
              for (int gq = 0; gq < 4; ++gq) {
                const int i = half * 16 + 4 * gq;
                const uint32_t d = v[i + 3] + 0x80u;
                w[3 * gq] = __byte_perm(v[i] + 0x80u, d, 0x5321);
                w[3 * gq + 1] = __byte_perm(v[i + 1] + 0x80u, d, 0x6321);
                w[3 * gq + 2] = __byte_perm(v[i + 2] + 0x80u, d, 0x7321);
              }
#pragma unroll
              for (int q = 0; q < 3; ++q)
                st_async_v4(xb + (uint32_t)((hb * 3 + q) * 128 * 16), __uint_as_float(w[4 * q]),
                            __uint_as_float(w[4 * q + 1]), __uint_as_float(w[4 * q + 2]),
                            __uint_as_float(w[4 * q + 3]), xbar);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(sm.s_empty[sb]));   // S buffer sb read
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static cudaError_t encode_fn(EncodeTiledFn* out) {
  static std::atomic<EncodeTiledFn> cached{nullptr};   // looked up once; callers may be on several threads
  EncodeTiledFn fn = cached.load(std::memory_order_acquire);
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || ptr == nullptr) return cudaErrorNotSupported;
    fn = reinterpret_cast<EncodeTiledFn>(ptr);
    cached.store(fn, std::memory_order_release);
  }
  *out = fn;
  return cudaSuccess;
}

// [rows, 512] pool view; box 128 bytes x box_rows rows; 128-byte swizzle.
cudaError_t encode_pool_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_stride, int dtype,
                            int box_rows) {
  EncodeTiledFn fn = nullptr;
  cudaError_t e = encode_fn(&fn);
  if (e != cudaSuccess) return e;
  const int elem = dtype == SMLA_BF16 ? 2 : 1;
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {(cuuint64_t)(row_stride * elem)};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / elem), (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype == SMLA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The query as [T, H, 512] (heads 512 elements apart, tokens q_stride_token
// apart); box 128 bytes x H heads x 1 token; 128-byte swizzle.  The call's
// checks make q 16-byte aligned and q_stride_token a multiple of 16 bytes.
static cudaError_t encode_query_map(CUtensorMap* map, const DecodeParams& p) {
  EncodeTiledFn fn = nullptr;
  cudaError_t e = encode_fn(&fn);
  if (e != cudaSuccess) return e;
  const int elem = p.dtype == SMLA_BF16 ? 2 : 1;
  const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)p.H, (cuuint64_t)(p.sum_q > 0 ? p.sum_q : 1)};
  const cuuint64_t strides[2] = {(cuuint64_t)(kHeadDim * elem), (cuuint64_t)(p.q_stride_token * elem)};
  const cuuint32_t box[3] = {(cuuint32_t)(128 / elem), (cuuint32_t)p.H, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, p.dtype == SMLA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                  const_cast<void*>(p.q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int tc_smem_bytes(int dtype) { return dtype == SMLA_BF16 ? Cfg<false>::kSmemBytes : Cfg<true>::kSmemBytes; }
int tc_threads() { return kThreads; }

cudaError_t launch_decode_tc(const DecodeParams& p, int grid, int clusters, __nv_bfloat16* piece_o, float* piece_lse,
                             uint32_t* piece_cnt, cudaStream_t stream) {
  TcParams P;
  memset(&P, 0, sizeof(P));
  P.p = p;
  P.clusters = clusters;
  P.piece_o = piece_o;
  P.piece_lse = piece_lse;
  P.piece_cnt = piece_cnt;
  // a pool of fewer than N rows holds no run of N rows: its run map is never used
  const int64_t run_rows = p.dtype == SMLA_BF16 ? Cfg<false>::kN : Cfg<true>::kN;
  const int swa_run = (int)std::max<int64_t>(1, std::min(run_rows, p.swa_rows));
  const int comp_run = (int)std::max<int64_t>(1, std::min(run_rows, p.comp_rows));
  cudaError_t e = encode_pool_map(&P.tm_swa, p.swa, p.swa_rows, p.swa_stride, p.dtype, 1);
  if (e == cudaSuccess) e = encode_pool_map(&P.tm_comp, p.comp, p.comp_rows, p.comp_stride, p.dtype, 1);
  if (e == cudaSuccess) e = encode_pool_map(&P.tm_swa_run, p.swa, p.swa_rows, p.swa_stride, p.dtype, swa_run);
  if (e == cudaSuccess) e = encode_pool_map(&P.tm_comp_run, p.comp, p.comp_rows, p.comp_stride, p.dtype, comp_run);
  if (e == cudaSuccess) e = encode_query_map(&P.tm_q, p);
  if (e != cudaSuccess) return e;
  const int smem = tc_smem_bytes(p.dtype);
  auto launch = [&](auto kernel) -> cudaError_t {
    // The softmax warpgroups' setmaxnreg.inc waits for registers that the
    // launch must hold: refuse to launch a build whose per-thread count is
    // below the one the split was sized for (the wait would never end).
    static std::atomic<int> launch_regs[2];            // per kernel (BF16, E4M3); 0 = not queried yet
    std::atomic<int>& cached = launch_regs[p.dtype == SMLA_BF16 ? 0 : 1];
    int regs = cached.load(std::memory_order_relaxed);
    if (regs == 0) {
      cudaFuncAttributes fa;
      cudaError_t err = cudaFuncGetAttributes(&fa, kernel);
      if (err != cudaSuccess) return err;
      regs = fa.numRegs;
      cached.store(regs, std::memory_order_relaxed);
    }
    if (regs < kLaunchRegs) return cudaErrorInvalidConfiguration;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    kernel<<<grid, kThreads, smem, stream>>>(P);
    return cudaSuccess;
  };
  e = p.dtype == SMLA_BF16 ? launch(decode_tc_kernel<false>) : launch(decode_tc_kernel<true>);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace smla
