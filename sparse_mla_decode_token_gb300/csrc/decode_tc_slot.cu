// tcgen05 / TMEM sparse MLA decode kernel for E4M3 rows, slot-split pair
// (sm_103a).
//
// Work unit: one (token, split) on a cluster of two CTAs, as in the grid
// kernel (decode_tc_grid.cu).  An fp32 accumulator for 128 heads x 512 dims
// fills the whole tensor memory of one SM, so CTA r still keeps output dims
// [256 r, 256 r + 256) of every head; but the logits are split by slot, not
// by dim.  A tile is up to 128 selected slots; CTA r owns the tile's slots
// [64 r, 64 r + 64), gathers their full rows and computes their logits over
// all 512 dims, so no partial logits cross between the CTAs:
//
//   producer warps 0-3  the own slots' full rows (four 128-byte column
//                       blocks) with TMA tile::gather4 into 128-byte-swizzled,
//                       UMMA-canonical tiles: this CTA's output half into an
//                       entry of the V ring, the peer's half into one of the
//                       K ring (rings below); the tile's 64 requests spread
//                       over the four warps; 64 consecutive rows are one box
//                       copy per column block
//   QK warps 4-5        warp 4 first copies the peer's output half of the
//                       landed own rows (16 KB) into the peer's stage with one
//                       DSMEM bulk copy, then S_r = Q K_own^T (M = 128 heads, N = 64 own
//                       slots, K = 512 dims; Q is read from tensor memory):
//                       warp 4 + q issues the eight MMAs of dims
//                       [256 q, 256 q + 256) into half q of the TMEM S area,
//                       so a tile's QK runs as two chains that the softmax adds
//   PV warp 7           O_r += P V_r (M = 128 heads, N = 256 output dims, K =
//                       128 slots): P from shared memory (this CTA's half
//                       written by its softmax, the peer's half copied in), V
//                       of the own slots from the stage, V of the peer's slots
//                       from the peer's copy
//   softmax warps 8-15  two warpgroups taking whole tiles in turn, one thread
//                       per head: read the own slots' logits, send the per-head
//                       tile maximum to the peer (4 bytes, st.async) and take
//                       the peer's, settle the running reference maximum m(j)
//                       (the same in both CTAs), P = 2^(x - m(j)) in E4M3 into
//                       shared memory, whose 8 KB half one thread then copies
//                       to the peer (DSMEM bulk copy); lazy rescaling of O;
//                       finally the two CTAs' row sums (each over its own
//                       slots) meet once, O is normalised and stored
//
// Per 128 slots each CTA sends 16 KB of rows, 8 KB of P and 512 bytes of
// maxima to its peer, against 48 KB of 24-bit partial logits in the dims-split
// kernel, and runs the exponentials of its own 64 slots only.
//
// kPair (64 heads): a unit holds two tokens, their heads in MMA rows 0-63 and
// 64-127, over the union of their selected rows (built in the set-up, see
// kPairCols); each softmax row masks the other token's entries.  The P halves
// and maxima already carry 128 rows, so the second token's heads travel free
// and the per-unit fixed cost is paid once per two tokens.
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

constexpr int kNH = 64;                          // own slots per CTA per tile
constexpr int kNT = 2 * kNH;                     // slots per tile (the pair's)
constexpr int kHalfDims = 256;                   // output dims per CTA
constexpr int kProducerWarps = 4;
constexpr int kMmaWarp = kProducerWarps;         // first QK issuer; allocates and frees TMEM
constexpr int kQkWarps = 2;                      // one per half of the QK (K steps 0-7, 8-15); warp 6 has no role
constexpr int kPvWarp = 7;
constexpr int kSoftmaxWarp0 = 8;
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = (kSoftmaxWarp0 + kSoftmaxWarps) * 32;
constexpr int kWarps = kThreads / 32;
// Registers per thread of each warpgroup after the role split (setmaxnreg):
// the launch gives every thread kLaunchRegs; the producer and MMA warpgroups
// hand registers back, the two softmax warpgroups take them.
constexpr int kLaunchRegs = 65536 / kThreads / 8 * 8;
constexpr int kRegsProducer = 80;
constexpr int kRegsMma = 56;
constexpr int kRegsSoftmax = 184;
static_assert(128 * (kRegsProducer + kRegsMma) + 256 * kRegsSoftmax <= kThreads * kLaunchRegs,
              "the warpgroups' registers after the split fit in what the launch holds");
static_assert(kProducerWarps == 4 && kSoftmaxWarp0 == 8, "roles are whole warpgroups");
constexpr int kMaxCols = SMLA_TC_MAX_SPLIT_COLS;
constexpr int kMaxChunks = kMaxCols / 32;
constexpr int kChunksPerWarp = (kMaxChunks + kWarps - 1) / kWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;                    // O: 256 fp32 columns
constexpr uint32_t kQCol = 256;                  // Q: 128 columns of four E4M3 values (dims 4c .. 4c + 3)
constexpr uint32_t kSCol = 384;                  // S: a tile's two partial logits (64 fp32 columns each)
constexpr int kSBufs = 2;                        // s_full / s_empty barrier sets, one per softmax warpgroup
static_assert(kQkWarps == 2, "one QK issuer per half of the S area");
static_assert(kSCol + kSBufs * kNH == kTmemCols, "tensor memory budget");
constexpr float kRescaleThreshold = 8.f;         // log2 units: P stays <= 2^8
constexpr int kExactRefSlots = 512;              // E4M3 P: splits of at most this many slots follow the exact maximum
// Three rings of 16 KB entries (64 rows x two 128-byte column blocks), each
// released as soon as its last reader is done:
//   V ring  the own rows' blocks of this CTA's output half: QK and the PV of the own slots
//   K ring  the own rows' blocks of the peer's output half: QK and the copy to the peer
//   R ring  the peer's rows, this CTA's output half (the peer's copy): the PV of the peer's slots
constexpr int kRegion = kNH * 128;               // one 128-byte column block of 64 rows
constexpr int kEntry = 2 * kRegion;
constexpr int kNV = 4, kNK = 3, kNR = 4;
constexpr int kPHalf = 128 * kNH;                // P of one CTA's 64 slots: 128 rows x 64 bytes
constexpr int kPBytes = 2 * kPHalf;              // one P buffer (the tile's 128 slots)
constexpr int kOffV = 0;
constexpr int kOffK = kOffV + kNV * kEntry;
constexpr int kOffR = kOffK + kNK * kEntry;
constexpr int kOffP = kOffR + kNR * kEntry;
constexpr int kQStageBytes = 128 * 512;          // Q rows staged in the R ring during the set-up
static_assert(kNR * kEntry >= kQStageBytes, "Q staging fits in the R ring");
constexpr int kOffIdx = kOffP + 2 * kPBytes;
constexpr int kOffSmall = kOffIdx + kMaxCols * 4;
// Token pairs (H = 64): a unit holds two tokens (heads in MMA rows 0-63 and
// 64-127) over the union of their selected rows, each token at most
// kPairCols columns per split so that the union fits the kMaxCols list.  The
// union is built in the set-up with scratch in the V and K rings: a hash of
// token A's rows (keys, A's list indices), each token's compacted list, one
// membership byte per union entry, and one "B selects it too" byte per entry
// of A's list.
constexpr int kPairCols = kMaxCols / 2;
constexpr int kPairTiles = kMaxCols / kNT + 2;   // the SWA and compressed runs may each end in a partial tile
constexpr int kPairHash = 4096;                  // > kMaxCols: probing always ends
constexpr int kScrVals = kPairHash * 4;
constexpr int kScrListA = 2 * kPairHash * 4;
constexpr int kScrListB = kScrListA + kPairCols * 4;
constexpr int kScrMemb = kScrListB + kPairCols * 4;
constexpr int kScrShared = kScrMemb + kMaxCols;
static_assert(kScrShared + kPairCols <= kOffR - kOffV, "token-pair scratch fits in the V and K rings");
constexpr uint32_t kBarStride = (uint32_t)sizeof(uint64_t);

struct TcSmall {
  uint64_t kv_full[kNV];                 // tile j's own rows (V and K entries) landed
  uint64_t v_empty[kNV];                 // this CTA's PV of the entry's tile (own slots) done
  uint64_t k_empty[kNK];                 // this CTA's QK done, and the peer saw the copy land (remote)
  uint64_t r_full[kNR];                  // the peer's copy landed
  uint64_t r_empty[kNR];                 // this CTA's PV of the entry's tile (the peer's slots) done
  uint64_t r_free[kNR];                  // the peer's R entry may take this CTA's copy (remote)
  uint64_t r_seen[kNR];                  // the QK warp of the entry's tile has seen the copy land
  uint64_t s_full[kSBufs], s_empty[kSBufs];
  uint64_t p_ready[2];                   // P half of warpgroup g written by its four warps
  uint64_t pin_full[2];                  // both halves of P buffer g in place
  uint64_t p_empty[2];                   // PV of P buffer g done
  uint64_t pout_free[2];                 // the peer's PV of its P buffer g done
  uint64_t mx_full[2][2];                // the peer's tile maxima [warpgroup][(j >> 1) & 1]
  uint64_t m_ready[2];
  uint64_t lsum_full;
  uint64_t l_full;                       // the peer's row sums
  uint64_t o_full;
  uint64_t qk0_done;
  uint64_t qk_done;
  uint64_t mask_a[kPairTiles];           // token pairs: this CTA's own entries of tile j that token A selects
  uint64_t mask_b[kPairTiles];           //              ... and token B
  float mx[2][2][128];
  float lpeer[128];
  float m_end[2][128];
  float m_buf[2][128];
  float lsum[2][128];
  int32_t chunk_off[kMaxChunks];
  int32_t nswa;
  int32_t nvalid;
  // token pairs: token B's chunk counts, the chunk counts of B's rows that
  // token A does not select, and the per-token list sizes
  int32_t chunk_off_b[kMaxChunks];
  int32_t only_b_chunk[kMaxChunks];
  int32_t nswa_a, nswa_b, n_a, n_b, only_b_swa, dup;
  uint32_t tmem_base;
  int32_t abort_flag;
};

constexpr int kSmemBytes = kOffSmall + (int)sizeof(TcSmall) + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kNV * kEntry == 2 * 128 * 256, "BF16 partial staging: the V ring holds 128 rows x 256 bytes per warpgroup");
static_assert(kOffR == kOffK + kNK * kEntry && kOffK == kOffV + kNV * kEntry, "the set-up zeroes the V and K rings in one sweep");
static_assert(kEntry % 1024 == 0 && kPBytes % 1024 == 0, "swizzle atoms");

// Kernel parameters: the shared decode parameters plus two TMA descriptors per
// KV pool ([rows, 512] with the pool's row stride; 128-byte swizzle): box =
// 128 bytes x 1 row for tile::gather4, and 128 bytes x 64 rows for runs.
struct SlotParams {
  CUtensorMap tm_swa;
  CUtensorMap tm_comp;
  CUtensorMap tm_swa_run;
  CUtensorMap tm_comp_run;
  DecodeParams p;
};

// kPartial: split partials (num_splits > 1).  kPair: H = 64 and a unit is
// (token pair, split), see kPairCols.
template <bool kPartial, bool kPair>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_tc_slot_kernel(const __grid_constant__ SlotParams P) {
  const DecodeParams& p = P.p;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_addr - raw_addr);
  TcSmall& sm = *reinterpret_cast<TcSmall*>(base + kOffSmall);
  int32_t* idx_s = reinterpret_cast<int32_t*>(base + kOffIdx);
  const uint32_t v_addr = base_addr + kOffV;
  const uint32_t k_addr = base_addr + kOffK;
  const uint32_t r_addr = base_addr + kOffR;
  const uint32_t p_addr = base_addr + kOffP;

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
  // column range of this split (the grid kernel's rule)
  int per_split = (p.W + S - 1) / S;
  if (p.bt) per_split = (per_split + kNH - 1) / kNH * kNH;
  const int c0 = min(p.W, s * per_split);
  int c1 = min(p.W, c0 + per_split);
  if (c1 - c0 > (kPair ? kPairCols : kMaxCols)) {   // the planner prevents this
    if (p.err && tid == 0) atomicOr(p.err, SMLA_DEVERR_INTERNAL);
    c1 = c0 + (kPair ? kPairCols : kMaxCols);
  }

  auto bar = [&](const uint64_t& b) { return smem_addr(&b); };

  // ---------------------------------------------------------------- set-up
  const bool softmax_warp = warp >= kSoftmaxWarp0;
  const int g_sm = softmax_warp ? (warp - kSoftmaxWarp0) >> 2 : 0;
  // the split's index columns first: they lead to the first gathers, while Q
  // is needed only by the first QK
  const int nchunks = (c1 - c0 + 31) / 32;
  auto load_cols = [&](int tok, int32_t (&r)[kChunksPerWarp]) {
    const int32_t* irow = p.ind + (int64_t)tok * p.ind_stride;
    if (p.bt == nullptr) {
#pragma unroll
      for (int q = 0; q < kChunksPerWarp; ++q) {
        const int col = c0 + (warp + q * kWarps) * 32 + lane;
        r[q] = (col < c1) ? __ldg(irow + col) : -1;
      }
    } else {
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
  // Q rows staged in the R ring (free until the set-up's cluster barrier):
  // row h at 512 h, its 16-byte chunk c at chunk position c ^ (h % 32) so
  // that the per-head reads below spread over the banks (a token pair: MMA
  // row h is head h & 63 of token t + (h >> 6))
  for (int c = tid; c < rows_used * 32; c += kThreads) {
    const int h = c >> 5, cc = c & 31;
    const unsigned char* qrow = reinterpret_cast<const unsigned char*>(p.q) +
                                (int64_t)(kPair ? t + (h >> 6) : t) * p.q_stride_token;
    cp_async_16(r_addr + h * 512 + ((cc ^ (h & 31)) << 4), qrow + (int64_t)(kPair ? h & 63 : h) * kHeadDim + cc * 16);
  }
  const TokenInfo ti = token_info(p, t);
  const int c1b_full = c1;
  c1 = min(c1, max(c0, ti.n_lim));
  int c1b = c0, w_swa_b = 0;
  if (has_b) {
    const TokenInfo tib = token_info(p, t + 1);
    c1b = min(c1b_full, max(c0, tib.n_lim));
    w_swa_b = tib.w_swa;
  }
  {
    // P rows of absent heads must read 0 (the softmax writes only the rows
    // of present heads).  The V and K rings are not zeroed whole: rows past
    // a tile's slot count must only be finite, which every row a gather has
    // written is, so only those rows of an entry's first use are zeroed,
    // once the tiles are known (below; the R ring's entries are copies of
    // the peer's K entries)
    if (rows_used < 128) {
      const uint4 z = make_uint4(0, 0, 0, 0);
      uint4* zp = reinterpret_cast<uint4*>(base + kOffP);
      for (int i = tid; i < 2 * kPBytes / 16; i += kThreads) zp[i] = z;
    }
    uint32_t* hkeys = reinterpret_cast<uint32_t*>(base + kOffV);              // token pairs: set-up scratch
    int32_t* hvals = reinterpret_cast<int32_t*>(base + kOffV + kScrVals);
    int32_t* list_a = reinterpret_cast<int32_t*>(base + kOffV + kScrListA);
    int32_t* list_b = reinterpret_cast<int32_t*>(base + kOffV + kScrListB);
    uint8_t* memb = base + kOffV + kScrMemb;
    uint8_t* shared_a = base + kOffV + kScrShared;
    if constexpr (kPair) {
      const uint4 e4 = make_uint4(kPairEmpty, kPairEmpty, kPairEmpty, kPairEmpty), z = make_uint4(0, 0, 0, 0);
      for (int i = tid; i < kPairHash / 4; i += kThreads) reinterpret_cast<uint4*>(hkeys)[i] = e4;
      for (int i = tid; i < kPairCols / 16; i += kThreads) reinterpret_cast<uint4*>(shared_a)[i] = z;
      for (int i = tid; i < 2 * kPairTiles; i += kThreads) sm.mask_a[i] = 0ull;   // mask_b follows mask_a
    }
    if (tid == 0) {
      for (int i = 0; i < kNV; ++i) {
        mbar_init(bar(sm.kv_full[i]), 1);
        mbar_init(bar(sm.v_empty[i]), 1);
      }
      for (int i = 0; i < kNK; ++i) mbar_init(bar(sm.k_empty[i]), 3);   // two QK halves + the peer's acknowledgement
      for (int i = 0; i < kNR; ++i) {
        mbar_init(bar(sm.r_full[i]), 1);
        mbar_init(bar(sm.r_empty[i]), 1);
        mbar_init(bar(sm.r_free[i]), 1);
        mbar_init(bar(sm.r_seen[i]), 1);
      }
      for (int b = 0; b < kSBufs; ++b) {
        mbar_init(bar(sm.s_full[b]), kQkWarps);   // one commit per QK half
        mbar_init(bar(sm.s_empty[b]), kSoftmaxWarps / 2);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(bar(sm.p_ready[b]), kSoftmaxWarps / 2);
        mbar_init(bar(sm.pin_full[b]), 1);
        mbar_init(bar(sm.p_empty[b]), 1);
        mbar_init(bar(sm.pout_free[b]), kSoftmaxWarps / 2);
        mbar_init(bar(sm.mx_full[b][0]), 1);
        mbar_init(bar(sm.mx_full[b][1]), 1);
        mbar_init(bar(sm.m_ready[b]), kSoftmaxWarps / 2);
      }
      mbar_init(bar(sm.lsum_full), kSoftmaxWarps);
      mbar_init(bar(sm.l_full), 1);
      mbar_init(bar(sm.o_full), 1);
      mbar_init(bar(sm.qk0_done), 1);
      mbar_init(bar(sm.qk_done), kQkWarps);
      sm.abort_flag = 0;
      sm.nswa = 0;
      sm.nswa_a = sm.nswa_b = sm.only_b_swa = sm.dup = 0;
      fence_mbar_init_cluster();
    }
    if (warp == kMmaWarp) {
      tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
      tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
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
    // per-chunk valid counts of this warp's chunks (k = warp + q * kWarps)
    // and the valid SWA slots, for one token's loaded columns (valid rows
    // stay in r)
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
    // every warp scans the chunk counts itself: lane L sums chunks 3L .. 3L + 2
    // (3 x 32 >= kMaxChunks), one shuffle ladder over the lanes, and each of
    // the warp's chunks reads its base from the lane that holds it; returns
    // the total
    static_assert(3 * 32 >= kMaxChunks, "three chunks per lane");
    auto scan_chunks = [&](const int32_t* cnt, int nch, int (&chunk_base)[kChunksPerWarp]) -> int {
      const int k3 = 3 * lane;
      const int e0 = k3 < nch ? cnt[k3] : 0;
      const int e1 = k3 + 1 < nch ? cnt[k3 + 1] : 0;
      const int e2 = k3 + 2 < nch ? cnt[k3 + 2] : 0;
      const int own = e0 + e1 + e2;
      int incl = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
#pragma unroll
      for (int q = 0; q < kChunksPerWarp; ++q) {
        const int kq = warp + q * kWarps;              // warp-uniform
        const int src = min(kq / 3, 31), r = kq - 3 * src;
        const int ex = __shfl_sync(0xffffffffu, incl - own, src);
        const int a0 = __shfl_sync(0xffffffffu, e0, src);
        const int a1 = __shfl_sync(0xffffffffu, e1, src);
        chunk_base[q] = ex + (r >= 1 ? a0 : 0) + (r >= 2 ? a1 : 0);
      }
      return __shfl_sync(0xffffffffu, incl, 31);
    };
    if constexpr (!kPair) {
      // compaction of the split's columns [c0, c1) into idx_s: valid SWA
      // slots first, then valid compressed slots, each in column order
      count_chunks(rv, c1, ti.w_swa, sm.chunk_off, &sm.nswa);
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
    } else {
      // f1, the rows shared by a pair's tokens gathered once (as in the
      // token-pair form of the dims-split kernel): both tokens compacted,
      // every valid (pool, row) hashed with a flag per token, and the union
      //   [A SWA] [B-only SWA] [A compressed] [B-only compressed]
      // built in B's order by ballot scans, so both CTAs build the same list;
      // a token that selects a row twice makes the unit share nothing.
      count_chunks(rv, c1, ti.w_swa, sm.chunk_off, &sm.nswa_a);
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
              pair_insert_a<kPairHash>(hkeys, hvals, &sm.dup, pair_key(rv[q], e >= nswa_a), e);
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
              const int ia = pair_claim_a<kPairHash>(hkeys, hvals, &sm.dup, pair_key(list_b[i], i >= nswa_b));
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
      if (dup && !dup_a) {                 // B repeats a shared row: share nothing after all
        if (tid == 0) sm.only_b_swa = 0;
        __syncthreads();
        count_only_b(true);
        __syncthreads();
      }
      const int bs = sm.only_b_swa;        // B-only SWA entries (they come first in B's order)
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
        // this CTA's own entries of every 128-entry tile: bit i of mask_x[j]
        // is own entry i (list entry tile_start(j) + 64 rank + i)
        const int nsw = sm.nswa, nva = sm.nvalid;
        const int tsw = (nsw + kNT - 1) / kNT;
        const int nt = tsw + (nva - nsw + kNT - 1) / kNT;
        for (int j = warp; j < nt; j += kWarps) {
          const int start = (j < tsw ? j * kNT : nsw + (j - tsw) * kNT) + kNH * (int)rank;
          const int n = max(0, min(kNH, (j < tsw ? nsw : nva) - start));
          uint64_t ma = 0ull, mb = 0ull;
#pragma unroll
          for (int hb = 0; hb < kNH / 32; ++hb) {
            const int i = hb * 32 + lane;
            const uint32_t m = i < n ? memb[start + i] : 0u;
            ma |= (uint64_t)__ballot_sync(0xffffffffu, (m & 1u) != 0u) << (32 * hb);
            mb |= (uint64_t)__ballot_sync(0xffffffffu, (m & 2u) != 0u) << (32 * hb);
          }
          if (lane == 0) {
            sm.mask_a[j] = ma;
            sm.mask_b[j] = mb;
          }
        }
      }
    }
    // Q into tensor memory: softmax warp (g, quadrant) writes dims
    // [256 g, 256 g + 256) of its 32 heads (64 columns); absent heads get 0
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (!softmax_warp) {
      // first use of a V or K entry by a partial tile: rows [n4, 64) of its
      // column blocks must be finite (they meet P = 0 in the PV, and the K
      // entry travels to the peer); later uses find rows an earlier tile
      // wrote there.  n4 = the tile's own slots rounded up to 4 (gather4).
      const int nsw = sm.nswa, nva = sm.nvalid;
      const int tsw = (nsw + kNT - 1) / kNT;
      const int nt = tsw + (nva - nsw + kNT - 1) / kNT;
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int j = 0; j < kNV; ++j) {
        const int start = j < tsw ? j * kNT : nsw + (j - tsw) * kNT;
        const int n = j < nt ? max(0, min(kNH, min(kNT, (j < tsw ? nsw : nva) - start) - kNH * (int)rank)) : kNH;
        const int n4 = (n + 3) & ~3;
        if (n4 >= kNH) continue;
        const int per_block = (kNH - n4) * 8;            // 16-byte chunks per column block
        for (int i = tid; i < 4 * per_block; i += kSoftmaxWarp0 * 32) {
          const int kb = i / per_block, c = i % per_block;
          if (kb >= 2 && j >= kNK) continue;
          unsigned char* blk = kb < 2 ? base + kOffV + j * kEntry + kb * kRegion
                                      : base + kOffK + j * kEntry + (kb - 2) * kRegion;
          reinterpret_cast<uint4*>(blk + n4 * 128)[c] = z;
        }
      }
    }
    if (softmax_warp) {
      const int h = (warp & 3) * 32 + lane;
      const unsigned char* qs = base + kOffR + h * 512;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int cc = g_sm * 16 + half * 8 + i;
          const uint4 x = h < rows_used ? *reinterpret_cast<const uint4*>(qs + ((cc ^ (h & 31)) << 4)) : make_uint4(0, 0, 0, 0);
          r[4 * i] = x.x;
          r[4 * i + 1] = x.y;
          r[4 * i + 2] = x.z;
          r[4 * i + 3] = x.w;
        }
        tmem_st32(sm.tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + kQCol + 64 * g_sm + 32 * half, r);
      }
      tmem_wait_st();
    }
    // the zeroed rows are read by the tensor core, the staged Q's area is
    // overwritten by the peer's copies (async proxy)
    fence_proxy_async_smem();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
  }
  const uint32_t tmem = sm.tmem_base;
  const Ctx cx{&sm.abort_flag, p.err};
  // tiles: runs of up to 128 compacted slots of one pool; CTA rr owns list
  // entries [tile_start(j) + 64 rr, tile_start(j) + 64 rr + own_n(j, rr))
  const int nswa = sm.nswa, nvalid = sm.nvalid;
  const int tswa = (nswa + kNT - 1) / kNT;
  const int ntiles = tswa + (nvalid - nswa + kNT - 1) / kNT;
  auto tile_start = [&](int j) { return j < tswa ? j * kNT : nswa + (j - tswa) * kNT; };
  auto tile_n = [&](int j) { return min(kNT, (j < tswa ? nswa : nvalid) - tile_start(j)); };
  auto own_n = [&](int j, int rr) { return max(0, min(kNH, tile_n(j) - kNH * rr)); };

  if (warp < kProducerWarps) {
    // ============================================================ producer
    regs_decrease<kRegsProducer>();
    if (tid == 0) {
      prefetch_tensormap(&P.tm_swa);
      prefetch_tensormap(&P.tm_comp);
      prefetch_tensormap(&P.tm_swa_run);
      prefetch_tensormap(&P.tm_comp_run);
    }
    const uint32_t r_free_peer = map_to_rank(bar(sm.r_free[0]), peer);
    int issued = 0;                          // tiles whose gathers were issued
    for (int j = 0; j < ntiles; ++j) {
      const int iv = j % kNV, ik = j % kNK, ir = j % kNR;
      // the V entry is free once this CTA's PV of the own slots of tile j - 4
      // is done; the K entry once the QK of tile j - 3 is done and its copy
      // has landed in the peer
      if (!warp_wait(cx, bar(sm.v_empty[iv]), ((j / kNV) & 1) ^ 1)) break;
      if (!warp_wait(cx, bar(sm.k_empty[ik]), ((j / kNK) & 1) ^ 1, true)) break;
      const int n = own_n(j, (int)rank);
      const int n4 = (n + 3) & ~3;           // gather4 moves four rows: the last row repeats
      if (warp == 0 && lane == 0) mbar_arrive_expect_tx(bar(sm.kv_full[iv]), (uint32_t)(4 * n4 * 128));
      if (n > 0) {
      // column block kb of the own rows: blocks 2 rank, 2 rank + 1 in the V
      // entry, blocks 2 peer, 2 peer + 1 in the K entry
      auto block_dst = [&](int kb) {
        return (kb >> 1) == (int)rank ? v_addr + iv * kEntry + (kb & 1) * kRegion
                                      : k_addr + ik * kEntry + (kb & 1) * kRegion;
      };
      const int32_t* rows = idx_s + tile_start(j) + kNH * (int)rank;
      bool run = false;                      // rows[r] == rows[0] + r for every r < 64
      if (n == kNH) {
        const uint32_t r0 = (uint32_t)rows[0];
        bool ok = true;
#pragma unroll
        for (int r = lane; r < kNH; r += 32) ok = ok && (uint32_t)rows[r] == r0 + (uint32_t)r;
        run = __all_sync(0xffffffffu, ok);
      }
      if (run) {
        const void* tmap = j < tswa ? static_cast<const void*>(&P.tm_swa_run) : static_cast<const void*>(&P.tm_comp_run);
        if (warp == 0 && lane < 4) tma_load_2d(block_dst(lane), tmap, lane * 128, rows[0], bar(sm.kv_full[iv]));
      } else {
        const void* tmap = j < tswa ? static_cast<const void*>(&P.tm_swa) : static_cast<const void*>(&P.tm_comp);
        for (int gi = warp + kProducerWarps * lane; gi < n4; gi += kProducerWarps * 32) {
          const int kb = gi & 3, r0 = (gi >> 2) * 4;
          tma_gather4(block_dst(kb) + r0 * 128, tmap, kb * 128, rows[r0], rows[min(r0 + 1, n - 1)],
                      rows[min(r0 + 2, n - 1)], rows[min(r0 + 3, n - 1)], bar(sm.kv_full[iv]));
        }
      }
      }
      issued = j + 1;
      // the R entry of tile j is free once this CTA's PV of the peer's slots
      // of tile j - 4 is done: arm it and let the peer send its copy
      if (!warp_wait(cx, bar(sm.r_empty[ir]), ((j / kNR) & 1) ^ 1)) break;
      if (warp == 0 && lane == 0) {
        mbar_arrive_expect_tx(bar(sm.r_full[ir]), (uint32_t)kEntry);
        mbar_arrive_cluster_relaxed(r_free_peer + (uint32_t)ir * kBarStride);
      }
    }
    // leave no TMA write in flight (bounded, not cut short by the abort
    // flag): the last tiles issued (also one whose R entry wait gave up), at
    // most one per V entry
    for (int jj = max(0, issued - kNV); jj < issued; ++jj) drain_wait(bar(sm.kv_full[jj % kNV]), (jj / kNV) & 1);
  } else if (warp < kSoftmaxWarp0) {
    regs_decrease<kRegsMma>();
    if (warp < kMmaWarp + kQkWarps) {
    // ============================================================ QK issue
    // Both QK warps take every tile: warp 4 + qi issues the K steps
    // 8 qi .. 8 qi + 7 (dims 256 qi .. 256 qi + 255) into half qi of the S
    // area, so a tile's 16 dependent MMAs run as two chains of eight that the
    // softmax adds.  Warp 4 also copies the tile's K entry to the peer and
    // acknowledges the peer's copy of the tile.
    constexpr uint32_t idesc_qk = idesc(true, 128, kNH, false);
    const int qi = warp - kMmaWarp;
    const uint32_t r_dst0 = map_to_rank(r_addr, peer);
    const uint32_t r_full_peer = map_to_rank(bar(sm.r_full[0]), peer);
    const uint32_t k_empty_peer = map_to_rank(bar(sm.k_empty[0]), peer);
    for (int k = 0; k < ntiles; ++k) {
      const int iv = k % kNV, ik = k % kNK, ir = k % kNR;
      if (!warp_wait(cx, bar(sm.kv_full[iv]), (k / kNV) & 1)) break;
      if (qi == 0) {
        // the peer's output half of the own rows (the K entry) into the
        // peer's R entry, once the peer has released it
        if (!warp_wait(cx, bar(sm.r_free[ir]), (k / kNR) & 1, true)) break;
        if (lane == 0)
          bulk_copy_to_cluster(r_dst0 + ir * kEntry, k_addr + ik * kEntry, (uint32_t)kEntry,
                               r_full_peer + (uint32_t)ir * kBarStride);
      }
      // the second issuer starts its MMAs once the CTA's first QK half has
      // completed (as in the grid kernel)
      if (k == 0 && qi > 0 && !warp_wait(cx, bar(sm.qk0_done), 0)) break;
      // the S area is free once the softmax of tile k - 1 (the other
      // warpgroup's) has read it
      if (k > 0 && !warp_wait(cx, bar(sm.s_empty[(k - 1) & 1]), ((k - 1) >> 1) & 1)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t d = tmem + kSCol + qi * kNH;
#pragma unroll
        for (int h8 = 0; h8 < 8; ++h8) {
          const int kk = 8 * qi + h8;
          const int kb = kk >> 2;            // column block of the own rows
          const uint32_t blk = (kb >> 1) == (int)rank ? v_addr + iv * kEntry + (kb & 1) * kRegion
                                                      : k_addr + ik * kEntry + (kb & 1) * kRegion;
          const uint64_t kd = desc_sw128(blk + (kk & 3) * 32, 16, 1024);
          mma_tmem_a<true>(d, tmem + kQCol + kk * 8, kd, idesc_qk, h8 > 0 ? 1u : 0u);
        }
        mma_commit(bar(sm.s_full[k & 1]));   // (two commits per tile)
        mma_commit(bar(sm.k_empty[ik]));     // this CTA's reads of the K entry
        if (k == 0 && qi == 0) mma_commit(bar(sm.qk0_done));
      }
      __syncwarp();
      if (qi == 0) {
        // the peer's copy of tile k has landed here: tell the peer (its K
        // entry's other reader), then the PV warp (which waits for this, so
        // that the entry's next phase cannot complete before this wait)
        if (!warp_wait(cx, bar(sm.r_full[ir]), (k / kNR) & 1, true)) break;
        if (lane == 0) {
          mbar_arrive_cluster_relaxed(k_empty_peer + (uint32_t)ik * kBarStride);
          mbar_arrive(bar(sm.r_seen[ir]));
        }
      }
    }
    if (lane == 0) mma_commit(bar(sm.qk_done));
    __syncwarp();
    } else if (warp == kPvWarp) {
    // ============================================================ PV issue
    constexpr uint32_t idesc_pv = idesc(true, 128, kHalfDims, true);
    // per tile: the own slots' PV as soon as this CTA's P half is written
    // (it releases the V entry), then the peer's slots' PV once the peer's P
    // half and rows have landed
    for (int jj = 0; jj < ntiles; ++jj) {
      const int b = jj & 1, iv = jj % kNV, ir = jj % kNR;
      const uint32_t pb = p_addr + b * kPBytes;
      if (!warp_wait(cx, bar(sm.p_ready[b]), (jj >> 1) & 1)) break;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint64_t a = desc_noswizzle(pb + rank * kPHalf + kk * 256, 128, 512);
          const uint64_t v = desc_sw128(v_addr + iv * kEntry + kk * (32 * 128), kRegion, 1024);
          mma<true>(tmem + kOCol, a, v, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(sm.v_empty[iv]));
      }
      __syncwarp();
      if (!warp_wait(cx, bar(sm.r_seen[ir]), (jj / kNR) & 1)) break;
      if (!warp_wait(cx, bar(sm.pin_full[b]), (jj >> 1) & 1, true)) break;
      if (!warp_wait(cx, bar(sm.r_full[ir]), (jj / kNR) & 1, true)) break;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint64_t a = desc_noswizzle(pb + peer * kPHalf + kk * 256, 128, 512);
          const uint64_t v = desc_sw128(r_addr + ir * kEntry + kk * (32 * 128), kRegion, 1024);
          mma<true>(tmem + kOCol, a, v, idesc_pv, 1u);
        }
        mma_commit(bar(sm.p_empty[b]));
        mma_commit(bar(sm.r_empty[ir]));
      }
      __syncwarp();
    }
    if (lane == 0) mma_commit(bar(sm.o_full));
    __syncwarp();
    }
  } else {
    // ============================================================ softmax / epilogue
    regs_increase<kRegsSoftmax>();
    const int g = (warp - kSoftmaxWarp0) >> 2;        // warpgroup: tiles j with j % 2 == g
    const int q4 = warp & 3;                           // TMEM lane quadrant of this warp
    const int h = q4 * 32 + lane;                      // MMA row (a token pair: head h & 63 of token t + (h >> 6))
    const bool active = q4 * 32 < rows_used;           // warp-uniform
    const uint64_t* my_mask = (h < 64) ? sm.mask_a : sm.mask_b;   // token pairs: this row's own entries
    const bool leader = (warp - kSoftmaxWarp0) % 4 == 0 && lane == 0;   // one thread per warpgroup (quadrant 0: active)
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    // BF16 partial staging: warpgroup g's 128 rows of 256 bytes in half of
    // the V ring (read by nothing but this CTA's QK and PV, done by then)
    auto stage_row = [&](int sg, int r) -> unsigned char* { return base + kOffV + sg * (128 * 256) + r * 256; };
    const float c = load_scale(p.bmm1, p.bmm1_dev) * kLog2e;
    const uint32_t mx_bytes = (uint32_t)(rows_used * 4);
    // the peer's copy of a TcSmall field: one mapped base plus the field's offset
    const uint32_t small_local = smem_addr(&sm);
    const uint32_t small_peer = map_to_rank(small_local, peer);
    auto at_peer = [&](const void* field) { return small_peer + (smem_addr(field) - small_local); };
    const uint32_t p_mine = p_addr + g * kPBytes + rank * kPHalf;                     // this CTA's half of P buffer g
    // this thread's P row in the no-swizzle K-major layout: 16-byte chunk cc
    // of row h at (h / 8) * 512 + cc * 128 + (h % 8) * 16
    const uint32_t p_row = p_mine + (uint32_t)((h >> 3) * 512 + (h & 7) * 16);
    if (leader) {
      mbar_arrive_expect_tx(bar(sm.mx_full[g][0]), mx_bytes);
      mbar_arrive_expect_tx(bar(sm.mx_full[g][1]), mx_bytes);
      if (g == 0) mbar_arrive_expect_tx(bar(sm.l_full), mx_bytes);
    }

    float m_last = -INFINITY, l_run = 0.f;
    // E4M3 P keeps 3 mantissa bits: short splits move the reference on every
    // new maximum (the same choice in both CTAs: nvalid is the pair's)
    // (a token pair: by the slot count of the row's own token)
    const int n_row = kPair ? (h < 64 ? sm.n_a : sm.n_b) : nvalid;
    const float thr = n_row <= kExactRefSlots ? 0.f : kRescaleThreshold;
    bool ok = true;
    int j = g;
    const uint64_t c2 = f2_pack(c, c);
    for (; ok && j < ntiles; j += 2) {
      const int n_own = own_n(j, (int)rank);
      const int sb = j % kSBufs, q = (j >> 1) & 1;
      if (!(ok = warp_wait(cx, bar(sm.s_full[sb]), (j / kSBufs) & 1))) break;
      tc_fence_after();
      float sv[kNH];
      if (active) {
        // the two QK halves' partial logits (dims 0-255 and 256-511)
#pragma unroll
        for (int hb = 0; hb < kNH / 32; ++hb) {
          uint32_t r[32];
          tmem_ld32(tl + kSCol + hb * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[hb * 32 + i] = __uint_as_float(r[i]);
        }
        tmem_wait_ld();
#pragma unroll
        for (int hb = 0; hb < kNH / 32; ++hb) {
          uint32_t r[32];
          tmem_ld32(tl + kSCol + kNH + hb * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[hb * 32 + i] += __uint_as_float(r[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(sm.s_empty[sb]));     // the S area may be overwritten (by tile j + 1)
      // ---- this CTA's tile maximum to the peer, the peer's back
      float mt = -INFINITY;
      if (active) {
#pragma unroll
        for (int i = 0; i < kNH; i += 2) f2_unpack(f2_mul(f2_pack(sv[i], sv[i + 1]), c2), sv[i], sv[i + 1]);
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if constexpr (kPair) {
          // only the entries of this row's token (the tile's other entries are the other token's)
          const uint64_t mrow = my_mask[j];
#pragma unroll
          for (int i = 0; i < kNH; ++i)
            if ((mrow >> i) & 1ull) m4[i & 3] = fmaxf(m4[i & 3], sv[i]);
        } else if (n_own >= kNH) {
#pragma unroll
          for (int i = 0; i < kNH; ++i) m4[i & 3] = fmaxf(m4[i & 3], sv[i]);
        } else {
#pragma unroll
          for (int i = 0; i < kNH; ++i)
            if (i < n_own) m4[i & 3] = fmaxf(m4[i & 3], sv[i]);
        }
        mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        st_async_b32(at_peer(&sm.mx[g][q][h]), __float_as_uint(mt), at_peer(&sm.mx_full[g][q]));
        // absent heads' warps neither send nor wait: the peer's next use of
        // this slot needs every active warp's maximum of tile j + 2 first
        if (!(ok = warp_wait(cx, bar(sm.mx_full[g][q]), (j >> 2) & 1, true))) break;
        mt = fmaxf(mt, sm.mx[g][q][h]);
      }
      if (leader) mbar_arrive_expect_tx(bar(sm.mx_full[g][q]), mx_bytes);   // for tile j + 4
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
      // ---- P buffer g: this CTA's PV(j - 2) done (then tell the peer, whose
      // P half this CTA has read), and the peer's PV(j - 2) done
      if (!(ok = warp_wait(cx, bar(sm.p_empty[g]), ((j >> 1) & 1) ^ 1))) break;
      if (j >= 2 && lane == 0) mbar_arrive_cluster_relaxed(at_peer(&sm.pout_free[g]));
      if (!(ok = warp_wait(cx, bar(sm.pout_free[g]), ((j >> 1) & 1) ^ 1, true))) break;
      tc_fence_after();
      // ---- P = 2^(x - m(j)) for the own slots; this warpgroup's row sum, rescaled to m(j)
      if (active) {
        l_run *= (m_last == -INFINITY) ? 0.f : fast_exp2(m_last - m_cur);
        m_last = m_cur;
        const uint64_t nm2 = f2_pack(-m_cur, -m_cur);
#pragma unroll
        for (int i = 0; i < kNH; i += 2) {
          float x0, x1;
          f2_unpack(f2_add(f2_pack(sv[i], sv[i + 1]), nm2), x0, x1);
          sv[i] = fast_exp2(x0);
          sv[i + 1] = fast_exp2(x1);
        }
        if constexpr (kPair) {
          const uint64_t mrow = my_mask[j];
#pragma unroll
          for (int i = 0; i < kNH; ++i)
            if (!((mrow >> i) & 1ull)) sv[i] = 0.f;
        } else if (n_own < kNH) {
#pragma unroll
          for (int i = 0; i < kNH; ++i)
            if (i >= n_own) sv[i] = 0.f;
        }
        uint64_t s4[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < kNH; i += 2) s4[(i >> 1) & 1] = f2_add(s4[(i >> 1) & 1], f2_pack(sv[i], sv[i + 1]));
        float s0, s1, s2, s3;
        f2_unpack(s4[0], s0, s1);
        f2_unpack(s4[1], s2, s3);
        l_run += (s0 + s1) + (s2 + s3);
#pragma unroll
        for (int cc = 0; cc < kNH / 16; ++cc) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = cc * 16 + i * 4;
            w[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(sv[e], sv[e + 1]), __NV_SATFINITE, __NV_E4M3) |
                   ((uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(sv[e + 2], sv[e + 3]), __NV_SATFINITE, __NV_E4M3) << 16);
          }
          st_shared_v4(p_row + cc * 128, make_uint4(w[0], w[1], w[2], w[3]));
        }
      }
      fence_proxy_async_smem();                       // the P rows are read by the tensor core and the bulk copy
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
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(sm.p_ready[g]));
      // ---- one thread: this CTA's P half to the peer, and the tile's P buffer armed
      if (leader) {
        bool lok = wait_bar(cx, bar(sm.p_ready[g]), (j >> 1) & 1, false);
        if (lok) {
          mbar_arrive_expect_tx(bar(sm.pin_full[g]), (uint32_t)kPHalf);
          bulk_copy_to_cluster(map_to_rank(p_mine, peer), p_mine, (uint32_t)kPHalf, at_peer(&sm.pin_full[g]));
        }
        ok = lok;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    // ---- row sums: both warpgroups brought to the final reference (the
    // same in both CTAs), then this CTA's sum (its own slots) and the peer's
    if (active) {
      sm.lsum[g][h] = l_run;
      sm.m_end[g][h] = m_last;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(sm.lsum_full));
    if (ok) ok = warp_wait(cx, bar(sm.lsum_full), 0);
    if (active) {
      float l_tot = 0.f, m_fin = -INFINITY;
      if (ok) {
        const float ma = sm.m_end[0][h], mb = sm.m_end[1][h];
        m_fin = fmaxf(ma, mb);
        float l_loc = 0.f;
        if (m_fin != -INFINITY) {
          if (ma != -INFINITY) l_loc += sm.lsum[0][h] * fast_exp2(ma - m_fin);
          if (mb != -INFINITY) l_loc += sm.lsum[1][h] * fast_exp2(mb - m_fin);
        }
        if (g == 0)
          st_async_b32(at_peer(&sm.lpeer[h]), __float_as_uint(l_loc), at_peer(&sm.l_full));
        ok = warp_wait(cx, bar(sm.l_full), 0, true);
        if (ok) l_tot = l_loc + sm.lpeer[h];
      }
      if (ok && ntiles > 0) {
        ok = warp_wait(cx, bar(sm.o_full), 0);
        tc_fence_after();
      }
      const bool have = ok && ntiles > 0 && l_tot > 0.f;
      const float lse = have ? m_fin + fast_log2(l_tot) : -INFINITY;
      float f = have ? 1.f / l_tot : 0.f;
      if (S == 1) {
        f *= load_scale(p.bmm2, p.bmm2_dev);
        if (p.sinks != nullptr && have) f *= 1.f / (1.f + fast_exp2(__ldg(p.sinks + (kPair ? (h & 63) : h)) * kLog2e - lse));
      }
      const int64_t row_th = kPair ? (int64_t)(t + (h >> 6)) * H + (h & 63) : (int64_t)t * H + h;
      // The normalised BF16 rows go through shared memory, so that the
      // global stores below are whole 256-byte row segments rather than one
      // 16-byte piece per row per warp instruction: warpgroup g stages its
      // 128 columns in half of the V ring (read by nothing but this CTA's QK
      // and PV, done by now; no copy to the peer reads it), 16-byte chunks
      // XOR-swizzled by the row to spread the banks
      unsigned char* row = stage_row(g, h);
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
    named_bar_sync(1 + g, 128);
    {
      const int w4 = (warp - kSoftmaxWarp0) & 3;
      const int col0 = (int)rank * kHalfDims + g * (kHalfDims / 2);
      const int cidx = lane & 15;
      for (int r = w4 + 4 * (lane >> 4); r < rows_used; r += 8) {
        const uint4 x = *reinterpret_cast<const uint4*>(stage_row(g, r) + ((cidx ^ (r & 7)) << 4));
        const int64_t row = kPair ? (int64_t)(t + (r >> 6)) * H + (r & 63) : (int64_t)t * H + r;
        const int64_t orow = kPartial ? row * S + s : row;
        *reinterpret_cast<uint4*>((kPartial ? p.part_o : p.out) + orow * kHeadDim + col0 + cidx * 8) = x;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == kMmaWarp) {
    drain_wait(bar(sm.qk_done), 0);
    drain_wait(bar(sm.o_full), 0);
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  tc_fence_before();
  cluster_sync();                          // the peer is done with this CTA's shared memory
}

}  // namespace

int tc_slot_smem_bytes() { return kSmemBytes; }
int tc_slot_threads() { return kThreads; }

cudaError_t launch_decode_tc_slot(const DecodeParams& p, int grid, bool pair, cudaStream_t stream) {
  if (p.dtype != SMLA_E4M3) return cudaErrorInvalidValue;
  if (pair && p.H != 64) return cudaErrorInvalidValue;   // two tokens of 64 heads fill the 128 MMA rows
  SlotParams P;
  memset(&P, 0, sizeof(P));
  P.p = p;
  // a pool of fewer than 64 rows holds no run of 64 rows: its run map is never used
  const int swa_run = (int)std::max<int64_t>(1, std::min<int64_t>(kNH, p.swa_rows));
  const int comp_run = (int)std::max<int64_t>(1, std::min<int64_t>(kNH, p.comp_rows));
  cudaError_t e = encode_pool_map(&P.tm_swa, p.swa, p.swa_rows, p.swa_stride, p.dtype, 1);
  if (e == cudaSuccess) e = encode_pool_map(&P.tm_comp, p.comp, p.comp_rows, p.comp_stride, p.dtype, 1);
  if (e == cudaSuccess) e = encode_pool_map(&P.tm_swa_run, p.swa, p.swa_rows, p.swa_stride, p.dtype, swa_run);
  if (e == cudaSuccess) e = encode_pool_map(&P.tm_comp_run, p.comp, p.comp_rows, p.comp_stride, p.dtype, comp_run);
  if (e != cudaSuccess) return e;
  auto launch = [&](auto kernel) -> cudaError_t {
    // the register split waits until the launch holds the registers it hands
    // out: refuse a build whose per-thread count is below the one it was sized for
    static std::atomic<int> launch_regs[4];            // per kernel (single split, split partials; x token pairs)
    std::atomic<int>& cached = launch_regs[(p.num_splits > 1 ? 1 : 0) + (pair ? 2 : 0)];
    int regs = cached.load(std::memory_order_relaxed);
    if (regs == 0) {
      cudaFuncAttributes fa;
      cudaError_t err = cudaFuncGetAttributes(&fa, kernel);
      if (err != cudaSuccess) return err;
      regs = fa.numRegs;
      cached.store(regs, std::memory_order_relaxed);
    }
    if (regs < kLaunchRegs) return cudaErrorInvalidConfiguration;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    kernel<<<grid, kThreads, kSmemBytes, stream>>>(P);
    return cudaSuccess;
  };
  if (pair)
    e = p.num_splits > 1 ? launch(decode_tc_slot_kernel<true, true>) : launch(decode_tc_slot_kernel<false, true>);
  else
    e = p.num_splits > 1 ? launch(decode_tc_slot_kernel<true, false>) : launch(decode_tc_slot_kernel<false, false>);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace smla
