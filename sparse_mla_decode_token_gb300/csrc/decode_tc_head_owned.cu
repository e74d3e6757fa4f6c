// tcgen05 / TMEM sparse MLA decode kernel for E4M3 rows with head-owned
// softmax (sm_103a).
//
// Work unit: one (token, split) on a cluster of two CTAs.  An fp32
// accumulator for 128 heads x 512 dims fills the whole tensor memory of one
// SM, so CTA r of the pair keeps output dims [256 r, 256 r + 256) of every
// head and gathers only that half of every selected row.  Each CTA's QK is
// then a partial sum over its 256 dims, and the two partials must meet before
// the softmax.  Here they meet per head: heads 32 q .. 32 q + 31 (TMEM lane
// quadrant q) belong to CTA q % 2, which alone runs their softmax.  Per tile
// of up to 128 selected slots:
//
//   producer warps 0-3  this CTA's half of every selected row (two 128-byte
//                       column blocks) with TMA tile::gather4 (four rows per
//                       request) into a 128-byte-swizzled, UMMA-canonical
//                       tile of a 3-stage ring; two groups of two warps take
//                       alternate tiles; a tile of 128 consecutive rows is one
//                       box copy per column block
//   QK warps 4-5        S_r = Q_r K_r^T (M = 128 heads, N = 128 slots, K = 256
//                       dims) into TMEM S buffer k % 2; warp 4 + b issues the
//                       tiles of buffer b (each issuing thread's chain of
//                       dependent MMAs runs at about one instruction per 150
//                       ns, so two chains overlap); warp 4 also allocates
//                       and frees TMEM
//   PV warp 6           O_r += P V_r (M = 128 heads, N = 256 dims, K = 128
//                       slots), P read from the first 32 columns of the tile's
//                       S buffer, where the softmax warps put it
//   softmax warps 8-15  two warpgroups taking whole tiles in turn (warpgroup
//                       g takes tiles j with j % 2 == g), one thread per head
//                       (TMEM lane).  In each warpgroup the two warps of the
//                       quadrants the peer owns ("push" warps) send their
//                       heads' partial S to the peer (st.async, 24-bit
//                       floats), then take the peer's E4M3 P rows and rescale
//                       factors for those heads, write the P rows into TMEM
//                       and rescale their O rows; the two warps of this CTA's
//                       own quadrants ("own" warps) add the peer's partial to
//                       their own, settle the running reference maximum
//                       (handed between the warpgroups through shared
//                       memory), compute P = 2^(x - m) in E4M3, write it into
//                       TMEM and send it, with the factor by which O must be
//                       rescaled, to the peer.
//
// Per slot each CTA thus sends 64 heads x 3 bytes of partial S and 64 heads x
// 1 byte of P instead of 128 x 3 bytes of partial S, and runs the
// exponentials of its own 64 heads only.  The price is a round trip between
// the CTAs inside every tile (partial S out, P back) while tensor memory
// holds only two 128-slot S buffers next to O, so the tile chain is latency
// bound: on a GB300 the 128-token E4M3 workload takes ~145 us here against
// ~94 us with the replicated softmax (decode_tcgen05.cu), which is why this
// form is opt-in (SMLA_KERNEL_TCGEN05_HEAD_OWNED).
//
// The operation follows the FlashInfer trtllm_batch_decode_sparse_mla_dsv4 page
// (description, SM100/SM103 paragraph; Parameters); the base-2 LSE, the sink in
// the normaliser and the split partials follow the cake_sparse_mla_sm120 page
// (Parameters: out_lse, attn_sink, mid_out / mid_lse).
//
// Every mbarrier wait is bounded (2 s); on expiry the CTA raises an abort flag,
// ORs SMLA_DEVERR_TIMEOUT into the error word, lets every role leave its loop,
// waits for its own copies and MMAs, frees its TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kN = 128;                    // slots per tile
constexpr int kHalfDims = 256;             // output dims per CTA
constexpr int kRegions = 2;                // 128-byte column blocks per half row
constexpr int kStages = 3;                 // KV ring
constexpr int kProducerWarps = 4;
constexpr int kProducerGroups = 2;         // tiles alternate between two groups of two warps
constexpr int kQkWarp0 = kProducerWarps;   // QK issuers 4 and 5; warp 4 allocates and frees TMEM
constexpr int kQkWarps = 2;
constexpr int kPvWarp = kQkWarp0 + kQkWarps;
constexpr int kSoftmaxWarp0 = 8;
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = (kSoftmaxWarp0 + kSoftmaxWarps) * 32;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCols = SMLA_TC_MAX_SPLIT_COLS;
constexpr int kMaxChunks = kMaxCols / 32;
constexpr int kChunksPerWarp = (kMaxChunks + kWarps - 1) / kWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;              // O: 256 fp32 columns
constexpr uint32_t kSCol = 256;            // S buffer b at 256 + 128 b; P of its tile in its first 32 columns
constexpr int kPCols = kN / 4;             // E4M3 P: four per column
constexpr float kRescaleThreshold = 8.f;   // log2 units: P stays <= 2^8
constexpr int kExactRefTiles = 4;          // chains of at most 4 tiles (512 slots) follow the exact maximum
constexpr int kKStep = 32;                 // E4M3 MMA K per instruction
constexpr int kOwnMax = 64;                // heads one CTA owns (H = 128)

constexpr int kRegionQ = 128 * 128;        // 128 head rows x 128 B
constexpr int kRegionKV = kN * 128;        // 128 slot rows x 128 B
constexpr int kQBytes = kRegions * kRegionQ;
constexpr int kStageBytes = kRegions * kRegionKV;
constexpr int kXBytes = (kN / 16) * 3 * kOwnMax * 16;   // peer's partial S of my heads: 16-slot groups x 3 words x 64 heads
constexpr int kPinAlpha = kOwnMax * kN;                 // offset of the rescale factors in a P-in buffer
constexpr int kPinBytes = kPinAlpha + kOwnMax * 4;      // peer's P rows (128 B each) + factors
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kQBytes;
constexpr int kOffX = kOffKV + kStages * kStageBytes;
constexpr int kOffPin = kOffX + 2 * kXBytes;
constexpr int kOffFin = kOffPin + 2 * kPinBytes;
constexpr int kOffIdx = kOffFin + kOwnMax * 4;

struct Small {
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2], s_empty[2];        // QK done / PV done (S buffer, and the P in it, free)
  uint64_t xs_full[2];                   // the peer's partial S of my heads landed (bytes)
  uint64_t xs_free[2];                   // the peer's own warps read what my push warps sent (remote arrivals)
  uint64_t pin_full[2];                  // the peer's P rows and factors landed (bytes)
  uint64_t pin_free[2];                  // the peer's push warps read what my own warps sent (remote arrivals)
  uint64_t m_ready[2];                   // m_buf[g] written by warpgroup g's own warps
  uint64_t pv_ready[2];                  // P of the tile in TMEM, O rescaled
  uint64_t lsum_full;
  uint64_t fin_full;                     // the peer's output factors of its heads landed (bytes)
  uint64_t o_full;                       // every PV done
  uint64_t qk0_done;                     // the CTA's first QK done (single use)
  uint64_t qk_done;                      // every QK done (one commit per QK warp)
  float m_end[2][kOwnMax];               // reference maximum after warpgroup g's last tile, per own head
  float m_buf[2][kOwnMax];               // reference maximum after warpgroup g's latest tile
  float lsum[2][kOwnMax];
  int32_t chunk_off[kMaxChunks];
  int32_t nswa;
  int32_t nvalid;
  uint32_t tmem_base;
  int32_t abort_flag;
};

constexpr int kOffSmall = kOffIdx + kMaxCols * 4;
constexpr int kSmemBytes = kOffSmall + (int)sizeof(Small) + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kSCol + 2 * kN <= kTmemCols, "tensor memory budget");
static_assert(kStages * kStageBytes >= 2 * 128 * 256, "BF16 partial staging fits in the KV stages");

struct TcParams {
  CUtensorMap tm_swa;
  CUtensorMap tm_comp;
  CUtensorMap tm_swa_run;
  CUtensorMap tm_comp_run;
  DecodeParams p;
};

__device__ __forceinline__ uint32_t fp8x4(float a, float b, float c, float d) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3) |
         ((uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3) << 16);
}

// 24-bit logits: the low mantissa byte is dropped after rounding; values a, b,
// c, d travel as [a1 a2 a3 d1] [b1 b2 b3 d2] [c1 c2 c3 d3].
__device__ __forceinline__ void pack24(const uint32_t (&v)[16], uint32_t (&w)[12]) {
#pragma unroll
  for (int gq = 0; gq < 4; ++gq) {
    const uint32_t d = v[4 * gq + 3] + 0x80u;
    w[3 * gq] = __byte_perm(v[4 * gq] + 0x80u, d, 0x5321);
    w[3 * gq + 1] = __byte_perm(v[4 * gq + 1] + 0x80u, d, 0x6321);
    w[3 * gq + 2] = __byte_perm(v[4 * gq + 2] + 0x80u, d, 0x7321);
  }
}

__device__ __forceinline__ void unpack24(const uint32_t (&w)[12], float (&x)[16]) {
#pragma unroll
  for (int gq = 0; gq < 4; ++gq) {
    const uint32_t w0 = w[3 * gq], w1 = w[3 * gq + 1], w2 = w[3 * gq + 2];
    x[4 * gq] = __uint_as_float(w0 << 8);
    x[4 * gq + 1] = __uint_as_float(w1 << 8);
    x[4 * gq + 2] = __uint_as_float(w2 << 8);
    x[4 * gq + 3] = __uint_as_float(__byte_perm(__byte_perm(w0, w1, 0x7373), w2, 0x7103));
  }
}

// kPartial: the launch has num_splits > 1 and writes BF16 split partials.
template <bool kPartial>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_tc_head_owned_kernel(const __grid_constant__ TcParams P) {
  const DecodeParams& p = P.p;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_addr - raw_addr);
  Small& sm = *reinterpret_cast<Small*>(base + kOffSmall);
  int32_t* idx_s = reinterpret_cast<int32_t*>(base + kOffIdx);
  const uint32_t q_addr = base_addr + kOffQ;
  const uint32_t kv_addr = base_addr + kOffKV;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const int S = p.num_splits;
  const int unit = blockIdx.x >> 1;
  const int s = unit % S;
  const int t = unit / S;
  const int H = p.H;
  const int nown = H / 64;                 // own (and push) quadrants per warpgroup: 2 for H = 128, 1 for H = 64
  // Column range of this split, from the table width only; in the page-table
  // form rounded up to whole tiles, so that full compressed tiles lie on one
  // page when pages hold a multiple of 128 rows.
  int per_split = (p.W + S - 1) / S;
  if (p.bt) per_split = (per_split + kN - 1) / kN * kN;
  const int c0 = min(p.W, s * per_split);
  int c1 = min(p.W, c0 + per_split);
  if (c1 - c0 > kMaxCols) {           // the planner prevents this; never read past the staging buffer
    if (p.err && tid == 0) atomicOr(p.err, SMLA_DEVERR_INTERNAL);
    c1 = c0 + kMaxCols;
  }

  auto bar = [&](const uint64_t& b) { return smem_addr(&b); };

  // ---------------------------------------------------------------- set-up
  {
    const unsigned char* qb = reinterpret_cast<const unsigned char*>(p.q) +
                              ((int64_t)t * p.q_stride_token + (int64_t)rank * kHalfDims);
    constexpr int kChunks = kHalfDims / 16;   // 16-byte chunks per half row
    for (int c = tid; c < H * kChunks; c += kThreads) {
      const int h = c / kChunks, cc = c % kChunks;
      cp_async_16(q_addr + (cc >> 3) * kRegionQ + sw128_offset(h, cc & 7), qb + (int64_t)h * kHeadDim + cc * 16);
    }
  }
  const int nchunks = (c1 - c0 + 31) / 32;
  const int32_t* irow = p.ind + (int64_t)t * p.ind_stride;
  int32_t rv[kChunksPerWarp];
  if (p.bt == nullptr) {
#pragma unroll
    for (int q = 0; q < kChunksPerWarp; ++q) {
      const int col = c0 + (warp + q * kWarps) * 32 + lane;
      rv[q] = (col < c1) ? __ldg(irow + col) : -1;
    }
  } else {
#pragma unroll
    for (int q = 0; q < kChunksPerWarp; ++q) {
      const int col = c0 + (warp + q * kWarps) * 32 + lane;
      rv[q] = -1;
      if (col < c1) rv[q] = col >= kSwaCols ? paged_row(p, t, col - kSwaCols) : __ldg(irow + col);
    }
  }
  const TokenInfo ti = token_info(p, t);
  c1 = min(c1, max(c0, ti.n_lim));
  {
    // zero the KV stages (rows past a tile's slot count then hold finite data)
    // and the Q rows of absent heads (their S, and so their P, is then 0)
    const uint4 z = make_uint4(0, 0, 0, 0);
    uint4* zp = reinterpret_cast<uint4*>(base + kOffKV);
    for (int i = tid; i < kStages * kStageBytes / 16; i += kThreads) zp[i] = z;
    if (H < 128) {
      for (int kb = 0; kb < kRegions; ++kb) {
        uint4* qz = reinterpret_cast<uint4*>(base + kOffQ + kb * kRegionQ + H * 128);
        for (int i = tid; i < (128 - H) * 8; i += kThreads) qz[i] = z;
      }
    }
    if (tid == 0) {
      for (int i = 0; i < kStages; ++i) {
        mbar_init(bar(sm.kv_full[i]), 1);
        mbar_init(bar(sm.kv_empty[i]), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(bar(sm.s_full[b]), 1);
        mbar_init(bar(sm.s_empty[b]), 1);
        mbar_init(bar(sm.xs_full[b]), 1);
        mbar_init(bar(sm.xs_free[b]), nown);
        mbar_init(bar(sm.pin_full[b]), 1);
        mbar_init(bar(sm.pin_free[b]), nown);
        mbar_init(bar(sm.m_ready[b]), nown);
        mbar_init(bar(sm.pv_ready[b]), 2 * nown);
      }
      mbar_init(bar(sm.lsum_full), 2 * nown);
      mbar_init(bar(sm.fin_full), 1);
      mbar_init(bar(sm.o_full), 1);
      mbar_init(bar(sm.qk0_done), 1);
      mbar_init(bar(sm.qk_done), kQkWarps);
      sm.abort_flag = 0;
      sm.nswa = 0;
      fence_mbar_init_cluster();
    }
    __syncthreads();
    // a2: compaction of the split's columns [c0, c1): valid SWA slots first,
    // then valid compressed slots, each in column order
#pragma unroll
    for (int q = 0; q < kChunksPerWarp; ++q) {
      const int k = warp + q * kWarps;
      if (k < nchunks) {
        const int col = c0 + k * 32 + lane;
        const int idx = rv[q];
        rv[q] = -1;
        if (col < c1) {
          const bool swa = col < kSwaCols;
          bool ok = idx != -1 && (!swa || col < ti.w_swa);
          if (ok) {
            const int64_t nrows = swa ? p.swa_rows : p.comp_rows;
            if (idx < 0 || (int64_t)idx >= nrows) {
              ok = false;
              if (p.err && rank == 0) atomicOr(p.err, SMLA_DEVERR_INDEX_OUT_OF_RANGE);
            }
          }
          if (ok) rv[q] = idx;
        }
        const unsigned ball = __ballot_sync(0xffffffffu, rv[q] >= 0);
        const unsigned ball_swa = __ballot_sync(0xffffffffu, rv[q] >= 0 && col < kSwaCols);
        if (lane == 0) {
          sm.chunk_off[k] = __popc(ball);
          if (ball_swa) atomicAdd(&sm.nswa, __popc(ball_swa));
        }
      }
    }
    __syncthreads();
    int chunk_base[kChunksPerWarp];
    {
      int carry = 0;
#pragma unroll
      for (int q = 0; q < kChunksPerWarp; ++q) chunk_base[q] = 0;
      for (int base0 = 0; base0 < nchunks; base0 += 32) {
        const int k = base0 + lane;
        const int v = k < nchunks ? sm.chunk_off[k] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += u;
        }
#pragma unroll
        for (int q = 0; q < kChunksPerWarp; ++q) {
          const int kq = warp + q * kWarps;
          const int excl = __shfl_sync(0xffffffffu, incl - v, kq & 31);
          if ((kq >> 5) == (base0 >> 5)) chunk_base[q] = carry + excl;
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (warp == 0 && lane == 0) sm.nvalid = carry;
    }
#pragma unroll
    for (int q = 0; q < kChunksPerWarp; ++q) {
      const int k = warp + q * kWarps;
      if (k < nchunks) {
        const unsigned ball = __ballot_sync(0xffffffffu, rv[q] >= 0);
        if (rv[q] >= 0) idx_s[chunk_base[q] + __popc(ball & ((1u << lane) - 1u))] = rv[q];
      }
    }
    if (warp == kQkWarp0) tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
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
  const int nswa = sm.nswa, nvalid = sm.nvalid;
  const int tswa = (nswa + kN - 1) / kN;
  const int ntiles = tswa + (nvalid - nswa + kN - 1) / kN;
  auto tile_start = [&](int j) { return j < tswa ? j * kN : nswa + (j - tswa) * kN; };
  auto tile_n = [&](int j) { return min(kN, (j < tswa ? nswa : nvalid) - tile_start(j)); };

  if (warp < kProducerWarps) {
    // ============================================================ producer
    if (tid == 0) {
      prefetch_tensormap(&P.tm_swa);
      prefetch_tensormap(&P.tm_comp);
      prefetch_tensormap(&P.tm_swa_run);
      prefetch_tensormap(&P.tm_comp_run);
    }
    constexpr int kWarpsPerGroup = kProducerWarps / kProducerGroups;
    const int pg = warp / kWarpsPerGroup, pw = warp % kWarpsPerGroup;
    int j = pg;
    for (; j < ntiles; j += kProducerGroups) {
      const int st = j % kStages;
      if (!warp_wait(cx, bar(sm.kv_empty[st]), ((j / kStages) & 1) ^ 1)) break;
      const int start = tile_start(j), n = tile_n(j);
      const int n4 = (n + 3) & ~3;           // gather4 moves four rows: the last row repeats
      if (pw == 0 && lane == 0) mbar_arrive_expect_tx(bar(sm.kv_full[st]), (uint32_t)(kRegions * n4 * 128));
      const uint32_t stage = kv_addr + st * kStageBytes;
      const int32_t* rows = idx_s + start;
      bool run = false;                      // rows[r] == rows[0] + r for every r < N
      if (n == kN) {
        const uint32_t r0 = (uint32_t)rows[0];
        bool ok = true;
#pragma unroll
        for (int r = lane; r < kN; r += 32) ok = ok && (uint32_t)rows[r] == r0 + (uint32_t)r;
        run = __all_sync(0xffffffffu, ok);
      }
      if (run) {
        const void* tmap = j < tswa ? static_cast<const void*>(&P.tm_swa_run) : static_cast<const void*>(&P.tm_comp_run);
        if (pw == 0 && lane < kRegions)
          tma_load_2d(stage + lane * kRegionKV, tmap, (int)rank * kHalfDims + lane * 128, rows[0], bar(sm.kv_full[st]));
      } else {
        const void* tmap = j < tswa ? static_cast<const void*>(&P.tm_swa) : static_cast<const void*>(&P.tm_comp);
        const int groups = (n4 / 4) * kRegions;
        for (int gi = pw + kWarpsPerGroup * lane; gi < groups; gi += kWarpsPerGroup * 32) {
          const int kb = gi % kRegions, r0 = (gi / kRegions) * 4;
          tma_gather4(stage + kb * kRegionKV + r0 * 128, tmap, (int)rank * kHalfDims + kb * 128, rows[r0],
                      rows[min(r0 + 1, n - 1)], rows[min(r0 + 2, n - 1)], rows[min(r0 + 3, n - 1)],
                      bar(sm.kv_full[st]));
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // leave no TMA write of this group in flight, also after an abort
    for (int jj = max(pg, min(j, ntiles) - kStages); jj < min(j, ntiles); ++jj)
      if ((jj - pg) % kProducerGroups == 0) drain_wait(bar(sm.kv_full[jj % kStages]), (jj / kStages) & 1);
  } else if (warp < kQkWarp0 + kQkWarps) {
    // ============================================================ QK issue
    constexpr uint32_t idesc_qk = idesc(true, 128, kN, false);
    const int qi = warp - kQkWarp0;
    // The other issuers start only once the CTA's first QK has completed:
    // on a GB300, a QK issued by a second warp before the first one finished
    // gave wrong logits for some heads in repeated runs (observed, cause
    // not identified); after that the issuers' chains overlap freely.
    bool ok = qi == 0 || ntiles <= qi || warp_wait(cx, bar(sm.qk0_done), 0);
    for (int k = qi; ok && k < ntiles; k += kQkWarps) {
      const int st = k % kStages;
      const int b = k & 1;
      if (!warp_wait(cx, bar(sm.kv_full[st]), (k / kStages) & 1)) break;
      // S buffer b (and the P of tile k - 2 in it) is free once PV(k - 2) is done
      if (!warp_wait(cx, bar(sm.s_empty[b]), ((k >> 1) & 1) ^ 1)) break;
      fence_proxy_async_smem();
      tc_fence_after();
      if (lane == 0) {
        const uint32_t stage = kv_addr + st * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < kRegions * (128 / kKStep); ++kk) {
          const uint64_t a = desc_sw128(q_addr + (kk >> 2) * kRegionQ + (kk & 3) * 32, 16, 1024);
          const uint64_t kd = desc_sw128(stage + (kk >> 2) * kRegionKV + (kk & 3) * 32, 16, 1024);
          mma<true>(tmem + kSCol + b * kN, a, kd, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(sm.s_full[b]));
        if (k == 0) mma_commit(bar(sm.qk0_done));
      }
      __syncwarp();
    }
    if (lane == 0) mma_commit(bar(sm.qk_done));
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ============================================================ PV issue
    constexpr uint32_t idesc_pv = idesc(true, 128, kHalfDims, true);
    for (int jj = 0; jj < ntiles; ++jj) {
      const int b = jj & 1, st = jj % kStages;
      if (!warp_wait(cx, bar(sm.pv_ready[b]), (jj >> 1) & 1)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t stage = kv_addr + st * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < kN / kKStep; ++kk) {
          const uint64_t v = desc_sw128(stage + kk * (kKStep / 8) * 1024, kRegionKV, 1024);
          mma_tmem_a<true>(tmem + kOCol, tmem + kSCol + b * kN + kk * (kKStep / 4), v, idesc_pv,
                           (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(sm.kv_empty[st]));
        mma_commit(bar(sm.s_empty[b]));
      }
      __syncwarp();
    }
    if (lane == 0) mma_commit(bar(sm.o_full));
    __syncwarp();
  } else if (warp >= kSoftmaxWarp0) {
    // ============================================================ softmax / epilogue
    const int g = (warp - kSoftmaxWarp0) >> 2;         // warpgroup: tiles j % 2 == g
    const int q4 = warp & 3;                            // TMEM lane quadrant
    const int h = q4 * 32 + lane;
    const bool active = q4 * 32 < H;                    // warp-uniform
    const bool own = active && (q4 & 1) == (int)rank;   // this CTA runs the softmax of these heads
    const int oh = (q4 >> 1) * 32 + lane;               // index among the owner's heads
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    const float c = load_scale(p.bmm1, p.bmm1_dev) * kLog2e;
    constexpr uint32_t kBarStride = (uint32_t)sizeof(uint64_t);
    const uint32_t xs_bytes = (uint32_t)(nown * 32 * kN * 3);         // the peer's partial S of my heads
    const uint32_t pin_bytes = (uint32_t)(nown * 32 * (kN + 4));      // the peer's P rows and factors
    const uint32_t x_mine = base_addr + kOffX + g * kXBytes;
    const uint32_t pin_mine = base_addr + kOffPin + g * kPinBytes;
    const bool own_leader = own && (q4 >> 1) == 0 && lane == 0;       // one own thread per warpgroup
    const bool push_leader = active && !own && (q4 >> 1) == 0 && lane == 0;
    if (own_leader && g < ntiles) mbar_arrive_expect_tx(bar(sm.xs_full[g]), xs_bytes);
    if (push_leader && g < ntiles) mbar_arrive_expect_tx(bar(sm.pin_full[g]), pin_bytes);
    if (push_leader && g == 0) mbar_arrive_expect_tx(bar(sm.fin_full), (uint32_t)(nown * 32 * 4));
    const float thr = ntiles <= kExactRefTiles ? 0.f : kRescaleThreshold;
    float m_last = -INFINITY, l_run = 0.f;             // own heads: reference and row sum of my tiles
    bool ok = true;

    if (own) {
      const uint32_t x_peer_free = map_to_rank(bar(sm.xs_free[0]), peer) + g * kBarStride;
      const uint32_t pin_peer = map_to_rank(pin_mine, peer);
      const uint32_t pin_full_peer = map_to_rank(bar(sm.pin_full[0]), peer) + g * kBarStride;
      const uint4* xp = reinterpret_cast<const uint4*>(base + kOffX + g * kXBytes) + oh;
      for (int j = g; j < ntiles; j += 2) {
        const int n_cur = tile_n(j);
        const uint32_t sb = kSCol + g * kN;
        if (!(ok = warp_wait(cx, bar(sm.s_full[g]), (j >> 1) & 1))) break;
        if (!(ok = warp_wait(cx, bar(sm.xs_full[g]), (j >> 1) & 1, true))) break;
        tc_fence_after();
        // pass 1: the tile's maximum of x = (S_own + S_peer) * bmm1 * log2(e)
        float mt = -INFINITY;
#pragma unroll 1
        for (int hb = 0; hb < kN / 16; ++hb) {
          uint32_t v[16], w[12];
          float xv[16];
          tmem_ld16(tl + sb + hb * 16, v);
#pragma unroll
          for (int q = 0; q < 3; ++q) {
            const uint4 x = xp[(hb * 3 + q) * kOwnMax];
            w[4 * q] = x.x;
            w[4 * q + 1] = x.y;
            w[4 * q + 2] = x.z;
            w[4 * q + 3] = x.w;
          }
          unpack24(w, xv);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float x = (__uint_as_float(v[i]) + xv[i]) * c;
            if (hb * 16 + i < n_cur) mt = fmaxf(mt, x);
          }
        }
        // reference maximum: m(j) = mt if it exceeds m(j-1) by the threshold, else m(j-1)
        float m_prev = -INFINITY;
        if (j > 0) {
          if (!(ok = warp_wait(cx, bar(sm.m_ready[g ^ 1]), ((j - 1) >> 1) & 1))) break;
          m_prev = sm.m_buf[g ^ 1][oh];
        }
        const float m_cur = (mt > m_prev + thr) ? mt : m_prev;
        sm.m_buf[g][oh] = m_cur;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(sm.m_ready[g]));
        // pass 2: P = 2^(x - m(j)) in E4M3, and the row sum
        uint32_t pr[kPCols];
        float lt = 0.f;
#pragma unroll
        for (int hb = 0; hb < kN / 16; ++hb) {
          uint32_t v[16], w[12];
          float xv[16];
          tmem_ld16(tl + sb + hb * 16, v);
#pragma unroll
          for (int q = 0; q < 3; ++q) {
            const uint4 x = xp[(hb * 3 + q) * kOwnMax];
            w[4 * q] = x.x;
            w[4 * q + 1] = x.y;
            w[4 * q + 2] = x.z;
            w[4 * q + 3] = x.w;
          }
          unpack24(w, xv);
          tmem_wait_ld();
          float pv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float x = (__uint_as_float(v[i]) + xv[i]) * c;
            pv[i] = (hb * 16 + i < n_cur) ? fast_exp2(x - m_cur) : 0.f;
            lt += pv[i];
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) pr[hb * 4 + k] = fp8x4(pv[4 * k], pv[4 * k + 1], pv[4 * k + 2], pv[4 * k + 3]);
        }
        // this buffer of the peer's partials is read out: the peer may send tile j + 2
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_release(x_peer_free);
        if (own_leader && j + 2 < ntiles) mbar_arrive_expect_tx(bar(sm.xs_full[g]), xs_bytes);
        const float alpha = (j > 0 && m_cur != m_prev) ? fast_exp2(m_prev - m_cur) : 1.f;
        // P and the O factor to the peer, whose O rows of these heads need both
        if (j >= 2 && !(ok = warp_wait(cx, bar(sm.pin_free[g]), ((j >> 1) & 1) ^ 1, true))) break;
        {
          const uint32_t row = pin_peer + (uint32_t)(oh * kN);
#pragma unroll
          for (int k = 0; k < kN / 16; ++k)
            st_async_v4u(row + (uint32_t)(((k ^ (oh & 7)) << 4)),
                         make_uint4(pr[4 * k], pr[4 * k + 1], pr[4 * k + 2], pr[4 * k + 3]), pin_full_peer);
          st_async_b32(pin_peer + (uint32_t)(kPinAlpha + oh * 4), __float_as_uint(alpha), pin_full_peer);
        }
        // P of my heads into the S buffer (the A operand of PV)
        tmem_st32(tl + sb, pr);
        l_run *= (m_last == -INFINITY) ? 0.f : fast_exp2(m_last - m_cur);
        m_last = m_cur;
        l_run += lt;
        // O rescale when the reference moved (O holds tiles < j at m(j-1))
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          if (!(ok = warp_wait(cx, bar(sm.s_empty[g ^ 1]), ((j - 1) >> 1) & 1))) break;   // PV(j - 1) done
          tc_fence_after();
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
        if (lane == 0) mbar_arrive(bar(sm.pv_ready[g]));
      }
      sm.lsum[g][oh] = l_run;
      sm.m_end[g][oh] = m_last;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(sm.lsum_full));
    } else if (active) {
      const uint32_t x_peer = map_to_rank(x_mine, peer);
      const uint32_t xs_full_peer = map_to_rank(bar(sm.xs_full[0]), peer) + g * kBarStride;
      const uint32_t pin_free_peer = map_to_rank(bar(sm.pin_free[0]), peer) + g * kBarStride;
      const unsigned char* pin = base + kOffPin + g * kPinBytes;
      for (int j = g; j < ntiles; j += 2) {
        const uint32_t sb = kSCol + g * kN;
        if (!(ok = warp_wait(cx, bar(sm.s_full[g]), (j >> 1) & 1))) break;
        // the peer's own warps have read tile j - 2 out of the buffer this tile goes to
        if (j >= 2 && !(ok = warp_wait(cx, bar(sm.xs_free[g]), ((j >> 1) & 1) ^ 1, true))) break;
        tc_fence_after();
#pragma unroll
        for (int hb = 0; hb < kN / 16; ++hb) {
          uint32_t v[16], w[12];
          tmem_ld16(tl + sb + hb * 16, v);
          tmem_wait_ld();
          pack24(v, w);
#pragma unroll
          for (int q = 0; q < 3; ++q)
            st_async_v4u(x_peer + (uint32_t)(((hb * 3 + q) * kOwnMax + oh) * 16),
                         make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]), xs_full_peer);
        }
        // the peer's P rows and O factors of these heads
        if (!(ok = warp_wait(cx, bar(sm.pin_full[g]), (j >> 1) & 1, true))) break;
        uint32_t pr[kPCols];
        {
          const unsigned char* row = pin + oh * kN;
#pragma unroll
          for (int k = 0; k < kN / 16; ++k) {
            const uint4 x = *reinterpret_cast<const uint4*>(row + ((k ^ (oh & 7)) << 4));
            pr[4 * k] = x.x;
            pr[4 * k + 1] = x.y;
            pr[4 * k + 2] = x.z;
            pr[4 * k + 3] = x.w;
          }
        }
        const float alpha = *reinterpret_cast<const float*>(pin + kPinAlpha + oh * 4);
        tmem_st32(tl + sb, pr);
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_release(pin_free_peer);
        if (push_leader && j + 2 < ntiles) mbar_arrive_expect_tx(bar(sm.pin_full[g]), pin_bytes);
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          if (!(ok = warp_wait(cx, bar(sm.s_empty[g ^ 1]), ((j - 1) >> 1) & 1))) break;   // PV(j - 1) done
          tc_fence_after();
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
        if (lane == 0) mbar_arrive(bar(sm.pv_ready[g]));
      }
    }

    // ---- epilogue: factor per head, then this CTA's O rows (columns [128 g, 128 g + 128))
    if (active) {
      if (ok) ok = warp_wait(cx, bar(sm.lsum_full), 0);
      if (ok && ntiles > 0) {
        ok = warp_wait(cx, bar(sm.o_full), 0);
        tc_fence_after();
      }
      float f = 0.f;
      if (own) {
        float l_tot = 0.f, m_fin = -INFINITY;
        if (ok) {
          const float ma = sm.m_end[0][oh], mb = sm.m_end[1][oh];
          m_fin = fmaxf(ma, mb);
          if (m_fin != -INFINITY) {
            if (ma != -INFINITY) l_tot += sm.lsum[0][oh] * fast_exp2(ma - m_fin);
            if (mb != -INFINITY) l_tot += sm.lsum[1][oh] * fast_exp2(mb - m_fin);
          }
        }
        const bool have = ok && ntiles > 0 && l_tot > 0.f;
        const float lse = have ? m_fin + fast_log2(l_tot) : -INFINITY;
        f = have ? 1.f / l_tot : 0.f;
        if (S == 1) {
          f *= load_scale(p.bmm2, p.bmm2_dev);
          if (p.sinks != nullptr && have) f *= 1.f / (1.f + fast_exp2(__ldg(p.sinks + h) * kLog2e - lse));
        }
        if (g == 0) {
          const int64_t row_th = (int64_t)t * H + h;
          if (S == 1) {
            if (p.out_lse) p.out_lse[row_th] = lse;
          } else {
            p.part_lse[row_th * S + s] = lse;
          }
          st_async_b32(map_to_rank(base_addr + kOffFin + oh * 4, peer), __float_as_uint(f),
                       map_to_rank(bar(sm.fin_full), peer));
        }
      } else {
        if (ok) ok = warp_wait(cx, bar(sm.fin_full), 0, true);
        f = ok ? *reinterpret_cast<const float*>(base + kOffFin + oh * 4) : 0.f;
      }
      const bool have = ok && ntiles > 0;
      const int64_t row_th = (int64_t)t * H + h;
      __nv_bfloat16* dst = kPartial ? p.part_o + (row_th * S + s) * kHeadDim : p.out + row_th * kHeadDim;
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
        uint4* o = reinterpret_cast<uint4*>(dst + (int)rank * kHalfDims + col);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          o[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                            pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == kQkWarp0) {
    drain_wait(bar(sm.qk_done), 0);
    drain_wait(bar(sm.o_full), 0);
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  tc_fence_before();
  cluster_sync();
}

}  // namespace

int tc_head_owned_smem_bytes() { return kSmemBytes; }
int tc_head_owned_threads() { return kThreads; }

cudaError_t launch_decode_tc_head_owned(const DecodeParams& p, int grid, cudaStream_t stream) {
  TcParams P;
  memset(&P, 0, sizeof(P));
  P.p = p;
  const int swa_run = (int)std::max<int64_t>(1, std::min<int64_t>(kN, p.swa_rows));
  const int comp_run = (int)std::max<int64_t>(1, std::min<int64_t>(kN, p.comp_rows));
  cudaError_t e = encode_pool_map(&P.tm_swa, p.swa, p.swa_rows, p.swa_stride, p.dtype, 1);
  if (e == cudaSuccess) e = encode_pool_map(&P.tm_comp, p.comp, p.comp_rows, p.comp_stride, p.dtype, 1);
  if (e == cudaSuccess) e = encode_pool_map(&P.tm_swa_run, p.swa, p.swa_rows, p.swa_stride, p.dtype, swa_run);
  if (e == cudaSuccess) e = encode_pool_map(&P.tm_comp_run, p.comp, p.comp_rows, p.comp_stride, p.dtype, comp_run);
  if (e != cudaSuccess) return e;
  auto launch = [&](auto kernel) -> cudaError_t {
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    kernel<<<grid, kThreads, kSmemBytes, stream>>>(P);
    return cudaSuccess;
  };
  e = p.num_splits > 1 ? launch(decode_tc_head_owned_kernel<true>) : launch(decode_tc_head_owned_kernel<false>);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace smla
