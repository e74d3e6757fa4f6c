// tcgen05 / TMEM sparse MLA decode kernel for sm_103a.
//
// Work unit: one (token, split) runs on a cluster of two CTAs.  CTA r of the
// pair owns output dims [256 r, 256 r + 256): an fp32 accumulator for 128 heads
// x 512 dims is 256 KB, the whole tensor memory of one SM, so the output is
// split across the pair.  Per tile of up to 64 selected slots:
//
//   producer warps 0-3  gather the pair's half of every selected row (256 dims)
//                       with 16-byte cp.async into a 128-byte-swizzled,
//                       UMMA-canonical shared-memory tile (index compaction first:
//                       masked slots are never loaded)
//   MMA warp 4          S_r = Q_r K_r^T   (M = 128 heads, N = 64 slots, K = 256 dims)
//                       O_r += P V_r      (M = 128 heads, N = 256 dims, K = 64 slots)
//                       one elected thread issues tcgen05.mma, accumulators in TMEM
//   softmax warps 5-8   one thread per head: read S_r from TMEM, send it to the
//                       peer CTA through distributed shared memory, add the
//                       peer's half (S = S_0 + S_1, identical in both CTAs),
//                       online softmax in base 2 with lazy rescaling of O, write
//                       P (BF16 or E4M3) for the PV MMA; finally normalise O and
//                       store it (BF16 output or fp32 split partial) plus LSE.
//
// The operation follows the FlashInfer trtllm_batch_decode_sparse_mla_dsv4 page
// (description, SM100/SM103 paragraph; Parameters); the base-2 LSE, the sink in
// the normaliser and the split partials follow the cake_sparse_mla_sm120 page
// (Parameters: out_lse, attn_sink, mid_out / mid_lse).
//
// Every mbarrier wait is bounded (2 s); on expiry the CTA raises an abort flag,
// ORs SMLA_DEVERR_TIMEOUT into the error word, lets every role leave its loop,
// waits for its own copies and MMAs, frees its TMEM and returns.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;

constexpr int kMaxN = 64;           // largest tile (slots per tile)
constexpr int kHalfDims = 256;      // output dims per CTA
constexpr int kThreads = 288;       // 4 producer warps, 1 MMA warp, 4 softmax warps
constexpr int kProducerThreads = 128;
constexpr int kMmaWarp = 4;          // warps 5-8 run the softmax and the epilogue
constexpr int kSoftmaxWarp0 = 5;
constexpr int kMaxCols = SMLA_TC_MAX_SPLIT_COLS;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;       // O: 256 fp32 columns
constexpr uint32_t kSCol = 256;     // S: two buffers of N fp32 columns, then P: two buffers of 16 columns
constexpr float kRescaleThreshold = 8.f;   // log2 units: P stays <= 2^8
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kMaxStages = 8;

struct TcSmall {
  uint64_t q_full;
  uint64_t kv_full[kMaxStages];
  uint64_t kv_empty[kMaxStages];
  uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2];
  uint64_t xin_full[2], xout_free[2];
  uint64_t o_full;
  int32_t meta_n[kMaxStages];
  int32_t rows[2][kMaxN];
  int32_t rows_n[2];
  uint32_t tmem_base;
  int32_t abort_flag;
};

template <bool kFp8>
struct Cfg {
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kN = kFp8 ? 64 : 32;                    // slots per tile
  static constexpr int kRegions = kHalfDims * kElem / 128;     // 128-byte column blocks per half row
  static constexpr int kChunks = kHalfDims * kElem / 16;       // 16-byte chunks per half row
  static constexpr int kStages = 6;
  static constexpr int kKStep = 32 / kElem;                    // MMA K per instruction
  static constexpr int kK1 = kHalfDims / kKStep;               // QK K steps
  static constexpr int kK2 = kN / kKStep;                      // PV K steps
  static constexpr int kPCols = kN * kElem / 4;                // TMEM columns of one P buffer
  static constexpr uint32_t kPCol = kSCol + 2 * kN;
  static constexpr int kRegionQ = 128 * 128;                   // 128 rows x 128 B
  static constexpr int kRegionKV = kN * 128;                   // N rows x 128 B
  static constexpr int kQBytes = kRegions * kRegionQ;
  static constexpr int kStageBytes = kRegions * kRegionKV;
  static constexpr int kXBytes = 128 * kN * 4;                 // one exchange buffer (fp32 S rows)
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQBytes;
  static constexpr int kOffX = kOffKV + kStages * kStageBytes;
  static constexpr int kOffIdx = kOffX + 2 * kXBytes;
  static constexpr int kOffSmall = kOffIdx + kMaxCols * 4;
  static constexpr int kSmemBytes = kOffSmall + (int)sizeof(TcSmall) + 1024;   // + alignment slack
  static_assert(kStages <= kMaxStages, "barrier arrays");
  static_assert(kN <= kMaxN, "row lists");
  static_assert(kPCol + 2 * kPCols <= kTmemCols, "tensor memory budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct Ctx {
  int32_t* abort_flag;
  int32_t* err;
};

__device__ __forceinline__ bool wait_bar(const Ctx& cx, uint32_t bar, uint32_t parity, bool cluster_scope) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    bool done = cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    if (done) return true;
    if ((it & 63u) == 63u) {
      if (*reinterpret_cast<volatile int32_t*>(cx.abort_flag)) return false;
      uint64_t now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kTimeoutNs) {
        *reinterpret_cast<volatile int32_t*>(cx.abort_flag) = 1;
        if (cx.err) atomicOr(cx.err, SMLA_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// All lanes of the warp wait; the result is warp-uniform.
__device__ __forceinline__ bool warp_wait(const Ctx& cx, uint32_t bar, uint32_t parity, bool cluster_scope = false) {
  bool ok = wait_bar(cx, bar, parity, cluster_scope);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Byte offset of 16-byte chunk `ch` (0..7) of row `r` in a 128-byte-swizzled
// K-major region whose 8-row groups are 1024 bytes apart.
__device__ __forceinline__ uint32_t sw128_offset(int r, int ch) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ DecodeParams p) {
  using C = Cfg<kFp8>;
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
  const int S = p.num_splits;
  const int unit = blockIdx.x >> 1;
  const int s = unit % S;
  const int t = unit / S;
  const TokenInfo ti = token_info(p, t);
  int c0, c1;
  split_range(ti.n_lim, S, s, &c0, &c1);
  if (c1 - c0 > kMaxCols) {           // the planner prevents this; never read past the staging buffer
    if (p.err && tid == 0) atomicOr(p.err, SMLA_DEVERR_INTERNAL);
    c1 = c0 + kMaxCols;
  }
  const int ncols = c1 - c0;
  const int H = p.H;

  auto bar = [&](const uint64_t& b) { return smem_addr(&b); };

  // ---------------------------------------------------------------- set-up
  {
    // zero the KV stages (rows past a tile's slot count then hold finite data)
    // and the Q rows of absent heads
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
    const int32_t* irow = p.ind + (int64_t)t * p.ind_stride + c0;
    for (int i = tid; i < ncols; i += kThreads) idx_s[i] = __ldg(irow + i);
    if (tid == 0) {
      mbar_init(bar(sm.q_full), kProducerThreads);
      for (int i = 0; i < C::kStages; ++i) {
        mbar_init(bar(sm.kv_full[i]), kProducerThreads + 1);
        mbar_init(bar(sm.kv_empty[i]), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(bar(sm.s_full[b]), 1);
        mbar_init(bar(sm.s_empty[b]), 4);
        mbar_init(bar(sm.p_full[b]), 4);
        mbar_init(bar(sm.p_empty[b]), 1);
        mbar_init(bar(sm.xin_full[b]), 1);
        mbar_init(bar(sm.xout_free[b]), 4);
      }
      mbar_init(bar(sm.o_full), 1);
      sm.abort_flag = 0;
      fence_mbar_init_cluster();
    }
    if (warp == kMmaWarp) tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
    fence_proxy_async_smem();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
  }
  const uint32_t tmem = sm.tmem_base;
  const Ctx cx{&sm.abort_flag, p.err};

  if (warp < kMmaWarp) {
    // ============================================================ producer
    const int ptid = tid;
    {
      const unsigned char* qb = reinterpret_cast<const unsigned char*>(p.q) +
                                ((int64_t)t * p.q_stride_token + (int64_t)rank * kHalfDims) * C::kElem;
      for (int c = ptid; c < H * C::kChunks; c += kProducerThreads) {
        const int h = c / C::kChunks, cc = c % C::kChunks;
        cp_async_16(q_addr + (cc >> 3) * C::kRegionQ + sw128_offset(h, cc & 7),
                    qb + (int64_t)h * kHeadDim * C::kElem + cc * 16);
      }
      cp_async_arrive_noinc(bar(sm.q_full));
    }
    // index compaction state (warp 0 only)
    int seg = 0, cursor = 0;
    for (int j = 0;; ++j) {
      const int st = j % C::kStages;
      wait_bar(cx, bar(sm.kv_empty[st]), ((j / C::kStages) & 1) ^ 1, false);
      if (warp == 0) {
        // next tile: up to N valid slots of one pool, in column order
        int cnt = 0, pool = 0;
        while (cnt < kN && seg < 2) {
          const int lo = seg == 0 ? c0 : max(c0, kSwaCols);
          const int hi = seg == 0 ? min(c1, kSwaCols) : c1;
          if (cursor < lo) cursor = lo;
          if (cursor >= hi) {
            ++seg;
            if (cnt > 0) break;
            continue;
          }
          const int col = cursor + lane;
          int row = -1;
          if (col < hi) {
            const int idx = idx_s[col - c0];
            bool ok = idx != -1 && (seg == 1 || col < ti.w_swa);
            if (ok) {
              const int64_t nrows = seg == 0 ? p.swa_rows : p.comp_rows;
              if (idx < 0 || (int64_t)idx >= nrows) {
                ok = false;
                if (p.err && rank == 0) atomicOr(p.err, SMLA_DEVERR_INDEX_OUT_OF_RANGE);
              }
            }
            if (ok) row = idx;
          }
          const unsigned ball = __ballot_sync(0xffffffffu, row >= 0);
          const int nv = __popc(ball);
          const int room = kN - cnt;
          const int rk = __popc(ball & ((1u << lane) - 1u));
          if (row >= 0 && rk < room) sm.rows[j & 1][cnt + rk] = row;
          if (nv > 0) pool = seg;
          if (nv <= room) {
            cnt += nv;
            cursor = min(cursor + 32, hi);
          } else {
            const unsigned last = __ballot_sync(0xffffffffu, row >= 0 && rk == room - 1);
            cursor += __ffs(last);       // column after the last slot taken
            cnt = kN;
          }
        }
        const bool stop = cnt == 0 || *reinterpret_cast<volatile int32_t*>(&sm.abort_flag) != 0;
        if (lane == 0) sm.rows_n[j & 1] = stop ? 0 : (cnt | (pool << 16));
      }
      named_barrier_sync(1, kProducerThreads);
      const int packed = sm.rows_n[j & 1];
      const int n = packed & 0xffff;
      if (n == 0) {
        cp_async_arrive_noinc(bar(sm.kv_full[st]));
        if (ptid == 0) {
          sm.meta_n[st] = 0;
          mbar_arrive(bar(sm.kv_full[st]));
        }
        break;
      }
      const bool swa_pool = (packed >> 16) == 0;
      const unsigned char* pool_base = reinterpret_cast<const unsigned char*>(swa_pool ? p.swa : p.comp);
      const int64_t stride = swa_pool ? p.swa_stride : p.comp_stride;
      const uint32_t stage = kv_addr + st * C::kStageBytes;
      for (int c = ptid; c < n * C::kChunks; c += kProducerThreads) {
        const int r = c / C::kChunks, cc = c % C::kChunks;
        const int64_t row = sm.rows[j & 1][r];
        cp_async_16(stage + (cc >> 3) * C::kRegionKV + sw128_offset(r, cc & 7),
                    pool_base + (row * stride + (int64_t)rank * kHalfDims) * C::kElem + cc * 16);
      }
      cp_async_arrive_noinc(bar(sm.kv_full[st]));
      if (ptid == 0) {
        sm.meta_n[st] = n;
        mbar_arrive(bar(sm.kv_full[st]));
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaWarp) {
    // ============================================================ MMA issue
    // Order: QK of tile k, then PV of tile k-2, so that QK runs two tiles ahead
    // of the softmax and PV never waits behind a QK.
    constexpr uint32_t idesc_qk = idesc(kFp8, 128, kN, false);
    constexpr uint32_t idesc_pv = idesc(kFp8, 128, kHalfDims, true);
    bool ok = warp_wait(cx, bar(sm.q_full), 0);
    int k = 0;
    auto issue_pv = [&](int jj) -> bool {
      const int b = jj & 1, st = jj % C::kStages;
      if (!warp_wait(cx, bar(sm.p_full[b]), (jj >> 1) & 1)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t stage = kv_addr + st * C::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < C::kK2; ++kk) {
          const uint64_t v = desc_sw128(stage + kk * (C::kKStep / 8) * 1024, C::kRegionKV, 1024);
          mma_tmem_a<kFp8>(tmem + kOCol, tmem + C::kPCol + b * C::kPCols + kk * (C::kKStep * C::kElem / 4), v,
                           idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(sm.p_empty[b]));
        mma_commit(bar(sm.kv_empty[st]));
      }
      __syncwarp();
      return true;
    };
    if (ok) {
      for (;; ++k) {
        const int st = k % C::kStages;
        if (!warp_wait(cx, bar(sm.kv_full[st]), (k / C::kStages) & 1)) { ok = false; break; }
        const int n = sm.meta_n[st];
        if (n == 0) break;
        const int b = k & 1;
        if (!warp_wait(cx, bar(sm.s_empty[b]), ((k >> 1) & 1) ^ 1)) { ok = false; break; }
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
        }
        __syncwarp();
        if (k >= 2 && !issue_pv(k - 2)) { ok = false; break; }
      }
      for (int jj = max(0, k - 2); ok && jj < k; ++jj) ok = issue_pv(jj);
    }
    if (lane == 0) mma_commit(bar(sm.o_full));    // completes once every MMA issued above is done
    __syncwarp();
  } else {
    // ============================================================ softmax / epilogue
    const int q4 = warp & 3;                           // TMEM lane quadrant of this warp
    const int h = q4 * 32 + lane;
    const bool active = q4 * 32 < H;                   // warp-uniform
    const bool leader = warp == kSoftmaxWarp0 && lane == 0;
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    const float c = load_scale(p.bmm1, p.bmm1_dev) * kLog2e;
    const uint32_t xbytes = (uint32_t)(H * kN * 4);    // bytes the peer pushes per tile
    // peer addresses of exchange buffer / barrier b are these plus b * (stride)
    const uint32_t x_peer0 = map_to_rank(x_addr, peer);
    const uint32_t xin_full_peer0 = map_to_rank(bar(sm.xin_full[0]), peer);
    const uint32_t xout_free_peer0 = map_to_rank(bar(sm.xout_free[0]), peer);
    constexpr uint32_t kBarStride = (uint32_t)sizeof(uint64_t);
    if (leader) {
      mbar_arrive_expect_tx(bar(sm.xin_full[0]), xbytes);
      mbar_arrive_expect_tx(bar(sm.xin_full[1]), xbytes);
    }
    if (!active) {
      // rows of absent heads: P = 0 in both buffers, so O and S stay 0 there
      uint32_t zr[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) zr[i] = 0u;
      tmem_st16(tl + C::kPCol, zr);
      tmem_st16(tl + C::kPCol + C::kPCols, zr);
      tmem_wait_st();
    }
    // load this CTA's partial S of tile jj into v (warp-collective)
    auto load_s = [&](int jj, float (&v)[kN]) {
      uint32_t r[32];
#pragma unroll
      for (int h32 = 0; h32 < kN / 32; ++h32) {
        tmem_ld32(tl + kSCol + (jj & 1) * kN + h32 * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[h32 * 32 + i] = __uint_as_float(r[i]);
      }
    };
    // send this CTA's partial S of tile jj to the peer (tile jj's S must be ready)
    auto push = [&](int jj) -> bool {
      const int b = jj & 1;
      if (!warp_wait(cx, bar(sm.s_full[b]), (jj >> 1) & 1)) return false;
      tc_fence_after();
      if (jj >= 2 && !warp_wait(cx, bar(sm.xout_free[b]), ((jj >> 1) & 1) ^ 1, true)) return false;
      if (active) {
        float v[kN];
        load_s(jj, v);
#pragma unroll
        for (int c4 = 0; c4 < kN / 4; ++c4)
          st_async_v4(x_peer0 + b * C::kXBytes + (uint32_t)((c4 * 128 + h) * 16), v[4 * c4], v[4 * c4 + 1],
                      v[4 * c4 + 2], v[4 * c4 + 3], xin_full_peer0 + b * kBarStride);
      }
      return true;
    };

    float m_run = -INFINITY, l_run = 0.f;
    bool ok = warp_wait(cx, bar(sm.kv_full[0]), 0);
    int n_cur = ok ? sm.meta_n[0] : 0;
    if (n_cur > 0) ok = push(0);
    int j = 0;
    while (ok && n_cur > 0) {
      // ---- consume tile j: S = S_0 + S_1
      const int b = j & 1;
      if (!(ok = warp_wait(cx, bar(sm.xin_full[b]), (j >> 1) & 1, true))) break;
      tc_fence_after();
      float sv[kN];
      if (active) {
        load_s(j, sv);
#pragma unroll
        for (int c4 = 0; c4 < kN / 4; ++c4) {
          const float4 v = ld_shared_v4(x_addr + b * C::kXBytes + (uint32_t)((c4 * 128 + h) * 16));
          sv[4 * c4] += v.x;
          sv[4 * c4 + 1] += v.y;
          sv[4 * c4 + 2] += v.z;
          sv[4 * c4 + 3] += v.w;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(sm.s_empty[b]));                    // S buffer b may be overwritten
        mbar_arrive_cluster_relaxed(xout_free_peer0 + b * kBarStride);   // exchange buffer b read out
      }
      if (leader) mbar_arrive_expect_tx(bar(sm.xin_full[b]), xbytes);   // for tile j + 2
      // ---- look ahead: push tile j+1 so that the exchange overlaps this tile's softmax
      const int st1 = (j + 1) % C::kStages;
      if (!(ok = warp_wait(cx, bar(sm.kv_full[st1]), ((j + 1) / C::kStages) & 1))) break;
      const int n_next = sm.meta_n[st1];
      if (n_next > 0 && !(ok = push(j + 1))) break;
      // ---- online softmax, base 2, lazy rescale
      bool rescale = false;
      float alpha = 1.f;
      if (active) {
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < kN; ++i) {
          sv[i] = (i < n_cur) ? sv[i] * c : -INFINITY;
          mx = fmaxf(mx, sv[i]);
        }
        if (mx > m_run + kRescaleThreshold) {
          rescale = true;
          alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - mx);
          l_run *= alpha;
          m_run = mx;
        }
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < kN; ++i) {
          sv[i] = fast_exp2(sv[i] - m_run);
          sum += sv[i];
        }
        l_run += sum;
      }
      if (!(ok = warp_wait(cx, bar(sm.p_empty[b]), ((j >> 1) & 1) ^ 1))) break;
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
        // O must hold tile j-1's contribution before it is rescaled
        if (!(ok = warp_wait(cx, bar(sm.p_empty[(j - 1) & 1]), ((j - 1) >> 1) & 1))) break;
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < kHalfDims / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32(tl + kOCol + cc * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tl + kOCol + cc * 32, r);
        }
        tmem_wait_st();
      }
      if (active) {
        uint32_t pr[16];
        if constexpr (kFp8) {
#pragma unroll
          for (int i = 0; i < 16; ++i) pr[i] = pack_e4m3x4(sv[4 * i], sv[4 * i + 1], sv[4 * i + 2], sv[4 * i + 3]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) pr[i] = pack_bf16x2(sv[2 * i], sv[2 * i + 1]);
        }
        tmem_st16(tl + C::kPCol + b * C::kPCols, pr);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(sm.p_full[b]));
      ++j;
      n_cur = n_next;
    }
    const int ntiles = j;
    if (ok && ntiles > 0) {
      ok = warp_wait(cx, bar(sm.o_full), 0);
      tc_fence_after();
    }
    if (active) {
      const bool have = ok && ntiles > 0 && l_run > 0.f;
      const float lse = have ? m_run + fast_log2(l_run) : -INFINITY;
      float f = have ? 1.f / l_run : 0.f;
      if (S == 1) {
        f *= load_scale(p.bmm2, p.bmm2_dev);
        if (p.sinks != nullptr && have) f *= 1.f / (1.f + fast_exp2(__ldg(p.sinks + h) * kLog2e - lse));
      }
      const int64_t row_th = (int64_t)t * H + h;
#pragma unroll 1
      for (int cc = 0; cc < kHalfDims / 32; ++cc) {
        float v[32];
        if (ok && ntiles > 0) {
          uint32_t r[32];
          tmem_ld32(tl + kOCol + cc * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * f;
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        const int d0 = (int)rank * kHalfDims + cc * 32;
        if (S == 1) {
          uint4* o = reinterpret_cast<uint4*>(p.out + row_th * kHeadDim + d0);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            o[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                              pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
        } else {
          float4* o = reinterpret_cast<float4*>(p.part_o + (row_th * S + s) * kHeadDim + d0);
#pragma unroll
          for (int q = 0; q < 8; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
      if (rank == 0) {
        if (S == 1) {
          if (p.out_lse) p.out_lse[row_th] = lse;
        } else {
          p.part_lse[row_th * S + s] = lse;
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == kMmaWarp) {
    warp_wait(cx, bar(sm.o_full), 0);     // no MMA may still write TMEM
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  tc_fence_before();
  cluster_sync();                          // the peer is done with this CTA's shared memory
}

}  // namespace

int tc_smem_bytes(int dtype) { return dtype == SMLA_BF16 ? Cfg<false>::kSmemBytes : Cfg<true>::kSmemBytes; }
int tc_threads() { return kThreads; }

cudaError_t launch_decode_tc(const DecodeParams& p, int grid, cudaStream_t stream) {
  const int smem = tc_smem_bytes(p.dtype);
  cudaError_t e;
  if (p.dtype == SMLA_BF16) {
    e = cudaFuncSetAttribute(decode_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    decode_tc_kernel<false><<<grid, kThreads, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(decode_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    decode_tc_kernel<true><<<grid, kThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace smla
