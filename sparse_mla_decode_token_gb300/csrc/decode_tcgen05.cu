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

constexpr int kN = 64;              // slots per tile
constexpr int kHalfDims = 256;      // output dims per CTA
constexpr int kThreads = 288;       // 4 producer warps, 1 MMA warp, 4 softmax warps
constexpr int kProducerThreads = 128;
constexpr int kMmaWarp = 4;          // warps 5-8 run the softmax and the epilogue
constexpr int kMaxCols = SMLA_TC_MAX_SPLIT_COLS;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;       // O: 256 fp32 columns
constexpr uint32_t kSCol = 256;     // S: two buffers of 64 fp32 columns
constexpr float kRescaleThreshold = 8.f;   // log2 units: P stays <= 2^8
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct TcSmall {
  uint64_t q_full;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2];
  uint64_t xin_full, xout_free, o_full;
  int32_t meta_n[8];
  int32_t rows[2][kN];
  int32_t rows_n[2];
  uint32_t tmem_base;
  int32_t abort_flag;
};

template <bool kFp8>
struct Cfg {
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kRegions = kHalfDims * kElem / 128;     // 128-byte column blocks per half row
  static constexpr int kChunks = kHalfDims * kElem / 16;       // 16-byte chunks per half row
  static constexpr int kStages = kFp8 ? 4 : 2;
  static constexpr int kKStep = 32 / kElem;                    // MMA K per instruction
  static constexpr int kK1 = kHalfDims / kKStep;               // QK K steps
  static constexpr int kK2 = kN / kKStep;                      // PV K steps
  static constexpr int kRegionQ = 128 * 128;                   // 128 rows x 128 B
  static constexpr int kRegionKV = kN * 128;                   // 64 rows x 128 B
  static constexpr int kQBytes = kRegions * kRegionQ;
  static constexpr int kStageBytes = kRegions * kRegionKV;
  static constexpr int kPBytes = 128 * 128;
  static constexpr int kXBytes = 128 * kN * 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQBytes;
  static constexpr int kOffP = kOffKV + kStages * kStageBytes;
  static constexpr int kOffX = kOffP + 2 * kPBytes;
  static constexpr int kOffIdx = kOffX + kXBytes;
  static constexpr int kOffSmall = kOffIdx + kMaxCols * 4;
  static constexpr int kSmemBytes = kOffSmall + (int)sizeof(TcSmall) + 1024;   // + alignment slack
  static_assert(kStages <= 8, "barrier arrays hold 8 stages");
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
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  unsigned char* base = smem_raw + (base_addr - raw_addr);
  TcSmall& sm = *reinterpret_cast<TcSmall*>(base + C::kOffSmall);
  int32_t* idx_s = reinterpret_cast<int32_t*>(base + C::kOffIdx);
  const uint32_t q_addr = base_addr + C::kOffQ;
  const uint32_t kv_addr = base_addr + C::kOffKV;
  const uint32_t p_addr = base_addr + C::kOffP;
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
    // zero the KV stages and P buffers (rows past a tile's slot count then hold
    // finite data), and the Q rows of absent heads
    const uint4 z = make_uint4(0, 0, 0, 0);
    uint4* zp = reinterpret_cast<uint4*>(base + C::kOffKV);
    const int zn = (C::kOffX - C::kOffKV) / 16;
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
        mbar_init(bar(sm.s_empty[b]), 128);
        mbar_init(bar(sm.p_full[b]), 128);
        mbar_init(bar(sm.p_empty[b]), 1);
      }
      mbar_init(bar(sm.xin_full), 128);
      mbar_init(bar(sm.xout_free), 128);
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
        // next tile: up to 64 valid slots of one pool, in column order
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
    constexpr uint32_t idesc_qk = idesc(kFp8, 128, kN, false);
    constexpr uint32_t idesc_pv = idesc(kFp8, 128, kHalfDims, true);
    bool ok = warp_wait(cx, bar(sm.q_full), 0);
    int j = 0;
    auto issue_pv = [&](int jj) -> bool {
      const int b = jj & 1, st = jj % C::kStages;
      if (!warp_wait(cx, bar(sm.p_full[b]), (jj >> 1) & 1)) return false;
      fence_proxy_async_smem();
      tc_fence_after();
      if (lane == 0) {
        const uint32_t stage = kv_addr + st * C::kStageBytes;
#pragma unroll
        for (int k = 0; k < C::kK2; ++k) {
          const uint64_t a = desc_sw128(p_addr + b * C::kPBytes + k * 32, 16, 1024);
          const uint64_t v = desc_sw128(stage + k * (C::kKStep / 8) * 1024, C::kRegionKV, 1024);
          mma<kFp8>(tmem + kOCol, a, v, idesc_pv, (jj > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(bar(sm.p_empty[b]));
        mma_commit(bar(sm.kv_empty[st]));
      }
      __syncwarp();
      return true;
    };
    if (ok) {
      for (;; ++j) {
        const int st = j % C::kStages;
        if (!warp_wait(cx, bar(sm.kv_full[st]), (j / C::kStages) & 1)) { ok = false; break; }
        const int n = sm.meta_n[st];
        if (n == 0) break;
        const int b = j & 1;
        if (!warp_wait(cx, bar(sm.s_empty[b]), ((j >> 1) & 1) ^ 1)) { ok = false; break; }
        fence_proxy_async_smem();
        tc_fence_after();
        if (lane == 0) {
          const uint32_t stage = kv_addr + st * C::kStageBytes;
#pragma unroll
          for (int k = 0; k < C::kK1; ++k) {
            const uint64_t a = desc_sw128(q_addr + (k >> 2) * C::kRegionQ + (k & 3) * 32, 16, 1024);
            const uint64_t kd = desc_sw128(stage + (k >> 2) * C::kRegionKV + (k & 3) * 32, 16, 1024);
            mma<kFp8>(tmem + kSCol + b * kN, a, kd, idesc_qk, k > 0 ? 1u : 0u);
          }
          mma_commit(bar(sm.s_full[b]));
        }
        __syncwarp();
        if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && j > 0) ok = issue_pv(j - 1);
    }
    if (lane == 0) mma_commit(bar(sm.o_full));    // completes once every MMA issued above is done
    __syncwarp();
  } else {
    // ============================================================ softmax / epilogue
    const int q4 = warp & 3;                           // TMEM lane quadrant of this warp
    const int h = q4 * 32 + lane;
    const bool active = q4 * 32 < H;                   // warp-uniform
    const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
    const float c = load_scale(p.bmm1, p.bmm1_dev) * kLog2e;
    const uint32_t x_peer = map_to_rank(x_addr, peer);
    const uint32_t xin_full_peer = map_to_rank(bar(sm.xin_full), peer);
    const uint32_t xout_free_peer = map_to_rank(bar(sm.xout_free), peer);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int j = 0;
    for (;; ++j) {
      const int st = j % C::kStages;
      if (!(ok = warp_wait(cx, bar(sm.kv_full[st]), (j / C::kStages) & 1))) break;
      const int n = sm.meta_n[st];
      if (n == 0) break;
      const int b = j & 1;
      if (!(ok = warp_wait(cx, bar(sm.s_full[b]), (j >> 1) & 1))) break;
      tc_fence_after();
      float sv[kN];
      if (active) {
        uint32_t r0[32], r1[32];
        tmem_ld32(tl + kSCol + b * kN, r0);
        tmem_ld32(tl + kSCol + b * kN + 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          sv[i] = __uint_as_float(r0[i]);
          sv[32 + i] = __uint_as_float(r1[i]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(sm.s_empty[b]));
      // S = S_0 + S_1: push my partial to the peer, add the peer's partial
      if (!(ok = warp_wait(cx, bar(sm.xout_free), (j & 1) ^ 1, true))) break;
      if (active) {
#pragma unroll
        for (int c4 = 0; c4 < kN / 4; ++c4)
          st_cluster_v4(x_peer + (uint32_t)((c4 * 128 + h) * 16), sv[4 * c4], sv[4 * c4 + 1], sv[4 * c4 + 2],
                        sv[4 * c4 + 3]);
      }
      mbar_arrive_cluster(xin_full_peer);
      if (!(ok = warp_wait(cx, bar(sm.xin_full), j & 1, true))) break;
      if (active) {
#pragma unroll
        for (int c4 = 0; c4 < kN / 4; ++c4) {
          const float4 v = ld_shared_v4(x_addr + (uint32_t)((c4 * 128 + h) * 16));
          sv[4 * c4] += v.x;
          sv[4 * c4 + 1] += v.y;
          sv[4 * c4 + 2] += v.z;
          sv[4 * c4 + 3] += v.w;
        }
      }
      mbar_arrive_cluster(xout_free_peer);
      // online softmax, base 2, lazy rescale
      bool rescale = false;
      float alpha = 1.f;
      if (active) {
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < kN; ++i) {
          sv[i] = (i < n) ? sv[i] * c : -INFINITY;
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
        const uint32_t prow = p_addr + b * C::kPBytes;
        if constexpr (kFp8) {
#pragma unroll
          for (int c16 = 0; c16 < kN / 16; ++c16) {
            const float* v = sv + 16 * c16;
            st_shared_v4(prow + sw128_offset(h, c16), pack_e4m3x4(v[0], v[1], v[2], v[3]),
                         pack_e4m3x4(v[4], v[5], v[6], v[7]), pack_e4m3x4(v[8], v[9], v[10], v[11]),
                         pack_e4m3x4(v[12], v[13], v[14], v[15]));
          }
        } else {
#pragma unroll
          for (int c8 = 0; c8 < kN / 8; ++c8) {
            const float* v = sv + 8 * c8;
            st_shared_v4(prow + sw128_offset(h, c8), pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                         pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(sm.p_full[b]));
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
          for (int k = 0; k < 4; ++k)
            o[k] = make_uint4(pack_bf16x2(v[8 * k], v[8 * k + 1]), pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                              pack_bf16x2(v[8 * k + 4], v[8 * k + 5]), pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
        } else {
          float4* o = reinterpret_cast<float4*>(p.part_o + (row_th * S + s) * kHeadDim + d0);
#pragma unroll
          for (int k = 0; k < 8; ++k) o[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
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
