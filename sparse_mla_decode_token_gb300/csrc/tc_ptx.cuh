// Thin inline-PTX wrappers for sm_103a: mbarriers, cp.async, cluster shared
// memory, tcgen05 (TMEM allocation, MMA, loads/stores, commits, fences).
// Each wrapper is one or two PTX instructions as documented in the PTX ISA.
#pragma once

#include <stdint.h>

namespace smla {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init_cluster() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// The waiting thread is suspended (it issues nothing) until the phase
// completes or the hinted time, in nanoseconds, has passed.
constexpr uint32_t kSuspendHintNs = 200000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity), "r"(kSuspendHintNs) : "memory");
  return ok != 0;
}

// Wait with cluster-scope acquire: for barriers that other CTAs arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity), "r"(kSuspendHintNs) : "memory");
  return ok != 0;
}

// ---------------------------------------------------------------- cp.async

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// The barrier receives one arrival once all of this thread's prior cp.async
// copies have landed (the arrival counts toward the expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T for kind::f16 (BF16 inputs) or kind::f8f6f4 (E4M3).
template <bool kFp8>
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                    uint32_t accumulate) {
  if constexpr (kFp8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// The barrier receives one arrival once every prior tcgen05 op of this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

#define SMLA_R32(i) "=r"(r[i])
// 32 consecutive 32-bit TMEM columns of this thread's lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : SMLA_R32(0), SMLA_R32(1), SMLA_R32(2), SMLA_R32(3), SMLA_R32(4), SMLA_R32(5), SMLA_R32(6), SMLA_R32(7),
        SMLA_R32(8), SMLA_R32(9), SMLA_R32(10), SMLA_R32(11), SMLA_R32(12), SMLA_R32(13), SMLA_R32(14),
        SMLA_R32(15), SMLA_R32(16), SMLA_R32(17), SMLA_R32(18), SMLA_R32(19), SMLA_R32(20), SMLA_R32(21),
        SMLA_R32(22), SMLA_R32(23), SMLA_R32(24), SMLA_R32(25), SMLA_R32(26), SMLA_R32(27), SMLA_R32(28),
        SMLA_R32(29), SMLA_R32(30), SMLA_R32(31)
      : "r"(taddr)
      : "memory");
}
#undef SMLA_R32


__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format: start,
// leading and stride byte offsets in 16-byte units, version 1 at bit 46,
// swizzle mode 2 at bits 61-63).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor for kind::f16 (BF16 A/B) or kind::f8f6f4 (E4M3 A/B),
// fp32 accumulator, A K-major, B K-major or MN-major.
__host__ __device__ constexpr uint32_t idesc(bool fp8, int M, int N, bool b_mn_major) {
  return (1u << 4)                                   // D format: f32
         | ((fp8 ? 0u : 1u) << 7)                    // A format: E4M3 = 0 / BF16 = 1
         | ((fp8 ? 0u : 1u) << 10)                   // B format
         | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
         | ((uint32_t)(N >> 3) << 17)                // N / 8
         | ((uint32_t)(M >> 4) << 24);               // M / 16
}

}  // namespace ptx
}  // namespace smla

namespace smla {
namespace ptx {

// Asynchronous 16-byte store into another CTA's shared memory that completes
// `16 bytes` of transaction count on that CTA's mbarrier (both addresses from
// map_to_rank).  No fence is needed on the sending side.
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, float a, float b, float c, float d,
                                            uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   remote_addr),
               "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Remote arrive without ordering of this thread's earlier memory accesses.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Remote arrive that orders this thread's earlier memory accesses before it
// (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster_release(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T (A read from tensor memory).
template <bool kFp8>
__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  if constexpr (kFp8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

#define SMLA_W16(i) "r"(r[i])
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      SMLA_W16(0), SMLA_W16(1), SMLA_W16(2), SMLA_W16(3), SMLA_W16(4), SMLA_W16(5), SMLA_W16(6), SMLA_W16(7),
      SMLA_W16(8), SMLA_W16(9), SMLA_W16(10), SMLA_W16(11), SMLA_W16(12), SMLA_W16(13), SMLA_W16(14),
      SMLA_W16(15)
      : "memory");
}
#undef SMLA_W16

}  // namespace ptx
}  // namespace smla

namespace smla {
namespace ptx {

#define SMLA_R16(i) "=r"(r[i])
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : SMLA_R16(0), SMLA_R16(1), SMLA_R16(2), SMLA_R16(3), SMLA_R16(4), SMLA_R16(5), SMLA_R16(6), SMLA_R16(7),
        SMLA_R16(8), SMLA_R16(9), SMLA_R16(10), SMLA_R16(11), SMLA_R16(12), SMLA_R16(13), SMLA_R16(14),
        SMLA_R16(15)
      : "r"(taddr)
      : "memory");
}
#undef SMLA_R16

// Packed pairs of fp32 (Blackwell f32x2 arithmetic).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

}  // namespace ptx
}  // namespace smla

namespace smla {
namespace ptx {

// TMA gather: four rows (r0..r3) of a 2-D tensor, columns [x, x + box width),
// into shared memory at dst as four consecutive box rows (swizzled as the
// tensor map says); completes its bytes on the mbarrier.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void* tmap, int x, int r0, int r1, int r2, int r3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}

// TMA tile load: the box at (x, y) of a 2-D tensor (box rows y .. y + box
// height - 1, swizzled as the tensor map says) into shared memory at dst;
// completes its bytes on the mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

}  // namespace ptx
}  // namespace smla

namespace smla {
namespace ptx {

// Asynchronous stores into another CTA's shared memory that complete their
// bytes on that CTA's mbarrier (addresses from map_to_rank).
__device__ __forceinline__ void st_async_v4u(uint32_t remote_addr, uint4 v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   remote_addr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
               : "memory");
}

__device__ __forceinline__ void st_async_b32(uint32_t remote_addr, uint32_t v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(remote_addr), "r"(v),
               "r"(remote_bar)
               : "memory");
}

#define SMLA_W32(i) "r"(r[i])
// 32 consecutive 32-bit TMEM columns of this thread's lane (warp-collective).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      SMLA_W32(0), SMLA_W32(1), SMLA_W32(2), SMLA_W32(3), SMLA_W32(4), SMLA_W32(5), SMLA_W32(6), SMLA_W32(7),
      SMLA_W32(8), SMLA_W32(9), SMLA_W32(10), SMLA_W32(11), SMLA_W32(12), SMLA_W32(13), SMLA_W32(14),
      SMLA_W32(15), SMLA_W32(16), SMLA_W32(17), SMLA_W32(18), SMLA_W32(19), SMLA_W32(20), SMLA_W32(21),
      SMLA_W32(22), SMLA_W32(23), SMLA_W32(24), SMLA_W32(25), SMLA_W32(26), SMLA_W32(27), SMLA_W32(28),
      SMLA_W32(29), SMLA_W32(30), SMLA_W32(31)
      : "memory");
}
#undef SMLA_W32

}  // namespace ptx
}  // namespace smla

namespace smla {
namespace ptx {

// Prefetch the 128-byte line holding addr into L1.
__device__ __forceinline__ void prefetch_l1(const void* addr) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(addr));
}

// Per-thread register limit of the executing warpgroup (all four warps run
// the same instruction): inc waits until the CTA's pool holds the registers.
template <uint32_t N>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// TMA tile load of a 3-D box at (x, y, z) into shared memory at dst (swizzled
// as the tensor map says); completes its bytes on the mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

}  // namespace ptx
}  // namespace smla

namespace smla {
namespace ptx {

// Shared-memory matrix descriptor without swizzle (K-major "interleaved"
// canonical layout: 8-row x 16-byte core matrices of 128 contiguous bytes;
// lbo = byte distance between core matrices adjacent along K, sbo = between
// 8-row groups), layout type 0 at bits 61-63.
__device__ __forceinline__ uint64_t desc_noswizzle(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory to
// another CTA's (destination and mbarrier addresses from map_to_rank); the
// bytes complete on that CTA's mbarrier.  Source and destination are read and
// written through the async proxy.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                                     uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(src_cta), "r"(bytes), "r"(bar_cluster)
      : "memory");
}

// 16-byte store to this CTA's shared memory.
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Prefetch the 128-byte line holding addr into L2.
__device__ __forceinline__ void prefetch_l2(const void* addr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(addr));
}

// Named barrier over `threads` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace ptx
}  // namespace smla
