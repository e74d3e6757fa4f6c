// Device helpers shared by the tcgen05 decode kernels: bounded mbarrier waits
// (a wait that expires raises the CTA's abort flag and ORs
// SMLA_DEVERR_TIMEOUT into the error word), the 128-byte-swizzle offset of
// UMMA-canonical tiles, BF16 packing; and the host encoder of the KV pool
// tensor maps.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace smla {

constexpr uint64_t kTimeoutNs = 2000000000ull;   // every on-device wait gives up after 2 s

// [rows, 512] pool view for TMA: box 128 bytes x box_rows rows, 128-byte
// swizzle (decode_tcgen05.cu).
cudaError_t encode_pool_map(CUtensorMap* map, const void* base, int64_t rows, int64_t row_stride, int dtype,
                            int box_rows);

namespace tc {

using namespace ptx;

struct Ctx {
  int32_t* abort_flag;
  int32_t* err;
};

__device__ __forceinline__ bool wait_bar(const Ctx& cx, uint32_t bar, uint32_t parity, bool cluster_scope) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    bool done = cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    if (done) return true;
    if ((it & 3u) == 3u) {
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

// Wait for a barrier that completes once already-issued asynchronous work is
// done; bounded by the same timeout but not cut short by the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > kTimeoutNs) return;
}

// All lanes of the warp wait; the result is warp-uniform.
__device__ __forceinline__ bool warp_wait(const Ctx& cx, uint32_t bar, uint32_t parity, bool cluster_scope = false) {
  bool ok = wait_bar(cx, bar, parity, cluster_scope);
  return __all_sync(0xffffffffu, ok);
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

// ---------------------------------------------------------------- token pairs
// The union of two tokens' selected rows (the token-pair forms of the
// tcgen05 kernels).  Token A's rows go into an open-addressing hash in shared
// memory, keyed by (pool, row), each key with A's list index; token B's rows
// look themselves up.  A B row found in A claims A's entry (the sign bit of
// the index): a second claim means B selects a row A selects twice over, and
// a key already present when A inserts means A selects a row twice; either
// sets *dup, and the unit then shares nothing (a shared entry cannot count
// one token's row twice).  B rows that A does not select stay B's own
// entries, repeats included.  kHashSlots is a power of two larger than the
// keys, so probing always ends.
// (Out of line: the set-up code of a unit runs once, cold in the instruction
// cache, so its size is what it costs.)
constexpr uint32_t kPairEmpty = 0xffffffffu;

__device__ __forceinline__ uint32_t pair_key(int row, bool comp) {
  return (uint32_t)row | (comp ? 0x80000000u : 0u);
}

template <int kHashSlots>
__device__ __forceinline__ uint32_t pair_slot(uint32_t key) {
  static_assert((kHashSlots & (kHashSlots - 1)) == 0, "power of two");
  return (key * 2654435761u) >> (32 - __builtin_ctz(kHashSlots));
}

// token A's row (list index a): one slot per key
template <int kHashSlots>
__device__ __noinline__ void pair_insert_a(uint32_t* keys, int32_t* vals, int32_t* dup, uint32_t key, int a) {
  if (key == kPairEmpty) {                                    // would read as empty
    *dup = 1;
    return;
  }
  uint32_t h = pair_slot<kHashSlots>(key);
  for (int probe = 0; probe < kHashSlots; ++probe) {
    const uint32_t prev = atomicCAS(keys + h, kPairEmpty, key);
    if (prev == kPairEmpty) {
      vals[h] = a;
      return;
    }
    if (prev == key) {                                        // token A selects the row twice
      *dup = 1;
      return;
    }
    h = (h + 1) & (kHashSlots - 1);
  }
  *dup = 1;                                                   // not reached: more slots than keys
}

// token B's row: A's list index of the same row (claimed for B), or -1
template <int kHashSlots>
__device__ __noinline__ int pair_claim_a(const uint32_t* keys, int32_t* vals, int32_t* dup, uint32_t key) {
  uint32_t h = pair_slot<kHashSlots>(key);
  for (int probe = 0; probe < kHashSlots; ++probe) {
    const uint32_t k = keys[h];
    if (k == key) {
      const int32_t old = atomicOr(vals + h, (int32_t)0x80000000);
      if (old < 0) *dup = 1;                                  // B's second entry of a row A selects
      return old & 0x7fffffff;
    }
    if (k == kPairEmpty) return -1;
    h = (h + 1) & (kHashSlots - 1);
  }
  return -1;
}

}  // namespace tc
}  // namespace smla
