// Tensor-core throughput of this GPU for the roofline's tensor term.
//
// One CTA per SM; two issuing warps per CTA, each with its own accumulator,
// issue back-to-back tcgen05.mma (cta_group::1, M = 128, N = 256, K = one
// 32-byte step) on operands resident in shared memory (128-byte swizzle,
// K-major), for kind::f8f6f4 (E4M3 x E4M3 -> fp32) and kind::f16 (BF16 x BF16
// -> fp32).  A single issuing thread with one dependent accumulator chain
// reaches only part of the rate (each instruction waits on the previous one),
// so two independent chains from two warps are used.  Timed with CUDA events:
// a burst of ~2 ms, and back-to-back launches for ~3 s (sustained, under the
// power cap).  Prints one JSON object.
//
// Build and run: nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o mma_peak mma_peak.cu && ./mma_peak
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>

#define CK(x)                                                                                   \
  do {                                                                                          \
    cudaError_t e_ = (x);                                                                       \
    if (e_ != cudaSuccess) {                                                                    \
      fprintf(stderr, "CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__); \
      exit(1);                                                                                  \
    }                                                                                           \
  } while (0)

namespace {

constexpr int kIssuers = 2;
constexpr int kM = 128, kN = 256;
constexpr int kSteps = 4;                 // K steps of 32 bytes inside one 128-byte swizzle row
constexpr uint64_t kTimeoutNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                 // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;       // 8-row groups 1024 bytes apart
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;                 // 128-byte swizzle
  return d;
}

__host__ __device__ constexpr uint32_t instr_desc(bool fp8) {
  return (1u << 4) | ((fp8 ? 0u : 1u) << 7) | ((fp8 ? 0u : 1u) << 10) | ((uint32_t)(kN >> 3) << 17) |
         ((uint32_t)(kM >> 4) << 24);
}

template <bool kFp8>
__global__ void __launch_bounds__(128, 1) mma_loop(int iters, int* err) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t done[kIssuers];
  __shared__ uint32_t tmem_base;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* b = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // A: 128 rows x 128 B, B: 256 rows x 128 B; finite, non-zero values
  for (int i = tid; i < (kM + kN) * 128 / 4; i += blockDim.x) {
    const uint32_t x = (uint32_t)i * 2654435761u ^ 0x9E3779B9u;
    reinterpret_cast<uint32_t*>(b)[i] = kFp8 ? (x & 0x37373737u) : (x & 0x3F7F3F7Fu);
  }
  if (tid == 0) {
    for (int i = 0; i < kIssuers; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&done[i])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;
  if (warp < kIssuers && lane == 0) {
    const uint32_t d = tmem + (uint32_t)(warp * kN);
    const uint32_t idesc = instr_desc(kFp8);
    for (int it = 0; it < iters; ++it) {
      for (int k = 0; k < kSteps; ++k) {
        const uint64_t a = desc_sw128(base + k * 32);
        const uint64_t bd = desc_sw128(base + kM * 128 + k * 32);
        const uint32_t acc = (it > 0 || k > 0) ? 1u : 0u;
        if (kFp8)
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
              "l"(a), "l"(bd), "r"(idesc), "r"(acc)
              : "memory");
        else
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
              "l"(a), "l"(bd), "r"(idesc), "r"(acc)
              : "memory");
      }
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(&done[warp]))
                 : "memory");
  }
  __syncwarp();
  if (lane == 0) {
    // every warp waits (bounded) for both issuers' MMAs before TMEM is freed
    for (int i = 0; i < kIssuers; ++i) {
      uint64_t start;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(start));
      for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(&done[i]))
            : "memory");
        if (ok) break;
        uint64_t now;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
        if (now - start > kTimeoutNs) {
          atomicOr(err, 1);
          break;
        }
      }
    }
  }
  __syncwarp();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
}

template <bool kFp8>
void measure(int sms, int* err, const char* name, bool last) {
  const int smem = (kM + kN) * 128 + 1024 + 120 * 1024;   // padding: one CTA per SM
  CK(cudaFuncSetAttribute(mma_loop<kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  const double flop_per_iter = 2.0 * kM * kN * (kFp8 ? 32 : 16) * kSteps * kIssuers;
  const int iters = (int)(2e-3 * (kFp8 ? 4.5e15 : 2.25e15) / sms / flop_per_iter);
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  mma_loop<kFp8><<<sms, 128, smem>>>(iters, err);
  CK(cudaGetLastError());
  CK(cudaDeviceSynchronize());
  float best = 1e30f;
  for (int r = 0; r < 10; ++r) {
    CK(cudaEventRecord(e0));
    mma_loop<kFp8><<<sms, 128, smem>>>(iters, err);
    CK(cudaEventRecord(e1));
    CK(cudaEventSynchronize(e1));
    float ms;
    CK(cudaEventElapsedTime(&ms, e0, e1));
    best = std::min(best, ms);
  }
  const double burst = flop_per_iter * iters * sms / (best * 1e-3) / 1e12;
  const int reps = std::max(1, (int)(3000.0 / best));
  CK(cudaEventRecord(e0));
  for (int r = 0; r < reps; ++r) mma_loop<kFp8><<<sms, 128, smem>>>(iters, err);
  CK(cudaEventRecord(e1));
  CK(cudaEventSynchronize(e1));
  float ms;
  CK(cudaEventElapsedTime(&ms, e0, e1));
  const double sustained = flop_per_iter * iters * sms * reps / (ms * 1e-3) / 1e12;
  printf("  \"%s_tflops\": %.1f, \"%s_tflops_sustained\": %.1f, \"%s_sustained_seconds\": %.2f%s\n", name, burst, name,
         sustained, name, ms * 1e-3, last ? "" : ",");
}

}  // namespace

int main() {
  int sms = 0, dev = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, dev));
  int* err = nullptr;
  CK(cudaMalloc(&err, sizeof(int)));
  CK(cudaMemset(err, 0, sizeof(int)));
  printf("{\n  \"gpu\": \"%s\", \"sms\": %d,\n  \"shape\": \"cta_group::1 M=%d N=%d, %d issuing warps with one accumulator each\",\n",
         prop.name, sms, kM, kN, kIssuers);
  measure<true>(sms, err, "e4m3", false);
  measure<false>(sms, err, "bf16", false);
  int h = 0;
  CK(cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost));
  printf("  \"timeouts\": %d\n}\n", h);
  return h != 0;
}
