// smla_decode_static_workspace: smla_decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// decode: an inference runtime's plugin "enqueue" callback that must not
// allocate, a process whose device memory is fully reserved by another
// allocator, or a plain C caller that links only this library and has no
// device allocator of its own.  This entry point serves them: the split-K
// scratch (partial outputs and their log-sum-exps) lives in one file-scope
// __device__ array of SMLA_STATIC_WORKSPACE_BYTES, which every GPU that loads
// the library holds until the process exits.  The entry point calls no
// allocator (no cudaMalloc, cudaFree or allocating library routine).
//
// Host code never hands the array's name to a kernel: on the host that name is
// a stand-in symbol, not a device address.  The runtime loads the module once
// per CUDA context, so the array has one device address per context.  The
// first call made in a context looks it up with cudaGetSymbolAddress (the
// caller's device and context being current), checks the result and caches
// it keyed by that context; later calls in the same context reuse it.
#include <cuda.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

__device__ __align__(256) unsigned char g_static_workspace[SMLA_STATIC_WORKSPACE_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

constexpr int kMaxContexts = 64;
struct CachedAddress {
  CUcontext ctx;
  void* ptr;
};
CachedAddress g_cache[kMaxContexts];
int g_cached = 0;
CtxGetCurrentFn g_ctx_get_current = nullptr;
std::mutex g_mutex;

// The device address of the static array in the current context.
cudaError_t static_workspace_address(void** out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_ctx_get_current == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
    // no context current yet: cudaGetSymbolAddress below makes the device's
    // primary context current, so read it again afterwards
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_workspace);
    if (e != cudaSuccess) return e;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  }
  for (int i = 0; i < g_cached; ++i)
    if (g_cache[i].ctx == ctx) {
      *out = g_cache[i].ptr;
      return cudaSuccess;
    }
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_workspace);
  if (e != cudaSuccess) return e;
  if (g_cached < kMaxContexts) g_cache[g_cached++] = CachedAddress{ctx, ptr};   // beyond that: looked up per call
  *out = ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" smla_status smla_decode_static_workspace(const smla_args* args, void* stream) {
  char msg[256];
  if (args == nullptr || args->sum_q == 0) return smla_decode(args, stream);  // NULL report / no-op
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
    return smla::record_error(SMLA_ERR_CUDA, msg);
  }
  size_t need = 0;
  smla_status st = smla_workspace_size(args, device, &need);
  if (st != SMLA_OK) return st;
  if (need > (size_t)SMLA_STATIC_WORKSPACE_BYTES) {
    snprintf(msg, sizeof(msg),
             "this call needs %zu bytes of split-K scratch but the static workspace holds %zu; "
             "lower num_splits / max_splits or use smla_decode with a caller workspace",
             need, (size_t)SMLA_STATIC_WORKSPACE_BYTES);
    return smla::record_error(SMLA_ERR_WORKSPACE_TOO_SMALL, msg);
  }
  void* ptr = nullptr;
  e = static_workspace_address(&ptr);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    return smla::record_error(SMLA_ERR_CUDA, msg);
  }
  smla_args a = *args;
  a.workspace = ptr;
  a.workspace_bytes = (size_t)SMLA_STATIC_WORKSPACE_BYTES;
  return smla_decode(&a, stream);
}
