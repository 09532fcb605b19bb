// kernels_noalloc.cu - attn_bwd_noalloc: the backward for callers that cannot allocate
// device memory themselves.
//
// Some callers of an attention backward have no way to allocate: a plugin that runs
// inside a host engine which owns all device memory and hands out no allocator or
// workspace, or a serving loop that bans cudaMalloc after start-up because it can
// synchronise the device and stall every other stream. For them this file keeps the
// backward's only scratch buffer (the per-row D values) in a fixed-size array of
// file-scope device memory, and passes its device address to the ordinary backward.
//
// The array is part of this library's device image: every GPU that loads the library
// reserves it until the process exits. Host code must not hand the array's name to a
// kernel (on the host it is only a stand-in for the symbol); its device address is looked
// up with cudaGetSymbolAddress, with the caller's context current, the first time a call
// runs in that context, and remembered per context: a module's device globals have one
// address per context, and a host engine may drive a device through a context of its own
// rather than the device's primary one.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "attn.h"

namespace {

// One float32 D value per query row of the whole batch: 16 MiB.
static __device__ __align__(256) float g_bwd_scratch[ATTN_NOALLOC_MAX_ROWS];

constexpr int kMaxContexts = 64;
std::mutex g_scratch_mu;
struct ScratchEntry {
  CUcontext ctx;
  float* addr;
};
ScratchEntry g_scratch[kMaxContexts] = {};
int g_scratch_n = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// The driver's cuCtxGetCurrent, through the runtime's entry-point query (the library
// does not link the driver library directly).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(p);
    return nullptr;
  }();
  return fn;
}

// Device address of g_bwd_scratch in the calling thread's current context. A thread with
// no current context gets its current device's primary context bound by the runtime's
// first call (cudaGetSymbolAddress), as any runtime call would.
cudaError_t scratch_in_current_context(float** out) {
  CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (ctx != nullptr)
    for (int i = 0; i < g_scratch_n; ++i)
      if (g_scratch[i].ctx == ctx) {
        *out = g_scratch[i].addr;
        return cudaSuccess;
      }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
  if (e != cudaSuccess) return e;
  if (ctx == nullptr && get(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  bool known = false;
  for (int i = 0; i < g_scratch_n && !known; ++i) known = g_scratch[i].ctx == ctx;
  if (!known && g_scratch_n < kMaxContexts) g_scratch[g_scratch_n++] = {ctx, static_cast<float*>(p)};
  *out = static_cast<float*>(p);
  return cudaSuccess;
}

}  // namespace

extern "C" attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                        const void* o, const float* lse, const void* dO,
                                        void* dq, void* dk, void* dv, int B, int H, int N,
                                        int d, attn_dtype dtype, int causal, float scale,
                                        void* cuda_stream) {
  if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if ((long long)B * H * N > (long long)ATTN_NOALLOC_MAX_ROWS) return ATTN_ERR_INVALID_ARG;
  float* scratch = nullptr;
  if (scratch_in_current_context(&scratch) != cudaSuccess) return ATTN_ERR_CUDA;
  // The backward's preprocess writes every D value it later reads, so the array's
  // previous contents never matter and nothing has to be cleared.
  return attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, scratch, B, H, N, d, dtype, causal, scale,
                  cuda_stream);
}
