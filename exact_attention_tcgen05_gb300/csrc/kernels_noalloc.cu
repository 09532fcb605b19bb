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
// kernel (on the host it is only a stand-in for the symbol); the device address is
// looked up once per device with cudaGetSymbolAddress, with that device current.
#include <cuda_runtime.h>

#include <mutex>

#include "attn.h"

namespace {

// One float32 D value per query row of the whole batch: 16 MiB.
static __device__ __align__(256) float g_bwd_scratch[ATTN_NOALLOC_MAX_ROWS];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device (looked up on first use).
cudaError_t scratch_on_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
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
  if (scratch_on_current_device(&scratch) != cudaSuccess) return ATTN_ERR_CUDA;
  // The backward's preprocess writes every D value it later reads, so the array's
  // previous contents never matter and nothing has to be cleared.
  return attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, scratch, B, H, N, d, dtype, causal, scale,
                  cuda_stream);
}
