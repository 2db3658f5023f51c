// naive_noalloc.cu -- the naive three-pass fp32 attention with its score
// matrix in a fixed array owned by the library, for callers that cannot
// allocate device memory.
//
// Who cannot allocate: a caller whose device memory is entirely reserved by
// its own pool or arena (a cudaMalloc would fail, or would fragment memory the
// pool expects to own), and a caller on a latency-critical path that must not
// pay cudaMalloc's cost and its implicit device-wide synchronisation. Such a
// caller still owns q, k, v and o; only the N*S*S score workspace moves into
// `g_naive_noalloc_scores` below.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds KB_NAIVE_NOALLOC_MAX_BYTES of it until the process exits. In
// host code its name is only a host-side stand-in for the symbol, so the
// device address is obtained with cudaGetSymbolAddress, once per device, with
// that device current, on the first call made on that device.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "internal.h"

namespace kb {

static __device__ __align__(256) float g_naive_noalloc_scores[KB_NAIVE_NOALLOC_MAX_BYTES / sizeof(float)];

namespace {

struct ScratchAddress {
  std::mutex mu;
  std::vector<float*> ptr;  // per device ordinal, nullptr until set up
};
ScratchAddress g_scratch;

// Device address of the array on the current device (set up on first use).
int scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return KB_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_scratch.mu);
  if ((int)g_scratch.ptr.size() <= dev) g_scratch.ptr.resize(dev + 1, nullptr);
  if (!g_scratch.ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_naive_noalloc_scores);
    if (e != cudaSuccess) {
      set_last_cuda_error(e);
      return KB_ERR_CUDA;
    }
    g_scratch.ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch.ptr[dev];
  return KB_OK;
}

}  // namespace
}  // namespace kb

using namespace kb;

extern "C" int kb_attn_fwd_naive_noalloc(const void* q, const void* k, const void* v, void* o, int B, int H,
                                         int S, int d, int causal, float scale, void* stream) {
  int var = 0;
  int st = validate_attention(q, k, v, o, B, H, S, d, causal, scale, KB_F32, KB_NAIVE, &var);
  if (st != KB_OK) return st;
  const int64_t N = (int64_t)B * H;
  if (naive_workspace_bytes(N, S) > KB_NAIVE_NOALLOC_MAX_BYTES) return KB_ERR_NO_MEMORY;
  if ((st = check_current_device()) != KB_OK) return st;
  float* scores = nullptr;
  if ((st = scratch_address(&scores)) != KB_OK) return st;
  // Every entry the three passes read is written earlier in the same call, so
  // nothing left in the array by a previous call needs clearing.
  AttnProblem p{q, k, v, o, N, S, d, causal, scale, KB_F32};
  cudaError_t e = launch_naive_f32(p, scores, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return KB_ERR_CUDA;
  }
  return KB_OK;
}
