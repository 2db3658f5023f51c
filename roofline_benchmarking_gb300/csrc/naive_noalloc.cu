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
// library holds KB_NAIVE_NOALLOC_MAX_BYTES of it until the process exits. With
// CUDA's lazy module loading (the default) the module that holds it, and so the
// 32 MiB, is loaded on a device by the first call made there, inside
// cudaGetSymbolAddress: that first call is where the memory is committed. In
// host code the array's name is only a host-side stand-in for the symbol, so
// the device address is obtained with cudaGetSymbolAddress with the device
// current, and cached together with the identity of the CUDA context it
// belongs to. A device reset (or a primary context torn down and created
// again) reloads the module at a possibly different address; the cached
// address is then looked up again instead of being reused.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "internal.h"

namespace kb {

static __device__ __align__(256) float g_naive_noalloc_scores[KB_NAIVE_NOALLOC_MAX_BYTES / sizeof(float)];

namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The driver's id of the calling thread's current context (unique over the
// process's lifetime, unlike the context handle, which can be reused); false
// when there is none or the driver does not provide the query.
bool current_context_id(unsigned long long* id) {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    (void)cudaGetLastError();
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

struct ScratchEntry {
  float* ptr = nullptr;        // device address of the array, nullptr until looked up
  unsigned long long ctx = 0;  // id of the context the address belongs to
  bool ctx_known = false;      // false: no context id was available, look up on every call
};

struct ScratchAddress {
  std::mutex mu;
  std::vector<ScratchEntry> dev;  // per device ordinal
};
ScratchAddress g_scratch;

// Device address of the array in the current device's current context.
int scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return KB_ERR_NO_DEVICE;
  }
  unsigned long long ctx = 0;
  bool known = current_context_id(&ctx);
  std::lock_guard<std::mutex> lk(g_scratch.mu);
  if ((int)g_scratch.dev.size() <= dev) g_scratch.dev.resize(dev + 1);
  ScratchEntry& s = g_scratch.dev[dev];
  if (s.ptr && known && s.ctx_known && s.ctx == ctx) {
    *out = s.ptr;
    return KB_OK;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_naive_noalloc_scores);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return KB_ERR_CUDA;
  }
  // the lookup made the device's primary context current if none was
  if (!known) known = current_context_id(&ctx);
  s.ptr = static_cast<float*>(p);
  s.ctx = ctx;
  s.ctx_known = known;
  *out = s.ptr;
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
