// api.cu -- the C ABI of libkbattn: argument validation, variant selection,
// launches on the caller's stream, CUDA-event timing and device properties.
//
// kbench page ("kbench -- Transformer Attention Micro-benchmark Harness"):
// "Architecture" (one problem definition behind run_attention(kernel, cfg)),
// "Implementation details" (events around the kernel only, configurable
// warm-up, per-iteration device times). The Triad timing follows the TileOPs
// "Hardware Microbenchmarks" README, section "Methodology".
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <limits>
#include <mutex>
#include <vector>

#include "internal.h"

namespace kb {

namespace {
thread_local int t_last_cuda_error = 0;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Longest sequence any kernel accepts: S + 256 (a tile's rows past S) stays in int.
constexpr int kMaxSeq = std::numeric_limits<int32_t>::max() - 256;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Validation shared by every attention entry point; no CUDA call is made, so a
// rejected request has no effect on any device.
int validate(const void* q, const void* k, const void* v, const void* o, int B, int H, int S, int d,
             int causal, float scale, int dtype, int variant, int* resolved) {
  if (!q || !k || !v || !o) return KB_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return KB_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S < 1 || d < 1) return KB_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return KB_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return KB_ERR_INVALID_ARG;
  if (dtype != KB_F32 && dtype != KB_BF16 && dtype != KB_F16 && dtype != KB_Q15) return KB_ERR_INVALID_ARG;
  if (variant < KB_AUTO || variant > KB_FIXEDPOINT) return KB_ERR_INVALID_ARG;
  // B*H*S*d elements, times 4 bytes, must fit in int64; B*H in int32.
  const int64_t N = (int64_t)B * H;
  if (N > std::numeric_limits<int32_t>::max()) return KB_ERR_INVALID_ARG;
  const int64_t lim = std::numeric_limits<int64_t>::max() / 4;
  if (N > lim / S || N * S > lim / d) return KB_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 128 && d != 256) return KB_ERR_UNSUPPORTED;
  // every kernel counts rows and tiles in 32 bits: S plus a tile's rows must fit
  if (S > kMaxSeq) return KB_ERR_UNSUPPORTED;
  int var = variant;
  if (var == KB_AUTO) var = dtype == KB_F32 ? KB_FLASH : (dtype == KB_Q15 ? KB_FIXEDPOINT : KB_TC);
  if ((dtype == KB_Q15) != (var == KB_FIXEDPOINT)) return KB_ERR_UNSUPPORTED;
  if (dtype == KB_F32 && var == KB_TC) return KB_ERR_UNSUPPORTED;
  if ((dtype == KB_BF16 || dtype == KB_F16) && var != KB_TC) return KB_ERR_UNSUPPORTED;
  if (d == 256 && var != KB_TC) return KB_ERR_UNSUPPORTED;  // d = 256: tensor-core path only
  // the tensor-core kernels index their work items (256-row pairs, 128-row tiles at d = 256) in 32 bits
  if (var == KB_TC && N * ceil_div(S, d == 256 ? 128 : 256) > std::numeric_limits<int32_t>::max())
    return KB_ERR_UNSUPPORTED;
  if (var == KB_FIXEDPOINT) {
    // keeps every fixed-point intermediate inside 64 bits
    if (S > 65536 || !q15_scale_ok(scale)) return KB_ERR_INVALID_ARG;
    if (N * ceil_div(S, 16) > std::numeric_limits<int32_t>::max()) return KB_ERR_UNSUPPORTED;  // 16-row blocks
  }
  // one block per query row (fused) or per 64-row tile (flash, naive)
  const int64_t grid_limit = std::numeric_limits<int32_t>::max();
  if (var == KB_FUSED && N * S > grid_limit) return KB_ERR_UNSUPPORTED;
  if ((var == KB_FLASH || var == KB_NAIVE) && N * ceil_div(S, 64) > grid_limit) return KB_ERR_UNSUPPORTED;
  if (var == KB_NAIVE && N > 65535) return KB_ERR_UNSUPPORTED;  // grid.z of the score pass
  if (var == KB_NAIVE && ceil_div(S, 64) > 65535) return KB_ERR_UNSUPPORTED;  // grid.y of the score pass
  // the naive score matrix, N*S*S fp32, must be addressable
  if (var == KB_NAIVE && N > lim / S / S) return KB_ERR_INVALID_ARG;
  *resolved = var;
  return KB_OK;
}

int cuda_fail(cudaError_t e) {
  set_last_cuda_error(e);
  return KB_ERR_CUDA;
}

// The current device must be an sm_103 part (this library carries sm_103a code only).
struct DeviceGate {
  std::mutex mu;
  std::vector<int> ok;  // per ordinal: 0 unknown, 1 usable, -1 not usable
};
DeviceGate g_gate;

int check_device() {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return KB_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_gate.mu);
  if ((int)g_gate.ok.size() <= dev) g_gate.ok.resize(dev + 1, 0);
  if (g_gate.ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return KB_ERR_NO_DEVICE;
    }
    g_gate.ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return g_gate.ok[dev] == 1 ? KB_OK : KB_ERR_NO_DEVICE;
}

// Per-device workspace of the naive variant, grown on demand.
struct Workspace {
  std::mutex mu;
  std::vector<void*> ptr;
  std::vector<size_t> bytes;
};
Workspace g_ws;

// The caller holds g_ws.mu, and keeps holding it until the kernels that use
// the returned buffer are enqueued: a concurrent call that replaces the buffer
// synchronises the device before freeing it, which covers only work already
// enqueued.
int cached_workspace_locked(size_t need, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((int)g_ws.ptr.size() <= dev) {
    g_ws.ptr.resize(dev + 1, nullptr);
    g_ws.bytes.resize(dev + 1, 0);
  }
  if (g_ws.bytes[dev] < need) {
    if (g_ws.ptr[dev]) {
      // in-flight work on any stream may still read the old buffer
      if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e);
      cudaFree(g_ws.ptr[dev]);
      g_ws.ptr[dev] = nullptr;
      g_ws.bytes[dev] = 0;
    }
    void* p = nullptr;
    if ((e = cudaMalloc(&p, need)) != cudaSuccess) {
      (void)cudaGetLastError();
      return KB_ERR_NO_MEMORY;
    }
    g_ws.ptr[dev] = p;
    g_ws.bytes[dev] = need;
  }
  *out = g_ws.ptr[dev];
  return KB_OK;
}

int run_attention(const void* q, const void* k, const void* v, void* o, int B, int H, int S, int d, int causal,
                  float scale, int dtype, int variant, void* stream, void* workspace, size_t ws_bytes,
                  bool caller_ws, float* lse = nullptr) {
  int var = 0;
  int st = validate(q, k, v, o, B, H, S, d, causal, scale, dtype, variant, &var);
  if (st != KB_OK) return st;
  AttnProblem p{q, k, v, o, (int64_t)B * H, S, d, causal, scale, dtype};
  p.lse = lse;
  float* scores = nullptr;
  std::unique_lock<std::mutex> ws_lock(g_ws.mu, std::defer_lock);  // held through the launch below
  if (var == KB_NAIVE) {
    const size_t need = naive_workspace_bytes(p.N, S);
    if (caller_ws) {
      if (!workspace || ws_bytes < need) return KB_ERR_NO_MEMORY;
      if (!aligned16(workspace)) return KB_ERR_INVALID_ARG;
      if ((st = check_device()) != KB_OK) return st;
      scores = static_cast<float*>(workspace);
    } else {
      if ((st = check_device()) != KB_OK) return st;
      void* w = nullptr;
      ws_lock.lock();
      if ((st = cached_workspace_locked(need, &w)) != KB_OK) return st;
      scores = static_cast<float*>(w);
    }
  } else if ((st = check_device()) != KB_OK) {
    return st;
  }
  if (var == KB_FLASH && flash_wants_split(p.N, S, causal)) {
    // split causal tiles need room for their partial states; without it (a caller's
    // workspace that is absent or too small) the kernel runs every tile whole
    const size_t need = flash_split_bytes(p.N, S, d);
    if (caller_ws) {
      if (workspace && ws_bytes >= need && aligned16(workspace)) p.work = static_cast<float*>(workspace);
    } else {
      void* w = nullptr;
      ws_lock.lock();
      if ((st = cached_workspace_locked(need, &w)) != KB_OK) return st;
      p.work = static_cast<float*>(w);
    }
  }
  if (var == KB_FUSED && (st = fused_f32_check(S, d)) != KB_OK) return st;
  if (var == KB_TC && (st = tc_check(S, d, dtype)) != KB_OK) return st;

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  switch (var) {
    case KB_NAIVE: e = launch_naive_f32(p, scores, cs); break;
    case KB_FUSED: e = launch_fused_f32(p, cs); break;
    case KB_FLASH: e = launch_flash_f32(p, cs); break;
    case KB_TC: e = launch_tc(p, cs); break;
    case KB_FIXEDPOINT: e = launch_q15(p, cs); break;
    default: return KB_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess ? KB_OK : cuda_fail(e);
}

// Records start[t] / stop[t] around each timed call; returns per-call times.
template <typename Call>
int time_calls(Call call, cudaStream_t cs, int warmup, int iters, float* ms) {
  for (int t = 0; t < warmup; ++t) {
    int st = call();
    if (st != KB_OK) return st;
  }
  std::vector<cudaEvent_t> ev(2 * (size_t)iters, nullptr);
  cudaError_t e = cudaSuccess;
  int st = KB_OK;
  for (auto& x : ev) {
    if ((e = cudaEventCreate(&x)) != cudaSuccess) break;
  }
  if (e == cudaSuccess) {
    for (int t = 0; t < iters && st == KB_OK && e == cudaSuccess; ++t) {
      e = cudaEventRecord(ev[2 * t], cs);
      if (e == cudaSuccess) st = call();
      if (e == cudaSuccess && st == KB_OK) e = cudaEventRecord(ev[2 * t + 1], cs);
    }
  }
  if (e == cudaSuccess && st == KB_OK && iters > 0) e = cudaEventSynchronize(ev[2 * iters - 1]);
  for (int t = 0; t < iters && e == cudaSuccess && st == KB_OK; ++t)
    e = cudaEventElapsedTime(&ms[t], ev[2 * t], ev[2 * t + 1]);
  for (auto& x : ev)
    if (x) cudaEventDestroy(x);
  if (st != KB_OK) return st;
  return e == cudaSuccess ? KB_OK : cuda_fail(e);
}

}  // namespace

void set_last_cuda_error(cudaError_t e) { t_last_cuda_error = (int)e; }

int validate_attention(const void* q, const void* k, const void* v, const void* o, int B, int H, int S, int d,
                       int causal, float scale, int dtype, int variant, int* resolved) {
  return validate(q, k, v, o, B, H, S, d, causal, scale, dtype, variant, resolved);
}

int check_current_device() { return check_device(); }

}  // namespace kb

using namespace kb;

extern "C" {

int kb_version(void) { return 101; }

int kb_binary_version(int* out) {
  if (!out) return KB_ERR_INVALID_ARG;
  int st = check_device();
  if (st != KB_OK) return st;
  cudaError_t e = tc_binary_version(out);
  return e == cudaSuccess ? KB_OK : cuda_fail(e);
}

int kb_q15_exp_table(unsigned short* out64) {
  if (!out64) return KB_ERR_INVALID_ARG;
  return kb::q15_exp_table(out64);
}

int kb_attn_work_lists(long long N, int S, int d, int causal, int grid, int* start, unsigned int* items, int cap,
                       int* count) {
  if (N <= 0 || S <= 0 || S > kMaxSeq || grid <= 0 || cap < 0 || !start || !items || !count)
    return KB_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 128 && d != 256) return KB_ERR_INVALID_ARG;
  return kb::tc_work_lists(N, S, d, causal != 0, grid, start, items, cap, count);
}

int kb_attn_fwd(const void* q, const void* k, const void* v, void* o, int B, int H, int S, int d, int causal,
                float scale, int dtype, int variant, void* stream) {
  return run_attention(q, k, v, o, B, H, S, d, causal, scale, dtype, variant, stream, nullptr, 0, false);
}

int kb_attn_fwd_lse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int S, int d,
                    int causal, float scale, int dtype, int variant, void* stream) {
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return KB_ERR_INVALID_ARG;
  int var = 0;
  int st = validate(q, k, v, o, B, H, S, d, causal, scale, dtype, variant, &var);
  if (st != KB_OK) return st;
  if (var != KB_TC && var != KB_FLASH) return KB_ERR_UNSUPPORTED;
  return run_attention(q, k, v, o, B, H, S, d, causal, scale, dtype, variant, stream, nullptr, 0, false, lse);
}

int kb_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, void* q_dev,
                     void* k_dev, void* v_dev, void* o_dev, int B, int H, int S, int d, int causal, float scale,
                     int dtype, int variant, void* stream) {
  if (!q_host || !k_host || !v_host || !o_host) return KB_ERR_INVALID_ARG;
  int var = 0;
  int st = validate(q_dev, k_dev, v_dev, o_dev, B, H, S, d, causal, scale, dtype, variant, &var);
  if (st != KB_OK) return st;
  if ((st = check_device()) != KB_OK) return st;
  const size_t bytes = (size_t)B * H * S * d * (dtype == KB_F32 ? 4u : 2u);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const void* src[3] = {q_host, k_host, v_host};
  void* dst[3] = {q_dev, k_dev, v_dev};
  for (int t = 0; t < 3; ++t) {
    cudaError_t e = cudaMemcpyAsync(dst[t], src[t], bytes, cudaMemcpyHostToDevice, cs);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  st = run_attention(q_dev, k_dev, v_dev, o_dev, B, H, S, d, causal, scale, dtype, variant, stream, nullptr, 0, false);
  if (st != KB_OK) return st;
  cudaError_t e = cudaMemcpyAsync(o_host, o_dev, bytes, cudaMemcpyDeviceToHost, cs);
  return e == cudaSuccess ? KB_OK : cuda_fail(e);
}

size_t kb_attn_workspace_bytes(int B, int H, int S, int d, int dtype, int variant) {
  int var = 0;
  const void* dummy = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  if (validate(dummy, dummy, dummy, dummy, B, H, S, d, 0, 1.0f, dtype, variant, &var) != KB_OK) return 0;
  if (var == KB_NAIVE) return naive_workspace_bytes((int64_t)B * H, S);
  if (var == KB_FLASH) return flash_split_bytes((int64_t)B * H, S, d);  // used by causal calls only
  return 0;
}

int kb_attn_fwd_ws(const void* q, const void* k, const void* v, void* o, int B, int H, int S, int d, int causal,
                   float scale, int dtype, int variant, void* stream, void* workspace, size_t ws_bytes) {
  return run_attention(q, k, v, o, B, H, S, d, causal, scale, dtype, variant, stream, workspace, ws_bytes, true);
}

int kb_attn_bench(const void* q, const void* k, const void* v, void* o, int B, int H, int S, int d, int causal,
                  float scale, int dtype, int variant, void* stream, void* workspace, size_t ws_bytes, int warmup,
                  int iters, float* ms_per_iter) {
  if (warmup < 0 || iters < 1 || !ms_per_iter) return KB_ERR_INVALID_ARG;
  int var = 0;
  int st = validate(q, k, v, o, B, H, S, d, causal, scale, dtype, variant, &var);
  if (st != KB_OK) return st;
  const bool use_ws = workspace != nullptr;
  auto call = [&]() {
    return run_attention(q, k, v, o, B, H, S, d, causal, scale, dtype, variant, stream, workspace, ws_bytes,
                         use_ws);
  };
  return time_calls(call, static_cast<cudaStream_t>(stream), warmup, iters, ms_per_iter);
}

int kb_attn_bench_graph(const void* q, const void* k, const void* v, void* o, int B, int H, int S, int d,
                        int causal, float scale, int dtype, int variant, void* stream, void* workspace,
                        size_t ws_bytes, int launches, int warmup, int iters, float* ms_per_graph) {
  if (launches < 1 || launches > 100000 || warmup < 0 || iters < 1 || !ms_per_graph) return KB_ERR_INVALID_ARG;
  int var = 0;
  int st = validate(q, k, v, o, B, H, S, d, causal, scale, dtype, variant, &var);
  if (st != KB_OK) return st;
  const bool use_ws = workspace != nullptr;
  // One plain call first: it checks the device and grows the cached workspace,
  // so nothing inside the capture allocates or synchronises.
  cudaStream_t user = static_cast<cudaStream_t>(stream);
  st = run_attention(q, k, v, o, B, H, S, d, causal, scale, dtype, variant, user, workspace, ws_bytes, use_ws);
  if (st != KB_OK) return st;
  cudaError_t e = cudaStreamSynchronize(user);
  if (e != cudaSuccess) return cuda_fail(e);
  // Capture on a private stream (the caller's may be the legacy stream, which
  // cannot be captured); the instantiated graph is then launched on `stream`.
  cudaStream_t cap = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  if ((e = cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking)) != cudaSuccess) return cuda_fail(e);
  e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) {
    for (int t = 0; t < launches && st == KB_OK; ++t)
      st = run_attention(q, k, v, o, B, H, S, d, causal, scale, dtype, variant, cap, workspace, ws_bytes, use_ws);
    cudaError_t e2 = cudaStreamEndCapture(cap, &graph);  // ends the capture even after a failed call
    if (st == KB_OK) e = e2;
  }
  if (st == KB_OK && e == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
  if (st == KB_OK && e == cudaSuccess) {
    auto call = [&]() {
      cudaError_t le = cudaGraphLaunch(exec, user);
      return le == cudaSuccess ? (int)KB_OK : cuda_fail(le);
    };
    st = time_calls(call, user, warmup, iters, ms_per_graph);
  }
  if (exec) cudaGraphExecDestroy(exec);
  if (graph) cudaGraphDestroy(graph);
  cudaStreamDestroy(cap);
  if (st != KB_OK) return st;
  return e == cudaSuccess ? KB_OK : cuda_fail(e);
}

int kb_triad(float* a, const float* b, const float* c, float s, size_t n, int block, void* stream) {
  if (n == 0) return KB_OK;
  if (!a || !b || !c) return KB_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(c)) return KB_ERR_INVALID_ARG;
  if (block == 0) block = 256;
  if (block != 128 && block != 256 && block != 512 && block != 1024) return KB_ERR_INVALID_ARG;
  int st = check_device();
  if (st != KB_OK) return st;
  cudaError_t e = launch_triad(a, b, c, s, n, block, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KB_OK : cuda_fail(e);
}

int kb_triad_bench(float* a, const float* b, const float* c, float s, size_t n, int block, void* stream, int warmup,
                   int iters, float* ms_per_iter) {
  if (warmup < 0 || iters < 1 || !ms_per_iter) return KB_ERR_INVALID_ARG;
  auto call = [&]() { return kb_triad(a, b, c, s, n, block, stream); };
  return time_calls(call, static_cast<cudaStream_t>(stream), warmup, iters, ms_per_iter);
}

namespace {
// Shared checks of the HBM kernels; 0 floats is a no-op (KB_OK, nothing launched).
int hbm_args(const void* a, const void* b, const void* c, size_t n, int* block) {
  if (!a || !b || !c) return KB_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(c)) return KB_ERR_INVALID_ARG;
  if (*block == 0) *block = 256;
  if (*block != 128 && *block != 256 && *block != 512 && *block != 1024) return KB_ERR_INVALID_ARG;
  return check_device();
}
}  // namespace

int kb_hbm_copy(float* a, const float* b, size_t n, int block, void* stream) {
  if (n == 0) return KB_OK;
  int st = hbm_args(a, b, b, n, &block);
  if (st != KB_OK) return st;
  cudaError_t e = launch_copy(a, b, n, block, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KB_OK : cuda_fail(e);
}

int kb_hbm_write(float* a, float s, size_t n, int block, void* stream) {
  if (n == 0) return KB_OK;
  int st = hbm_args(a, a, a, n, &block);
  if (st != KB_OK) return st;
  cudaError_t e = launch_fill(a, s, n, block, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KB_OK : cuda_fail(e);
}

int kb_hbm_read(const float* b, size_t n, int block, float* out, void* stream) {
  if (!out || (reinterpret_cast<uintptr_t>(out) & 3u)) return KB_ERR_INVALID_ARG;
  int st = n == 0 ? check_device() : hbm_args(b, b, b, n, &block);
  if (st != KB_OK) return st;
  cudaError_t e = n == 0 ? cudaMemsetAsync(out, 0, sizeof(float), static_cast<cudaStream_t>(stream))
                         : launch_read(b, n, out, block, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KB_OK : cuda_fail(e);
}

int kb_hbm_bench(int op, float* a, const float* b, const float* c, float s, size_t n, int block, float* out,
                 void* stream, int warmup, int iters, float* ms_per_iter) {
  if (warmup < 0 || iters < 1 || !ms_per_iter) return KB_ERR_INVALID_ARG;
  if (op < KB_HBM_TRIAD || op > KB_HBM_WRITE) return KB_ERR_INVALID_ARG;
  auto call = [&]() {
    switch (op) {
      case KB_HBM_TRIAD: return kb_triad(a, b, c, s, n, block, stream);
      case KB_HBM_COPY: return kb_hbm_copy(a, b, n, block, stream);
      case KB_HBM_READ: return kb_hbm_read(b, n, block, out, stream);
      default: return kb_hbm_write(a, s, n, block, stream);
    }
  };
  return time_calls(call, static_cast<cudaStream_t>(stream), warmup, iters, ms_per_iter);
}

int kb_device_info(int device, kb_device_info_t* out) {
  if (!out || device < 0) return KB_ERR_INVALID_ARG;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || device >= count) {
    (void)cudaGetLastError();
    return KB_ERR_NO_DEVICE;
  }
  std::memset(out, 0, sizeof(*out));
  out->device = device;
  struct {
    cudaDeviceAttr a;
    int* dst;
  } attrs[] = {
      {cudaDevAttrComputeCapabilityMajor, &out->cc_major},
      {cudaDevAttrComputeCapabilityMinor, &out->cc_minor},
      {cudaDevAttrMultiProcessorCount, &out->sm_count},
      {cudaDevAttrClockRate, &out->sm_clock_khz},
      {cudaDevAttrMemoryClockRate, &out->mem_clock_khz},
      {cudaDevAttrGlobalMemoryBusWidth, &out->mem_bus_width_bits},
      {cudaDevAttrL2CacheSize, &out->l2_bytes},
      {cudaDevAttrMaxSharedMemoryPerBlockOptin, &out->smem_per_block_optin},
      {cudaDevAttrMaxSharedMemoryPerMultiprocessor, &out->smem_per_sm},
  };
  for (auto& x : attrs) {
    cudaError_t e = cudaDeviceGetAttribute(x.dst, x.a, device);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) return cuda_fail(e);
  out->total_mem_bytes = prop.totalGlobalMem;
  std::strncpy(out->name, prop.name, sizeof(out->name) - 1);
  return KB_OK;
}

int kb_check_device_error(void* stream) {
  unsigned int word = 0;
  int st = check_device();
  if (st != KB_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  e = read_and_clear_error_word(&word, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return word ? KB_ERR_TIMEOUT : KB_OK;
}

int kb_selftest_timeout(unsigned long long limit_ns, void* stream) {
  int st = check_device();
  if (st != KB_OK) return st;
  if (limit_ns < 1000ull) limit_ns = 1000ull;
  if (limit_ns > 2000000000ull) limit_ns = 2000000000ull;
  cudaError_t e = launch_selftest_timeout(limit_ns, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KB_OK : cuda_fail(e);
}

const char* kb_status_string(int status) {
  switch (status) {
    case KB_OK: return "KB_OK";
    case KB_ERR_INVALID_ARG: return "KB_ERR_INVALID_ARG";
    case KB_ERR_UNSUPPORTED: return "KB_ERR_UNSUPPORTED";
    case KB_ERR_CUDA: return "KB_ERR_CUDA";
    case KB_ERR_NO_MEMORY: return "KB_ERR_NO_MEMORY";
    case KB_ERR_TIMEOUT: return "KB_ERR_TIMEOUT";
    case KB_ERR_NO_DEVICE: return "KB_ERR_NO_DEVICE";
  }
  return "KB_UNKNOWN_STATUS";
}

int kb_last_cuda_error(void) { return t_last_cuda_error; }

}  // extern "C"
