// hbm.cu -- the HBM bandwidth kernels: STREAM Triad a[i] = b[i] + s*c[i] (the
// roofline's bandwidth ceiling) and the copy, read-only and write-only
// reference kernels beside it.
//
// TileOPs "Hardware Microbenchmarks" README, section "HBM Bandwidth" and
// "Methodology": Triad (2 reads + 1 write) is the calibration kernel, float4
// vectorised, swept over block sizes 128/256/512, on a working set far larger
// than L2; copy (1:1), read-only and write-only are reference measurements.
//
// GB300 layout: a grid-stride loop over float4 with four independent float4
// accesses per stream in flight per thread before their uses, streaming
// (evict-first) cache hints on loads and stores (nothing is reused), and a grid
// of resident blocks sized to the SM count. a = fma(s, c, b): one rounding,
// which is also what a compiler emits for b + s*c by default.
#include <cuda_runtime.h>

#include <mutex>

#include "device_common.cuh"
#include "internal.h"

namespace kb {
namespace {

constexpr int kUnroll = 4;

struct TriadOp {
  static constexpr int kReads = 2;
  float s;
  __device__ __forceinline__ float4 operator()(float4 b, float4 c) const {
    return make_float4(__fmaf_rn(s, c.x, b.x), __fmaf_rn(s, c.y, b.y), __fmaf_rn(s, c.z, b.z),
                       __fmaf_rn(s, c.w, b.w));
  }
  __device__ __forceinline__ float operator()(float b, float c) const { return __fmaf_rn(s, c, b); }
};

struct CopyOp {
  static constexpr int kReads = 1;
  __device__ __forceinline__ float4 operator()(float4 b, float4) const { return b; }
  __device__ __forceinline__ float operator()(float b, float) const { return b; }
};

struct FillOp {
  static constexpr int kReads = 0;
  float s;
  __device__ __forceinline__ float4 operator()(float4, float4) const { return make_float4(s, s, s, s); }
  __device__ __forceinline__ float operator()(float, float) const { return s; }
};

// a[i] = op(b[i], c[i]) over n floats; b and c are read only when the op reads them.
template <int BLOCK, typename Op>
__global__ void __launch_bounds__(BLOCK) stream_kernel(float* __restrict__ a, const float* __restrict__ b,
                                                       const float* __restrict__ c, Op op, size_t n) {
  const size_t n4 = n / 4;
  float4* a4 = reinterpret_cast<float4*>(a);
  const float4* b4 = reinterpret_cast<const float4*>(b);
  const float4* c4 = reinterpret_cast<const float4*>(c);
  const size_t stride = (size_t)gridDim.x * BLOCK;
  size_t i = (size_t)blockIdx.x * BLOCK + threadIdx.x;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  // main body: kUnroll float4 per thread per trip, all loads issued first
  for (; i + (kUnroll - 1) * stride < n4; i += kUnroll * stride) {
    float4 bv[kUnroll], cv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      bv[u] = Op::kReads >= 1 ? __ldcs(b4 + i + u * stride) : z;
      cv[u] = Op::kReads >= 2 ? __ldcs(c4 + i + u * stride) : z;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) __stcs(a4 + i + u * stride, op(bv[u], cv[u]));
  }
  for (; i < n4; i += stride) {
    const float4 bv = Op::kReads >= 1 ? __ldcs(b4 + i) : z;
    const float4 cv = Op::kReads >= 2 ? __ldcs(c4 + i) : z;
    __stcs(a4 + i, op(bv, cv));
  }
  // scalar tail (n not a multiple of 4)
  if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
    const size_t t = n4 * 4 + threadIdx.x;
    a[t] = op(Op::kReads >= 1 ? b[t] : 0.f, Op::kReads >= 2 ? c[t] : 0.f);
  }
}

// Read-only: every float of b is loaded once and summed; one atomicAdd per
// block into *out (fp32 partial sums, so the result is exact for inputs whose
// partial sums are exactly representable).
template <int BLOCK>
__global__ void __launch_bounds__(BLOCK) read_kernel(const float* __restrict__ b, size_t n, float* __restrict__ out) {
  __shared__ float red[32];
  const size_t n4 = n / 4;
  const float4* b4 = reinterpret_cast<const float4*>(b);
  const size_t stride = (size_t)gridDim.x * BLOCK;
  size_t i = (size_t)blockIdx.x * BLOCK + threadIdx.x;
  float acc[kUnroll] = {0.f, 0.f, 0.f, 0.f};
  for (; i + (kUnroll - 1) * stride < n4; i += kUnroll * stride) {
    float4 bv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) bv[u] = __ldcs(b4 + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc[u] += (bv[u].x + bv[u].y) + (bv[u].z + bv[u].w);
  }
  for (; i < n4; i += stride) {
    const float4 bv = __ldcs(b4 + i);
    acc[0] += (bv.x + bv.y) + (bv.z + bv.w);
  }
  float t = (acc[0] + acc[1]) + (acc[2] + acc[3]);
  if (blockIdx.x == 0 && threadIdx.x < (n & 3)) t += b[n4 * 4 + threadIdx.x];
  t = block_sum(t, red);
  if (threadIdx.x == 0) atomicAdd(out, t);
}

struct GridCache {
  std::mutex mu;
  int device = -1;
  int sms = 0;
};
GridCache g_grid;

cudaError_t sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_grid.mu);
  if (g_grid.device != dev) {
    if ((e = cudaDeviceGetAttribute(&g_grid.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    g_grid.device = dev;
  }
  *sms = g_grid.sms;
  return cudaSuccess;
}

// Blocks for n floats: enough for one trip of kUnroll float4 per thread, at
// most the blocks that are resident on all SMs at once.
template <typename K>
cudaError_t grid_for(K kernel, int block, size_t n, unsigned* grid) {
  int sms = 0, per_sm = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, 0)) != cudaSuccess) return e;
  const size_t want = (n / 4 + (size_t)block * kUnroll - 1) / ((size_t)block * kUnroll);
  const size_t cap = (size_t)per_sm * (size_t)sms;
  size_t g = want < cap ? want : cap;
  *grid = (unsigned)(g < 1 ? 1 : g);
  return cudaSuccess;
}

template <int BLOCK, typename Op>
cudaError_t run_stream(float* a, const float* b, const float* c, Op op, size_t n, cudaStream_t st) {
  unsigned grid = 0;
  cudaError_t e = grid_for(stream_kernel<BLOCK, Op>, BLOCK, n, &grid);
  if (e != cudaSuccess) return e;
  stream_kernel<BLOCK, Op><<<grid, BLOCK, 0, st>>>(a, b, c, op, n);
  return cudaGetLastError();
}

template <typename Op>
cudaError_t dispatch_stream(float* a, const float* b, const float* c, Op op, size_t n, int block, cudaStream_t st) {
  switch (block) {
    case 128: return run_stream<128>(a, b, c, op, n, st);
    case 256: return run_stream<256>(a, b, c, op, n, st);
    case 512: return run_stream<512>(a, b, c, op, n, st);
  }
  return cudaErrorInvalidValue;
}

template <int BLOCK>
cudaError_t run_read(const float* b, size_t n, float* out, cudaStream_t st) {
  unsigned grid = 0;
  cudaError_t e = grid_for(read_kernel<BLOCK>, BLOCK, n, &grid);
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(out, 0, sizeof(float), st)) != cudaSuccess) return e;
  read_kernel<BLOCK><<<grid, BLOCK, 0, st>>>(b, n, out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_triad(float* a, const float* b, const float* c, float s, size_t n, int block,
                         cudaStream_t st) {
  return dispatch_stream(a, b, c, TriadOp{s}, n, block, st);
}

cudaError_t launch_copy(float* a, const float* b, size_t n, int block, cudaStream_t st) {
  return dispatch_stream(a, b, b, CopyOp{}, n, block, st);
}

cudaError_t launch_fill(float* a, float s, size_t n, int block, cudaStream_t st) {
  return dispatch_stream(a, a, a, FillOp{s}, n, block, st);
}

cudaError_t launch_read(const float* b, size_t n, float* out, int block, cudaStream_t st) {
  switch (block) {
    case 128: return run_read<128>(b, n, out, st);
    case 256: return run_read<256>(b, n, out, st);
    case 512: return run_read<512>(b, n, out, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kb
