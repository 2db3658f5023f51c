// triad.cu -- STREAM Triad a[i] = b[i] + s*c[i], the HBM bandwidth ceiling.
//
// TileOPs "Hardware Microbenchmarks" README, section "HBM Bandwidth" and
// "Methodology": Triad (2 reads + 1 write) is the calibration kernel, float4
// vectorised, swept over block sizes 128/256/512, on a working set far larger
// than L2.
//
// GB300 layout: a grid-stride loop over float4 with four independent float4
// loads of b and of c in flight per thread before their stores, streaming
// (evict-first) cache hints on loads and stores (nothing is reused), and a grid
// of resident blocks sized to the SM count. a = fma(s, c, b): one rounding,
// which is also what a compiler emits for b + s*c by default.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace kb {
namespace {

constexpr int kUnroll = 4;

template <int BLOCK>
__global__ void __launch_bounds__(BLOCK) triad_kernel(float* __restrict__ a, const float* __restrict__ b,
                                                      const float* __restrict__ c, float s, size_t n) {
  const size_t n4 = n / 4;
  float4* a4 = reinterpret_cast<float4*>(a);
  const float4* b4 = reinterpret_cast<const float4*>(b);
  const float4* c4 = reinterpret_cast<const float4*>(c);
  const size_t stride = (size_t)gridDim.x * BLOCK;
  size_t i = (size_t)blockIdx.x * BLOCK + threadIdx.x;
  // main body: kUnroll float4 per thread per trip, all loads issued first
  for (; i + (kUnroll - 1) * stride < n4; i += kUnroll * stride) {
    float4 bv[kUnroll], cv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      bv[u] = __ldcs(b4 + i + u * stride);
      cv[u] = __ldcs(c4 + i + u * stride);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float4 r;
      r.x = __fmaf_rn(s, cv[u].x, bv[u].x);
      r.y = __fmaf_rn(s, cv[u].y, bv[u].y);
      r.z = __fmaf_rn(s, cv[u].z, bv[u].z);
      r.w = __fmaf_rn(s, cv[u].w, bv[u].w);
      __stcs(a4 + i + u * stride, r);
    }
  }
  for (; i < n4; i += stride) {
    const float4 bv = __ldcs(b4 + i), cv = __ldcs(c4 + i);
    float4 r;
    r.x = __fmaf_rn(s, cv.x, bv.x);
    r.y = __fmaf_rn(s, cv.y, bv.y);
    r.z = __fmaf_rn(s, cv.z, bv.z);
    r.w = __fmaf_rn(s, cv.w, bv.w);
    __stcs(a4 + i, r);
  }
  // scalar tail (n not a multiple of 4)
  if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
    const size_t t = n4 * 4 + threadIdx.x;
    a[t] = __fmaf_rn(s, c[t], b[t]);
  }
}

struct GridCache {
  std::mutex mu;
  int device = -1;
  int blocks[3] = {0, 0, 0};  // resident blocks per SM for 128, 256, 512 threads
  int sms = 0;
};
GridCache g_grid;

template <int BLOCK>
cudaError_t run(float* a, const float* b, const float* c, float s, size_t n, int per_sm, int sms,
                cudaStream_t st) {
  const size_t n4 = n / 4;
  size_t want = (n4 + (size_t)BLOCK * kUnroll - 1) / ((size_t)BLOCK * kUnroll);
  size_t cap = (size_t)per_sm * (size_t)sms;
  size_t grid = want < cap ? want : cap;
  if (grid < 1) grid = 1;
  triad_kernel<BLOCK><<<(unsigned)grid, BLOCK, 0, st>>>(a, b, c, s, n);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_triad(float* a, const float* b, const float* c, float s, size_t n, int block,
                         cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int per_sm[3], sms;
  {
    std::lock_guard<std::mutex> lk(g_grid.mu);
    if (g_grid.device != dev) {
      if ((e = cudaDeviceGetAttribute(&g_grid.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
      if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_grid.blocks[0], triad_kernel<128>, 128, 0)) != cudaSuccess) return e;
      if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_grid.blocks[1], triad_kernel<256>, 256, 0)) != cudaSuccess) return e;
      if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_grid.blocks[2], triad_kernel<512>, 512, 0)) != cudaSuccess) return e;
      g_grid.device = dev;
    }
    for (int i = 0; i < 3; ++i) per_sm[i] = g_grid.blocks[i];
    sms = g_grid.sms;
  }
  switch (block) {
    case 128: return run<128>(a, b, c, s, n, per_sm[0], sms, st);
    case 256: return run<256>(a, b, c, s, n, per_sm[1], sms, st);
    case 512: return run<512>(a, b, c, s, n, per_sm[2], sms, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kb
