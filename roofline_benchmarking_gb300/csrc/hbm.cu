// hbm.cu -- the HBM bandwidth kernels: STREAM Triad a[i] = b[i] + s*c[i] (the
// roofline's bandwidth ceiling) and the copy, read-only and write-only
// reference kernels beside it.
//
// TileOPs "Hardware Microbenchmarks" README, section "HBM Bandwidth" and
// "Methodology": Triad (2 reads + 1 write) is the calibration kernel, float4
// vectorised, swept over block sizes 128/256/512, on a working set far larger
// than L2; copy (1:1), read-only and write-only are reference measurements.
//
// GB300 layout: each block streams one fixed tile of consecutive float4
// (thread t takes float4 t, t + blockDim, ...) and the grid holds one block
// per tile, so consecutive blocks walk consecutive memory as the block
// scheduler issues them (launches are split beyond 2^31 - 1 blocks). Measured on GB300 this order sustains 91-98 % of the theoretical DRAM
// bandwidth, where a grid of resident blocks striding over the whole array
// reached about 83 %. Loads and stores carry streaming (evict-first) hints.
// a = fma(s, c, b): one rounding, which is also what a compiler emits for
// b + s*c by default.
#include <cuda_runtime.h>


#include "device_common.cuh"
#include "internal.h"

namespace kb {
namespace {

struct TriadOp {
  static constexpr int kReads = 2;
  static constexpr int kTileF4 = 1024;  // float4 per block
  float s;
  __device__ __forceinline__ float4 operator()(float4 b, float4 c) const {
    return make_float4(__fmaf_rn(s, c.x, b.x), __fmaf_rn(s, c.y, b.y), __fmaf_rn(s, c.z, b.z),
                       __fmaf_rn(s, c.w, b.w));
  }
  __device__ __forceinline__ float operator()(float b, float c) const { return __fmaf_rn(s, c, b); }
};

struct CopyOp {
  static constexpr int kReads = 1;
  static constexpr int kTileF4 = 2048;
  __device__ __forceinline__ float4 operator()(float4 b, float4) const { return b; }
  __device__ __forceinline__ float operator()(float b, float) const { return b; }
};

struct FillOp {
  static constexpr int kReads = 0;
  static constexpr int kTileF4 = 1024;
  float s;
  __device__ __forceinline__ float4 operator()(float4, float4) const { return make_float4(s, s, s, s); }
  __device__ __forceinline__ float operator()(float, float) const { return s; }
};

constexpr int kReadTileF4 = 4096;  // float4 per block of the read-only kernel
constexpr size_t kMaxGrid = 0x7fffffff;

// a[i] = op(b[i], c[i]) for the float4 of tile first_tile + blockIdx.x (Op::kTileF4
// consecutive float4, thread t taking t, t + BLOCK, ...); b and c are read only
// when the op reads them. A fixed tile per block keeps the block count (and the
// block scheduler's rate) independent of BLOCK, and at most 32 registers keep
// 2048 threads resident per SM.
template <int BLOCK, typename Op>
__global__ void __launch_bounds__(BLOCK, 2048 / BLOCK) stream_kernel(float* __restrict__ a,
                                                                     const float* __restrict__ b,
                                                                     const float* __restrict__ c, Op op, size_t n,
                                                                     size_t first_tile) {
  constexpr int E = Op::kTileF4 / BLOCK;
  const size_t n4 = n / 4;
  float4* a4 = reinterpret_cast<float4*>(a);
  const float4* b4 = reinterpret_cast<const float4*>(b);
  const float4* c4 = reinterpret_cast<const float4*>(c);
  const size_t tile = first_tile + blockIdx.x;
  const size_t i0 = tile * (size_t)Op::kTileF4 + threadIdx.x;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int UMAX = Op::kReads == 2 ? 2 : 4;  // float4 per stream in flight per thread
  constexpr int U = E < UMAX ? E : UMAX;
#pragma unroll 1
  for (int e0 = 0; e0 < E; e0 += U) {
    float4 bv[U], cv[U];
#pragma unroll
    for (int e = 0; e < U; ++e) {
      const size_t i = i0 + (size_t)(e0 + e) * BLOCK;
      bv[e] = (Op::kReads >= 1 && i < n4) ? __ldcs(b4 + i) : z;
      cv[e] = (Op::kReads >= 2 && i < n4) ? __ldcs(c4 + i) : z;
    }
#pragma unroll
    for (int e = 0; e < U; ++e) {
      const size_t i = i0 + (size_t)(e0 + e) * BLOCK;
      if (i < n4) __stcs(a4 + i, op(bv[e], cv[e]));
    }
  }
  // scalar tail (n not a multiple of 4)
  if (tile == 0 && threadIdx.x < (n & 3)) {
    const size_t t = n4 * 4 + threadIdx.x;
    a[t] = op(Op::kReads >= 1 ? b[t] : 0.f, Op::kReads >= 2 ? c[t] : 0.f);
  }
}

// Read-only: every float of b is loaded once and summed; one atomicAdd per
// block into *out (fp32 partial sums, so the result is exact for inputs whose
// partial sums are exactly representable).
template <int BLOCK>
__global__ void __launch_bounds__(BLOCK, 2048 / BLOCK) read_kernel(const float* __restrict__ b, size_t n,
                                                                   float* __restrict__ out, size_t first_tile) {
  constexpr int E = kReadTileF4 / BLOCK;
  constexpr int U = 4;
  __shared__ float red[32];
  const size_t n4 = n / 4;
  const float4* b4 = reinterpret_cast<const float4*>(b);
  const size_t tile = first_tile + blockIdx.x;
  const size_t i0 = tile * (size_t)kReadTileF4 + threadIdx.x;
  float t = 0.f;
#pragma unroll 1
  for (int e0 = 0; e0 < E; e0 += U) {
    float4 bv[U];
#pragma unroll
    for (int e = 0; e < U; ++e) {
      const size_t i = i0 + (size_t)(e0 + e) * BLOCK;
      bv[e] = i < n4 ? __ldcs(b4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int e = 0; e < U; ++e) t += (bv[e].x + bv[e].y) + (bv[e].z + bv[e].w);
  }
  if (tile == 0 && threadIdx.x < (n & 3)) t += b[n4 * 4 + threadIdx.x];
  t = block_sum(t, red);
  if (threadIdx.x == 0) atomicAdd(out, t);
}

// One block per tile of tile_f4 float4 (at least one block, for the tail),
// launched in chunks of at most 2^31 - 1 blocks.
template <typename Launch>
cudaError_t for_tiles(size_t n, size_t tile_f4, Launch launch) {
  size_t tiles = (n / 4 + tile_f4 - 1) / tile_f4;
  if (tiles < 1) tiles = 1;
  for (size_t first = 0; first < tiles; first += kMaxGrid) {
    const size_t g = tiles - first < kMaxGrid ? tiles - first : kMaxGrid;
    launch((unsigned)g, first);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int BLOCK, typename Op>
cudaError_t run_stream(float* a, const float* b, const float* c, Op op, size_t n, cudaStream_t st) {
  return for_tiles(n, Op::kTileF4, [&](unsigned grid, size_t first) {
    stream_kernel<BLOCK, Op><<<grid, BLOCK, 0, st>>>(a, b, c, op, n, first);
  });
}

template <typename Op>
cudaError_t dispatch_stream(float* a, const float* b, const float* c, Op op, size_t n, int block, cudaStream_t st) {
  switch (block) {
    case 128: return run_stream<128>(a, b, c, op, n, st);
    case 256: return run_stream<256>(a, b, c, op, n, st);
    case 512: return run_stream<512>(a, b, c, op, n, st);
    case 1024: return run_stream<1024>(a, b, c, op, n, st);
  }
  return cudaErrorInvalidValue;
}

template <int BLOCK>
cudaError_t run_read(const float* b, size_t n, float* out, cudaStream_t st) {
  return for_tiles(n, kReadTileF4, [&](unsigned grid, size_t first) {
    read_kernel<BLOCK><<<grid, BLOCK, 0, st>>>(b, n, out, first);
  });
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
  if (block != 128 && block != 256 && block != 512 && block != 1024) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  switch (block) {
    case 128: return run_read<128>(b, n, out, st);
    case 256: return run_read<256>(b, n, out, st);
    case 512: return run_read<512>(b, n, out, st);
    default: return run_read<1024>(b, n, out, st);
  }
}

}  // namespace kb
