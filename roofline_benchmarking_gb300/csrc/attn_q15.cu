// attn_q15.cu -- the Q15 fixed-point attention path (integer arithmetic only).
//
// kbench page ("kbench -- Transformer Attention Micro-benchmark Harness"),
// section "CPU reference + cache profiling": the board's fixed-point path has
// Q15 inputs, Q15.16 score accumulation and a 64-entry exp table; section
// "ARM Cortex-M4 firmware": one query row at a time, keys streamed like the
// flash kernel with an online-rescaled softmax, no hardware exp.
//
// The fixed-point rules (the pages print none; the plainest readings):
//   score   z = floor(floor(sum_c q_c k_c / 2^14) * C / 2^16), Q15.16 in
//           base-2 units, C = round(scale * log2(e) * 2^16); the product sum
//           is exact (64-bit).
//   exp     2^(-t) = T[f] >> n for t >= 0 (n = floor(t), f = top 6 fraction
//           bits), T[f] = round(2^15 * 2^(-f/64)); 0 once n >= 16.
//   stream  keys in tiles of 32 from key 0; per tile the tile maximum, a
//           rescale of l and acc by 2^(-(m_new - m)) (floor of the product /
//           2^15) when the running maximum rose, then p = 2^(-(m - z)),
//           l += p, acc_c += p * v_c.
//   output  acc_c / l rounded to nearest, halves away from zero, saturated.
// Every step is integer arithmetic, so the result is defined bit for bit.
//
// GPU layout: one block per 32 query rows of one head, 256 threads, 8 per
// row. Per 32-key tile the block stages K and V in shared memory; thread g of
// a row computes the scores of keys g, g+8, g+16, g+24, the row's 8 threads
// combine the tile maximum and the weight sum with shuffles, and each thread
// accumulates d/8 contiguous output channels in 64-bit registers. The tiles
// are the model's tiles, and the block's rows all use the same tile bounds, so
// the sequence of rescales is exactly the model's.
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"

namespace kb {
namespace {

constexpr int kRows = 32;     // query rows per block
constexpr int kTile = 32;     // keys per tile
constexpr int kThreads = 256; // 8 threads per query row
constexpr double kLog2e = 1.4426950408889634074;

struct Q15Params {
  long long C;              // scale * log2(e) in Q0.16
  unsigned short t[64];     // 2^(-f/64) in Q15
};

// 2^(-t) in Q15 for t >= 0 given in Q15.16.
__device__ __forceinline__ long long pow2_neg(long long t, const unsigned short* tab) {
  const long long n = t >> 16;
  if (n >= 16) return 0;
  return (long long)(tab[(t >> 10) & 63] >> n);
}

// a / b for b > 0, nearest, halves away from zero.
__device__ __forceinline__ long long round_div(long long a, long long b) {
  return a >= 0 ? (a + b / 2) / b : -((-a + b / 2) / b);
}

__device__ __forceinline__ int lo16(int w) { return (int)(short)(w & 0xffff); }
__device__ __forceinline__ int hi16(int w) { return w >> 16; }  // arithmetic shift keeps the sign

template <int D>
__global__ void __launch_bounds__(kThreads) q15_attn_kernel(const short* __restrict__ Q,
                                                           const short* __restrict__ K,
                                                           const short* __restrict__ V, short* __restrict__ O,
                                                           int S, int tiles_per_head, int causal,
                                                           const Q15Params prm) {
  constexpr int LD = D + 8;        // int16 per staged row: 16-byte pad, 8 rows of one load hit distinct banks
  constexpr int VPR = D / 8;       // 16-byte vectors per row
  constexpr int CH = D / 8;        // output channels per thread
  __shared__ __align__(16) short Qs[kRows][LD];
  __shared__ __align__(16) short Ks[kTile][LD];
  __shared__ __align__(16) short Vs[kTile][D];
  __shared__ int Ps[kRows][kTile + 1];
  __shared__ unsigned short tab[64];

  const int tid = threadIdx.x;
  const int r = tid >> 3, g = tid & 7;
  const long long n = blockIdx.x / tiles_per_head;
  const int i0 = (int)(blockIdx.x % tiles_per_head) * kRows;
  const int i = i0 + r;
  const short* Qh = Q + n * S * D;
  const short* Kh = K + n * S * D;
  const short* Vh = V + n * S * D;

  if (tid < 64) tab[tid] = prm.t[tid];
  for (int f = tid; f < kRows * VPR; f += kThreads) {
    const int rr = f / VPR, c8 = f % VPR;
    int4 x = make_int4(0, 0, 0, 0);
    if (i0 + rr < S) x = *reinterpret_cast<const int4*>(Qh + (long long)(i0 + rr) * D + 8 * c8);
    *reinterpret_cast<int4*>(&Qs[rr][8 * c8]) = x;
  }

  // rows past S (the ragged tail) run on zeros and are not stored
  const int my_last = causal ? min(i, S - 1) : S - 1;
  const int block_last = causal ? min(i0 + kRows - 1, S - 1) : S - 1;
  long long m = 0, l = 0, acc[CH];
  bool have_m = false;
#pragma unroll
  for (int c = 0; c < CH; ++c) acc[c] = 0;

  for (int t0 = 0; t0 <= block_last; t0 += kTile) {
    __syncthreads();  // the previous tile is no longer read
    for (int f = tid; f < kTile * VPR; f += kThreads) {
      const int rr = f / VPR, c8 = f % VPR;
      int4 kx = make_int4(0, 0, 0, 0), vx = kx;
      if (t0 + rr < S) {
        kx = *reinterpret_cast<const int4*>(Kh + (long long)(t0 + rr) * D + 8 * c8);
        vx = *reinterpret_cast<const int4*>(Vh + (long long)(t0 + rr) * D + 8 * c8);
      }
      *reinterpret_cast<int4*>(&Ks[rr][8 * c8]) = kx;
      *reinterpret_cast<int4*>(&Vs[rr][8 * c8]) = vx;
    }
    __syncthreads();

    // scores of keys g, g+8, g+16, g+24 of the tile
    long long z[4];
    bool ok[4];
    long long mt = 0;
    bool any = false;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int kk = g + 8 * u;
      long long dot = 0;
#pragma unroll
      for (int c8 = 0; c8 < VPR; ++c8) {
        const int4 a = *reinterpret_cast<const int4*>(&Qs[r][8 * c8]);
        const int4 b = *reinterpret_cast<const int4*>(&Ks[kk][8 * c8]);
        dot += (long long)(lo16(a.x) * lo16(b.x)) + (long long)(hi16(a.x) * hi16(b.x));
        dot += (long long)(lo16(a.y) * lo16(b.y)) + (long long)(hi16(a.y) * hi16(b.y));
        dot += (long long)(lo16(a.z) * lo16(b.z)) + (long long)(hi16(a.z) * hi16(b.z));
        dot += (long long)(lo16(a.w) * lo16(b.w)) + (long long)(hi16(a.w) * hi16(b.w));
      }
      z[u] = ((dot >> 14) * prm.C) >> 16;  // arithmetic shifts: floor
      ok[u] = t0 + kk <= my_last;
      if (ok[u] && (!any || z[u] > mt)) mt = z[u];
      any = any || ok[u];
    }
    // tile maximum over the row's 8 threads (lanes 8r' .. 8r'+7 of the warp)
#pragma unroll
    for (int s = 1; s < 8; s <<= 1) {
      const long long om = __shfl_xor_sync(0xffffffffu, mt, s);
      const int oa = __shfl_xor_sync(0xffffffffu, (int)any, s);
      if (oa && (!any || om > mt)) mt = om;
      any = any || oa;
    }
    if (any) {
      if (!have_m) {
        m = mt;
        have_m = true;
      } else if (mt > m) {
        const long long a = pow2_neg(mt - m, tab);
        l = (l * a) >> 15;
#pragma unroll
        for (int c = 0; c < CH; ++c) acc[c] = (acc[c] * a) >> 15;
        m = mt;
      }
    }
    long long psum = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long p = (any && ok[u]) ? pow2_neg(m - z[u], tab) : 0;
      Ps[r][g + 8 * u] = (int)p;
      psum += p;
    }
#pragma unroll
    for (int s = 1; s < 8; s <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, s);
    l += psum;
    __syncwarp();  // the row's weights are written by, and read by, this warp only

    // acc_c += p_j * v_jc over the tile; this thread owns channels g*CH .. g*CH+CH-1
#pragma unroll 4
    for (int kk = 0; kk < kTile; ++kk) {
      const int p = Ps[r][kk];
      const short* vrow = &Vs[kk][g * CH];
#pragma unroll
      for (int c2 = 0; c2 < CH; c2 += 2) {
        const int w = *reinterpret_cast<const int*>(vrow + c2);
        acc[c2] += (long long)(p * lo16(w));
        acc[c2 + 1] += (long long)(p * hi16(w));
      }
    }
  }

  if (i < S) {
    __align__(8) short out[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      long long x = round_div(acc[c], l);
      x = x > 32767 ? 32767 : (x < -32768 ? -32768 : x);
      out[c] = (short)x;
    }
    short* dst = O + (n * S + i) * D + g * CH;
#pragma unroll
    for (int c = 0; c < CH; c += 4)
      *reinterpret_cast<int2*>(dst + c) = *reinterpret_cast<const int2*>(out + c);
  }
}

template <int D>
cudaError_t q15_launch(const AttnProblem& p, const Q15Params& prm, cudaStream_t st) {
  const int tiles = (p.S + kRows - 1) / kRows;
  q15_attn_kernel<D><<<(unsigned)(p.N * tiles), kThreads, 0, st>>>(
      static_cast<const short*>(p.q), static_cast<const short*>(p.k), static_cast<const short*>(p.v),
      static_cast<short*>(p.o), p.S, tiles, p.causal, prm);
  return cudaGetLastError();
}

}  // namespace

bool q15_scale_ok(float scale) {
  const double cd = (double)scale * kLog2e * 65536.0;
  return cd <= 1073741824.0;
}

int q15_exp_table(unsigned short* out) {
  for (int f = 0; f < 64; ++f) out[f] = (unsigned short)std::llround(32768.0 * std::exp2(-(double)f / 64.0));
  return KB_OK;
}

cudaError_t launch_q15(const AttnProblem& p, cudaStream_t st) {
  Q15Params prm;
  prm.C = std::llround((double)p.scale * kLog2e * 65536.0);
  q15_exp_table(prm.t);
  switch (p.d) {
    case 32: return q15_launch<32>(p, prm, st);
    case 64: return q15_launch<64>(p, prm, st);
    case 128: return q15_launch<128>(p, prm, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kb
