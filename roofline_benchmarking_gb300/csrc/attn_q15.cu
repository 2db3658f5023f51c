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
// GPU layout: one block per ROWS query rows of one head (32 rows; 16 under
// the causal mask, where short blocks balance the triangle), 8 threads per
// row. Per 32-key tile the block stages K (split into low and high bytes) and
// V (split and transposed to channel-major) in shared memory; thread g of a
// row computes the scores of keys g, g+8, g+16, g+24 with dp2a, the row's 8
// threads combine the tile maximum and the weight sum with shuffles, and each
// thread accumulates channels g, g+8, ... in 64-bit registers. The tiles
// are the model's tiles, and the block's rows all use the same tile bounds, so
// the sequence of rescales is exactly the model's.
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"

namespace kb {
namespace {

constexpr int kTile = 32;     // keys per tile
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

// Two-way 16-bit x 8-bit dot products (dp2a): d = c + a.h0 * b.byte(2s) + a.h1 * b.byte(2s+1),
// s = 0 (.lo) or 1 (.hi); the first type names a's halves, the second b's bytes.
__device__ __forceinline__ int dp2a_lo_su(int a, unsigned b, int c) {
  int d;
  asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi_su(int a, unsigned b, int c) {
  int d;
  asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_lo_ss(int a, unsigned b, int c) {
  int d;
  asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi_ss(int a, unsigned b, int c) {
  int d;
  asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ unsigned dp2a_lo_uu(unsigned a, unsigned b, unsigned c) {
  unsigned d;
  asm("dp2a.lo.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ unsigned dp2a_hi_uu(unsigned a, unsigned b, unsigned c) {
  unsigned d;
  asm("dp2a.hi.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_lo_us(unsigned a, unsigned b, int c) {
  int d;
  asm("dp2a.lo.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi_us(unsigned a, unsigned b, int c) {
  int d;
  asm("dp2a.hi.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Four int16 values (packed as two words) split into their low bytes
// (unsigned, x & 255) and high bytes (signed, x >> 8): x = 256 * hi + lo.
__device__ __forceinline__ void split4(int2 x, unsigned& lo, unsigned& hi) {
  const int a = (int)(short)(x.x & 0xffff), b = x.x >> 16, c = (int)(short)(x.y & 0xffff), d = x.y >> 16;
  lo = (unsigned)(a & 255) | ((unsigned)(b & 255) << 8) | ((unsigned)(c & 255) << 16) | ((unsigned)(d & 255) << 24);
  hi = (unsigned)((a >> 8) & 255) | ((unsigned)((b >> 8) & 255) << 8) | ((unsigned)((c >> 8) & 255) << 16) |
       ((unsigned)((d >> 8) & 255) << 24);
}

// The integer products are formed with dp2a: a key k = 256 kh + kl splits into
// a signed high byte and an unsigned low byte, so q . k = 256 (q . kh) + q . kl
// with both partial sums exact in 32 bits (|q kh| <= 2^22, 0 <= ... q kl < 2^23,
// at most 128 terms); likewise each tile's sum over 32 keys of p v (p <= 2^15).
template <int D, int ROWS>
__global__ void __launch_bounds__(8 * ROWS) q15_attn_kernel(const short* __restrict__ Q,
                                                           const short* __restrict__ K,
                                                           const short* __restrict__ V, short* __restrict__ O,
                                                           int S, int tiles_per_head, int causal,
                                                           const Q15Params prm) {
  constexpr int QW = D / 2;       // words (int16 pairs) of a query row
  constexpr int KW = D / 4;       // words (byte quads) of a split key row
  constexpr int KLD = KW + 4;     // padded: the 8 rows read by one load phase fall in distinct banks
  constexpr int VLD = kTile / 4 + 4;  // words of a split value column (32 keys), padded likewise
  constexpr int CH = D / 8;       // output channels per thread: g, g + 8, ...
  constexpr int kThreads = 8 * ROWS;
  __shared__ __align__(16) int Qw[ROWS][QW];
  __shared__ __align__(16) unsigned Kl[kTile][KLD], Kh[kTile][KLD];
  __shared__ __align__(16) short Vs[kTile][D];
  __shared__ __align__(16) unsigned Vl[D][VLD], Vh[D][VLD];
  __shared__ __align__(16) unsigned Pw[ROWS][kTile / 2];
  __shared__ unsigned short tab[64];

  const int tid = threadIdx.x;
  const int r = tid >> 3, g = tid & 7;
  // heads interleaved, the last (causal: heaviest) row tiles first, so that the
  // lightest blocks fill the last wave
  const long long nheads = gridDim.x / tiles_per_head;
  const long long n = blockIdx.x % nheads;
  const int i0 = (tiles_per_head - 1 - (int)(blockIdx.x / nheads)) * ROWS;
  const int i = i0 + r;
  const short* Qh = Q + n * S * D;
  const short* Kg = K + n * S * D;
  const short* Vg = V + n * S * D;

  if (tid < 64) tab[tid] = prm.t[tid];
  for (int f = tid; f < ROWS * (D / 8); f += kThreads) {
    const int rr = f / (D / 8), c8 = f % (D / 8);
    int4 x = make_int4(0, 0, 0, 0);
    if (i0 + rr < S) x = *reinterpret_cast<const int4*>(Qh + (long long)(i0 + rr) * D + 8 * c8);
    *reinterpret_cast<int4*>(&Qw[rr][4 * c8]) = x;
  }

  const int my_last = causal ? min(i, S - 1) : S - 1;
  const int block_last = causal ? min(i0 + ROWS - 1, S - 1) : S - 1;
  long long m = 0, l = 0, acc[CH];
  bool have_m = false;
#pragma unroll
  for (int c = 0; c < CH; ++c) acc[c] = 0;

  for (int t0 = 0; t0 <= block_last; t0 += kTile) {
    __syncthreads();  // the previous tile is no longer read (and Qw is written)
    // K: split each quad of features into low and high bytes
    for (int f = tid; f < kTile * KW; f += kThreads) {
      const int j = f / KW, w = f % KW;
      int2 x = make_int2(0, 0);
      if (t0 + j < S) x = *reinterpret_cast<const int2*>(Kg + (long long)(t0 + j) * D + 4 * w);
      unsigned lo, hi;
      split4(x, lo, hi);
      Kl[j][w] = lo;
      Kh[j][w] = hi;
    }
    // V: staged as is (coalesced), then split and transposed below
    for (int f = tid; f < kTile * (D / 8); f += kThreads) {
      const int j = f / (D / 8), c8 = f % (D / 8);
      int4 x = make_int4(0, 0, 0, 0);
      if (t0 + j < S) x = *reinterpret_cast<const int4*>(Vg + (long long)(t0 + j) * D + 8 * c8);
      *reinterpret_cast<int4*>(&Vs[j][8 * c8]) = x;
    }
    __syncthreads();
    for (int f = tid; f < D * (kTile / 4); f += kThreads) {
      const int c = f / (kTile / 4), kq = f % (kTile / 4);
      const int2 x = make_int2((int)((unsigned)(unsigned short)Vs[4 * kq][c] |
                                     ((unsigned)(unsigned short)Vs[4 * kq + 1][c] << 16)),
                               (int)((unsigned)(unsigned short)Vs[4 * kq + 2][c] |
                                     ((unsigned)(unsigned short)Vs[4 * kq + 3][c] << 16)));
      unsigned lo, hi;
      split4(x, lo, hi);
      Vl[c][kq] = lo;
      Vh[c][kq] = hi;
    }

    // scores of keys g, g+8, g+16, g+24 of the tile
    long long z[4];
    bool ok[4];
    long long mt = 0;
    bool any = false;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int kk = g + 8 * u;
      int accl = 0, acch = 0;
#pragma unroll
      for (int w = 0; w < KW; w += 4) {
        const uint4 kl = *reinterpret_cast<const uint4*>(&Kl[kk][w]);
        const uint4 kh = *reinterpret_cast<const uint4*>(&Kh[kk][w]);
        const int4 qa = *reinterpret_cast<const int4*>(&Qw[r][2 * w]);
        const int4 qb = *reinterpret_cast<const int4*>(&Qw[r][2 * w + 4]);
        accl = dp2a_lo_su(qa.x, kl.x, accl); accl = dp2a_hi_su(qa.y, kl.x, accl);
        acch = dp2a_lo_ss(qa.x, kh.x, acch); acch = dp2a_hi_ss(qa.y, kh.x, acch);
        accl = dp2a_lo_su(qa.z, kl.y, accl); accl = dp2a_hi_su(qa.w, kl.y, accl);
        acch = dp2a_lo_ss(qa.z, kh.y, acch); acch = dp2a_hi_ss(qa.w, kh.y, acch);
        accl = dp2a_lo_su(qb.x, kl.z, accl); accl = dp2a_hi_su(qb.y, kl.z, accl);
        acch = dp2a_lo_ss(qb.x, kh.z, acch); acch = dp2a_hi_ss(qb.y, kh.z, acch);
        accl = dp2a_lo_su(qb.z, kl.w, accl); accl = dp2a_hi_su(qb.w, kl.w, accl);
        acch = dp2a_lo_ss(qb.z, kh.w, acch); acch = dp2a_hi_ss(qb.w, kh.w, acch);
      }
      const long long dot = (long long)acch * 256 + accl;  // the exact sum of the d products
      z[u] = ((dot >> 14) * prm.C) >> 16;                   // arithmetic shifts: floor
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
      const unsigned p = (any && ok[u]) ? (unsigned)pow2_neg(m - z[u], tab) : 0u;  // <= 2^15
      psum += p;
      // weights of keys 2m and 2m+1 share a word: even threads take their odd neighbour's
      const unsigned pn = __shfl_down_sync(0xffffffffu, p, 1);
      if ((g & 1) == 0) Pw[r][(g + 8 * u) >> 1] = p | (pn << 16);
    }
#pragma unroll
    for (int s = 1; s < 8; s <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, s);
    l += psum;
    __syncthreads();  // Vl / Vh complete; the row's weights written

    // acc_c += sum_j p_j v_jc over the tile for channels c = g + 8 i
    uint4 pw[kTile / 8];
#pragma unroll
    for (int q4 = 0; q4 < kTile / 8; ++q4) pw[q4] = *reinterpret_cast<const uint4*>(&Pw[r][4 * q4]);
#pragma unroll
    for (int ci = 0; ci < CH; ++ci) {
      const int c = g + 8 * ci;
      unsigned al = 0;
      int ah = 0;
#pragma unroll
      for (int q4 = 0; q4 < kTile / 16; ++q4) {
        const uint4 vl = *reinterpret_cast<const uint4*>(&Vl[c][4 * q4]);
        const uint4 vh = *reinterpret_cast<const uint4*>(&Vh[c][4 * q4]);
        const uint4 pa = pw[2 * q4], pb = pw[2 * q4 + 1];  // keys 16 q4 .. 16 q4 + 15 as 8 pairs
        al = dp2a_lo_uu(pa.x, vl.x, al); al = dp2a_hi_uu(pa.y, vl.x, al);
        ah = dp2a_lo_us(pa.x, vh.x, ah); ah = dp2a_hi_us(pa.y, vh.x, ah);
        al = dp2a_lo_uu(pa.z, vl.y, al); al = dp2a_hi_uu(pa.w, vl.y, al);
        ah = dp2a_lo_us(pa.z, vh.y, ah); ah = dp2a_hi_us(pa.w, vh.y, ah);
        al = dp2a_lo_uu(pb.x, vl.z, al); al = dp2a_hi_uu(pb.y, vl.z, al);
        ah = dp2a_lo_us(pb.x, vh.z, ah); ah = dp2a_hi_us(pb.y, vh.z, ah);
        al = dp2a_lo_uu(pb.z, vl.w, al); al = dp2a_hi_uu(pb.w, vl.w, al);
        ah = dp2a_lo_us(pb.z, vh.w, ah); ah = dp2a_hi_us(pb.w, vh.w, ah);
      }
      acc[ci] += (long long)ah * 256 + (long long)al;
    }
  }

  if (i < S) {
    short* dst = O + (n * S + i) * D;
#pragma unroll
    for (int ci = 0; ci < CH; ++ci) {
      long long x = round_div(acc[ci], l);
      x = x > 32767 ? 32767 : (x < -32768 ? -32768 : x);
      dst[g + 8 * ci] = (short)x;
    }
  }
}

template <int D, int ROWS>
cudaError_t q15_launch_rows(const AttnProblem& p, const Q15Params& prm, cudaStream_t st) {
  const int tiles = (p.S + ROWS - 1) / ROWS;
  q15_attn_kernel<D, ROWS><<<(unsigned)(p.N * tiles), 8 * ROWS, 0, st>>>(
      static_cast<const short*>(p.q), static_cast<const short*>(p.k), static_cast<const short*>(p.v),
      static_cast<short*>(p.o), p.S, tiles, p.causal, prm);
  return cudaGetLastError();
}

template <int D>
cudaError_t q15_launch(const AttnProblem& p, const Q15Params& prm, cudaStream_t st) {
  return p.causal ? q15_launch_rows<D, 16>(p, prm, st) : q15_launch_rows<D, 32>(p, prm, st);
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
