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
// GPU layout: one block per ROWS = 16 query rows of one head (short blocks
// balance the causal triangle; 32-row blocks measured no faster without the
// mask), 8 threads per row. Per 32-key tile the block stages K (split into low and high bytes) and
// V (split and transposed to channel-major) in shared memory, one tile ahead in
// three rotating buffers, with one barrier per tile; thread g of a row keeps
// the row's query in registers, computes the scores of keys g, g+8, g+16, g+24
// with dp2a, the row's 8 threads combine the tile maximum and the weight sum
// with shuffles, and each thread accumulates channels g, g+8, ... in 64-bit
// registers. The tiles are the model's tiles, and the block's rows all use the
// same tile bounds, so the sequence of rescales is exactly the model's.
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

// Four int16 values (packed little-endian as two words) split into their low
// bytes (unsigned, x & 255) and high bytes (signed, x >> 8): x = 256 * hi + lo.
// Bytes 0, 2 of x.x and of x.y are the low bytes, 1, 3 the high ones: one byte
// permute each.
__device__ __forceinline__ void split4(int2 x, unsigned& lo, unsigned& hi) {
  lo = __byte_perm((unsigned)x.x, (unsigned)x.y, 0x6420);
  hi = __byte_perm((unsigned)x.x, (unsigned)x.y, 0x7531);
}

// The integer products are formed with dp2a: a key k = 256 kh + kl splits into
// a signed high byte and an unsigned low byte, so q . k = 256 (q . kh) + q . kl
// with both partial sums exact in 32 bits (|q kh| <= 2^22, 0 <= ... q kl < 2^23,
// at most 128 terms); likewise each tile's sum over 32 keys of p v (p <= 2^15).
//
// Per block: three staging buffers for the model's 32-key tiles (K split into
// low and high bytes, key-major; V split and channel-major, read straight from
// global memory in that order), two buffers of packed weights, one barrier per
// tile. Iteration t issues the global loads of tile t + 1 into registers, scores
// tile t, then stores tile t + 1 into buffer (t + 1) % 3; the barrier publishes
// tile t's weights and tile t + 1's staging; P V of tile t follows. A buffer is
// restaged only after the barrier that follows its last use two iterations
// earlier. Each thread keeps its row's query words in registers.
template <int D, int ROWS>
struct Q15Smem {
  static constexpr int KW = D / 4;            // words (byte quads) of a split key row
  static constexpr int KLD = KW + 4;          // padded: the 8 rows read by one load phase fall in distinct banks
  static constexpr int VLD = kTile / 4 + 4;   // words of a split value column (32 keys), padded likewise
  static constexpr int KBUF = kTile * KLD;    // one K half (low or high bytes) of a buffer
  static constexpr int VBUF = D * VLD;        // one V half of a buffer
  static constexpr int PBUF = ROWS * (kTile / 2);
  static constexpr int WORDS = 3 * (2 * KBUF + 2 * VBUF) + 2 * PBUF + 32;  // + the exp table (64 x 16 bits)
  static constexpr size_t BYTES = sizeof(unsigned) * (size_t)WORDS;
};

template <int D, int ROWS>
__global__ void __launch_bounds__(8 * ROWS) q15_attn_kernel(const short* __restrict__ Q,
                                                           const short* __restrict__ K,
                                                           const short* __restrict__ V, short* __restrict__ O,
                                                           int S, int tiles_per_head, int causal,
                                                           const Q15Params prm) {
  using L = Q15Smem<D, ROWS>;
  constexpr int QW = D / 2;       // words (int16 pairs) of a query row
  constexpr int KW = L::KW;
  constexpr int KLD = L::KLD;
  constexpr int VLD = L::VLD;
  constexpr int CH = D / 8;       // output channels per thread: g, g + 8, ...
  constexpr int kThreads = 8 * ROWS;
  extern __shared__ uint4 q15_smem[];
  unsigned* sm = reinterpret_cast<unsigned*>(q15_smem);
  unsigned* Kl = sm;                          // [3][kTile][KLD]
  unsigned* Kh = Kl + 3 * L::KBUF;            // [3][kTile][KLD]
  unsigned* Vl = Kh + 3 * L::KBUF;            // [3][D][VLD]
  unsigned* Vh = Vl + 3 * L::VBUF;            // [3][D][VLD]
  unsigned* Pw = Vh + 3 * L::VBUF;            // [2][ROWS][kTile / 2]
  unsigned short* tab = reinterpret_cast<unsigned short*>(Pw + 2 * L::PBUF);

  const int tid = threadIdx.x;
  const int r = tid >> 3, g = tid & 7;
  // heads interleaved, the last (causal: heaviest) row tiles first, so that the
  // lightest blocks fill the last wave
  const long long nheads = gridDim.x / tiles_per_head;
  const long long n = blockIdx.x % nheads;
  const int i0 = (tiles_per_head - 1 - (int)(blockIdx.x / nheads)) * ROWS;
  const int i = i0 + r;
  const short* Kg = K + n * S * D;
  const short* Vg = V + n * S * D;

  if (tid < 64) tab[tid] = prm.t[tid];
  int qreg[QW];  // the row's query values as int16 pairs
  {
    const int* qrow = reinterpret_cast<const int*>(Q + (n * S + (i < S ? i : 0)) * D);
#pragma unroll
    for (int w = 0; w < QW; w += 4) {
      int4 x = make_int4(0, 0, 0, 0);
      if (i < S) x = *reinterpret_cast<const int4*>(qrow + w);
      qreg[w] = x.x; qreg[w + 1] = x.y; qreg[w + 2] = x.z; qreg[w + 3] = x.w;
    }
  }

  // Staging of a tile in two halves, so that the global loads of tile t + 1
  // are in flight while tile t is scored: stage_load reads this thread's
  // share into registers (K as int16 quads, V as four keys of one channel),
  // stage_store splits it into low and high byte quads (V transposed to
  // channel-major) in buffer b. Keys >= S read as 0.
  constexpr int KT = (kTile * KW + kThreads - 1) / kThreads;        // K quads per thread
  constexpr int VT = (D * (kTile / 4) + kThreads - 1) / kThreads;  // V quads per thread
  int2 kreg[KT], vreg[VT];
  auto stage_load = [&](int tt) {
    const int t0 = tt * kTile;
#pragma unroll
    for (int x = 0; x < KT; ++x) {
      const int f = tid + x * kThreads;
      const int j = f / KW, w = f % KW;
      kreg[x] = make_int2(0, 0);
      if (f < kTile * KW && t0 + j < S) kreg[x] = *reinterpret_cast<const int2*>(Kg + (long long)(t0 + j) * D + 4 * w);
    }
#pragma unroll
    for (int x = 0; x < VT; ++x) {
      const int f = tid + x * kThreads;
      const int c = f / (kTile / 4), kq = f % (kTile / 4);
      unsigned e[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int key = t0 + 4 * kq + u;
        e[u] = (f < D * (kTile / 4) && key < S) ? (unsigned)(unsigned short)Vg[(long long)key * D + c] : 0u;
      }
      vreg[x] = make_int2((int)(e[0] | (e[1] << 16)), (int)(e[2] | (e[3] << 16)));
    }
  };
  auto stage_store = [&](int b) {
    unsigned* kl = Kl + b * L::KBUF;
    unsigned* kh = Kh + b * L::KBUF;
#pragma unroll
    for (int x = 0; x < KT; ++x) {
      const int f = tid + x * kThreads;
      if (f >= kTile * KW) continue;
      const int j = f / KW, w = f % KW;
      unsigned lo, hi;
      split4(kreg[x], lo, hi);
      kl[j * KLD + w] = lo;
      kh[j * KLD + w] = hi;
    }
    unsigned* vl = Vl + b * L::VBUF;
    unsigned* vh = Vh + b * L::VBUF;
#pragma unroll
    for (int x = 0; x < VT; ++x) {
      const int f = tid + x * kThreads;
      if (f >= D * (kTile / 4)) continue;
      const int c = f / (kTile / 4), kq = f % (kTile / 4);
      unsigned lo, hi;
      split4(vreg[x], lo, hi);
      vl[c * VLD + kq] = lo;
      vh[c * VLD + kq] = hi;
    }
  };

  const int my_last = causal ? min(i, S - 1) : S - 1;
  const int block_last = causal ? min(i0 + ROWS - 1, S - 1) : S - 1;
  const int nt = block_last / kTile + 1;
  long long m = 0, l = 0, acc[CH];
  bool have_m = false;
#pragma unroll
  for (int c = 0; c < CH; ++c) acc[c] = 0;

  stage_load(0);
  stage_store(0);
  __syncthreads();
  for (int tt = 0; tt < nt; ++tt) {
    const int t0 = tt * kTile;
    const int b = tt % 3;
    if (tt + 1 < nt) stage_load(tt + 1);  // consumed by stage_store after the scores

    // scores of keys g, g+8, g+16, g+24 of the tile
    const unsigned* kl = Kl + b * L::KBUF;
    const unsigned* kh = Kh + b * L::KBUF;
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
        const uint4 l4 = *reinterpret_cast<const uint4*>(&kl[kk * KLD + w]);
        const uint4 h4 = *reinterpret_cast<const uint4*>(&kh[kk * KLD + w]);
        const int qa0 = qreg[2 * w], qa1 = qreg[2 * w + 1], qa2 = qreg[2 * w + 2], qa3 = qreg[2 * w + 3];
        const int qb0 = qreg[2 * w + 4], qb1 = qreg[2 * w + 5], qb2 = qreg[2 * w + 6], qb3 = qreg[2 * w + 7];
        accl = dp2a_lo_su(qa0, l4.x, accl); accl = dp2a_hi_su(qa1, l4.x, accl);
        acch = dp2a_lo_ss(qa0, h4.x, acch); acch = dp2a_hi_ss(qa1, h4.x, acch);
        accl = dp2a_lo_su(qa2, l4.y, accl); accl = dp2a_hi_su(qa3, l4.y, accl);
        acch = dp2a_lo_ss(qa2, h4.y, acch); acch = dp2a_hi_ss(qa3, h4.y, acch);
        accl = dp2a_lo_su(qb0, l4.z, accl); accl = dp2a_hi_su(qb1, l4.z, accl);
        acch = dp2a_lo_ss(qb0, h4.z, acch); acch = dp2a_hi_ss(qb1, h4.z, acch);
        accl = dp2a_lo_su(qb2, l4.w, accl); accl = dp2a_hi_su(qb3, l4.w, accl);
        acch = dp2a_lo_ss(qb2, h4.w, acch); acch = dp2a_hi_ss(qb3, h4.w, acch);
      }
      const long long dot = (long long)acch * 256 + accl;  // the exact sum of the d products
      // arithmetic shifts: floor; |dot| < 2^38, so dot >> 14 fits in 32 bits, as C does
      // (scale checked on the host), and the product is one 32 x 32 -> 64-bit multiply
      z[u] = ((long long)(int)(dot >> 14) * (long long)(int)prm.C) >> 16;
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
    unsigned* pw_tile = Pw + (tt & 1) * L::PBUF;
    long long psum = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const unsigned p = (any && ok[u]) ? (unsigned)pow2_neg(m - z[u], tab) : 0u;  // <= 2^15
      psum += p;
      // weights of keys 2m and 2m+1 share a word: even threads take their odd neighbour's
      const unsigned pn = __shfl_down_sync(0xffffffffu, p, 1);
      if ((g & 1) == 0) pw_tile[r * (kTile / 2) + ((g + 8 * u) >> 1)] = p | (pn << 16);
    }
#pragma unroll
    for (int s = 1; s < 8; s <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, s);
    l += psum;
    if (tt + 1 < nt) stage_store((tt + 1) % 3);
    __syncthreads();  // the tile's weights written; tile tt + 1 staged

    // acc_c += sum_j p_j v_jc over the tile for channels c = g + 8 i
    const unsigned* vl = Vl + b * L::VBUF;
    const unsigned* vh = Vh + b * L::VBUF;
    uint4 pw[kTile / 8];
#pragma unroll
    for (int q4 = 0; q4 < kTile / 8; ++q4) pw[q4] = *reinterpret_cast<const uint4*>(&pw_tile[r * (kTile / 2) + 4 * q4]);
#pragma unroll
    for (int ci = 0; ci < CH; ++ci) {
      const int c = g + 8 * ci;
      unsigned al = 0;
      int ah = 0;
#pragma unroll
      for (int q4 = 0; q4 < kTile / 16; ++q4) {
        const uint4 l4 = *reinterpret_cast<const uint4*>(&vl[c * VLD + 4 * q4]);
        const uint4 h4 = *reinterpret_cast<const uint4*>(&vh[c * VLD + 4 * q4]);
        const uint4 pa = pw[2 * q4], pb = pw[2 * q4 + 1];  // keys 16 q4 .. 16 q4 + 15 as 8 pairs
        al = dp2a_lo_uu(pa.x, l4.x, al); al = dp2a_hi_uu(pa.y, l4.x, al);
        ah = dp2a_lo_us(pa.x, h4.x, ah); ah = dp2a_hi_us(pa.y, h4.x, ah);
        al = dp2a_lo_uu(pa.z, l4.y, al); al = dp2a_hi_uu(pa.w, l4.y, al);
        ah = dp2a_lo_us(pa.z, h4.y, ah); ah = dp2a_hi_us(pa.w, h4.y, ah);
        al = dp2a_lo_uu(pb.x, l4.z, al); al = dp2a_hi_uu(pb.y, l4.z, al);
        ah = dp2a_lo_us(pb.x, h4.z, ah); ah = dp2a_hi_us(pb.y, h4.z, ah);
        al = dp2a_lo_uu(pb.z, l4.w, al); al = dp2a_hi_uu(pb.w, l4.w, al);
        ah = dp2a_lo_us(pb.z, h4.w, ah); ah = dp2a_hi_us(pb.w, h4.w, ah);
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
  constexpr size_t smem = Q15Smem<D, ROWS>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(q15_attn_kernel<D, ROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int tiles = (p.S + ROWS - 1) / ROWS;
  q15_attn_kernel<D, ROWS><<<(unsigned)(p.N * tiles), 8 * ROWS, smem, st>>>(
      static_cast<const short*>(p.q), static_cast<const short*>(p.k), static_cast<const short*>(p.v),
      static_cast<short*>(p.o), p.S, tiles, p.causal, prm);
  return cudaGetLastError();
}

template <int D>
cudaError_t q15_launch(const AttnProblem& p, const Q15Params& prm, cudaStream_t st) {
  return q15_launch_rows<D, 16>(p, prm, st);
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
