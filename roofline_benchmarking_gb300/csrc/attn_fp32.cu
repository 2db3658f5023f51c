// attn_fp32.cu -- the three fp32 CUDA-core attention variants.
//
// kbench page ("kbench -- Transformer Attention Micro-benchmark Harness"),
// section "Implementation details / The three GPU kernels":
//  * naive: three global passes -- a GEMM that writes the S x S score matrix
//    to DRAM, a row softmax over it, a second GEMM for P*V;
//  * fused: one block per query row, the S-length score vector in shared
//    memory, one pass, shared memory O(S);
//  * flash: key/value tiles streamed through shared memory with an online
//    softmax (running max m and denominator l), shared memory O(Bc*d).
// All three compute O = softmax(Q K^T * scale [+ causal mask]) V over
// [N, S, d] row-major fp32 with fp32 arithmetic. Scores are carried in base 2
// (scale*log2(e) folded into one multiply) so that exp becomes exp2.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace kb {
namespace {

constexpr int kThreads = 256;  // 16 x 16 thread grid for the 64 x 64 tiles
constexpr int kBR = 64;        // query rows per tile
constexpr int kBC = 64;        // keys per tile
constexpr int kLD = kBR + 4;   // padded leading dimension of transposed tiles

template <int D>
struct Cols {
  // Output columns a thread owns: groups of W consecutive columns, G groups.
  static constexpr int W = D >= 64 ? 4 : 2;
  static constexpr int G = D / (16 * W);
  static_assert(G * 16 * W == D, "D must be 32, 64 or 128");
};

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// Loads rows [r0, r0+64) x D of a [S, D] matrix into a transposed shared tile
// dst[k * kLD + r] (feature-major), multiplied by `mul`; rows >= S read as 0.
// Consecutive threads take consecutive rows so that the shared stores do not
// conflict; the strided global reads are served from L1 across the k loop.
template <int D>
__device__ __forceinline__ void load_transposed(float* dst, const float* src, int r0, int S, float mul,
                                                int tid, int nthreads) {
  for (int f = tid; f < kBR * (D / 4); f += nthreads) {
    const int r = f % kBR, k4 = f / kBR;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r0 + r < S) x = ld4(src + (int64_t)(r0 + r) * D + 4 * k4);
    dst[(4 * k4 + 0) * kLD + r] = x.x * mul;
    dst[(4 * k4 + 1) * kLD + r] = x.y * mul;
    dst[(4 * k4 + 2) * kLD + r] = x.z * mul;
    dst[(4 * k4 + 3) * kLD + r] = x.w * mul;
  }
}

template <int D>
__device__ __forceinline__ void load_transposed(float* dst, const float* src, int r0, int S, float mul) {
  load_transposed<D>(dst, src, r0, S, mul, threadIdx.x, kThreads);
}

// Loads rows [r0, r0+64) x D of a [S, D] matrix into dst[r * D + k] (row-major).
template <int D>
__device__ __forceinline__ void load_rows(float* dst, const float* src, int r0, int S, int tid = 0,
                                          int nthreads = 0) {
  if (nthreads == 0) {
    tid = threadIdx.x;
    nthreads = kThreads;
  }
  for (int f = tid; f < kBC * (D / 4); f += nthreads) {
    const int r = f / (D / 4), k4 = f % (D / 4);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r0 + r < S) x = ld4(src + (int64_t)(r0 + r) * D + 4 * k4);
    *reinterpret_cast<float4*>(dst + r * D + 4 * k4) = x;
  }
}

// acc[a][*] += sum_c P[c][row a] * V[c][col]: P transposed in shared memory
// (Ps[c * kLD + r]), V row-major (Vs[c * D + col]); `kmax` keys.
template <int D>
__device__ __forceinline__ void pv_accumulate(float (&acc)[4][D / 16], const float* Ps, const float* Vs,
                                              int ty, int tx, int kmax) {
  using C = Cols<D>;
  for (int c = 0; c < kmax; ++c) {
    const float4 pa = ld4(Ps + c * kLD + ty * 4);
    const float pr[4] = {pa.x, pa.y, pa.z, pa.w};
#pragma unroll
    for (int g = 0; g < C::G; ++g) {
      float vv[C::W];
      const float* vp = Vs + c * D + g * 16 * C::W + tx * C::W;
      if constexpr (C::W == 4) {
        const float4 t = ld4(vp);
        vv[0] = t.x; vv[1] = t.y; vv[2] = t.z; vv[3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(vp);
        vv[0] = t.x; vv[1] = t.y;
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int e = 0; e < C::W; ++e) acc[a][g * C::W + e] = fmaf(pr[a], vv[e], acc[a][g * C::W + e]);
    }
  }
}

// ---------------------------------------------------------------------------
// flash at d = 128 (d <= 64 runs flash_f32x2_kernel below): one block per
// (head, 64-row query tile); grid.x = tiles * N with the heaviest causal tiles
// scheduled first. The block's 512 threads form two groups of 256 (each
// synchronised by its own named barrier) that take the even and the odd key
// tiles with their own K/V/P buffers and their own running max, sum and O, and
// are merged at the end -- twice the warps per query tile, so that small grids
// still hide the latency of shared memory. Two K/V buffers per group do not fit
// in shared memory at d = 128, so each group loads its tile, then computes.
// ---------------------------------------------------------------------------
constexpr int kFlashThreads = 2 * kThreads;

__device__ __forceinline__ void group_bar(int grp) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(kThreads) : "memory");
}

// Asynchronous global -> shared copies (cp.async): `bytes` (4 or 16) from src,
// or zeros when !valid (no byte is read then; src is still a mapped address).
template <int BYTES>
__device__ __forceinline__ void cp_async(float* dst, const float* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  if constexpr (BYTES == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d), "l"(src), "r"(valid ? 4 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Row stride of the flash kernel's row-major K tile: D + 4 floats, so that the
// rows a thread reads (consecutive keys across the 16 threads of a row group)
// fall in different 16-byte bank groups.
template <int D>
constexpr int flash_ldk() { return D + 4; }

// One group's copies of key tile [k0, k0 + 64): K row-major into Kr[r * (D + 4) + k]
// and V row-major into Vr[r * D + c], 16-byte copies by the group's `nthreads`
// threads; rows >= S are zero-filled.
template <int D>
__device__ __forceinline__ void flash_issue_kv(float* Kr, float* Vr, const float* Kh, const float* Vh, int k0, int S,
                                               int tid, int nthreads = kThreads) {
  for (int f = tid; f < kBC * (D / 4); f += nthreads) {
    const int r = f / (D / 4), c4 = f % (D / 4);
    const bool ok = k0 + r < S;
    cp_async<16>(Kr + r * flash_ldk<D>() + 4 * c4, Kh + (int64_t)(ok ? k0 + r : 0) * D + 4 * c4, ok);
  }
  for (int f = tid; f < kBC * (D / 4); f += nthreads) {
    const int r = f / (D / 4), c4 = f % (D / 4);
    const bool ok = k0 + r < S;
    cp_async<16>(Vr + r * D + 4 * c4, Vh + (int64_t)(ok ? k0 + r : 0) * D + 4 * c4, ok);
  }
}

// Floats of one group's K, V and P buffers in flash_f32_kernel.
template <int D>
constexpr int flash_group_floats() {
  return kBC * flash_ldk<D>() + kBC * D + kBC * kLD;
}

// s[a][b] = sum_k Qs[k][ty*4+a] * K[tx+16b][k]: Q transposed (Qs[k * kLD + r]), K
// row-major (Kr[key * (D + 4) + k]); the thread's keys are tx, tx+16, tx+32, tx+48.
template <int D>
__device__ __forceinline__ void qk_tile_rowk(float (&s)[4][4], const float* Qs, const float* Kr, int ty, int tx) {
  constexpr int LDK = flash_ldk<D>();
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) s[a][b] = 0.f;
#pragma unroll 2
  for (int k = 0; k < D; k += 4) {
    float4 q[4], kv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = ld4(Qs + (k + i) * kLD + ty * 4);
#pragma unroll
    for (int b = 0; b < 4; ++b) kv[b] = ld4(Kr + (tx + 16 * b) * LDK + k);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      s[0][b] = fmaf(q[0].x, kv[b].x, s[0][b]);
      s[1][b] = fmaf(q[0].y, kv[b].x, s[1][b]);
      s[2][b] = fmaf(q[0].z, kv[b].x, s[2][b]);
      s[3][b] = fmaf(q[0].w, kv[b].x, s[3][b]);
      s[0][b] = fmaf(q[1].x, kv[b].y, s[0][b]);
      s[1][b] = fmaf(q[1].y, kv[b].y, s[1][b]);
      s[2][b] = fmaf(q[1].z, kv[b].y, s[2][b]);
      s[3][b] = fmaf(q[1].w, kv[b].y, s[3][b]);
      s[0][b] = fmaf(q[2].x, kv[b].z, s[0][b]);
      s[1][b] = fmaf(q[2].y, kv[b].z, s[1][b]);
      s[2][b] = fmaf(q[2].z, kv[b].z, s[2][b]);
      s[3][b] = fmaf(q[2].w, kv[b].z, s[3][b]);
      s[0][b] = fmaf(q[3].x, kv[b].w, s[0][b]);
      s[1][b] = fmaf(q[3].y, kv[b].w, s[1][b]);
      s[2][b] = fmaf(q[3].z, kv[b].w, s[2][b]);
      s[3][b] = fmaf(q[3].w, kv[b].w, s[3][b]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kFlashThreads, 1) flash_f32_kernel(const float* __restrict__ Q,
                                                                  const float* __restrict__ K,
                                                                  const float* __restrict__ V,
                                                                  float* __restrict__ O, float* __restrict__ lse,
                                                                  int64_t N, int S, int causal, float scale_log2,
                                                                  float* __restrict__ part, int split_from) {
  // part / split_from: causal query tiles qt >= split_from are computed by two
  // blocks, over key tiles [0, h) and [h, qt] with h = ceil((qt + 1) / 2); each
  // writes its merged online-softmax state (m, l and the unnormalised O rows) to
  // `part` and flash_merge_kernel combines the two. split_from = tiles: no split.
  static_assert(D == 128, "d <= 64 runs flash_f32x2_kernel");
  using C = Cols<D>;
  constexpr int GROUP = flash_group_floats<D>();      // floats of one group's K, V and P buffers
  constexpr int KV = kBC * flash_ldk<D>() + kBC * D;  // the K + V buffer pair
  extern __shared__ float4 smem4[];
  float* Qs = reinterpret_cast<float*>(smem4);  // [D][kLD], both groups
  const int grp = threadIdx.x / kThreads, ltid = threadIdx.x % kThreads;
  float* Ks = Qs + D * kLD + grp * GROUP;       // [kBC][D + 4]
  float* Vs = Ks + kBC * flash_ldk<D>();        // [kBC][D]
  float* Ps = Ks + KV;                          // [kBC][kLD]

  const int ntiles = (S + kBR - 1) / kBR;
  const int nsplit = ntiles - split_from;  // split query tiles per head
  const int64_t n = blockIdx.x % N;
  const int u = (int)(blockIdx.x / N);  // heaviest units first: the split tiles' parts, then the rest
  int qt, kb, ke, pt = -1;              // query tile, key tiles [kb, ke], part (-1: whole tile)
  if (u < 2 * nsplit) {
    qt = ntiles - 1 - u / 2;
    pt = u & 1;
    const int h = (qt + 2) / 2;
    kb = pt ? h : 0;
    ke = pt ? qt : h - 1;
  } else {
    qt = split_from - 1 - (u - 2 * nsplit);
    kb = 0;
    ke = causal ? qt : ntiles - 1;
  }
  const int q0 = qt * kBR;
  const int tx = ltid & 15, ty = ltid >> 4;
  const float* Qh = Q + n * S * D;
  const float* Kh = K + n * S * D;
  const float* Vh = V + n * S * D;

  load_transposed<D>(Qs, Qh, q0, S, scale_log2, threadIdx.x, kFlashThreads);
  __syncthreads();

  float m[4], l[4], acc[4][D / 16];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    m[a] = -INFINITY;
    l[a] = 0.f;
#pragma unroll
    for (int c = 0; c < D / 16; ++c) acc[a][c] = 0.f;
  }

  for (int kt = kb + grp; kt <= ke; kt += 2) {
    const int k0 = kt * kBC;
    group_bar(grp);  // the group's previous K, V and P are no longer read
    flash_issue_kv<D>(Ks, Vs, Kh, Vh, k0, S, ltid);
    cp_async_commit();
    cp_async_wait<0>();
    group_bar(grp);

    float s[4][4];
    qk_tile_rowk<D>(s, Qs, Ks, ty, tx);

    // mask, then the online-softmax update for each of the thread's 4 rows
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int row = q0 + ty * 4 + a;
      float tmax = -INFINITY;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int key = k0 + tx + 16 * b;
        if (key >= S || (causal && key > row)) s[a][b] = -INFINITY;
        tmax = fmaxf(tmax, s[a][b]);
      }
      tmax = group_max<16>(tmax);
      const float m_new = fmaxf(m[a], tmax);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(m[a] - m_use);
      float rs = 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        s[a][b] = exp2f(s[a][b] - m_use);
        rs += s[a][b];
      }
      rs = group_sum<16>(rs);
      l[a] = l[a] * alpha + rs;
      m[a] = m_new;
#pragma unroll
      for (int c = 0; c < D / 16; ++c) acc[a][c] *= alpha;
    }
#pragma unroll
    for (int b = 0; b < 4; ++b)
      *reinterpret_cast<float4*>(Ps + (tx + 16 * b) * kLD + ty * 4) = make_float4(s[0][b], s[1][b], s[2][b], s[3][b]);
    group_bar(grp);
    pv_accumulate<D>(acc, Ps, Vs, ty, tx, kBC);
  }

  // merge: group 1 publishes its state (field-major, one column per thread) in
  // its own buffers, group 0 combines the two online softmaxes and writes O
  constexpr int F = 8 + 4 * (D / 16);  // m[4], l[4], acc[4][D/16]
  float* X = Qs + D * kLD + GROUP;     // group 1's buffers
  __syncthreads();
  if (grp == 1) {
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      X[a * kThreads + ltid] = m[a];
      X[(4 + a) * kThreads + ltid] = l[a];
#pragma unroll
      for (int c = 0; c < D / 16; ++c) X[(8 + a * (D / 16) + c) * kThreads + ltid] = acc[a][c];
    }
  }
  __syncthreads();
  if (grp == 1) return;
  static_assert(F * kThreads <= GROUP, "merge state fits in one group's buffers");
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int row = q0 + ty * 4 + a;
    const float m1 = X[a * kThreads + ltid], l1 = X[(4 + a) * kThreads + ltid];
    // group 0 always sees key kb * 64 <= every row of the tile, so m[a] and mm are finite
    const float mm = fmaxf(m[a], m1);
    const float s0 = exp2f(m[a] - mm);
    const float s1 = m1 == -INFINITY ? 0.f : exp2f(m1 - mm);
    const float lt = l[a] * s0 + l1 * s1;
    if (row >= S) continue;
    if (pt >= 0) {  // a part of a split tile: its state, for flash_merge_kernel
      const int lr = ty * 4 + a;
      float* st = part + ((n * nsplit + (ntiles - 1 - qt)) * 2 + pt) * (int64_t)(kBR * (D + 2));
      if (tx == 0) {
        st[lr] = mm;
        st[kBR + lr] = lt;
      }
#pragma unroll
      for (int g = 0; g < C::G; ++g)
#pragma unroll
        for (int e = 0; e < C::W; ++e) {
          const float a1 = X[(8 + a * (D / 16) + g * C::W + e) * kThreads + ltid];
          st[2 * kBR + lr * D + g * 16 * C::W + tx * C::W + e] = acc[a][g * C::W + e] * s0 + a1 * s1;
        }
      continue;
    }
    const float inv = 1.0f / lt;
    // natural log of sum_j exp(score): the scores sum to 2^mm * lt in base 2
    if (lse != nullptr && tx == 0) lse[n * S + row] = (mm + log2f(lt)) * 0.6931471805599453f;
    float* orow = O + (n * S + row) * D;
#pragma unroll
    for (int g = 0; g < C::G; ++g)
#pragma unroll
      for (int e = 0; e < C::W; ++e) {
        const float a1 = X[(8 + a * (D / 16) + g * C::W + e) * kThreads + ltid];
        orow[g * 16 * C::W + tx * C::W + e] = (acc[a][g * C::W + e] * s0 + a1 * s1) * inv;
      }
  }
}

// ---------------------------------------------------------------------------
// flash at d <= 64 with paired fp32 FMAs (fma.rn.f32x2: two products per lane
// and instruction; the FMA pipe's rate per product is that of the scalar FMA,
// measured on GB300, but each instruction issues two). The query tile, the two
// thread groups over even and odd key tiles, the causal split and the merge are
// those of flash_f32_kernel. What changes:
//  * Q K^T: Q and K row-major; one paired FMA takes features (k, k+1) of a
//    query row and of a key, so each score is carried as two partial sums
//    (even and odd features) that are added once per tile;
//  * P V: P row-major as the softmax writes it; V re-laid from its row-major
//    copy into key pairs, Vp[j/2][c] = (V[j][c], V[j+1][c]), so one paired FMA
//    takes keys (j, j+1) of a P row and of a V column; each output gathers
//    even-key and odd-key partial sums over a tile, added into O after it;
//  * register tiles of 8 rows x 4 keys (and 8 rows x 4 output columns), with
//    groups of 128 threads at up to 255 registers. A 16-byte shared load
//    costs about 4 wavefronts when the lanes read distinct rows (K, V) and 2
//    when each half-warp reads one row (Q, P) (measured); with 4 x 4 tiles a
//    warp's 32 paired FMAs per 4 features took 24 wavefronts for 16 cycles of
//    FMA-pipe work, with 8 x 4 tiles its 64 take 32 wavefronts for 32 cycles.
// Thread (tx, ty) of a group owns query rows ty + 8 a (a < 8), keys tx + 16 b
// (b < 4) and output columns 32 g + 2 tx + e (e < 2, g < D / 32).
// ---------------------------------------------------------------------------
constexpr int kFx2Group = 128;              // threads per key-tile group
constexpr int kFx2Threads = 2 * kFx2Group;  // two groups: even and odd key tiles

template <int D>
struct Fx2 {
  static constexpr int LDQ = D + 4;       // row stride of the Q and K tiles
  static constexpr int LDP = kBC + 16;    // row stride of the P tile: rows ty and ty + 1 16 banks apart
  static constexpr int G = D / 32;        // column groups of a thread
  static constexpr int NO = 2 * G;        // output columns of a thread per row
  static constexpr int KBUF = kBC * LDQ;  // one K buffer
  static constexpr int VBUF = kBC * D;    // one row-major V buffer (the cp.async target)
  static constexpr int GROUP = 2 * KBUF + 2 * VBUF + kBC * D + kBR * LDP;  // K x 2, V x 2, Vp, P
  static constexpr int SMEM_FLOATS = kBR * LDQ + 2 * GROUP;
};

__device__ __forceinline__ void st4(float* p, float4 x) { *reinterpret_cast<float4*>(p) = x; }

__device__ __forceinline__ void fx2_group_bar(int grp) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(kFx2Group) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kFx2Threads, 1) flash_f32x2_kernel(const float* __restrict__ Q,
                                                                  const float* __restrict__ K,
                                                                  const float* __restrict__ V,
                                                                  float* __restrict__ O, float* __restrict__ lse,
                                                                  int64_t N, int S, int causal, float scale_log2,
                                                                  float* __restrict__ part, int split_from) {
  static_assert(D == 32 || D == 64, "the paired-FMA flash kernel runs d = 32 and 64");
  using F = Fx2<D>;
  constexpr int RT = 8;  // query rows per thread
  extern __shared__ float4 smem4[];
  float* Qs = reinterpret_cast<float*>(smem4);  // [kBR][LDQ], scaled, both groups
  const int grp = threadIdx.x / kFx2Group, ltid = threadIdx.x % kFx2Group;
  float* Kb = Qs + kBR * F::LDQ + grp * F::GROUP;  // buffer b: [kBC][LDQ] at Kb + b KBUF
  float* Vb = Kb + 2 * F::KBUF;                    // buffer b: [kBC][D] at Vb + b VBUF
  float* Vp = Vb + 2 * F::VBUF;                    // [kBC / 2][2 D]: key pairs
  float* Pr = Vp + kBC * D;                        // [kBR][LDP]

  const int ntiles = (S + kBR - 1) / kBR;
  const int nsplit = ntiles - split_from;
  const int64_t n = blockIdx.x % N;
  const int u = (int)(blockIdx.x / N);
  int qt, kb, ke, pt = -1;
  if (u < 2 * nsplit) {
    qt = ntiles - 1 - u / 2;
    pt = u & 1;
    const int h = (qt + 2) / 2;
    kb = pt ? h : 0;
    ke = pt ? qt : h - 1;
  } else {
    qt = split_from - 1 - (u - 2 * nsplit);
    kb = 0;
    ke = causal ? qt : ntiles - 1;
  }
  const int q0 = qt * kBR;
  const int tx = ltid & 15, ty = ltid >> 4;  // a half-warp shares ty: its row's 16 key lanes
  const float* Qh = Q + n * S * D;
  const float* Kh = K + n * S * D;
  const float* Vh = V + n * S * D;

  for (int f = threadIdx.x; f < kBR * (D / 4); f += kFx2Threads) {  // Q rows, scaled; rows >= S read as 0
    const int r = f / (D / 4), c4 = f % (D / 4);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (q0 + r < S) x = ld4(Qh + (int64_t)(q0 + r) * D + 4 * c4);
    st4(Qs + r * F::LDQ + 4 * c4, make_float4(x.x * scale_log2, x.y * scale_log2, x.z * scale_log2,
                                               x.w * scale_log2));
  }
  __syncthreads();

  float m[RT], l[RT], o[RT][F::NO];
#pragma unroll
  for (int a = 0; a < RT; ++a) {
    m[a] = -INFINITY;
    l[a] = 0.f;
#pragma unroll
    for (int j = 0; j < F::NO; ++j) o[a][j] = 0.f;
  }

  if (kb + grp <= ke) flash_issue_kv<D>(Kb, Vb, Kh, Vh, (kb + grp) * kBC, S, ltid, kFx2Group);
  cp_async_commit();
  for (int kt = kb + grp, it = 0; kt <= ke; kt += 2, ++it) {
    const int k0 = kt * kBC;
    const float* Ks = Kb + (it & 1) * F::KBUF;
    const float* Vs = Vb + (it & 1) * F::VBUF;
    // the buffers of the group's previous tile: every thread of the group passed
    // the previous iteration's second barrier, after its last read of them
    if (kt + 2 <= ke)
      flash_issue_kv<D>(Kb + ((it + 1) & 1) * F::KBUF, Vb + ((it + 1) & 1) * F::VBUF, Kh, Vh, k0 + 2 * kBC, S,
                        ltid, kFx2Group);
    cp_async_commit();
    cp_async_wait<1>();  // this thread's copies of tile kt have landed
    fx2_group_bar(grp);  // everyone's have; the group's previous P and Vp are no longer read

    // V as key pairs. Per store instruction the lanes of one key pair write
    // 16-byte chunks 2 c4 + h with h = (c4 / 4) % 2: all eight bank groups.
    for (int w = ltid; w < (kBC / 2) * (D / 4); w += kFx2Group) {
      const int kp = w / (D / 4), c4 = w % (D / 4);
      const float4 a = ld4(Vs + (2 * kp) * D + 4 * c4), b = ld4(Vs + (2 * kp + 1) * D + 4 * c4);
      const float4 lo = make_float4(a.x, b.x, a.y, b.y), hi = make_float4(a.z, b.z, a.w, b.w);
      float* dst = Vp + kp * 2 * D + 8 * c4;
      const int sw = ((c4 >> 2) & 1) * 4;
      st4(dst + sw, sw ? hi : lo);
      st4(dst + 4 - sw, sw ? lo : hi);
    }

    // scores of rows ty + 8 a and keys tx + 16 b, as even- and odd-feature sums
    float s[RT][4];
    {
      float2 s2[RT][4];
#pragma unroll
      for (int a = 0; a < RT; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) s2[a][b] = make_float2(0.f, 0.f);
      // per 4 features: all 32 products of features (k, k+1), then those of
      // (k+2, k+3), so that the two FMAs into one accumulator are 32 apart
#pragma unroll
      for (int k = 0; k < D; k += 4) {
        float4 kv[4], qv[RT];
#pragma unroll
        for (int b = 0; b < 4; ++b) kv[b] = ld4(Ks + (tx + 16 * b) * F::LDQ + k);
#pragma unroll
        for (int a = 0; a < RT; ++a) qv[a] = ld4(Qs + (ty + 8 * a) * F::LDQ + k);
#pragma unroll
        for (int a = 0; a < RT; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b)
            s2[a][b] = __ffma2_rn(make_float2(qv[a].x, qv[a].y), make_float2(kv[b].x, kv[b].y), s2[a][b]);
#pragma unroll
        for (int a = 0; a < RT; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b)
            s2[a][b] = __ffma2_rn(make_float2(qv[a].z, qv[a].w), make_float2(kv[b].z, kv[b].w), s2[a][b]);
      }
#pragma unroll
      for (int a = 0; a < RT; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) s[a][b] = s2[a][b].x + s2[a][b].y;
    }

    // mask, online-softmax update, P row-major
#pragma unroll
    for (int a = 0; a < RT; ++a) {
      const int row = q0 + ty + 8 * a;
      float tmax = -INFINITY;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int key = k0 + tx + 16 * b;
        if (key >= S || (causal && key > row)) s[a][b] = -INFINITY;
        tmax = fmaxf(tmax, s[a][b]);
      }
      tmax = group_max<16>(tmax);
      const float m_new = fmaxf(m[a], tmax);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(m[a] - m_use);
      float rs = 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        s[a][b] = exp2f(s[a][b] - m_use);
        rs += s[a][b];
      }
      rs = group_sum<16>(rs);
      l[a] = l[a] * alpha + rs;
      m[a] = m_new;
#pragma unroll
      for (int j = 0; j < F::NO; ++j) o[a][j] *= alpha;
#pragma unroll
      for (int b = 0; b < 4; ++b) Pr[(ty + 8 * a) * F::LDP + tx + 16 * b] = s[a][b];
    }
    fx2_group_bar(grp);  // P and Vp of this tile are visible to the group

    // O += P V over the tile's 64 keys, two keys per paired FMA, as even-key and
    // odd-key partial sums added into O at the end of the tile
    float2 acc[RT][F::NO];
#pragma unroll
    for (int a = 0; a < RT; ++a)
#pragma unroll
      for (int j = 0; j < F::NO; ++j) acc[a][j] = make_float2(0.f, 0.f);
#pragma unroll 2
    for (int c4 = 0; c4 < kBC / 4; ++c4) {
      float4 v[2][F::G];
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int g = 0; g < F::G; ++g) v[kk][g] = ld4(Vp + (2 * c4 + kk) * 2 * D + 64 * g + 4 * tx);
      float4 p[RT];
#pragma unroll
      for (int a = 0; a < RT; ++a) p[a] = ld4(Pr + (ty + 8 * a) * F::LDP + 4 * c4);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)  // key pair 2 c4 + kk for every row, then the next
#pragma unroll
        for (int a = 0; a < RT; ++a) {
          const float2 pp = kk == 0 ? make_float2(p[a].x, p[a].y) : make_float2(p[a].z, p[a].w);
#pragma unroll
          for (int g = 0; g < F::G; ++g) {
            acc[a][2 * g] = __ffma2_rn(pp, make_float2(v[kk][g].x, v[kk][g].y), acc[a][2 * g]);
            acc[a][2 * g + 1] = __ffma2_rn(pp, make_float2(v[kk][g].z, v[kk][g].w), acc[a][2 * g + 1]);
          }
        }
    }
#pragma unroll
    for (int a = 0; a < RT; ++a)
#pragma unroll
      for (int j = 0; j < F::NO; ++j) o[a][j] += acc[a][j].x + acc[a][j].y;
  }

  // merge of the two groups' online softmaxes, as in flash_f32_kernel; output
  // column of the thread's value j: 32 (j / 2) + 2 tx + j % 2
  float* X = Qs + kBR * F::LDQ + F::GROUP;  // group 1's buffers
  constexpr int FIELDS = 2 * RT + RT * F::NO;
  static_assert(FIELDS * kFx2Group <= F::GROUP, "merge state fits in one group's buffers");
  __syncthreads();
  if (grp == 1) {
#pragma unroll
    for (int a = 0; a < RT; ++a) {
      X[a * kFx2Group + ltid] = m[a];
      X[(RT + a) * kFx2Group + ltid] = l[a];
#pragma unroll
      for (int j = 0; j < F::NO; ++j) X[(2 * RT + a * F::NO + j) * kFx2Group + ltid] = o[a][j];
    }
  }
  __syncthreads();
  if (grp == 1) return;
#pragma unroll
  for (int a = 0; a < RT; ++a) {
    const int lr = ty + 8 * a, row = q0 + lr;
    const float m1 = X[a * kFx2Group + ltid], l1 = X[(RT + a) * kFx2Group + ltid];
    const float mm = fmaxf(m[a], m1);
    const float s0 = exp2f(m[a] - mm);
    const float s1 = m1 == -INFINITY ? 0.f : exp2f(m1 - mm);
    const float lt = l[a] * s0 + l1 * s1;
    if (row >= S) continue;
    float val[F::NO];
#pragma unroll
    for (int j = 0; j < F::NO; ++j) val[j] = o[a][j] * s0 + X[(2 * RT + a * F::NO + j) * kFx2Group + ltid] * s1;
    if (pt >= 0) {  // a part of a split tile: its state, for flash_merge_kernel
      float* st = part + ((n * nsplit + (ntiles - 1 - qt)) * 2 + pt) * (int64_t)(kBR * (D + 2));
      if (tx == 0) {
        st[lr] = mm;
        st[kBR + lr] = lt;
      }
#pragma unroll
      for (int g = 0; g < F::G; ++g)
        *reinterpret_cast<float2*>(st + 2 * kBR + lr * D + 32 * g + 2 * tx) = make_float2(val[2 * g], val[2 * g + 1]);
      continue;
    }
    const float inv = 1.0f / lt;
    if (lse != nullptr && tx == 0) lse[n * S + row] = (mm + log2f(lt)) * 0.6931471805599453f;
    float* orow = O + (n * S + row) * D;
#pragma unroll
    for (int g = 0; g < F::G; ++g)
      *reinterpret_cast<float2*>(orow + 32 * g + 2 * tx) = make_float2(val[2 * g] * inv, val[2 * g + 1] * inv);
  }
}

// Combines the two parts of every split query tile: O = (acc0 s0 + acc1 s1) / l
// with s_p = 2^(m_p - max(m0, m1)), l = l0 s0 + l1 s1 (two online-softmax states
// over disjoint key ranges, combined like the flash kernel's own group merge).
// One block of 256 threads per split tile: thread t takes row t / 4 and the
// columns c = t % 4 + 4 i.
template <int D>
__global__ void __launch_bounds__(256) flash_merge_kernel(const float* __restrict__ part, float* __restrict__ O,
                                                        float* __restrict__ lse, int S, int nsplit) {
  const int64_t n = blockIdx.x / nsplit;
  const int j = (int)(blockIdx.x % nsplit);
  const int ntiles = (S + kBR - 1) / kBR;
  const int qt = ntiles - 1 - j;
  const int lr = threadIdx.x >> 2, c0 = threadIdx.x & 3;
  const int row = qt * kBR + lr;
  if (row >= S) return;
  const float* p0 = part + (n * nsplit + j) * 2 * (int64_t)(kBR * (D + 2));
  const float* p1 = p0 + kBR * (D + 2);
  const float m0 = p0[lr], m1 = p1[lr];
  const float mm = fmaxf(m0, m1);
  const float s0 = m0 == -INFINITY ? 0.f : exp2f(m0 - mm);
  const float s1 = m1 == -INFINITY ? 0.f : exp2f(m1 - mm);
  const float lt = p0[kBR + lr] * s0 + p1[kBR + lr] * s1;
  const float inv = 1.0f / lt;
  if (lse != nullptr && c0 == 0) lse[n * S + row] = (mm + log2f(lt)) * 0.6931471805599453f;
  float* orow = O + (n * S + row) * D;
  for (int c = c0; c < D; c += 4)
    orow[c] = (p0[2 * kBR + lr * D + c] * s0 + p1[2 * kBR + lr * D + c] * s1) * inv;
}

// ---------------------------------------------------------------------------
// naive pass 1: scores[n][i][j] = scale * q_i . k_j as a tiled GEMM; causal
// entries j > i are written as -inf in the diagonal tile and tiles wholly
// above the diagonal are skipped (pass 2 and 3 never read them).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads) naive_scores_kernel(const float* __restrict__ Q,
                                                                const float* __restrict__ K,
                                                                float* __restrict__ Sc, int64_t N, int S,
                                                                int causal, float scale) {
  extern __shared__ float4 smem4[];
  constexpr int LDK = flash_ldk<D>();
  float* Qs = reinterpret_cast<float*>(smem4);  // [D][kLD] (transposed)
  float* Ks = Qs + D * kLD;                      // [kBC][D + 4] (row-major)
  const int kt = blockIdx.x, qt = blockIdx.y;
  const int64_t n = blockIdx.z;
  if (causal && kt > qt) return;
  const int q0 = qt * kBR, k0 = kt * kBC;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  load_transposed<D>(Qs, Q + n * S * D, q0, S, scale);
  const float* Kh = K + n * S * D;
  for (int f = tid; f < kBC * (D / 4); f += kThreads) {  // coalesced 16-byte loads; rows >= S read as 0
    const int r = f / (D / 4), c4 = f % (D / 4);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (k0 + r < S) x = ld4(Kh + (int64_t)(k0 + r) * D + 4 * c4);
    *reinterpret_cast<float4*>(Ks + r * LDK + 4 * c4) = x;
  }
  __syncthreads();
  float s[4][4];
  qk_tile_rowk<D>(s, Qs, Ks, ty, tx);  // the thread's keys: tx, tx + 16, tx + 32, tx + 48
  float* Sh = Sc + n * (int64_t)S * S;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int row = q0 + ty * 4 + a;
    if (row >= S) continue;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int key = k0 + tx + 16 * b;
      if (key >= S) continue;
      Sh[(int64_t)row * S + key] = (causal && key > row) ? -INFINITY : s[a][b];
    }
  }
}

// naive pass 2: in-place row softmax, one warp per row over its visible keys.
// When S is a multiple of 4 every row starts 16 bytes aligned and the row is
// read and written as float4 (the running max rescales the sum once per four
// scores); the remaining keys, and every key otherwise, one float at a time.
__global__ void __launch_bounds__(kThreads) naive_softmax_kernel(float* __restrict__ Sc, int64_t rows, int S,
                                                                 int causal) {
  const int64_t r = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int lane = threadIdx.x & 31;
  const int i = (int)(r % S);
  const int len = causal ? i + 1 : S;
  float* row = Sc + r * S;
  const int n4 = (S & 3) == 0 ? len >> 2 : 0;  // whole float4s of the visible keys
  float4* row4 = reinterpret_cast<float4*>(row);
  // one read pass: lane-local running max and sum, then combined across lanes
  float m = -INFINITY, l = 0.f;
  for (int q = lane; q < n4; q += 32) {
    const float4 v = row4[q];
    const float x0 = v.x * kLog2e, x1 = v.y * kLog2e, x2 = v.z * kLog2e, x3 = v.w * kLog2e;
    const float m_new = fmaxf(m, fmaxf(fmaxf(x0, x1), fmaxf(x2, x3)));
    l = l * exp2f(m - m_new) + ((exp2f(x0 - m_new) + exp2f(x1 - m_new)) + (exp2f(x2 - m_new) + exp2f(x3 - m_new)));
    m = m_new;
  }
  for (int j = 4 * n4 + lane; j < len; j += 32) {
    const float x = row[j] * kLog2e;
    const float m_new = fmaxf(m, x);
    l = l * exp2f(m - m_new) + exp2f(x - m_new);
    m = m_new;
  }
  const float mw = warp_max(m);
  l = warp_sum(m == -INFINITY ? 0.f : l * exp2f(m - mw));
  const float inv = 1.0f / l;
  for (int q = lane; q < n4; q += 32) {
    const float4 v = row4[q];
    row4[q] = make_float4(exp2f(v.x * kLog2e - mw) * inv, exp2f(v.y * kLog2e - mw) * inv,
                          exp2f(v.z * kLog2e - mw) * inv, exp2f(v.w * kLog2e - mw) * inv);
  }
  for (int j = 4 * n4 + lane; j < len; j += 32) row[j] = exp2f(row[j] * kLog2e - mw) * inv;
}

// naive pass 3: O = P V as a tiled GEMM over the visible key tiles. As in the
// flash kernel, two groups of 256 threads take the even and the odd key tiles
// with their own buffers, and group 0 adds group 1's partial sums. Each group
// double-buffers its P and V tiles with cp.async; P stays row-major as the
// softmax pass left it (16-byte copies when S is a multiple of 4, so that every
// copied row segment is 16-byte aligned, else 4-byte copies), and the entries
// above the diagonal of the causal diagonal tile (still -inf) are zeroed.
constexpr int kLDP = kBC + 4;  // row stride of a P tile

template <int D>
__device__ __forceinline__ void naive_pv_issue(float* Pr, float* Vr, const float* Sh, const float* Vh, int q0, int k0,
                                               int S, int tid, bool vec16) {
  if (vec16) {
    for (int f = tid; f < kBR * (kBC / 4); f += kThreads) {
      const int r = f / (kBC / 4), c4 = f % (kBC / 4);
      const int row = q0 + r, col = k0 + 4 * c4;
      const bool ok = row < S && col < S;  // S % 4 == 0: a 4-key chunk is wholly in or out
      cp_async<16>(Pr + r * kLDP + 4 * c4, Sh + (ok ? (int64_t)row * S + col : 0), ok);
    }
  } else {
    for (int f = tid; f < kBR * kBC; f += kThreads) {
      const int r = f / kBC, c = f % kBC;
      const int row = q0 + r, col = k0 + c;
      const bool ok = row < S && col < S;
      cp_async<4>(Pr + r * kLDP + c, Sh + (ok ? (int64_t)row * S + col : 0), ok);
    }
  }
  for (int f = tid; f < kBC * (D / 4); f += kThreads) {
    const int r = f / (D / 4), c4 = f % (D / 4);
    const bool ok = k0 + r < S;
    cp_async<16>(Vr + r * D + 4 * c4, Vh + (int64_t)(ok ? k0 + r : 0) * D + 4 * c4, ok);
  }
}

// acc[a][*] += sum_c P[ty*4+a][c] * V[c][col], P row-major (Pr[r * kLDP + c]), four keys per step.
template <int D>
__device__ __forceinline__ void pv_accumulate_rowp(float (&acc)[4][D / 16], const float* Pr, const float* Vs, int ty,
                                                   int tx) {
  using C = Cols<D>;
#pragma unroll 2
  for (int c = 0; c < kBC; c += 4) {
    float4 p4[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) p4[a] = ld4(Pr + (ty * 4 + a) * kLDP + c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float pr[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) pr[a] = i == 0 ? p4[a].x : i == 1 ? p4[a].y : i == 2 ? p4[a].z : p4[a].w;
#pragma unroll
      for (int g = 0; g < C::G; ++g) {
        float vv[C::W];
        const float* vp = Vs + (c + i) * D + g * 16 * C::W + tx * C::W;
        if constexpr (C::W == 4) {
          const float4 t = ld4(vp);
          vv[0] = t.x; vv[1] = t.y; vv[2] = t.z; vv[3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2*>(vp);
          vv[0] = t.x; vv[1] = t.y;
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int e = 0; e < C::W; ++e) acc[a][g * C::W + e] = fmaf(pr[a], vv[e], acc[a][g * C::W + e]);
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kFlashThreads, 1) naive_pv_kernel(const float* __restrict__ Sc,
                                                                    const float* __restrict__ V,
                                                                    float* __restrict__ O, int64_t N, int S,
                                                                    int causal) {
  using C = Cols<D>;
  constexpr int BUF = kBR * kLDP + kBC * D;  // floats of one P + V buffer pair
  constexpr int GROUP = 2 * BUF;              // a group's two buffer pairs
  extern __shared__ float4 smem4[];
  const int grp = threadIdx.x / kThreads, ltid = threadIdx.x % kThreads;
  float* B0 = reinterpret_cast<float*>(smem4) + grp * GROUP;  // buffer b: P [kBR][kLDP] at B0 + b BUF, V after it
  const int ntiles = (S + kBR - 1) / kBR;
  const int64_t n = blockIdx.x % N;
  const int qt = ntiles - 1 - (int)(blockIdx.x / N);
  const int q0 = qt * kBR;
  const int tx = ltid & 15, ty = ltid >> 4;
  const float* Sh = Sc + n * (int64_t)S * S;
  const float* Vh = V + n * S * D;
  const bool vec16 = (S & 3) == 0;
  float acc[4][D / 16];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < D / 16; ++c) acc[a][c] = 0.f;

  const int kt_last = causal ? qt : ntiles - 1;
  if (grp <= kt_last) naive_pv_issue<D>(B0, B0 + kBR * kLDP, Sh, Vh, q0, grp * kBC, S, ltid, vec16);
  cp_async_commit();
  for (int kt = grp, it = 0; kt <= kt_last; kt += 2, ++it) {
    float* Pr = B0 + (it & 1) * BUF;
    float* Vs = Pr + kBR * kLDP;
    group_bar(grp);  // the group's other buffer pair is no longer read
    if (kt + 2 <= kt_last) {
      float* Pn = B0 + ((it + 1) & 1) * BUF;
      naive_pv_issue<D>(Pn, Pn + kBR * kLDP, Sh, Vh, q0, (kt + 2) * kBC, S, ltid, vec16);
    }
    cp_async_commit();
    cp_async_wait<1>();  // this thread's copies of tile kt have landed
    group_bar(grp);
    if (causal && kt == qt) {  // the diagonal tile: keys after the row are masked
      for (int f = ltid; f < kBR * kBC; f += kThreads) {
        const int r = f / kBC, c = f % kBC;
        if (c > r) Pr[r * kLDP + c] = 0.f;
      }
      group_bar(grp);
    }
    pv_accumulate_rowp<D>(acc, Pr, Vs, ty, tx);
  }
  float* X = reinterpret_cast<float*>(smem4) + GROUP;  // group 1's buffers hold its partial sums
  static_assert(4 * (D / 16) * kThreads <= GROUP, "partial sums fit in one group's buffers");
  __syncthreads();
  if (grp == 1) {
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < D / 16; ++c) X[(a * (D / 16) + c) * kThreads + ltid] = acc[a][c];
  }
  __syncthreads();
  if (grp == 1) return;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int row = q0 + ty * 4 + a;
    if (row >= S) continue;
    float* orow = O + (n * S + row) * D;
#pragma unroll
    for (int g = 0; g < C::G; ++g)
#pragma unroll
      for (int e = 0; e < C::W; ++e)
        orow[g * 16 * C::W + tx * C::W + e] =
            acc[a][g * C::W + e] + X[(a * (D / 16) + g * C::W + e) * kThreads + ltid];
  }
}

// ---------------------------------------------------------------------------
// naive passes 1 and 3 at d <= 64 with paired FMAs and 8 x 4 register tiles,
// the tile products of flash_f32x2_kernel (the softmax pass is shared):
//  * scores: a block of 128 threads per 64 x 64 score tile, Q (scaled) and K
//    row-major in shared memory, features paired; thread (tx, ty) owns rows
//    ty + 8 a and keys tx + 16 b;
//  * P V: per 64-row query tile two groups of 128 threads take the even and the
//    odd key tiles; each double-buffers its P tile (row-major, as pass 2 left
//    it) and V tile with cp.async (the next tile's copies issued once every
//    thread of the group is past the tile that last read that buffer), re-lays
//    V as key pairs and accumulates rows ty + 8 a, columns 32 g + 2 tx + e over
//    key pairs; group 0 adds group 1's sums at the end.
// ---------------------------------------------------------------------------
constexpr int kNx2Threads = 128;

template <int D>
__global__ void __launch_bounds__(kNx2Threads) naive_scores_x2_kernel(const float* __restrict__ Q,
                                                                       const float* __restrict__ K,
                                                                       float* __restrict__ Sc, int64_t N, int S,
                                                                       int causal, float scale) {
  static_assert(D == 32 || D == 64, "paired-FMA naive score pass: d = 32 and 64");
  constexpr int RT = 8;
  constexpr int LDQ = D + 4;
  extern __shared__ float4 smem4[];
  float* Qs = reinterpret_cast<float*>(smem4);  // [kBR][LDQ], scaled
  float* Ks = Qs + kBR * LDQ;                    // [kBC][LDQ]
  const int kt = blockIdx.x, qt = blockIdx.y;
  const int64_t n = blockIdx.z;
  if (causal && kt > qt) return;
  const int q0 = qt * kBR, k0 = kt * kBC;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const float* Qh = Q + n * S * D;
  const float* Kh = K + n * S * D;
  for (int f = tid; f < kBR * (D / 4); f += kNx2Threads) {  // coalesced 16-byte loads; rows >= S read as 0
    const int r = f / (D / 4), c4 = f % (D / 4);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
    if (q0 + r < S) x = ld4(Qh + (int64_t)(q0 + r) * D + 4 * c4);
    if (k0 + r < S) y = ld4(Kh + (int64_t)(k0 + r) * D + 4 * c4);
    *reinterpret_cast<float4*>(Qs + r * LDQ + 4 * c4) = make_float4(x.x * scale, x.y * scale, x.z * scale, x.w * scale);
    *reinterpret_cast<float4*>(Ks + r * LDQ + 4 * c4) = y;
  }
  __syncthreads();
  float2 s2[RT][4];
#pragma unroll
  for (int a = 0; a < RT; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) s2[a][b] = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < D; k += 4) {
    float4 kv[4], qv[RT];
#pragma unroll
    for (int b = 0; b < 4; ++b) kv[b] = ld4(Ks + (tx + 16 * b) * LDQ + k);
#pragma unroll
    for (int a = 0; a < RT; ++a) qv[a] = ld4(Qs + (ty + 8 * a) * LDQ + k);
#pragma unroll
    for (int a = 0; a < RT; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        s2[a][b] = __ffma2_rn(make_float2(qv[a].x, qv[a].y), make_float2(kv[b].x, kv[b].y), s2[a][b]);
#pragma unroll
    for (int a = 0; a < RT; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        s2[a][b] = __ffma2_rn(make_float2(qv[a].z, qv[a].w), make_float2(kv[b].z, kv[b].w), s2[a][b]);
  }
  float* Sh = Sc + n * (int64_t)S * S;
#pragma unroll
  for (int a = 0; a < RT; ++a) {
    const int row = q0 + ty + 8 * a;
    if (row >= S) continue;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int key = k0 + tx + 16 * b;
      if (key >= S) continue;
      Sh[(int64_t)row * S + key] = (causal && key > row) ? -INFINITY : s2[a][b].x + s2[a][b].y;
    }
  }
}

template <int D>
struct Nx2 {
  static constexpr int LDP = kBC + 16;   // P rows ty and ty + 1 16 banks apart
  static constexpr int G = D / 32;
  static constexpr int NO = 2 * G;
  static constexpr int PBUF = kBR * LDP;
  static constexpr int VBUF = kBC * D;
  static constexpr int GROUP = 2 * (PBUF + VBUF) + kBC * D;  // P + V x 2, Vp
  static constexpr int SMEM_FLOATS = 2 * GROUP;
};

template <int D>
__global__ void __launch_bounds__(2 * kNx2Threads, 1) naive_pv_x2_kernel(const float* __restrict__ Sc,
                                                                      const float* __restrict__ V,
                                                                      float* __restrict__ O, int64_t N, int S,
                                                                      int causal) {
  static_assert(D == 32 || D == 64, "paired-FMA naive P V pass: d = 32 and 64");
  using F = Nx2<D>;
  constexpr int RT = 8;
  extern __shared__ float4 smem4[];
  const int grp = threadIdx.x / kNx2Threads, ltid = threadIdx.x % kNx2Threads;
  float* B0 = reinterpret_cast<float*>(smem4) + grp * F::GROUP;  // buffer b: P at B0 + b (PBUF + VBUF), V after it
  float* Vp = B0 + 2 * (F::PBUF + F::VBUF);                      // [kBC / 2][2 D]
  const int ntiles = (S + kBR - 1) / kBR;
  const int64_t n = blockIdx.x % N;
  const int qt = ntiles - 1 - (int)(blockIdx.x / N);
  const int q0 = qt * kBR;
  const int tx = ltid & 15, ty = ltid >> 4;
  const float* Sh = Sc + n * (int64_t)S * S;
  const float* Vh = V + n * S * D;
  const bool vec16 = (S & 3) == 0;
  // cp.async copies of key tile kt: the P rows q0 .. q0 + 63 (row-major, keys
  // kt*64 ..) and the V rows; entries past S are zero-filled
  auto issue = [&](int kt, float* Pr, float* Vr) {
    const int k0 = kt * kBC;
    if (vec16) {
      for (int f = ltid; f < kBR * (kBC / 4); f += kNx2Threads) {
        const int r = f / (kBC / 4), c4 = f % (kBC / 4);
        const int row = q0 + r, col = k0 + 4 * c4;
        const bool ok = row < S && col < S;  // S % 4 == 0: a 4-key chunk is wholly in or out
        cp_async<16>(Pr + r * F::LDP + 4 * c4, Sh + (ok ? (int64_t)row * S + col : 0), ok);
      }
    } else {
      for (int f = ltid; f < kBR * kBC; f += kNx2Threads) {
        const int r = f / kBC, c = f % kBC;
        const int row = q0 + r, col = k0 + c;
        const bool ok = row < S && col < S;
        cp_async<4>(Pr + r * F::LDP + c, Sh + (ok ? (int64_t)row * S + col : 0), ok);
      }
    }
    for (int f = ltid; f < kBC * (D / 4); f += kNx2Threads) {
      const int r = f / (D / 4), c4 = f % (D / 4);
      const bool ok = k0 + r < S;
      cp_async<16>(Vr + r * D + 4 * c4, Vh + (int64_t)(ok ? k0 + r : 0) * D + 4 * c4, ok);
    }
    cp_async_commit();
  };
  auto pbuf = [&](int it) { return B0 + (it & 1) * (F::PBUF + F::VBUF); };

  float o[RT][F::NO];
#pragma unroll
  for (int a = 0; a < RT; ++a)
#pragma unroll
    for (int j = 0; j < F::NO; ++j) o[a][j] = 0.f;

  const int kt_last = causal ? qt : ntiles - 1;
  if (grp <= kt_last) issue(grp, pbuf(0), pbuf(0) + F::PBUF);
  for (int kt = grp, it = 0; kt <= kt_last; kt += 2, ++it) {
    float* Pr = pbuf(it);
    const float* Vs = Pr + F::PBUF;
    cp_async_wait<0>();  // this thread's copies of tile kt have landed
    fx2_group_bar(grp);  // everyone's have, and everyone finished the previous tile (its P, V and Vp)
    // tile kt + 2 into the other buffer pair, whose P the previous tile's P V read
    if (kt + 2 <= kt_last) issue(kt + 2, pbuf(it + 1), pbuf(it + 1) + F::PBUF);
    if (causal && kt == qt)  // the diagonal tile: keys after the row are masked (-inf from pass 1)
      for (int f = ltid; f < kBR * kBC; f += kNx2Threads) {
        const int r = f / kBC, c = f % kBC;
        if (c > r) Pr[r * F::LDP + c] = 0.f;
      }
    for (int w = ltid; w < (kBC / 2) * (D / 4); w += kNx2Threads) {  // V as key pairs
      const int kp = w / (D / 4), c4 = w % (D / 4);
      const float4 a = ld4(Vs + (2 * kp) * D + 4 * c4), b = ld4(Vs + (2 * kp + 1) * D + 4 * c4);
      const float4 lo = make_float4(a.x, b.x, a.y, b.y), hi = make_float4(a.z, b.z, a.w, b.w);
      float* dst = Vp + kp * 2 * D + 8 * c4;
      const int sw = ((c4 >> 2) & 1) * 4;
      st4(dst + sw, sw ? hi : lo);
      st4(dst + 4 - sw, sw ? lo : hi);
    }
    fx2_group_bar(grp);  // Vp and the masked P are visible to the group
    float2 acc[RT][F::NO];
#pragma unroll
    for (int a = 0; a < RT; ++a)
#pragma unroll
      for (int j = 0; j < F::NO; ++j) acc[a][j] = make_float2(0.f, 0.f);
#pragma unroll 2
    for (int c4 = 0; c4 < kBC / 4; ++c4) {
      float4 v[2][F::G];
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int g = 0; g < F::G; ++g) v[kk][g] = ld4(Vp + (2 * c4 + kk) * 2 * D + 64 * g + 4 * tx);
      float4 pv[RT];
#pragma unroll
      for (int a = 0; a < RT; ++a) pv[a] = ld4(Pr + (ty + 8 * a) * F::LDP + 4 * c4);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int a = 0; a < RT; ++a) {
          const float2 pp = kk == 0 ? make_float2(pv[a].x, pv[a].y) : make_float2(pv[a].z, pv[a].w);
#pragma unroll
          for (int g = 0; g < F::G; ++g) {
            acc[a][2 * g] = __ffma2_rn(pp, make_float2(v[kk][g].x, v[kk][g].y), acc[a][2 * g]);
            acc[a][2 * g + 1] = __ffma2_rn(pp, make_float2(v[kk][g].z, v[kk][g].w), acc[a][2 * g + 1]);
          }
        }
    }
#pragma unroll
    for (int a = 0; a < RT; ++a)
#pragma unroll
      for (int j = 0; j < F::NO; ++j) o[a][j] += acc[a][j].x + acc[a][j].y;
  }
  // group 0 adds group 1's sums (group 1's buffers hold them)
  float* X = reinterpret_cast<float*>(smem4) + F::GROUP;
  static_assert(RT * F::NO * kNx2Threads <= F::GROUP, "partial sums fit in one group's buffers");
  __syncthreads();
  if (grp == 1) {
#pragma unroll
    for (int a = 0; a < RT; ++a)
#pragma unroll
      for (int j = 0; j < F::NO; ++j) X[(a * F::NO + j) * kNx2Threads + ltid] = o[a][j];
  }
  __syncthreads();
  if (grp == 1) return;
#pragma unroll
  for (int a = 0; a < RT; ++a) {
    const int row = q0 + ty + 8 * a;
    if (row >= S) continue;
    float* orow = O + (n * S + row) * D;
#pragma unroll
    for (int g = 0; g < F::G; ++g)
      *reinterpret_cast<float2*>(orow + 32 * g + 2 * tx) =
          make_float2(o[a][2 * g] + X[(a * F::NO + 2 * g) * kNx2Threads + ltid],
                      o[a][2 * g + 1] + X[(a * F::NO + 2 * g + 1) * kNx2Threads + ltid]);
  }
}

// ---------------------------------------------------------------------------
// fused: the S-length score rows live in shared memory, one pass over the keys
// (kbench, "The three GPU kernels": one block per query row, shared memory
// O(S)). A block takes R consecutive query rows of one head (R = 4 where their
// R score rows fit in shared memory and the grid keeps two blocks per SM, else
// 2 or 1 -- R = 1 is the page's layout and sets the same S cap), so every K and
// V element read from L2 serves R rows. Key tiles of 64 keys, of K in the score
// pass and of V in the P V pass, are staged in two shared-memory buffers by
// cp.async, the next tile's copies in flight while the current one is used;
// each dot product is split over 4 threads, thread q of a key taking float4 q,
// q + 4, ...; K rows are padded by 16 floats so that the 8 threads of one
// 128-bit load phase (2 keys x 4 parts) touch 8 distinct bank groups. In the
// P V pass a thread takes one output column and every G-th quad of keys, the
// four weights of a quad read with one 16-byte load per row.
// Masked keys (past a row's causal limit) hold -inf, so every row of the block
// runs over the same key range and gets probability 0 there.
// ---------------------------------------------------------------------------
constexpr int kFusedThreads = 256;
constexpr int kFusedKeys = 64;  // keys per staged tile
constexpr int kFusedWarps = kFusedThreads / 32;

// Per-row maxima (MAX) or sums over the block for R values per thread; every
// thread receives the results. Uses red[kFusedWarps * R]; contains barriers.
template <int R, bool MAX>
__device__ __forceinline__ void block_rows(float (&v)[R], float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float x = v[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float y = __shfl_xor_sync(0xffffffffu, x, o);
      x = MAX ? fmaxf(x, y) : x + y;
    }
    if (lane == 0) red[warp * R + r] = x;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float x = red[r];
#pragma unroll
    for (int w = 1; w < kFusedWarps; ++w) x = MAX ? fmaxf(x, red[w * R + r]) : x + red[w * R + r];
    v[r] = x;
  }
  __syncthreads();  // red may be reused
}

template <int D, int R>
__global__ void __launch_bounds__(kFusedThreads) fused_row_f32_kernel(const float* __restrict__ Q,
                                                                      const float* __restrict__ K,
                                                                      const float* __restrict__ V,
                                                                      float* __restrict__ O, int S, int causal,
                                                                      float scale_log2) {
  constexpr int LDK = D + 16;
  constexpr int G = kFusedThreads / D;  // key groups of the P V pass
  constexpr int QUADS = kFusedKeys / 4;  // key quads of a tile
  static_assert(QUADS % G == 0, "the key quads of a tile split evenly over the key groups");
  extern __shared__ float4 smem4[];
  float* buf = reinterpret_cast<float*>(smem4);  // two tile buffers: K [kFusedKeys][LDK], later V [kFusedKeys][D]
  float* qs = buf + 2 * kFusedKeys * LDK;        // [R][D]
  float* red = qs + R * D;                       // [kFusedWarps * R]
  float* part = red + kFusedWarps * R;           // [R][kFusedThreads]
  float* sc = part + R * kFusedThreads;          // [R][SP]
  const int SP = (S + 3) & ~3;                   // score row stride: 16-byte aligned rows
  const int tiles = (S + R - 1) / R;
  // heads interleaved, the last (causal: heaviest) row tiles first
  const int64_t nheads = gridDim.x / tiles;
  const int64_t n = blockIdx.x % nheads;
  const int i0 = (tiles - 1 - (int)(blockIdx.x / nheads)) * R;
  const int tid = threadIdx.x;
  const int last_block = causal ? min(i0 + R - 1, S - 1) : S - 1;  // keys any row of the block sees
  const int nt = last_block / kFusedKeys + 1;                       // key tiles
  const float* Kh = K + n * S * D;
  const float* Vh = V + n * S * D;
  auto tile_buf = [&](int b) { return buf + (b & 1) * kFusedKeys * LDK; };
  // cp.async copies of key tile t of K or V (row stride ld) into dst; rows past
  // last_block are zero-filled and read nothing
  auto issue = [&](const float* src, int ld, int t, float* dst) {
    const int k0 = t * kFusedKeys;
    for (int f = tid; f < kFusedKeys * (D / 4); f += kFusedThreads) {
      const int r = f / (D / 4), c4 = f % (D / 4);
      const bool ok = k0 + r <= last_block;
      cp_async<16>(dst + r * ld + 4 * c4, src + (int64_t)(ok ? k0 + r : 0) * D + 4 * c4, ok);
    }
    cp_async_commit();
  };

  issue(Kh, LDK, 0, tile_buf(0));
  for (int f = tid; f < R * D; f += kFusedThreads) {
    const int r = f / D, c = f % D;
    qs[f] = i0 + r < S ? Q[(n * S + i0 + r) * D + c] * scale_log2 : 0.f;
  }

  // scores: thread tid works on key tid / 4 of the tile, float4 (tid % 4) + 4 t, for all R rows;
  // the next K tile's copies are in flight while the current one is used
  const int kl = tid >> 2, qp = tid & 3;
  float tmax[R];
#pragma unroll
  for (int r = 0; r < R; ++r) tmax[r] = -INFINITY;
  for (int t = 0; t < nt; ++t) {
    cp_async_wait<0>();  // this thread's copies of tile t have landed
    __syncthreads();     // everyone's have (and qs is written); tile t - 1 is no longer read
    if (t + 1 < nt) issue(Kh, LDK, t + 1, tile_buf(t + 1));
    const float* Ks = tile_buf(t);
    float dot[R];
#pragma unroll
    for (int r = 0; r < R; ++r) dot[r] = 0.f;
#pragma unroll
    for (int c = 4 * qp; c < D; c += 16) {
      const float4 kv = ld4(Ks + kl * LDK + c);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float4 qv = ld4(qs + r * D + c);
        dot[r] = fmaf(qv.x, kv.x, dot[r]);
        dot[r] = fmaf(qv.y, kv.y, dot[r]);
        dot[r] = fmaf(qv.z, kv.z, dot[r]);
        dot[r] = fmaf(qv.w, kv.w, dot[r]);
      }
    }
    const int key = t * kFusedKeys + kl;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float x = dot[r];
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      const int last_r = causal ? min(i0 + r, S - 1) : S - 1;
      if (qp == 0 && key <= last_block) {
        const float sv = key <= last_r ? x : -INFINITY;
        sc[r * SP + key] = sv;
        tmax[r] = fmaxf(tmax[r], sv);
      }
    }
  }
  // the first V tile into the buffer the last K tile does not occupy (every
  // thread passed the barrier after its last read of that buffer)
  issue(Vh, D, 0, tile_buf(nt));
  block_rows<R, true>(tmax, red);  // its barriers also publish sc[]
  // weights; the up to three entries past last_block that its last key quad
  // spans are set to 0 (never written above, and their V rows are zero-filled)
  const int jend = (last_block + 4) & ~3;  // <= SP
  float tsum[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    tsum[r] = 0.f;
    for (int j = tid; j < jend; j += kFusedThreads) {
      const float p = j <= last_block ? exp2f(sc[r * SP + j] - tmax[r]) : 0.f;
      sc[r * SP + j] = p;
      tsum[r] += p;
    }
  }
  block_rows<R, false>(tsum, red);  // its barriers also publish the new sc[]

  // O = P V: thread (c, g) takes column c and the key quads g, g + G, ... of every
  // tile (a warp shares g, so its weight loads are broadcasts); V tiles are
  // double-buffered like K
  const int c = tid % D, g = tid / D;
  float acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = 0.f;
  for (int t = 0; t < nt; ++t) {
    cp_async_wait<0>();
    __syncthreads();
    if (t + 1 < nt) issue(Vh, D, t + 1, tile_buf(nt + t + 1));
    const float* Vs = tile_buf(nt + t);
    const int k0 = t * kFusedKeys;
#pragma unroll
    for (int qd = g; qd < QUADS; qd += G) {
      if (k0 + 4 * qd > last_block) break;
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = Vs[(4 * qd + i) * D + c];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float4 p = ld4(sc + r * SP + k0 + 4 * qd);
        acc[r] = fmaf(p.x, v[0], acc[r]);
        acc[r] = fmaf(p.y, v[1], acc[r]);
        acc[r] = fmaf(p.z, v[2], acc[r]);
        acc[r] = fmaf(p.w, v[3], acc[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) part[r * kFusedThreads + tid] = acc[r];
  if (tid == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r) red[r] = tsum[r];  // row sums, indexed by a runtime row below
  }
  __syncthreads();
  for (int f = tid; f < R * D; f += kFusedThreads) {
    const int r = f / D, cc = f % D;
    if (i0 + r >= S) continue;
    float t = 0.f;
#pragma unroll
    for (int gg = 0; gg < G; ++gg) t += part[r * kFusedThreads + gg * D + cc];
    O[(n * S + i0 + r) * D + cc] = t / red[r];
  }
}

size_t flash_smem(int d) {
  if (d == 32) return sizeof(float) * (size_t)Fx2<32>::SMEM_FLOATS;
  if (d == 64) return sizeof(float) * (size_t)Fx2<64>::SMEM_FLOATS;
  return sizeof(float) * (size_t)(d * kLD + 2 * flash_group_floats<128>());
}
size_t naive_scores_smem(int d) { return sizeof(float) * (size_t)(d * kLD + kBC * (d + 4)); }
size_t naive_pv_smem(int d) { return sizeof(float) * (size_t)(2 * 2 * (kBR * kLDP + kBC * d)); }
size_t fused_smem(int S, int d, int rows = 1) {
  return sizeof(float) * (size_t)(2 * kFusedKeys * (d + 16) + rows * d + kFusedWarps * rows + rows * kFusedThreads +
                                  (size_t)rows * (size_t)((S + 3) & ~3));
}

template <typename F>
cudaError_t set_smem(F* kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// d <= 64: the paired-FMA kernel; d = 128: flash_f32_kernel (its two groups'
// single-buffered K/V tiles and the re-laid V would not fit beside each other).
template <int D, typename Kernel>
cudaError_t flash_launch(Kernel kernel, int threads, const AttnProblem& p, cudaStream_t st) {
  const size_t smem = flash_smem(D);
  cudaError_t e = set_smem(kernel, smem);
  if (e != cudaSuccess) return e;
  const int tiles = (p.S + kBR - 1) / kBR;
  const int split_from = p.work ? (tiles + 1) / 2 : tiles;
  const int nsplit = tiles - split_from;
  kernel<<<(unsigned)((tiles + nsplit) * p.N), threads, smem, st>>>(
      (const float*)p.q, (const float*)p.k, (const float*)p.v, (float*)p.o, p.lse, p.N, p.S, p.causal,
      p.scale * kLog2e, p.work, split_from);
  if (nsplit > 0 && (e = cudaGetLastError()) == cudaSuccess)
    flash_merge_kernel<D><<<(unsigned)(nsplit * p.N), 256, 0, st>>>(p.work, (float*)p.o, p.lse, p.S, nsplit);
  return cudaGetLastError();
}

template <int D>
cudaError_t flash_launch(const AttnProblem& p, cudaStream_t st) {
  if constexpr (D <= 64)
    return flash_launch<D>(flash_f32x2_kernel<D>, kFx2Threads, p, st);
  else
    return flash_launch<D>(flash_f32_kernel<D>, kFlashThreads, p, st);
}

// d <= 64: the paired-FMA score and P V passes; d = 128: the scalar ones.
template <int D>
cudaError_t naive_launch(const AttnProblem& p, float* scores, cudaStream_t st) {
  constexpr bool X2 = D <= 64;
  constexpr int XD = X2 ? D : 64;  // keeps the paired kernels' templates instantiable at d = 128
  const size_t sc_smem = X2 ? sizeof(float) * (size_t)(2 * kBR * (D + 4)) : naive_scores_smem(D);
  const size_t pv_smem = X2 ? sizeof(float) * (size_t)Nx2<XD>::SMEM_FLOATS : naive_pv_smem(D);
  cudaError_t e = X2 ? set_smem(naive_scores_x2_kernel<XD>, sc_smem) : set_smem(naive_scores_kernel<D>, sc_smem);
  if (e == cudaSuccess)
    e = X2 ? set_smem(naive_pv_x2_kernel<XD>, pv_smem) : set_smem(naive_pv_kernel<D>, pv_smem);
  if (e != cudaSuccess) return e;
  const int tiles = (p.S + kBR - 1) / kBR;
  if constexpr (X2)
    naive_scores_x2_kernel<XD><<<dim3(tiles, tiles, (unsigned)p.N), kNx2Threads, sc_smem, st>>>(
        (const float*)p.q, (const float*)p.k, scores, p.N, p.S, p.causal, p.scale);
  else
    naive_scores_kernel<D><<<dim3(tiles, tiles, (unsigned)p.N), kThreads, sc_smem, st>>>(
        (const float*)p.q, (const float*)p.k, scores, p.N, p.S, p.causal, p.scale);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t rows = p.N * p.S;
  naive_softmax_kernel<<<(unsigned)((rows + kThreads / 32 - 1) / (kThreads / 32)), kThreads, 0, st>>>(
      scores, rows, p.S, p.causal);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if constexpr (X2)
    naive_pv_x2_kernel<XD><<<(unsigned)(tiles * p.N), 2 * kNx2Threads, pv_smem, st>>>(
        scores, (const float*)p.v, (float*)p.o, p.N, p.S, p.causal);
  else
    naive_pv_kernel<D><<<(unsigned)(tiles * p.N), kFlashThreads, pv_smem, st>>>(
        scores, (const float*)p.v, (float*)p.o, p.N, p.S, p.causal);
  return cudaGetLastError();
}

template <int D, int R>
cudaError_t fused_launch_rows(const AttnProblem& p, size_t smem, cudaStream_t st) {
  cudaError_t e = set_smem(fused_row_f32_kernel<D, R>, smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = p.N * ((p.S + R - 1) / R);
  fused_row_f32_kernel<D, R><<<(unsigned)blocks, kFusedThreads, smem, st>>>(
      (const float*)p.q, (const float*)p.k, (const float*)p.v, (float*)p.o, p.S, p.causal, p.scale * kLog2e);
  return cudaGetLastError();
}

// R = 8 query rows per block where two such blocks fit in one SM's shared
// memory (each K or V element then serves 8 rows; measured faster than R = 4
// up to S = 1024 at d = 64, slower at S = 2048 where only one fits), else R = 4
// where the block fits, else 2, else 1; the grid keeps at least two blocks per SM.
template <int D>
cudaError_t fused_launch(const AttnProblem& p, cudaStream_t st) {
  int dev = 0, optin = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e != cudaSuccess) return e;
  const int64_t rows = p.N * p.S;
  auto fits = [&](int r) { return fused_smem(p.S, D, r) <= (size_t)optin && rows / r >= 2 * (int64_t)sms; };
  // 1 KB of each block's shared memory is reserved by the system
  if (fits(8) && 2 * (fused_smem(p.S, D, 8) + 1024) <= (size_t)per_sm)
    return fused_launch_rows<D, 8>(p, fused_smem(p.S, D, 8), st);
  if (fits(4)) return fused_launch_rows<D, 4>(p, fused_smem(p.S, D, 4), st);
  if (fits(2)) return fused_launch_rows<D, 2>(p, fused_smem(p.S, D, 2), st);
  return fused_launch_rows<D, 1>(p, fused_smem(p.S, D, 1), st);
}

}  // namespace

cudaError_t launch_flash_f32(const AttnProblem& p, cudaStream_t st) {
  switch (p.d) {
    case 32: return flash_launch<32>(p, st);
    case 64: return flash_launch<64>(p, st);
    case 128: return flash_launch<128>(p, st);
  }
  return cudaErrorInvalidValue;
}

size_t naive_workspace_bytes(int64_t N, int S) { return (size_t)N * (size_t)S * (size_t)S * sizeof(float); }

bool flash_wants_split(int64_t N, int S, int causal) {
  const int tiles = (S + kBR - 1) / kBR;
  if (!causal || tiles < 4) return false;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return N * tiles <= 2 * (int64_t)sms;
}

size_t flash_split_bytes(int64_t N, int S, int d) {
  const int tiles = (S + kBR - 1) / kBR;
  const int nsplit = tiles - (tiles + 1) / 2;
  return (size_t)N * (size_t)nsplit * 2 * kBR * (size_t)(d + 2) * sizeof(float);
}

cudaError_t launch_naive_f32(const AttnProblem& p, float* scores, cudaStream_t st) {
  switch (p.d) {
    case 32: return naive_launch<32>(p, scores, st);
    case 64: return naive_launch<64>(p, scores, st);
    case 128: return naive_launch<128>(p, scores, st);
  }
  return cudaErrorInvalidValue;
}

int fused_f32_check(int S, int d) {
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KB_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return KB_ERR_CUDA;
  return fused_smem(S, d) <= (size_t)optin ? KB_OK : KB_ERR_UNSUPPORTED;
}

cudaError_t launch_fused_f32(const AttnProblem& p, cudaStream_t st) {
  switch (p.d) {
    case 32: return fused_launch<32>(p, st);
    case 64: return fused_launch<64>(p, st);
    case 128: return fused_launch<128>(p, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kb
