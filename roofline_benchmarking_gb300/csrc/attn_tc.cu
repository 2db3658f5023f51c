// attn_tc.cu -- attention forward on the sm_103a tensor cores (bf16 / f16).
//
// The algorithm is the tiled online softmax of the kbench page ("kbench --
// Transformer Attention Micro-benchmark Harness", section "Implementation
// details / The three GPU kernels", the flash kernel: keys and values stream
// through in tiles, a running max m and denominator l are kept per query row,
// the score matrix is never materialised). It is laid out for GB300:
//
//  * a work item is a pair of 128-row query tiles A and B of one head; the two
//    tiles share every K and V tile loaded for them. The grid is persistent
//    (at most one CTA per SM): items are sorted heaviest first (causal) and
//    dealt to the CTAs in a snake order. Within a CTA the next item's Q load
//    starts as soon as the current item's last score MMA has completed, and
//    its first P V waits only for the current epilogue to have read O;
//  * warp 8 (one lane) stages both Q tiles and rings of K and V tiles with TMA
//    (128-byte swizzle, 3-D tensor maps [N, S, d], rows past S zero-filled);
//  * warp 9 issues the tcgen05 MMAs, the whole warp running the issue loop and
//    one elected lane issuing each instruction: S = Q K^T from shared memory
//    into a 128x128 fp32 TMEM tile per query tile, and O += P V with P read
//    from TMEM and V from shared memory into a 128 x d fp32 TMEM accumulator
//    per query tile; completion is signalled by tcgen05.commit on mbarriers;
//  * warps 0-3 (tile A) and 4-7 (tile B) own one query row per thread (TMEM
//    lane = row): they load the score row from TMEM, apply scale and the
//    causal/tail masks, update the running max in base 2 (scale*log2(e) in one
//    FMA), write P = exp2(s - m) as 16-bit pairs back into the first 64 columns
//    of the score tile, and rescale O in TMEM only when the row max grew by
//    more than 8 (factor 256; the final O / l is exact either way);
//  * the MMA order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1) keeps the tensor core on
//    one tile while the other tile's softmax runs. S_A(j+1) overwrites P_A(j)
//    only after PV_A(j) has read it: MMAs issued by one thread execute in order.
// Every mbarrier wait is bounded by %globaltimer; a wait that runs out sets the
// library's device error word and an abort flag, every role then leaves its
// loop, waits (bounded) for its own TMA copies and MMAs in flight, and the
// tensor memory is released before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <functional>
#include <map>
#include <memory>
#include <mutex>
#include <queue>
#include <tuple>
#include <utility>
#include <vector>

#include "internal.h"
#include "tc_ptx.cuh"

namespace kb {

// Device error word: bit 0 = a bounded wait ran out.
__device__ unsigned int g_kb_error_word;

namespace {

constexpr int kBM = 128;  // query rows per tile (TMEM lanes)
constexpr int kBN = 128;  // keys per tile
constexpr int kPairRows = 2 * kBM;
// Three warpgroups: 0 and 1 run the softmax of tiles A and B; in the third,
// warp 8 drives TMA and warp 9 issues MMAs (warps 10 and 11 only hand their
// registers over). Launch budget 384 x 168 = 64512 registers, rebalanced as
// 2 x 128 x 200 + 128 x 104 = 64512.
constexpr int kThreadsTC = 384;
constexpr int kWarpTMA = 8;
constexpr int kWarpMMA = 9;
constexpr int kRegsSoftmax = 200;
constexpr int kRegsControl = 104;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColBlock = 16384;  // one 128-row x 128-byte swizzled block
constexpr unsigned long long kDefaultWaitLimitNs = 1000000000ull;

template <int D>
struct TcCfg {
  static_assert(D == 64 || D == 128, "tensor-core path supports d = 64 and 128");
  static constexpr int DB = D / 64;           // 128-byte column blocks per tile row
  static constexpr int TILE = kBM * D * 2;    // bytes of a Q, K or V tile
  static constexpr int KS = D == 128 ? 2 : 3;  // K ring stages
  static constexpr int VS = D == 128 ? 2 : 3;  // V ring stages
  static constexpr int OFF_Q = 0;              // Q_A then Q_B
  static constexpr int OFF_K = OFF_Q + 2 * TILE;
  static constexpr int OFF_V = OFF_K + KS * TILE;
  // d = 128: output staging of the eight softmax warps, 32 rows x 64 columns each,
  // in the 128-byte swizzled layout of the output tensor map's boxes (TMA stores).
  // d = 64 stores O from registers (measured faster there: its smaller K/V loads
  // come more often and would share the TMA unit with the stores).
  static constexpr bool TMA_STORE = D == 128;
  static constexpr int STG = 32 * 64 * 2;
  static constexpr int OFF_O = OFF_V + VS * TILE;
  static constexpr int OFF_BAR = OFF_O + (TMA_STORE ? 8 * STG : 0);
  enum {
    B_Q = 0,
    B_KFULL = 1,
    B_KEMPTY = B_KFULL + KS,
    B_VFULL = B_KEMPTY + KS,
    B_VEMPTY = B_VFULL + VS,
    B_SFULL = B_VEMPTY + VS,  // [2]: S of tile A / B computed
    B_PFULL = B_SFULL + 2,    // [2]: P of tile A / B written (and O rescaled)
    B_OFINAL = B_PFULL + 2,   // [2]: last P V of tile A / B of an item done
    B_OFREE = B_OFINAL + 2,   // [2]: O of tile A / B read out by the epilogue
    B_QFREE = B_OFREE + 2,    // last score MMA of an item done: Q may be replaced
    B_DRAIN = B_QFREE + 1,
    NBAR = B_DRAIN + 1
  };
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int SMEM = BYTES + 1024;  // slack to align the base to 1024 bytes
  static_assert(SMEM <= 232448, "at most 227 KB of shared memory per CTA");
  // TMEM columns of tile g: S (and P in its first 64 columns) at 128 g, O at 256 + 128 g.
  __host__ __device__ static constexpr uint32_t tm_s(int g) { return 128u * (uint32_t)g; }
  __host__ __device__ static constexpr uint32_t tm_o(int g) { return 256u + 128u * (uint32_t)g; }
};

// Bounded wait on phase `parity` of `bar`. Gives up when the abort flag is set
// (if `honor_abort`) or after `limit` ns, recording the timeout.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                      unsigned long long limit, bool honor_abort) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *abort_flag) return false;
    if (ptx::globaltimer() - t0 > limit) {
      *abort_flag = 1;
      atomicOr(&g_kb_error_word, 1u);
      return false;
    }
  }
}

// All lanes wait; the warp proceeds only if every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long limit) {
  const bool ok = wait_bar(bar, parity, abort_flag, limit, true);
  return __all_sync(0xffffffffu, ok);
}

// Warp-wide wait that can ignore the abort flag (used to drain copies and MMAs in flight).
__device__ __forceinline__ bool warp_wait_all(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned long long limit, bool honor_abort) {
  const bool ok = wait_bar(bar, parity, abort_flag, limit, honor_abort);
  return __all_sync(0xffffffffu, ok);
}

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// A weight as the P V MMA sees it: p rounded to 16 bits (the packing's
// round-to-nearest-even), widened back to fp32.
template <bool F16>
__device__ __forceinline__ float rounded16(float p) {
  const uint32_t w = pack2<F16>(p, 0.f);
  if constexpr (F16) {
    return __low2float(*reinterpret_cast<const __half2*>(&w));
  } else {
    return __uint_as_float(w << 16);
  }
}

// Sixteen fp32 values of one O row, times inv, rounded to 16 bits and stored at
// dst: one 32-byte store (a whole L2 sector) when the output base is 32-byte
// aligned (st32; every row and chunk offset is a multiple of 32 bytes), else two
// 16-byte stores.
template <bool F16>
__device__ __forceinline__ void store_o16(uint8_t* dst, const uint32_t* u, float inv, bool st32) {
  uint32_t w[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) w[e] = pack2<F16>(__uint_as_float(u[2 * e]) * inv, __uint_as_float(u[2 * e + 1]) * inv);
  if (st32) {
    ptx::st_global_v8(dst, w);
  } else {
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// Per-CTA work lists built on the host (passed by value as a kernel parameter):
// CTA c runs units item[start[c]], item[start[c] + 1], ... < start[c + 1], an
// entry holding head << 16 | unit. The lists come from list scheduling over
// the heads in groups whose K and V fit in L2 (each group's units heaviest
// first): the CTAs work on one group's heads at a time, so every K/V tile is
// fetched from DRAM about once and shared in L2 by all the units of its head,
// while the per-CTA totals stay within a few per cent of each other. count = 0
// (more units than the table holds) selects the snake order below.
constexpr int kSchedMaxGrid = 256;
constexpr int kSchedMaxItems = 4096;
struct SchedTable {
  int count;
  unsigned short start[kSchedMaxGrid + 1];
  unsigned int item[kSchedMaxItems];
};

// Snake order (the fallback). Work item i (0 <= i < N * pairs) is query rows
// [256 t, 256 t + 256) of head n with t = pairs - 1 - i / N, so the heaviest
// causal items come first. CTA c takes, in round r, item r G + c when r is
// even and item r G + G - 1 - c when r is odd: a snake over the list sorted
// by cost keeps the per-CTA totals within a few per cent of each other.
struct Item {
  int n, t, q0, nA, nB;  // head, pair, first row, key tiles of tile A and of tile B
};

struct Schedule {
  int N, S, causal, pairs, nkv, total;
  const SchedTable* tab;
  __device__ Schedule(int N_, int S_, int causal_, const SchedTable* tab_)
      : N(N_), S(S_), causal(causal_), tab(tab_) {
    pairs = (S + kPairRows - 1) / kPairRows;
    nkv = (S + kBN - 1) / kBN;
    total = N * pairs;
  }
  // Item of this CTA's round `round`; false once the list is exhausted (the
  // index grows with the round, so every later round is exhausted too).
  __device__ bool get(int round, Item& it) const {
    const int c = (int)blockIdx.x;
    if (tab->count > 0) {
      const int k = (int)tab->start[c] + round;
      if (k >= (int)tab->start[c + 1]) return false;
      const unsigned int e = tab->item[k];
      it.n = (int)(e >> 16);
      it.t = (int)(e & 0xFFFFu);
    } else {
      const int G = (int)gridDim.x;
      const int i = round * G + ((round & 1) ? G - 1 - c : c);
      if (i >= total) return false;
      it.n = i % N;
      it.t = pairs - 1 - i / N;
    }
    it.q0 = it.t * kPairRows;
    it.nA = causal ? min(2 * it.t + 1, nkv) : nkv;
    it.nB = causal ? min(2 * it.t + 2, nkv) : nkv;  // never shorter than nA
    return true;
  }
};

template <int D, bool F16>
__global__ void __launch_bounds__(kThreadsTC, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                   const __grid_constant__ SchedTable tab,
                   uint8_t* __restrict__ out, float* __restrict__ lse, int dout, int N, int S, int causal,
                   float scale_log2, unsigned long long limit) {
  // dout: output columns per row (D, or 32 when a d = 32 problem runs on the 64-wide kernel
  // with its tiles zero-filled by TMA past column 32)
  using C = TcCfg<D>;
  constexpr uint32_t kAB = F16 ? 0u : 1u;
  constexpr uint32_t IDESC_QK = ptx::f16_idesc(kBM, kBN, kAB, 0);
  constexpr uint32_t IDESC_PV = ptx::f16_idesc(kBM, D, kAB, 1);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 4);
  auto bar = [&](int i) -> uint32_t { return base + C::OFF_BAR + 8u * (uint32_t)i; };

  const Schedule sched(N, S, causal, &tab);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    ptx::mbar_init(bar(C::B_Q), 1);
    for (int s = 0; s < C::KS; ++s) {
      ptx::mbar_init(bar(C::B_KFULL + s), 1);
      ptx::mbar_init(bar(C::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < C::VS; ++s) {
      ptx::mbar_init(bar(C::B_VFULL + s), 1);
      ptx::mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    for (int g = 0; g < 2; ++g) {
      ptx::mbar_init(bar(C::B_SFULL + g), 1);
      ptx::mbar_init(bar(C::B_PFULL + g), 4 * 32);
      ptx::mbar_init(bar(C::B_OFINAL + g), 1);
      ptx::mbar_init(bar(C::B_OFREE + g), 4 * 32);
    }
    ptx::mbar_init(bar(C::B_QFREE), 1);
    ptx::mbar_init(bar(C::B_DRAIN), 1);
    ptx::fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    ptx::tmem_alloc(base + C::OFF_MISC, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + C::OFF_MISC);

  if (warp >= kWarpTMA) {
    ptx::regs_decrease<kRegsControl>();
    if (warp == kWarpTMA) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        ptx::tma_prefetch_desc(&tmq);
        ptx::tma_prefetch_desc(&tmk);
        ptx::tma_prefetch_desc(&tmv);
        ptx::tma_prefetch_desc(&tmo);
        int kdone = 0, vdone = 0, items = 0;  // K tiles, V tiles and items whose loads were issued
        bool ok = true;
        Item it;
        for (int round = 0; ok && sched.get(round, it); ++round) {
          // Q of both tiles, once the previous item's last score MMA has read the old Q
          if (items > 0) ok = wait_bar(bar(C::B_QFREE), (items - 1) & 1, abort_flag, limit, true);
          if (!ok) break;
          ptx::mbar_arrive_expect_tx(bar(C::B_Q), 2 * C::TILE);
          for (int g = 0; g < 2; ++g)
            for (int b = 0; b < C::DB; ++b)
              ptx::tma_load_3d(base + C::OFF_Q + g * C::TILE + b * kColBlock, &tmq, bar(C::B_Q), b * 64,
                               it.q0 + g * kBM, it.n);
          for (int j = 0; j < it.nB && ok; ++j) {
            const int ks = kdone % C::KS, vs = vdone % C::VS;
            if (kdone >= C::KS) ok = wait_bar(bar(C::B_KEMPTY + ks), ((kdone / C::KS) & 1) ^ 1, abort_flag, limit, true);
            if (!ok) break;
            ptx::mbar_arrive_expect_tx(bar(C::B_KFULL + ks), C::TILE);
            for (int b = 0; b < C::DB; ++b)
              ptx::tma_load_3d(base + C::OFF_K + ks * C::TILE + b * kColBlock, &tmk, bar(C::B_KFULL + ks), b * 64,
                               j * kBN, it.n);
            ++kdone;
            if (vdone >= C::VS) ok = wait_bar(bar(C::B_VEMPTY + vs), ((vdone / C::VS) & 1) ^ 1, abort_flag, limit, true);
            if (!ok) break;
            ptx::mbar_arrive_expect_tx(bar(C::B_VFULL + vs), C::TILE);
            for (int b = 0; b < C::DB; ++b)
              ptx::tma_load_3d(base + C::OFF_V + vs * C::TILE + b * kColBlock, &tmv, bar(C::B_VFULL + vs), b * 64,
                               j * kBN, it.n);
            ++vdone;
          }
          ++items;
        }
        // Every copy this CTA started must land before the CTA exits.
        if (items > 0) wait_bar(bar(C::B_Q), (items - 1) & 1, abort_flag, limit, false);
        for (int x = kdone - C::KS < 0 ? 0 : kdone - C::KS; x < kdone; ++x)
          wait_bar(bar(C::B_KFULL + x % C::KS), (x / C::KS) & 1, abort_flag, limit, false);
        for (int x = vdone - C::VS < 0 ? 0 : vdone - C::VS; x < vdone; ++x)
          wait_bar(bar(C::B_VFULL + x % C::VS), (x / C::VS) & 1, abort_flag, limit, false);
      }
      __syncwarp();
    } else if (warp == kWarpMMA) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs the issue loop (descriptors and waits are warp-uniform);
      // one elected lane issues each MMA and commit.
      {
        // S_g = Q_g K_j^T (K-major operands, both from shared memory)
        auto issue_s = [&](int g, int ks) {
          // descriptors of k-step 0; a k-step moves the start address field (bytes >> 4)
          const uint64_t a0 = ptx::sw128_desc(base + C::OFF_Q + g * C::TILE, 16, 1024);
          const uint64_t b0 = ptx::sw128_desc(base + C::OFF_K + ks * C::TILE, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * kColBlock + (kk & 3) * 32) >> 4;
            ptx::mma_f16_ss_elect(tmem + C::tm_s(g), a0 + off, b0 + off, IDESC_QK, kk > 0 ? 1u : 0u);
          }
          ptx::mma_commit_elect(bar(C::B_SFULL + g));
        };
        // O_g += P_g V_j (P from TMEM, V MN-major from shared memory)
        auto issue_pv = [&](int g, int vs, bool first) {
          const uint64_t b0 = ptx::sw128_desc(base + C::OFF_V + vs * C::TILE, kColBlock, 1024);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)  // a k-step is 16 keys = 16 rows of 128 bytes
            ptx::mma_f16_ts_elect(tmem + C::tm_o(g), tmem + C::tm_s(g) + kk * 8, b0 + ((kk * 16 * 128) >> 4), IDESC_PV,
                            (!first || kk > 0) ? 1u : 0u);
        };
        bool ok = true;
        int kbase = 0, vbase = 0;  // ring positions of the current item's first K and V tiles
        int pa = 0, pb = 0;        // P tiles of tile A and of tile B consumed
        Item it;
        for (int item = 0; ok && sched.get(item, it); ++item) {
          const int nA = it.nA, nB = it.nB;
          ok = warp_wait(bar(C::B_Q), item & 1, abort_flag, limit);
          const int ks0 = kbase % C::KS;
          if (ok) ok = warp_wait(bar(C::B_KFULL + ks0), (kbase / C::KS) & 1, abort_flag, limit);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_s(0, ks0);
          issue_s(1, ks0);
          ptx::mma_commit_elect(bar(C::B_KEMPTY + ks0));
          if (nB == 1) ptx::mma_commit_elect(bar(C::B_QFREE));
          for (int j = 0; j < nB && ok; ++j) {
            const int vp = vbase + j, vs = vp % C::VS;
            const int jn = j + 1, kpn = kbase + jn, ksn = kpn % C::KS;
            ok = warp_wait(bar(C::B_VFULL + vs), (vp / C::VS) & 1, abort_flag, limit);
            if (ok && j < nA) {  // tile A
              ok = warp_wait(bar(C::B_PFULL + 0), pa & 1, abort_flag, limit);
              if (ok && j == 0 && item > 0) ok = warp_wait(bar(C::B_OFREE + 0), (item - 1) & 1, abort_flag, limit);
              if (ok) {
                ++pa;
                ptx::tc_fence_after();
                issue_pv(0, vs, j == 0);
                if (jn < nA) {
                  ok = warp_wait(bar(C::B_KFULL + ksn), (kpn / C::KS) & 1, abort_flag, limit);
                  if (ok) {
                    ptx::tc_fence_after();
                    issue_s(0, ksn);
                  }
                } else {
                  ptx::mma_commit_elect(bar(C::B_OFINAL + 0));
                }
              }
            }
            if (ok) ok = warp_wait(bar(C::B_PFULL + 1), pb & 1, abort_flag, limit);
            if (ok && j == 0 && item > 0) ok = warp_wait(bar(C::B_OFREE + 1), (item - 1) & 1, abort_flag, limit);
            if (!ok) break;
            ++pb;
            ptx::tc_fence_after();
            issue_pv(1, vs, j == 0);  // tile B
            ptx::mma_commit_elect(bar(C::B_VEMPTY + vs));
            if (jn < nB) {
              ok = warp_wait(bar(C::B_KFULL + ksn), (kpn / C::KS) & 1, abort_flag, limit);
              if (!ok) break;
              ptx::tc_fence_after();
              issue_s(1, ksn);
              ptx::mma_commit_elect(bar(C::B_KEMPTY + ksn));
              if (jn == nB - 1) ptx::mma_commit_elect(bar(C::B_QFREE));  // the item's last score MMA
            } else {
              ptx::mma_commit_elect(bar(C::B_OFINAL + 1));
            }
          }
          kbase += nB;
          vbase += nB;
        }
        // No MMA may still be running when the tensor memory is released.
        ptx::mma_commit_elect(bar(C::B_DRAIN));
        warp_wait_all(bar(C::B_DRAIN), 0, abort_flag, limit, false);
      }
    }
  } else {
    ptx::regs_increase<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax, warps 0-7
    const int g = warp >> 2;  // query tile of this warpgroup
    const int wq = warp & 3;  // TMEM lane quarter
    const int r = wq * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t ts = tl + C::tm_s(g), to = tl + C::tm_o(g);
    int scnt = 0;  // score tiles consumed
    bool ok = true;
    Item it;
    for (int item = 0; ok && sched.get(item, it); ++item) {
      const int row = it.q0 + g * kBM + r;
      const int nj = g ? it.nB : it.nA;
      const int diag = 2 * it.t + g;  // the key tile on the diagonal (causal)
      // l_run sums the unrounded weights (the log-sum-exp uses it). The P V MMA sees
      // each weight rounded to 16 bits; l_corr adds, for the largest weight of every
      // tile, the difference its rounding made, so that O / (l_run + l_corr) is the
      // mean of V under the weights the MMA used where it matters: a dominant
      // weight's rounding error then cancels instead of scaling O (the smaller
      // weights' errors are relatively small and of both signs).
      float m_run = -INFINITY, l_run = 0.f, l_corr = 0.f;
      for (int j = 0; j < nj; ++j) {
        if (!(ok = warp_wait(bar(C::B_SFULL + g), scnt & 1, abort_flag, limit))) break;
        ++scnt;
        ptx::tc_fence_after();
        float s[kBN];
        {
          uint32_t u0[32], u1[32], u2[32], u3[32];
          ptx::tmem_ld32(ts + 0, u0);
          ptx::tmem_ld32(ts + 32, u1);
          ptx::tmem_ld32(ts + 64, u2);
          ptx::tmem_ld32(ts + 96, u3);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            s[e] = __uint_as_float(u0[e]);
            s[32 + e] = __uint_as_float(u1[e]);
            s[64 + e] = __uint_as_float(u2[e]);
            s[96 + e] = __uint_as_float(u3[e]);
          }
        }
        const int k0 = j * kBN;
        if ((causal && j == diag) || k0 + kBN > S) {
          const int lim = min(causal ? row - k0 : kBN - 1, S - 1 - k0);  // last visible column
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c > lim) s[c] = -INFINITY;
        }
        // row max with 3-input max over 8 accumulators
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = fmaxf(s[e], s[8 + e]);
#pragma unroll
        for (int c = 16; c < kBN; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = ptx::max3(mx[e], s[c + e], s[c + 8 + e]);
        const float s_max =
            fmaxf(ptx::max3(mx[0], mx[1], mx[2]), ptx::max3(mx[3], mx[4], ptx::max3(mx[5], mx[6], mx[7])));
        const float m_tile = s_max * scale_log2;
        float alpha = 1.f;
        bool corr = false;
        if (j == 0) {
          m_run = m_tile == -INFINITY ? 0.f : m_tile;
        } else if (m_tile > m_run + 8.0f) {
          alpha = ptx::ex2(m_run - m_tile);
          m_run = m_tile;
          l_run *= alpha;
          l_corr *= alpha;
          corr = true;
        }
        // P = exp2(s * scale_log2 - m) as 16-bit pairs into columns [0, 64) of S;
        // the scale-and-shift and the row sum run two lanes per instruction
        const float2 sl2 = make_float2(scale_log2, scale_log2);
        const float2 nm2 = make_float2(-m_run, -m_run);
        float2 sum2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sum2[e] = make_float2(0.f, 0.f);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 x = ptx::fma2(make_float2(s[h * 64 + 2 * c], s[h * 64 + 2 * c + 1]), sl2, nm2);
            const float2 pv = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
            sum2[c & 3] = ptx::add2(sum2[c & 3], pv);
            pk[c] = pack2<F16>(pv.x, pv.y);
          }
          ptx::tmem_st32(ts + h * 32, pk);
        }
        const float2 t2 = ptx::add2(ptx::add2(sum2[0], sum2[1]), ptx::add2(sum2[2], sum2[3]));
        l_run += t2.x + t2.y;
        {
          // the tile's largest weight, computed exactly as the loop above computes it
          const float p_max = ptx::ex2(fmaf(s_max, scale_log2, -m_run));
          l_corr += rounded16<F16>(p_max) - p_max;
        }
        if (__any_sync(0xffffffffu, corr)) {
          // Rescale O after P is out (the scores are dead by now). S_g(j)
          // completing implies P V of tile j-1 has completed (one issuing
          // thread, in-order commits), so O holds exactly tiles < j here; P V
          // of tile j waits for the PFULL arrival below.
          uint32_t u[32];
#pragma unroll 1
          for (int cb = 0; cb < D / 32; ++cb) {
            ptx::tmem_ld32(to + cb * 32, u);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
            ptx::tmem_st32(to + cb * 32, u);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(C::B_PFULL + g));
      }
      if (ok) ok = warp_wait(bar(C::B_OFINAL + g), item & 1, abort_flag, limit);
      if (ok) {
        ptx::tc_fence_after();
        const float inv = 1.0f / (l_run + l_corr);
        // natural log of sum_j exp(score): the scores sum to 2^m_run * l_run in base 2
        if (lse != nullptr && row < S) lse[(size_t)it.n * S + row] = (m_run + log2f(l_run)) * 0.6931471805599453f;
        // the whole O row in one round trip to TMEM (the score registers are free by now);
        // then the accumulator may take the next item while this one is scaled and stored
        uint32_t u[D / 32][32];
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) ptx::tmem_ld32(to + cb * 32, u[cb]);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(C::B_OFREE + g));
        if constexpr (!C::TMA_STORE) {
          uint8_t* orow = out + ((size_t)it.n * S + row) * (size_t)dout * 2;
          const bool st32 = (reinterpret_cast<uintptr_t>(out) & 31) == 0;
#pragma unroll
          for (int cb = 0; cb < D / 32; ++cb) {
            if (row < S && cb * 32 < dout) {
              store_o16<F16>(orow + cb * 64, &u[cb][0], inv, st32);
              store_o16<F16>(orow + cb * 64 + 32, &u[cb][16], inv, st32);
            }
          }
        } else {
          // O / l, rounded to 16 bits, through this warp's staging buffer: one TMA store
          // per 64 columns of its 32 rows. Rows past S and columns past dout lie outside
          // the output tensor and are not written.
          const uint32_t stg = base + C::OFF_O + (uint32_t)warp * C::STG;
          const int y0 = it.q0 + g * kBM + wq * 32;  // first row of this warp (warp-uniform)
#pragma unroll
          for (int h = 0; h < (y0 < S ? D / 64 : 0); ++h) {
            if (lane == 0) ptx::bulk_wait_read_all();  // the buffer's previous store has read it
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c) {  // 16-byte chunk c of the row, at chunk c ^ (row % 8)
              const uint32_t* v = &u[2 * h + c / 4][(c % 4) * 8];
              ptx::st_shared_v4(stg + (uint32_t)lane * 128u + ((uint32_t)(c ^ (lane & 7)) << 4),
                                pack2<F16>(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                                pack2<F16>(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                                pack2<F16>(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                                pack2<F16>(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_3d(&tmo, stg, h * 64, y0, it.n);
              ptx::bulk_commit();
            }
          }
        }
      }
    }
    if (C::TMA_STORE && lane == 0) ptx::bulk_wait_all();  // this warp's output stores are complete
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// d <= 64: P in tensor-memory columns of its own. At d = 64 the two O
// accumulators take 128 columns, which leaves room for the packed P tiles
// beside the score tiles: S_A 0-127, S_B 128-255, P_A 256-319, P_B 320-383,
// O_A 384-447, O_B 448-511. The next score tile S_g(j+1) is then issued as
// soon as the softmax of tile g has copied S_g(j) into registers (SFREE), and
// O_g += P_g(j) V_j as soon as P_g(j) is written (PFULL): the score MMA no longer
// waits for the P V that used to read P out of the score tile's columns, so
// the tensor core computes the next scores while the softmax exponentiates the
// current ones, and each softmax warpgroup finds its next tile ready. The
// softmax writes P_g(j) only after P V(j-1) has read P_g(j-1) (PVDONE, which
// also makes O hold exactly tiles < j when it must be rescaled).
// MMA issue order per key tile j: S_A(j+1), S_B(j+1), then P V_A(j), P V_B(j).
// ---------------------------------------------------------------------------
struct Tc64 {
  static constexpr int D = 64;
  static constexpr int TILE = kBM * D * 2;  // bytes of a Q, K or V tile (128 rows x 128 bytes)
  static constexpr int KS = 4, VS = 4;      // K and V ring stages
  static constexpr int OFF_Q = 0;           // Q_A then Q_B
  static constexpr int OFF_K = OFF_Q + 2 * TILE;
  static constexpr int OFF_V = OFF_K + KS * TILE;
  static constexpr int OFF_BAR = OFF_V + VS * TILE;
  enum {
    B_Q = 0,
    B_KFULL = 1,
    B_KEMPTY = B_KFULL + KS,
    B_VFULL = B_KEMPTY + KS,
    B_VEMPTY = B_VFULL + VS,
    B_SFULL = B_VEMPTY + VS,  // [2]: S of tile A / B computed
    B_SFREE = B_SFULL + 2,    // [2]: S of tile A / B copied into registers by the softmax
    B_PFULL = B_SFREE + 2,    // [2]: P of tile A / B written (and O rescaled)
    B_PVDONE = B_PFULL + 2,   // [2]: a P V of tile A / B completed (each one commits)
    B_OFREE = B_PVDONE + 2,   // [2]: O of tile A / B read out by the epilogue
    B_QFREE = B_OFREE + 2,    // last score MMA of an item done: Q may be replaced
    B_DRAIN = B_QFREE + 1,
    NBAR = B_DRAIN + 1
  };
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int SMEM = BYTES + 1024;
  static_assert(SMEM <= 232448, "at most 227 KB of shared memory per CTA");
  __host__ __device__ static constexpr uint32_t tm_s(int g) { return 128u * (uint32_t)g; }
  __host__ __device__ static constexpr uint32_t tm_p(int g) { return 256u + 64u * (uint32_t)g; }
  __host__ __device__ static constexpr uint32_t tm_o(int g) { return 384u + 64u * (uint32_t)g; }
};

template <bool F16>
__global__ void __launch_bounds__(kThreadsTC, 1)
    attn_tc64_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const __grid_constant__ SchedTable tab,
                     uint8_t* __restrict__ out, float* __restrict__ lse, int dout, int N, int S, int causal,
                     float scale_log2, unsigned long long limit) {
  // dout: output columns per row (64, or 32 when a d = 32 problem runs here with its
  // tiles zero-filled by TMA past column 32)
  using C = Tc64;
  constexpr int D = C::D;
  constexpr uint32_t kAB = F16 ? 0u : 1u;
  constexpr uint32_t IDESC_QK = ptx::f16_idesc(kBM, kBN, kAB, 0);
  constexpr uint32_t IDESC_PV = ptx::f16_idesc(kBM, D, kAB, 1);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 4);
  auto bar = [&](int i) -> uint32_t { return base + C::OFF_BAR + 8u * (uint32_t)i; };

  const Schedule sched(N, S, causal, &tab);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    ptx::mbar_init(bar(C::B_Q), 1);
    for (int s = 0; s < C::KS; ++s) {
      ptx::mbar_init(bar(C::B_KFULL + s), 1);
      ptx::mbar_init(bar(C::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < C::VS; ++s) {
      ptx::mbar_init(bar(C::B_VFULL + s), 1);
      ptx::mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    for (int g = 0; g < 2; ++g) {
      ptx::mbar_init(bar(C::B_SFULL + g), 1);
      ptx::mbar_init(bar(C::B_SFREE + g), 4 * 32);
      ptx::mbar_init(bar(C::B_PFULL + g), 4 * 32);
      ptx::mbar_init(bar(C::B_PVDONE + g), 1);
      ptx::mbar_init(bar(C::B_OFREE + g), 4 * 32);
    }
    ptx::mbar_init(bar(C::B_QFREE), 1);
    ptx::mbar_init(bar(C::B_DRAIN), 1);
    ptx::fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    ptx::tmem_alloc(base + C::OFF_MISC, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + C::OFF_MISC);

  if (warp >= kWarpTMA) {
    ptx::regs_decrease<kRegsControl>();
    if (warp == kWarpTMA) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        ptx::tma_prefetch_desc(&tmq);
        ptx::tma_prefetch_desc(&tmk);
        ptx::tma_prefetch_desc(&tmv);
        int kdone = 0, vdone = 0, items = 0;
        bool ok = true;
        Item it;
        for (int round = 0; ok && sched.get(round, it); ++round) {
          if (items > 0) ok = wait_bar(bar(C::B_QFREE), (items - 1) & 1, abort_flag, limit, true);
          if (!ok) break;
          ptx::mbar_arrive_expect_tx(bar(C::B_Q), 2 * C::TILE);
          for (int g = 0; g < 2; ++g)
            ptx::tma_load_3d(base + C::OFF_Q + g * C::TILE, &tmq, bar(C::B_Q), 0, it.q0 + g * kBM, it.n);
          for (int j = 0; j < it.nB && ok; ++j) {
            const int ks = kdone % C::KS, vs = vdone % C::VS;
            if (kdone >= C::KS) ok = wait_bar(bar(C::B_KEMPTY + ks), ((kdone / C::KS) & 1) ^ 1, abort_flag, limit, true);
            if (!ok) break;
            ptx::mbar_arrive_expect_tx(bar(C::B_KFULL + ks), C::TILE);
            ptx::tma_load_3d(base + C::OFF_K + ks * C::TILE, &tmk, bar(C::B_KFULL + ks), 0, j * kBN, it.n);
            ++kdone;
            if (vdone >= C::VS) ok = wait_bar(bar(C::B_VEMPTY + vs), ((vdone / C::VS) & 1) ^ 1, abort_flag, limit, true);
            if (!ok) break;
            ptx::mbar_arrive_expect_tx(bar(C::B_VFULL + vs), C::TILE);
            ptx::tma_load_3d(base + C::OFF_V + vs * C::TILE, &tmv, bar(C::B_VFULL + vs), 0, j * kBN, it.n);
            ++vdone;
          }
          ++items;
        }
        if (items > 0) wait_bar(bar(C::B_Q), (items - 1) & 1, abort_flag, limit, false);
        for (int x = kdone - C::KS < 0 ? 0 : kdone - C::KS; x < kdone; ++x)
          wait_bar(bar(C::B_KFULL + x % C::KS), (x / C::KS) & 1, abort_flag, limit, false);
        for (int x = vdone - C::VS < 0 ? 0 : vdone - C::VS; x < vdone; ++x)
          wait_bar(bar(C::B_VFULL + x % C::VS), (x / C::VS) & 1, abort_flag, limit, false);
      }
      __syncwarp();
    } else if (warp == kWarpMMA) {
      // ------------------------------------------------------------ MMA issuer
      auto issue_s = [&](int g, int ks) {
        const uint64_t a0 = ptx::sw128_desc(base + C::OFF_Q + g * C::TILE, 16, 1024);
        const uint64_t b0 = ptx::sw128_desc(base + C::OFF_K + ks * C::TILE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(kk * 32) >> 4;
          ptx::mma_f16_ss_elect(tmem + C::tm_s(g), a0 + off, b0 + off, IDESC_QK, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit_elect(bar(C::B_SFULL + g));
      };
      auto issue_pv = [&](int g, int vs, bool first) {
        const uint64_t b0 = ptx::sw128_desc(base + C::OFF_V + vs * C::TILE, kColBlock, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          ptx::mma_f16_ts_elect(tmem + C::tm_o(g), tmem + C::tm_p(g) + kk * 8, b0 + ((kk * 16 * 128) >> 4), IDESC_PV,
                                (!first || kk > 0) ? 1u : 0u);
        ptx::mma_commit_elect(bar(C::B_PVDONE + g));
      };
      bool ok = true;
      int kbase = 0, vbase = 0;  // ring positions of the current item's first K and V tiles
      int sa = 0, sb = 0;        // score tiles of tile A / B issued
      int pa = 0, pb = 0;        // P tiles of tile A / B consumed
      Item it;
      for (int item = 0; ok && sched.get(item, it); ++item) {
        const int nA = it.nA, nB = it.nB;
        ok = warp_wait(bar(C::B_Q), item & 1, abort_flag, limit);
        const int ks0 = kbase % C::KS;
        if (ok) ok = warp_wait(bar(C::B_KFULL + ks0), (kbase / C::KS) & 1, abort_flag, limit);
        // a score tile is overwritten only after the softmax has copied the previous one out
        if (ok && sa > 0) ok = warp_wait(bar(C::B_SFREE + 0), (sa - 1) & 1, abort_flag, limit);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_s(0, ks0);
        ++sa;
        if (sb > 0) ok = warp_wait(bar(C::B_SFREE + 1), (sb - 1) & 1, abort_flag, limit);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_s(1, ks0);
        ++sb;
        ptx::mma_commit_elect(bar(C::B_KEMPTY + ks0));
        if (nB == 1) ptx::mma_commit_elect(bar(C::B_QFREE));
        for (int j = 0; j < nB && ok; ++j) {
          const int jn = j + 1, kpn = kbase + jn, ksn = kpn % C::KS;
          if (jn < nB) {  // the next scores first: the softmax waits for them, P V is off its path
            ok = warp_wait(bar(C::B_KFULL + ksn), (kpn / C::KS) & 1, abort_flag, limit);
            if (ok && jn < nA) {
              ok = warp_wait(bar(C::B_SFREE + 0), (sa - 1) & 1, abort_flag, limit);
              if (ok) {
                ptx::tc_fence_after();
                issue_s(0, ksn);
                ++sa;
              }
            }
            if (ok) ok = warp_wait(bar(C::B_SFREE + 1), (sb - 1) & 1, abort_flag, limit);
            if (!ok) break;
            ptx::tc_fence_after();
            issue_s(1, ksn);
            ++sb;
            ptx::mma_commit_elect(bar(C::B_KEMPTY + ksn));
            if (jn == nB - 1) ptx::mma_commit_elect(bar(C::B_QFREE));  // the item's last score MMA
          }
          const int vp = vbase + j, vs = vp % C::VS;
          ok = warp_wait(bar(C::B_VFULL + vs), (vp / C::VS) & 1, abort_flag, limit);
          if (ok && j < nA) {
            ok = warp_wait(bar(C::B_PFULL + 0), pa & 1, abort_flag, limit);
            if (ok && j == 0 && item > 0) ok = warp_wait(bar(C::B_OFREE + 0), (item - 1) & 1, abort_flag, limit);
            if (ok) {
              ++pa;
              ptx::tc_fence_after();
              issue_pv(0, vs, j == 0);
            }
          }
          if (ok) ok = warp_wait(bar(C::B_PFULL + 1), pb & 1, abort_flag, limit);
          if (ok && j == 0 && item > 0) ok = warp_wait(bar(C::B_OFREE + 1), (item - 1) & 1, abort_flag, limit);
          if (!ok) break;
          ++pb;
          ptx::tc_fence_after();
          issue_pv(1, vs, j == 0);
          ptx::mma_commit_elect(bar(C::B_VEMPTY + vs));
        }
        kbase += nB;
        vbase += nB;
      }
      ptx::mma_commit_elect(bar(C::B_DRAIN));
      warp_wait_all(bar(C::B_DRAIN), 0, abort_flag, limit, false);
    }
  } else {
    ptx::regs_increase<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax, warps 0-7
    const int g = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t ts = tl + C::tm_s(g), tp = tl + C::tm_p(g), to = tl + C::tm_o(g);
    int scnt = 0;  // score tiles consumed
    int pcnt = 0;  // P tiles written (= P V of this tile issued or to be issued)
    bool ok = true;
    Item it;
    for (int item = 0; ok && sched.get(item, it); ++item) {
      const int row = it.q0 + g * kBM + r;
      const int nj = g ? it.nB : it.nA;
      const int diag = 2 * it.t + g;
      // l_run sums the unrounded weights (the log-sum-exp uses it). The P V MMA sees
      // each weight rounded to 16 bits; l_corr adds, for the largest weight of every
      // tile, the difference its rounding made, so that O / (l_run + l_corr) is the
      // mean of V under the weights the MMA used where it matters: a dominant
      // weight's rounding error then cancels instead of scaling O (the smaller
      // weights' errors are relatively small and of both signs).
      float m_run = -INFINITY, l_run = 0.f, l_corr = 0.f;
      for (int j = 0; j < nj; ++j) {
        if (!(ok = warp_wait(bar(C::B_SFULL + g), scnt & 1, abort_flag, limit))) break;
        ++scnt;
        ptx::tc_fence_after();
        float s[kBN];
        {
          uint32_t u0[32], u1[32], u2[32], u3[32];
          ptx::tmem_ld32(ts + 0, u0);
          ptx::tmem_ld32(ts + 32, u1);
          ptx::tmem_ld32(ts + 64, u2);
          ptx::tmem_ld32(ts + 96, u3);
          ptx::tmem_wait_ld();
          // the score columns may take the next tile's scores now
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(C::B_SFREE + g));
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            s[e] = __uint_as_float(u0[e]);
            s[32 + e] = __uint_as_float(u1[e]);
            s[64 + e] = __uint_as_float(u2[e]);
            s[96 + e] = __uint_as_float(u3[e]);
          }
        }
        const int k0 = j * kBN;
        if ((causal && j == diag) || k0 + kBN > S) {
          const int lim = min(causal ? row - k0 : kBN - 1, S - 1 - k0);
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c > lim) s[c] = -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = fmaxf(s[e], s[8 + e]);
#pragma unroll
        for (int c = 16; c < kBN; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = ptx::max3(mx[e], s[c + e], s[c + 8 + e]);
        const float s_max =
            fmaxf(ptx::max3(mx[0], mx[1], mx[2]), ptx::max3(mx[3], mx[4], ptx::max3(mx[5], mx[6], mx[7])));
        const float m_tile = s_max * scale_log2;
        float alpha = 1.f;
        bool corr = false;
        if (j == 0) {
          m_run = m_tile == -INFINITY ? 0.f : m_tile;
        } else if (m_tile > m_run + 8.0f) {
          alpha = ptx::ex2(m_run - m_tile);
          m_run = m_tile;
          l_run *= alpha;
          l_corr *= alpha;
          corr = true;
        }
        const float2 sl2 = make_float2(scale_log2, scale_log2);
        const float2 nm2 = make_float2(-m_run, -m_run);
        float2 sum2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sum2[e] = make_float2(0.f, 0.f);
        uint32_t pk[2][32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 x = ptx::fma2(make_float2(s[h * 64 + 2 * c], s[h * 64 + 2 * c + 1]), sl2, nm2);
            const float2 pv = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
            sum2[c & 3] = ptx::add2(sum2[c & 3], pv);
            pk[h][c] = pack2<F16>(pv.x, pv.y);
          }
        }
        const float2 t2 = ptx::add2(ptx::add2(sum2[0], sum2[1]), ptx::add2(sum2[2], sum2[3]));
        l_run += t2.x + t2.y;
        {
          // the tile's largest weight, computed exactly as the loop above computes it
          const float p_max = ptx::ex2(fmaf(s_max, scale_log2, -m_run));
          l_corr += rounded16<F16>(p_max) - p_max;
        }
        // P V of the previous tile has read P and added into O: P may be overwritten,
        // and O holds exactly the tiles before j for the rescale
        if (pcnt > 0 && !(ok = warp_wait(bar(C::B_PVDONE + g), (pcnt - 1) & 1, abort_flag, limit))) break;
        ptx::tc_fence_after();
        ptx::tmem_st32(tp + 0, pk[0]);
        ptx::tmem_st32(tp + 32, pk[1]);
        if (__any_sync(0xffffffffu, corr)) {
          uint32_t u[32];
#pragma unroll 1
          for (int cb = 0; cb < D / 32; ++cb) {
            ptx::tmem_ld32(to + cb * 32, u);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
            ptx::tmem_st32(to + cb * 32, u);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(C::B_PFULL + g));
        ++pcnt;
      }
      // the item's last P V of this tile complete: O is final
      if (ok) ok = warp_wait(bar(C::B_PVDONE + g), (pcnt - 1) & 1, abort_flag, limit);
      if (ok) {
        ptx::tc_fence_after();
        const float inv = 1.0f / (l_run + l_corr);
        if (lse != nullptr && row < S) lse[(size_t)it.n * S + row] = (m_run + log2f(l_run)) * 0.6931471805599453f;
        uint32_t u[D / 32][32];
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) ptx::tmem_ld32(to + cb * 32, u[cb]);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(C::B_OFREE + g));
        uint8_t* orow = out + ((size_t)it.n * S + row) * (size_t)dout * 2;
        const bool st32 = (reinterpret_cast<uintptr_t>(out) & 31) == 0;
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          if (row < S && cb * 32 < dout) {
            store_o16<F16>(orow + cb * 64, &u[cb][0], inv, st32);
            store_o16<F16>(orow + cb * 64 + 32, &u[cb][16], inv, st32);
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// d = 256. Two 128 x 256 fp32 O accumulators would take all 512 TMEM columns,
// so here a work item is ONE 128-row query tile, and TMEM holds two 128 x 64
// score buffers (the scores of key tile j+1 are computed while the softmax
// works on tile j), the item's Q tile as 16-bit pairs (the A operand of the
// score MMAs, so that they read only K from shared memory: with Q read from
// shared memory as well, the MMAs' operand reads and the TMA writes of K and V
// took more of the shared-memory port than the tensor pipe had work) and the
// 128 x 256 O. The softmax warps copy each Q tile from its TMA landing zone in
// shared memory into TMEM: the first item's before its first tile, every later
// one during the previous item's last tile, as soon as that tile's scores are
// in registers (all of that item's score MMAs have then completed). Key tiles are 64 keys; K and V rings
// of two 32 KB stages each plus the 64 KB Q tile use 192 KB of shared memory.
// Warps 0-3 run the softmax (thread = row = TMEM lane), warp 4 loads Q and K
// with TMA, warp 6 loads V (so K tiles are not held behind V's ring), warp 5
// issues the MMAs. MMA order per item: S(0), S(1), then for each j:
// PV(j), S(j+2). S(j+2) reuses the buffer of P(j) only after PV(j) read it
// (in-order execution); since PV(j) is no longer ordered before S(j+1), a
// softmax that must rescale O first waits for the PVDONE commit of PV(j-1).
// ---------------------------------------------------------------------------
constexpr int kThreads256 = 224;
constexpr int kWarpTMA256 = 4;   // Q and K tiles
constexpr int kWarpMMA256 = 5;
constexpr int kWarpTMAV256 = 6;  // V tiles: a producer of its own, so K loads run ahead of V's
constexpr int kBN256 = 64;

struct Tc256 {
  static constexpr int D = 256;
  static constexpr int QTILE = kBM * D * 2;      // 64 KB
  static constexpr int KTILE = kBN256 * D * 2;   // 32 KB (K or V)
  static constexpr int KS = 2, VS = 2;
  static constexpr uint32_t QBLK = kBM * 128;     // a 64-feature column block of Q: 128 rows x 128 bytes
  static constexpr uint32_t KBLK = kBN256 * 128;  // a 64-feature column block of K or V: 64 rows x 128 bytes
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QTILE;
  static constexpr int OFF_V = OFF_K + KS * KTILE;
  // output staging: two 32-row x 64-column buffers per softmax warp, in the
  // 128-byte swizzled layout of the output tensor map's boxes (TMA stores)
  static constexpr int STG = 32 * 64 * 2;
  static constexpr int OFF_O = OFF_V + VS * KTILE;
  static constexpr int OFF_BAR = OFF_O + 4 * 2 * STG;
  enum {
    B_Q = 0,
    B_KFULL = 1,
    B_KEMPTY = B_KFULL + KS,
    B_VFULL = B_KEMPTY + KS,
    B_VEMPTY = B_VFULL + VS,
    B_SFULL = B_VEMPTY + VS,  // [2]: score buffer b computed
    B_PFULL = B_SFULL + 2,    // [2]: P written into buffer b (and O rescaled)
    B_PVDONE = B_PFULL + 2,   // every P V completed, in order
    B_OFINAL = B_PVDONE + 1,  // last P V of an item completed
    B_OFREE = B_OFINAL + 1,   // O read out by the epilogue
    B_QTM = B_OFREE + 1,      // the item's Q copied from shared memory into TMEM
    B_DRAIN = B_QTM + 1,
    NBAR = B_DRAIN + 1
  };
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int SMEM = BYTES + 1024;
  static_assert(SMEM <= 232448, "at most 227 KB of shared memory per CTA");
  static constexpr uint32_t TM_O = 256;  // O in columns 256-511; score buffer b in 64 b .. 64 b + 63
  static constexpr uint32_t TM_Q = 128;  // Q in columns 128-255: column c holds features 2c, 2c + 1
};

// One query tile per item: from the host's work lists (same construction as for
// the pair kernel), or heaviest (causal) first in a snake order.
struct Item256 {
  int n, q0, nk;  // head, first row, key tiles
};

struct Schedule256 {
  int N, S, causal, tiles, nkv, total;
  const SchedTable* tab;
  __device__ Schedule256(int N_, int S_, int causal_, const SchedTable* tab_)
      : N(N_), S(S_), causal(causal_), tab(tab_) {
    tiles = (S + kBM - 1) / kBM;
    nkv = (S + kBN256 - 1) / kBN256;
    total = N * tiles;
  }
  __device__ bool get(int round, Item256& it) const {
    const int c = (int)blockIdx.x;
    int t;
    if (tab->count > 0) {
      const int k = (int)tab->start[c] + round;
      if (k >= (int)tab->start[c + 1]) return false;
      const unsigned int e = tab->item[k];
      it.n = (int)(e >> 16);
      t = (int)(e & 0xFFFFu);
    } else {
      const int G = (int)gridDim.x;
      const int i = round * G + ((round & 1) ? G - 1 - c : c);
      if (i >= total) return false;
      t = tiles - 1 - i / N;
      it.n = i % N;
    }
    it.q0 = t * kBM;
    it.nk = causal ? min(2 * t + 2, nkv) : nkv;
    return true;
  }
};

template <bool F16>
__global__ void __launch_bounds__(kThreads256, 1)
    attn_tc256_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                      const __grid_constant__ SchedTable tab,
                      uint8_t* __restrict__ out, float* __restrict__ lse, int N, int S, int causal,
                      float scale_log2, unsigned long long limit) {
  using C = Tc256;
  constexpr uint32_t kAB = F16 ? 0u : 1u;
  constexpr uint32_t IDESC_QK = ptx::f16_idesc(kBM, kBN256, kAB, 0);
  constexpr uint32_t IDESC_PV = ptx::f16_idesc(kBM, C::D, kAB, 1);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 4);
  auto bar = [&](int i) -> uint32_t { return base + C::OFF_BAR + 8u * (uint32_t)i; };

  const Schedule256 sched(N, S, causal, &tab);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    ptx::mbar_init(bar(C::B_Q), 1);
    for (int s = 0; s < C::KS; ++s) {
      ptx::mbar_init(bar(C::B_KFULL + s), 1);
      ptx::mbar_init(bar(C::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < C::VS; ++s) {
      ptx::mbar_init(bar(C::B_VFULL + s), 1);
      ptx::mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(bar(C::B_SFULL + b), 1);
      ptx::mbar_init(bar(C::B_PFULL + b), 4 * 32);
    }
    ptx::mbar_init(bar(C::B_PVDONE), 1);
    ptx::mbar_init(bar(C::B_OFINAL), 1);
    ptx::mbar_init(bar(C::B_OFREE), 4 * 32);
    ptx::mbar_init(bar(C::B_QTM), 4 * 32);
    ptx::mbar_init(bar(C::B_DRAIN), 1);
    ptx::fence_mbar_init();
  }
  if (warp == kWarpMMA256) {
    ptx::tmem_alloc(base + C::OFF_MISC, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + C::OFF_MISC);

  if (warp == kWarpTMA256) {
    // ------------------------------------------------------------ TMA producer: Q and K
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmq);
      ptx::tma_prefetch_desc(&tmk);
      int kdone = 0, items = 0;
      bool ok = true;
      Item256 it;
      for (int round = 0; ok && sched.get(round, it); ++round) {
        // the previous Q tile has been copied into TMEM: its landing zone may be reused
        if (items > 0) ok = wait_bar(bar(C::B_QTM), (items - 1) & 1, abort_flag, limit, true);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(bar(C::B_Q), C::QTILE);
        for (int b = 0; b < 4; ++b)
          ptx::tma_load_3d(base + C::OFF_Q + b * C::QBLK, &tmq, bar(C::B_Q), b * 64, it.q0, it.n);
        for (int j = 0; j < it.nk && ok; ++j) {
          const int ks = kdone % C::KS;
          if (kdone >= C::KS) ok = wait_bar(bar(C::B_KEMPTY + ks), ((kdone / C::KS) & 1) ^ 1, abort_flag, limit, true);
          if (!ok) break;
          ptx::mbar_arrive_expect_tx(bar(C::B_KFULL + ks), C::KTILE);
          for (int b = 0; b < 4; ++b)
            ptx::tma_load_3d(base + C::OFF_K + ks * C::KTILE + b * C::KBLK, &tmk, bar(C::B_KFULL + ks), b * 64,
                             j * kBN256, it.n);
          ++kdone;
        }
        ++items;
      }
      if (items > 0) wait_bar(bar(C::B_Q), (items - 1) & 1, abort_flag, limit, false);
      for (int x = kdone - C::KS < 0 ? 0 : kdone - C::KS; x < kdone; ++x)
        wait_bar(bar(C::B_KFULL + x % C::KS), (x / C::KS) & 1, abort_flag, limit, false);
    }
    __syncwarp();
  } else if (warp == kWarpTMAV256) {
    // ------------------------------------------------------------ TMA producer: V
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmv);
      ptx::tma_prefetch_desc(&tmo);
      int vdone = 0;
      bool ok = true;
      Item256 it;
      for (int round = 0; ok && sched.get(round, it); ++round) {
        for (int j = 0; j < it.nk && ok; ++j) {
          const int vs = vdone % C::VS;
          if (vdone >= C::VS) ok = wait_bar(bar(C::B_VEMPTY + vs), ((vdone / C::VS) & 1) ^ 1, abort_flag, limit, true);
          if (!ok) break;
          ptx::mbar_arrive_expect_tx(bar(C::B_VFULL + vs), C::KTILE);
          for (int b = 0; b < 4; ++b)
            ptx::tma_load_3d(base + C::OFF_V + vs * C::KTILE + b * C::KBLK, &tmv, bar(C::B_VFULL + vs), b * 64,
                             j * kBN256, it.n);
          ++vdone;
        }
      }
      for (int x = vdone - C::VS < 0 ? 0 : vdone - C::VS; x < vdone; ++x)
        wait_bar(bar(C::B_VFULL + x % C::VS), (x / C::VS) & 1, abort_flag, limit, false);
    }
    __syncwarp();
  } else if (warp == kWarpMMA256) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop; one elected lane issues each MMA and commit.
    {
      // S(buffer b) = Q K^T: 16 k-steps of 16 features; Q from TMEM (8 columns a
      // k-step), K K-major from shared memory
      auto issue_s = [&](int b, int ks) {
        const uint64_t b0 = ptx::sw128_desc(base + C::OFF_K + ks * C::KTILE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk) {
          const uint32_t offb = ((kk >> 2) * C::KBLK + (kk & 3) * 32) >> 4;
          ptx::mma_f16_ts_elect(tmem + 64u * (uint32_t)b, tmem + C::TM_Q + kk * 8, b0 + offb, IDESC_QK,
                                kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit_elect(bar(C::B_SFULL + b));
      };
      // O += P(buffer b) V: 4 k-steps of 16 keys; V MN-major, column blocks KBLK apart
      auto issue_pv = [&](int b, int vs, bool first) {
        const uint64_t b0 = ptx::sw128_desc(base + C::OFF_V + vs * C::KTILE, C::KBLK, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN256 / 16; ++kk)
          ptx::mma_f16_ts_elect(tmem + C::TM_O, tmem + 64u * (uint32_t)b + kk * 8, b0 + ((kk * 16 * 128) >> 4), IDESC_PV,
                          (!first || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      int kcons = 0, vcons = 0, scnt = 0, pcnt = 0;
      Item256 it;
      for (int item = 0; ok && sched.get(item, it); ++item) {
        const int nk = it.nk;
        ok = warp_wait(bar(C::B_QTM), item & 1, abort_flag, limit);
        // S(0) and S(1)
        for (int j = 0; j < 2 && j < nk && ok; ++j) {
          const int ks = kcons % C::KS;
          ok = warp_wait(bar(C::B_KFULL + ks), (kcons / C::KS) & 1, abort_flag, limit);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_s(scnt & 1, ks);
          ptx::mma_commit_elect(bar(C::B_KEMPTY + ks));
          ++kcons;
          ++scnt;
        }
        for (int j = 0; j < nk && ok; ++j) {
          const int vs = vcons % C::VS;
          ok = warp_wait(bar(C::B_VFULL + vs), (vcons / C::VS) & 1, abort_flag, limit);
          if (ok) ok = warp_wait(bar(C::B_PFULL + (pcnt & 1)), (pcnt >> 1) & 1, abort_flag, limit);
          if (ok && j == 0 && item > 0) ok = warp_wait(bar(C::B_OFREE), (item - 1) & 1, abort_flag, limit);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_pv(pcnt & 1, vs, j == 0);
          ptx::mma_commit_elect(bar(C::B_PVDONE));
          ptx::mma_commit_elect(bar(C::B_VEMPTY + vs));
          ++vcons;
          ++pcnt;
          if (j + 2 < nk) {
            const int ks = kcons % C::KS;
            ok = warp_wait(bar(C::B_KFULL + ks), (kcons / C::KS) & 1, abort_flag, limit);
            if (!ok) break;
            ptx::tc_fence_after();
            issue_s(scnt & 1, ks);
            ptx::mma_commit_elect(bar(C::B_KEMPTY + ks));
            ++kcons;
            ++scnt;
          }
        }
        if (ok) ptx::mma_commit_elect(bar(C::B_OFINAL));
      }
      ptx::mma_commit_elect(bar(C::B_DRAIN));
      warp_wait_all(bar(C::B_DRAIN), 0, abort_flag, limit, false);
    }
  } else {
    // ------------------------------------------------------------ softmax, warps 0-3
    const int r = warp * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t to = tl + C::TM_O;
    // Q tile of item k: this thread's row of the 128-byte-swizzled landing zone
    // (16-byte chunk c of a 64-feature block at chunk c ^ (row % 8)) into TMEM
    // columns TM_Q + 32 b + 4 c .. + 3 (four feature pairs per chunk)
    auto copy_q = [&](int k) -> bool {
      if (!warp_wait(bar(C::B_Q), k & 1, abort_flag, limit)) return false;
#pragma unroll 1
      for (int blk = 0; blk < C::D / 64; ++blk) {
        uint32_t u[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 x = *reinterpret_cast<const uint4*>(sm + C::OFF_Q + blk * C::QBLK + r * 128 +
                                                          ((c ^ (r & 7)) << 4));
          u[4 * c] = x.x;
          u[4 * c + 1] = x.y;
          u[4 * c + 2] = x.z;
          u[4 * c + 3] = x.w;
        }
        ptx::tmem_st32(tl + C::TM_Q + blk * 32, u);
      }
      ptx::tmem_wait_st();
      ptx::fence_proxy_async_smem();  // the reads of the landing zone before TMA rewrites it
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(C::B_QTM));
      return true;
    };
    int scnt = 0;  // score tiles consumed (global)
    bool ok = true;
    Item256 it;
    for (int item = 0; ok && sched.get(item, it); ++item) {
      if (item == 0 && !(ok = copy_q(0))) break;
      const int row = it.q0 + r;
      // l_run sums the unrounded weights (the log-sum-exp uses it). The P V MMA sees
      // each weight rounded to 16 bits; l_corr adds, for the largest weight of every
      // tile, the difference its rounding made, so that O / (l_run + l_corr) is the
      // mean of V under the weights the MMA used where it matters: a dominant
      // weight's rounding error then cancels instead of scaling O (the smaller
      // weights' errors are relatively small and of both signs).
      float m_run = -INFINITY, l_run = 0.f, l_corr = 0.f;
      for (int j = 0; j < it.nk; ++j) {
        const int b = scnt & 1;
        if (!(ok = warp_wait(bar(C::B_SFULL + b), (scnt >> 1) & 1, abort_flag, limit))) break;
        ptx::tc_fence_after();
        const uint32_t ts = tl + 64u * (uint32_t)b;
        float s[kBN256];
        {
          uint32_t u0[32], u1[32];
          ptx::tmem_ld32(ts + 0, u0);
          ptx::tmem_ld32(ts + 32, u1);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            s[e] = __uint_as_float(u0[e]);
            s[32 + e] = __uint_as_float(u1[e]);
          }
        }
        if (j == it.nk - 1) {
          // every score MMA of this item has completed: the next item's Q may replace it
          Item256 nx;
          if (sched.get(item + 1, nx) && !(ok = copy_q(item + 1))) break;
        }
        const int k0 = j * kBN256;
        if ((causal && k0 + kBN256 - 1 > it.q0) || k0 + kBN256 > S) {
          const int lim = min(causal ? row - k0 : kBN256 - 1, S - 1 - k0);  // last visible column
#pragma unroll
          for (int c = 0; c < kBN256; ++c)
            if (c > lim) s[c] = -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = fmaxf(s[e], s[8 + e]);
#pragma unroll
        for (int c = 16; c < kBN256; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e) mx[e] = ptx::max3(mx[e], s[c + e], s[c + 8 + e]);
        const float s_max =
            fmaxf(ptx::max3(mx[0], mx[1], mx[2]), ptx::max3(mx[3], mx[4], ptx::max3(mx[5], mx[6], mx[7])));
        const float m_tile = s_max * scale_log2;
        float alpha = 1.f;
        bool corr = false;
        if (j == 0) {
          m_run = m_tile == -INFINITY ? 0.f : m_tile;
        } else if (m_tile > m_run + 8.0f) {
          alpha = ptx::ex2(m_run - m_tile);
          m_run = m_tile;
          l_run *= alpha;
          l_corr *= alpha;
          corr = true;
        }
        const float2 sl2 = make_float2(scale_log2, scale_log2);
        const float2 nm2 = make_float2(-m_run, -m_run);
        float2 sum2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sum2[e] = make_float2(0.f, 0.f);
        {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 x = ptx::fma2(make_float2(s[2 * c], s[2 * c + 1]), sl2, nm2);
            const float2 pv = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
            sum2[c & 3] = ptx::add2(sum2[c & 3], pv);
            pk[c] = pack2<F16>(pv.x, pv.y);
          }
          ptx::tmem_st32(ts, pk);
        }
        const float2 t2 = ptx::add2(ptx::add2(sum2[0], sum2[1]), ptx::add2(sum2[2], sum2[3]));
        l_run += t2.x + t2.y;
        {
          // the tile's largest weight, computed exactly as the loop above computes it
          const float p_max = ptx::ex2(fmaf(s_max, scale_log2, -m_run));
          l_corr += rounded16<F16>(p_max) - p_max;
        }
        if (__any_sync(0xffffffffu, corr)) {
          // O must hold exactly the tiles before j: wait for P V of tile j-1
          // (global index scnt - 1). Its phase is unambiguous: S of this tile
          // was issued after P V of tile j-2, so that one has completed.
          if (!(ok = warp_wait(bar(C::B_PVDONE), (scnt - 1) & 1, abort_flag, limit))) break;
          ptx::tc_fence_after();
          uint32_t u[32];
#pragma unroll 1
          for (int cb = 0; cb < C::D / 32; ++cb) {
            ptx::tmem_ld32(to + cb * 32, u);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
            ptx::tmem_st32(to + cb * 32, u);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(C::B_PFULL + b));
        ++scnt;
      }
      if (ok) ok = warp_wait(bar(C::B_OFINAL), item & 1, abort_flag, limit);
      if (ok) {
        ptx::tc_fence_after();
        const float inv = 1.0f / (l_run + l_corr);
        if (lse != nullptr && row < S) lse[(size_t)it.n * S + row] = (m_run + log2f(l_run)) * 0.6931471805599453f;
        // O / l, rounded to 16 bits, 64 columns at a time through this warp's two
        // staging buffers (alternating), one TMA store each; rows past S lie outside
        // the output tensor and are not written.
        const int y0 = it.q0 + warp * 32;  // first row of this warp (warp-uniform)
        uint32_t u[2][32];
#pragma unroll 1
        for (int h = 0; h < C::D / 64; ++h) {
          ptx::tmem_ld32(to + h * 64, u[0]);
          ptx::tmem_ld32(to + h * 64 + 32, u[1]);
          ptx::tmem_wait_ld();
          if (h == C::D / 64 - 1) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(C::B_OFREE));
          }
          if (y0 >= S) continue;
          const uint32_t stg = base + C::OFF_O + (uint32_t)(warp * 2 + (h & 1)) * C::STG;
          if (lane == 0) ptx::bulk_wait_read_1();  // the store that last used this buffer has read it
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // 16-byte chunk c of the row, at chunk c ^ (row % 8)
            const uint32_t* v = &u[c / 4][(c % 4) * 8];
            ptx::st_shared_v4(stg + (uint32_t)lane * 128u + ((uint32_t)(c ^ (lane & 7)) << 4),
                              pack2<F16>(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                              pack2<F16>(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                              pack2<F16>(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                              pack2<F16>(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d(&tmo, stg, h * 64, y0, it.n);
            ptx::bulk_commit();
          }
        }
      }
    }
    if (lane == 0) ptx::bulk_wait_all();  // this warp's output stores are complete
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA256) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// One thread waits on an mbarrier nothing will complete; the bounded wait must
// record a timeout and return.
__global__ void selftest_timeout_kernel(unsigned long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_bar(ptx::smem_u32(&bar), 0, &abort_flag, limit, false);
}

// ---- host side ----------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    (void)cudaGetLastError();
  });
  return fn;
}

// K and V bytes that one head group may keep in L2: about a quarter of the
// 129 MB, leaving room for the Q, O and next-group traffic around them.
constexpr double kGroupKvBytes = 32.0 * 1024 * 1024;

// Work lists for `grid` persistent CTAs over N heads x `units` query units. A
// unit t costs min(2 t + 2, nkv) key tiles when causal (nkv otherwise) plus one
// for its pipeline fill and epilogue. Heads are split into contiguous groups
// whose K and V fit kGroupKvBytes; within a group the units go heaviest first,
// and each goes to the CTA with the least work so far (lowest index on ties).
void build_table(SchedTable& tab, int64_t N, int units, int nkv, bool causal, int grid, double kv_bytes_per_head) {
  tab.count = 0;
  const int64_t total = N * units;
  if (grid <= 0 || grid > kSchedMaxGrid || total <= grid || total > kSchedMaxItems || N > 65535 || units > 65535)
    return;
  int groups = (int)std::ceil((double)N * kv_bytes_per_head / kGroupKvBytes);
  groups = std::max(1, std::min(groups, (int)N));
  std::vector<std::vector<unsigned int>> lists((size_t)grid);
  using Slot = std::pair<double, int>;  // work so far, CTA
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int c = 0; c < grid; ++c) heap.push({0.0, c});
  for (int g = 0; g < groups; ++g) {
    const int64_t h0 = N * g / groups, h1 = N * (g + 1) / groups;
    for (int t = units - 1; t >= 0; --t) {
      const double cost = (causal ? std::min(2 * t + 2, nkv) : nkv) + 1.0;
      for (int64_t n = h0; n < h1; ++n) {
        const Slot s = heap.top();
        heap.pop();
        lists[(size_t)s.second].push_back((unsigned int)(n << 16) | (unsigned int)t);
        heap.push({s.first + cost, s.second});
      }
    }
  }
  int k = 0;
  for (int c = 0; c < grid; ++c) {
    tab.start[c] = (unsigned short)k;
    for (unsigned int e : lists[(size_t)c]) tab.item[k++] = e;
  }
  tab.start[grid] = (unsigned short)k;
  tab.count = k;
}

// The table for one problem shape, built once and kept (a few shapes at most in
// practice; the cache is emptied if it ever grows past 64 entries).
SchedTable sched_table(int64_t N, int units, int nkv, bool causal, int grid, double kv_bytes_per_head) {
  using Key = std::tuple<int64_t, int, int, int, int, double>;
  static std::mutex mu;
  static std::map<Key, std::unique_ptr<SchedTable>> cache;
  const Key key{N, units, nkv, (int)causal, grid, kv_bytes_per_head};
  std::lock_guard<std::mutex> lock(mu);
  auto f = cache.find(key);
  if (f == cache.end()) {
    if (cache.size() >= 64) cache.clear();
    auto t = std::make_unique<SchedTable>();
    build_table(*t, N, units, nkv, causal, grid, kv_bytes_per_head);
    f = cache.emplace(key, std::move(t)).first;
  }
  return *f->second;
}

// [N, S, d] row-major 16-bit tensor, boxes of 64 features x `rows` rows x 1 head.
bool make_map(CUtensorMap* m, const void* ptr, int64_t N, int S, int d, bool f16, int rows = kBM) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)S, (cuuint64_t)N};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)S * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// d = 32 runs on the 64-wide kernel: the tensor maps describe the real
// 32-feature rows, TMA fills features 32-63 of every box with zeros (they add
// nothing to Q K^T and give O columns that are never stored).
template <int D, bool F16>
cudaError_t tc_launch(const AttnProblem& p, cudaStream_t st) {
  using C = TcCfg<D>;
  constexpr int smem = D == 64 ? Tc64::SMEM : C::SMEM;
  // per-device attribute, so it is set on every launch
  cudaError_t e;
  if constexpr (D == 64)
    e = cudaFuncSetAttribute(attn_tc64_kernel<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  else
    e = cudaFuncSetAttribute(attn_tc_kernel<D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int dreal = p.d;  // D, or 32 with D = 64
  CUtensorMap mq, mk, mv;
  CUtensorMap mo;  // output boxes: 64 columns x the 32 rows of one softmax warp
  if (!make_map(&mq, p.q, p.N, p.S, dreal, F16) || !make_map(&mk, p.k, p.N, p.S, dreal, F16) ||
      !make_map(&mv, p.v, p.N, p.S, dreal, F16) || !make_map(&mo, p.o, p.N, p.S, dreal, F16, 32))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int units = (p.S + kPairRows - 1) / kPairRows;
  const int64_t items = (int64_t)units * p.N;
  const int64_t grid = items < sms ? items : sms;  // persistent: at most one CTA per SM
  const SchedTable tab = sched_table(p.N, units, (p.S + kBN - 1) / kBN, p.causal != 0, (int)grid,
                                     2.0 * p.S * dreal * 2.0);
  if constexpr (D == 64)
    attn_tc64_kernel<F16><<<(unsigned)grid, kThreadsTC, smem, st>>>(
        mq, mk, mv, tab, static_cast<uint8_t*>(p.o), p.lse, dreal, (int)p.N, p.S, p.causal,
        p.scale * 1.4426950408889634f, kDefaultWaitLimitNs);
  else
    attn_tc_kernel<D, F16><<<(unsigned)grid, kThreadsTC, smem, st>>>(
        mq, mk, mv, mo, tab, static_cast<uint8_t*>(p.o), p.lse, dreal, (int)p.N, p.S, p.causal,
        p.scale * 1.4426950408889634f, kDefaultWaitLimitNs);
  return cudaGetLastError();
}

template <bool F16>
cudaError_t tc256_launch(const AttnProblem& p, cudaStream_t st) {
  using C = Tc256;
  cudaError_t e = cudaFuncSetAttribute(attn_tc256_kernel<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mv;
  CUtensorMap mo;  // output boxes: 64 columns x the 32 rows of one softmax warp
  if (!make_map(&mq, p.q, p.N, p.S, C::D, F16, kBM) || !make_map(&mk, p.k, p.N, p.S, C::D, F16, kBN256) ||
      !make_map(&mv, p.v, p.N, p.S, C::D, F16, kBN256) || !make_map(&mo, p.o, p.N, p.S, C::D, F16, 32))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int units = (p.S + kBM - 1) / kBM;
  const int64_t items = (int64_t)units * p.N;
  const int64_t grid = items < sms ? items : sms;
  const SchedTable tab = sched_table(p.N, units, (p.S + kBN256 - 1) / kBN256, p.causal != 0, (int)grid,
                                     2.0 * p.S * C::D * 2.0);
  attn_tc256_kernel<F16><<<(unsigned)grid, kThreads256, C::SMEM, st>>>(
      mq, mk, mv, mo, tab, static_cast<uint8_t*>(p.o), p.lse, (int)p.N, p.S, p.causal, p.scale * 1.4426950408889634f,
      kDefaultWaitLimitNs);
  return cudaGetLastError();
}

}  // namespace

int tc_check(int S, int d, int dtype) {
  (void)S;
  if (d != 32 && d != 64 && d != 128 && d != 256) return KB_ERR_UNSUPPORTED;
  if (dtype != KB_BF16 && dtype != KB_F16) return KB_ERR_UNSUPPORTED;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KB_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return KB_ERR_CUDA;
  const int need = d == 256 ? Tc256::SMEM : (d == 128 ? TcCfg<128>::SMEM : Tc64::SMEM);  // d = 32: the 64 kernel
  return need <= optin ? KB_OK : KB_ERR_UNSUPPORTED;
}

// The work lists tc_launch / tc256_launch build for these arguments (host only).
int tc_work_lists(int64_t N, int S, int d, bool causal, int grid, int* start, unsigned int* items, int cap,
                  int* count) {
  const bool wide = d == 256;
  const int units = wide ? (S + kBM - 1) / kBM : (S + kPairRows - 1) / kPairRows;
  const int nkv = wide ? (S + kBN256 - 1) / kBN256 : (S + kBN - 1) / kBN;
  const SchedTable tab = sched_table(N, units, nkv, causal, grid, 2.0 * S * d * 2.0);
  *count = tab.count;
  if (tab.count == 0) return KB_OK;
  if (cap < tab.count) return KB_ERR_INVALID_ARG;
  for (int c = 0; c <= grid; ++c) start[c] = tab.start[c];
  for (int k = 0; k < tab.count; ++k) items[k] = tab.item[k];
  return KB_OK;
}

cudaError_t launch_tc(const AttnProblem& p, cudaStream_t st) {
  const bool f16 = p.dtype == KB_F16;
  if (p.d == 128) return f16 ? tc_launch<128, true>(p, st) : tc_launch<128, false>(p, st);
  if (p.d == 64 || p.d == 32) return f16 ? tc_launch<64, true>(p, st) : tc_launch<64, false>(p, st);
  if (p.d == 256) return f16 ? tc256_launch<true>(p, st) : tc256_launch<false>(p, st);
  return cudaErrorInvalidValue;
}

cudaError_t read_and_clear_error_word(unsigned int* out, cudaStream_t st) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_kb_error_word, sizeof(unsigned int), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  if ((e = cudaMemcpyToSymbolAsync(g_kb_error_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st)) !=
      cudaSuccess)
    return e;
  return cudaStreamSynchronize(st);
}

cudaError_t launch_selftest_timeout(unsigned long long limit_ns, cudaStream_t st) {
  selftest_timeout_kernel<<<1, 32, 0, st>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t tc_binary_version(int* out) {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, attn_tc_kernel<128, false>);
  if (e == cudaSuccess) *out = a.binaryVersion;
  return e;
}

}  // namespace kb
