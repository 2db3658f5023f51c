/*
 * Sanitizer driver for the library's host-only logic (test infrastructure):
 * linked with libkbattn's objects built under AddressSanitizer and
 * UndefinedBehaviorSanitizer, it exercises the calls that never reach a
 * device -- argument validation of every attention entry point, the
 * workspace sizing, the tensor-core path's per-CTA work lists, the Q15 exp
 * table, the status strings -- with exactly sized heap buffers, so an
 * out-of-bounds access, an overflow or another undefined operation stops the
 * run. No call here launches a kernel: every attention call is given an
 * argument that validation rejects before any CUDA call. Exit status: 0 when
 * every check passed.
 */
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "kbattn.h"

static int failures = 0;
#define CHECK(c)                                                      \
  do {                                                                \
    if (!(c)) {                                                       \
      std::fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
      ++failures;                                                     \
    }                                                                 \
  } while (0)

static void* const FAKE = reinterpret_cast<void*>(static_cast<uintptr_t>(1) << 20);

// Work lists: sizing call, exact-size buffers, every unit exactly once.
static void work_lists(long long N, int S, int d, int causal, int grid) {
  int count = -1;
  int* start0 = static_cast<int*>(std::malloc(sizeof(int) * (grid + 1)));
  unsigned int dummy = 0;
  int st = kb_attn_work_lists(N, S, d, causal, grid, start0, &dummy, 0, &count);
  std::free(start0);
  if (st == KB_OK) {
    CHECK(count == 0);  // the kernel orders the units itself
    return;
  }
  CHECK(st == KB_ERR_INVALID_ARG && count > 0);
  int* start = static_cast<int*>(std::malloc(sizeof(int) * (grid + 1)));
  unsigned int* items = static_cast<unsigned int*>(std::malloc(sizeof(unsigned int) * count));
  int count2 = -1;
  CHECK(kb_attn_work_lists(N, S, d, causal, grid, start, items, count, &count2) == KB_OK && count2 == count);
  const int rows = d == 256 ? 128 : 256;
  const long long units = (S + rows - 1) / rows;
  CHECK(count == N * units);
  CHECK(start[0] == 0 && start[grid] == count);
  std::vector<int> seen(static_cast<size_t>(N * units), 0);
  for (int c = 0; c < grid; ++c) {
    CHECK(start[c] <= start[c + 1]);
    for (int e = start[c]; e < start[c + 1]; ++e) {
      const long long n = items[e] >> 16, t = items[e] & 0xFFFFu;
      CHECK(n < N && t < units);
      if (n < N && t < units) ++seen[static_cast<size_t>(n * units + t)];
    }
  }
  for (int x : seen) CHECK(x == 1);
  std::free(start);
  std::free(items);
}

static void validation() {
  const float scale = 0.125f;
  // one rejected argument per call: null, misaligned, sizes, flags, scale, dtype, variant
  CHECK(kb_attn_fwd(nullptr, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, scale, KB_F32, KB_FLASH, nullptr) == KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd(FAKE, static_cast<char*>(FAKE) + 4, FAKE, FAKE, 1, 1, 64, 64, 0, scale, KB_F32, KB_FLASH, nullptr) ==
        KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 0, 1, 64, 64, 0, scale, KB_F32, KB_FLASH, nullptr) == KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 2, scale, KB_F32, KB_FLASH, nullptr) == KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, NAN, KB_F32, KB_FLASH, nullptr) == KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, -1.f, KB_F32, KB_FLASH, nullptr) == KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, scale, 9, KB_FLASH, nullptr) == KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, scale, KB_F32, 17, nullptr) == KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 48, 0, scale, KB_F32, KB_FLASH, nullptr) == KB_ERR_UNSUPPORTED);
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, scale, KB_F32, KB_TC, nullptr) == KB_ERR_UNSUPPORTED);
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, scale, KB_BF16, KB_FLASH, nullptr) == KB_ERR_UNSUPPORTED);
  // sizes at the edges of the integer ranges
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 65536, 65536, 64, 64, 0, scale, KB_F32, KB_FLASH, nullptr) ==
        KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 2147483647, 2147483647, 2147483647, 256, 1, scale, KB_BF16, KB_TC,
                    nullptr) == KB_ERR_INVALID_ARG);
  for (int variant : {KB_NAIVE, KB_FUSED, KB_FLASH, KB_TC})
    for (int S : {2147483647, 2147483647 - 255})
      CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 1, 1, S, 64, 1, scale, variant == KB_TC ? KB_BF16 : KB_F32, variant,
                        nullptr) == KB_ERR_UNSUPPORTED);
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 1, 1, 70000, 64, 1, 0.125f, KB_Q15, KB_FIXEDPOINT, nullptr) ==
        KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 1, 1e9f, KB_Q15, KB_FIXEDPOINT, nullptr) == KB_ERR_INVALID_ARG);
  // the other entry points share the validation
  float ms[4];
  CHECK(kb_attn_fwd_ws(FAKE, FAKE, FAKE, nullptr, 1, 1, 64, 64, 0, scale, KB_F32, KB_NAIVE, nullptr, FAKE, 1 << 20) ==
        KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd_lse(FAKE, FAKE, FAKE, FAKE, nullptr, 1, 1, 64, 64, 0, scale, KB_F32, KB_FLASH, nullptr) ==
        KB_ERR_INVALID_ARG);
  CHECK(kb_attn_bench(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, scale, KB_F32, KB_FLASH, nullptr, nullptr, 0, 0, 0, ms) ==
        KB_ERR_INVALID_ARG);
  CHECK(kb_attn_bench_graph(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, scale, KB_F32, KB_FLASH, nullptr, nullptr, 0, 0, 1,
                            1, ms) == KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd_host(FAKE, FAKE, nullptr, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 0, scale, KB_F32, KB_FLASH,
                         nullptr) == KB_ERR_INVALID_ARG);
  CHECK(kb_attn_fwd_host(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 96, 0, scale, KB_F32, KB_FLASH,
                         nullptr) == KB_ERR_UNSUPPORTED);
  CHECK(kb_attn_fwd_naive_noalloc(FAKE, FAKE, FAKE, FAKE, 1, 8, 1025, 64, 0, scale, nullptr) == KB_ERR_NO_MEMORY);
  CHECK(kb_triad(static_cast<float*>(FAKE), nullptr, static_cast<float*>(FAKE), 1.f, 16, 256, nullptr) ==
        KB_ERR_INVALID_ARG);
  CHECK(kb_triad(static_cast<float*>(FAKE), static_cast<float*>(FAKE), static_cast<float*>(FAKE), 1.f, 16, 100,
                 nullptr) == KB_ERR_INVALID_ARG);
  CHECK(kb_hbm_bench(7, nullptr, nullptr, nullptr, 0.f, 0, 0, nullptr, nullptr, 0, 1, ms) == KB_ERR_INVALID_ARG);
  CHECK(kb_binary_version(nullptr) == KB_ERR_INVALID_ARG);
  CHECK(kb_device_info(0, nullptr) == KB_ERR_INVALID_ARG);
}

static void sizing() {
  const int dtypes[] = {KB_F32, KB_BF16, KB_F16, KB_Q15};
  const int ds[] = {32, 64, 128, 256, 48};
  for (int variant = KB_AUTO; variant <= KB_FIXEDPOINT + 1; ++variant)
    for (int dt : dtypes)
      for (int d : ds)
        for (int S : {1, 63, 1024, 65536})
          (void)kb_attn_workspace_bytes(2, 3, S, d, dt, variant);
  CHECK(kb_attn_workspace_bytes(1, 8, 1024, 64, KB_F32, KB_NAIVE) == 8ull * 1024 * 1024 * 4);
  CHECK(kb_attn_workspace_bytes(1, 1, 64, 64, KB_BF16, KB_TC) == 0);
  CHECK(kb_attn_workspace_bytes(0, 1, 64, 64, KB_F32, KB_NAIVE) == 0);
  CHECK(kb_attn_workspace_bytes(65536, 65536, 65536, 64, KB_F32, KB_NAIVE) == 0);  // not addressable
  // the longest sequence accepted, and one past it
  const int max_seq = 2147483647 - 256;
  for (int d : {32, 64, 128, 256})
    for (int variant : {KB_NAIVE, KB_FLASH, KB_FUSED, KB_TC}) {
      (void)kb_attn_workspace_bytes(1, 1, max_seq, d, d == 256 ? KB_BF16 : KB_F32, variant);
      CHECK(kb_attn_workspace_bytes(1, 1, max_seq + 1, d, KB_F32, variant) == 0);
    }
}

int main() {
  validation();
  sizing();
  // the benchmarked shapes, ragged lengths, every d, causal and not, odd grids, fallbacks
  const long long Ns[] = {1, 3, 24, 64, 192};
  const int Ss[] = {1, 129, 300, 2048, 4096};
  const int dsz[] = {32, 64, 128, 256};
  const int grids[] = {1, 7, 152, 256, 300};
  for (long long N : Ns)
    for (int S : Ss)
      for (int d : dsz)
        for (int causal = 0; causal < 2; ++causal)
          for (int grid : grids) work_lists(N, S, d, causal, grid);
  work_lists(32, 16384, 128, 1, 152);
  work_lists(4096, 4096, 128, 1, 152);
  work_lists(1, 2147483647 - 256, 128, 1, 152);
  work_lists(1, 2147483647 - 256, 256, 0, 152);
  {
    int start[3], count = 0;
    unsigned int items[4];
    CHECK(kb_attn_work_lists(1, 2147483647 - 255, 128, 1, 2, start, items, 4, &count) == KB_ERR_INVALID_ARG);
  }
  unsigned short* tab = static_cast<unsigned short*>(std::malloc(64 * sizeof(unsigned short)));
  CHECK(kb_q15_exp_table(tab) == KB_OK && tab[0] == 32768);
  std::free(tab);
  CHECK(kb_q15_exp_table(nullptr) == KB_ERR_INVALID_ARG);
  for (int s = -2; s < 9; ++s) CHECK(kb_status_string(s) != nullptr && std::strlen(kb_status_string(s)) > 0);
  CHECK(kb_version() >= 100);
  if (failures) std::fprintf(stderr, "%d checks failed\n", failures);
  else std::printf("host sanitizer driver: all checks passed\n");
  return failures ? 1 : 0;
}
