/*
 * ThreadSanitizer driver for the library's host-only logic (test
 * infrastructure): linked with libkbattn's objects built under
 * -fsanitize=thread, it calls the host-only entry points from several threads
 * at once -- the tensor-core path's work lists (whose per-shape cache is shared
 * by every caller and emptied when it grows past its bound), argument
 * validation that rejects each call before any CUDA call, the Q15 exp table,
 * the status strings and the per-thread last CUDA error -- so that a data race
 * in the shared host state stops the run. No call launches a kernel or needs a
 * GPU. Exit status: 0 when every check passed.
 */
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <thread>
#include <vector>

#include "kbattn.h"

static std::atomic<int> failures{0};
#define CHECK(c)                                                              \
  do {                                                                        \
    if (!(c)) {                                                               \
      std::fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c);    \
      failures.fetch_add(1);                                                  \
    }                                                                         \
  } while (0)

struct Shape {
  long long N;
  int S, d, causal, grid;
};

// Fills the lists of one shape and checks that every (head, query unit) pair
// appears exactly once across the CTAs.
static void work_lists(const Shape& s) {
  int count = -1;
  std::vector<int> start((size_t)s.grid + 1);
  unsigned int dummy = 0;
  int st = kb_attn_work_lists(s.N, s.S, s.d, s.causal, s.grid, start.data(), &dummy, 0, &count);
  if (st == KB_OK) {
    CHECK(count == 0);
    return;
  }
  CHECK(st == KB_ERR_INVALID_ARG && count > 0);
  std::vector<unsigned int> items((size_t)count);
  int count2 = -1;
  CHECK(kb_attn_work_lists(s.N, s.S, s.d, s.causal, s.grid, start.data(), items.data(), count, &count2) == KB_OK);
  CHECK(count2 == count);
  CHECK(start[0] == 0 && start[(size_t)s.grid] == count);
  const int rows = s.d == 256 ? 128 : 256;
  const long long units = (s.S + rows - 1) / rows;
  CHECK((long long)count == s.N * units);
}

static void worker(int id, const std::vector<Shape>* shapes, int iters) {
  unsigned int x = 2463534242u + 977u * (unsigned)id;
  void* const fake = reinterpret_cast<void*>(static_cast<uintptr_t>(1) << 20);
  for (int it = 0; it < iters; ++it) {
    x ^= x << 13;
    x ^= x >> 17;
    x ^= x << 5;
    work_lists((*shapes)[x % shapes->size()]);
    // rejected before any CUDA call: a null output pointer, an unsupported head dimension
    CHECK(kb_attn_fwd(fake, fake, fake, nullptr, 1, 1, 64, 64, 0, 0.125f, KB_F32, KB_FLASH, nullptr) ==
          KB_ERR_INVALID_ARG);
    CHECK(kb_attn_fwd(fake, fake, fake, fake, 1, 1, 64, 48, 0, 0.125f, KB_BF16, KB_TC, nullptr) ==
          KB_ERR_UNSUPPORTED);
    CHECK(kb_attn_workspace_bytes(1, 2, 128, 64, KB_F32, KB_NAIVE) == (size_t)2 * 128 * 128 * 4);
    unsigned short tab[64];
    CHECK(kb_q15_exp_table(tab) == KB_OK && tab[0] == 32768u);
    CHECK(std::strlen(kb_status_string(it % 7)) > 0);
    CHECK(kb_last_cuda_error() == 0);
  }
}

int main() {
  std::vector<Shape> shapes;
  const int dims[] = {32, 64, 128, 256};
  const int seqs[] = {1, 77, 128, 300, 1000, 2048, 4096};
  const long long heads[] = {1, 3, 12, 64};
  const int grids[] = {1, 7, 152};
  for (int d : dims)
    for (int S : seqs)
      for (long long N : heads)
        for (int c = 0; c < 2; ++c) shapes.push_back({N, S, d, c, grids[(d + S + (int)N + c) % 3]});
  // more shapes than the work-list cache keeps, so that it is emptied while other threads use it
  const int nthreads = 8, iters = 150;
  std::vector<std::thread> ts;
  for (int t = 0; t < nthreads; ++t) ts.emplace_back(worker, t, &shapes, iters);
  for (auto& t : ts) t.join();
  if (failures.load() != 0) {
    std::fprintf(stderr, "%d checks failed\n", failures.load());
    return 1;
  }
  std::printf("all checks passed (%zu shapes, %d threads x %d iterations)\n", shapes.size(), nthreads, iters);
  return 0;
}
