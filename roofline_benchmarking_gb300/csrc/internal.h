// internal.h -- declarations shared by the library's translation units (not
// part of the ABI; the public interface is include/kbattn.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kbattn.h"

namespace kb {

// Attention problem as validated by the API layer.
struct AttnProblem {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  int64_t N;  // B*H
  int S;
  int d;
  int causal;
  float scale;
  int dtype;
  float* lse = nullptr;  // optional [N, S] fp32 log-sum-exp of the score rows
  float* work = nullptr;  // fp32 flash: the split tiles' partial states (null: no split)
};

// Launchers return a cudaError_t from the launch (or cudaSuccess).
cudaError_t launch_flash_f32(const AttnProblem& p, cudaStream_t st);
cudaError_t launch_fused_f32(const AttnProblem& p, cudaStream_t st);
cudaError_t launch_naive_f32(const AttnProblem& p, float* scores, cudaStream_t st);
size_t naive_workspace_bytes(int64_t N, int S);
// fp32 flash, causal: the heavier half of the query tiles is split over two blocks
// when the grid is small (a single wave of blocks would otherwise wait on the
// heaviest tile); these give the decision and the partial-state bytes it needs.
bool flash_wants_split(int64_t N, int S, int causal);
size_t flash_split_bytes(int64_t N, int S, int d);
// 0 if the fused-row kernel can run S keys on the current device, else an error code.
int fused_f32_check(int S, int d);

cudaError_t launch_tc(const AttnProblem& p, cudaStream_t st);
int tc_check(int S, int d, int dtype);
// cudaFuncAttributes::binaryVersion (10 * major + minor) of the tensor-core
// kernel's code on the current device.
cudaError_t tc_binary_version(int* out);
// The per-CTA work lists of the tensor-core path (host only); *count = 0 when
// the kernel falls back to its snake order.
int tc_work_lists(int64_t N, int S, int d, bool causal, int grid, int* start, unsigned int* items, int cap,
                  int* count);

// Q15 fixed-point path: launcher, the scale limit (scale*log2(e)*2^16 <= 2^30)
// and the 64-entry exp table it uses.
cudaError_t launch_q15(const AttnProblem& p, cudaStream_t st);
bool q15_scale_ok(float scale);
int q15_exp_table(unsigned short* out);

cudaError_t launch_triad(float* a, const float* b, const float* c, float s, size_t n, int block,
                         cudaStream_t st);
cudaError_t launch_copy(float* a, const float* b, size_t n, int block, cudaStream_t st);
cudaError_t launch_fill(float* a, float s, size_t n, int block, cudaStream_t st);
cudaError_t launch_read(const float* b, size_t n, float* out, int block, cudaStream_t st);

// Device error word (bounded waits that ran out).
cudaError_t read_and_clear_error_word(unsigned int* out, cudaStream_t st);
cudaError_t launch_selftest_timeout(unsigned long long limit_ns, cudaStream_t st);

// Per-thread record of the last CUDA error returned as KB_ERR_CUDA.
void set_last_cuda_error(cudaError_t e);

// The API layer's argument validation (no CUDA call) and device gate.
int validate_attention(const void* q, const void* k, const void* v, const void* o, int B, int H, int S, int d,
                       int causal, float scale, int dtype, int variant, int* resolved);
int check_current_device();

}  // namespace kb
