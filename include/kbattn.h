/*
 * kbattn.h -- C ABI of libkbattn, scaled-dot-product attention forward and
 * the STREAM Triad bandwidth ceiling on one GB300 (sm_103a).
 *
 * No CUDA or PyTorch type appears here: a stream is passed as `void*` (a
 * cudaStream_t; NULL is the legacy default stream) and every tensor as a
 * plain device pointer.
 *
 * The problem definition follows the kbench page ("kbench -- Transformer
 * Attention Micro-benchmark Harness"):
 *  - section "Implementation details / The three GPU kernels": all kernels
 *    compute O = softmax(Q K^T / sqrt(d)) V over a flattened (batch*heads)
 *    axis laid out [head, seq, dim] row-major; here the scale is a parameter;
 *  - "Architecture" diagram: one shared problem definition behind a dispatch
 *    call run_attention(kernel, cfg) with CUDA-event timing in the launch layer;
 *  - sequence diagram "One MCU measurement": the request carries seq, dim and
 *    a causal flag;
 *  - section "Implementation details", the paragraph on gpu/src/launch.cu:
 *    events around the kernel only, no host<->device copy in the window,
 *    configurable warm-up, per-iteration times.
 * The Triad follows the TileOPs "Hardware Microbenchmarks" README, section
 * "HBM Bandwidth" and "Methodology": a[i] = b[i] + s*c[i], float4 vectorised,
 * cudaEvent timing, block sizes 128/256/512.
 *
 * Conventions for every call:
 *  - Layout: q, k, v, o are contiguous [B, H, S, d] row-major (head
 *    n = b*H + h, then query/key row, then feature), i.e. [N, S, d].
 *  - Causal: key j is visible to query i iff j <= i.
 *  - Ownership: the caller owns every pointer. The library never frees,
 *    retains or synchronises caller memory or streams, except where a call
 *    says so (the *_bench calls synchronise on their own events).
 *  - Alignment: device pointers must be 16-byte aligned.
 *  - Errors: every call returns a kb_status; no exception or abort crosses the
 *    ABI. Arguments are validated before any launch, so a rejected call has
 *    no effect on the device. KB_ERR_CUDA leaves the CUDA error code in
 *    kb_last_cuda_error() (per thread).
 *  - Asynchrony: launches are asynchronous on `stream`; results are valid
 *    once the stream reaches that point. Waits inside the kernels are
 *    bounded; a wait that runs out sets a device error word that
 *    kb_check_device_error() reports as KB_ERR_TIMEOUT.
 */
#ifndef KBATTN_H
#define KBATTN_H

#include <stddef.h>
#include <stdint.h>

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define KB_API __attribute__((visibility("default")))
#else
#define KB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KB_OK = 0,
  KB_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad scale, overflow */
  KB_ERR_UNSUPPORTED = 2, /* valid request the library has no kernel for */
  KB_ERR_CUDA = 3,        /* a CUDA runtime call failed; see kb_last_cuda_error() */
  KB_ERR_NO_MEMORY = 4,   /* workspace too small or allocation failed */
  KB_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out */
  KB_ERR_NO_DEVICE = 6    /* no usable sm_103 device */
} kb_status;

/*
 * Element types. KB_Q15 is int16 fixed point, value = x / 2^15 (the kbench
 * page's fixed-point path, section "CPU reference + cache profiling").
 */
typedef enum { KB_F32 = 0, KB_BF16 = 1, KB_F16 = 2, KB_Q15 = 3 } kb_dtype;

/*
 * Variants (kbench page, "The three GPU kernels"; the tensor-core variant is
 * this library's sm_103a kernel):
 *  KB_NAIVE : three passes, the N*S*S fp32 score matrix goes through global
 *             memory (score GEMM, row softmax in place, P*V GEMM). fp32 only.
 *  KB_FUSED : a block per query row (or per 2, 4 or 8 consecutive rows where
 *             they fit), the S-length score rows kept in shared memory beside
 *             two 64-key staging buffers. fp32 only; UNSUPPORTED when one row's
 *             S*4 bytes and the buffers exceed the shared memory a block may
 *             use (on GB300: S up to about 39,000 at d = 128, 47,000 at d = 64,
 *             51,000 at d = 32).
 *  KB_FLASH : tiled, online softmax (running max and denominator), the score
 *             matrix never materialised; CUDA cores. fp32 only.
 *  KB_TC    : tiled, online softmax on the 5th-generation tensor cores
 *             (tcgen05 MMAs into tensor memory, TMA-staged tiles). bf16/f16.
 *  KB_FIXEDPOINT : the Q15 fixed-point path (kbench page, "CPU reference +
 *             cache profiling" and "ARM Cortex-M4 firmware"), integer
 *             arithmetic only, defined bit for bit. KB_Q15 only. Q15 inputs;
 *             score = floor(floor(sum_c q_c*k_c / 2^14) * C / 2^16) in Q15.16
 *             base-2 units with C = round(scale*log2(e)*2^16); keys in tiles of
 *             32 from key 0 with an online-rescaled softmax whose weights come
 *             from a 64-entry table T[f] = round(2^15 * 2^(-f/64))
 *             (2^(-t) = T[top 6 fraction bits of t] >> floor(t), 0 once
 *             floor(t) >= 16); l and the 64-bit accumulators are rescaled by
 *             floor(x * 2^(-dm) / 2^15) when the running maximum rises by dm;
 *             o = acc / l rounded to nearest (halves away from zero),
 *             saturated to int16. Requires S <= 65536 and
 *             scale*log2(e)*2^16 <= 2^30 (else KB_ERR_INVALID_ARG).
 *  KB_AUTO  : KB_TC for bf16/f16, KB_FLASH for fp32, KB_FIXEDPOINT for Q15.
 */
typedef enum { KB_AUTO = 0, KB_NAIVE = 1, KB_FUSED = 2, KB_FLASH = 3, KB_TC = 4,
               KB_FIXEDPOINT = 5 } kb_variant;

/* Device properties used by the roofline peak formulas. */
typedef struct {
  int device;               /* CUDA ordinal */
  int cc_major, cc_minor;   /* compute capability */
  int sm_count;             /* streaming multiprocessors */
  int sm_clock_khz;         /* cudaDevAttrClockRate */
  int mem_clock_khz;        /* cudaDevAttrMemoryClockRate */
  int mem_bus_width_bits;   /* cudaDevAttrGlobalMemoryBusWidth */
  int l2_bytes;             /* L2 cache size */
  int smem_per_block_optin; /* opt-in shared memory per block */
  int smem_per_sm;          /* shared memory per SM */
  size_t total_mem_bytes;   /* device memory */
  char name[256];           /* device name, NUL-terminated */
} kb_device_info_t;

/*
 * kb_attn_fwd -- O = softmax(Q K^T * scale [+ causal mask]) V.
 *   q, k, v : const device pointers, [B, H, S, d] of `dtype`
 *   o       : device pointer, [B, H, S, d] of `dtype`, written in full
 *             (bf16/f16 outputs are rounded to nearest even from fp32)
 *   B, H, S : >= 1; B*H*S*d must fit in int64 and B*H in int32;
 *             S <= 2^31 - 257 (longer -> KB_ERR_UNSUPPORTED)
 *   d       : head dimension: 32, 64 or 128, and 256 for KB_TC (others -> UNSUPPORTED)
 *   causal  : 0 or 1
 *   scale   : finite and > 0 (callers normally pass 1/sqrt(d))
 *   dtype   : kb_dtype of q, k, v and o
 *   variant : kb_variant; see the support matrix above
 *   stream  : cudaStream_t or NULL
 * KB_TC supports d = 32 (run by the d = 64 kernel on tiles whose features
 * 32-63 are zero-filled by TMA), 64, 128 and 256 (one 128-row query tile per
 * CTA); KB_NAIVE, KB_FUSED and KB_FLASH support d = 32, 64 and 128.
 * KB_NAIVE needs N*S*S*4 bytes of workspace, and a causal KB_FLASH call on a
 * small grid the partial states of its split query tiles (see
 * kb_attn_workspace_bytes): this call takes them from a per-device cache that
 * it grows with cudaMalloc, synchronising the device first when it replaces a
 * smaller buffer (so it may allocate and block); calls on different streams
 * share that cache and must not overlap on the device. The cache's lock is
 * held until a call's kernels are enqueued, so a call from another host thread
 * that grows the cache never frees a buffer under a launch still being made.
 * kb_attn_fwd_ws lets the caller supply the workspace instead.
 */
KB_API int kb_attn_fwd(const void* q, const void* k, const void* v, void* o,
                int B, int H, int S, int d, int causal, float scale,
                int dtype, int variant, void* stream);

/*
 * kb_attn_fwd_lse -- kb_attn_fwd that also writes the log-sum-exp of every
 * score row, lse[n, i] = log(sum over visible keys j of exp(scale * q_i.k_j)),
 * the natural log of the softmax denominator (the flash kernel's running max m
 * and denominator l give it as m + log l; kbench page, "The three GPU kernels").
 *   lse     : device pointer, [B, H, S] fp32 (4-byte aligned), written in full
 *   others  : as kb_attn_fwd
 * Supported for KB_TC and KB_FLASH (and KB_AUTO); KB_NAIVE and KB_FUSED return
 * KB_ERR_UNSUPPORTED.
 */
KB_API int kb_attn_fwd_lse(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int S, int d, int causal, float scale,
                           int dtype, int variant, void* stream);

/*
 * kb_attn_fwd_host -- kb_attn_fwd from host memory to host memory: on
 * `stream`, copies Q, K and V from the host buffers into the caller's device
 * buffers, runs the forward pass there, and copies O back into o_host (the
 * kbench page's launch layer keeps these copies outside its timed window; this
 * call is the whole round trip a host caller makes).
 *   q_host, k_host, v_host : host pointers, [B, H, S, d] of `dtype`, read
 *   o_host  : host pointer, [B, H, S, d] of `dtype`, written
 *   q_dev, k_dev, v_dev, o_dev : device pointers as in kb_attn_fwd (the
 *             caller's staging buffers; overwritten)
 *   others  : as kb_attn_fwd
 * Asynchronous: o_host holds the result once `stream` reaches the end of the
 * call. Page-locked host buffers let the copies run asynchronously and overlap
 * other streams' work; with pageable buffers the CUDA runtime may stage them and
 * block the calling thread. The host buffers must stay valid until then.
 * Validation, workspace and errors are those of kb_attn_fwd (plus
 * KB_ERR_INVALID_ARG for a null host pointer); copies are issued only after
 * the arguments have been validated.
 */
KB_API int kb_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                            void* q_dev, void* k_dev, void* v_dev, void* o_dev,
                            int B, int H, int S, int d, int causal, float scale,
                            int dtype, int variant, void* stream);

/* Workspace bytes kb_attn_fwd_ws uses: KB_NAIVE's N*S*S*4 score matrix; for
 * KB_FLASH, the partial states of its split causal query tiles (the heavier
 * half of them runs as two blocks over two key ranges when N * ceil(S/64) is
 * at most twice the SM count, and a merge kernel combines the halves); 0 for
 * the other variants and for an invalid request. */
KB_API size_t kb_attn_workspace_bytes(int B, int H, int S, int d, int dtype, int variant);

/* kb_attn_fwd with a caller-owned device workspace of ws_bytes bytes (16-byte
 * aligned). KB_NAIVE: KB_ERR_NO_MEMORY if ws_bytes < kb_attn_workspace_bytes(...).
 * KB_FLASH: with less (or none), its causal tiles simply run unsplit.
 * The library allocates nothing in this call. */
KB_API int kb_attn_fwd_ws(const void* q, const void* k, const void* v, void* o,
                   int B, int H, int S, int d, int causal, float scale,
                   int dtype, int variant, void* stream,
                   void* workspace, size_t ws_bytes);

/*
 * kb_attn_bench -- `warmup` untimed calls, then `iters` calls each bracketed
 * by CUDA events on `stream`; ms_per_iter[t] (host array of `iters` floats)
 * receives the t-th call's device time. Synchronises on its own events only.
 * Uses kb_attn_fwd_ws when workspace != NULL, else kb_attn_fwd.
 */
KB_API int kb_attn_bench(const void* q, const void* k, const void* v, void* o,
                  int B, int H, int S, int d, int causal, float scale,
                  int dtype, int variant, void* stream,
                  void* workspace, size_t ws_bytes,
                  int warmup, int iters, float* ms_per_iter);

/*
 * kb_attn_bench_graph -- the kbench page, section "Implementation details"
 * (launch overhead of tiny problems, measured with the launches captured in
 * a CUDA graph): `launches` consecutive kb_attn_fwd(_ws) calls are captured
 * into one CUDA graph on a private stream, then the graph is launched on
 * `stream` `warmup` times untimed and `iters` times between CUDA events;
 * ms_per_graph[t] (host array of `iters` floats) receives the t-th graph's
 * device time, so one call costs ms_per_graph[t] / launches.
 *   launches : 1 ... 100000 (else KB_ERR_INVALID_ARG)
 * Before capturing, one plain call runs and `stream` is synchronised (it
 * validates the arguments and sets up any cached workspace). Arguments are
 * validated as in kb_attn_fwd; a failed call inside the capture ends the
 * capture and its status is returned. The graph is destroyed before return.
 */
KB_API int kb_attn_bench_graph(const void* q, const void* k, const void* v, void* o,
                               int B, int H, int S, int d, int causal, float scale,
                               int dtype, int variant, void* stream,
                               void* workspace, size_t ws_bytes,
                               int launches, int warmup, int iters, float* ms_per_graph);

/*
 * kb_triad -- STREAM Triad a[i] = b[i] + s*c[i] for i < n, fp32, computed as
 * one fused multiply-add (a single rounding of the exact value).
 *   a       : device pointer, n floats, written
 *   b, c    : const device pointers, n floats
 *   n       : element count (0 is a no-op)
 *   block   : threads per block, one of 128, 256, 512 (the TileOPs sweep) or
 *             1024 (0 picks 256)
 * Pointers must be 16-byte aligned (float4 accesses); any n is accepted, the
 * tail that is not a multiple of 4 is handled with scalar accesses.
 */
KB_API int kb_triad(float* a, const float* b, const float* c, float s, size_t n,
             int block, void* stream);

/*
 * The Triad's reference kernels (TileOPs README, "HBM Bandwidth" /
 * "Methodology": copy 1:1 read:write, read-only and write-only), float4
 * vectorised with streaming cache hints, same pointer and block rules as
 * kb_triad:
 *   kb_hbm_copy  : a[i] = b[i]                       (4 bytes read, 4 written)
 *   kb_hbm_write : a[i] = s                          (4 bytes written)
 *   kb_hbm_read  : *out = sum of b[0..n) in fp32     (4 bytes read); out is a
 *                  4-byte aligned device float that the call first zeroes on
 *                  `stream` (partial sums are fp32, so the value is exact only
 *                  where every partial sum is representable)
 */
KB_API int kb_hbm_copy(float* a, const float* b, size_t n, int block, void* stream);
KB_API int kb_hbm_write(float* a, float s, size_t n, int block, void* stream);
KB_API int kb_hbm_read(const float* b, size_t n, int block, float* out, void* stream);

typedef enum { KB_HBM_TRIAD = 0, KB_HBM_COPY = 1, KB_HBM_READ = 2, KB_HBM_WRITE = 3 } kb_hbm_op;

/*
 * kb_hbm_bench -- one of the four HBM kernels (`op`, a kb_hbm_op) timed like
 * kb_attn_bench; arguments a kernel does not use are ignored (but pointers
 * must still be valid device pointers).
 */
KB_API int kb_hbm_bench(int op, float* a, const float* b, const float* c, float s, size_t n, int block,
                        float* out, void* stream, int warmup, int iters, float* ms_per_iter);

/* kb_triad timed like kb_attn_bench. */
KB_API int kb_triad_bench(float* a, const float* b, const float* c, float s, size_t n,
                   int block, void* stream, int warmup, int iters, float* ms_per_iter);

/* Device properties of `device` (an ordinal), no launch. */
KB_API int kb_device_info(int device, kb_device_info_t* out);

/*
 * kb_check_device_error -- synchronise `stream`, then read and clear the
 * device error word of the current device. KB_ERR_TIMEOUT if a bounded wait
 * in any kernel of this library ran out since the last check, else KB_OK
 * (or KB_ERR_CUDA if synchronising failed).
 */
KB_API int kb_check_device_error(void* stream);

/*
 * kb_selftest_timeout -- launch one block whose thread waits, with the same
 * bounded wait the tensor-core kernel uses, on an mbarrier that nothing ever
 * completes; the wait gives up after `limit_ns` nanoseconds (clamped to
 * [1e3, 2e9]) and records the timeout in the device error word. Exists so
 * that the timeout path can be tested without hanging a GPU. Asynchronous.
 */
KB_API int kb_selftest_timeout(unsigned long long limit_ns, void* stream);

/*
 * Size in bytes of the library-owned score array of kb_attn_fwd_naive_noalloc:
 * 32 MiB, i.e. N*S*S <= 8388608 (for example 8 heads at S = 1024). A GPU holds
 * this array from the moment the library's module is loaded there until the
 * process exits: under CUDA's default lazy module loading that is the first
 * kb_attn_fwd_naive_noalloc call on that GPU (with CUDA_MODULE_LOADING=EAGER,
 * the library's load).
 */
#define KB_NAIVE_NOALLOC_MAX_BYTES (32u * 1024u * 1024u)

/*
 * kb_attn_fwd_naive_noalloc -- the KB_NAIVE fp32 forward (score GEMM, row
 * softmax, P*V GEMM, the N*S*S scores through global memory) that allocates
 * nothing. The pages have no counterpart: it exists for callers that cannot
 * call cudaMalloc -- a caller whose device memory is entirely reserved by its
 * own pool (an allocation would fail or fragment that pool), or a caller on a
 * latency-critical path that must not pay cudaMalloc's cost and its implicit
 * device synchronisation. The caller still passes inputs and outputs; the
 * score workspace is a fixed array inside the library.
 *   q, k, v, o, B, H, S, d, causal, scale, stream : as kb_attn_fwd, fp32 only
 * Returns KB_ERR_NO_MEMORY, before any device work, when N*S*S*4 bytes exceed
 * KB_NAIVE_NOALLOC_MAX_BYTES. Calls no cudaMalloc, cudaFree or other
 * allocating routine. The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; that lookup may
 * load the library's module and commit the 32 MiB array on the device, so
 * make the first call before the caller's own pool reserves the device's
 * memory (else it can fail with KB_ERR_CUDA), and before any stream capture.
 * The address is cached with the identity of the CUDA context; after a device
 * reset the next call looks it up again (and commits the array again). All
 * calls share the one array and it keeps the last call's contents (nothing
 * needs clearing: every score a call reads it has written first), so calls
 * whose work overlaps on the GPU -- on different streams or from different
 * host threads -- race on it.
 */
KB_API int kb_attn_fwd_naive_noalloc(const void* q, const void* k, const void* v, void* o,
                                     int B, int H, int S, int d, int causal, float scale,
                                     void* stream);

/*
 * kb_attn_work_lists -- the per-CTA work lists the KB_TC path launches with, for
 * inspection (host only, no CUDA call). A unit is query rows [256 u, 256 u + 256)
 * of one head (d <= 128: the two 128-row tiles of a work item) or [128 u, 128 u +
 * 128) (d = 256). The heads are split into contiguous groups whose K and V fit
 * 32 MB of L2; within a group the units go heaviest first (causal: most key
 * tiles), each to the CTA with the least modelled work so far (key tiles + 1).
 * The kernel runs CTA c's units in list order. The lists are deterministic.
 *   N      : heads (B * H), > 0;  0 < S <= 2^31 - 257;  d : 32, 64, 128 or 256
 *   grid   : persistent CTAs (the launch uses min(units, SMs))
 *   start  : host array of grid + 1 ints; CTA c runs items[start[c] .. start[c + 1])
 *   items  : host array of `cap` entries, head << 16 | unit
 *   count  : receives the number of entries; 0 means the kernel orders the units
 *            itself (heaviest first, a snake over the CTAs): more than 4096
 *            units, no more units than CTAs, or more than 256 CTAs; start and
 *            items are then left untouched
 * Returns KB_ERR_INVALID_ARG for null pointers, non-positive sizes, another d,
 * or cap smaller than the count (which is then still stored in *count).
 */
KB_API int kb_attn_work_lists(long long N, int S, int d, int causal, int grid, int* start, unsigned int* items,
                              int cap, int* count);

/* Human-readable name of a kb_status (static storage, never NULL). */
KB_API const char* kb_status_string(int status);

/* cudaError_t of the last call on this thread that returned KB_ERR_CUDA. */
KB_API int kb_last_cuda_error(void);

/* Library ABI version: 100 * major + minor. */
KB_API int kb_version(void);

/*
 * kb_binary_version -- the architecture the library's kernels were compiled
 * for, as the CUDA runtime reports it for the tensor-core attention kernel on
 * the current device (cudaFuncAttributes::binaryVersion, 10 * major + minor:
 * 103 for sm_103a code). *out receives it. KB_ERR_INVALID_ARG for a null
 * pointer, KB_ERR_NO_DEVICE without a usable sm_103 device.
 */
KB_API int kb_binary_version(int* out);

/*
 * kb_q15_exp_table -- the 64-entry table of the KB_FIXEDPOINT path,
 * out64[f] = round(2^15 * 2^(-f/64)) (out64: host array of 64 entries).
 * Host only, no CUDA call. KB_ERR_INVALID_ARG for a null pointer.
 */
KB_API int kb_q15_exp_table(unsigned short* out64);

#ifdef __cplusplus
}
#endif

#endif /* KBATTN_H */
