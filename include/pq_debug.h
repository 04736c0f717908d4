/*
 * pq_debug.h — test-only hooks of libpq.  Not part of the computation; used by
 * the failure-detection tests.  The Phobos pages have no counterpart: their
 * kernels trap on a bad extent ("Kernel ABI", "Entry checks") and a trapping
 * CTA of a persistent kernel leaves the others waiting for good, which a
 * shared GPU must never see.  libpq instead bounds every on-device wait.
 */
#ifndef PQ_DEBUG_H
#define PQ_DEBUG_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Makes the next launches of the pipelined kernels skip pipeline stage
 * `skip_stage` in the producer (-1 turns it off): the tensor-core kernels
 * (PQ_PATH_TC; in the prompt-shape kernel that holds the weights in tensor
 * memory a stage is one scale group of 128 K) and the TMA-fed warp-level MMA
 * kernel of few rows (PQ_PATH_MMA, and the automatic path where it runs that
 * kernel; a stage is 128 weight rows x 4 blocks of one CTA's K chunk), so
 * that every consumer's bounded wait gives up after `timeout_cycles` SM clock
 * cycles (0 restores the default limit of about two seconds).  The kernel
 * then drains its copies and MMAs in flight, frees its tensor memory and
 * returns; C is left undefined.  The next pq_check_device returns
 * PQ_ERR_TIMEOUT.  Host state, process-wide, not thread-safe; returns
 * PQ_ERR_INVALID_ARG for skip_stage < -1.
 */
int pq_debug_set_tc_fault(int skip_stage, unsigned long long timeout_cycles);

/*
 * Chooses the tensor-core kernel of the prompt shapes (M > 64, Q8_0 or Q5_0
 * weights): 1 (the default) the kernel that applies the scales in registers
 * and hands two blocks at a time between its roles, wherever it takes the
 * call (scaled output, K a multiple of 128, a call that may allocate its
 * activation workspace); 0 the kernel with the scale-product MMA, which also
 * serves small batches, block sums and the allocation-free entry.  Both
 * compute the same qdot_t (q50_qdot_t) within its tolerance; the hook lets the
 * tests and measurements run either.  Host state, process-wide, not
 * thread-safe; PQ_ERR_INVALID_ARG for any other value.
 */
int pq_debug_set_prompt_kernel(int which);

/*
 * Chooses the warp-level MMA kernel of few rows (PQ_PATH_MMA, 1 <= M <= 64,
 * and the automatic paths that use it): 1 (the default) the kernel whose
 * producer warp streams the weights into shared memory by TMA, with K split
 * over a thread-block cluster, wherever it takes the shape; 0 the kernel whose
 * computing warps load their own weight bytes.  Both compute the same qdot_t
 * within its tolerance; the hook lets the tests and measurements run either.
 * Host state, process-wide, not thread-safe; PQ_ERR_INVALID_ARG for any other
 * value.
 */
int pq_debug_set_small_kernel(int which);

/*
 * The TMA-fed kernel of few rows splits K over a thread-block cluster whose
 * size (1, 2, 4 or 8 CTAs) it chooses by a cost model.  pq_debug_set_small_split
 * restricts it to clusters of `ks` CTAs (0 restores its own choice); a shape
 * whose K chunk then does not fit shared memory, or whose chunking gives
 * another cluster size, goes to the register-fed kernel.
 * pq_debug_small_kernel_config writes the last launch of that kernel's cluster
 * size, number of clusters, ring stages and K chunk in blocks to out4[0..3]
 * (zeros before the first launch).  Host state, process-wide, not
 * thread-safe; PQ_ERR_INVALID_ARG for another ks or a null out4.
 */
int pq_debug_set_small_split(int ks);
int pq_debug_small_kernel_config(int* out4);

/*
 * Registers a thread of the build of the second prompt kernel (see
 * pq_debug_set_prompt_kernel) that the current device admits with its 704
 * threads (several builds with different register limits exist; the largest
 * that fits is used), or 0 if the device admits none and the prompt shapes
 * run the first kernel.
 */
int pq_debug_prompt_kernel_regs(void);

/*
 * A streaming reader with the memory traffic of the one-row decode step and
 * none of its arithmetic, for measuring the floor that launch chaining and the
 * weight stream set on that step: `rows` weight rows W [rows, K] int8
 * (32-byte aligned base) and their scales WS [rows, K/32] f32 are read with
 * the step's grid (32 rows per CTA), L2 prefetch, 256-bit evict-first loads and
 * programmatic launch chaining; out[row] receives a checksum of the row (so no
 * load can be dropped).  early = 1 issues the first round of loads before the
 * wait for the preceding kernel (valid here because the reader's inputs are
 * never written while it runs).  Device
 * pointers; asynchronous on `stream`; PQ_ERR_INVALID_ARG / PQ_ERR_ALIGN on bad
 * arguments.
 */
int pq_debug_stream_read(const int8_t* W, const float* WS, int64_t rows, int64_t K, float* out, int early,
                         cudaStream_t stream);

/*
 * How pq_quantize_qdot_q8_0_host reaches its result buffer: 0 (the default)
 * the kernels write C_host in place when it is page-locked host memory the
 * device can address, else through a copy; 1 always through a copy.  Both give the same results; the
 * hook lets the tests and measurements run either.  Host state, process-wide,
 * not thread-safe; PQ_ERR_INVALID_ARG for any other value.
 */
int pq_debug_set_host_path(int which);

#ifdef __cplusplus
}
#endif

#endif /* PQ_DEBUG_H */
