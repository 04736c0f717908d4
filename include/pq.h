/*
 * pq.h — C ABI of the Q8_0 block-scaled contraction library (libpq.so) for
 * NVIDIA GB300 (sm_103a).
 *
 * What it computes (Phobos documentation, "Quantized built-ins and formats",
 * section "Q8_0", and "Phobos Language Spec", section 10 "Quantized
 * built-ins", Q8_0 table):
 *
 *   Q8_0 stores signed bytes with one scale per block of 32 values;
 *   activations are quantized the same way, so
 *
 *     C[i, j] = sum over blocks b of AS[i, b] * WS[j, b]
 *                 * sum over k in b of A[i, k] * W[j, k]
 *
 *   with the inner (block) sum in integers.  A is [M, K] int8, AS [M, K/32]
 *   f32, W [N, K] int8, WS [N, K/32] f32 (qdot_t's layout; qmma_t's
 *   [K/32, N] is selected with PQ_WS_KB_N), C [M, N] f32.
 *
 * Conventions shared by every entry point:
 *
 *   Memory.  All tensors are row-major and dense (the innermost index is
 *   contiguous, no padding).  Every pointer is a DEVICE pointer owned by the
 *   caller; the library never frees it or keeps it.  The only device memory
 *   the library allocates is the workspace some entry points keep per
 *   (device, stream) pair (documented with each).  It is allocated with
 *   cudaMallocAsync on that stream on first use (ordered with the stream's
 *   work, no device-wide synchronization) and replaced by one at least twice
 *   as large when a larger call arrives; a replaced workspace is kept until
 *   exit, never freed, so work enqueued or captured earlier that refers to it
 *   stays valid.  No entry point calls cudaFree.
 *   Base alignment: int8 tensors (A, W, q) and f32 inputs read as vectors
 *   (x) start on a 16-byte boundary; the f32 scale planes and C on a 4-byte
 *   boundary.  (The pages ask 16 bytes of every tensor base, "Kernel ABI",
 *   section "Memory layout and alignment".)
 *
 *   Streams.  Work is enqueued on `stream` (0 = the legacy default stream) and
 *   runs asynchronously: PQ_OK means "validated and enqueued".  Results are
 *   visible after the stream is synchronized.
 *
 *   Errors.  Every precondition is checked on the host BEFORE anything is
 *   launched, and a failed check returns a negative pq_status with nothing
 *   enqueued and no byte written (the pages' kernels trap on a bad extent and
 *   leave the CUDA context unusable, "Kernel ABI", "Entry checks"; this
 *   library never traps).  PQ_ERR_CUDA reports a launch failure returned by
 *   the CUDA runtime.  Empty problems (M == 0, N == 0 or rows == 0) return
 *   PQ_OK and launch nothing.
 *
 *   Shapes.  K must be a positive multiple of 32 (one whole Q8_0 block).  M
 *   and N need not be multiples of any tile: the kernels mask ragged edges
 *   themselves.  All sizes are int64; products such as M*K must fit in int64
 *   and the grid limits of the device (checked, PQ_ERR_SHAPE).
 *
 *   Values.  Any int8 is a valid qdot operand, including -128 (which the
 *   quantizer never emits).  Scales may be any finite f32.  NaN or Inf inputs
 *   give unspecified outputs.
 */
#ifndef PQ_H
#define PQ_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PQ_OK = 0,
    PQ_ERR_INVALID_ARG = -1, /* null pointer, unknown path or layout code */
    PQ_ERR_SHAPE = -2,       /* negative size, K not a positive multiple of 32, size overflow */
    PQ_ERR_ALIGN = -3,       /* a base pointer below the alignment stated above */
    PQ_ERR_CUDA = -4,        /* the CUDA runtime refused a launch or a query */
    PQ_ERR_TIMEOUT = -5,     /* a bounded on-device wait gave up (reported by pq_check_device) */
    PQ_ERR_UNSUPPORTED = -6, /* the device is not sm_103 / the path cannot take this shape */
    PQ_ERR_SCRATCH = -7      /* the problem does not fit the fixed scratch of pq_quantize_qdot_q8_0_noalloc */
} pq_status;

/* Bytes of device memory that pq_quantize_qdot_q8_0_noalloc keeps for itself on every GPU. */
#define PQ_NOALLOC_SCRATCH_BYTES (1u << 20)

/* Kernel path selector for pq_qdot_q8_0_ex / pq_qdot_q8_0_blocksums. */
enum {
    PQ_PATH_AUTO = 0,  /* by M: dp4a up to M = 8, the warp-level MMA for 9..16, tcgen05 above */
    PQ_PATH_SIMT = 1,  /* dp4a (CUDA-core) streaming kernel, any M */
    PQ_PATH_TC = 2,    /* tcgen05 tensor-core kernel (f16 operands, exact integer block sums) */
    PQ_PATH_MMA = 3    /* warp-level tensor-core path (mma.sync m16n8k16, f16 operands, exact
                          integer block sums), M <= 64: the kernel fed by TMA through a
                          shared-memory ring, or the one whose warps load their own weight
                          bytes (block-sum mode; shapes the first declines) */
};

/* Layout of the weight-scale plane WS. */
enum {
    PQ_WS_N_KB = 0,  /* WS [N, K/32]: qdot_t */
    PQ_WS_KB_N = 1   /* WS [K/32, N]: qmma_t ("w_scales is [K/32, N], transposed relative to qdot_t") */
};

/*
 * Row quantizer f32 -> Q8_0 ("Quantized built-ins and formats", section
 * "Q8_0": one f32 scale per 32 signed bytes; activations are quantized the
 * same way as weights).  For every row r and block b of 32 elements:
 *   amax = max |x|,  d = amax / 127 (IEEE f32 division),
 *   q = round(x / d) with ties to even (the spec's round(), section 9),
 *   clamped to [-127, 127];  a block with d == 0 stores q = 0.
 * x: f32 [rows, K] (16-byte aligned), q: int8 [rows, K] (16-byte aligned),
 * s: f32 [rows, K/32] (4-byte aligned).  Outputs are overwritten.  x must
 * not overlap q or s.
 */
int pq_quantize_q8_0(const float* x, int8_t* q, float* s,
                     int64_t rows, int64_t K, cudaStream_t stream);

/*
 * qdot_t: C[M, N] = Q8_0 contraction of A [M, K] with W [N, K] as stated at
 * the top of this header ("Quantized built-ins and formats", section "Q8_0";
 * the example kernel's argument order A, AS, W, WS, C).  C is overwritten
 * (the pages' example assigns the result).  The kernel is chosen by M.
 * C must not overlap any input.
 *
 * Workspace (tensor-core path, M > 64): the activations are converted once
 * per call, by a small kernel enqueued before the contraction, into a
 * workspace that belongs to the (device, stream) pair (allocated and grown
 * as stated at the top of this header).  A call made while its stream is
 * being captured, whose workspace does
 * not exist yet or is too small, allocates nothing and lets the kernel convert
 * the activations itself (same results); so does
 * pq_quantize_qdot_q8_0_noalloc, and so does every stream past the 64th.
 */
int pq_qdot_q8_0(const int8_t* A, const float* AS, const int8_t* W, const float* WS,
                 float* C, int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * As pq_qdot_q8_0, with the weight-scale layout (PQ_WS_N_KB for qdot_t,
 * PQ_WS_KB_N for qmma_t, spec section 10) and the kernel path chosen by the
 * caller (PQ_PATH_*).  PQ_ERR_UNSUPPORTED if the chosen path cannot take
 * the shape.  PQ_PATH_TC works on groups of four Q8_0 blocks and loads the
 * scale planes with TMA, so it needs K a multiple of 128, AS and WS 16-byte
 * aligned, and N a multiple of 4 for PQ_WS_KB_N (TMA row strides are
 * multiples of 16 bytes); otherwise it returns PQ_ERR_UNSUPPORTED, and
 * PQ_PATH_AUTO takes the dp4a kernel instead.
 */
int pq_qdot_q8_0_ex(const int8_t* A, const float* AS, const int8_t* W, const float* WS,
                    float* C, int64_t M, int64_t N, int64_t K,
                    int ws_layout, int path, cudaStream_t stream);

/*
 * One decode step in one call: quantize the activation rows x [M, K] f32 to
 * Q8_0 (exactly as pq_quantize_q8_0) and contract them with W (as
 * pq_qdot_q8_0_ex with the given weight-scale layout, automatic path) -- the
 * quantizer feeding qdot_t that "Quantized built-ins and formats", section
 * "Q8_0", describes ("the activations are quantized the same way").  For one
 * row (M == 1) this is one kernel, in which every CTA quantizes x into its
 * shared memory while L2 prefetches its weight rows, then streams them (at
 * most one CTA per SM; its warps take further columns when N needs more).
 * Otherwise it is the quantizer followed by qdot_t, launched so that the
 * second overlaps the first (for 9 to 16 rows this is faster than a one-kernel
 * step whose every CTA quantizes its K range of the rows again; that one-kernel
 * step remains with the register-fed warp-level MMA kernel selected by
 * pq_debug_set_small_kernel(0)).  A [M, K] int8 and AS [M, K/32] f32
 * optionally receive the quantized rows (both null, or both non-null).  When
 * they are null and the two-kernel route is taken, the rows go to a
 * workspace of this (device, stream) pair, allocated on the first such call
 * on the stream and grown when a larger one arrives (that call must not be
 * inside a stream capture; see the top of this header).  x: 16-byte aligned f32
 * [M, K]; A 16-byte aligned; AS, WS, C 4-byte aligned.  C must not overlap
 * any input, and A, AS must not overlap x, W, WS or C.
 */
int pq_quantize_qdot_q8_0(const float* x, int8_t* A, float* AS, const int8_t* W, const float* WS,
                          float* C, int64_t M, int64_t N, int64_t K, int ws_layout, cudaStream_t stream);

/*
 * One decode step with the activations and the result in host memory:
 * x_host [M, K] f32 in, C_host [M, N] f32 out, the rules of the contraction as
 * for pq_quantize_qdot_q8_0 (A = AS = NULL).  The call returns once the work is
 * enqueued on `stream`: synchronize the stream before reading C_host.
 *   - When C_host is page-locked host memory that the device can address
 *     (cudaHostAlloc / cudaHostRegister, mapped: on GB300 the host memory is
 *     reached over the coherent chip-to-chip link), the host-to-device copy of
 *     x and the step are enqueued, and the step's kernels write C into C_host
 *     directly (no device-to-host copy).
 *   - Otherwise (pageable C_host) the host-to-device copy of x, the step, and
 *     the device-to-host copy of C are enqueued in that order.
 * The device copies of x (and of C) live in a workspace of this (device,
 * stream) pair, allocated on the first such call on the stream and grown when a
 * larger one arrives (that call must not be inside a stream capture; see the
 * top of this header).  Pageable buffers make the copies synchronous.
 * W and WS as for pq_quantize_qdot_q8_0.
 */
int pq_quantize_qdot_q8_0_host(const float* x_host, const int8_t* W, const float* WS, float* C_host,
                               int64_t M, int64_t N, int64_t K, int ws_layout, cudaStream_t stream);

/*
 * pq_quantize_qdot_q8_0 without any device allocation.  (The Phobos pages
 * have no counterpart: this is a property of the library, not of the method.)
 *
 * For callers that cannot have the library allocate device memory -- code
 * whose work is recorded into a CUDA graph (no allocation while a stream is
 * being captured), serving loops that must never stall on cudaMalloc or
 * cudaFree (both may synchronize the device), hosts that give a plugin a
 * fixed memory budget and make every allocation themselves.  Same result as
 * pq_quantize_qdot_q8_0 with A = AS = NULL (the quantizer, then qdot_t on the
 * automatic path), but the quantized rows and their scales are kept in a
 * fixed array of PQ_NOALLOC_SCRATCH_BYTES (1 MiB) that is part of the library
 * and that every GPU which loads the library holds until the process exits.
 * Where pq_quantize_qdot_q8_0 runs one kernel (one row) this call runs the
 * same kernel and leaves the array alone.
 * The caller still passes x, W, WS and C (same layouts and alignment as
 * pq_quantize_qdot_q8_0); nothing else is allocated, by this call or by the
 * kernels it starts.
 *
 * Limits: M * K bytes (rounded up to 256) plus M * K / 8 bytes of scales must
 * fit PQ_NOALLOC_SCRATCH_BYTES -- e.g. M <= 227 for K = 4096, M <= 65 for
 * K = 14336 -- else PQ_ERR_SCRATCH and nothing is launched.
 *
 * The first call on a device resolves the array's device address there (a
 * runtime query, no allocation); make that first call before any stream
 * capture on that device.  Every call on a device uses the same array, and
 * each call overwrites all of it that it reads, so nothing carries over from
 * an earlier call; but calls that can run at the same time on the GPU (on
 * different streams, without an ordering between them) race on the array and
 * give wrong results.
 */
int pq_quantize_qdot_q8_0_noalloc(const float* x, const int8_t* W, const float* WS, float* C,
                                  int64_t M, int64_t N, int64_t K, int ws_layout, cudaStream_t stream);

/*
 * The integer stage alone, for verification: S[i, j, b] = sum over k in
 * block b of A[i, k] * W[j, k] ("Quantized built-ins and formats": "the
 * inner sum in integers"), computed by the engine of `path` (PQ_PATH_SIMT:
 * dp4a; PQ_PATH_TC and PQ_PATH_MMA (M <= 64): the tensor-core MMAs with f32
 * accumulation, exact because every partial sum is an integer below 2^24).  S: int32 [M, N, K/32],
 * 4-byte aligned, overwritten.  |S| <= 32 * 128 * 128 = 524288.
 */
int pq_qdot_q8_0_blocksums(const int8_t* A, const int8_t* W, int32_t* S,
                           int64_t M, int64_t N, int64_t K, int path, cudaStream_t stream);

/*
 * q50_qdot_t: C[M, N] = the Q8_0 contraction of A [M, K] with a Q5_0 weight
 * ("Phobos Language Spec", section 10, Q5_0 row; "Quantized built-ins and
 * formats", built-in table):
 *
 *   C[i, j] = sum over blocks b of AS[i, b] * WS[j, b]
 *               * sum over e < 32 of A[i, 32b + e] * (q[j, 32b + e] - 16)
 *
 * W5 holds the weight's Q5_0 blocks without their scale, row-major
 * [N, K/32 * 20] bytes: per 32 elements a 4-byte qh word, then 16 bytes whose
 * byte e holds element e in its low nibble and element e + 16 in its high
 * nibble.  qh is read as a little-endian 32-bit word whose bit e is the fifth
 * bit (value 16) of element e (the pages do not state the bit order; this is
 * the reading taken).  WS is f32 [N, K/32] (PQ_WS_N_KB) or [K/32, N]
 * (PQ_WS_KB_N, q50_qmma_t's layout); A and AS as for pq_qdot_q8_0.  C is
 * overwritten.  Alignment: A 16 bytes; W5, AS, WS, C 4 bytes.  M <= 64 runs
 * the dp4a kernel; M > 64 runs a tensor-core kernel, which decodes the blocks
 * to f16 in shared memory (it needs K a multiple of 128 and W5 and WS 16-byte
 * aligned, and uses the per-stream workspace of pq_qdot_q8_0; inside a stream
 * capture before that workspace exists, the other tensor-core kernel, which
 * also needs AS 16-byte aligned; shapes and operands both decline run the
 * dp4a kernel).
 */
int pq_q50_qdot(const int8_t* A, const float* AS, const uint8_t* W5, const float* WS, float* C,
                int64_t M, int64_t N, int64_t K, int ws_layout, cudaStream_t stream);

/*
 * One decode step against Q5_0 weights in one call: quantize the activation
 * rows x [M, K] f32 to Q8_0 (exactly as pq_quantize_q8_0) and contract them
 * with the Q5_0 weight W5 as pq_q50_qdot does -- the Q5_0 counterpart of
 * pq_quantize_qdot_q8_0 ("Quantized built-ins and formats", built-in table:
 * q50_qdot_t takes Q8_0 activations).  For one row (M == 1) and N up to
 * 64 x the SM count this is one kernel, in which every CTA quantizes x into
 * its shared memory while L2 prefetches the start of its weight rows, then
 * streams them; otherwise it is the quantizer followed by pq_q50_qdot.
 * A / AS, the workspace, alignment and overlap rules are those of
 * pq_quantize_qdot_q8_0; W5 as for pq_q50_qdot.
 */
int pq_quantize_q50_qdot(const float* x, int8_t* A, float* AS, const uint8_t* W5, const float* WS, float* C,
                         int64_t M, int64_t N, int64_t K, int ws_layout, cudaStream_t stream);

/*
 * The integer stage of pq_q50_qdot alone, for verification: S[i, j, b] =
 * sum over e < 32 of A[i, 32b + e] * (q[j, 32b + e] - 16), int32 [M, N, K/32],
 * 4-byte aligned, overwritten.
 */
int pq_q50_blocksums(const int8_t* A, const uint8_t* W5, int32_t* S, int64_t M, int64_t N, int64_t K,
                     cudaStream_t stream);

/*
 * Synchronizes `stream`, then reads and clears this library's device status
 * word for the current device.  Returns PQ_OK, PQ_ERR_TIMEOUT if a kernel's
 * bounded wait gave up since the last check (its output is then invalid), or
 * PQ_ERR_CUDA if the synchronize failed.
 */
int pq_check_device(cudaStream_t stream);

/* A static, human-readable name for a pq_status code. */
const char* pq_strerror(int code);

/* ABI version of this header: major * 100 + minor (1.01: pq_quantize_qdot_q8_0; 1.02: Q5_0 weights;
   1.03: pq_quantize_q50_qdot and PQ_PATH_MMA; 1.04: pq_quantize_qdot_q8_0_host; 1.05: one kernel
   for 9..16 rows in pq_quantize_qdot_q8_0). */
int pq_version(void);

/*
 * The CUDA runtime error (a cudaError_t value) behind the last PQ_ERR_CUDA or
 * PQ_ERR_UNSUPPORTED that an entry point returned on the calling thread, or 0
 * if there was none.  For diagnostics only; it is not reset by later calls
 * that succeed.
 */
int pq_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PQ_H */
