// Host-side interface between the C-ABI layer (pq_api.cu) and the kernel
// launchers.  Launchers assume validated arguments and return a cudaError_t.
#pragma once
#include <cstdint>
#include <cuda_runtime_api.h>

namespace pq {

struct QdotArgs {
    const int8_t* A;
    const float* AS;
    const int8_t* W;
    const float* WS;
    float* C;        // f32 [M, N] result, or null in block-sum mode
    int32_t* S;      // int32 [M, N, K/32] block sums, or null
    int64_t M, N, K;
    int ws_layout;   // 0: WS [N, K/32]; 1: WS [K/32, N]
    int no_alloc = 0;  // 1: the call must not allocate device memory (no workspace)
    // 1: the kernel just before this launch on the stream is this library's
    // quantizer launched with late_trigger, so every kernel before that one
    // has completed when this one starts and W, WS may be read before
    // griddepcontrol.wait (the TMA-fed kernel then streams its first stages)
    int early_weights = 0;
};

struct FusedArgs {
    const float* x;  // f32 [M, K] activations
    int8_t* A;       // optional int8 [M, K] output of the quantizer (with AS), or null
    float* AS;
    const int8_t* W;
    const float* WS;
    float* C;
    int64_t M, N, K;
    int ws_layout;
};

// Launches `kernel` with programmatic stream serialization allowed: it may be
// scheduled while the previous kernel on the stream is still running, and
// orders itself with griddepcontrol.wait (pdl_wait) before touching data that
// kernel may have written.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// late_trigger: the next kernel on the stream is let in only after this one
// has waited for its own predecessor (see QdotArgs::early_weights).
cudaError_t launch_quantize(const float* x, int8_t* q, float* s, int64_t rows, int64_t K,
                            cudaStream_t stream, bool late_trigger = false);

// dp4a streaming kernel: any M; returns cudaErrorInvalidConfiguration when the
// grid would exceed the device limits.
cudaError_t launch_qdot_simt(const QdotArgs& a, cudaStream_t stream);

// Fused quantize + dp4a contraction for one activation row (cudaErrorNotSupported
// for M != 1, when the grid would need more than one wave, or when the
// quantized row does not fit a CTA's shared memory).
cudaError_t launch_qdot_fused(const FusedArgs& a, cudaStream_t stream);

// Test-only streaming reader: reads `rows` weight rows of K bytes and their
// K/32 f32 scales exactly as the fused decode step does (same grid, loads and
// launch chaining), computes nothing but a checksum per row (out[row]).
// early = 1 issues the first round of loads before griddepcontrol.wait.
cudaError_t launch_stream_read(const int8_t* W, const float* WS, int64_t rows, int64_t K, float* out, int early,
                               cudaStream_t stream);

// dp4a kernel for Q5_0 weights (q50_qdot_t): a.W points at the 20-byte Q5_0
// blocks, [N, K/32 * 20] bytes; any M.
cudaError_t launch_qdot_q50(const QdotArgs& a, cudaStream_t stream);

// Fused quantize + dp4a contraction against Q5_0 weights (a.W points at the
// Q5_0 blocks) for one activation row; cudaErrorNotSupported as for
// launch_qdot_fused.
cudaError_t launch_qdot_q50_fused(const FusedArgs& a, cudaStream_t stream);

// tcgen05 tensor-core kernel for Q5_0 weights (a.W points at the Q5_0 blocks,
// 16-byte aligned): prompt shapes only (M > 64), no block-sum mode;
// cudaErrorNotSupported otherwise or when the device is not sm_103.
cudaError_t launch_qdot_tc_q50(const QdotArgs& a, cudaStream_t stream);

// tcgen05 tensor-core kernels.  cudaErrorNotSupported if the device is not
// sm_103.  The prompt shapes that the kernel of qdot_tcw.cu takes (M > 64,
// scaled output, K % 128 == 0, a call that may allocate; Q8_0 or Q5_0 weights)
// run it (scales applied in registers, two blocks per hand-off) unless
// set_prompt_kernel(0) asks for the kernel of qdot_tc.cu, which runs every
// other shape.
cudaError_t launch_qdot_tc(const QdotArgs& a, cudaStream_t stream);
cudaError_t launch_qdot_tcw(const QdotArgs& a, cudaStream_t stream, bool q5 = false);
void set_prompt_kernel(int which);

// Warp-level MMA kernel (mma.sync m16n8k16, f16 operands, exact block sums) for
// 1 <= M <= 64; cudaErrorNotSupported otherwise.
cudaError_t launch_qdot_mma(const QdotArgs& a, cudaStream_t stream);

// Fused quantize + warp-level MMA contraction (1 <= M <= 64): every CTA
// quantizes the rows of its K range itself; a.A / a.AS, when given, receive the
// quantized rows.  cudaErrorNotSupported as for launch_qdot_mma.
cudaError_t launch_qdot_mma_fused(const FusedArgs& a, cudaStream_t stream);

// Warp-level MMA kernel fed by TMA (qdot_mmt.cu) for 1 <= M <= 64, scaled
// output only: weights streamed into a shared-memory ring by a producer warp,
// K split over a thread-block cluster.  cudaErrorNotSupported for shapes or
// alignments it does not take (block-sum mode, K < 128, N < 32, W or WS not
// 16-byte aligned, K/32 % 4 != 0 with WS [N, K/32], N % 4 != 0 with WS
// [K/32, N], shared memory too small for the K chunk) and when
// set_small_kernel(0) selected the register-fed kernel of qdot_mma.cu.
// small_kernel() returns the selection (1: this kernel where it applies).
cudaError_t launch_qdot_mmt(const QdotArgs& a, cudaStream_t stream);
void set_small_kernel(int which);
int small_kernel();
// Test hooks: restrict the TMA-fed kernel to clusters of ks CTAs (0: its own
// choice); the last launch's (cluster size, clusters, ring stages, K chunk).
void set_small_split(int ks);
void small_kernel_config(int* out4);

// A workspace of at least `bytes` for work enqueued on `stream` of the current
// device (one per device, stream and kind, so calls on different streams never
// share it; allocated stream-ordered on first use, replaced by one at least
// twice as large when a larger call arrives, never freed before exit).  Fails
// without allocating while `stream` is being captured and the workspace is too
// small, or when the table of streams is full; callers then take a path that
// needs no workspace.
cudaError_t stream_workspace(cudaStream_t stream, size_t bytes, void** out, int kind = 0);

// Shape checks of the qdot entry points (sizes >= 0, K a positive multiple of
// 32, element counts representable in int64); returns a pq_status.
int check_qdot_shape(int64_t M, int64_t N, int64_t K);

// qdot_t (automatic kernel path) without any device allocation; returns a pq_status.
int qdot_noalloc(const int8_t* A, const float* AS, const int8_t* W, const float* WS, float* C, int64_t M, int64_t N,
                 int64_t K, int ws_layout, cudaStream_t stream);

// Reads and clears the device status words of the tensor-core kernels (set by
// a bounded wait that gave up).
cudaError_t read_and_clear_status(unsigned* status);
cudaError_t read_and_clear_status_w(unsigned* status);
cudaError_t read_and_clear_status_mmt(unsigned* status);
cudaError_t read_and_clear_status_simt(unsigned* status);

// Test hooks of the tensor-core kernel: skip one producer stage so that the
// consumers' bounded waits give up (-1: off), and the wait limit in SM clock
// cycles (0: the default of about two seconds).
void set_tc_test_hooks(int inject_skip_stage, unsigned long long timeout_cycles);
void set_tcw_test_hooks(int inject_skip_group, unsigned long long timeout_cycles);
void set_mmt_test_hooks(int inject_skip_stage, unsigned long long timeout_cycles);
// Registers a thread of the prompt kernel build chosen for the current device
// (0: the device admits none, the shared-memory kernel runs instead).
int tcw_kernel_regs();

}  // namespace pq
