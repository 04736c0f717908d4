// Allocation-free form of the one-call decode step (pq_quantize_qdot_q8_0).
//
// pq_quantize_qdot_q8_0 keeps the quantized activation rows in a workspace it
// allocates (cudaMallocAsync) on first use.  Some callers cannot let a library
// allocate device memory: code that records its work into a CUDA graph
// (allocation is not allowed while a stream is being captured), serving loops
// that must never stall on cudaMalloc / cudaFree (both can synchronize the
// whole device), and hosts that hand a plugin a fixed memory budget and own
// every allocation themselves.  For them this entry point keeps the rows in a
// fixed array of device memory that is part of the library image instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kScratchBytes of it until the process exits.  Host code
// cannot use the array's name as a device address (on the host it names a
// stand-in object), so the device address is resolved once per device with
// cudaGetSymbolAddress, with that device current, and handed to the kernels.
#include <cstdint>
#include <mutex>

#include <cuda_runtime_api.h>

#include "pq.h"
#include "pq_internal.h"

namespace {

constexpr size_t kScratchBytes = PQ_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Quantized rows (M*K bytes, rounded up to 256) followed by their scales
// (M*K/32 floats).  Shared by every call on a device; each call overwrites
// what it reads, so nothing carries over from the previous call's contents.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (resolved on the
// first call on that device).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

}  // namespace

extern "C" int pq_quantize_qdot_q8_0_noalloc(const float* x, const int8_t* W, const float* WS, float* C,
                                             int64_t M, int64_t N, int64_t K, int ws_layout,
                                             cudaStream_t stream) {
    if (ws_layout != PQ_WS_N_KB && ws_layout != PQ_WS_KB_N) return PQ_ERR_INVALID_ARG;
    // the same shape rules as the allocating entry point
    const int shape = pq::check_qdot_shape(M, N, K);
    if (shape != PQ_OK) return shape;
    if (M == 0 || N == 0) return PQ_OK;
    // the quantized rows and their scales must fit the fixed array
    if (M > static_cast<int64_t>(kScratchBytes) || K > static_cast<int64_t>(kScratchBytes)) return PQ_ERR_SCRATCH;
    const size_t qbytes = (static_cast<size_t>(M) * static_cast<size_t>(K) + 255) & ~size_t(255);
    const size_t sbytes = static_cast<size_t>(M) * static_cast<size_t>(K / 32) * sizeof(float);
    if (qbytes + sbytes > kScratchBytes) return PQ_ERR_SCRATCH;
    if (!x || !W || !WS || !C) return PQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(W, 16) || !aligned(WS, 4) || !aligned(C, 4)) return PQ_ERR_ALIGN;

    // one kernel where the one-call step has one (one row; 9..16 rows with the
    // register-fed warp-level MMA kernel selected): its CTAs quantize the rows
    // themselves and the scratch is not touched
    const pq::FusedArgs f{x, nullptr, nullptr, W, WS, C, M, N, K, ws_layout};
    cudaError_t e = pq::launch_qdot_fused(f, stream);
    if (e == cudaErrorNotSupported && M > 8 && M <= 16 && pq::small_kernel() == 0)
        e = pq::launch_qdot_mma_fused(f, stream);
    if (e != cudaErrorNotSupported)
        return e == cudaSuccess ? PQ_OK : e == cudaErrorInvalidConfiguration ? PQ_ERR_UNSUPPORTED : PQ_ERR_CUDA;

    void* base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return PQ_ERR_CUDA;
    int8_t* A = static_cast<int8_t*>(base);
    float* AS = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + qbytes);
    const int st = pq_quantize_q8_0(x, A, AS, M, K, stream);
    if (st != PQ_OK) return st;
    // qdot_t on the path that allocates nothing (the tensor-core kernel then
    // converts the activations itself instead of pre-tiling them in a workspace)
    return pq::qdot_noalloc(A, AS, W, WS, C, M, N, K, ws_layout, stream);
}
