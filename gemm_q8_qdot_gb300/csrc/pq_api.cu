// C ABI of libpq: argument checks, kernel selection by M, launch.
//
// Every check runs on the host before anything is enqueued; a failed check
// returns a pq_status and writes nothing.  The pages' kernels instead trap at
// entry on a bad extent, which leaves the CUDA context unusable ("Kernel ABI",
// section "Entry checks"); a shared GPU must never see that.
#include <cstdint>
#include <mutex>
#include <cuda_runtime_api.h>

#include "pq.h"
#include "pq_debug.h"
#include "pq_internal.h"

namespace pq {

// Per-(device, stream, kind) workspaces (kind 0: the tensor-core path's
// pre-tiled activations; kind 1: the host-buffer step's device copies of x
// and C; kind 2: the quantized rows of a two-kernel pq_quantize_qdot_q8_0 /
// pq_quantize_q50_qdot call without A / AS), at most 64 triples.
//
// A workspace is allocated on the first call that needs it on its stream,
// with cudaMallocAsync on that stream: the allocation is ordered with the
// stream's work and synchronizes nothing else.  A larger call replaces it by
// one at least twice as large; the replaced one is kept (never freed before
// exit), so work enqueued earlier on the stream, and graphs captured earlier
// that refer to it, stay valid, and no call ever waits on a cudaFree.  With
// the doubling, the replaced workspaces of a triple add up to less than its
// current one.
cudaError_t stream_workspace(cudaStream_t stream, size_t bytes, void** out, int kind) {
    struct Slot {
        int dev;
        cudaStream_t stream;
        int kind;
        void* ptr;
        size_t size;
    };
    static std::mutex mu;
    static Slot slots[64];
    static int nslots = 0;
    // replaced workspaces are never freed (work already enqueued or captured may
    // still use them); they stay listed here, reachable, until the process exits
    [[maybe_unused]] static void* retired[64 * 48] = {};
    static int nretired = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    Slot* sl = nullptr;
    for (int i = 0; i < nslots; ++i)
        if (slots[i].dev == dev && slots[i].stream == stream && slots[i].kind == kind) sl = &slots[i];
    if (sl && sl->size >= bytes) {
        *out = sl->ptr;
        return cudaSuccess;
    }
    // allocating is not allowed while the stream is being captured
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) {
        cudaGetLastError();  // leave no sticky error behind for the caller's next check
        return e;
    }
    if (cs != cudaStreamCaptureStatusNone) return cudaErrorNotPermitted;
    if (!sl && nslots == 64) return cudaErrorMemoryAllocation;
    if (sl && sl->ptr && nretired == 64 * 48) return cudaErrorMemoryAllocation;
    size_t want = bytes < (size_t(1) << 20) ? (size_t(1) << 20) : bytes;
    if (sl && want < 2 * sl->size) want = 2 * sl->size;
    void* p = nullptr;
    e = cudaMallocAsync(&p, want, stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e;
    }
    if (!sl) {
        sl = &slots[nslots++];
        *sl = Slot{dev, stream, kind, nullptr, 0};
    }
    if (sl->ptr) retired[nretired++] = sl->ptr;
    sl->ptr = p;
    sl->size = want;
    *out = p;
    return cudaSuccess;
}

}  // namespace pq

namespace {

constexpr int64_t kMaxDim = int64_t(1) << 40;

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

// The CUDA error behind this thread's last PQ_ERR_CUDA / PQ_ERR_UNSUPPORTED.
thread_local int g_last_cuda_error = 0;

// 0: host buffers the device can address are used in place; 1: always copied
// (test hook, pq_debug_set_host_path).
int g_host_path = 0;

// The device address of a page-locked host buffer that the device can access
// (registered or allocated with cudaHostAlloc, mapped), or null for any other
// pointer (pageable or device memory); leaves no CUDA error behind.
void* device_view(const void* p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
    return at.devicePointer;
}

int map_cuda(cudaError_t e) {
    if (e == cudaSuccess) return PQ_OK;
    g_last_cuda_error = static_cast<int>(e);
    if (e == cudaErrorInvalidConfiguration || e == cudaErrorNotSupported) return PQ_ERR_UNSUPPORTED;
    return PQ_ERR_CUDA;
}

}  // namespace

// Shape checks shared by the qdot entry points: sizes >= 0, K a positive
// multiple of 32, every element count representable.
int pq::check_qdot_shape(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K <= 0 || (K % 32) != 0) return PQ_ERR_SHAPE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return PQ_ERR_SHAPE;
    // M*K, N*K, M*N and M*N*K/32 must fit in int64
    const __int128 mk = (__int128)M * K, nk = (__int128)N * K, mn = (__int128)M * N;
    const __int128 lim = (__int128)INT64_MAX;
    if (mk > lim || nk > lim || mn > lim || mn * (K / 32) > lim) return PQ_ERR_SHAPE;
    return PQ_OK;
}

namespace {

using pq::check_qdot_shape;

int qdot_impl(const int8_t* A, const float* AS, const int8_t* W, const float* WS, float* C,
              int32_t* S, int64_t M, int64_t N, int64_t K, int ws_layout, int path,
              cudaStream_t stream, int no_alloc = 0, int early_weights = 0) {
    if (path != PQ_PATH_AUTO && path != PQ_PATH_SIMT && path != PQ_PATH_TC && path != PQ_PATH_MMA)
        return PQ_ERR_INVALID_ARG;
    if (ws_layout != PQ_WS_N_KB && ws_layout != PQ_WS_KB_N) return PQ_ERR_INVALID_ARG;
    int st = check_qdot_shape(M, N, K);
    if (st != PQ_OK) return st;
    if (M == 0 || N == 0) return PQ_OK;
    const bool sums = S != nullptr;
    if (!A || !W) return PQ_ERR_INVALID_ARG;
    if (!sums && (!AS || !WS || !C)) return PQ_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(W, 16)) return PQ_ERR_ALIGN;
    if (sums && !aligned(S, 4)) return PQ_ERR_ALIGN;
    if (!sums && (!aligned(AS, 4) || !aligned(WS, 4) || !aligned(C, 4))) return PQ_ERR_ALIGN;

    pq::QdotArgs a{A, AS, W, WS, C, S, M, N, K, ws_layout, no_alloc, early_weights};
    if (path == PQ_PATH_SIMT) return map_cuda(pq::launch_qdot_simt(a, stream));
    if (path == PQ_PATH_TC) return map_cuda(pq::launch_qdot_tc(a, stream));
    if (path == PQ_PATH_MMA) return map_cuda(pq::launch_qdot_mma(a, stream));
    // automatic, by M (measured on GB300 at K = 4096, N = 11008, graphs of
    // back-to-back calls): the dp4a streaming kernel up to 8 rows (12.6 us at
    // M = 4, 17.3 us at M = 8, against 19.1 us for the TMA-fed warp-level MMA
    // kernel), the warp-level MMA path for 9..16 rows (19.1 us at M = 16 with
    // its TMA-fed kernel, against 31.9 us for dp4a and 29.2 us for tcgen05),
    // the tcgen05 kernel above (30.8 us at M = 32, 34.2 us at M = 64, against
    // 32.8 and 47.5 us for the TMA-fed kernel); a shape a kernel declines
    // (K % 128 != 0 for tcgen05) goes to the dp4a kernel, which takes every
    // shape
    cudaError_t e = cudaErrorNotSupported;
    if (M > 16) e = pq::launch_qdot_tc(a, stream);
    else if (M > 8) e = pq::launch_qdot_mma(a, stream);
    if (e != cudaErrorNotSupported) return map_cuda(e);
    return map_cuda(pq::launch_qdot_simt(a, stream));
}

}  // namespace

int pq::qdot_noalloc(const int8_t* A, const float* AS, const int8_t* W, const float* WS, float* C, int64_t M,
                     int64_t N, int64_t K, int ws_layout, cudaStream_t stream) {
    return qdot_impl(A, AS, W, WS, C, nullptr, M, N, K, ws_layout, PQ_PATH_AUTO, stream, 1);
}

extern "C" {

int pq_quantize_q8_0(const float* x, int8_t* q, float* s, int64_t rows, int64_t K, cudaStream_t stream) {
    if (rows < 0 || K <= 0 || (K % 32) != 0 || rows > kMaxDim || K > kMaxDim) return PQ_ERR_SHAPE;
    if ((__int128)rows * K > (__int128)INT64_MAX) return PQ_ERR_SHAPE;
    if (rows == 0) return PQ_OK;
    if (!x || !q || !s) return PQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(s, 4)) return PQ_ERR_ALIGN;
    return map_cuda(pq::launch_quantize(x, q, s, rows, K, stream));
}

int pq_qdot_q8_0(const int8_t* A, const float* AS, const int8_t* W, const float* WS, float* C,
                 int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    return qdot_impl(A, AS, W, WS, C, nullptr, M, N, K, PQ_WS_N_KB, PQ_PATH_AUTO, stream);
}

int pq_qdot_q8_0_ex(const int8_t* A, const float* AS, const int8_t* W, const float* WS, float* C,
                    int64_t M, int64_t N, int64_t K, int ws_layout, int path, cudaStream_t stream) {
    return qdot_impl(A, AS, W, WS, C, nullptr, M, N, K, ws_layout, path, stream);
}

int pq_quantize_qdot_q8_0(const float* x, int8_t* A, float* AS, const int8_t* W, const float* WS, float* C,
                          int64_t M, int64_t N, int64_t K, int ws_layout, cudaStream_t stream) {
    if (ws_layout != PQ_WS_N_KB && ws_layout != PQ_WS_KB_N) return PQ_ERR_INVALID_ARG;
    int st = check_qdot_shape(M, N, K);
    if (st != PQ_OK) return st;
    if (M == 0 || N == 0) return PQ_OK;
    if (!x || !W || !WS || !C) return PQ_ERR_INVALID_ARG;
    if ((A == nullptr) != (AS == nullptr)) return PQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(W, 16) || !aligned(WS, 4) || !aligned(C, 4)) return PQ_ERR_ALIGN;
    if (A && (!aligned(A, 16) || !aligned(AS, 4))) return PQ_ERR_ALIGN;
    // one kernel for a single row whose grid fits one wave
    pq::FusedArgs f{x, A, AS, W, WS, C, M, N, K, ws_layout};
    cudaError_t e = pq::launch_qdot_fused(f, stream);
    if (e != cudaErrorNotSupported) return map_cuda(e);
    // 9..16 rows with the register-fed warp-level MMA kernel selected
    // (pq_debug_set_small_kernel(0)): one kernel as well, whose CTAs quantize
    // the rows of their K ranges themselves.  With the TMA-fed kernel (the
    // default) the quantizer followed by qdot_t is faster (21.0 against 25.0
    // us at K = 4096, N = 11008: every CTA of a one-kernel step quantizes its
    // K chunk of all rows again)
    if (M > 8 && M <= 16 && pq::small_kernel() == 0) {
        e = pq::launch_qdot_mma_fused(f, stream);
        if (e != cudaErrorNotSupported) return map_cuda(e);
    }
    // otherwise the quantizer, then qdot_t (the second launch overlaps the first);
    // the quantized rows go to A / AS, or to this stream's workspace
    if (!A) {
        void* ws = nullptr;
        const size_t qbytes = (static_cast<size_t>(M * K) + 255) & ~size_t(255);
        e = pq::stream_workspace(stream, qbytes + static_cast<size_t>(M * (K / 32)) * sizeof(float), &ws, 2);
        if (e != cudaSuccess) return map_cuda(e);
        A = static_cast<int8_t*>(ws);
        AS = reinterpret_cast<float*>(static_cast<char*>(ws) + qbytes);
    }
    // 9..16 rows on the TMA-fed kernel: the quantizer lets qdot_t in only
    // after its own wait, and qdot_t then streams its first weight stages
    // while the quantizer runs
    const bool early = M > 8 && M <= 16 && pq::small_kernel() == 1;
    if (!aligned(A, 16) || !aligned(AS, 4)) return PQ_ERR_ALIGN;
    e = pq::launch_quantize(x, A, AS, M, K, stream, early);
    if (e != cudaSuccess) return map_cuda(e);
    return qdot_impl(A, AS, W, WS, C, nullptr, M, N, K, ws_layout, PQ_PATH_AUTO, stream, 0, early ? 1 : 0);
}

int pq_quantize_qdot_q8_0_host(const float* x_host, const int8_t* W, const float* WS, float* C_host, int64_t M,
                               int64_t N, int64_t K, int ws_layout, cudaStream_t stream) {
    if (ws_layout != PQ_WS_N_KB && ws_layout != PQ_WS_KB_N) return PQ_ERR_INVALID_ARG;
    int st = check_qdot_shape(M, N, K);
    if (st != PQ_OK) return st;
    if (M == 0 || N == 0) return PQ_OK;
    if (!x_host || !W || !WS || !C_host) return PQ_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(WS, 4)) return PQ_ERR_ALIGN;
    // C in page-locked host memory the device can address (on GB300 host memory
    // is reached over the coherent chip-to-chip link): the step writes it there
    // itself, with no device-to-host copy.  x is still copied in (one copy into
    // this stream's workspace): read in place, every CTA of the step would pull
    // the whole row over the link.
    float* cd = g_host_path == 0 ? static_cast<float*>(device_view(C_host)) : nullptr;
    if (cd && aligned(cd, 4)) {
        const size_t xbytes = static_cast<size_t>(M * K) * sizeof(float);
        void* ws = nullptr;
        cudaError_t e = pq::stream_workspace(stream, xbytes, &ws, 1);
        if (e != cudaSuccess) return map_cuda(e);
        e = cudaMemcpyAsync(ws, x_host, xbytes, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return map_cuda(e);
        return pq_quantize_qdot_q8_0(static_cast<const float*>(ws), nullptr, nullptr, W, WS, cd, M, N, K, ws_layout,
                                     stream);
    }
    // device copies of x and C in this stream's staging workspace
    const size_t xbytes = static_cast<size_t>(M * K) * sizeof(float);
    const size_t cbytes = static_cast<size_t>(M * N) * sizeof(float);
    const size_t coff = (xbytes + 255) & ~size_t(255);
    void* ws = nullptr;
    cudaError_t e = pq::stream_workspace(stream, coff + cbytes, &ws, 1);
    if (e != cudaSuccess) return map_cuda(e);
    float* x = static_cast<float*>(ws);
    float* C = reinterpret_cast<float*>(static_cast<char*>(ws) + coff);
    e = cudaMemcpyAsync(x, x_host, xbytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return map_cuda(e);
    st = pq_quantize_qdot_q8_0(x, nullptr, nullptr, W, WS, C, M, N, K, ws_layout, stream);
    if (st != PQ_OK) return st;
    return map_cuda(cudaMemcpyAsync(C_host, C, cbytes, cudaMemcpyDeviceToHost, stream));
}

int pq_qdot_q8_0_blocksums(const int8_t* A, const int8_t* W, int32_t* S, int64_t M, int64_t N,
                           int64_t K, int path, cudaStream_t stream) {
    int st = check_qdot_shape(M, N, K);
    if (st != PQ_OK) return st;
    if (M == 0 || N == 0) return PQ_OK;
    if (!S) return PQ_ERR_INVALID_ARG;
    if (path == PQ_PATH_AUTO) path = PQ_PATH_SIMT;
    return qdot_impl(A, nullptr, W, nullptr, nullptr, S, M, N, K, PQ_WS_N_KB, path, stream);
}

int pq_q50_qdot(const int8_t* A, const float* AS, const uint8_t* W5, const float* WS, float* C,
                int64_t M, int64_t N, int64_t K, int ws_layout, cudaStream_t stream) {
    if (ws_layout != PQ_WS_N_KB && ws_layout != PQ_WS_KB_N) return PQ_ERR_INVALID_ARG;
    int st = check_qdot_shape(M, N, K);
    if (st != PQ_OK) return st;
    if ((__int128)N * (K / 32) * 20 > (__int128)INT64_MAX) return PQ_ERR_SHAPE;
    if (M == 0 || N == 0) return PQ_OK;
    if (!A || !AS || !W5 || !WS || !C) return PQ_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(W5, 4) || !aligned(AS, 4) || !aligned(WS, 4) || !aligned(C, 4))
        return PQ_ERR_ALIGN;
    pq::QdotArgs a{A, AS, reinterpret_cast<const int8_t*>(W5), WS, C, nullptr, M, N, K, ws_layout};
    // prompt shapes on the tensor cores (Q5_0 blocks decoded to f16 in the
    // kernel); every other shape, and whatever that kernel declines (K not a
    // multiple of 128, bases not 16-byte aligned), on the dp4a kernel
    if (M > 64) {
        cudaError_t e = pq::launch_qdot_tc_q50(a, stream);
        if (e != cudaErrorNotSupported) return map_cuda(e);
    }
    return map_cuda(pq::launch_qdot_q50(a, stream));
}

int pq_quantize_q50_qdot(const float* x, int8_t* A, float* AS, const uint8_t* W5, const float* WS, float* C,
                         int64_t M, int64_t N, int64_t K, int ws_layout, cudaStream_t stream) {
    if (ws_layout != PQ_WS_N_KB && ws_layout != PQ_WS_KB_N) return PQ_ERR_INVALID_ARG;
    int st = check_qdot_shape(M, N, K);
    if (st != PQ_OK) return st;
    if ((__int128)N * (K / 32) * 20 > (__int128)INT64_MAX) return PQ_ERR_SHAPE;
    if (M == 0 || N == 0) return PQ_OK;
    if (!x || !W5 || !WS || !C) return PQ_ERR_INVALID_ARG;
    if ((A == nullptr) != (AS == nullptr)) return PQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(W5, 4) || !aligned(WS, 4) || !aligned(C, 4)) return PQ_ERR_ALIGN;
    if (A && (!aligned(A, 16) || !aligned(AS, 4))) return PQ_ERR_ALIGN;
    // one kernel for a single row whose grid fits two waves
    pq::FusedArgs f{x, A, AS, reinterpret_cast<const int8_t*>(W5), WS, C, M, N, K, ws_layout};
    cudaError_t e = pq::launch_qdot_q50_fused(f, stream);
    if (e != cudaErrorNotSupported) return map_cuda(e);
    // otherwise the quantizer, then q50_qdot_t; the quantized rows go to A / AS,
    // or to this stream's workspace
    if (!A) {
        void* ws = nullptr;
        const size_t qbytes = (static_cast<size_t>(M * K) + 255) & ~size_t(255);
        e = pq::stream_workspace(stream, qbytes + static_cast<size_t>(M * (K / 32)) * sizeof(float), &ws, 2);
        if (e != cudaSuccess) return map_cuda(e);
        A = static_cast<int8_t*>(ws);
        AS = reinterpret_cast<float*>(static_cast<char*>(ws) + qbytes);
    }
    st = pq_quantize_q8_0(x, A, AS, M, K, stream);
    if (st != PQ_OK) return st;
    return pq_q50_qdot(A, AS, W5, WS, C, M, N, K, ws_layout, stream);
}

int pq_q50_blocksums(const int8_t* A, const uint8_t* W5, int32_t* S, int64_t M, int64_t N, int64_t K,
                     cudaStream_t stream) {
    int st = check_qdot_shape(M, N, K);
    if (st != PQ_OK) return st;
    if ((__int128)N * (K / 32) * 20 > (__int128)INT64_MAX) return PQ_ERR_SHAPE;
    if (M == 0 || N == 0) return PQ_OK;
    if (!A || !W5 || !S) return PQ_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(W5, 4) || !aligned(S, 4)) return PQ_ERR_ALIGN;
    pq::QdotArgs a{A, nullptr, reinterpret_cast<const int8_t*>(W5), nullptr, nullptr, S, M, N, K, PQ_WS_N_KB};
    return map_cuda(pq::launch_qdot_q50(a, stream));
}

int pq_check_device(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PQ_ERR_CUDA;
    unsigned status = 0, status_w = 0, status_m = 0, status_s = 0;
    if (pq::read_and_clear_status(&status) != cudaSuccess) return PQ_ERR_CUDA;
    if (pq::read_and_clear_status_w(&status_w) != cudaSuccess) return PQ_ERR_CUDA;
    if (pq::read_and_clear_status_mmt(&status_m) != cudaSuccess) return PQ_ERR_CUDA;
    if (pq::read_and_clear_status_simt(&status_s) != cudaSuccess) return PQ_ERR_CUDA;
    return (status | status_w | status_m | status_s) ? PQ_ERR_TIMEOUT : PQ_OK;
}

const char* pq_strerror(int code) {
    switch (code) {
        case PQ_OK: return "ok";
        case PQ_ERR_INVALID_ARG: return "invalid argument (null pointer or unknown code)";
        case PQ_ERR_SHAPE: return "bad shape (negative size, K not a positive multiple of 32, or overflow)";
        case PQ_ERR_ALIGN: return "misaligned base pointer";
        case PQ_ERR_CUDA: return "CUDA runtime error";
        case PQ_ERR_TIMEOUT: return "a bounded on-device wait gave up";
        case PQ_ERR_UNSUPPORTED: return "unsupported device or shape for this path";
        case PQ_ERR_SCRATCH: return "problem larger than the fixed scratch of the allocation-free entry point";
        default: return "unknown pq_status";
    }
}

int pq_version(void) { return 105; }

int pq_last_cuda_error(void) { return g_last_cuda_error; }

int pq_debug_set_tc_fault(int skip_stage, unsigned long long timeout_cycles) {
    if (skip_stage < -1) return PQ_ERR_INVALID_ARG;
    pq::set_tc_test_hooks(skip_stage, timeout_cycles);
    pq::set_tcw_test_hooks(skip_stage, timeout_cycles);
    pq::set_mmt_test_hooks(skip_stage, timeout_cycles);
    return PQ_OK;
}

int pq_debug_set_small_kernel(int which) {
    if (which != 0 && which != 1) return PQ_ERR_INVALID_ARG;
    pq::set_small_kernel(which);
    return PQ_OK;
}

int pq_debug_set_small_split(int ks) {
    if (ks != 0 && ks != 1 && ks != 2 && ks != 4 && ks != 8) return PQ_ERR_INVALID_ARG;
    pq::set_small_split(ks);
    return PQ_OK;
}

int pq_debug_small_kernel_config(int* out4) {
    if (!out4) return PQ_ERR_INVALID_ARG;
    pq::small_kernel_config(out4);
    return PQ_OK;
}

int pq_debug_prompt_kernel_regs(void) { return pq::tcw_kernel_regs(); }

int pq_debug_set_host_path(int which) {
    if (which != 0 && which != 1) return PQ_ERR_INVALID_ARG;
    g_host_path = which;
    return PQ_OK;
}

int pq_debug_stream_read(const int8_t* W, const float* WS, int64_t rows, int64_t K, float* out, int early,
                         cudaStream_t stream) {
    if (!W || !WS || !out || rows <= 0 || K < 32 || K % 32 != 0 || (early != 0 && early != 1))
        return PQ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 31u) != 0 || !aligned(WS, 4) || !aligned(out, 4)) return PQ_ERR_ALIGN;
    return map_cuda(pq::launch_stream_read(W, WS, rows, K, out, early, stream));
}

int pq_debug_set_prompt_kernel(int which) {
    if (which != 0 && which != 1) return PQ_ERR_INVALID_ARG;
    pq::set_prompt_kernel(which);
    return PQ_OK;
}

}  // extern "C"
