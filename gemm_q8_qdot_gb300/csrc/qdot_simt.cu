// qdot_t on CUDA cores with dp4a: the decode (M = 1) matvec and the small-M
// streaming kernel.
//
// "Quantized built-ins and formats", section "Q8_0":
//   out[i, j] = sum_b a_scales[i, b] * w_scales[j, b] * sum_{k in b} a[i, k] * w[j, k]
// with the inner sum in integers, four bytes at a time with dp4a.  The weights
// cross the memory bus at their stored size (1.125 bytes per weight), which
// bounds this kernel by HBM bandwidth.
//
// Work layout (the warp-per-output pattern of the pages' lanes_matvec, "Uniform,
// warp-uniform and varying", carried to whole Q8_0 blocks):
//   * a warp owns COLS output columns j and MR activation rows i;
//   * lane l takes blocks b = l, l + 32, l + 64, ... of K; per block it loads the
//     32 weight bytes of each of its columns with ONE 256-bit load (the warp
//     reads 1 KB contiguous per column per instruction), the 32 activation
//     bytes of each row (L1-resident: every warp of the CTA reads the same
//     rows), and the block's two scales;
//   * the block sum is 8 dp4a in int32 (|S| <= 2^19, exact), then one f32
//     FMA: acc += (a_scale * w_scale) * S;
//   * U blocks per lane are loaded before any is consumed, so each lane has
//     U * COLS * 32 bytes of weights in flight;
//   * the lanes' partial sums meet in an xor butterfly (sum<over ctx.lane>)
//     and lane 0 stores.
// The kernel is launched as a programmatic dependent: before
// griddepcontrol.wait it only asks L2 to prefetch its weight rows (a hint that
// cannot return stale data), so the weight stream from HBM overlaps the tail
// of the kernel that produced the activations (normally the quantizer); every
// load proper comes after the wait.
// Ragged M and N are masked (no slice has to be in bounds, unlike the pages'
// @aligned(N = TN) example).
//
// SUMS = true instead stores every block sum S[i, j, b] as int32 (the
// verification entry point pq_qdot_q8_0_blocksums).
#include <algorithm>
#include <atomic>

#include "pq_internal.h"
#include "pq_device.cuh"

namespace pq {

// Nonzero after the fused step's bounded wait for its copy of x gave up.
__device__ unsigned g_pq_status_simt;

cudaError_t read_and_clear_status_simt(unsigned* status) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_pq_status_simt, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_pq_status_simt, &zero, sizeof(unsigned));
}

namespace {

constexpr int kWarps = 8;
// bytes of each weight row a CTA asks L2 to prefetch before griddepcontrol.wait
// (GB300, graphs of back-to-back steps: at K = 14336, 4 KB per row gives 14.0 us
// per fused decode step against 15.1 us with whole rows, and 13.6 us against
// 16.4 us for qdot_t alone; at K = 4096 it is the whole row either way)
constexpr int64_t kPrefetchBytes = 4096;
// warps (= output columns) per CTA of the fused step.  Short rows take 32: the
// grid then leaves SMs free for the next launch's first CTAs, which prefetch
// during this launch's tail (K = N = 4096: 4.76 us per step, against 5.7 us
// with 27 or 28).  Long rows take 28, so that the grid covers every SM for the
// much longer stream (K = 14336, N = 4096: 13.1 us against 14.2 us with 32).
constexpr int kFusedWarps = 32;
constexpr int kFusedWarpsLongRows = 28;
constexpr int64_t kLongRowK = 8192;

template <int MR, int COLS, int U, bool V8, bool SUMS, int WSL>
__global__ void __launch_bounds__(kWarps * 32)
qdot_simt_kernel(QdotArgs p) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t N = p.N, M = p.M, K = p.K, KB = K >> 5;
    const int64_t j0 = (static_cast<int64_t>(blockIdx.x) * kWarps + warp) * COLS;
    const int64_t i0 = static_cast<int64_t>(blockIdx.y) * MR;
    pdl_trigger();
    if (j0 >= N) return;  // warp-uniform; no CTA-wide synchronisation below
    if (lane < COLS && j0 + lane < N) {
        // one bulk L2 prefetch per weight row and scale row, of the row's first
        // kPrefetchBytes (whole rows up to K = 4096; prefetching whole long rows,
        // K = 14336, measured slower); rows of a 16-byte aligned base stay 16-byte
        // aligned since K % 32 == 0
        const int64_t kb = K < kPrefetchBytes ? K : kPrefetchBytes;
        prefetch_l2(p.W + (j0 + lane) * K, static_cast<uint32_t>(kb));
        if (WSL == 0 && !SUMS && (kb / 32 * 4) % 16 == 0 &&
            (reinterpret_cast<uintptr_t>(p.WS + (j0 + lane) * KB) & 15) == 0)
            prefetch_l2(p.WS + (j0 + lane) * KB, static_cast<uint32_t>(kb / 32 * 4));
    }
    pdl_wait();

    bool jv[COLS];
    const int8_t* wrow[COLS];
#pragma unroll
    for (int c = 0; c < COLS; ++c) {
        jv[c] = (j0 + c) < N;
        wrow[c] = p.W + (jv[c] ? (j0 + c) : j0) * K;
    }
    bool iv[MR];
    const int8_t* arow[MR];
#pragma unroll
    for (int r = 0; r < MR; ++r) {
        iv[r] = (i0 + r) < M;
        arow[r] = p.A + (iv[r] ? (i0 + r) : i0) * K;
    }

    float acc[MR][COLS];
#pragma unroll
    for (int r = 0; r < MR; ++r)
#pragma unroll
        for (int c = 0; c < COLS; ++c) acc[r][c] = 0.0f;

    for (int64_t bb = 0; bb < KB; bb += 32 * U) {
        u32x8 wv[U][COLS];
        u32x8 av[U][MR];
        float wsv[U][COLS];
        float asv[U][MR];
        // issue every load of this round first: weights (HBM stream) ...
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t b = bb + u * 32 + lane;
            const bool bv = b < KB;
#pragma unroll
            for (int c = 0; c < COLS; ++c) {
                if (bv && jv[c]) {
                    wv[u][c] = ld_block<V8, true>(wrow[c] + b * 32);
                    if constexpr (!SUMS)
                        wsv[u][c] = ld_f32(WSL == 0 ? p.WS + (j0 + c) * KB + b : p.WS + b * N + (j0 + c));
                } else {
#pragma unroll
                    for (int t = 0; t < 8; ++t) wv[u][c].v[t] = 0u;
                    wsv[u][c] = 0.0f;
                }
            }
        }
        // ... then the activations (L1 / L2 hits)
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t b = bb + u * 32 + lane;
            const bool bv = b < KB;
#pragma unroll
            for (int r = 0; r < MR; ++r) {
                if (bv && iv[r]) {
                    av[u][r] = ld_block<V8, false>(arow[r] + b * 32);
                    if constexpr (!SUMS) asv[u][r] = ld_f32(p.AS + (i0 + r) * KB + b);
                } else {
#pragma unroll
                    for (int t = 0; t < 8; ++t) av[u][r].v[t] = 0u;
                    asv[u][r] = 0.0f;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t b = bb + u * 32 + lane;
#pragma unroll
            for (int r = 0; r < MR; ++r)
#pragma unroll
                for (int c = 0; c < COLS; ++c) {
                    const int s = block_dot(av[u][r], wv[u][c]);
                    if constexpr (SUMS) {
                        if (b < KB && iv[r] && jv[c]) p.S[((i0 + r) * N + (j0 + c)) * KB + b] = s;
                    } else {
                        acc[r][c] = fmaf(asv[u][r] * wsv[u][c], static_cast<float>(s), acc[r][c]);
                    }
                }
        }
    }
    if constexpr (!SUMS) {
#pragma unroll
        for (int r = 0; r < MR; ++r)
#pragma unroll
            for (int c = 0; c < COLS; ++c) {
                const float v = warp_sum(acc[r][c]);
                if (lane == 0 && iv[r] && jv[c]) p.C[(i0 + r) * N + (j0 + c)] = v;
            }
    }
}

template <int MR, int COLS, int U, bool SUMS, int WSL>
cudaError_t launch_tile(const QdotArgs& a, bool v8, cudaStream_t stream) {
    const int64_t gx = (a.N + kWarps * COLS - 1) / (kWarps * COLS);
    const int64_t gy = (a.M + MR - 1) / MR;
    if (gx > 0x7fffffffLL || gy > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
    if (v8) return launch_pdl(qdot_simt_kernel<MR, COLS, U, true, SUMS, WSL>, grid, dim3(kWarps * 32), 0, stream, a);
    return launch_pdl(qdot_simt_kernel<MR, COLS, U, false, SUMS, WSL>, grid, dim3(kWarps * 32), 0, stream, a);
}

template <bool SUMS, int WSL>
cudaError_t launch_by_m(const QdotArgs& a, bool v8, cudaStream_t stream) {
    if (a.M == 1) return launch_tile<1, 1, 4, SUMS, WSL>(a, v8, stream);
    if (a.M == 2) return launch_tile<2, 2, 2, SUMS, WSL>(a, v8, stream);
    if (a.M <= 4) return launch_tile<4, 2, 2, SUMS, WSL>(a, v8, stream);
    // 8 rows per CTA row, one block per lane in flight: measured fastest for
    // 8 <= M <= 32 at K = 4096, N = 11008 (M = 16: 32.7 us against 37.6 us
    // with 4 rows and 2 blocks per lane)
    return launch_tile<8, 2, 1, SUMS, WSL>(a, v8, stream);
}

// ---------------------------------------------------------------------------
// Fused decode step: quantize the activation row x [1, K] into this CTA's
// shared memory with the quantizer's exact arithmetic, then contract it with W
// like qdot_simt_kernel (one output column per warp).  One launch per step
// instead of two.
//
// Order of the memory traffic (measured on GB300 in a graph of back-to-back
// steps at K = 4096, N = 4096: 4.7 us per step, against 5.6 us with the weight
// loads issued before x):
//   1. before griddepcontrol.wait the CTA asks L2 to prefetch the first 4 KB
//      of its weight rows (a hint that cannot return stale data);
//   2. after it, the CTA loads x first: x is small and sits in L2, and its
//      loads do not queue behind the CTA's own 128 KB of weight loads;
//   3. the first round of weight loads is issued once the first round of x is
//      quantized; by then most of the prefetched rows are in L2;
//   4. the next kernel on the stream is let in (griddepcontrol.launch_dependents)
//      once the quantized row is in shared memory, so that its CTAs take the SMs
//      this grid leaves free and prefetch their own weights during our tail.
// When the quantized row is requested (A / AS), every CTA writes a few 16-byte
// pieces of it from shared memory: a single writer CTA would be the last to
// finish and delay the step.
// MULTI: N exceeds the grid (one CTA per SM), so each warp takes further
// columns; otherwise one column per warp (the loop costs the single-column
// grids ~3 %, measured).
// XB: x arrives by one bulk copy into shared memory (the async proxy) and the
// first weight round is issued at once, before x is there; otherwise x is
// loaded by the threads and the first weight round follows its quantization
// (issuing it earlier delayed x's loads behind the weights').  Measured on
// GB300 (graphs of back-to-back steps): XB takes K = 4096, N = 14336 from
// 11.90 to 11.24 us and K = 14336, N = 4096 from 13.27 to 12.32 us, but
// K = N = 4096 (one column per warp) from 4.75 to 4.83 us, so it serves long
// rows and several columns per warp.
template <int U, bool V8, int WSL, int NW, bool MULTI, bool XB>
__global__ void __launch_bounds__(NW * 32)
qdot_fused_kernel(FusedArgs p) {
    extern __shared__ __align__(16) uint8_t fsm[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t N = p.N, K = p.K, KB = K >> 5;
    int8_t* a_s = reinterpret_cast<int8_t*>(fsm);           // [K]
    float* as_s = reinterpret_cast<float*>(fsm + K);        // [KB]
    // XB: x as f32 [K] after them, 16-byte aligned
    float* x_s = reinterpret_cast<float*>(fsm + ((K + KB * 4 + 15) & ~int64_t(15)));
    __shared__ __align__(8) uint64_t xbar;
    const uint32_t xbar_a = static_cast<uint32_t>(__cvta_generic_to_shared(&xbar));
    if constexpr (XB) {
        if (threadIdx.x == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(xbar_a) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncthreads();
    }
    // the warp's columns: j0, j0 + jstride, ... (one each unless N exceeds the grid)
    const int64_t j0 = static_cast<int64_t>(blockIdx.x) * NW + warp;
    const int64_t jstride = static_cast<int64_t>(gridDim.x) * NW;
    int64_t j = j0;
    bool jv = j < N;
    const int8_t* wrow = p.W + (jv ? j : 0) * K;

    if (lane == 0) {
        // each column's first kPrefetchBytes (the whole row up to K = 4096):
        // prefetching whole long rows (K = 14336) measured slower than this
        const int64_t kb = K < kPrefetchBytes ? K : kPrefetchBytes;
        for (int64_t jj = j0; jj < (MULTI ? N : (j0 < N ? j0 + 1 : j0)); jj += jstride) {
            prefetch_l2(p.W + jj * K, static_cast<uint32_t>(kb));
            if (WSL == 0 && (reinterpret_cast<uintptr_t>(p.WS + jj * KB) & 15) == 0 && (kb / 32 * 4) % 16 == 0)
                prefetch_l2(p.WS + jj * KB, static_cast<uint32_t>(kb / 32 * 4));
        }
    }
    pdl_wait();
    if constexpr (XB) {
        if (threadIdx.x == 0) {
            const uint32_t bytes = static_cast<uint32_t>(K * 4);
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(xbar_a), "r"(bytes) : "memory");
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                         ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(x_s))), "l"(p.x), "r"(bytes), "r"(xbar_a)
                         : "memory");
        }
    }

    // weights of round `bb`: U blocks per lane, read once per launch
    const uint64_t wpol = l2_weight_policy(true);
    u32x8 wv[U];
    float wsv[U];
    auto load_round = [&](int64_t bb) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t b = bb + u * 32 + lane;
            if (jv && b < KB) {  // jv: the first column exists (the later ones do by the loop)
                wv[u] = ld_wblock<V8>(wrow + b * 32, wpol);
                wsv[u] = ld_wscale(WSL == 0 ? p.WS + j * KB + b : p.WS + b * N + j, wpol);
            } else {
#pragma unroll
                for (int t = 0; t < 8; ++t) wv[u].v[t] = 0u;
                wsv[u] = 0.0f;
            }
        }
    };

    // quantize x: 8 lanes per Q8_0 block, 4 floats each, so every thread of the
    // CTA works; the next round's x load is issued before the current round is
    // quantized, and the first weight round right after the first x round
    const int64_t nthr = KB * 8;    // one float4 of x per thread and round
    constexpr int64_t kRound = NW * 32;
    const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 xv;
    if constexpr (XB) {
        load_round(0);
        // bounded wait for the copy of x (about a second at 2 GHz; giving up
        // records the failure in this file's status word, C is then undefined)
        uint32_t ok = 0;
        const long long t0 = clock64();
        for (uint32_t n = 0; !ok; ++n) {
            asm volatile("{\n\t.reg .pred q;\n\tmbarrier.try_wait.parity.shared::cta.b64 q, [%1], 0;\n\t"
                         "selp.b32 %0, 1, 0, q;\n\t}"
                         : "=r"(ok) : "r"(xbar_a) : "memory");
            if (!ok && (n & 15) == 15 && clock64() - t0 > 2000000000LL) {
                atomicOr(&g_pq_status_simt, 1u);
                break;
            }
        }
        xv = threadIdx.x < nthr ? reinterpret_cast<const float4*>(x_s)[threadIdx.x] : zero4;
    } else {
        xv = threadIdx.x < nthr ? ld_stream_f4(p.x + threadIdx.x * 4) : zero4;
    }
    for (int64_t base = 0; base < nthr; base += kRound) {  // CTA-uniform
        const int64_t t = base + threadIdx.x;
        const int64_t tn = t + kRound;
        const float4 xn = tn < nthr ? (XB ? reinterpret_cast<const float4*>(x_s)[tn] : ld_stream_f4(p.x + tn * 4))
                                    : zero4;
        const float d = q8_scale_of<8>(amax4(xv));  // every lane of the warp takes part
        if (t < nthr) {
            *reinterpret_cast<uint32_t*>(a_s + t * 4) = q8_pack4(xv, d, __frcp_rn(d));
            if ((threadIdx.x & 7) == 0) as_s[t >> 3] = d;
        }
        xv = xn;
        if (!XB && base == 0) load_round(0);
    }
    __syncthreads();
    pdl_trigger();

    if (p.A != nullptr) {
        // piece q (16 bytes of A, or one scale of AS) goes to CTA q % grid
        const int64_t g = gridDim.x;
        for (int64_t q = threadIdx.x * g + blockIdx.x; q < K / 16; q += kRound * g)
            reinterpret_cast<uint4*>(p.A)[q] = reinterpret_cast<const uint4*>(a_s)[q];
        for (int64_t q = threadIdx.x * g + blockIdx.x; q < KB; q += kRound * g) p.AS[q] = as_s[q];
    }
    if (!jv) return;
    for (;;) {
        float acc = 0.0f;
        for (int64_t bb = 0; bb < KB; bb += 32 * U) {
            if (bb > 0) load_round(bb);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t b = bb + u * 32 + lane;
                if (b >= KB) continue;
                const uint4* pa = reinterpret_cast<const uint4*>(a_s + b * 32);
                const uint4 a0 = pa[0], a1 = pa[1];
                u32x8 av;
                av.v[0] = a0.x; av.v[1] = a0.y; av.v[2] = a0.z; av.v[3] = a0.w;
                av.v[4] = a1.x; av.v[5] = a1.y; av.v[6] = a1.z; av.v[7] = a1.w;
                acc = fmaf(as_s[b] * wsv[u], static_cast<float>(block_dot(av, wv[u])), acc);
            }
        }
        const float v = warp_sum(acc);
        if (lane == 0) p.C[j] = v;
        if constexpr (!MULTI) break;
        j += jstride;  // a further column: its first round (the first column's was loaded above)
        if (j >= N) break;
        wrow = p.W + j * K;
        load_round(0);
    }
}

template <int U, int WSL, int NW, bool MULTI, bool XB>
auto fused_kernel_for(bool v8) {
    return v8 ? qdot_fused_kernel<U, true, WSL, NW, MULTI, XB> : qdot_fused_kernel<U, false, WSL, NW, MULTI, XB>;
}

template <int U, int WSL, int NW>
cudaError_t launch_fused(const FusedArgs& a, bool v8, int sms, bool long_rows, cudaStream_t stream) {
    const size_t smem0 = static_cast<size_t>(a.K) + static_cast<size_t>(a.K / 32) * 4;
    if (smem0 > 200 * 1024) return cudaErrorNotSupported;
    // one output column per warp; NW warps per CTA quantize x once for NW columns
    // one CTA per SM at most (its 1024 or 896 threads hold the SM's registers);
    // beyond that each warp takes further columns
    const int64_t grid = std::min<int64_t>((a.N + NW - 1) / NW, sms);
    const bool multi = (a.N + NW - 1) / NW > sms;
    // x by bulk copy for long rows and several columns per warp, where it fits
    const size_t smem_xb = ((smem0 + 15) & ~size_t(15)) + static_cast<size_t>(a.K) * 4;
    const bool xb = (multi || long_rows) && smem_xb <= 200 * 1024;
    const size_t smem = xb ? smem_xb : smem0;
    auto kern = multi ? (xb ? fused_kernel_for<U, WSL, NW, true, true>(v8) : fused_kernel_for<U, WSL, NW, true, false>(v8))
                      : (xb ? fused_kernel_for<U, WSL, NW, false, true>(v8) : fused_kernel_for<U, WSL, NW, false, false>(v8));
    // beyond the default 48 KB of dynamic shared memory (K > 43690) the kernel's
    // limit is raised once for the largest size met (it is per function, not per call)
    if (smem > 48 * 1024) {
        static std::atomic<int> raised[64][8];  // per device (the attribute is set in its context) and kernel
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorNotSupported;
        std::atomic<int>& r = raised[dev][(v8 ? 1 : 0) + (multi ? 2 : 0) + (xb ? 4 : 0)];
        if (static_cast<int>(smem) > r.load()) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            r.store(static_cast<int>(smem));
        }
    }
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(NW * 32), smem, stream, a);
}

}  // namespace

cudaError_t launch_qdot_fused(const FusedArgs& a, cudaStream_t stream) {
    // one row (the decode step); at most one CTA per SM, whose warps take further
    // columns when N exceeds the grid
    if (a.M != 1) return cudaErrorNotSupported;
    // the SM count of each device, queried once
    static std::atomic<int> sm_count[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorNotSupported;
    int sms = sm_count[dev].load(std::memory_order_relaxed);
    if (sms <= 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return cudaErrorNotSupported;
        sm_count[dev].store(sms, std::memory_order_relaxed);
    }
    const bool long_rows = a.K >= kLongRowK;
    const bool v8 = (reinterpret_cast<uintptr_t>(a.W) & 31u) == 0;
    if (long_rows)
        return a.ws_layout == 0 ? launch_fused<4, 0, kFusedWarpsLongRows>(a, v8, sms, true, stream)
                                : launch_fused<4, 1, kFusedWarpsLongRows>(a, v8, sms, true, stream);
    return a.ws_layout == 0 ? launch_fused<4, 0, kFusedWarps>(a, v8, sms, false, stream)
                            : launch_fused<4, 1, kFusedWarps>(a, v8, sms, false, stream);
}

namespace {

// Test-only streaming reader: the fused decode step's memory traffic without
// its arithmetic.  One warp per weight row (kFusedWarps rows per CTA, at most
// one CTA per SM), the same L2 prefetch before griddepcontrol.wait, the same
// 256-bit evict-first loads of U blocks per lane and of their scales; the
// loaded words are folded into a checksum per row so that no load is dead.
template <bool EARLY>
__global__ void __launch_bounds__(kFusedWarps * 32)
stream_read_kernel(const int8_t* __restrict__ W, const float* __restrict__ WS, int64_t rows, int64_t K,
                   float* __restrict__ out) {
    constexpr int U = 4;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t KB = K >> 5;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kFusedWarps + warp;
    const bool jv = j < rows;
    const int8_t* wrow = W + (jv ? j : 0) * K;
    if (lane == 0 && jv) {
        const int64_t kb = K < kPrefetchBytes ? K : kPrefetchBytes;
        prefetch_l2(wrow, static_cast<uint32_t>(kb));
        if ((reinterpret_cast<uintptr_t>(WS + j * KB) & 15) == 0 && (kb / 32 * 4) % 16 == 0)
            prefetch_l2(WS + j * KB, static_cast<uint32_t>(kb / 32 * 4));
    }
    const uint64_t wpol = l2_weight_policy(true);
    u32x8 wv[U];
    float wsv[U];
    auto load_round = [&](int64_t bb) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t b = bb + u * 32 + lane;
            if (jv && b < KB) {
                wv[u] = ld_wblock<true>(wrow + b * 32, wpol);
                wsv[u] = ld_wscale(WS + j * KB + b, wpol);
            } else {
#pragma unroll
                for (int t = 0; t < 8; ++t) wv[u].v[t] = 0u;
                wsv[u] = 0.0f;
            }
        }
    };
    if constexpr (EARLY) load_round(0);
    pdl_wait();
    pdl_trigger();
    if constexpr (!EARLY) load_round(0);
    uint32_t h = 0;
    float s = 0.0f;
    for (int64_t bb = 0; bb < KB; bb += 32 * U) {
        if (bb > 0) load_round(bb);
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int t = 0; t < 8; ++t) h += wv[u].v[t];
            s += wsv[u];
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        h += __shfl_xor_sync(0xffffffffu, h, o);
        s += __shfl_xor_sync(0xffffffffu, s, o);
    }
    if (lane == 0 && jv) out[j] = s + static_cast<float>(h & 0xffu);
}

}  // namespace

cudaError_t launch_stream_read(const int8_t* W, const float* WS, int64_t rows, int64_t K, float* out, int early,
                               cudaStream_t stream) {
    if ((reinterpret_cast<uintptr_t>(W) & 31u) != 0 || K % 32 != 0 || rows <= 0) return cudaErrorInvalidValue;
    const int64_t grid = (rows + kFusedWarps - 1) / kFusedWarps;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    return early ? launch_pdl(stream_read_kernel<true>, dim3(static_cast<unsigned>(grid)), dim3(kFusedWarps * 32), 0,
                              stream, W, WS, rows, K, out)
                 : launch_pdl(stream_read_kernel<false>, dim3(static_cast<unsigned>(grid)), dim3(kFusedWarps * 32), 0,
                              stream, W, WS, rows, K, out);
}

cudaError_t launch_qdot_simt(const QdotArgs& a, cudaStream_t stream) {
    // 256-bit loads need 32-byte aligned blocks: every row starts at a multiple
    // of 32 bytes from its base (K % 32 == 0), so only the bases decide.
    const bool v8 = ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.W)) & 31u) == 0;
    if (a.S != nullptr) return launch_by_m<true, 0>(a, v8, stream);
    if (a.ws_layout == 0) return launch_by_m<false, 0>(a, v8, stream);
    return launch_by_m<false, 1>(a, v8, stream);
}

}  // namespace pq
