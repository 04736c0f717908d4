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
#include "pq_internal.h"
#include "pq_device.cuh"

namespace pq {
namespace {

constexpr int kWarps = 8;

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
        // one bulk L2 prefetch per weight row (K bytes) and scale row; rows of a
        // 16-byte aligned base stay 16-byte aligned since K % 32 == 0
        prefetch_l2(p.W + (j0 + lane) * K, static_cast<uint32_t>(K < (int64_t(1) << 30) ? K : (int64_t(1) << 30)));
        if (WSL == 0 && !SUMS && (KB * 4) % 16 == 0 &&
            (reinterpret_cast<uintptr_t>(p.WS + (j0 + lane) * KB) & 15) == 0)
            prefetch_l2(p.WS + (j0 + lane) * KB, static_cast<uint32_t>(KB * 4));
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
    return launch_tile<4, 2, 2, SUMS, WSL>(a, v8, stream);
}

}  // namespace

cudaError_t launch_qdot_simt(const QdotArgs& a, cudaStream_t stream) {
    // 256-bit loads need 32-byte aligned blocks: every row starts at a multiple
    // of 32 bytes from its base (K % 32 == 0), so only the bases decide.
    const bool v8 = ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.W)) & 31u) == 0;
    if (a.S != nullptr) return launch_by_m<true, 0>(a, v8, stream);
    if (a.ws_layout == 0) return launch_by_m<false, 0>(a, v8, stream);
    return launch_by_m<false, 1>(a, v8, stream);
}

}  // namespace pq
