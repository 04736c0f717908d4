// q50_qdot_t on CUDA cores with dp4a: Q8_0 activations against Q5_0 weights.
//
// "Phobos Language Spec", section 10 (Quantized built-ins), Q5_0 row, and
// "Quantized built-ins and formats", built-in table: qdot_t against a Q5_0
// weight held as its blocks without their f16 scale.  A weight block is 20
// bytes per 32 elements: the qh word, then 16 bytes whose byte e holds element
// e in its low nibble and element e + 16 in its high nibble; each element is
// q - 16.  qh is read as a little-endian word whose bit e is the fifth bit of
// element e.  The scales are as for qdot_t: w_scales [N, K/32] f32, or
// [K/32, N] (q50_qmma_t's layout).
//
//   out[i, j] = sum_b a_scales[i, b] * w_scales[j, b] * sum_{e<32} a[i, 32b+e] * (q[j, 32b+e] - 16)
//
// Work layout as the Q8_0 streaming kernel: a warp owns COLS output columns
// and MR activation rows; lane l takes blocks l, l + 32, ... of K.  A weight
// row is K/32 * 20 bytes, so the 32 blocks a warp reads at once are 640
// contiguous bytes: each lane loads its block as five 32-bit words, the first
// of which brings every line of the 640 bytes into L1, so the other four hit.
// The weights cross HBM at their stored size: 0.625 bytes per weight plus
// 0.125 of scale.
//
// Decode in registers: the low and high nibbles of the four data words give
// elements 0..15 and 16..31 in dp4a word order; the matching four qh bits go
// to bit 4 of each byte ((x * 0x02040810) & 0x10101010 puts bit i of x at bit
// 8i + 4, no carries), giving the unsigned q in [0, 31] per byte.  Then
//   sum_e a_e (q_e - 16) = sum_e a_e q_e - 16 sum_e a_e:
// 8 dp4a of signed activation bytes with unsigned q bytes, minus 16 times the
// activation block's byte sum, exact in int32.
#include <atomic>

#include "pq_internal.h"
#include "pq_device.cuh"

namespace pq {
namespace {

constexpr int kWarps = 8;
constexpr int kQ50Bytes = 20;

struct Q50Block {
    uint32_t w[5];  // qh, then the 16 nibble bytes as four words
};

__device__ __forceinline__ Q50Block ld_q50(const uint8_t* p, uint64_t pol) {
    Q50Block b;
#pragma unroll
    for (int t = 0; t < 5; ++t) b.w[t] = ld_wword(p + 4 * t, pol);
    return b;
}

// The four bits of x at bit 4 of the four bytes.
__device__ __forceinline__ uint32_t spread4_bit4(uint32_t x) { return (x * 0x02040810u) & 0x10101010u; }

// The block's 32 elements as unsigned q in [0, 31], word t = elements 4t .. 4t+3.
__device__ __forceinline__ u32x8 q50_unpack(const Q50Block& b) {
    u32x8 r;
    const uint32_t qh = b.w[0];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t w = b.w[1 + t];
        r.v[t] = (w & 0x0F0F0F0Fu) | spread4_bit4((qh >> (4 * t)) & 0xFu);
        r.v[4 + t] = ((w >> 4) & 0x0F0F0F0Fu) | spread4_bit4((qh >> (16 + 4 * t)) & 0xFu);
    }
    return r;
}

// sum of a_e * q_e over a block: signed activation bytes, unsigned q bytes
__device__ __forceinline__ int block_dot_su(const u32x8& a, const u32x8& q) {
    int s = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) asm("dp4a.s32.u32 %0, %1, %2, %0;" : "+r"(s) : "r"(a.v[t]), "r"(q.v[t]));
    return s;
}

// sum of the 32 signed activation bytes of a block
__device__ __forceinline__ int block_sum(const u32x8& a) {
    int s = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) s = __dp4a(static_cast<int>(a.v[t]), 0x01010101, s);
    return s;
}

// sum_e a_e (q_e - 16) of a block
__device__ __forceinline__ int q50_block_dot(const u32x8& a, const u32x8& q, int a_sum) {
    return block_dot_su(a, q) - 16 * a_sum;
}

template <int MR, int COLS, int U, bool V8, bool SUMS, int WSL>
__global__ void __launch_bounds__(kWarps * 32)
qdot_q50_kernel(QdotArgs p) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t N = p.N, M = p.M, K = p.K, KB = K >> 5;
    const int64_t row_bytes = KB * kQ50Bytes;
    const uint8_t* W5 = reinterpret_cast<const uint8_t*>(p.W);
    const int64_t j0 = (static_cast<int64_t>(blockIdx.x) * kWarps + warp) * COLS;
    const int64_t i0 = static_cast<int64_t>(blockIdx.y) * MR;
    pdl_trigger();
    if (j0 >= N) return;  // warp-uniform; no CTA-wide synchronisation below
    if (lane < COLS && j0 + lane < N) {
        // bulk L2 prefetch of the weight row when it is 16-byte aligned and sized
        const uint8_t* row = W5 + (j0 + lane) * row_bytes;
        if ((row_bytes % 16) == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0 && row_bytes < (int64_t(1) << 30))
            prefetch_l2(row, static_cast<uint32_t>(row_bytes));
    }
    pdl_wait();

    const uint64_t wpol = l2_weight_policy(gridDim.y == 1);
    bool jv[COLS];
    const uint8_t* wrow[COLS];
#pragma unroll
    for (int c = 0; c < COLS; ++c) {
        jv[c] = (j0 + c) < N;
        wrow[c] = W5 + (jv[c] ? (j0 + c) : j0) * row_bytes;
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
        Q50Block wb[U][COLS];
        float wsv[U][COLS];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t b = bb + u * 32 + lane;
#pragma unroll
            for (int c = 0; c < COLS; ++c) {
                if (b < KB && jv[c]) {
                    wb[u][c] = ld_q50(wrow[c] + b * kQ50Bytes, wpol);
                    if constexpr (!SUMS)
                        wsv[u][c] = ld_wscale(WSL == 0 ? p.WS + (j0 + c) * KB + b : p.WS + b * N + (j0 + c), wpol);
                } else {
#pragma unroll
                    for (int t = 0; t < 5; ++t) wb[u][c].w[t] = 0u;
                    wsv[u][c] = 0.0f;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t b = bb + u * 32 + lane;
            if (b >= KB) continue;
            u32x8 wq[COLS];
#pragma unroll
            for (int c = 0; c < COLS; ++c) wq[c] = q50_unpack(wb[u][c]);
#pragma unroll
            for (int r = 0; r < MR; ++r) {
                if (!iv[r]) continue;
                const u32x8 av = ld_block<V8, false>(arow[r] + b * 32);
                const int asum = block_sum(av);
                float as = 0.0f;
                if constexpr (!SUMS) as = ld_f32(p.AS + (i0 + r) * KB + b);
#pragma unroll
                for (int c = 0; c < COLS; ++c) {
                    const int s = q50_block_dot(av, wq[c], asum);
                    if constexpr (SUMS) {
                        if (jv[c]) p.S[((i0 + r) * N + (j0 + c)) * KB + b] = s;
                    } else {
                        acc[r][c] = fmaf(as * wsv[u][c], static_cast<float>(s), acc[r][c]);
                    }
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
    if (v8) return launch_pdl(qdot_q50_kernel<MR, COLS, U, true, SUMS, WSL>, grid, dim3(kWarps * 32), 0, stream, a);
    return launch_pdl(qdot_q50_kernel<MR, COLS, U, false, SUMS, WSL>, grid, dim3(kWarps * 32), 0, stream, a);
}

template <bool SUMS, int WSL>
cudaError_t launch_by_m(const QdotArgs& a, bool v8, cudaStream_t stream) {
    if (a.M == 1) return launch_tile<1, 1, 4, SUMS, WSL>(a, v8, stream);
    if (a.M == 2) return launch_tile<2, 2, 2, SUMS, WSL>(a, v8, stream);
    return launch_tile<4, 2, 2, SUMS, WSL>(a, v8, stream);
}

// ---------------------------------------------------------------------------
// Fused decode step against Q5_0 weights: quantize the activation row x [1, K]
// into this CTA's shared memory with the quantizer's exact arithmetic, then
// contract it with the Q5_0 rows as qdot_q50_kernel does (one output column
// per warp).  The order of the memory traffic is that of the Q8_0 fused step:
// an L2 prefetch of the start of the CTA's weight rows before
// griddepcontrol.wait, x loaded and quantized first after it, the first round
// of weight loads issued once the first round of x is quantized, the next
// kernel let in once the quantized row is in shared memory, and the optional
// A / AS outputs written in 16-byte pieces spread over all CTAs.
constexpr int kQ50FusedWarps = 32;            // warps (= output columns) per CTA
constexpr int64_t kQ50PrefetchBytes = 4096;   // bytes of each weight row prefetched into L2

template <int U, int WSL, int NW>
__global__ void __launch_bounds__(NW * 32)
qdot_q50_fused_kernel(FusedArgs p) {
    extern __shared__ __align__(16) uint8_t fsm[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t N = p.N, K = p.K, KB = K >> 5;
    const int64_t row_bytes = KB * kQ50Bytes;
    int8_t* a_s = reinterpret_cast<int8_t*>(fsm);       // [K]
    float* as_s = reinterpret_cast<float*>(fsm + K);    // [KB]
    int* sum_s = reinterpret_cast<int*>(fsm + K + KB * 4);  // [KB] byte sums of the quantized blocks
    const int64_t j = static_cast<int64_t>(blockIdx.x) * NW + warp;
    const bool jv = j < N;
    const uint8_t* wrow = reinterpret_cast<const uint8_t*>(p.W) + (jv ? j : 0) * row_bytes;

    if (lane == 0 && jv) {
        const int64_t kb = row_bytes < kQ50PrefetchBytes ? row_bytes : kQ50PrefetchBytes;
        if ((kb % 16) == 0 && (reinterpret_cast<uintptr_t>(wrow) & 15) == 0)
            prefetch_l2(wrow, static_cast<uint32_t>(kb));
    }
    pdl_wait();

    // weights of round `bb`: U blocks per lane, read once per launch
    const uint64_t wpol = l2_weight_policy(true);
    Q50Block wb[U];
    float wsv[U];
    auto load_round = [&](int64_t bb) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t b = bb + u * 32 + lane;
            if (jv && b < KB) {
                wb[u] = ld_q50(wrow + b * kQ50Bytes, wpol);
                wsv[u] = ld_wscale(WSL == 0 ? p.WS + j * KB + b : p.WS + b * N + j, wpol);
            } else {
#pragma unroll
                for (int t = 0; t < 5; ++t) wb[u].w[t] = 0u;
                wsv[u] = 0.0f;
            }
        }
    };

    // quantize x: 8 lanes per Q8_0 block, 4 floats each (every thread of the CTA
    // works); the next round's x load is issued before the current round is
    // quantized, and the first weight round right after the first x round
    const int64_t nthr = KB * 8;
    constexpr int64_t kRound = NW * 32;
    const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 xv = threadIdx.x < nthr ? ld_stream_f4(p.x + threadIdx.x * 4) : zero4;
    for (int64_t base = 0; base < nthr; base += kRound) {  // CTA-uniform
        const int64_t t = base + threadIdx.x;
        const int64_t tn = t + kRound;
        const float4 xn = tn < nthr ? ld_stream_f4(p.x + tn * 4) : zero4;
        const float d = q8_scale_of<8>(amax4(xv));  // every lane of the warp takes part
        const uint32_t packed = q8_pack4(xv, d, __frcp_rn(d));
        int bsum = __dp4a(static_cast<int>(packed), 0x01010101, 0);  // the block's byte sum over its 8 lanes
        bsum += __shfl_xor_sync(0xffffffffu, bsum, 1);
        bsum += __shfl_xor_sync(0xffffffffu, bsum, 2);
        bsum += __shfl_xor_sync(0xffffffffu, bsum, 4);
        if (t < nthr) {
            *reinterpret_cast<uint32_t*>(a_s + t * 4) = packed;
            if ((threadIdx.x & 7) == 0) {
                as_s[t >> 3] = d;
                sum_s[t >> 3] = bsum;
            }
        }
        xv = xn;
        if (base == 0) load_round(0);
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
            acc = fmaf(as_s[b] * wsv[u], static_cast<float>(q50_block_dot(av, q50_unpack(wb[u]), sum_s[b])), acc);
        }
    }
    const float v = warp_sum(acc);
    if (lane == 0) p.C[j] = v;
}

template <int WSL>
cudaError_t launch_q50_fused(const FusedArgs& a, cudaStream_t stream) {
    constexpr int NW = kQ50FusedWarps;
    const size_t smem = static_cast<size_t>(a.K) + static_cast<size_t>(a.K / 32) * 8;
    if (smem > 200 * 1024) return cudaErrorNotSupported;
    const int64_t grid = (a.N + NW - 1) / NW;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    auto kern = qdot_q50_fused_kernel<4, WSL, NW>;
    if (smem > 48 * 1024) {
        static std::atomic<int> raised[64];  // per device (the attribute is set in its context)
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorNotSupported;
        if (static_cast<int>(smem) > raised[dev].load()) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            raised[dev].store(static_cast<int>(smem));
        }
    }
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(NW * 32), smem, stream, a);
}

}  // namespace

cudaError_t launch_qdot_q50_fused(const FusedArgs& a, cudaStream_t stream) {
    // one row (the decode step), at most two waves of CTAs (one 1024-thread CTA per SM)
    if (a.M != 1) return cudaErrorNotSupported;
    static std::atomic<int> sm_count[64];  // the SM count of each device, queried once
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorNotSupported;
    int sms = sm_count[dev].load(std::memory_order_relaxed);
    if (sms <= 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return cudaErrorNotSupported;
        sm_count[dev].store(sms, std::memory_order_relaxed);
    }
    if ((a.N + kQ50FusedWarps - 1) / kQ50FusedWarps > 2 * static_cast<int64_t>(sms)) return cudaErrorNotSupported;
    return a.ws_layout == 0 ? launch_q50_fused<0>(a, stream) : launch_q50_fused<1>(a, stream);
}

cudaError_t launch_qdot_q50(const QdotArgs& a, cudaStream_t stream) {
    // the activation blocks take 256-bit loads when A is 32-byte aligned
    const bool v8 = (reinterpret_cast<uintptr_t>(a.A) & 31u) == 0;
    if (a.S != nullptr) return launch_by_m<true, 0>(a, v8, stream);
    if (a.ws_layout == 0) return launch_by_m<false, 0>(a, v8, stream);
    return launch_by_m<false, 1>(a, v8, stream);
}

}  // namespace pq
