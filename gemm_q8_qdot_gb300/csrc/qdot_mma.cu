// qdot_t for a few activation rows (M <= 64) on the warp-level tensor-core MMA.
//
// What it computes (the Q8_0 contraction of the qdot_t built-in, "the inner
// sum in integers, one scale multiply per block"):
//   C[m, n] = sum_b AS[m, b] * WS[n, b] * S_b[m, n],
//   S_b[m, n] = sum over the 32 k of block b of A[m, k] * W[n, k]   (exact integer),
// or, in block-sum mode, S itself.
//
// Why this MMA for few rows.  With M <= 64 the contraction is bound by the
// weight stream (N * K bytes), not by multiply-adds.  The tcgen05 MMA needs 128
// rows on its A side, so there the weights must be that operand: converter
// warps turn every weight byte into f16 in shared memory before a small
// 128 x M x 16 MMA reads it back.  mma.sync.m16n8k16 takes its operands from
// registers: a warp turns the weight bytes it has just loaded straight into B
// fragments, and the activations (m-tiles of 16 rows) are the A side.  On this
// GPU the f16 form issues one m16n8k16 per 2 cycles per SM (~600 TFLOP/s
// dense, measured), while the int8 form (m16n8k32.s8) takes 16 cycles, so the
// int8 operands are widened to f16.
//
// Exactness.  f16 holds every int8 value; products of two of them are exact
// in f32, and a block sum (two k16 steps from zero) is an integer of magnitude
// <= 32 * 128 * 128 = 2^19, so every partial sum the MMA forms is exact.
//
// Work layout.
//   CTA: 4 warps and 128 weight rows (each warp 32 rows = four n-tiles of 8)
//   over one K range; a cluster of KS CTAs along grid y splits K, and the
//   cluster sums its partial tiles through distributed shared memory, so C is
//   written once, with no zeroing pass and no atomics.
//   The CTA converts its activation rows over its K range to f16 in shared
//   memory once; the warps read A fragments from there and the weights from
//   global memory (8 bytes per lane and block, after an L2 prefetch of the
//   CTA's rows issued before the launch waits on its predecessor).
//   In the fused step the CTA quantizes the f32 activation rows of its K range
//   itself, with the row quantizer's arithmetic, instead of reading A and AS;
//   the CTAs of the first weight-row tile also store the quantized rows.
//   K order inside a block: lane q of a row group holds k = 8q .. 8q + 7 of
//   the block; MMA step 0 takes 8q .. 8q + 3 and step 1 takes 8q + 4 .. 8q + 7
//   (as K positions 2q, 2q + 1, 2q + 8, 2q + 9).  Weights and activations use
//   the same assignment, so each block sum covers the block's 32 k once.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <atomic>

#include "pq_device.cuh"
#include "pq_internal.h"

namespace cg = cooperative_groups;

namespace pq {
namespace {

constexpr int kMmaWarps = 4;
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr int kNT = 4;                    // n-tiles of 8 weight rows per warp
constexpr int kWarpRows = 8 * kNT;
constexpr int kMmaRows = kMmaWarps * kWarpRows;  // weight rows per CTA
constexpr int kUnroll = 2;                // blocks per group of weight loads (two groups in flight)
constexpr int kMaxSplits = 8;             // portable cluster size
constexpr int kWsStride = kMmaRows + 2;   // floats per block of the weight-scale tile (bank spread)

struct MmaParams {
    const int8_t* A;    // [M, K]
    const float* AS;    // [M, K/32]
    const int8_t* W;    // [N, K]
    const float* WS;    // WS[n * ws_r + b * ws_b]
    float* C;           // [M, N]
    int32_t* S;         // block-sum mode: [M, N, K/32]
    const float* X;     // fused step: f32 [M, K] rows quantized in the staging (A, AS unused), or null
    int8_t* Aq;         // fused step: optional outputs, the quantized rows [M, K] and their scales [M, K/32]
    float* ASq;
    int64_t M, N, K;
    int64_t ws_r, ws_b;
    int nb;             // blocks per K split (the last split may have fewer)
    int nbp;            // nb rounded up to whole groups of kUnroll
    int a_stride;       // bytes per row of the f16 activation tile in shared memory
};

// Shared memory of one CTA, in order:
//   region 0: the f16 activation tile [16 * MT rows][a_stride bytes] (blocks of
//             the split, zero past its end); after the main loop the same bytes
//             hold the partial-sum tile for the cluster reduction,
//             [4 warps][MT][kNT n-tiles][32 lanes] float4;
//   the activation scales of the split [nbp][16 * MT], each as a pair (s, s);
//   the weight scales of the split [nbp][kWsStride] (rows 0..63; zero past N
//             and past nb).
template <int MT>
__host__ __device__ constexpr int64_t mma_region0(int a_stride) {
    return (static_cast<int64_t>(16 * MT) * a_stride > int64_t(kMmaWarps) * MT * kNT * 32 * 16)
               ? static_cast<int64_t>(16 * MT) * a_stride
               : int64_t(kMmaWarps) * MT * kNT * 32 * 16;
}
template <int MT>
__host__ __device__ constexpr int64_t mma_smem_bytes(int a_stride, int nbp) {
    return mma_region0<MT>(a_stride) + static_cast<int64_t>(nbp) * 16 * MT * 8 +
           static_cast<int64_t>(nbp) * kWsStride * 4;
}

__device__ __forceinline__ uint2 ld_w8(const int8_t* p) {
    uint2 r;
    asm volatile("ld.global.L1::no_allocate.v2.b32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

// D += A * B on one m16n8k16 tile: A 16 x 16 f16 (row), B 16 x 8 f16 (column), D f32.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// CTAs per SM the register budget is sized for: with one m-tile, five (the
// whole grid of a 4096 x 11008 problem then runs at once)
template <int MT, bool SUMS>
constexpr int mma_min_blocks() { return SUMS ? 1 : MT == 1 ? 5 : MT == 2 ? 4 : 2; }

template <int MT, bool SUMS>
__global__ void __launch_bounds__(kMmaThreads, mma_min_blocks<MT, SUMS>()) qdot_mma_kernel(const MmaParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int R = 16 * MT;  // activation rows of the tile (rows past M are zero)
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;  // fragment row group and K quarter
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kMmaRows;
    const int KB = static_cast<int>(p.K / 32);
    const int b0 = static_cast<int>(blockIdx.y) * p.nb;  // first block of this K split
    const int nb = max(0, min(p.nb, KB - b0));
    const int nbp = p.nbp;

    // this CTA's weight rows into L2 before waiting on the preceding kernel (a
    // hint: L2 is the point of coherence, so loads after the wait still see
    // that kernel's writes)
    if (tid < kMmaRows && nb > 0) {
        const int64_t n = n0 + tid;
        if (n < p.N) prefetch_l2(p.W + n * p.K + static_cast<int64_t>(b0) * 32, static_cast<uint32_t>(nb) * 32);
    }
    pdl_wait();

    // B fragments: lane loads row g of each n-tile (rows past N read the last
    // row: their scales are zero); blocks past nb read the split's last block
    // (their activation scales are zero).  The first group of weight bytes is
    // in flight while the CTA stages the rest.
    const int8_t* wp[kNT];
#pragma unroll
    for (int t = 0; t < kNT; ++t) {
        const int64_t n = min(n0 + warp * kWarpRows + 8 * t + g, p.N - 1);
        wp[t] = p.W + n * p.K + static_cast<int64_t>(b0) * 32 + 8 * q;
    }
    const int blast = max(nb - 1, 0);
    uint2 wv[kUnroll][kNT], wn[kUnroll][kNT];
    auto load_group = [&](int bb, uint2 (&dst)[kUnroll][kNT]) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
            for (int t = 0; t < kNT; ++t) dst[u][t] = ld_w8(wp[t] + min(bb + u, blast) * 32);
    };
    if (nb > 0) load_group(0, wv);

    // staging: the split's activations -> f16 tile (zero past M and past nb),
    // their scales, and the weight scales of the CTA's rows; every load of a
    // pass is issued before its first use
    uint8_t* a16 = smem;
    const int64_t r0 = mma_region0<MT>(p.a_stride);
    uint64_t* as_s = reinterpret_cast<uint64_t*>(smem + r0);
    float* ws_s = reinterpret_cast<float*>(smem + r0 + static_cast<int64_t>(nbp) * R * 8);
    // weight scales when nbp <= 32: 32 per thread, in two passes of 16 held in
    // registers across the activation staging (layout [N, K/32]: a warp's lanes
    // read 32 consecutive blocks of one row; [K/32, N]: 32 consecutive rows of
    // one block)
    constexpr int kWsPer = kMmaRows * 32 / kMmaThreads / 2;
    const bool ws_fast = !SUMS && nbp <= 32;
    auto ws_index = [&](int i, int& r, int& b) {
        if (p.ws_b == 1) {
            r = warp + kMmaWarps * i;
            b = lane;
        } else {
            r = lane + 32 * (i & 3);
            b = warp + kMmaWarps * (i >> 2);
        }
    };
    float wsr[kWsPer];
    auto ws_load = [&](int h) {
#pragma unroll
        for (int j = 0; j < kWsPer; ++j) {
            int r, b;
            ws_index(j + kWsPer * h, r, b);
            const int64_t n = n0 + r;
            wsr[j] = (n < p.N && b < nb) ? p.WS[n * p.ws_r + (b0 + b) * p.ws_b] : 0.0f;
        }
    };
    auto ws_store = [&](int h) {
#pragma unroll
        for (int j = 0; j < kWsPer; ++j) {
            int r, b;
            ws_index(j + kWsPer * h, r, b);
            if (b < nbp) ws_s[b * kWsStride + r] = wsr[j];
        }
    };
    if (ws_fast) ws_load(0);
    if (SUMS || p.X == nullptr) {
        constexpr int kPass = 8;  // 16-byte chunks per lane per pass
        const int cpr = nbp * 2;  // chunks per row
        for (int base = 0; base < R * cpr; base += kMmaWarps * 32 * kPass) {
            uint4 v[kPass];
#pragma unroll
            for (int j = 0; j < kPass; ++j) {
                const int i = base + (j * kMmaWarps + warp) * 32 + lane;  // chunk index, row-major
                const int r = i / cpr, c = i - r * cpr;
                v[j] = make_uint4(0u, 0u, 0u, 0u);
                if (i < R * cpr && r < p.M && c < nb * 2)
                    v[j] = *reinterpret_cast<const uint4*>(p.A + r * p.K + static_cast<int64_t>(b0) * 32 + c * 16);
            }
#pragma unroll
            for (int j = 0; j < kPass; ++j) {
                const int i = base + (j * kMmaWarps + warp) * 32 + lane;
                const int r = i / cpr, c = i - r * cpr;
                if (i < R * cpr) {
                    uint4 o0, o1;
                    i8x4_to_f16x4(v[j].x, o0.x, o0.y);
                    i8x4_to_f16x4(v[j].y, o0.z, o0.w);
                    i8x4_to_f16x4(v[j].z, o1.x, o1.y);
                    i8x4_to_f16x4(v[j].w, o1.z, o1.w);
                    *reinterpret_cast<uint4*>(a16 + r * p.a_stride + c * 32) = o0;
                    *reinterpret_cast<uint4*>(a16 + r * p.a_stride + c * 32 + 16) = o1;
                }
            }
        }
    } else {
        // the fused step: two lanes per Q8_0 block, 16 floats each; the block's
        // scale is the max over both lanes, then the quantizer's per-element
        // rounding (bytes and scales bit-identical to pq_quantize_q8_0); rows
        // past M and blocks past nb quantize zeros (q = 0, d = 0)
        constexpr int kPass = 2;  // block halves per lane per pass
        const int cpr = nbp * 2;  // 16-element chunks per row
        const bool store_q = p.Aq != nullptr && blockIdx.x == 0;
        for (int base = 0; base < R * cpr; base += kMmaWarps * 32 * kPass) {
            float4 v[kPass][4];
#pragma unroll
            for (int j = 0; j < kPass; ++j) {
                const int i = base + (j * kMmaWarps + warp) * 32 + lane;  // chunk index, row-major
                const int r = i / cpr, c = i - r * cpr;
                const bool live = i < R * cpr && r < p.M && c < nb * 2;
                const float* src = p.X + (live ? r * p.K + static_cast<int64_t>(b0) * 32 + c * 16 : 0);
#pragma unroll
                for (int h = 0; h < 4; ++h) v[j][h] = live ? ld_stream_f4(src + 4 * h) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < kPass; ++j) {
                const int i = base + (j * kMmaWarps + warp) * 32 + lane;
                const int r = i / cpr, c = i - r * cpr;
                // lanes 2t and 2t + 1 hold one block (cpr is even); every lane takes part
                const float d = q8_scale_of<2>(fmaxf(fmaxf(amax4(v[j][0]), amax4(v[j][1])),
                                                     fmaxf(amax4(v[j][2]), amax4(v[j][3]))));
                if (i < R * cpr) {
                    const float rc = __frcp_rn(d);
                    const uint4 q = make_uint4(q8_pack4(v[j][0], d, rc), q8_pack4(v[j][1], d, rc),
                                               q8_pack4(v[j][2], d, rc), q8_pack4(v[j][3], d, rc));
                    uint4 o0, o1;
                    i8x4_to_f16x4(q.x, o0.x, o0.y);
                    i8x4_to_f16x4(q.y, o0.z, o0.w);
                    i8x4_to_f16x4(q.z, o1.x, o1.y);
                    i8x4_to_f16x4(q.w, o1.z, o1.w);
                    *reinterpret_cast<uint4*>(a16 + r * p.a_stride + c * 32) = o0;
                    *reinterpret_cast<uint4*>(a16 + r * p.a_stride + c * 32 + 16) = o1;
                    if ((lane & 1) == 0) as_s[(c >> 1) * R + r] = f2_pack(__float_as_uint(d), __float_as_uint(d));
                    if (store_q && r < p.M && c < nb * 2) {
                        *reinterpret_cast<uint4*>(p.Aq + r * p.K + static_cast<int64_t>(b0) * 32 + c * 16) = q;
                        if ((lane & 1) == 0) p.ASq[r * static_cast<int64_t>(KB) + b0 + (c >> 1)] = d;
                    }
                }
            }
        }
    }
    if constexpr (!SUMS) {
        if (p.X == nullptr) {
#pragma unroll 4
            for (int i = tid; i < nbp * R; i += kMmaThreads) {
                const int b = i / R, r = i - b * R;
                const float v = (r < p.M && b < nb) ? p.AS[r * static_cast<int64_t>(KB) + b0 + b] : 0.0f;
                as_s[i] = f2_pack(__float_as_uint(v), __float_as_uint(v));
            }
        }
        if (ws_fast) {
            ws_store(0);
            ws_load(1);
            ws_store(1);
        } else {
            for (int i = tid; i < nbp * kMmaRows; i += kMmaThreads) {
                const int b = i / kMmaRows, r = i - b * kMmaRows;
                const int64_t n = n0 + r;
                ws_s[b * kWsStride + r] = (n < p.N && b < nb) ? p.WS[n * p.ws_r + (b0 + b) * p.ws_b] : 0.0f;
            }
        }
    }
    __syncthreads();
    pdl_trigger();

    uint64_t acc[MT][kNT][2];  // f32 pairs: (row g, cols 2q, 2q + 1), (row g + 8, same cols)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int t = 0; t < kNT; ++t) acc[mt][t][0] = acc[mt][t][1] = 0ull;

    for (int bb = 0; bb < (nb > 0 ? nbp : 0); bb += kUnroll) {
        if (bb + kUnroll < nbp) load_group(bb + kUnroll, wn);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int b = bb + u;
            uint32_t bf[kNT][4];  // per n-tile: step 0 (b0, b1), step 1 (b0, b1)
#pragma unroll
            for (int t = 0; t < kNT; ++t) {
                i8x4_to_f16x4(wv[u][t].x, bf[t][0], bf[t][1]);
                i8x4_to_f16x4(wv[u][t].y, bf[t][2], bf[t][3]);
            }
            uint64_t ws2[kNT];
            if constexpr (!SUMS) {
#pragma unroll
                for (int t = 0; t < kNT; ++t)
                    ws2[t] = *reinterpret_cast<const uint64_t*>(ws_s + b * kWsStride + warp * kWarpRows + 8 * t + 2 * q);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const uint8_t* ar = a16 + (16 * mt + g) * p.a_stride + b * 64 + q * 16;
                const uint4 lo = *reinterpret_cast<const uint4*>(ar);                   // row g
                const uint4 hi = *reinterpret_cast<const uint4*>(ar + 8 * p.a_stride);  // row g + 8
                uint64_t al = 0, ah = 0;
                if constexpr (!SUMS) {
                    al = as_s[b * R + 16 * mt + g];
                    ah = as_s[b * R + 16 * mt + g + 8];
                }
#pragma unroll
                for (int t = 0; t < kNT; ++t) {
                    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    mma_16816(s, lo.x, hi.x, lo.y, hi.y, bf[t][0], bf[t][1]);
                    mma_16816(s, lo.z, hi.z, lo.w, hi.w, bf[t][2], bf[t][3]);
                    if constexpr (SUMS) {
                        // s = (row g, col 2q), (g, 2q + 1), (g + 8, 2q), (g + 8, 2q + 1)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int64_t m = 16 * mt + g + (i >> 1) * 8;
                            const int64_t c = n0 + warp * kWarpRows + 8 * t + 2 * q + (i & 1);
                            if (b < nb && m < p.M && c < p.N)
                                p.S[(m * p.N + c) * KB + b0 + b] = static_cast<int32_t>(s[i]);
                        }
                    } else {
                        acc[mt][t][0] = f2_fma(f2_mul(al, ws2[t]), f2_pack(__float_as_uint(s[0]), __float_as_uint(s[1])),
                                               acc[mt][t][0]);
                        acc[mt][t][1] = f2_fma(f2_mul(ah, ws2[t]), f2_pack(__float_as_uint(s[2]), __float_as_uint(s[3])),
                                               acc[mt][t][1]);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
            for (int t = 0; t < kNT; ++t) wv[u][t] = wn[u][t];
    }
    if constexpr (SUMS) return;

    auto lo32 = [](uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); };
    auto hi32 = [](uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); };
    // one 2 x 2 piece of C per (warp, m-tile, n-tile, lane): rows m, m + 8, columns c, c + 1
    auto store = [&](int slot, float4 v) {
        const int l = slot & 31, t = (slot >> 5) % kNT, mt = (slot >> 5) / kNT % MT, w = (slot >> 5) / kNT / MT;
        const int64_t m = 16 * mt + (l >> 2);
        const int64_t c = n0 + w * kWarpRows + 8 * t + 2 * (l & 3);
        if (c < p.N) {
            if (m < p.M) p.C[m * p.N + c] = v.x;
            if (m + 8 < p.M) p.C[(m + 8) * p.N + c] = v.z;
        }
        if (c + 1 < p.N) {
            if (m < p.M) p.C[m * p.N + c + 1] = v.y;
            if (m + 8 < p.M) p.C[(m + 8) * p.N + c + 1] = v.w;
        }
    };
    if (gridDim.y == 1) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int t = 0; t < kNT; ++t)
                store(((warp * MT + mt) * kNT + t) * 32 + lane,
                      make_float4(lo32(acc[mt][t][0]), hi32(acc[mt][t][0]), lo32(acc[mt][t][1]), hi32(acc[mt][t][1])));
        return;
    }
    // the cluster holds this tile's K splits (cluster = grid y): each CTA puts its
    // partial tile in shared memory (over the activation tile, once every warp
    // is done with it), then sums one share of the slots over all CTAs of the
    // cluster and writes it
    __syncthreads();
    float4* red = reinterpret_cast<float4*>(smem);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int t = 0; t < kNT; ++t)
            red[((warp * MT + mt) * kNT + t) * 32 + lane] =
                make_float4(lo32(acc[mt][t][0]), hi32(acc[mt][t][0]), lo32(acc[mt][t][1]), hi32(acc[mt][t][1]));
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int ks = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    constexpr int kSlots = kMmaWarps * MT * kNT * 32;
    for (int i = tid; i * ks + rank < kSlots; i += kMmaThreads) {
        const int slot = i * ks + rank;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int j = 0; j < ks; ++j) {
            const float4 o = cluster.map_shared_rank(red, j)[slot];
            v.x += o.x;
            v.y += o.y;
            v.z += o.z;
            v.w += o.w;
        }
        store(slot, v);
    }
    cluster.sync();  // no CTA leaves while another still reads its shared memory
}

template <int MT, bool SUMS>
cudaError_t launch_mt(const MmaParams& p, int64_t tiles, int ks, cudaStream_t stream) {
    auto kern = qdot_mma_kernel<MT, SUMS>;
    const int64_t smem = mma_smem_bytes<MT>(p.a_stride, p.nbp);
    if (smem > 48 * 1024) {
        static std::atomic<int> raised[64];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorNotSupported;
        const int have = raised[dev].load(std::memory_order_relaxed);
        if (have < smem) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            raised[dev].store(static_cast<int>(smem), std::memory_order_relaxed);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(ks));
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = static_cast<unsigned>(ks);
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

int sm_count_of_current_device() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int sms = cached[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 0;
        cached[dev].store(sms, std::memory_order_relaxed);
    }
    return sms;
}

// Chooses the K split and launches; p holds the operands, the shape and the
// weight-scale layout (ws_r, ws_b) on entry.
cudaError_t launch_mma(MmaParams p, bool sums, cudaStream_t stream) {
    if (p.M < 1 || p.M > 64 || p.N < 1 || p.K % 32 != 0 || p.K > 0x7fffffffLL ||
        p.N > 0x7fffffffLL * int64_t(kMmaRows))
        return cudaErrorNotSupported;
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return cudaErrorNotSupported;
    const int MT = static_cast<int>((p.M + 15) / 16);
    const int64_t KB = p.K / 32;
    const int64_t tiles = (p.N + kMmaRows - 1) / kMmaRows;
    auto smem_of = [&](int64_t nb) {
        const int64_t nbp = (nb + kUnroll - 1) / kUnroll * kUnroll;
        const int a_stride = static_cast<int>((nbp * 64 + 127) / 128 * 128 + 64);
        switch (MT) {
            case 1: return mma_smem_bytes<1>(a_stride, static_cast<int>(nbp));
            case 2: return mma_smem_bytes<2>(a_stride, static_cast<int>(nbp));
            case 3: return mma_smem_bytes<3>(a_stride, static_cast<int>(nbp));
            default: return mma_smem_bytes<4>(a_stride, static_cast<int>(nbp));
        }
    };
    // K split: the fewest splits that give every SM about four CTAs, each split
    // at least four blocks long, with shared memory for five CTAs per SM (the
    // whole grid then runs at once)
    int ks = 1;
    for (int s = 1; s <= kMaxSplits; ++s) {
        const int64_t nb = (KB + s - 1) / s;
        if (s > 1 && nb < 4) break;
        ks = s;
        if (smem_of(nb) <= 44 * 1024 && tiles * s >= 4 * static_cast<int64_t>(sms)) break;
    }
    p.nb = static_cast<int>((KB + ks - 1) / ks);
    ks = static_cast<int>((KB + p.nb - 1) / p.nb);  // no empty split
    p.nbp = (p.nb + kUnroll - 1) / kUnroll * kUnroll;
    p.a_stride = static_cast<int>((static_cast<int64_t>(p.nbp) * 64 + 127) / 128 * 128 + 64);
    if (smem_of(p.nb) > 227 * 1024) return cudaErrorNotSupported;
    switch (MT) {
        case 1: return sums ? launch_mt<1, true>(p, tiles, ks, stream) : launch_mt<1, false>(p, tiles, ks, stream);
        case 2: return sums ? launch_mt<2, true>(p, tiles, ks, stream) : launch_mt<2, false>(p, tiles, ks, stream);
        case 3: return sums ? launch_mt<3, true>(p, tiles, ks, stream) : launch_mt<3, false>(p, tiles, ks, stream);
        default: return sums ? launch_mt<4, true>(p, tiles, ks, stream) : launch_mt<4, false>(p, tiles, ks, stream);
    }
}

}  // namespace

cudaError_t launch_qdot_mma(const QdotArgs& a, cudaStream_t stream) {
    // the TMA-fed kernel where it applies, else this file's
    if (a.S == nullptr) {
        const cudaError_t e = launch_qdot_mmt(a, stream);
        if (e != cudaErrorNotSupported) return e;
    }
    MmaParams p{};
    p.A = a.A;
    p.AS = a.AS;
    p.W = a.W;
    p.WS = a.WS;
    p.C = a.C;
    p.S = a.S;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.ws_r = a.ws_layout == 0 ? a.K / 32 : 1;
    p.ws_b = a.ws_layout == 0 ? 1 : a.N;
    return launch_mma(p, a.S != nullptr, stream);
}

cudaError_t launch_qdot_mma_fused(const FusedArgs& f, cudaStream_t stream) {
    MmaParams p{};
    p.X = f.x;
    p.Aq = f.A;
    p.ASq = f.AS;
    p.W = f.W;
    p.WS = f.WS;
    p.C = f.C;
    p.M = f.M;
    p.N = f.N;
    p.K = f.K;
    p.ws_r = f.ws_layout == 0 ? f.K / 32 : 1;
    p.ws_b = f.ws_layout == 0 ? 1 : f.N;
    return launch_mma(p, false, stream);
}

}  // namespace pq
