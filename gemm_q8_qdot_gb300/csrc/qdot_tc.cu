// qdot_t on the sm_103a tensor cores (tcgen05), for prompt-sized M and, with
// the operands swapped, for small batches.
//
// What it computes ("Quantized built-ins and formats", section "Q8_0"; the
// integer-tensor-core variant qmma_t in "Phobos Language Spec" section 10):
//   out[i, j] = sum_b a_scales[i, b] * w_scales[j, b] * S[i, j, b],
//   S[i, j, b] = sum_{k in block b} a[i, k] * w[j, k]   (an integer).
//
// Engine.  int8 values are exact in f16, every product (|.| <= 16384) and
// every partial sum of one 32-element block (|S| <= 524288 < 2^24) is exact in
// an f32 accumulator, so a kind::f16 MMA with f32 accumulation gives the
// integer block sums S exactly, whatever order the tensor core adds in.  Each
// Q8_0 block is two K = 16 MMAs into a fresh TMEM accumulator; the epilogue
// warps read S back (tcgen05.ld) and apply acc += (xs * ys) * S in f32
// registers.  (GB300's dense int8 tensor rate is far below its f16 rate, so
// the integer MMA kind is not used.)
//
// Tile.  The "P" operand X (128 rows per tile, the MMA M and the TMEM lanes)
// and the "Q" operand Y (BN rows, the MMA N) are both K-major int8 [rows, K].
// For M > 64, X = A and Y = W (output C[p * N + q]); for M <= 64, X = W and
// Y = A with BN = M rounded up to 16 (output C[q * N + p]), so that the large
// weight matrix fills the 128-row side.  Optional split-K over gridDim.z adds
// the partial sums into a zeroed C with atomics.
//
// Pipeline (one CTA per tile, warp-specialised):
//   warp 0      TMA: int8 tiles of X and Y, 64 K per stage, 64-byte swizzle
//               -> int8 ring (full8 / empty8 mbarriers);
//   warps 2..   converters: int8 -> f16 (magic-number trick: the byte b is
//               biased to b + 128, placed under the f16 exponent of 1024 and
//               1152 is subtracted, all exact) into the UMMA K-major layout
//               with the 128-byte swizzle -> f16 ring (full16 / empty16);
//   warp 1      MMA issuer: 2 x tcgen05.mma per block into one of NBUF TMEM
//               buffers, tcgen05.commit -> tfull; commits free f16 stages;
//   epilogue    tcgen05.ld of S, f32 scale-and-accumulate in registers,
//   warps       scales prefetched one group of 4 blocks ahead (tempty).
//
// Safety.  Every mbarrier wait is bounded (a clock64 limit).  A wait that
// gives up sets the library's device status word and a CTA-wide abort flag;
// every role then runs out its loops without waiting or working (so no
// barrier is skipped), TMA loads and MMAs still in flight are drained with
// bounded waits, TMEM is freed and the kernel returns.  The host reads the
// status with pq_check_device.  No trap, no unbounded spin.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "pq_device.cuh"
#include "pq_internal.h"
#include "tc_ptx.cuh"

namespace pq {

// Nonzero after a bounded on-device wait gave up (read and cleared by
// pq_check_device through read_and_clear_status).
__device__ unsigned g_pq_status;

namespace {

constexpr int BM = 128;      // X rows per tile (MMA M, TMEM lanes)
constexpr int KS = 64;       // K elements per pipeline stage (two Q8_0 blocks)
constexpr int GROUP = 4;     // Q8_0 blocks per scale group (128 K, two stages)

struct TcParams {
    const float* xs;          // scale of X row p, block b: xs[p * xs_r + b * xs_b]
    int64_t xs_r, xs_b;
    const float* ys;          // scale of Y row q, block b: ys[q * ys_r + b * ys_b]
    int64_t ys_r, ys_b;
    float* C;                 // C[p * ldp + q * ldq]
    int64_t ldp, ldq;
    int32_t* S;               // block sums (verification): S[p * sp + q * sq + b]
    int64_t sp, sq;
    int64_t P, Q, K;
    int groups_per_split;
    int atomic;               // split-K: red.add into a zeroed C
    int vec_store;            // ldq == 1, Q % 4 == 0, C 16-byte aligned: float4 stores
    int inject_skip_stage;    // test hook: the producer skips this stage (-1: off)
    unsigned long long timeout_cycles;
};

template <int BN, int NCONV, int NEPI, int S8, int S16>
struct Cfg {
    static constexpr int kThreads = 32 * (2 + NCONV + NEPI);
    static constexpr int kE0 = 2 + NCONV;                 // first epilogue warp
    static constexpr int kNbuf = (512 / BN) < 4 ? (512 / BN) : 4;
    static constexpr int kTmemCols = (kNbuf * BN <= 32) ? 32 : (kNbuf * BN <= 64) ? 64 : (kNbuf * BN <= 128) ? 128
                                     : (kNbuf * BN <= 256) ? 256 : 512;
    static constexpr int kCW = BN / (NEPI / 4);          // columns per epilogue warp
    static constexpr int kCH = kCW < 32 ? kCW : 32;       // columns per tcgen05.ld
    static constexpr int kX8 = BM * KS;                   // int8 X tile bytes
    static constexpr int kY8 = BN * KS;
    static constexpr int kX16 = BM * KS * 2;              // f16 X tile bytes
    static constexpr int kY16 = BN * KS * 2;
    static constexpr int kOffX8 = 0;
    static constexpr int kOffY8 = kOffX8 + S8 * kX8;
    static constexpr int kOffX16 = kOffY8 + S8 * kY8;
    static constexpr int kOffY16 = kOffX16 + S16 * kX16;
    static constexpr int kOffYs = kOffY16 + S16 * kY16;   // 2 x [GROUP][BN] f32
    static constexpr int kOffBar = kOffYs + 2 * GROUP * BN * 4;
    static constexpr int kNumBars = 2 * S8 + 2 * S16 + 2 * kNbuf + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmem = kOffMisc + 16 + 1024;    // + alignment slack
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
    static_assert(NEPI == 4 || NEPI == 8, "epilogue warps cover the four TMEM lane quadrants");
    static_assert(kCW % kCH == 0 && kCH % 8 == 0, "epilogue column chunks");
    static_assert(kX8 % 1024 == 0 && kY8 % 1024 == 0 && kX16 % 1024 == 0 && kY16 % 1024 == 0, "1024-B tiles");
};

__device__ __forceinline__ void set_abort(volatile int* abort_flag) {
    if (*abort_flag == 0) {
        *abort_flag = 1;
        atomicOr(&g_pq_status, 1u);
    }
}

// Waits for the phase of `bar` with the given parity; false if the CTA is
// aborting or the wait ran past its limit (which starts the abort).
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned long long limit) {
    if (*abort_flag) return false;
    if (tc::mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (tc::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (static_cast<unsigned long long>(clock64() - t0) > limit) {
            set_abort(abort_flag);
            return false;
        }
    }
}

// Drain wait for work already in flight: ignores the abort flag, still bounded.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, unsigned long long limit) {
    const long long t0 = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (static_cast<unsigned long long>(clock64() - t0) > limit) {
            atomicOr(&g_pq_status, 2u);
            return;
        }
    }
}

// int8x4 -> two f16x2 (exact): bias the bytes to unsigned, put them under the
// f16 exponent of 1024 (0x64xx = 1024 + u), subtract 1152 = 1024 + 128.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140u);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342u);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = *reinterpret_cast<const uint32_t*>(&ha);
    hi = *reinterpret_cast<const uint32_t*>(&hb);
}

template <int BN, int NCONV, int NEPI, int S8, int S16, int MINB, bool SUMS>
__global__ void __launch_bounds__(Cfg<BN, NCONV, NEPI, S8, S16>::kThreads, MINB)
qdot_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
               const TcParams prm) {
    using CF = Cfg<BN, NCONV, NEPI, S8, S16>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + CF::kOffBar);
    uint64_t* full8 = bars;
    uint64_t* empty8 = full8 + S8;
    uint64_t* full16 = empty8 + S8;
    uint64_t* empty16 = full16 + S16;
    uint64_t* tfull = empty16 + S16;
    uint64_t* tempty = tfull + CF::kNbuf;
    uint64_t* drain = tempty + CF::kNbuf;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + CF::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + CF::kOffMisc + 4);
    float* ys_s = reinterpret_cast<float*>(smem + CF::kOffYs);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long limit = prm.timeout_cycles;

    const int64_t p0 = static_cast<int64_t>(blockIdx.x) * BM;
    const int64_t q0 = static_cast<int64_t>(blockIdx.y) * BN;
    const int ngroups = static_cast<int>(prm.K / (KS * 2));
    const int g_begin = static_cast<int>(blockIdx.z) * prm.groups_per_split;
    const int g_end = min(ngroups, g_begin + prm.groups_per_split);
    const int nst = 2 * max(0, g_end - g_begin);  // stages of this CTA
    const int st0 = 2 * g_begin;

    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int i = 0; i < S8; ++i) {
            tc::mbar_init(&full8[i], 1);
            tc::mbar_init(&empty8[i], NCONV);
        }
        for (int i = 0; i < S16; ++i) {
            tc::mbar_init(&full16[i], NCONV);
            tc::mbar_init(&empty16[i], 1);
        }
        for (int i = 0; i < CF::kNbuf; ++i) {
            tc::mbar_init(&tfull[i], 1);
            tc::mbar_init(&tempty[i], NEPI);
        }
        tc::mbar_init(drain, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::tma_prefetch_map(&tmX);
        tc::tma_prefetch_map(&tmY);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, CF::kTmemCols);
        tc::tmem_relinquish();
        tc::tc_fence_before_sync();
    }
    __syncthreads();
    tc::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // everything below reads global memory the preceding kernel may have written
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nst; ++i) {
                const int s = i % S8;
                if (!bounded_wait(&empty8[s], ((i / S8) & 1) ^ 1, abort_flag, limit)) continue;
                issued = i + 1;
                if (i == prm.inject_skip_stage) continue;  // test hook: never arrives
                tc::mbar_arrive_expect_tx(&full8[s], CF::kX8 + CF::kY8);
                const int kx = (st0 + i) * KS;
                tc::tma_load_2d(smem + CF::kOffX8 + s * CF::kX8, &tmX, &full8[s], kx, static_cast<int>(p0));
                tc::tma_load_2d(smem + CF::kOffY8 + s * CF::kY8, &tmY, &full8[s], kx, static_cast<int>(q0));
            }
            // copies in flight land before the CTA may exit
            for (int i = max(0, issued - S8); i < issued; ++i)
                if (i != prm.inject_skip_stage) drain_wait(&full8[i % S8], (i / S8) & 1, limit);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_f16_f32(BM, BN);
            int g = 0;
            for (int i = 0; i < nst; ++i) {
                const int s = i % S16;
                const bool ok = bounded_wait(&full16[s], (i / S16) & 1, abort_flag, limit);
                if (ok) tc::tc_fence_after_sync();
                const uint32_t xa = tc::smem_u32(smem + CF::kOffX16 + s * CF::kX16);
                const uint32_t ya = tc::smem_u32(smem + CF::kOffY16 + s * CF::kY16);
#pragma unroll
                for (int bb = 0; bb < 2; ++bb, ++g) {
                    const int buf = g % CF::kNbuf;
                    if (!ok || !bounded_wait(&tempty[buf], ((g / CF::kNbuf) & 1) ^ 1, abort_flag, limit)) continue;
                    tc::tc_fence_after_sync();
                    const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint32_t koff = static_cast<uint32_t>((bb * 2 + kk) * 32);  // 16 f16 = 32 B
                        tc::umma_f16(d, tc::sw128_kmajor_desc(xa + koff), tc::sw128_kmajor_desc(ya + koff), idesc,
                                     kk);
                    }
                    tc::umma_commit(&tfull[buf]);
                }
                if (ok) tc::umma_commit(&empty16[s]);
            }
            tc::umma_commit(drain);  // arrives when every MMA issued above has completed
            drain_wait(drain, 0, limit);
        }
    } else if (warp < CF::kE0) {
        // ------------------------------------------------------------ converters
        const int cw = warp - 2;
        const int r_in = lane & 7;  // row within an octet
        const int c8 = lane >> 3;   // 16-byte chunk of a 64-byte int8 row
        constexpr int kOctets = (BM + BN) / 8;
        for (int i = 0; i < nst; ++i) {
            const int s8 = i % S8, s16 = i % S16;
            int ok = 0;
            if (lane == 0)
                ok = bounded_wait(&full8[s8], (i / S8) & 1, abort_flag, limit) &&
                     bounded_wait(&empty16[s16], ((i / S16) & 1) ^ 1, abort_flag, limit);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok) {
                const uint8_t* x8 = smem + CF::kOffX8 + s8 * CF::kX8;
                const uint8_t* y8 = smem + CF::kOffY8 + s8 * CF::kY8;
                uint8_t* x16 = smem + CF::kOffX16 + s16 * CF::kX16;
                uint8_t* y16 = smem + CF::kOffY16 + s16 * CF::kY16;
                for (int o = cw; o < kOctets; o += NCONV) {
                    const bool isx = o < BM / 8;
                    const int row = (isx ? o : o - BM / 8) * 8 + r_in;
                    const uint8_t* src = (isx ? x8 : y8) + row * KS + ((c8 ^ ((row >> 1) & 3)) << 4);
                    uint8_t* dst = (isx ? x16 : y16) + row * (KS * 2);
                    const uint4 v = *reinterpret_cast<const uint4*>(src);
                    uint4 o0, o1;
                    i8x4_to_f16x4(v.x, o0.x, o0.y);
                    i8x4_to_f16x4(v.y, o0.z, o0.w);
                    i8x4_to_f16x4(v.z, o1.x, o1.y);
                    i8x4_to_f16x4(v.w, o1.z, o1.w);
                    const int j0 = 2 * c8, j1 = 2 * c8 + 1;
                    *reinterpret_cast<uint4*>(dst + ((j0 ^ (row & 7)) << 4)) = o0;
                    *reinterpret_cast<uint4*>(dst + ((j1 ^ (row & 7)) << 4)) = o1;
                }
                tc::fence_proxy_async_smem();
            }
            __syncwarp();
            if (ok && lane == 0) {
                tc::mbar_arrive(&empty8[s8]);
                tc::mbar_arrive(&full16[s16]);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int e = warp - CF::kE0;
        const int quad = warp & 3;
        const int cb = (e >> 2) * CF::kCW;
        const int et = e * 32 + lane;  // 0 .. 32 * NEPI - 1
        const int64_t p = p0 + quad * 32 + lane;
        const bool pv = p < prm.P;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
        const int ngs = nst / 2;  // scale groups of this CTA

        float acc[CF::kCW];
#pragma unroll
        for (int t = 0; t < CF::kCW; ++t) acc[t] = 0.0f;

        // scale prefetch: own row's 4 X scales, and one Y column's 4 scales per thread
        auto load_scales = [&](int G, float (&xr)[GROUP], float (&yr)[GROUP]) {
            const int64_t b0 = static_cast<int64_t>(g_begin + G) * GROUP;
#pragma unroll
            for (int bb = 0; bb < GROUP; ++bb) {
                xr[bb] = pv ? ld_f32(prm.xs + p * prm.xs_r + (b0 + bb) * prm.xs_b) : 0.0f;
                const int64_t q = q0 + et;
                yr[bb] = (et < BN && q < prm.Q) ? ld_f32(prm.ys + q * prm.ys_r + (b0 + bb) * prm.ys_b) : 0.0f;
            }
        };
        auto store_ys = [&](int buf, const float (&yr)[GROUP]) {
            if (et < BN) {
#pragma unroll
                for (int bb = 0; bb < GROUP; ++bb) ys_s[(buf * GROUP + bb) * BN + et] = yr[bb];
            }
        };

        float xs_cur[GROUP], xs_nxt[GROUP], ysr[GROUP];
        if (!SUMS && ngs > 0) {
            load_scales(0, xs_cur, ysr);
            store_ys(0, ysr);
        }
        tc::named_bar_sync(1, NEPI * 32);
        int g = 0;
        for (int G = 0; G < ngs; ++G) {
            if (!SUMS && G + 1 < ngs) load_scales(G + 1, xs_nxt, ysr);
#pragma unroll
            for (int bb = 0; bb < GROUP; ++bb, ++g) {
                const int buf = g % CF::kNbuf;
                int ok = 0;
                if (lane == 0) ok = bounded_wait(&tfull[buf], (g / CF::kNbuf) & 1, abort_flag, limit);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) continue;
                tc::tc_fence_after_sync();
                const float* ysb = ys_s + ((G & 1) * GROUP + bb) * BN + cb;
                const int64_t b = static_cast<int64_t>(g_begin) * GROUP + g;
#pragma unroll
                for (int c = 0; c < CF::kCW / CF::kCH; ++c) {
                    float sv[CF::kCH];
                    tc::TmemLd<CF::kCH>::run(t_lane + static_cast<uint32_t>(buf * BN + cb + c * CF::kCH), sv);
                    if constexpr (SUMS) {
                        if (pv) {
#pragma unroll
                            for (int t = 0; t < CF::kCH; ++t) {
                                const int64_t q = q0 + cb + c * CF::kCH + t;
                                if (q < prm.Q) prm.S[p * prm.sp + q * prm.sq + b] = static_cast<int32_t>(sv[t]);
                            }
                        }
                    } else {
                        const float xsb = xs_cur[bb];
#pragma unroll
                        for (int t = 0; t < CF::kCH; t += 4) {
                            const float4 y4 = *reinterpret_cast<const float4*>(ysb + c * CF::kCH + t);
                            acc[c * CF::kCH + t + 0] = fmaf(xsb * y4.x, sv[t + 0], acc[c * CF::kCH + t + 0]);
                            acc[c * CF::kCH + t + 1] = fmaf(xsb * y4.y, sv[t + 1], acc[c * CF::kCH + t + 1]);
                            acc[c * CF::kCH + t + 2] = fmaf(xsb * y4.z, sv[t + 2], acc[c * CF::kCH + t + 2]);
                            acc[c * CF::kCH + t + 3] = fmaf(xsb * y4.w, sv[t + 3], acc[c * CF::kCH + t + 3]);
                        }
                    }
                }
                tc::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&tempty[buf]);
            }
            if (!SUMS && G + 1 < ngs) {
                store_ys((G + 1) & 1, ysr);
#pragma unroll
                for (int bb = 0; bb < GROUP; ++bb) xs_cur[bb] = xs_nxt[bb];
            }
            tc::named_bar_sync(1, NEPI * 32);
        }
        if (!SUMS && *abort_flag == 0 && pv) {
            if (prm.vec_store) {
#pragma unroll
                for (int t = 0; t < CF::kCW; t += 4) {
                    const int64_t q = q0 + cb + t;
                    if (q < prm.Q)
                        *reinterpret_cast<float4*>(prm.C + p * prm.ldp + q) =
                            make_float4(acc[t], acc[t + 1], acc[t + 2], acc[t + 3]);
                }
            } else {
#pragma unroll
                for (int t = 0; t < CF::kCW; ++t) {
                    const int64_t q = q0 + cb + t;
                    if (q < prm.Q) {
                        float* dst = prm.C + p * prm.ldp + q * prm.ldq;
                        if (prm.atomic)
                            atomicAdd(dst, acc[t]);
                        else
                            *dst = acc[t];
                    }
                }
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after_sync();
        tc::tmem_dealloc(tmem_base, CF::kTmemCols);
    }
}

// ---------------------------------------------------------------------- host

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// int8 [rows, K] row-major, box {64 bytes of K, box_rows}, 64-byte swizzle,
// zero fill outside the tensor (ragged rows read as 0).
bool make_i8_map(CUtensorMap* map, const int8_t* base, int64_t rows, int64_t K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(KS), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
    int sms = 0;
    bool ok = false;
};

DeviceInfo device_info() {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return {};
    std::lock_guard<std::mutex> lk(mu);
    if (!have[dev]) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cache[dev].sms = sms;
        cache[dev].ok = (major == 10 && minor == 3);
        have[dev] = true;
    }
    return cache[dev];
}

int g_inject_skip_stage = -1;
unsigned long long g_timeout_cycles = 4000000000ull;  // ~2 s at 2 GHz

template <int BN, int NCONV, int NEPI, int S8, int S16, int MINB, bool SUMS>
cudaError_t launch_cfg(const CUtensorMap& mx, const CUtensorMap& my, const TcParams& prm, int64_t gx, int64_t gy,
                       int splits, cudaStream_t stream) {
    using CF = Cfg<BN, NCONV, NEPI, S8, S16>;
    auto kern = qdot_tc_kernel<BN, NCONV, NEPI, S8, S16, MINB, SUMS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::kSmem);
    if (e != cudaSuccess) return e;
    if (gx > 0x7fffffffLL || gy > 65535 || splits > 65535) return cudaErrorInvalidConfiguration;
    return launch_pdl(kern, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(splits)),
                      dim3(CF::kThreads), static_cast<size_t>(CF::kSmem), stream, mx, my, prm);
}

template <bool SUMS>
cudaError_t launch_tc(const QdotArgs& a, cudaStream_t stream) {
    const DeviceInfo dev = device_info();
    if (!dev.ok) return cudaErrorNotSupported;
    if (a.K % (KS * 2) != 0) return cudaErrorNotSupported;
    if (a.K > 0x7fffffffLL || a.M > 0x7fffffffLL || a.N > 0x7fffffffLL) return cudaErrorNotSupported;
    const int64_t KB = a.K / 32;
    const bool swap = a.M <= 64;
    TcParams prm{};
    const int64_t P = swap ? a.N : a.M;
    const int64_t Q = swap ? a.M : a.N;
    const int8_t* X = swap ? a.W : a.A;
    const int8_t* Y = swap ? a.A : a.W;
    // scale planes: AS [M, KB]; WS [N, KB] (layout 0) or [KB, N] (layout 1)
    const int64_t ws_r = a.ws_layout == 0 ? KB : 1, ws_b = a.ws_layout == 0 ? 1 : a.N;
    if (swap) {
        prm.xs = a.WS; prm.xs_r = ws_r; prm.xs_b = ws_b;
        prm.ys = a.AS; prm.ys_r = KB; prm.ys_b = 1;
        prm.ldp = 1; prm.ldq = a.N;
        prm.sp = KB; prm.sq = a.N * KB;
    } else {
        prm.xs = a.AS; prm.xs_r = KB; prm.xs_b = 1;
        prm.ys = a.WS; prm.ys_r = ws_r; prm.ys_b = ws_b;
        prm.ldp = a.N; prm.ldq = 1;
        prm.sp = a.N * KB; prm.sq = KB;
    }
    prm.C = a.C;
    prm.S = a.S;
    prm.P = P;
    prm.Q = Q;
    prm.K = a.K;
    prm.inject_skip_stage = g_inject_skip_stage;
    prm.timeout_cycles = g_timeout_cycles;

    const int BN = !swap ? 128 : (Q <= 16 ? 16 : Q <= 32 ? 32 : 64);
    const int64_t gx = (P + BM - 1) / BM;
    const int64_t gy = (Q + BN - 1) / BN;
    const int ngroups = static_cast<int>(a.K / (KS * 2));
    // split K when the tiles alone leave SMs idle (two CTAs fit an SM on the swapped path)
    int splits = 1;
    const int64_t tiles = gx * gy;
    const int64_t slots = static_cast<int64_t>(dev.sms) * (swap ? 2 : 1);
    if (tiles < slots) splits = static_cast<int>(std::min<int64_t>(ngroups, std::max<int64_t>(1, slots / tiles)));
    prm.groups_per_split = (ngroups + splits - 1) / splits;
    splits = (ngroups + prm.groups_per_split - 1) / prm.groups_per_split;
    prm.atomic = (!SUMS && splits > 1) ? 1 : 0;
    prm.vec_store = (!SUMS && !swap && !prm.atomic && (Q % 4 == 0) &&
                     (reinterpret_cast<uintptr_t>(a.C) & 15u) == 0) ? 1 : 0;

    CUtensorMap mx, my;
    if (!make_i8_map(&mx, X, P, a.K, BM) || !make_i8_map(&my, Y, Q, a.K, BN)) return cudaErrorInvalidValue;
    if (prm.atomic) {
        cudaError_t e = cudaMemsetAsync(a.C, 0, static_cast<size_t>(a.M * a.N) * sizeof(float), stream);
        if (e != cudaSuccess) return e;
    }
    if (!swap) return launch_cfg<128, 2, 8, 4, 4, 1, SUMS>(mx, my, prm, gx, gy, splits, stream);
    if (BN == 16) return launch_cfg<16, 2, 4, 3, 3, 2, SUMS>(mx, my, prm, gx, gy, splits, stream);
    if (BN == 32) return launch_cfg<32, 2, 4, 3, 3, 2, SUMS>(mx, my, prm, gx, gy, splits, stream);
    return launch_cfg<64, 2, 4, 3, 3, 2, SUMS>(mx, my, prm, gx, gy, splits, stream);
}

}  // namespace

cudaError_t launch_qdot_tc(const QdotArgs& a, cudaStream_t stream) {
    return a.S != nullptr ? launch_tc<true>(a, stream) : launch_tc<false>(a, stream);
}

cudaError_t read_and_clear_status(unsigned* status) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_pq_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_pq_status, &zero, sizeof(unsigned));
}

void set_tc_test_hooks(int inject_skip_stage, unsigned long long timeout_cycles) {
    g_inject_skip_stage = inject_skip_stage;
    g_timeout_cycles = timeout_cycles ? timeout_cycles : 4000000000ull;
}

}  // namespace pq
